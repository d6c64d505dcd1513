// simt.cu - CUDA-core attention kernels (float32 path, and any head dim up to 256).
//
// The float32 workload needs these: tensor-core tf32 products cannot meet a
// 1e-5 max-abs bound, so the fp32 path keeps every product and sum in fp32 FMA.
// They also serve bf16 problems whose head dim the tensor-core kernels do not
// take.  One warp owns one query row (forward, dQ) or one key row (dK/dV) and
// walks the allowed keys (queries) 32 at a time, one per lane, folding them
// into the running (max, numerator, denominator) carry of "bpt.py",
// _blockwise_attention_fwd / scan_kv_block.
#include <math.h>

#include "bpa_internal.h"
#include "common.cuh"

namespace bpa {
namespace {

constexpr int kMaxD = 512;
constexpr int kWarps = 4;       // warps per CTA
constexpr int kRows = kWarps;   // rows per CTA: one per warp (small problems still fill the GPU)
// KP: channels per lane (lane owns dims lane + 32 i, i < KP): 2 up to 64 channels, 4 up to
// 128, 8 up to 256, 16 above

template <typename T>
__device__ __forceinline__ float ldf(const T* p);
template <>
__device__ __forceinline__ float ldf<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float ldf<__nv_bfloat16>(const __nv_bfloat16* p) {
    return __bfloat162float(*p);
}
template <typename T>
__device__ __forceinline__ void stf(T* p, float v);
template <>
__device__ __forceinline__ void stf<float>(float* p, float v) { *p = v; }
template <>
__device__ __forceinline__ void stf<__nv_bfloat16>(__nv_bfloat16* p, float v) {
    *p = __float2bfloat16_rn(v);
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Keys of the ring super-block query q meets at step `idx` (whole sequence
// when the problem has no ring or the launch is not a ring step).
__device__ __forceinline__ void ring_range(const Problem& P, bool ring, int idx, int q, int& lo,
                                           int& hi) {
    if (!ring) {
        lo = 0;
        hi = P.S - 1;
        return;
    }
    int i = q / P.ring_blk;
    int j = ((i - idx) % P.ring_n + P.ring_n) % P.ring_n;
    lo = j * P.ring_blk;
    hi = lo + P.ring_blk - 1;
}

// Whether key block kb is selected for query q (only blocks before q's own block count).
__device__ __forceinline__ bool selected(const Problem& P, int b, int h, int q, int kb) {
    const int nblk = P.S / P.sel_block;
    if (kb >= q / P.sel_block) return false;
    const int32_t* sel = P.block_idx + ((static_cast<int64_t>(b) * P.Hq + h) * nblk + q / P.sel_block) * P.top_n;
    for (int t = 0; t < P.top_n; ++t)
        if (sel[t] == kb) return true;
    return false;
}

__device__ __forceinline__ bool allowed(const Problem& P, int b, int h, int q, int k) {
    const Lens L = lens_of(P, b);
    if (q >= L.lq || k >= L.lk) return false;   // padding
    const int c = q + L.off;                    // the diagonal key of row q
    if (P.causal && k > c) return false;
    if (P.wl >= 0 && k < c - P.wl) return false;
    if (P.wr >= 0 && k > c + P.wr) return false;
    if (P.block_idx) {
        bool local = k <= q && k > q - P.local_window;
        if (!local && !selected(P, b, h, q, k / P.sel_block)) return false;
    }
    // attention dropout: a dropped entry leaves the softmax like a masked one
    if (P.drop_thr && !dropout_keep(P.drop_thr, P.drop_k0, P.drop_k1, b, h, q, k)) return false;
    return true;
}

// Narrows [lo, hi] to the keys that can be allowed for query q of batch entry b
// (lengths, causal / window diagonal).
__device__ __forceinline__ void key_span(const Problem& P, int b, int q, int& lo, int& hi) {
    const Lens L = lens_of(P, b);
    const int c = q + L.off;
    hi = min(hi, L.lk - 1);
    if (q >= L.lq) hi = -1;
    if (P.causal) hi = min(hi, c);
    if (P.wr >= 0) hi = min(hi, c + P.wr);
    if (P.wl >= 0) lo = max(lo, c - P.wl);
}

__device__ __forceinline__ float bias_at(const Problem& P, int b, int h, int q, int k) {
    if (!P.bias) return 0.f;
    return P.bias[b * P.bs[0] + h * P.bs[1] + q * P.bs[2] + k * P.bs[3]];
}

// Forward state of one query row, spread over the warp (lane owns dims lane + 32 i).
template <int KP>
struct RowState {
    float m, l;
    float acc[KP];
};

template <typename T, int KP>
__device__ void fold_keys(const Problem& P, int b, int h, int g, int q, int klo, int khi,
                          const float* sq, RowState<KP>& st) {
    const int lane = threadIdx.x & 31;
    const T* K = static_cast<const T*>(P.k);
    const T* V = static_cast<const T*>(P.v);
    for (int k0 = klo; k0 <= khi; k0 += 32) {
        const int k = k0 + lane;
        const bool ok = k <= khi && allowed(P, b, h, q, k);
        float s = -INFINITY;
        if (ok) {
            const T* kr = K + b * P.ks[0] + static_cast<int64_t>(k) * P.ks[1] + g * P.ks[2];
            float dot = 0.f;
#pragma unroll 8
            for (int c = 0; c < P.d; ++c) dot = fmaf(sq[c], ldf(kr + c), dot);
            s = dot * P.scale + bias_at(P, b, h, q, k);
        }
        const float cmax = warp_max(s);
        const float mnew = fmaxf(st.m, cmax);
        if (mnew == -INFINITY) continue;  // warp-uniform: nothing allowed yet
        const float corr = st.m == -INFINITY ? 0.f : expf(st.m - mnew);
        const float p = ok ? expf(s - mnew) : 0.f;
        st.l = st.l * corr + warp_sum(p);
#pragma unroll
        for (int i = 0; i < KP; ++i) st.acc[i] *= corr;
        const int nt = min(32, khi - k0 + 1);   // keys of this chunk inside the range
#pragma unroll 8
        for (int t = 0; t < 32; ++t) {
            const float pt = __shfl_sync(0xffffffffu, p, t);
            if (t >= nt) continue;
            const T* vr = V + b * P.vs[0] + static_cast<int64_t>(k0 + t) * P.vs[1] + g * P.vs[2];
#pragma unroll
            for (int i = 0; i < KP; ++i) {
                const int c = lane + 32 * i;
                if (c < P.dv) st.acc[i] = fmaf(pt, ldf(vr + c), st.acc[i]);
            }
        }
        st.m = mnew;
    }
}

template <typename T, int KP>
__global__ void __launch_bounds__(kWarps * 32) k_fwd_simt(const FwdArgs a) {
    const Problem& P = a.P;
    const int b = blockIdx.z, h = blockIdx.y, g = h / P.G;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __shared__ float sq[kWarps][kMaxD];
    const T* Q = static_cast<const T*>(P.q);
    const bool ring = a.acc != nullptr;
    for (int r = warp; r < kRows; r += kWarps) {
        const int q = blockIdx.x * kRows + r;
        if (q >= P.S) break;
        for (int c = lane; c < P.d; c += 32)
            sq[warp][c] = ldf(Q + b * P.qs[0] + static_cast<int64_t>(q) * P.qs[1] + h * P.qs[2] + c);
        __syncwarp();
        int lo, hi;
        ring_range(P, ring, a.ring_idx, q, lo, hi);
        key_span(P, b, q, lo, hi);
        RowState<KP> st;
        st.m = -INFINITY;
        st.l = 0.f;
#pragma unroll
        for (int i = 0; i < KP; ++i) st.acc[i] = 0.f;
        if (lo <= hi) {
            if (!P.block_idx) {
                fold_keys<T, KP>(P, b, h, g, q, lo, hi, sq[warp], st);
            } else {
                // visit each key block once: selected blocks and the blocks of
                // the local window, in ascending order (a set union)
                for (int kb = lo / P.sel_block; kb <= hi / P.sel_block; ++kb) {
                    const int k0 = max(lo, kb * P.sel_block);
                    const int k1 = min(hi, kb * P.sel_block + P.sel_block - 1);
                    const bool local = k1 > q - P.local_window && k0 <= q;
                    if (!local && !selected(P, b, h, q, kb)) continue;
                    fold_keys<T, KP>(P, b, h, g, q, k0, k1, sq[warp], st);
                }
            }
        }
        const int64_t mi = (static_cast<int64_t>(b) * P.Hq + h) * P.S + q;
        if (!ring && P.sink && q < lens_of(P, b).lq) {
            // sink logit: joins the max and the denominator, contributes no value
            const float sk = __ldg(P.sink + h);
            const float mn = fmaxf(st.m, sk);
            const float f = st.m == -INFINITY ? 0.f : expf(st.m - mn);
#pragma unroll
            for (int i = 0; i < KP; ++i) st.acc[i] *= f;
            st.l = st.l * f + expf(sk - mn);
            st.m = mn;
        }
        if (!ring) {
            const float inv = st.l > 0.f ? 1.f / st.l : 0.f;
            T* O = static_cast<T*>(a.o) + b * P.os[0] + static_cast<int64_t>(q) * P.os[1] + h * P.os[2];
#pragma unroll
            for (int i = 0; i < KP; ++i) {
                const int c = lane + 32 * i;
                if (c < P.dv) stf(O + c, st.acc[i] * inv);
            }
            if (lane == 0) {
                a.m[mi] = st.m;
                a.l[mi] = st.l;
            }
        } else {
            // merge this step's (m, l, numerator) into the carry
            const float mc = a.m[mi], lc = a.l[mi];
            const float mn = fmaxf(mc, st.m);
            if (mn != -INFINITY) {
                const float fa = mc == -INFINITY ? 0.f : expf(mc - mn);
                const float fb = st.m == -INFINITY ? 0.f : expf(st.m - mn);
                float* C = a.acc + ((static_cast<int64_t>(b) * P.S + q) * P.Hq + h) * P.dv;
#pragma unroll
                for (int i = 0; i < KP; ++i) {
                    const int c = lane + 32 * i;
                    if (c < P.dv) C[c] = C[c] * fa + st.acc[i] * fb;
                }
                __syncwarp();
                if (lane == 0) {
                    a.m[mi] = mn;
                    a.l[mi] = lc * fa + st.l * fb;
                }
            }
        }
        __syncwarp();
    }
}

// dQ contribution of the keys [klo, khi] to one query row (lane owns dims lane + 32 i):
//   acc += sum_k P (dP - D) K_k   (the scale is applied by the caller)
template <typename T, int KP>
__device__ void dq_keys(const Problem& P, int b, int h, int g, int q, int klo, int khi, const float* sq,
                        const float* sdo, float lse, float Dq, float* acc) {
    const int lane = threadIdx.x & 31;
    const T* K = static_cast<const T*>(P.k);
    const T* V = static_cast<const T*>(P.v);
    for (int k0 = klo; k0 <= khi; k0 += 32) {
        const int k = k0 + lane;
        float dS = 0.f;
        if (k <= khi && allowed(P, b, h, q, k)) {
            const T* kr = K + b * P.ks[0] + static_cast<int64_t>(k) * P.ks[1] + g * P.ks[2];
            const T* vr = V + b * P.vs[0] + static_cast<int64_t>(k) * P.vs[1] + g * P.vs[2];
            float dot = 0.f, dp = 0.f;
#pragma unroll 8
            for (int c = 0; c < P.d; ++c) dot = fmaf(sq[c], ldf(kr + c), dot);
#pragma unroll 8
            for (int c = 0; c < P.dv; ++c) dp = fmaf(sdo[c], ldf(vr + c), dp);
            const float z = dot * P.scale + bias_at(P, b, h, q, k);
            dS = expf(z - lse) * (dp - Dq);
        }
        const int nt = min(32, khi - k0 + 1);
#pragma unroll 8
        for (int t = 0; t < 32; ++t) {
            const float st = __shfl_sync(0xffffffffu, dS, t);
            if (t >= nt) continue;
            const T* kr = K + b * P.ks[0] + static_cast<int64_t>(k0 + t) * P.ks[1] + g * P.ks[2];
#pragma unroll
            for (int i = 0; i < KP; ++i) {
                const int c = lane + 32 * i;
                if (c < P.d) acc[i] = fmaf(st, ldf(kr + c), acc[i]);
            }
        }
    }
}

// dQ of one query row per warp:  dQ = scale * sum_k P (dP - D) K_k
template <typename T, int KP>
__global__ void __launch_bounds__(kWarps * 32) k_bwd_dq_simt(const BwdArgs a) {
    const Problem& P = a.P;
    const int b = blockIdx.z, h = blockIdx.y, g = h / P.G;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __shared__ float sq[kWarps][kMaxD];
    __shared__ float sdo[kWarps][kMaxD];
    const T* Q = static_cast<const T*>(P.q);
    const T* dO = static_cast<const T*>(a.dout);
    for (int r = warp; r < kRows; r += kWarps) {
        const int q = blockIdx.x * kRows + r;
        if (q >= P.S) break;
        const int64_t qoff = b * P.qs[0] + static_cast<int64_t>(q) * P.qs[1] + h * P.qs[2];
        const int64_t ooff = b * P.os[0] + static_cast<int64_t>(q) * P.os[1] + h * P.os[2];
        for (int c = lane; c < P.d; c += 32) sq[warp][c] = ldf(Q + qoff + c);
        for (int c = lane; c < P.dv; c += 32) sdo[warp][c] = ldf(dO + ooff + c);
        __syncwarp();
        const int64_t mi = (static_cast<int64_t>(b) * P.Hq + h) * a.Spad + q;
        const float lse = a.lse[mi], Dq = a.Dvec[mi];
        float acc[KP];
#pragma unroll
        for (int i = 0; i < KP; ++i) acc[i] = 0.f;
        int lo = 0, hi = P.S - 1;
        key_span(P, b, q, lo, hi);
        if (lse != INFINITY && lo <= hi) {
            if (!P.block_idx) {
                dq_keys<T, KP>(P, b, h, g, q, lo, hi, sq[warp], sdo[warp], lse, Dq, acc);
            } else {
                // the key blocks the forward visited: the local window's and the selected ones
                for (int kb = lo / P.sel_block; kb <= hi / P.sel_block; ++kb) {
                    const int k0 = max(lo, kb * P.sel_block);
                    const int k1 = min(hi, kb * P.sel_block + P.sel_block - 1);
                    const bool local = k1 > q - P.local_window && k0 <= q;
                    if (!local && !selected(P, b, h, q, kb)) continue;
                    dq_keys<T, KP>(P, b, h, g, q, k0, k1, sq[warp], sdo[warp], lse, Dq, acc);
                }
            }
        }
        T* dQ = static_cast<T*>(a.dq) + qoff;
#pragma unroll
        for (int i = 0; i < KP; ++i) {
            const int c = lane + 32 * i;
            if (c < P.d) stf(dQ + c, acc[i] * P.scale);
        }
        __syncwarp();
    }
}

// dK, dV contributions of the queries [qlo, qhi] of q head h to one key row:
//   dk += sum_q dS Q_q,   dv += sum_q P dO_q   (the scale on dk is applied by the caller)
template <typename T, int KP>
__device__ void dkdv_queries(const BwdArgs& a, int b, int h, int k, int qlo, int qhi, const float* sk,
                             const float* sv, float* dk, float* dv) {
    const Problem& P = a.P;
    const int lane = threadIdx.x & 31;
    const T* Q = static_cast<const T*>(P.q);
    const T* dO = static_cast<const T*>(a.dout);
    for (int q0 = qlo; q0 <= qhi; q0 += 32) {
        const int q = q0 + lane;
        float p = 0.f, dS = 0.f;
        if (q <= qhi && allowed(P, b, h, q, k)) {
            const int64_t mi = (static_cast<int64_t>(b) * P.Hq + h) * a.Spad + q;
            const float lse = a.lse[mi];
            if (lse != INFINITY) {
                const int64_t qoff = b * P.qs[0] + static_cast<int64_t>(q) * P.qs[1] + h * P.qs[2];
                const int64_t ooff = b * P.os[0] + static_cast<int64_t>(q) * P.os[1] + h * P.os[2];
                float dot = 0.f, dp = 0.f;
#pragma unroll 8
                for (int c = 0; c < P.d; ++c) dot = fmaf(ldf(Q + qoff + c), sk[c], dot);
#pragma unroll 8
                for (int c = 0; c < P.dv; ++c) dp = fmaf(ldf(dO + ooff + c), sv[c], dp);
                const float z = dot * P.scale + bias_at(P, b, h, q, k);
                p = expf(z - lse);
                dS = p * (dp - a.Dvec[mi]);
            }
        }
        const int nt = min(32, qhi - q0 + 1);
#pragma unroll 8
        for (int t = 0; t < 32; ++t) {
            const float pt = __shfl_sync(0xffffffffu, p, t);
            const float st = __shfl_sync(0xffffffffu, dS, t);
            if (t >= nt) continue;
            const int64_t qoff = b * P.qs[0] + static_cast<int64_t>(q0 + t) * P.qs[1] + h * P.qs[2];
            const int64_t ooff = b * P.os[0] + static_cast<int64_t>(q0 + t) * P.os[1] + h * P.os[2];
#pragma unroll
            for (int i = 0; i < KP; ++i) {
                const int c = lane + 32 * i;
                if (c < P.d) dk[i] = fmaf(st, ldf(Q + qoff + c), dk[i]);
                if (c < P.dv) dv[i] = fmaf(pt, ldf(dO + ooff + c), dv[i]);
            }
        }
    }
}

// dK, dV of one key row per warp, summed over the q heads of its group:
//   dK = scale * sum_q dS Q_q,   dV = sum_q P dO_q
// In block-selected mode (AnnAttention, faiss_block_attention) a key is seen by the
// queries whose local window holds it and by every query of the query blocks that
// selected its block; the warp finds those query blocks 32 at a time with a ballot
// (selection is per query block) and visits only them.
template <typename T, int KP>
__global__ void __launch_bounds__(kWarps * 32) k_bwd_dkdv_simt(const BwdArgs a) {
    const Problem& P = a.P;
    const int b = blockIdx.z, g = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __shared__ float sk[kWarps][kMaxD];
    __shared__ float sv[kWarps][kMaxD];
    const T* K = static_cast<const T*>(P.k);
    const T* V = static_cast<const T*>(P.v);
    for (int r = warp; r < kRows; r += kWarps) {
        const int k = blockIdx.x * kRows + r;
        if (k >= P.S) break;
        const int64_t koff = b * P.ks[0] + static_cast<int64_t>(k) * P.ks[1] + g * P.ks[2];
        const int64_t voff = b * P.vs[0] + static_cast<int64_t>(k) * P.vs[1] + g * P.vs[2];
        for (int c = lane; c < P.d; c += 32) sk[warp][c] = ldf(K + koff + c);
        for (int c = lane; c < P.dv; c += 32) sv[warp][c] = ldf(V + voff + c);
        __syncwarp();
        float dk[KP], dv[KP];
#pragma unroll
        for (int i = 0; i < KP; ++i) dk[i] = dv[i] = 0.f;
        int lo = 0, hi = P.S - 1;  // queries that may see key k
        {
            const Lens L = lens_of(P, b);
            hi = k < L.lk ? L.lq - 1 : -1;
            if (P.causal) lo = max(lo, k - L.off);
            if (P.wr >= 0) lo = max(lo, k - L.off - P.wr);
            if (P.wl >= 0) hi = min(hi, k - L.off + P.wl);
        }
        for (int h = g * P.G; h < (g + 1) * P.G && lo <= hi; ++h) {
            if (!P.block_idx) {
                dkdv_queries<T, KP>(a, b, h, k, lo, hi, sk[warp], sv[warp], dk, dv);
                continue;
            }
            const int sb = P.sel_block, kb = k / sb;
            const int llo = max(lo, k), lhi = min(hi, k + P.local_window - 1);   // local-window queries
            for (int qb0 = lo / sb; qb0 <= hi / sb; qb0 += 32) {
                const int qb = qb0 + lane;
                bool visit = false;
                if (qb <= hi / sb) {
                    const int q0 = qb * sb, q1 = q0 + sb - 1;
                    visit = (q0 <= lhi && q1 >= llo) || selected(P, b, h, q0, kb);
                }
                unsigned todo = __ballot_sync(0xffffffffu, visit);
                while (todo) {
                    const int qv = qb0 + __ffs(todo) - 1;
                    todo &= todo - 1;
                    dkdv_queries<T, KP>(a, b, h, k, max(lo, qv * sb), min(hi, qv * sb + sb - 1), sk[warp], sv[warp],
                                    dk, dv);
                }
            }
        }
        T* dK = static_cast<T*>(a.dk) + koff;
        T* dV = static_cast<T*>(a.dv) + voff;
#pragma unroll
        for (int i = 0; i < KP; ++i) {
            const int c = lane + 32 * i;
            if (c < P.d) stf(dK + c, dk[i] * P.scale);
            if (c < P.dv) stf(dV + c, dv[i]);
        }
        __syncwarp();
    }
}

}  // namespace

namespace {

template <int KP>
cudaError_t fwd_simt_kp(const FwdArgs& a, cudaStream_t s) {
    const Problem& P = a.P;
    dim3 grid((P.S + kRows - 1) / kRows, P.Hq, P.B);
    if (P.dtype == BPA_FP32)
        k_fwd_simt<float, KP><<<grid, kWarps * 32, 0, s>>>(a);
    else
        k_fwd_simt<__nv_bfloat16, KP><<<grid, kWarps * 32, 0, s>>>(a);
    return cudaGetLastError();
}

template <int KP>
cudaError_t bwd_simt_kp(const BwdArgs& a, cudaStream_t s) {
    const Problem& P = a.P;
    dim3 gq((P.S + kRows - 1) / kRows, P.Hq, P.B);
    dim3 gk((P.S + kRows - 1) / kRows, P.Hkv, P.B);
    if (P.dtype == BPA_FP32) {
        k_bwd_dq_simt<float, KP><<<gq, kWarps * 32, 0, s>>>(a);
        k_bwd_dkdv_simt<float, KP><<<gk, kWarps * 32, 0, s>>>(a);
    } else {
        k_bwd_dq_simt<__nv_bfloat16, KP><<<gq, kWarps * 32, 0, s>>>(a);
        k_bwd_dkdv_simt<__nv_bfloat16, KP><<<gk, kWarps * 32, 0, s>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace

// Channels per lane for the wider of the two head dims.
static int simt_kp(const Problem& P) {
    const int w = P.d > P.dv ? P.d : P.dv;
    return w <= 64 ? 2 : (w <= 128 ? 4 : (w <= 256 ? 8 : 16));
}

cudaError_t launch_fwd_simt(const FwdArgs& a, cudaStream_t s) {
    switch (simt_kp(a.P)) {
        case 2: return fwd_simt_kp<2>(a, s);
        case 4: return fwd_simt_kp<4>(a, s);
        case 8: return fwd_simt_kp<8>(a, s);
        default: return fwd_simt_kp<16>(a, s);
    }
}

cudaError_t launch_bwd_simt(const BwdArgs& a, cudaStream_t s) {
    switch (simt_kp(a.P)) {
        case 2: return bwd_simt_kp<2>(a, s);
        case 4: return bwd_simt_kp<4>(a, s);
        case 8: return bwd_simt_kp<8>(a, s);
        default: return bwd_simt_kp<16>(a, s);
    }
}

}  // namespace bpa
