// aux.cu - the memory-bound helper kernels around the attention kernels.
//
//   ring init / finalize: the carry of the ring sweep ("bpt.py",
//     _ring_attention_fwd: numerator = 0, denominator = 0, max = -inf before
//     the first step; output = numerator / denominator after the last);
//   backward pre-pass: D = rowsum(dO * O) ("bpt.py", _blockwise_attention_bwd,
//     dl_part) and the per-row log-sum-exp m + log(l), zeroing the float32
//     dQ accumulator;
//   backward post-pass: float32 accumulators -> output dtype;
//   a self-test of the bounded wait (a barrier that never completes).
#include <math.h>

#include "bpa_internal.h"
#include "common.cuh"

namespace bpa {
namespace {

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

__global__ void k_ring_init(float* acc, float* m, float* l, int64_t n_acc, int64_t n_rows) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n_acc; i += stride)
        acc[i] = 0.f;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n_rows; i += stride) {
        m[i] = -INFINITY;
        l[i] = 0.f;
    }
}

// one thread per (b, q, h, 8-channel group)
template <typename T>
__global__ void k_ring_finalize(const FwdArgs a) {
    const Problem& P = a.P;
    const int groups = (P.dv + 7) / 8;
    const int64_t total = static_cast<int64_t>(P.B) * P.S * P.Hq * groups;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total; i += stride) {
        const int gi = static_cast<int>(i % groups);
        int64_t r = i / groups;
        const int h = static_cast<int>(r % P.Hq);
        r /= P.Hq;
        const int q = static_cast<int>(r % P.S);
        const int b = static_cast<int>(r / P.S);
        const float lv = a.l[(static_cast<int64_t>(b) * P.Hq + h) * P.S + q];
        const float inv = lv > 0.f ? 1.f / lv : 0.f;
        const float* C = a.acc + ((static_cast<int64_t>(b) * P.S + q) * P.Hq + h) * P.dv;
        T* O = static_cast<T*>(a.o) + b * P.os[0] + static_cast<int64_t>(q) * P.os[1] + h * P.os[2];
        for (int c = gi * 8; c < min(P.dv, gi * 8 + 8); ++c) stf(O + c, C[c] * inv);
    }
}

// one warp per (b, h, q) row of the padded [B, Hq, Spad] statistics
// A backward split over two CTAs per key tile adds its dK, dV halves (bf16 pairs) into dk, dv,
// which must start at zero (contiguous bf16 [B, S, Hkv, d] and [.., dv], 16-byte aligned).
__device__ __forceinline__ void zero_split_kv(const BwdArgs& a) {
    if (a.hsplit <= 1) return;
    const Problem& P = a.P;
    const int64_t nk = static_cast<int64_t>(P.B) * P.S * P.Hkv * P.d / 8, nv = static_cast<int64_t>(P.B) * P.S * P.Hkv * P.dv / 8;
    const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < nk + nv; i += nthreads) {
        uint4* z = i < nk ? static_cast<uint4*>(a.dk) + i : static_cast<uint4*>(a.dv) + (i - nk);
        *z = make_uint4(0u, 0u, 0u, 0u);
    }
}

template <typename T>
__global__ void k_bwd_pre(const BwdArgs a, int zero_dq) {
    const Problem& P = a.P;
    const int lane = threadIdx.x & 31;
    const int64_t rows = static_cast<int64_t>(P.B) * P.Hq * a.Spad;
    const int64_t wstride = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t r = blockIdx.x * static_cast<int64_t>(blockDim.x >> 5) + (threadIdx.x >> 5); r < rows;
         r += wstride) {
        const int q = static_cast<int>(r % a.Spad);
        const int h = static_cast<int>((r / a.Spad) % P.Hq);
        const int b = static_cast<int>(r / (static_cast<int64_t>(a.Spad) * P.Hq));
        float D = 0.f, lse = INFINITY;
        if (q < P.S) {
            const int64_t off = b * P.os[0] + static_cast<int64_t>(q) * P.os[1] + h * P.os[2];
            const T* O = static_cast<const T*>(a.o) + off;
            const T* dO = static_cast<const T*>(a.dout) + off;
            float s = 0.f;
            for (int c = lane; c < P.dv; c += 32) s = fmaf(ldf(O + c), ldf(dO + c), s);
#pragma unroll
            for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            D = s;
            const int64_t mi = (static_cast<int64_t>(b) * P.Hq + h) * P.S + q;
            const float lv = a.l[mi];
            if (lv > 0.f) lse = a.m[mi] + logf(lv);
        }
        if (lane == 0) {
            a.Dvec[r] = D;
            a.lse[r] = lse;
        }
    }
    if (zero_dq) {
        const int64_t n4 = static_cast<int64_t>(P.B) * a.Spad * P.Hq * P.d / 4;
        float4* z = reinterpret_cast<float4*>(a.dq_acc);
        const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
        for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n4; i += stride)
            z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    zero_split_kv(a);
}

// bf16 rows, d % 8 == 0 and d / 8 a power of two (<= 32): each thread loads 16 bytes
// of O and of dO; the d/8 threads of a row reduce with shuffles.
__global__ void k_bwd_pre_bf16v(const BwdArgs a, int zero_dq) {
    const Problem& P = a.P;
    const int tpr = P.dv / 8;                      // threads per row (O, dO have dv channels)
    const int rpw = 32 / tpr;                      // rows per warp and step
    const int lane = threadIdx.x & 31, sub = lane % tpr;
    const int64_t rows = static_cast<int64_t>(P.B) * P.Hq * a.Spad;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    const int64_t warp_id = blockIdx.x * static_cast<int64_t>(blockDim.x >> 5) + (threadIdx.x >> 5);
    // the loop bound is uniform across the warp, so the shuffles see every lane; row indices
    // fit 32 bits (the launcher checks), so no 64-bit division is needed
    const int nrows = static_cast<int>(rows), spad = a.Spad;
    for (int rbase = static_cast<int>(warp_id) * rpw; rbase < nrows; rbase += static_cast<int>(warps) * rpw) {
        const int r = rbase + lane / tpr;
        const bool live = r < nrows;
        const int rr = live ? r : 0;
        const int q = rr % spad;
        const int bh = rr / spad;
        const int h = bh % P.Hq;
        const int b = bh / P.Hq;
        // the row's saved statistics are fetched first, so that they are in flight together
        // with O and dO
        float lv = 0.f, mv = 0.f;
        if (live && sub == 0 && q < P.S) {
            const int64_t mi = static_cast<int64_t>(bh) * P.S + q;
            lv = a.l[mi];
            mv = a.m[mi];
        }
        float s = 0.f;
        if (live && q < P.S) {
            const int64_t off = b * P.os[0] + static_cast<int64_t>(q) * P.os[1] + h * P.os[2] + sub * 8;
            const uint4 o = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.o) + off);
            const uint4 g = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.dout) + off);
            const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&o);
            const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&g);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 x = __bfloat1622float2(o2[i]), y = __bfloat1622float2(g2[i]);
                s = fmaf(x.x, y.x, s);
                s = fmaf(x.y, y.y, s);
            }
        }
        for (int o = tpr >> 1; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o, tpr);
        if (a.dq_direct && live && q < P.S)   // band backward: dq is accumulated in place (d == dv)
            *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.dq) + b * P.qs[0] + static_cast<int64_t>(q) * P.qs[1] +
                                      h * P.qs[2] + sub * 8) = make_uint4(0u, 0u, 0u, 0u);
        if (live && sub == 0) {
            const float lse = q < P.S && lv > 0.f ? mv + logf(lv) : INFINITY;
            a.Dvec[r] = q < P.S ? s : 0.f;
            a.lse[r] = lse;
        }
    }
    if (zero_dq) {
        const int64_t n4 = static_cast<int64_t>(P.B) * a.Spad * P.Hq * P.d / 4;
        float4* z = reinterpret_cast<float4*>(a.dq_acc);
        const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
        for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n4; i += nthreads)
            z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    zero_split_kv(a);
}

// float32 [B, S, H, d] accumulator -> bf16 tensor with strides (s0, s1, s2); d % 8 == 0:
// 8 consecutive channels per thread (two 16-byte loads, one 16-byte store).
__global__ void k_cast_out_bf16v(const float* src, __nv_bfloat16* dst, int B, int S, int H, int d, int64_t s0,
                                 int64_t s1, int64_t s2) {
    const int g8 = d / 8;
    const int64_t total = static_cast<int64_t>(B) * S * H * g8;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total; i += stride) {
        const int c = static_cast<int>(i % g8) * 8;
        const int64_t row = i / g8;                 // (b * S + q) * H + h
        const int h = static_cast<int>(row % H);
        const int64_t bq = row / H;
        const int q = static_cast<int>(bq % S);
        const int b = static_cast<int>(bq / S);
        const int64_t so = i * 8;
        const float4 x = *reinterpret_cast<const float4*>(src + so);
        const float4 y = *reinterpret_cast<const float4*>(src + so + 4);
        uint4 w;
        w.x = pack_bf16(x.x, x.y);
        w.y = pack_bf16(x.z, x.w);
        w.z = pack_bf16(y.x, y.y);
        w.w = pack_bf16(y.z, y.w);
        *reinterpret_cast<uint4*>(dst + b * s0 + static_cast<int64_t>(q) * s1 + h * s2 + c) = w;
    }
}

// float32 dQ accumulator of the tensor-core backward, [B, H, src_rows / 4, d, 4] (four
// consecutive queries of one channel side by side) -> bf16 tensor with strides (s0, s1, s2);
// d % 32 == 0.  One warp per group of four queries: lane l loads channels l, l+32, ... (512
// contiguous bytes per load), neighbouring lanes swap halves so that each holds a channel pair
// for two of the queries, and a store writes 64 contiguous bytes of a row.
__global__ void k_cast_dq4_bf16(const float* src, __nv_bfloat16* dst, int B, int S, int H, int d, int64_t s0,
                                int64_t s1, int64_t s2, int src_rows) {
    const int lane = threadIdx.x & 31, r4 = src_rows / 4, n4 = (S + 3) / 4;
    const bool even = (lane & 1) == 0;
    const int groups = B * H * n4;   // < 2^31 (the launcher checks): 32-bit index arithmetic
    const int wstride = gridDim.x * (blockDim.x >> 5);
    for (int g = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); g < groups; g += wstride) {
        const int q4 = g % n4;
        const int bh = g / n4;
        const int h = bh % H;
        const int b = bh / H;
        const float4* in = reinterpret_cast<const float4*>(src + (static_cast<int64_t>(bh) * r4 + q4) * d * 4);
        const int qa = q4 * 4 + (even ? 0 : 2);   // the two rows this lane writes: qa, qa + 1
        __nv_bfloat16* out = dst + b * s0 + h * s2;
        auto emit = [&](const float4& x, int c0) {
            const float y0 = __shfl_xor_sync(0xffffffffu, even ? x.z : x.x, 1);
            const float y1 = __shfl_xor_sync(0xffffffffu, even ? x.w : x.y, 1);
            const int c = c0 + lane - (even ? 0 : 1);   // first channel of this lane's pair
            const uint32_t w0 = even ? pack_bf16(x.x, y0) : pack_bf16(y0, x.z);
            const uint32_t w1 = even ? pack_bf16(x.y, y1) : pack_bf16(y1, x.w);
            if (qa < S) *reinterpret_cast<uint32_t*>(out + static_cast<int64_t>(qa) * s1 + c) = w0;
            if (qa + 1 < S) *reinterpret_cast<uint32_t*>(out + static_cast<int64_t>(qa + 1) * s1 + c) = w1;
        };
        if (d == 128) {   // the tensor-core backward's head dim: the four loads go out together
            float4 xs[4];
#pragma unroll
            for (int g = 0; g < 4; ++g) xs[g] = in[g * 32 + lane];
#pragma unroll
            for (int g = 0; g < 4; ++g) emit(xs[g], g * 32);
        } else {
            for (int c0 = 0; c0 < d; c0 += 32) emit(in[c0 + lane], c0);
        }
    }
}

__global__ void k_wait_selftest(uint32_t* status, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(smem_u32(&bar), 1);
        fence_mbar_init();
    }
    __syncthreads();
    // nothing ever arrives on `bar`: the wait must give up and report
    if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, &abort_flag, status, 0x5E1F, limit_ns);
    __syncthreads();
}

int grid_for(int64_t work, int threads) {
    int64_t g = (work + threads - 1) / threads;
    if (g < 1) g = 1;
    if (g > 152 * 32) g = 152 * 32;
    return static_cast<int>(g);
}

}  // namespace

cudaError_t launch_ring_init(const FwdArgs& a, cudaStream_t s) {
    const Problem& P = a.P;
    const int64_t n_acc = static_cast<int64_t>(P.B) * P.S * P.Hq * P.dv;
    const int64_t n_rows = static_cast<int64_t>(P.B) * P.Hq * P.S;
    k_ring_init<<<grid_for(n_acc, 256), 256, 0, s>>>(a.acc, a.m, a.l, n_acc, n_rows);
    return cudaGetLastError();
}

cudaError_t launch_ring_finalize(const FwdArgs& a, cudaStream_t s) {
    const Problem& P = a.P;
    const int64_t work = static_cast<int64_t>(P.B) * P.S * P.Hq * ((P.dv + 7) / 8);
    if (P.dtype == BPA_FP32)
        k_ring_finalize<float><<<grid_for(work, 256), 256, 0, s>>>(a);
    else
        k_ring_finalize<__nv_bfloat16><<<grid_for(work, 256), 256, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_bwd_pre(const BwdArgs& a, cudaStream_t s) {
    const Problem& P = a.P;
    const int64_t rows = static_cast<int64_t>(P.B) * P.Hq * a.Spad;
    const int zero = a.dq_acc != nullptr && !P.det;   // deterministic slices are written, not added to
    const int tpr = P.dv / 8;
    const bool vec_ok = ((reinterpret_cast<uintptr_t>(a.o) | reinterpret_cast<uintptr_t>(a.dout)) & 15u) == 0 &&
                        ((P.os[0] | P.os[1] | P.os[2]) & 7) == 0;
    if (P.dtype == BPA_BF16 && vec_ok && P.dv % 8 == 0 && tpr <= 32 && (tpr & (tpr - 1)) == 0 && rows < (1ll << 31)) {
        const int threads = 256;   // a multiple of every tpr
        const int64_t work = rows * tpr;
        k_bwd_pre_bf16v<<<grid_for(work, threads), threads, 0, s>>>(a, zero);
    } else if (P.dtype == BPA_FP32)
        k_bwd_pre<float><<<grid_for(rows * 32, 256), 256, 0, s>>>(a, zero);
    else
        k_bwd_pre<__nv_bfloat16><<<grid_for(rows * 32, 256), 256, 0, s>>>(a, zero);
    return cudaGetLastError();
}

cudaError_t launch_bwd_post(const BwdArgs& a, cudaStream_t s) {
    const Problem& P = a.P;
    const int64_t nk = static_cast<int64_t>(P.B) * P.S * P.Hkv * P.d;
    const int64_t nv = static_cast<int64_t>(P.B) * P.S * P.Hkv * P.dv;
    if (P.dtype != BPA_BF16) return cudaErrorInvalidValue;
    const bool vec_ok =
        ((reinterpret_cast<uintptr_t>(a.dq) | reinterpret_cast<uintptr_t>(a.dk) | reinterpret_cast<uintptr_t>(a.dv)) &
         15u) == 0 &&
        ((P.qs[0] | P.qs[1] | P.qs[2] | P.ks[0] | P.ks[1] | P.ks[2] | P.vs[0] | P.vs[1] | P.vs[2]) & 7) == 0;
    if (vec_ok && P.d % 32 == 0 && P.dv % 8 == 0 && static_cast<int64_t>(P.B) * P.Hq * ((P.S + 3) / 4) < (1ll << 31)) {
        const int64_t dq_threads = static_cast<int64_t>(P.B) * P.Hq * ((P.S + 3) / 4) * 32;   // a warp per 4 rows
        k_cast_dq4_bf16<<<grid_for(dq_threads, 256), 256, 0, s>>>(
            a.dq_acc, static_cast<__nv_bfloat16*>(a.dq), P.B, P.S, P.Hq, P.d, P.qs[0], P.qs[1], P.qs[2], a.Spad);
        if (a.dk_acc) {
            k_cast_out_bf16v<<<grid_for(nk / 8, 256), 256, 0, s>>>(
                a.dk_acc, static_cast<__nv_bfloat16*>(a.dk), P.B, P.S, P.Hkv, P.d, P.ks[0], P.ks[1], P.ks[2]);
            k_cast_out_bf16v<<<grid_for(nv / 8, 256), 256, 0, s>>>(
                a.dv_acc, static_cast<__nv_bfloat16*>(a.dv), P.B, P.S, P.Hkv, P.dv, P.vs[0], P.vs[1], P.vs[2]);
        }
        return cudaGetLastError();
    }
    return cudaErrorInvalidValue;   // the tensor-core backward always meets the vector conditions
}

cudaError_t launch_cast_dkdv(const BwdArgs& a, cudaStream_t s) {
    const Problem& P = a.P;
    const int64_t nk = static_cast<int64_t>(P.B) * P.S * P.Hkv * P.d;
    const int64_t nv = static_cast<int64_t>(P.B) * P.S * P.Hkv * P.dv;
    const bool vec_ok = P.dtype == BPA_BF16 && P.d % 8 == 0 && P.dv % 8 == 0 &&
                        ((reinterpret_cast<uintptr_t>(a.dk) | reinterpret_cast<uintptr_t>(a.dv)) & 15u) == 0 &&
                        ((P.ks[0] | P.ks[1] | P.ks[2] | P.vs[0] | P.vs[1] | P.vs[2]) & 7) == 0;
    if (!vec_ok) return cudaErrorInvalidValue;
    k_cast_out_bf16v<<<grid_for(nk / 8, 256), 256, 0, s>>>(a.dk_acc, static_cast<__nv_bfloat16*>(a.dk), P.B, P.S,
                                                           P.Hkv, P.d, P.ks[0], P.ks[1], P.ks[2]);
    k_cast_out_bf16v<<<grid_for(nv / 8, 256), 256, 0, s>>>(a.dv_acc, static_cast<__nv_bfloat16*>(a.dv), P.B, P.S,
                                                           P.Hkv, P.dv, P.vs[0], P.vs[1], P.vs[2]);
    return cudaGetLastError();
}

// Gradient of the sink logits: dsink[h] = -sum over (b, row) of P_sink <dO, O> with
// P_sink = exp(sink[h] - LSE); padding rows (LSE = +inf) add nothing.  One CTA per q head,
// rows in a fixed order and a fixed reduction tree: the result does not depend on timing.
__global__ void __launch_bounds__(256) k_sink_grad(const BwdArgs a) {
    const Problem& P = a.P;
    const int h = blockIdx.x;
    const float sk = P.sink[h];
    float acc = 0.f;
    for (int b = 0; b < P.B; ++b) {
        const int64_t base = (static_cast<int64_t>(b) * P.Hq + h) * a.Spad;
        for (int r = threadIdx.x; r < a.Spad; r += blockDim.x) {
            const float lse = a.lse[base + r];
            if (lse != INFINITY) acc -= expf(sk - lse) * a.Dvec[base + r];
        }
    }
    __shared__ float red[256];
    red[threadIdx.x] = acc;
    __syncthreads();
    for (int o = 128; o > 0; o >>= 1) {
        if (threadIdx.x < o) red[threadIdx.x] += red[threadIdx.x + o];
        __syncthreads();
    }
    if (threadIdx.x == 0) P.dsink[h] = red[0];
}

// m = -inf, l = 0 on the padding rows (q >= Lq) of a variable-length problem.
__global__ void k_pad_stats(const FwdArgs a) {
    const Problem& P = a.P;
    const int64_t rows = static_cast<int64_t>(P.B) * P.Hq * P.S;
    for (int64_t r = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; r < rows;
         r += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int q = static_cast<int>(r % P.S);
        const int b = static_cast<int>(r / (static_cast<int64_t>(P.S) * P.Hq));
        if (q >= lens_of(P, b).lq) {
            a.m[r] = -INFINITY;
            a.l[r] = 0.f;
        }
    }
}

cudaError_t launch_pad_stats(const FwdArgs& a, cudaStream_t s) {
    const int64_t rows = static_cast<int64_t>(a.P.B) * a.P.Hq * a.P.S;
    k_pad_stats<<<grid_for(rows, 256), 256, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_sink_grad(const BwdArgs& a, cudaStream_t s) {
    k_sink_grad<<<a.P.Hq, 256, 0, s>>>(a);
    return cudaGetLastError();
}

// Block-selected mode: every entry of block_idx [B, Hq, S / sel_block, top_n] must be -1 or a
// block strictly before its query block (what bpa_select_blocks produces).  Entries outside
// that range are ignored by the attention kernels and reported here as a device-side check
// failure (the index array is only read, so a bad entry cannot make an access go astray).
__global__ void k_check_blocks(const Problem P, uint32_t* status) {
    const int nblk = P.S / P.sel_block;
    const int64_t rows = static_cast<int64_t>(P.B) * P.Hq * nblk;
    for (int64_t r = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; r < rows;
         r += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int i = static_cast<int>(r % nblk);
        const int32_t* sel = P.block_idx + r * P.top_n;
        bool bad = false;
        for (int t = 0; t < P.top_n; ++t) {
            const int32_t e = sel[t];
            bad = bad || (e != -1 && (e < 0 || e >= i));
        }
        if (bad) report(status, ST_CHECK, 0xB0);
    }
}

cudaError_t launch_check_blocks(const Problem& P, uint32_t* status, cudaStream_t s) {
    const int64_t rows = static_cast<int64_t>(P.B) * P.Hq * (P.S / P.sel_block);
    k_check_blocks<<<grid_for(rows, 256), 256, 0, s>>>(P, status);
    return cudaGetLastError();
}

cudaError_t launch_wait_selftest(uint32_t* status, uint64_t limit_ns, cudaStream_t s) {
    k_wait_selftest<<<1, 32, 0, s>>>(status, limit_ns);
    return cudaGetLastError();
}

}  // namespace bpa
