// gather.cu - block-selected attention over gathered key blocks, forward and backward
// (bf16, head dim d = 64 NW with NW in {1, 2, 4, 8}, 32-row blocks).
//
// For query q in block i the allowed keys are the local window q-W+1..q
// united with the key blocks selected for block i ("AnnAttention",
// faiss_block_attention.py: sliding window plus the blocks select_block
// returns; read as a set union, each key once).  One warp owns one 32-row
// query block: it builds the sorted list of distinct key blocks it must
// visit (the selected ones and those the local window touches), then folds
// them one at a time into a running (max, numerator, denominator) carry in
// registers ("bpt.py", _blockwise_attention_fwd / scan_kv_block).
// The products are small (32 x 32 x 64 per block and warp), gathered from
// scattered blocks, so they run on mma.sync m16n8k16 from registers: Q stays
// in A fragments, K and V blocks are staged in XOR-swizzled shared memory and
// read with ldmatrix.  The kernels are bound by L2 / HBM traffic of the
// gathered blocks, not by the tensor cores.
// Head dims above 64 (the joint view of "AnnAttention", which flattens the heads
// into one embedding of H d channels) split the channels over NW warps per query
// block: each warp keeps its 64-channel slice of Q, K, V, O (and of dO, dQ, dK, dV),
// and only the 32 x 32 partial sums of S (and dP) are exchanged through shared
// memory, added in a fixed order so that every warp holds the same bits.
#include <math.h>

#include "bpa_internal.h"
#include "common.cuh"

namespace bpa {
namespace {

constexpr int BS = 32;        // block size (query rows and keys)
constexpr int D = 64;         // channels per warp (one slice of the head dim)
constexpr int kMaxList = 24;  // key blocks per query block (top_n + window blocks)

// 128-byte aligned so that every warp's tiles start on a 16-byte boundary
// (16-byte shared stores and ldmatrix row addresses)
struct __align__(128) WarpSmem {
    __nv_bfloat16 k[BS * D];    // 4 KB, rows of 128 B, 16-byte chunks XOR-swizzled by row
    __nv_bfloat16 v[BS * D];
    int list[kMaxList];
    int n;
};

__device__ __forceinline__ uint32_t swz(int row, int chunk) {   // byte offset in a [32][128 B] tile
    return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D (16x8 f32) += A (16x16 bf16) * B (16x8 bf16)
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// CTA geometry for NW warps per query block.  Shared memory (dynamic): the warps' own
// tiles, then one float exchange buffer [NW][32 fragments][32 lanes] per query block
// (two in the backward, for S and dP) when NW > 1.
template <int NW>
struct Geom {
    static constexpr int QB_F = NW >= 4 ? 1 : 4 / NW;   // query blocks per CTA, forward
    static constexpr int QB_B = NW >= 2 ? 1 : 2;        // backward
    static constexpr int XCH = NW > 1 ? NW * 32 * 32 : 0;   // floats of one exchange buffer
};

// Barrier over the NW warps of one query block (named barrier slot + 1; 0 is __syncthreads).
template <int NW>
__device__ __forceinline__ void group_sync(int slot) {
    if (NW == 1)
        __syncwarp();
    else
        asm volatile("bar.sync %0, %1;" ::"r"(slot + 1), "r"(NW * 32) : "memory");
}

__device__ __forceinline__ void put_partial(float* xch_w, const float (&x)[2][4][4], int lane) {
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) xch_w[((mt * 4 + nt) * 4 + e) * 32 + lane] = x[mt][nt][e];
}

template <int NW>
__device__ __forceinline__ void sum_partials(float (&x)[2][4][4], const float* xch, int lane) {
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int j = ((mt * 4 + nt) * 4 + e) * 32 + lane;
                float v = 0.f;
#pragma unroll
                for (int w = 0; w < NW; ++w) v += xch[w * 1024 + j];
                x[mt][nt][e] = v;
            }
}

// mma.sync m16n8k16 fragment layouts (g = lane / 4, t = lane % 4):
//   A 16x16 row-major:  a0 (row g, k 2t..2t+1), a1 (row g+8, k 2t..), a2 (row g, k 2t+8..), a3 (row g+8, k 2t+8..)
//   B 16x8:             b0 (k 2t..2t+1, col g), b1 (k 2t+8..2t+9, col g)
//   C 16x8 float:       c0, c1 (row g, cols 2t, 2t+1), c2, c3 (row g+8, cols 2t, 2t+1)
// ldmatrix gives lane i row i/4, elements 2(i%4), 2(i%4)+1 of each 8x8 matrix (.trans: the
// transpose), so row-major tiles load as A or K-major B fragments and column-major ones
// with .trans.

// The distinct key blocks query block i visits, ascending: the blocks its local window
// touches and its selected blocks (selected entries outside [0, i) are ignored; a separate
// check reports them).  Run by one lane.
__device__ int visit_list(const Problem& P, int64_t unit, int i, int* list) {
    int n = 0;
    const int32_t* sel = P.block_idx + unit * P.top_n;
    const int wfirst = max(0, (BS * i - (P.local_window - 1))) / BS;
    auto add = [&](int kb) {
        if (kb < 0 || kb > i) return;
        for (int x = 0; x < n; ++x)
            if (list[x] == kb) return;
        if (n < kMaxList) list[n++] = kb;
    };
    if (P.local_window > 0)
        for (int kb = wfirst; kb <= i; ++kb) add(kb);
    for (int x = 0; x < P.top_n; ++x)
        if (sel[x] < i) add(sel[x]);
    for (int x = 1; x < n; ++x) {   // ascending
        const int key = list[x];
        int y = x - 1;
        while (y >= 0 && list[y] > key) {
            list[y + 1] = list[y];
            --y;
        }
        list[y + 1] = key;
    }
    return n;
}

// DROP: the attention-dropout instantiation (dropped entries leave the softmax)
template <int NW, bool DROP>
__global__ void __launch_bounds__(Geom<NW>::QB_F * NW * 32, NW == 1 ? 3 : 1) k_gather_fwd(const FwdArgs a) {
    using G = Geom<NW>;
    const Problem& P = a.P;
    extern __shared__ __align__(128) uint8_t gsm[];
    static_assert(sizeof(WarpSmem) % 128 == 0, "per-warp tiles must stay 16-byte aligned");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slot = warp / NW, c0 = D * (warp % NW);   // query block of the CTA, channel slice
    const int g = lane >> 2, t = lane & 3;
    const int nblk = P.S / BS;
    const int64_t unit = static_cast<int64_t>(blockIdx.x) * G::QB_F + slot;   // (b, h, i)
    if (unit >= static_cast<int64_t>(P.B) * P.Hq * nblk) return;   // the whole query block's warps
    const int i = static_cast<int>(unit % nblk);
    const int h = static_cast<int>((unit / nblk) % P.Hq);
    const int b = static_cast<int>(unit / (static_cast<int64_t>(nblk) * P.Hq));
    const int hkv = h / P.G;
    WarpSmem& S = reinterpret_cast<WarpSmem*>(gsm)[warp];
    float* xch = reinterpret_cast<float*>(gsm + sizeof(WarpSmem) * G::QB_F * NW) + slot * G::XCH;
    const uint32_t sk = smem_u32(S.k), sv = smem_u32(S.v);

    // ---- key blocks to visit: selected blocks and the blocks the local window touches
    if (lane == 0) S.n = visit_list(P, unit, i, S.list);
    __syncwarp();
    const int nlist = S.n;

    // ---- Q fragments (A operand): rows mt*16 + {g, g+8}, channels ks*16 + {2t, 2t+1, 2t+8, 2t+9}
    const __nv_bfloat16* Q = static_cast<const __nv_bfloat16*>(P.q) + b * P.qs[0] + h * P.qs[2] + c0;
    uint32_t qa[2][4][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            const int r0 = BS * i + mt * 16 + g, cc = ks * 16 + 2 * t;
            const __nv_bfloat16* p0 = Q + static_cast<int64_t>(r0) * P.qs[1];
            const __nv_bfloat16* p1 = Q + static_cast<int64_t>(r0 + 8) * P.qs[1];
            qa[mt][ks][0] = *reinterpret_cast<const uint32_t*>(p0 + cc);
            qa[mt][ks][1] = *reinterpret_cast<const uint32_t*>(p1 + cc);
            qa[mt][ks][2] = *reinterpret_cast<const uint32_t*>(p0 + cc + 8);
            qa[mt][ks][3] = *reinterpret_cast<const uint32_t*>(p1 + cc + 8);
        }

    const float sl2 = P.scale * kLog2e;
    float o[2][8][4];    // [m tile][d n-tile][frag]
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[mt][nt][e] = 0.f;
    float mrow[2][2], lrow[2][2];   // [m tile][row g / g+8]
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            mrow[mt][hh] = -INFINITY;
            lrow[mt][hh] = 0.f;
        }

    const __nv_bfloat16* K = static_cast<const __nv_bfloat16*>(P.k) + b * P.ks[0] + hkv * P.ks[2] + c0;
    const __nv_bfloat16* V = static_cast<const __nv_bfloat16*>(P.v) + b * P.vs[0] + hkv * P.vs[2] + c0;
    const int32_t* selrow = P.block_idx + static_cast<int64_t>(unit) * P.top_n;

    for (int x = 0; x < nlist; ++x) {
        const int kb = S.list[x];
        bool selected = false;
        for (int y = 0; y < P.top_n; ++y) selected |= selrow[y] == kb;
        // a selected block wholly before query block i with no window bounds: no key is masked
        const bool full = !DROP && selected && kb < i && P.wl < 0 && P.wr < 0;
        // stage K and V of the block: 32 rows x 8 chunks of 16 B each, 8 chunks per lane
        __syncwarp();
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int idx = u * 32 + lane, row = idx >> 3, chunk = idx & 7;
            const int64_t key = static_cast<int64_t>(BS) * kb + row;
            const uint4 kv = *reinterpret_cast<const uint4*>(K + key * P.ks[1] + chunk * 8);
            const uint4 vv = *reinterpret_cast<const uint4*>(V + key * P.vs[1] + chunk * 8);
            st_shared_v4(sk + swz(row, chunk), kv.x, kv.y, kv.z, kv.w);
            st_shared_v4(sv + swz(row, chunk), vv.x, vv.y, vv.z, vv.w);
        }
        __syncwarp();

        // ---- S = Q K^T (32 x 32): B fragments of K^T straight from K's rows (ldmatrix, no transpose)
        float s[2][4][4];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) s[mt][nt][e] = 0.f;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
            for (int np = 0; np < 2; ++np) {   // two key n-tiles per ldmatrix.x4
                // matrices: (keys np*16 + 0..7, ch ks*16 + 0..7), (same keys, ch +8), (keys +8, ch), (keys +8, ch +8)
                const int mi = lane >> 3, rr = lane & 7;
                const int row = np * 16 + (mi >> 1) * 8 + rr, chunk = ks * 2 + (mi & 1);
                uint32_t b00, b01, b10, b11;
                ldsm_x4(sk + swz(row, chunk), b00, b01, b10, b11);
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    mma16816(s[mt][np * 2 + 0], qa[mt][ks], b00, b01);
                    mma16816(s[mt][np * 2 + 1], qa[mt][ks], b10, b11);
                }
            }
        }
        if (NW > 1) {   // S over all channels: add the slices' partial sums
            put_partial(xch + (warp % NW) * 1024, s, lane);
            group_sync<NW>(slot);
            sum_partials<NW>(s, xch, lane);
            group_sync<NW>(slot);
        }
        // ---- scale, mask, online softmax
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int q = BS * i + mt * 16 + g + hh * 8;
                float mx = -INFINITY;
                if (full) {   // a selected block wholly before the query block: every key allowed
#pragma unroll
                    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const float v = s[mt][nt][hh * 2 + e] * sl2;
                            s[mt][nt][hh * 2 + e] = v;
                            mx = fmaxf(mx, v);
                        }
                } else {
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    uint32_t dw[2] = {0u, 0u};   // draws of keys (e = 0, 1), dropout only
                    if constexpr (DROP) {
                        const uint4 w = dropout_draws(P.drop_k0, P.drop_k1, b, h, q, (BS * kb + nt * 8 + 2 * t) >> 2);
                        dw[0] = (t & 1) ? w.z : w.x;
                        dw[1] = (t & 1) ? w.w : w.y;
                    }
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int k = BS * kb + nt * 8 + 2 * t + e;
                        const bool ok = k <= q && (selected || k > q - P.local_window) &&
                                        (!P.causal || k <= q) && (P.wl < 0 || k >= q - P.wl) &&
                                        (P.wr < 0 || k <= q + P.wr) && (!DROP || dw[e] >= P.drop_thr);
                        float v = s[mt][nt][hh * 2 + e] * sl2;
                        v = ok ? v : -INFINITY;
                        s[mt][nt][hh * 2 + e] = v;
                        mx = fmaxf(mx, v);
                    }
                }
                }
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                const float mnew = fmaxf(mrow[mt][hh], mx);
                const float mref = mnew == -INFINITY ? 0.f : mnew;
                const float corr = mrow[mt][hh] == -INFINITY ? 0.f : ex2(mrow[mt][hh] - mref);
                float rs = 0.f;
#pragma unroll
                for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float p = ex2(s[mt][nt][hh * 2 + e] - mref);
                        s[mt][nt][hh * 2 + e] = p;
                        rs += p;
                    }
                rs += __shfl_xor_sync(0xffffffffu, rs, 1);
                rs += __shfl_xor_sync(0xffffffffu, rs, 2);
                lrow[mt][hh] = lrow[mt][hh] * corr + rs;
                mrow[mt][hh] = mnew;
#pragma unroll
                for (int nt = 0; nt < 8; ++nt) {
                    o[mt][nt][hh * 2 + 0] *= corr;
                    o[mt][nt][hh * 2 + 1] *= corr;
                }
            }
        // ---- O += P V: P from the S fragments (C layout -> A layout), V^T fragments by ldmatrix.trans
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {       // 16 keys per k step
            uint32_t pa[2][4];
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                pa[mt][0] = pack_bf16(s[mt][2 * kk][0], s[mt][2 * kk][1]);
                pa[mt][1] = pack_bf16(s[mt][2 * kk][2], s[mt][2 * kk][3]);
                pa[mt][2] = pack_bf16(s[mt][2 * kk + 1][0], s[mt][2 * kk + 1][1]);
                pa[mt][3] = pack_bf16(s[mt][2 * kk + 1][2], s[mt][2 * kk + 1][3]);
            }
#pragma unroll
            for (int np = 0; np < 4; ++np) {   // two d n-tiles per ldmatrix.x4.trans
                // matrices: (keys kk*16 + 0..7, ch np*16 + 0..7), (keys +8, same ch), (keys, ch +8), (keys +8, ch +8)
                const int mi = lane >> 3, rr = lane & 7;
                const int row = kk * 16 + (mi & 1) * 8 + rr, chunk = np * 2 + (mi >> 1);
                uint32_t b00, b01, b10, b11;
                ldsm_x4_t(sv + swz(row, chunk), b00, b01, b10, b11);
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    mma16816(o[mt][np * 2 + 0], pa[mt], b00, b01);
                    mma16816(o[mt][np * 2 + 1], pa[mt], b10, b11);
                }
            }
        }
    }

    // ---- epilogue: O = num / den, m, l
    __nv_bfloat16* O = static_cast<__nv_bfloat16*>(a.o) + b * P.os[0] + h * P.os[2] + c0;
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int q = BS * i + mt * 16 + g + hh * 8;
            float scale_o = 1.f;
            if (P.sink) {   // sink logit: joins the max and the denominator, contributes no value
                const float s2 = __ldg(P.sink + h) * kLog2e, mn = fmaxf(mrow[mt][hh], s2);
                scale_o = mrow[mt][hh] == -INFINITY ? 0.f : ex2(mrow[mt][hh] - mn);
                lrow[mt][hh] = lrow[mt][hh] * scale_o + ex2(s2 - mn);
                mrow[mt][hh] = mn;
            }
            const float inv = lrow[mt][hh] > 0.f ? scale_o / lrow[mt][hh] : 0.f;
            __nv_bfloat16* orow = O + static_cast<int64_t>(q) * P.os[1];
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
                *reinterpret_cast<uint32_t*>(orow + nt * 8 + 2 * t) =
                    pack_bf16(o[mt][nt][hh * 2 + 0] * inv, o[mt][nt][hh * 2 + 1] * inv);
            if (t == 0 && c0 == 0) {
                const int64_t mi = (static_cast<int64_t>(b) * P.Hq + h) * P.S + q;
                a.m[mi] = mrow[mt][hh] == -INFINITY ? -INFINITY : mrow[mt][hh] * kLn2;
                a.l[mi] = lrow[mt][hh];
            }
        }
}


// ---- backward -------------------------------------------------------------------------
// Same unit of work and visiting order as the forward.  Per key block kb of the list:
//   S = Q K^T, P = exp(s S - LSE) under the forward's mask, dP = dO V^T, dS = P (dP - D),
//   dQ += dS K                       (registers; written once, scaled, at the end),
//   dV[kb] += P^T dO, dK[kb] += s dS^T Q   (float32 accumulators, vector reductions: a key
//                                          block is shared by every query block that
//                                          selected it and by its local windows).
// "AnnAttention", faiss_block_attention.py trains through the gathered attention with the
// selection held fixed; the gradients are those of "bpt.py", _blockwise_attention_bwd
// restricted to the visited blocks.
struct __align__(128) WarpSmemB {
    __nv_bfloat16 k[BS * D];      // [key][ch], 128-byte rows, swz()
    __nv_bfloat16 v[BS * D];
    __nv_bfloat16 q[BS * D];      // [query][ch] of the warp's query block
    __nv_bfloat16 dout[BS * D];
    __nv_bfloat16 p[BS * BS];     // P and dS of the current key block: [query][key], 64-byte rows, swz32()
    __nv_bfloat16 ds[BS * BS];
    int list[kMaxList];
    int n;
};

__device__ __forceinline__ uint32_t swz32(int row, int chunk) {   // byte offset in a [32][64 B] tile
    return static_cast<uint32_t>(row * 64 + ((chunk ^ ((row >> 1) & 3)) << 4));
}

// Copies 32 rows x 64 bf16 channels (row stride rs elements) into a swizzled tile.
__device__ __forceinline__ void stage_rows(uint32_t dst, const __nv_bfloat16* src, int64_t rs, int lane) {
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const int idx = u * 32 + lane, row = idx >> 3, chunk = idx & 7;
        const uint4 x = *reinterpret_cast<const uint4*>(src + row * rs + chunk * 8);
        st_shared_v4(dst + swz(row, chunk), x.x, x.y, x.z, x.w);
    }
}

// acc (32 rows x 64 channels, C fragments) = X^T Y, X a swizzled [query][row] 32 x 32 tile,
// Y a swizzled [query][ch] 32 x 64 tile: rows of the result are X's columns (keys).
__device__ __forceinline__ void tn_product(float (&acc)[2][8][4], uint32_t x, uint32_t y, int lane) {
    const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[mt][nt][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {   // 16 queries per k step
        uint32_t xa[2][4];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
            // A = X^T (keys x queries) from [query][key] storage by .trans:
            // matrix mi holds keys mt*16 + (mi & 1) * 8 + 0..7, queries kk*16 + (mi >> 1) * 8 + 0..7
            const int row = kk * 16 + (mi >> 1) * 8 + rr, chunk = mt * 2 + (mi & 1);
            ldsm_x4_t(x + swz32(row, chunk), xa[mt][0], xa[mt][1], xa[mt][2], xa[mt][3]);
        }
#pragma unroll
        for (int np = 0; np < 4; ++np) {
            // B = Y (queries x channels) from [query][ch] storage by .trans, two channel n-tiles
            const int row = kk * 16 + (mi & 1) * 8 + rr, chunk = np * 2 + (mi >> 1);
            uint32_t b00, b01, b10, b11;
            ldsm_x4_t(y + swz(row, chunk), b00, b01, b10, b11);
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                mma16816(acc[mt][np * 2 + 0], xa[mt], b00, b01);
                mma16816(acc[mt][np * 2 + 1], xa[mt], b10, b11);
            }
        }
    }
}

// S (32 x 32, C fragments) = A B^T with A a swizzled [row][ch] 32 x 64 tile (queries) and B
// one of the same shape (keys): A fragments by ldmatrix, B fragments straight from B's rows.
__device__ __forceinline__ void nt_product(float (&s)[2][4][4], uint32_t a, uint32_t b, int lane) {
    const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) s[mt][nt][e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
        uint32_t fa[2][4];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
            // matrix mi: rows mt*16 + (mi & 1) * 8 + 0..7, channels ks*16 + (mi >> 1) * 8 + 0..7
            const int row = mt * 16 + (mi & 1) * 8 + rr, chunk = ks * 2 + (mi >> 1);
            ldsm_x4(a + swz(row, chunk), fa[mt][0], fa[mt][1], fa[mt][2], fa[mt][3]);
        }
#pragma unroll
        for (int np = 0; np < 2; ++np) {
            const int row = np * 16 + (mi >> 1) * 8 + rr, chunk = ks * 2 + (mi & 1);
            uint32_t b00, b01, b10, b11;
            ldsm_x4(b + swz(row, chunk), b00, b01, b10, b11);
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                mma16816(s[mt][np * 2 + 0], fa[mt], b00, b01);
                mma16816(s[mt][np * 2 + 1], fa[mt], b10, b11);
            }
        }
    }
}

// Writes a 32 x 32 C-fragment tile as bf16 into a swizzled [query][key] tile.
__device__ __forceinline__ void store_tile32(uint32_t dst, const float (&s)[2][4][4], int lane) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int row = mt * 16 + g + hh * 8;
                st_shared_u32(dst + swz32(row, nt) + 4 * t, pack_bf16(s[mt][nt][hh * 2], s[mt][nt][hh * 2 + 1]));
            }
}

// Adds a 32 x 64 C-fragment tile (times mul) to rows key0.. of a float32 [B, S, Hkv, 64] accumulator.
__device__ __forceinline__ void reduce_rows(float* acc_row0, int64_t row_stride, const float (&x)[2][8][4], float mul,
                                            int lane) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            float* row = acc_row0 + (mt * 16 + g + hh * 8) * row_stride + 2 * t;
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) red_add_v2(row + nt * 8, x[mt][nt][hh * 2] * mul, x[mt][nt][hh * 2 + 1] * mul);
        }
}

template <int NW, bool DROP>
__global__ void __launch_bounds__(Geom<NW>::QB_B * NW * 32) k_gather_bwd(const BwdArgs a) {
    using G = Geom<NW>;
    const Problem& P = a.P;
    extern __shared__ __align__(128) uint8_t gsm[];
    static_assert(sizeof(WarpSmemB) % 128 == 0, "per-warp tiles must stay 16-byte aligned");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slot = warp / NW, c0 = D * (warp % NW);   // query block of the CTA, channel slice
    const int g = lane >> 2, t = lane & 3, mi = lane >> 3, rr = lane & 7;
    const int nblk = P.S / BS;
    const int64_t unit = static_cast<int64_t>(blockIdx.x) * G::QB_B + slot;   // (b, h, i)
    if (unit >= static_cast<int64_t>(P.B) * P.Hq * nblk) return;   // the whole query block's warps
    const int i = static_cast<int>(unit % nblk);
    const int h = static_cast<int>((unit / nblk) % P.Hq);
    const int b = static_cast<int>(unit / (static_cast<int64_t>(nblk) * P.Hq));
    const int hkv = h / P.G;
    WarpSmemB& W = reinterpret_cast<WarpSmemB*>(gsm)[warp];
    float* xch = reinterpret_cast<float*>(gsm + sizeof(WarpSmemB) * G::QB_B * NW) + slot * 2 * G::XCH;
    const uint32_t sk = smem_u32(W.k), sv = smem_u32(W.v), sq = smem_u32(W.q), sdo = smem_u32(W.dout),
                   sp = smem_u32(W.p), sds = smem_u32(W.ds);

    if (lane == 0) W.n = visit_list(P, unit, i, W.list);
    const __nv_bfloat16* Q = static_cast<const __nv_bfloat16*>(P.q) + b * P.qs[0] + h * P.qs[2] + c0;
    const __nv_bfloat16* dO = static_cast<const __nv_bfloat16*>(a.dout) + b * P.os[0] + h * P.os[2] + c0;
    stage_rows(sq, Q + static_cast<int64_t>(BS) * i * P.qs[1], P.qs[1], lane);
    stage_rows(sdo, dO + static_cast<int64_t>(BS) * i * P.os[1], P.os[1], lane);
    __syncwarp();
    const int nlist = W.n;

    // per-row statistics: rows mt*16 + g + hh*8 of the block
    float lse2[2][2], Drow[2][2];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int64_t r = (static_cast<int64_t>(b) * P.Hq + h) * a.Spad + BS * i + mt * 16 + g + hh * 8;
            lse2[mt][hh] = a.lse[r] * kLog2e;   // +inf on rows with no allowed key: P = 0
            Drow[mt][hh] = a.Dvec[r];
        }
    const float sl2 = P.scale * kLog2e;
    float dq[2][8][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) dq[mt][nt][e] = 0.f;

    const __nv_bfloat16* K = static_cast<const __nv_bfloat16*>(P.k) + b * P.ks[0] + hkv * P.ks[2] + c0;
    const __nv_bfloat16* V = static_cast<const __nv_bfloat16*>(P.v) + b * P.vs[0] + hkv * P.vs[2] + c0;
    const int64_t acc_rs = static_cast<int64_t>(P.Hkv) * D * NW;   // float32 accumulators [B, S, Hkv, d]
    float* dKacc = a.dk_acc + (static_cast<int64_t>(b) * P.S * P.Hkv + hkv) * (D * NW) + c0;
    float* dVacc = a.dv_acc + (static_cast<int64_t>(b) * P.S * P.Hkv + hkv) * (D * NW) + c0;
    const int32_t* selrow = P.block_idx + unit * P.top_n;

    for (int x = 0; x < nlist; ++x) {
        const int kb = W.list[x];
        bool selected = false;
        for (int y = 0; y < P.top_n; ++y) selected |= selrow[y] == kb;
        // a selected block wholly before query block i with no window bounds: no key is masked
        const bool full = !DROP && selected && kb < i && P.wl < 0 && P.wr < 0;
        __syncwarp();   // the previous block's reads of K, V and the P / dS tiles are done
        stage_rows(sk, K + static_cast<int64_t>(BS) * kb * P.ks[1], P.ks[1], lane);
        stage_rows(sv, V + static_cast<int64_t>(BS) * kb * P.vs[1], P.vs[1], lane);
        __syncwarp();

        float s[2][4][4], dp[2][4][4];
        nt_product(s, sq, sk, lane);     // Q K^T
        nt_product(dp, sdo, sv, lane);   // dO V^T
        if (NW > 1) {   // over all channels: add the slices' partial sums
            put_partial(xch + (warp % NW) * 1024, s, lane);
            put_partial(xch + G::XCH + (warp % NW) * 1024, dp, lane);
            group_sync<NW>(slot);
            sum_partials<NW>(s, xch, lane);
            sum_partials<NW>(dp, xch + G::XCH, lane);
            group_sync<NW>(slot);
        }
        // P and dS under the forward's mask
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int q = BS * i + mt * 16 + g + hh * 8;
                if (full) {   // a selected block wholly before the query block: every key allowed
#pragma unroll
                    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const float p = ex2(s[mt][nt][hh * 2 + e] * sl2 - lse2[mt][hh]);
                            s[mt][nt][hh * 2 + e] = p;
                            dp[mt][nt][hh * 2 + e] = p * (dp[mt][nt][hh * 2 + e] - Drow[mt][hh]);
                        }
                } else {
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    uint32_t dw[2] = {0u, 0u};   // draws of keys (e = 0, 1), dropout only
                    if constexpr (DROP) {
                        const uint4 w = dropout_draws(P.drop_k0, P.drop_k1, b, h, q, (BS * kb + nt * 8 + 2 * t) >> 2);
                        dw[0] = (t & 1) ? w.z : w.x;
                        dw[1] = (t & 1) ? w.w : w.y;
                    }
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int k = BS * kb + nt * 8 + 2 * t + e;
                        const bool ok = k <= q && (selected || k > q - P.local_window) &&
                                        (!P.causal || k <= q) && (P.wl < 0 || k >= q - P.wl) &&
                                        (P.wr < 0 || k <= q + P.wr) && (!DROP || dw[e] >= P.drop_thr);
                        const float p = ok ? ex2(s[mt][nt][hh * 2 + e] * sl2 - lse2[mt][hh]) : 0.f;
                        s[mt][nt][hh * 2 + e] = p;
                        dp[mt][nt][hh * 2 + e] = p * (dp[mt][nt][hh * 2 + e] - Drow[mt][hh]);
                    }
                }
                }
            }
        store_tile32(sp, s, lane);
        store_tile32(sds, dp, lane);
        __syncwarp();
        // dQ += dS K: dS fragments from its [query][key] tile, K^T fragments by ldmatrix.trans
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
            uint32_t da[2][4];
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                const int row = mt * 16 + (mi & 1) * 8 + rr, chunk = kk * 2 + (mi >> 1);
                ldsm_x4(sds + swz32(row, chunk), da[mt][0], da[mt][1], da[mt][2], da[mt][3]);
            }
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                const int row = kk * 16 + (mi & 1) * 8 + rr, chunk = np * 2 + (mi >> 1);
                uint32_t b00, b01, b10, b11;
                ldsm_x4_t(sk + swz(row, chunk), b00, b01, b10, b11);
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    mma16816(dq[mt][np * 2 + 0], da[mt], b00, b01);
                    mma16816(dq[mt][np * 2 + 1], da[mt], b10, b11);
                }
            }
        }
        float acc[2][8][4];
        // dV[kb] += P^T dO
        tn_product(acc, sp, sdo, lane);
        reduce_rows(dVacc + static_cast<int64_t>(BS) * kb * acc_rs, acc_rs, acc, 1.f, lane);
        // dK[kb] += scale dS^T Q
        tn_product(acc, sds, sq, lane);
        reduce_rows(dKacc + static_cast<int64_t>(BS) * kb * acc_rs, acc_rs, acc, P.scale, lane);
    }

    // ---- dQ = scale * sum dS K, written once
    __nv_bfloat16* dQ = static_cast<__nv_bfloat16*>(a.dq) + b * P.qs[0] + h * P.qs[2] + c0;
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            __nv_bfloat16* row = dQ + static_cast<int64_t>(BS * i + mt * 16 + g + hh * 8) * P.qs[1];
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
                *reinterpret_cast<uint32_t*>(row + nt * 8 + 2 * t) =
                    pack_bf16(dq[mt][nt][hh * 2 + 0] * P.scale, dq[mt][nt][hh * 2 + 1] * P.scale);
        }
}
}  // namespace

bool gather_supported(const Problem& P) {
    if (P.dtype != BPA_BF16 || P.d != P.dv || !P.block_idx || P.sel_block != BS) return false;
    if (P.d != 64 && P.d != 128 && P.d != 256 && P.d != 512) return false;
    if (P.top_n + 3 > kMaxList || P.local_window > 2 * BS) return false;
    if (P.ring_n != 1 || P.bias) return false;
    // 16-byte rows for the staged copies, 4-byte fragment loads
    if ((reinterpret_cast<uintptr_t>(P.q) | reinterpret_cast<uintptr_t>(P.k) | reinterpret_cast<uintptr_t>(P.v)) & 15)
        return false;
    if ((P.qs[0] | P.qs[1] | P.qs[2] | P.ks[0] | P.ks[1] | P.ks[2] | P.vs[0] | P.vs[1] | P.vs[2] | P.os[0] | P.os[1] |
         P.os[2]) & 7)
        return false;
    return true;
}

namespace {

template <int NW>
cudaError_t gather_fwd_nw(const FwdArgs& a, cudaStream_t s) {
    using G = Geom<NW>;
    const int64_t units = static_cast<int64_t>(a.P.B) * a.P.Hq * (a.P.S / BS);
    const size_t smem = sizeof(WarpSmem) * G::QB_F * NW + sizeof(float) * G::XCH * G::QB_F;
    void (*kern)(const FwdArgs) = a.P.drop_thr ? k_gather_fwd<NW, true> : k_gather_fwd<NW, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    kern<<<static_cast<unsigned>((units + G::QB_F - 1) / G::QB_F), G::QB_F * NW * 32, smem, s>>>(a);
    return cudaGetLastError();
}

template <int NW>
cudaError_t gather_bwd_nw(const BwdArgs& a, cudaStream_t s) {
    using G = Geom<NW>;
    const int64_t units = static_cast<int64_t>(a.P.B) * a.P.Hq * (a.P.S / BS);
    const size_t smem = sizeof(WarpSmemB) * G::QB_B * NW + sizeof(float) * 2 * G::XCH * G::QB_B;
    void (*kern)(const BwdArgs) = a.P.drop_thr ? k_gather_bwd<NW, true> : k_gather_bwd<NW, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    kern<<<static_cast<unsigned>((units + G::QB_B - 1) / G::QB_B), G::QB_B * NW * 32, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gather_fwd(const FwdArgs& a, cudaStream_t s) {
    switch (a.P.d) {
        case 64: return gather_fwd_nw<1>(a, s);
        case 128: return gather_fwd_nw<2>(a, s);
        case 256: return gather_fwd_nw<4>(a, s);
        case 512: return gather_fwd_nw<8>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_gather_bwd(const BwdArgs& a, cudaStream_t s) {
    switch (a.P.d) {
        case 64: return gather_bwd_nw<1>(a, s);
        case 128: return gather_bwd_nw<2>(a, s);
        case 256: return gather_bwd_nw<4>(a, s);
        case 512: return gather_bwd_nw<8>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace bpa
