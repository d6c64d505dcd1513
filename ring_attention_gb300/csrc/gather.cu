// gather.cu - block-selected attention forward over gathered key blocks (bf16, d = 64, 32-key blocks).
//
// For query q in block i the allowed keys are the local window q-W+1..q
// united with the key blocks selected for block i ("AnnAttention",
// faiss_block_attention.py: sliding window plus the blocks select_block
// returns; read as a set union, each key once).  One warp owns one 32-row
// query block: it builds the sorted list of distinct key blocks it must
// visit (the selected ones and those the local window touches), then folds
// them one at a time into a running (max, numerator, denominator) carry in
// registers ("bpt.py", _blockwise_attention_fwd / scan_kv_block).
// The products are small (32 x 32 x 64 per block), gathered from scattered
// blocks, so they run on mma.sync m16n8k16 from registers: Q stays in A
// fragments, K and V blocks are staged in XOR-swizzled shared memory and
// read with ldmatrix.  The kernel is bound by L2 / HBM traffic of the
// gathered blocks, not by the tensor cores.
#include <math.h>

#include "bpa_internal.h"
#include "common.cuh"

namespace bpa {
namespace {

constexpr int BS = 32;        // block size (query rows and keys)
constexpr int D = 64;         // head dim
constexpr int kWarps = 4;     // query blocks per CTA
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

__global__ void __launch_bounds__(kWarps * 32) k_gather_fwd(const FwdArgs a) {
    const Problem& P = a.P;
    __shared__ WarpSmem sm[kWarps];
    static_assert(sizeof(WarpSmem) % 128 == 0, "per-warp tiles must stay 16-byte aligned");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int nblk = P.S / BS;
    const int64_t unit = static_cast<int64_t>(blockIdx.x) * kWarps + warp;   // (b, h, i)
    if (unit >= static_cast<int64_t>(P.B) * P.Hq * nblk) return;
    const int i = static_cast<int>(unit % nblk);
    const int h = static_cast<int>((unit / nblk) % P.Hq);
    const int b = static_cast<int>(unit / (static_cast<int64_t>(nblk) * P.Hq));
    const int hkv = h / P.G;
    WarpSmem& S = sm[warp];
    const uint32_t sk = smem_u32(S.k), sv = smem_u32(S.v);

    // ---- key blocks to visit: selected blocks and the blocks the local window touches
    if (lane == 0) {
        int n = 0;
        const int32_t* sel = P.block_idx + (static_cast<int64_t>(unit)) * P.top_n;
        const int wfirst = max(0, (BS * i - (P.local_window - 1))) / BS;
        auto add = [&](int kb) {
            if (kb < 0 || kb > i) return;
            for (int x = 0; x < n; ++x)
                if (S.list[x] == kb) return;
            if (n < kMaxList) S.list[n++] = kb;
        };
        if (P.local_window > 0)
            for (int kb = wfirst; kb <= i; ++kb) add(kb);
        for (int x = 0; x < P.top_n; ++x) add(sel[x]);
        for (int x = 1; x < n; ++x) {   // ascending
            const int key = S.list[x];
            int y = x - 1;
            while (y >= 0 && S.list[y] > key) {
                S.list[y + 1] = S.list[y];
                --y;
            }
            S.list[y + 1] = key;
        }
        S.n = n;
    }
    __syncwarp();
    const int nlist = S.n;

    // ---- Q fragments (A operand): rows mt*16 + {g, g+8}, channels ks*16 + {2t, 2t+1, 2t+8, 2t+9}
    const __nv_bfloat16* Q = static_cast<const __nv_bfloat16*>(P.q) + b * P.qs[0] + h * P.qs[2];
    uint32_t qa[2][4][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            const int r0 = BS * i + mt * 16 + g, c0 = ks * 16 + 2 * t;
            const __nv_bfloat16* p0 = Q + static_cast<int64_t>(r0) * P.qs[1];
            const __nv_bfloat16* p1 = Q + static_cast<int64_t>(r0 + 8) * P.qs[1];
            qa[mt][ks][0] = *reinterpret_cast<const uint32_t*>(p0 + c0);
            qa[mt][ks][1] = *reinterpret_cast<const uint32_t*>(p1 + c0);
            qa[mt][ks][2] = *reinterpret_cast<const uint32_t*>(p0 + c0 + 8);
            qa[mt][ks][3] = *reinterpret_cast<const uint32_t*>(p1 + c0 + 8);
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

    const __nv_bfloat16* K = static_cast<const __nv_bfloat16*>(P.k) + b * P.ks[0] + hkv * P.ks[2];
    const __nv_bfloat16* V = static_cast<const __nv_bfloat16*>(P.v) + b * P.vs[0] + hkv * P.vs[2];
    const int32_t* selrow = P.block_idx + static_cast<int64_t>(unit) * P.top_n;

    for (int x = 0; x < nlist; ++x) {
        const int kb = S.list[x];
        bool selected = false;
        for (int y = 0; y < P.top_n; ++y) selected |= selrow[y] == kb;
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
        // ---- scale, mask, online softmax
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int q = BS * i + mt * 16 + g + hh * 8;
                float mx = -INFINITY;
#pragma unroll
                for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int k = BS * kb + nt * 8 + 2 * t + e;
                        const bool ok = k <= q && (selected || k > q - P.local_window) &&
                                        (!P.causal || k <= q) && (P.wl < 0 || k >= q - P.wl) &&
                                        (P.wr < 0 || k <= q + P.wr);
                        float v = s[mt][nt][hh * 2 + e] * sl2;
                        v = ok ? v : -INFINITY;
                        s[mt][nt][hh * 2 + e] = v;
                        mx = fmaxf(mx, v);
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
    __nv_bfloat16* O = static_cast<__nv_bfloat16*>(a.o) + b * P.os[0] + h * P.os[2];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int q = BS * i + mt * 16 + g + hh * 8;
            const float inv = lrow[mt][hh] > 0.f ? 1.f / lrow[mt][hh] : 0.f;
            __nv_bfloat16* orow = O + static_cast<int64_t>(q) * P.os[1];
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
                *reinterpret_cast<uint32_t*>(orow + nt * 8 + 2 * t) =
                    pack_bf16(o[mt][nt][hh * 2 + 0] * inv, o[mt][nt][hh * 2 + 1] * inv);
            if (t == 0) {
                const int64_t mi = (static_cast<int64_t>(b) * P.Hq + h) * P.S + q;
                a.m[mi] = mrow[mt][hh] == -INFINITY ? -INFINITY : mrow[mt][hh] * kLn2;
                a.l[mi] = lrow[mt][hh];
            }
        }
}

}  // namespace

bool gather_supported(const Problem& P) {
    if (P.dtype != BPA_BF16 || P.d != D || P.dv != D || !P.block_idx || P.sel_block != BS) return false;
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

cudaError_t launch_gather_fwd(const FwdArgs& a, cudaStream_t s) {
    const int64_t units = static_cast<int64_t>(a.P.B) * a.P.Hq * (a.P.S / BS);
    k_gather_fwd<<<static_cast<unsigned>((units + kWarps - 1) / kWarps), kWarps * 32, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace bpa
