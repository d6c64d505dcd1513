// select.cu - exact top-n block selection ("AnnAttention", faiss_block_attention.py,
// select_block, made exact: brute-force dot products of block sums).
//
// Arithmetic contract (it makes the result bit-identical to any
// implementation that performs the same IEEE operations in the same order):
//   Qs[i][c] = ((0 + x_0) + x_1) + ... + x_{bs-1}      float64, rows in order
//   score    = ((0 + a_0*b_0) + a_1*b_1) + ...         float64, channels in
//              order, every product and sum rounded separately (no FMA)
//   ranking  : larger score first, the lower block index on equal scores; a NaN
//              score below every number, NaNs in block order.
//
// GB300 runs float64 at a small fraction of its float32 rate, so the float64 scores
// are computed only where they can decide the result.  For query block i and every
// candidate j < i a float32 score s_j (block sums rounded to float32, fused
// multiply-adds) and a float32 magnitude a_j = sum_c |q_c| |k_c| come first.  With
// u = 2^-24, d channels and z_j = sum_c (|q_c| + |k_c|) (float32 values),
//   |s_j - score_j| <= e_j = 2 * 1.01 * ((d + 4) u a_j + 2^-149 z_j) + d * 2^-120
// covers the float32 rounding of the inputs (relative u, or 2^-150 absolute below the
// normal range), the float32 accumulation of s_j, a_j and z_j (one rounding per fused
// step) and the float64 rounding of the contract score, with a factor of two to spare.
// So score_j lies in [L_j, U_j] = [s_j - e_j, s_j + e_j].  If T is the n-th largest L_j,
// n blocks score at least T, and any j with U_j < T scores below all of them: it cannot be
// selected.  When exactly n candidates remain they are the selection (every other block
// scores below each of them, and the output lists the selected blocks in block order), so
// no contract score is needed; otherwise the contract scores of the candidates decide the
// ranking exactly as the definition does.  L_j and U_j are rounded outwards in float32.
// A row whose float32 values are not all finite takes the contract score of every block.
// Comparisons use integer keys that order like the scores: float64 comparisons would run
// on the slow float64 pipe, and they outnumber the arithmetic in the ranking passes.
#include <climits>

#include "bpa_internal.h"
#include "common.cuh"

namespace bpa {
namespace {

template <typename T>
__device__ __forceinline__ double ldd(const T* p);
template <>
__device__ __forceinline__ double ldd<float>(const float* p) { return static_cast<double>(*p); }
template <>
__device__ __forceinline__ double ldd<__nv_bfloat16>(const __nv_bfloat16* p) {
    return static_cast<double>(__bfloat162float(*p));
}

// A float32 or bfloat16 value as sign, significand and the exponent of its last bit
// (value = (-1)^neg * mant * 2^w), with w of a subnormal that of the smallest normal.
struct Parts {
    uint32_t mant;
    int w;
    bool neg, finite;
};
template <typename T>
__device__ __forceinline__ Parts parts(const T* p);
template <>
__device__ __forceinline__ Parts parts<float>(const float* p) {
    const uint32_t u = __float_as_uint(*p), e = (u >> 23) & 0xFFu, f = u & 0x7FFFFFu;
    return {e ? (f | 0x800000u) : f, static_cast<int>(e ? e : 1u) - 150, (u >> 31) != 0, e != 0xFFu};
}
template <>
__device__ __forceinline__ Parts parts<__nv_bfloat16>(const __nv_bfloat16* p) {
    const uint32_t u = __bfloat16_as_ushort(*p), e = (u >> 7) & 0xFFu, f = u & 0x7Fu;
    return {e ? (f | 0x80u) : f, static_cast<int>(e ? e : 1u) - 134, (u >> 15) != 0, e != 0xFFu};
}
template <typename T>
constexpr int kMantBits = sizeof(T) == 4 ? 24 : 8;

// The float64 sum ((0 + x_0) + x_1) + ... of one channel over the rows of a block, x_r at
// p + r * stride.  When every nonzero x_r is a multiple of 2^wmin and below 2^(wmax + m) in
// magnitude (m significand bits) with wmax - wmin + m + ceil(log2 rows) <= 53, every partial
// sum is a multiple of 2^wmin below 2^(53 + wmin): each float64 addition is exact and the
// sum equals the exact one, which 64-bit integer additions of the significands (scaled to
// the common last bit) give without the float64 pipe.  Other columns (a wide exponent
// range, an infinity or a NaN) take the float64 additions in row order.
template <typename T>
__device__ __forceinline__ double column_sum(const T* p, int64_t stride, int rows, int lg_rows) {
    int wmin = INT_MAX, wmax = INT_MIN;
    bool finite = true;
#pragma unroll 8
    for (int r = 0; r < rows; ++r) {
        const Parts x = parts(p + r * stride);
        finite = finite && x.finite;
        if (x.mant) {
            wmin = min(wmin, x.w);
            wmax = max(wmax, x.w);
        }
    }
    if (finite && wmin == INT_MAX) return 0.0;   // all zeros: +0, as the float64 additions give
    if (finite && wmax - wmin + kMantBits<T> + lg_rows <= 53) {
        long long acc = 0;
#pragma unroll 8
        for (int r = 0; r < rows; ++r) {
            const Parts x = parts(p + r * stride);
            if (!x.mant) continue;   // a zero (its w may lie below wmin)
            const long long m = static_cast<long long>(x.mant) << (x.w - wmin);
            acc += x.neg ? -m : m;
        }
        // |acc| < 2^53: exact as a float64, and the scaling by 2^wmin (a normal float64) too
        return __dmul_rn(__ll2double_rn(acc), __longlong_as_double(static_cast<long long>(wmin + 1023) << 52));
    }
    double s = 0.0;
#pragma unroll 8
    for (int r = 0; r < rows; ++r) s = __dadd_rn(s, ldd(p + r * stride));
    return s;
}

// grid (nblk, H, B), one thread per channel: the float64 block sums of Q and K, and the
// float32 copy of the key sums, channel-major [B, H, d, nblk] for the pre-filter
template <typename T>
__global__ void k_block_sums(const SelectArgs a) {
    const int i = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int nblk = a.S / a.block;
    const int lg_rows = a.block > 1 ? 32 - __clz(a.block - 1) : 0;
    const T* Q = static_cast<const T*>(a.q) + b * a.qs[0] + static_cast<int64_t>(i) * a.block * a.qs[1] + h * a.qs[2];
    const T* K = static_cast<const T*>(a.k) + b * a.ks[0] + static_cast<int64_t>(i) * a.block * a.ks[1] + h * a.ks[2];
    for (int c = threadIdx.x; c < a.d; c += blockDim.x) {
        const double sq = column_sum(Q + c, a.qs[1], a.block, lg_rows);
        const double sk = column_sum(K + c, a.ks[1], a.block, lg_rows);
        const int64_t bh = static_cast<int64_t>(b) * a.H + h;
        const int64_t o = (bh * nblk + i) * a.d + c;
        a.qsum[o] = sq;
        a.ksum[o] = sk;
        a.kt32[(bh * a.d + c) * nblk + i] = __double2float_rn(sk);
    }
}

// The same sums for blocks of at most 32 rows from values held in registers: each value is
// read from global memory once (both passes run on the registers), Q and K columns go to
// separate threads, and with NC = 2 a thread takes two adjacent bfloat16 channels (4-byte
// loads, so a warp reads 128 contiguous bytes of a row).
template <typename T>
__device__ __forceinline__ Parts parts_bits(uint32_t u);
template <>
__device__ __forceinline__ Parts parts_bits<float>(uint32_t u) {
    const uint32_t e = (u >> 23) & 0xFFu, f = u & 0x7FFFFFu;
    return {e ? (f | 0x800000u) : f, static_cast<int>(e ? e : 1u) - 150, (u >> 31) != 0, e != 0xFFu};
}
template <>
__device__ __forceinline__ Parts parts_bits<__nv_bfloat16>(uint32_t u) {
    const uint32_t e = (u >> 7) & 0xFFu, f = u & 0x7Fu;
    return {e ? (f | 0x80u) : f, static_cast<int>(e ? e : 1u) - 134, ((u >> 15) & 1u) != 0, e != 0xFFu};
}
template <typename T>
__device__ __forceinline__ double value_bits(uint32_t u) {
    return sizeof(T) == 4 ? static_cast<double>(__uint_as_float(u)) : static_cast<double>(__uint_as_float(u << 16));
}

template <typename T>
__device__ __forceinline__ double column_sum_regs(const uint32_t (&v)[32], int shift, int rows, int lg_rows) {
    const uint32_t msk = sizeof(T) == 4 ? 0xFFFFFFFFu : 0xFFFFu;
    int wmin = INT_MAX, wmax = INT_MIN;
    bool finite = true;
#pragma unroll
    for (int r = 0; r < 32; ++r) {
        if (r >= rows) break;
        const Parts x = parts_bits<T>((v[r] >> shift) & msk);
        finite = finite && x.finite;
        if (x.mant) {
            wmin = min(wmin, x.w);
            wmax = max(wmax, x.w);
        }
    }
    if (finite && wmin == INT_MAX) return 0.0;   // all zeros: +0, as the float64 additions give
    if (finite && wmax - wmin + kMantBits<T> + lg_rows <= 53) {
        long long acc = 0;
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            if (r >= rows) break;
            const Parts x = parts_bits<T>((v[r] >> shift) & msk);
            if (!x.mant) continue;   // a zero (its w may lie below wmin)
            const long long m = static_cast<long long>(x.mant) << (x.w - wmin);
            acc += x.neg ? -m : m;
        }
        return __dmul_rn(__ll2double_rn(acc), __longlong_as_double(static_cast<long long>(wmin + 1023) << 52));
    }
    double s = 0.0;
#pragma unroll
    for (int r = 0; r < 32; ++r) {
        if (r >= rows) break;
        s = __dadd_rn(s, value_bits<T>((v[r] >> shift) & msk));
    }
    return s;
}

// bfloat16 columns: the exponent range comes from the largest and the smallest nonzero
// magnitude (integer min / max of the low 15 bits), and where the span leaves room
// (wmax - wmin + 8 + ceil(log2 rows) <= 24, and no partial sum can reach 2^128) every float32
// addition in row order is exact too, so the sum runs on the float32 pipe; wider spans take
// the integer or float64 paths above.
__device__ __forceinline__ double column_sum_regs_bf16(const uint32_t (&v)[32], int shift, int rows, int lg_rows) {
    uint32_t mx = 0, mn = 0xFFFFFFFFu;
#pragma unroll
    for (int r = 0; r < 32; ++r) {
        if (r >= rows) break;
        const uint32_t m = (v[r] >> shift) & 0x7FFFu;
        mx = max(mx, m);
        mn = min(mn, m ? m : 0xFFFFFFFFu);
    }
    if (mx >= 0x7F80u) return column_sum_regs<__nv_bfloat16>(v, shift, rows, lg_rows);   // an infinity or a NaN
    if (mn == 0xFFFFFFFFu) return 0.0;   // all zeros: +0, as the float64 additions give
    const int wmax = static_cast<int>(max(mx >> 7, 1u)) - 134, wmin = static_cast<int>(max(mn >> 7, 1u)) - 134;
    if (wmax - wmin + 8 + lg_rows <= 24 && wmax + 8 + lg_rows <= 127) {
        float s = 0.f;
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            if (r >= rows) break;
            s = __fadd_rn(s, __uint_as_float(((v[r] >> shift) & 0xFFFFu) << 16));
        }
        return static_cast<double>(s);
    }
    return column_sum_regs<__nv_bfloat16>(v, shift, rows, lg_rows);
}

// grid (nblk, H, B); threads [0, half) take Q, [half, 2 half) take K, NC channels each
template <typename T, int NC>
__global__ void k_block_sums_reg(const SelectArgs a, int half) {
    const int i = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int nblk = a.S / a.block;
    const int lg_rows = a.block > 1 ? 32 - __clz(a.block - 1) : 0;
    const bool isk = threadIdx.x >= half;
    const int c0 = (isk ? threadIdx.x - half : threadIdx.x) * NC;
    if (c0 >= a.d) return;
    const T* base = isk ? static_cast<const T*>(a.k) + b * a.ks[0] + static_cast<int64_t>(i) * a.block * a.ks[1] + h * a.ks[2]
                        : static_cast<const T*>(a.q) + b * a.qs[0] + static_cast<int64_t>(i) * a.block * a.qs[1] + h * a.qs[2];
    const int64_t stride = isk ? a.ks[1] : a.qs[1];
    uint32_t v[32];
#pragma unroll
    for (int r = 0; r < 32; ++r) {
        if (r >= a.block) break;
        const T* p = base + r * stride + c0;
        if (NC == 2)
            v[r] = *reinterpret_cast<const uint32_t*>(p);
        else if (sizeof(T) == 4)
            v[r] = __float_as_uint(*reinterpret_cast<const float*>(p));
        else
            v[r] = __bfloat16_as_ushort(*reinterpret_cast<const __nv_bfloat16*>(p));
    }
    const int64_t bh = static_cast<int64_t>(b) * a.H + h;
#pragma unroll
    for (int k = 0; k < NC; ++k) {
        const int c = c0 + k;
        const double s = sizeof(T) == 2 ? column_sum_regs_bf16(v, 16 * k, a.block, lg_rows)
                                         : column_sum_regs<T>(v, 16 * k, a.block, lg_rows);
        const int64_t o = (bh * nblk + i) * a.d + c;
        if (isk) {
            a.ksum[o] = s;
            a.kt32[(bh * a.d + c) * nblk + i] = __double2float_rn(s);
        } else {
            a.qsum[o] = s;
        }
    }
}

// The ranking, in integers (float64 comparisons run on GB300's slow float64 pipe):
// a score maps to a signed 64-bit key that orders like the score, with both zeros equal
// and a NaN below every number; equal keys go to the lower block.
__device__ __forceinline__ long long rank_key(double s) {
    const long long bits = __double_as_longlong(s);
    const long long mag = bits & 0x7FFFFFFFFFFFFFFFll;
    if (mag > 0x7FF0000000000000ll) return LLONG_MIN;   // NaN
    if (mag == 0) return 0;                              // +0 and -0
    return bits >= 0 ? bits : (bits ^ 0x7FFFFFFFFFFFFFFFll);
}

// A finite float32 as a signed 32-bit key in the same order (for the pre-filter threshold).
__device__ __forceinline__ int f32_key(float f) {
    const int bits = __float_as_int(f);
    return bits >= 0 ? bits : (bits ^ 0x7FFFFFFF);
}

// The contract score of query block sums qs and key block sums ks.
// (Unrolled so that several loads are in flight; the additions stay in channel order.)
__device__ __forceinline__ double contract_dot(const double* qs, const double* ks, int d) {
    double acc = 0.0;
#pragma unroll 8
    for (int c = 0; c < d; ++c) acc = __dadd_rn(acc, __dmul_rn(qs[c], ks[c]));
    return acc;
}

// Warps per CTA (at most; fewer where the per-warp arrays of long rows need the space) and
// the tile of float32 key sums (channels x blocks) staged in shared memory: the CTA's warps
// take consecutive query blocks of one (batch, head) and read the staged tile.
constexpr int kSelMaxWarps = 8, kStageC = 64, kStageJ = 256;
// Head dims up to this take the float32 pre-filter (every head dim the selection accepts);
// wider ones would score every block in float64.
constexpr int kPrefilterMaxD = 512;

// The untaken entry with the largest key (the lower index on equal keys); every lane gets it.
template <typename K>
__device__ __forceinline__ int warp_best(const K* key, const unsigned char* taken, int n, int lane, K& best) {
    K bk = 0;
    int bj = -1;
    for (int j = lane; j < n; j += 32) {
        if (taken[j]) continue;
        const K k = key[j];
        if (bj < 0 || k > bk) {   // ascending j per lane: a later equal key never wins
            bk = k;
            bj = j;
        }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        const K ok = __shfl_xor_sync(0xffffffffu, bk, o);
        const int oj = __shfl_xor_sync(0xffffffffu, bj, o);
        if (oj >= 0 && (bj < 0 || ok > bk || (ok == bk && oj < bj))) {
            bk = ok;
            bj = oj;
        }
    }
    best = bk;
    return bj;
}

// One warp per (b, h, query block i); a CTA of nw warps takes query blocks nw y .. nw y + nw - 1
// of one (b, h) = blockIdx.x.  Shared memory per warp: keys[nblk] 64-bit words (the 32-bit keys
// of the lower bounds L_j, then the 64-bit rank keys of the candidates' contract scores),
// up[nblk] floats (the upper bounds U_j), taken[nblk] bytes, and the query block's float32 sums
// q32[d]; per CTA the staged tile of float32 key sums.
__global__ void __launch_bounds__(kSelMaxWarps * 32) k_select(const SelectArgs a) {
    extern __shared__ long long sm_all[];
    const int nblk = a.S / a.block;
    const int nw = blockDim.x >> 5;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    long long* key64 = sm_all + static_cast<int64_t>(warp) * nblk;
    int* key32 = reinterpret_cast<int*>(key64);
    float* up_all = reinterpret_cast<float*>(sm_all + static_cast<int64_t>(nw) * nblk);
    float* up = up_all + static_cast<int64_t>(warp) * nblk;
    float* q32_all = up_all + static_cast<int64_t>(nw) * nblk;
    float* q32 = q32_all + static_cast<int64_t>(warp) * a.d;
    unsigned char* taken_all = reinterpret_cast<unsigned char*>(q32_all + static_cast<int64_t>(nw) * a.d);
    unsigned char* taken = taken_all + static_cast<int64_t>(warp) * nblk;
    float* kts = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(taken_all + static_cast<int64_t>(nw) * nblk) + 15) &
                                          ~static_cast<uintptr_t>(15));
    const int64_t bh = blockIdx.x;
    const int i = blockIdx.y * nw + warp;
    const bool active = i < nblk;
    const double* qs = a.qsum + (bh * nblk + (active ? i : 0)) * a.d;
    const int take = !active ? 0 : (i < a.top_n ? i : a.top_n);
    int picks[64];
    // ---- float32 pre-filter: L_j and U_j for every earlier block, rounded outwards
    if (take > 0)
        for (int c = lane; c < a.d; c += 32) q32[c] = __double2float_rn(qs[c]);
    const float* kt = a.kt32 + bh * a.d * static_cast<int64_t>(nblk);
    const float cb = 2.0f * 1.01f * static_cast<float>(a.d + 4) * 5.9604645e-8f * 1.0001f;   // >= 2 * 1.01 * (d + 4) * 2^-24
    const float zb = 2.0f * 1.01f * 1.4012985e-45f * 2.0f;                                // >= 2 * 1.01 * 2^-149
    const float eb = static_cast<float>(a.d) * 7.5231638e-37f * 1.0001f;                    // >= d * 2^-120
    const bool pre = a.d <= kPrefilterMaxD;
    bool finite = pre;
    // blocks [jb, jb + kStageJ) at a time (eight per lane), channels kStageC at a time through
    // the staged tile; every warp of the CTA joins the staging, also those with nothing to do
    const int imax = min(nblk, static_cast<int>(blockIdx.y + 1) * nw) - 1;   // the CTA's last query block
    const bool vec4 = nblk % 4 == 0 && (reinterpret_cast<uintptr_t>(a.kt32) & 15u) == 0;
    for (int jb = 0; pre && jb < imax; jb += kStageJ) {
        float s[8], m[8], z[8];
#pragma unroll
        for (int w = 0; w < 8; ++w) s[w] = m[w] = z[w] = 0.f;
        const bool mine = take > 0 && jb < i;
        // the blocks any warp of the CTA needs from this tile: j < imax (a multiple of 4 with
        // 16-byte loads; nblk % 4 == 0 keeps them inside the row)
        const int jn = vec4 ? min(kStageJ, (imax - jb + 3) / 4 * 4) : min(kStageJ, imax - jb);
        for (int cb0 = 0; cb0 < a.d; cb0 += kStageC) {
            const int cn = min(kStageC, a.d - cb0);
            __syncthreads();   // the previous tile has been read
            if (vec4) {   // 16-byte loads (rows of the key sums start 16-byte aligned)
#pragma unroll 4
                for (int idx = threadIdx.x; idx < cn * (kStageJ / 4); idx += blockDim.x) {
                    const int c = idx / (kStageJ / 4), q4 = idx % (kStageJ / 4);
                    if (4 * q4 < jn)
                        *reinterpret_cast<float4*>(kts + c * kStageJ + 4 * q4) =
                            *reinterpret_cast<const float4*>(kt + static_cast<int64_t>(cb0 + c) * nblk + jb + 4 * q4);
                }
            } else {
#pragma unroll 4
                for (int idx = threadIdx.x; idx < cn * kStageJ; idx += blockDim.x) {
                    const int c = idx / kStageJ, jj = idx % kStageJ;
                    if (jj < jn) kts[idx] = kt[static_cast<int64_t>(cb0 + c) * nblk + jb + jj];
                }
            }
            __syncthreads();
            if (mine) {
#pragma unroll 4
                for (int c = 0; c < cn; ++c) {
                    const float x = q32[cb0 + c];
                    const float* row = kts + c * kStageJ + lane;
#pragma unroll
                    for (int w = 0; w < 8; ++w) {
                        const float y = row[32 * w];
                        s[w] = fmaf(x, y, s[w]);
                        m[w] = fmaf(fabsf(x), fabsf(y), m[w]);
                        z[w] += fabsf(x) + fabsf(y);
                    }
                }
            }
        }
        if (mine) {
#pragma unroll
            for (int w = 0; w < 8; ++w) {
                const int j = jb + lane + 32 * w;
                if (j >= i) break;
                const float e = __fmaf_ru(cb, m[w], __fmaf_ru(zb, z[w], eb));
                const float lo = __fsub_rd(s[w], e), hi = __fadd_ru(s[w], e);
                finite = finite && isfinite(lo) && isfinite(hi);
                key32[j] = isfinite(lo) ? f32_key(lo) : 0;
                up[j] = hi;
                taken[j] = 0;
            }
        }
    }
    if (!active) return;
    if (take > 0) {
        __syncwarp();
        const bool exact_all = !__all_sync(0xffffffffu, finite);   // also every row of a wide head
        __syncwarp();
        float T = -INFINITY;   // the take-th largest lower bound
        if (!exact_all && take < i) {
            for (int t = 0; t < take; ++t) {
                int bk;
                const int bj = warp_best(key32, taken, i, lane, bk);
                if (lane == 0 && bj >= 0) taken[bj] = 1;
                __syncwarp();
                // the key decodes back to the float lower bound
                const int bits = bk >= 0 ? bk : (bk ^ 0x7FFFFFFF);
                T = __int_as_float(bits);
            }
        }
        __syncwarp();
        // ---- contract scores of the candidates (U_j >= T); the rest leave the ranking.  The
        // candidates are first packed into a list (over the upper bounds, no longer needed),
        // so that their float64 dot products run side by side, one per lane.
        for (int j = lane; j < i; j += 32) taken[j] = (exact_all || take >= i || up[j] >= T) ? 0 : 1;
        __syncwarp();
        int* list = reinterpret_cast<int*>(up);
        int count = 0;
        for (int base = 0; base < i; base += 32) {
            const int j = base + lane;
            const bool cand = j < i && !taken[j];
            const unsigned mask = __ballot_sync(0xffffffffu, cand);
            if (cand) list[count + __popc(mask & ((1u << lane) - 1u))] = j;
            count += __popc(mask);
        }
        __syncwarp();
        if (count == take) {
            // The set is decided without a contract score: the take blocks with the largest
            // lower bounds have U_j >= L_j >= T, so they are the whole list, and every other
            // block scores below T, i.e. below each of them (or all blocks are taken).  The
            // list is in block order, as the output is.
            int32_t* out = a.out + (bh * nblk + i) * a.top_n;
            for (int t = lane; t < a.top_n; t += 32) out[t] = t < take ? list[t] : -1;
            return;
        }
        for (int t = lane; t < count; t += 32) {
            const int j = list[t];
            key64[j] = rank_key(contract_dot(qs, a.ksum + (bh * nblk + j) * a.d, a.d));
        }
        __syncwarp();
        // ---- exact ranking among the candidates
        int pick0 = -1, pick1 = -1;   // pick t sits in lane t (t < 32) or lane t - 32
        for (int t = 0; t < take; ++t) {
            long long bk;
            const int bj = warp_best(key64, taken, i, lane, bk);
            if (t < 32 && lane == t) pick0 = bj;
            if (t >= 32 && lane == t - 32) pick1 = bj;
            __syncwarp();
            // at least `take` candidates exist, so bj >= 0 here
            if (lane == 0 && bj >= 0) taken[bj] = 1;
            __syncwarp();
        }
        for (int t = 0; t < 32; ++t) {
            picks[t] = __shfl_sync(0xffffffffu, pick0, t);
            picks[t + 32] = __shfl_sync(0xffffffffu, pick1, t);
        }
    }
    if (lane == 0) {
        for (int x = 1; x < take; ++x) {
            const int k = picks[x];
            int y = x - 1;
            while (y >= 0 && picks[y] > k) {
                picks[y + 1] = picks[y];
                --y;
            }
            picks[y + 1] = k;
        }
        int32_t* out = a.out + (bh * nblk + i) * a.top_n;
        for (int t = 0; t < a.top_n; ++t) out[t] = t < take ? picks[t] : -1;
    }
}

}  // namespace

// Per warp: keys[nblk] 64-bit words, up[nblk] floats, taken[nblk] bytes, q32[d] floats; per
// CTA: the staged key-sum tile (16-byte aligned).
size_t select_smem_bytes(int nblk, int d, int nw) {
    return static_cast<size_t>(nw) * (static_cast<size_t>(nblk) * (sizeof(long long) + sizeof(float) + 1) +
                                      sizeof(float) * static_cast<size_t>(d)) +
           16 + sizeof(float) * kStageC * kStageJ;
}

cudaError_t launch_select(const SelectArgs& a, cudaStream_t s) {
    const int nblk = a.S / a.block;
    dim3 g1(nblk, a.H, a.B);
    if (a.block <= 32) {
        // two bfloat16 channels per thread where every row of every head starts 4-byte aligned
        const bool pairs = a.dtype != BPA_FP32 && a.d % 2 == 0 && a.qs[0] % 2 == 0 && a.qs[1] % 2 == 0 &&
                           a.qs[2] % 2 == 0 && a.ks[0] % 2 == 0 && a.ks[1] % 2 == 0 && a.ks[2] % 2 == 0 &&
                           reinterpret_cast<uintptr_t>(a.q) % 4 == 0 && reinterpret_cast<uintptr_t>(a.k) % 4 == 0;
        const int nc = pairs ? 2 : 1;
        const int half = ((a.d + nc - 1) / nc + 31) / 32 * 32;
        if (a.dtype == BPA_FP32)
            k_block_sums_reg<float, 1><<<g1, 2 * half, 0, s>>>(a, half);
        else if (pairs)
            k_block_sums_reg<__nv_bfloat16, 2><<<g1, 2 * half, 0, s>>>(a, half);
        else
            k_block_sums_reg<__nv_bfloat16, 1><<<g1, 2 * half, 0, s>>>(a, half);
    } else {
        const int threads = a.d < 32 ? 32 : (a.d > 256 ? 256 : (a.d + 31) / 32 * 32);
        if (a.dtype == BPA_FP32)
            k_block_sums<float><<<g1, threads, 0, s>>>(a);
        else
            k_block_sums<__nv_bfloat16><<<g1, threads, 0, s>>>(a);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    int nw = kSelMaxWarps;
    while (nw > 1 && select_smem_bytes(nblk, a.d, nw) > 200 * 1024) nw /= 2;
    const size_t smem = select_smem_bytes(nblk, a.d, nw);
    if (smem > 48 * 1024) {
        e = cudaFuncSetAttribute(k_select, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    const dim3 g2(static_cast<unsigned>(static_cast<int64_t>(a.B) * a.H), static_cast<unsigned>((nblk + nw - 1) / nw));
    k_select<<<g2, nw * 32, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace bpa
