// select.cu - exact top-n block selection ("AnnAttention", faiss_block_attention.py,
// select_block, made exact: brute-force dot products of block sums).
//
// Arithmetic contract (it makes the result bit-identical to any
// implementation that performs the same IEEE operations in the same order):
//   Qs[i][c] = ((0 + x_0) + x_1) + ... + x_{bs-1}      float64, rows in order
//   score    = ((0 + a_0*b_0) + a_1*b_1) + ...         float64, channels in
//              order, every product and sum rounded separately (no FMA)
//   ranking  : larger score first, the lower block index on equal scores.
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

// grid (nblk, H, B), one thread per channel
template <typename T>
__global__ void k_block_sums(const SelectArgs a) {
    const int i = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int nblk = a.S / a.block;
    const T* Q = static_cast<const T*>(a.q);
    const T* K = static_cast<const T*>(a.k);
    for (int c = threadIdx.x; c < a.d; c += blockDim.x) {
        double sq = 0.0, sk = 0.0;
        for (int r = 0; r < a.block; ++r) {
            const int64_t s = static_cast<int64_t>(i) * a.block + r;
            sq = __dadd_rn(sq, ldd(Q + b * a.qs[0] + s * a.qs[1] + h * a.qs[2] + c));
            sk = __dadd_rn(sk, ldd(K + b * a.ks[0] + s * a.ks[1] + h * a.ks[2] + c));
        }
        const int64_t o = ((static_cast<int64_t>(b) * a.H + h) * nblk + i) * a.d + c;
        a.qsum[o] = sq;
        a.ksum[o] = sk;
    }
}

// Ranking: a larger score first, the lower block on equal scores; a NaN score
// (non-finite inputs) ranks below every number, NaNs in block order.
__device__ __forceinline__ bool better(double sa, int ja, double sb, int jb) {
    const bool na = sa != sa, nb = sb != sb;
    if (na != nb) return nb;
    if (na) return ja < jb;
    return sa > sb || (sa == sb && ja < jb);
}

constexpr int kSelWarps = 4;

// one warp per (b, h, query block i); the scores of the i earlier blocks live
// in shared memory (kSelWarps * nblk doubles), followed by one "taken" byte
// per block and warp.
__global__ void __launch_bounds__(kSelWarps * 32) k_select(const SelectArgs a) {
    extern __shared__ double sc_all[];
    const int nblk = a.S / a.block;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t unit = static_cast<int64_t>(blockIdx.x) * kSelWarps + warp;
    if (unit >= static_cast<int64_t>(a.B) * a.H * nblk) return;
    const int i = static_cast<int>(unit % nblk);
    const int64_t bh = unit / nblk;
    double* sc = sc_all + static_cast<int64_t>(warp) * nblk;
    unsigned char* taken = reinterpret_cast<unsigned char*>(sc_all + static_cast<int64_t>(kSelWarps) * nblk) +
                           static_cast<int64_t>(warp) * nblk;
    const double* qs = a.qsum + (bh * nblk + i) * a.d;
    for (int j = lane; j < i; j += 32) {
        const double* ks = a.ksum + (bh * nblk + j) * a.d;
        double acc = 0.0;
        for (int c = 0; c < a.d; ++c) acc = __dadd_rn(acc, __dmul_rn(qs[c], ks[c]));
        sc[j] = acc;
        taken[j] = 0;
    }
    __syncwarp();
    const int take = i < a.top_n ? i : a.top_n;
    int pick0 = -1, pick1 = -1;   // pick t sits in lane t (t < 32) or lane t - 32
    for (int t = 0; t < take; ++t) {
        double bs = 0.0;
        int bj = -1;
        for (int j = lane; j < i; j += 32) {
            if (taken[j]) continue;
            const double s = sc[j];
            if (bj < 0 || better(s, j, bs, bj)) {
                bs = s;
                bj = j;
            }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            const double os = __shfl_xor_sync(0xffffffffu, bs, o);
            const int oj = __shfl_xor_sync(0xffffffffu, bj, o);
            if (oj >= 0 && (bj < 0 || better(os, oj, bs, bj))) {
                bs = os;
                bj = oj;
            }
        }
        if (t < 32 && lane == t) pick0 = bj;
        if (t >= 32 && lane == t - 32) pick1 = bj;
        __syncwarp();
        // t < take <= i leaves an untaken candidate, so bj >= 0 here
        if (lane == 0 && bj >= 0) taken[bj] = 1;
        __syncwarp();
    }
    int picks[64];
    for (int t = 0; t < 32; ++t) {
        const int x0 = __shfl_sync(0xffffffffu, pick0, t);
        const int x1 = __shfl_sync(0xffffffffu, pick1, t);
        picks[t] = x0;
        picks[t + 32] = x1;
    }
    if (lane == 0) {
        for (int x = 1; x < take; ++x) {
            const int key = picks[x];
            int y = x - 1;
            while (y >= 0 && picks[y] > key) {
                picks[y + 1] = picks[y];
                --y;
            }
            picks[y + 1] = key;
        }
        int32_t* out = a.out + (bh * nblk + i) * a.top_n;
        for (int t = 0; t < a.top_n; ++t) out[t] = t < take ? picks[t] : -1;
    }
}

}  // namespace

cudaError_t launch_select(const SelectArgs& a, cudaStream_t s) {
    const int nblk = a.S / a.block;
    dim3 g1(nblk, a.H, a.B);
    const int threads = a.d < 32 ? 32 : (a.d > 256 ? 256 : (a.d + 31) / 32 * 32);
    if (a.dtype == BPA_FP32)
        k_block_sums<float><<<g1, threads, 0, s>>>(a);
    else
        k_block_sums<__nv_bfloat16><<<g1, threads, 0, s>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t units = static_cast<int64_t>(a.B) * a.H * nblk;
    const size_t smem = (sizeof(double) + 1) * kSelWarps * static_cast<size_t>(nblk);
    if (smem > 48 * 1024) {
        e = cudaFuncSetAttribute(k_select, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    k_select<<<static_cast<unsigned>((units + kSelWarps - 1) / kSelWarps), kSelWarps * 32, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace bpa
