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
    const int groups = (P.d + 7) / 8;
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
        const float* C = a.acc + ((static_cast<int64_t>(b) * P.S + q) * P.Hq + h) * P.d;
        T* O = static_cast<T*>(a.o) + b * P.qs[0] + static_cast<int64_t>(q) * P.qs[1] + h * P.qs[2];
        for (int c = gi * 8; c < min(P.d, gi * 8 + 8); ++c) stf(O + c, C[c] * inv);
    }
}

// one warp per (b, h, q) row of the padded [B, Hq, Spad] statistics
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
            const int64_t off = b * P.qs[0] + static_cast<int64_t>(q) * P.qs[1] + h * P.qs[2];
            const T* O = static_cast<const T*>(a.o) + off;
            const T* dO = static_cast<const T*>(a.dout) + off;
            float s = 0.f;
            for (int c = lane; c < P.d; c += 32) s = fmaf(ldf(O + c), ldf(dO + c), s);
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
        const int64_t n4 = static_cast<int64_t>(P.B) * P.S * P.Hq * P.d / 4;
        float4* z = reinterpret_cast<float4*>(a.dq_acc);
        const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
        for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n4; i += stride)
            z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

// float32 [B, S, H, d] accumulator -> dtype tensor with strides st
template <typename T>
__global__ void k_cast_out(const float* src, T* dst, int B, int S, int H, int d, int64_t s0,
                           int64_t s1, int64_t s2, float mul) {
    const int64_t total = static_cast<int64_t>(B) * S * H * d;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total; i += stride) {
        const int c = static_cast<int>(i % d);
        int64_t r = i / d;
        const int h = static_cast<int>(r % H);
        r /= H;
        const int q = static_cast<int>(r % S);
        const int b = static_cast<int>(r / S);
        stf(dst + b * s0 + static_cast<int64_t>(q) * s1 + h * s2 + c, src[i] * mul);
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
    const int64_t n_acc = static_cast<int64_t>(P.B) * P.S * P.Hq * P.d;
    const int64_t n_rows = static_cast<int64_t>(P.B) * P.Hq * P.S;
    k_ring_init<<<grid_for(n_acc, 256), 256, 0, s>>>(a.acc, a.m, a.l, n_acc, n_rows);
    return cudaGetLastError();
}

cudaError_t launch_ring_finalize(const FwdArgs& a, cudaStream_t s) {
    const Problem& P = a.P;
    const int64_t work = static_cast<int64_t>(P.B) * P.S * P.Hq * ((P.d + 7) / 8);
    if (P.dtype == BPA_FP32)
        k_ring_finalize<float><<<grid_for(work, 256), 256, 0, s>>>(a);
    else
        k_ring_finalize<__nv_bfloat16><<<grid_for(work, 256), 256, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_bwd_pre(const BwdArgs& a, cudaStream_t s) {
    const Problem& P = a.P;
    const int64_t rows = static_cast<int64_t>(P.B) * P.Hq * a.Spad;
    const int zero = a.dq_acc != nullptr;
    if (P.dtype == BPA_FP32)
        k_bwd_pre<float><<<grid_for(rows * 32, 256), 256, 0, s>>>(a, zero);
    else
        k_bwd_pre<__nv_bfloat16><<<grid_for(rows * 32, 256), 256, 0, s>>>(a, zero);
    return cudaGetLastError();
}

cudaError_t launch_bwd_post(const BwdArgs& a, cudaStream_t s) {
    const Problem& P = a.P;
    const int64_t nq = static_cast<int64_t>(P.B) * P.S * P.Hq * P.d;
    const int64_t nk = static_cast<int64_t>(P.B) * P.S * P.Hkv * P.d;
    if (P.dtype != BPA_BF16) return cudaErrorInvalidValue;
    k_cast_out<__nv_bfloat16><<<grid_for(nq, 256), 256, 0, s>>>(
        a.dq_acc, static_cast<__nv_bfloat16*>(a.dq), P.B, P.S, P.Hq, P.d, P.qs[0], P.qs[1], P.qs[2],
        1.f);
    if (a.dk_acc) {
        k_cast_out<__nv_bfloat16><<<grid_for(nk, 256), 256, 0, s>>>(
            a.dk_acc, static_cast<__nv_bfloat16*>(a.dk), P.B, P.S, P.Hkv, P.d, P.ks[0], P.ks[1],
            P.ks[2], 1.f);
        k_cast_out<__nv_bfloat16><<<grid_for(nk, 256), 256, 0, s>>>(
            a.dv_acc, static_cast<__nv_bfloat16*>(a.dv), P.B, P.S, P.Hkv, P.d, P.vs[0], P.vs[1],
            P.vs[2], 1.f);
    }
    return cudaGetLastError();
}

cudaError_t launch_wait_selftest(uint32_t* status, uint64_t limit_ns, cudaStream_t s) {
    k_wait_selftest<<<1, 32, 0, s>>>(status, limit_ns);
    return cudaGetLastError();
}

}  // namespace bpa
