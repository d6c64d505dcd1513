// noalloc.cu - block selection for callers that cannot allocate device memory.
//
// bpa_select_blocks needs scratch (the float64 block sums and a status word)
// and expects the caller to provide it.  Some callers cannot: a plain C or
// C++ host program with no device allocator of its own, running next to
// other GPU work, should not call cudaMalloc, because cudaMalloc may
// synchronise the device and stall every other stream; other embedders
// (inference servers, plugins inside a host framework) forbid device
// allocations once they have started.  bpa_select_blocks_noalloc serves
// them with a scratch buffer that lives inside this library: a fixed-size
// __device__ array that every GPU loading the library keeps until the
// process exits.  No cudaMalloc, cudaFree or other allocating call is made.
#include <cuda_runtime.h>
#include <stdio.h>

#include <mutex>

#include "bpa.h"
#include "bpa_internal.h"

namespace {

// Largest scratch the variant can use: 16 MiB per GPU.
constexpr size_t kScratchBytes = static_cast<size_t>(16) << 20;

static __device__ __align__(256) unsigned char g_select_scratch[kScratchBytes];

// Device address of g_select_scratch, looked up once per device and kept for
// the life of the process: it does not survive cudaDeviceReset (or any other
// teardown of the device's primary context), after which this entry point must
// not be called again in the same process.
std::mutex g_mu;
void* g_addr[64] = {};

cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
        void* p = nullptr;
        // `g_select_scratch` names a host-side stand-in; only this call yields
        // the address the kernels can use on the current device.
        e = cudaGetSymbolAddress(&p, g_select_scratch);
        if (e != cudaSuccess) return e;
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" {

size_t bpa_select_noalloc_max_bytes(void) { return kScratchBytes; }

bpa_status bpa_select_blocks_noalloc(const void* q, const void* k, int32_t dtype, int32_t B, int32_t S,
                                     int32_t H, int32_t d, const int64_t q_strides[3],
                                     const int64_t k_strides[3], int32_t block_size, int32_t top_n,
                                     int32_t* block_idx_out, void* stream) {
    // the argument errors first, the same as bpa_select_blocks reports them
    const bpa_status st = bpa::check_select_args(q, k, dtype, B, S, H, d, q_strides, k_strides, block_size,
                                                 top_n, block_idx_out);
    if (st != BPA_OK) return st;
    const size_t need = bpa_select_workspace_size(B, S, H, d, block_size);
    if (need > kScratchBytes) {
        char msg[256];
        snprintf(msg, sizeof msg,
                 "bpa_select_blocks_noalloc: this problem needs %zu bytes of scratch, more than the "
                 "built-in %zu bytes; use bpa_select_blocks with a caller-provided workspace",
                 need, kScratchBytes);
        bpa::set_last_error(msg);
        return BPA_ERR_UNSUPPORTED;
    }
    void* scratch = nullptr;
    const cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess) {
        char msg[256];
        snprintf(msg, sizeof msg, "bpa_select_blocks_noalloc: cudaGetSymbolAddress failed: %s",
                 cudaGetErrorString(e));
        bpa::set_last_error(msg);
        return BPA_ERR_CUDA;
    }
    // The regular entry point clears the status word and overwrites every
    // block sum it reads, so stale contents of the shared buffer never leak
    // into a result.
    return bpa_select_blocks(q, k, dtype, B, S, H, d, q_strides, k_strides, block_size, top_n,
                             block_idx_out, scratch, kScratchBytes, stream);
}

}  // extern "C"
