// bpa_internal.h - validated problem description and kernel launchers of libbpa.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "bpa.h"

namespace bpa {

// A validated attention problem (scale resolved, ring geometry derived).
struct Problem {
    int B, S, Hq, Hkv, G, d;
    int dv;                    // head dim of v, o, dout (== d unless separate value head dims)
    int dtype;                 // bpa_dtype
    float scale;
    int causal, wl, wr;        // window bounds, -1 = unbounded
    const void* q;
    const void* k;
    const void* v;
    int64_t qs[3], ks[3], vs[3];
    int64_t os[3];             // strides of o and dout
    const float* bias;
    int64_t bs[4];
    int ring_n, ring_blk;      // ring_blk = S / ring_n
    const int32_t* block_idx;
    int sel_block, top_n, local_window;
    const int32_t* seqlens_q;  // device [B] or nullptr: valid queries per batch entry
    const int32_t* seqlens_kv; // device [B] or nullptr (then the query lengths)
    int bottom_right;          // diagonal at k = q + Lk - Lq instead of k = q
    const float* sink;         // device [Hq] sink logits (natural log units) or nullptr
    float* dsink;              // device [Hq] sink gradient (backward output) or nullptr
    int det;                   // deterministic backward (no atomic adds anywhere)
    uint32_t drop_thr;         // attention dropout: entries whose draw is below this are dropped (0: none)
    uint32_t drop_k0, drop_k1; // Philox4x32-10 key: the 64-bit seed's low and high words
};

// Valid query / key counts of one batch entry and the offset of the causal / window
// diagonal (k is compared with q + off).
struct Lens {
    int lq, lk, off;
};

#ifdef __CUDACC__
__device__ __forceinline__ Lens lens_of(const Problem& P, int b) {
    Lens L;
    L.lq = P.seqlens_q ? min(max(__ldg(P.seqlens_q + b), 0), P.S) : P.S;
    L.lk = P.seqlens_kv ? min(max(__ldg(P.seqlens_kv + b), 0), P.S) : L.lq;
    L.off = P.bottom_right ? L.lk - L.lq : 0;
    return L;
}
#endif

struct FwdArgs {
    Problem P;
    void* o;            // output (one-shot) - unused by ring steps
    float* m;           // [B, Hq, S]
    float* l;           // [B, Hq, S]
    float* acc;         // ring carry [B, S, Hq, dv] float32, or nullptr (one-shot)
    int ring_idx;       // ring step run by this launch
    uint32_t* status;   // device status word
    uint32_t* sched;    // work-item counter of the tensor-core forward; zero before each launch
};

struct BwdArgs {
    Problem P;
    const void* o;
    const void* dout;
    const float* m;
    const float* l;
    void* dq;
    void* dk;
    void* dv;
    float* Dvec;        // [B, Hq, Spad] rowsum(dO * O); padding rows hold 0
    float* lse;         // [B, Hq, Spad] m + log(l) (natural log); +inf on padding / empty rows
    int Spad;           // S rounded up to 64
    float* dq_acc;      // [B, Hq, Spad / 4, d, 4] float32 (four consecutive queries of a channel together);
                        // deterministic mode: one such slice per 128-key tile, [nkt][B, Hq, Spad / 4, d, 4]
    int dq_direct;      // band backward: dQ added in bf16 pairs straight into dq (zeroed by the pre-pass)
    int hsplit;         // band backward: CTAs per key tile, each taking G / hsplit q heads (1 or 2); with 2
                        // the halves add dK, dV in bf16 pairs into dk, dv (zeroed by the pre-pass)
    float* dk_acc;      // ring carries / block-selected accumulators [B, S, Hkv, d] float32, or nullptr
    float* dv_acc;
    int ring_idx;
    uint32_t* status;
};

struct SelectArgs {
    const void* q;
    const void* k;
    int dtype, B, S, H, d;
    int64_t qs[3], ks[3];
    int block, top_n;
    int32_t* out;
    double* qsum;       // [B, H, nblk, d]
    double* ksum;
    float* kt32;        // [B, H, d, nblk] float32 copies of the key sums (the pre-filter's)
    uint32_t* status;
};

// ---- launchers (return the launch error, if any) --------------------------
cudaError_t launch_fwd_simt(const FwdArgs& a, cudaStream_t s);
cudaError_t launch_bwd_simt(const BwdArgs& a, cudaStream_t s);
cudaError_t launch_fwd_tc(const FwdArgs& a, const CUtensorMap* maps, cudaStream_t s);
cudaError_t launch_bwd_tc(const BwdArgs& a, const CUtensorMap* maps, cudaStream_t s);
// Band backward (every 64-row query tile seen by at most two key tiles): the tensor-core
// kernel adding dQ straight into dq; bwd_band_supported says when it applies.
bool bwd_band_supported(const Problem& P);
cudaError_t launch_bwd_tc_band(const BwdArgs& a, const CUtensorMap* maps, cudaStream_t s);
cudaError_t launch_gather_fwd(const FwdArgs& a, cudaStream_t s);
cudaError_t launch_gather_bwd(const BwdArgs& a, cudaStream_t s);   // needs dk_acc / dv_acc cleared
cudaError_t launch_cast_dkdv(const BwdArgs& a, cudaStream_t s);    // dk_acc / dv_acc -> dk / dv (bf16)
cudaError_t launch_ring_init(const FwdArgs& a, cudaStream_t s);
cudaError_t launch_ring_finalize(const FwdArgs& a, cudaStream_t s);
cudaError_t launch_bwd_pre(const BwdArgs& a, cudaStream_t s);
cudaError_t launch_bwd_post(const BwdArgs& a, cudaStream_t s);
cudaError_t launch_sink_grad(const BwdArgs& a, cudaStream_t s);   // after the pre-pass (LSE, D)
cudaError_t launch_pad_stats(const FwdArgs& a, cudaStream_t s);   // m, l of padding rows
cudaError_t launch_dq_reduce(const BwdArgs& a, cudaStream_t s);   // deterministic mode: slices -> dq
cudaError_t launch_select(const SelectArgs& a, cudaStream_t s);
cudaError_t launch_wait_selftest(uint32_t* status, uint64_t limit_ns, cudaStream_t s);
cudaError_t launch_check_blocks(const Problem& P, uint32_t* status, cudaStream_t s);   // block_idx contract

void set_last_error(const char* msg);

// Most blocks per sequence the selection takes (its per-warp score list lives in shared memory).
constexpr int kSelectMaxBlocks = 4096;

// The argument checks of bpa_select_blocks other than the workspace's (sets the last error).
bpa_status check_select_args(const void* q, const void* k, int32_t dtype, int32_t B, int32_t S, int32_t H,
                             int32_t d, const int64_t q_strides[3], const int64_t k_strides[3],
                             int32_t block_size, int32_t top_n, const int32_t* block_idx_out);

bool fwd_tc_supported(const Problem& P);
// Narrow key bands with grouped heads take the band forward (fwd_band.cu).
bool fwd_band_supported(const Problem& P);
cudaError_t launch_fwd_band(const FwdArgs& a, const CUtensorMap* maps, cudaStream_t s);
bool bwd_tc_supported(const Problem& P);
bool gather_supported(const Problem& P);

}  // namespace bpa
