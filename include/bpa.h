/*
 * bpa.h - blockwise exact attention on NVIDIA GB300 (sm_103a): the C ABI of libbpa.so.
 *
 * What the library computes (the sources are the pages this project follows;
 * each entry point names the passage that defines it):
 *
 *   For batch b, query head h, kv head g = h / (Hq / Hkv), query position q:
 *     z_k = scale * <Q[b,q,h,:], K[b,k,g,:]> + bias[b,h,q,k]      (allowed k only)
 *     m   = max_k z_k,  l = sum_k exp(z_k - m),
 *     O[b,q,h,:] = sum_k exp(z_k - m) / l * V[b,k,g,:]
 *   computed one KV tile at a time and folded into a running
 *   (max, numerator, denominator) carry with the exp(previous max - max)
 *   correction ("bpt.py", _blockwise_attention_fwd / scan_kv_block), and
 *   its gradients recomputed from the saved O, m and l
 *   ("bpt.py", _blockwise_attention_bwd and the einsum version in
 *   _ring_attention_bwd).
 *
 *   allowed(q, k) = (!causal || k <= q)
 *                && (window_left  < 0 || k >= q - window_left)
 *                && (window_right < 0 || k <= q + window_right)
 *                && (block mode: k in [q - local_window + 1, q] or in a selected block)
 *   (bounds inclusive; "JAX: Single-GPU Attention with TransformerEngine",
 *   section 1, _make_causal_swa_mask; the GQA head map is _repeat_kv_for_gqa).
 *   Masked entries are excluded exactly.  A row with no allowed key yields
 *   O = 0, m = -inf, l = 0 and zero gradients.
 *
 * Conventions shared by every entry point:
 *   - Tensors are BSHD: element (b, s, h, c) of a tensor with strides
 *     (sb, ss, sh) sits at base + b*sb + s*ss + h*sh + c (strides counted in
 *     elements, the last dimension contiguous).  Q, O, dO and dQ share
 *     q_strides; K and dK share k_strides; V and dV share v_strides.
 *     For the bf16 tensor-core path every stride must be a multiple of 8
 *     elements and every base pointer 16-byte aligned.
 *   - m and l are float32 [B, Hq, S], contiguous, natural-log units of z.
 *   - All pointers are device pointers owned by the caller.  The library
 *     allocates no device memory at run time and keeps no per-call state;
 *     scratch lives in the caller's workspace (size from bpa_workspace_size).
 *     The one exception is static: every GPU that loads the library holds a
 *     fixed 16 MiB __device__ array until the process exits, the scratch of
 *     bpa_select_blocks_noalloc (unused by every other entry point).
 *   - Calls are asynchronous on the given stream (a cudaStream_t passed as
 *     void*; NULL is the legacy default stream).  Argument errors are
 *     returned before anything is launched.  Launch failures return
 *     BPA_ERR_CUDA.  Faults detected by the kernels themselves (a bounded
 *     wait that ran out, a failed device-side check) are recorded in the
 *     workspace's status word, which each call clears first; read it with
 *     bpa_check() after the stream has been synchronised.
 *   - Not thread-safe with respect to one workspace: concurrent calls must
 *     use separate workspaces.
 */
#ifndef BPA_H
#define BPA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define BPA_VERSION 6

typedef enum {
    BPA_OK = 0,
    BPA_ERR_INVALID_ARG = 1,   /* a null pointer, a bad size, stride or mode */
    BPA_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. head dim) */
    BPA_ERR_WORKSPACE = 3,     /* workspace missing, misaligned or too small */
    BPA_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
    BPA_ERR_TIMEOUT = 5,       /* (bpa_check) a kernel's bounded wait ran out */
    BPA_ERR_DEVICE_CHECK = 6   /* (bpa_check) a kernel's own bounds check failed */
} bpa_status;

typedef enum { BPA_BF16 = 0, BPA_FP32 = 1 } bpa_dtype;

typedef enum { BPA_OP_FWD = 0, BPA_OP_BWD = 1 } bpa_op;

/* Describes one attention problem.  Zero-initialise, then set struct_size. */
typedef struct bpa_attn_desc {
    uint32_t struct_size;      /* = sizeof(bpa_attn_desc) */
    int32_t dtype;             /* bpa_dtype of q, k, v, o, dout, dq, dk, dv */
    int32_t B, S, Hq, Hkv, d;  /* q, k, v share the padded length S (shorter sequences: the
                                * version-3 lengths below); Hq % Hkv == 0; 1 <= d <= 512 (head
                                * dim of q, k) */
    const void* q;             /* [B, S, Hq, d] */
    const void* k;             /* [B, S, Hkv, d] */
    const void* v;             /* [B, S, Hkv, dv] */
    int64_t q_strides[3];      /* (b, s, h) strides of q, dq (and of o, dout unless o_strides is set) */
    int64_t k_strides[3];      /* (b, s, h) strides of k, dk */
    int64_t v_strides[3];      /* (b, s, h) strides of v, dv */
    float scale;               /* <= 0 selects d^-0.5 */
    int32_t causal;            /* nonzero: k <= q (positions share one origin) */
    int32_t window_left;       /* inclusive; -1 = unbounded */
    int32_t window_right;      /* inclusive; -1 = unbounded */
    const float* bias;         /* optional additive float32 bias, NULL = none */
    int64_t bias_strides[4];   /* (b, h, q, k) strides in elements; 0 broadcasts */
    int32_t query_chunk;       /* the pages' chunk sizes: 0 or a divisor of S/ring_size; */
    int32_t key_chunk;         /* they never change the result (tiling is the kernel's) */
    int32_t ring_size;         /* >= 1: KV super-blocks swept in ring order, S % ring_size == 0 */
    int32_t ring_step_begin;   /* first ring step of this call, 0 <= begin < end */
    int32_t ring_step_end;     /* one past the last step; 0 selects ring_size */
    const int32_t* block_idx;  /* block-selected mode: [B, Hq, S/sel_block, top_n] from
                                *   bpa_select_blocks: each entry -1 (ignored) or a block before
                                *   the query block.  Other entries are ignored too, and the
                                *   call records BPA_ERR_DEVICE_CHECK for bpa_check */
    int32_t sel_block;
    int32_t top_n;
    int32_t local_window;      /* keys q - local_window + 1 .. q are always allowed */
    /* Fields below were added in descriptor version 2 (bpa_version() >= 2).  A caller
     * that sets struct_size = offsetof(bpa_attn_desc, dv) (version 1) gets dv = d and
     * o_strides = q_strides.  Separate value head dims follow "JAX: Single-GPU Attention
     * with TransformerEngine", section 4 (DeepSeek-style MLA head dimensions: q, k with
     * head dim d, v and the output with head dim dv). */
    int32_t dv;                /* head dim of v, o, dout and the dv gradient; 0 selects d; <= 512 */
    int64_t o_strides[3];      /* (b, s, h) strides of o and dout; all 0 selects q_strides */
    /* Fields below were added in descriptor version 3 (bpa_version() >= 3); a version-2
     * caller (struct_size = offsetof(bpa_attn_desc, seqlens_q)) gets full-length sequences.
     * Variable lengths follow the sequence descriptor of "JAX: Single-GPU Attention with
     * TransformerEngine", section 1 (SequenceDescriptor.from_seqlens): batch entry b holds
     * Lq = seqlens_q[b] queries and Lk = seqlens_kv[b] keys at positions 0..L-1 of the
     * padded [B, S, H, d] tensors.  Later positions are padding: they attend to nothing
     * and nothing attends to them; their rows of o, dq get 0, of m -inf, of l 0, and
     * their rows of dk, dv get 0.  Padding must hold finite numbers (it is read by the
     * tiled loads and weighted by exactly 0).  Values are clamped to [0, S].  Needs
     * ring_size 1 and no block selection. */
    const int32_t* seqlens_q;  /* device int32 [B] or NULL (every entry S) */
    const int32_t* seqlens_kv; /* device int32 [B] or NULL (the query lengths) */
    int32_t bottom_right;      /* 0: causal / window diagonal at k = q (top-left, both
                                * sequences start together); 1: at k = q + Lk - Lq (the
                                * queries are the last Lq positions of the key sequence) */
    /* Fields below were added in descriptor version 4 (bpa_version() >= 4); a version-3
     * caller (struct_size = offsetof(bpa_attn_desc, sink)) gets plain softmax.  Sink
     * attention: "JAX: Single-GPU Attention with TransformerEngine", Other attention knobs
     * (softmax_type "off_by_one" or "learnable"), read as one extra logit per q head with
     * no value vector in every valid row's softmax:  P = exp(z) / (exp(sink[h]) + sum exp(z))
     * (off_by_one: sink = 0).  m and l include it (m = max(max z, sink)); a row with no
     * allowed key gets O = 0, m = sink, l = 1.  Needs ring_size 1. */
    const float* sink;         /* device float32 [Hq] or NULL (plain softmax) */
    float* dsink;              /* device float32 [Hq] or NULL: bpa_bwd writes
                                * dsink[h] = -sum over valid rows of P_sink <dO, O> */
    /* Field added in descriptor version 5 (bpa_version() >= 5); a version-4 caller
     * (struct_size = offsetof(bpa_attn_desc, deterministic)) gets 0.  The determinism knob
     * of "JAX: Single-GPU Attention with TransformerEngine", Other attention knobs
     * (NVTE_ALLOW_NONDETERMINISTIC_ALGO=0): with 1, bpa_bwd gives bit-identical dq, dk, dv
     * on every call: each key tile's dQ contribution goes to its own float32 slice of the
     * workspace (no atomic adds) and the slices are added in ascending key order.  The
     * workspace then holds one dQ slice per 128-key tile (bpa_workspace_size grows by about
     * that factor).  Needs ring_size 1. */
    int32_t deterministic;
    /* Fields below were added in descriptor version 6 (bpa_version() >= 6); a version-5
     * caller (struct_size = offsetof(bpa_attn_desc, dropout_threshold)) gets no dropout.
     * Attention dropout as "bpt.py" applies it (_blockwise_attention_fwd / _bwd with
     * attn_pdrop, _chunk_attention_bias): each score entry (b, h, q, k) is dropped with
     * probability p, and a dropped entry leaves the softmax (the dtype minimum is added to
     * its score), so the row renormalises over the kept keys; no 1/(1-p) factor.  m and l
     * cover the kept keys only.  The decision is an integer comparison, identical on every
     * path and in both passes: the 32-bit draw of entry (b, h, q, k) is word k % 4 of
     * Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC 2011) with key (seed low 32 bits, seed
     * high 32 bits) and counter (k / 4, q, h, b), at the entry's positions in the padded
     * [B, S, ...] tensors, and the entry is dropped when the draw is below
     * dropout_threshold = round(p * 2^32) (capped at 2^32 - 1).  bpa_bwd must be given the
     * threshold and seed of the forward call. */
    uint32_t dropout_threshold;   /* 0: no dropout */
    uint32_t dropout_reserved;    /* must be 0 */
    uint64_t dropout_seed;
} bpa_attn_desc;

/* Bytes of workspace bpa_fwd (op = BPA_OP_FWD) or bpa_bwd (op = BPA_OP_BWD)
 * needs for this problem, a multiple of 256.  0 if the descriptor is invalid.
 * Forward: a status header, plus, when ring_size > 1, the float32 running
 * numerator [B, S, Hq, dv].  Backward: the header, D = rowsum(dO * O) and
 * the log-sum-exp [B, Hq, S'] (S' = S rounded up to 64), the float32 dQ
 * accumulator [B, Hq, S', d], plus, when ring_size > 1 or in block-selected
 * mode, float32 dK and dV carries / accumulators [B, S, Hkv, d] and
 * [B, S, Hkv, dv]. */
size_t bpa_workspace_size(int32_t op, const bpa_attn_desc* desc);

/* Forward pass.
 * Defined by "bpt.py", _blockwise_attention_fwd (scan_kv_block: scores,
 * running max, exp correction, numerator and denominator) and
 * _ring_attention_fwd (ring order: query block i meets KV block
 * (i - idx) mod n at step idx; output = numerator / denominator).
 * Writes o [B, S, Hq, dv] (dtype of the inputs, strides o_strides) and m, l [B, Hq, S].
 * With ring_size = n > 1 the sequence is cut into n query blocks and n KV
 * super-blocks; steps [ring_step_begin, ring_step_end) run, carrying the
 * float32 numerator in the workspace and the running max / denominator in
 * m and l between steps, so a sweep may stop after any step and resume
 * with the same workspace, m and l.  o is written by the call that runs
 * the last step (n - 1).  The workspace must not be touched between
 * partial calls.  Block-selected mode (block_idx != NULL) needs ring_size 1.
 * Returns BPA_OK or an error code; see the conventions above. */
bpa_status bpa_fwd(const bpa_attn_desc* desc, void* o, float* m, float* l,
                   void* workspace, size_t workspace_bytes, void* stream);

/* Backward pass: dq, dk, dv from the saved output o, the row statistics
 * m and l of bpa_fwd, and the output gradient dout.
 * Defined by "bpt.py", _blockwise_attention_bwd and the einsum version in
 * _ring_attention_bwd:  D = rowsum(dO * O);  P = exp(z - m) / l;
 * dP = dO V^T;  dS = P (dP - D);  dQ = scale dS K;  dK = scale dS^T Q;
 * dV = P^T dO, with dK and dV summed over the q heads of each kv group.
 * No gradient is produced for the bias.  With ring_size > 1 the steps run
 * in ring order like the forward pass, the float32 dK / dV carries stand
 * in for the gradients that travel around the ring, and all steps run in
 * one call (ring_step_begin / ring_step_end must select the whole sweep).
 * dq, dk, dv have the dtype of the inputs and the strides of q, k, v; o and
 * dout are [B, S, Hq, dv] with o_strides.  dq, dk, dv must not overlap any input:
 * some paths zero them first and add partial results into them (narrow windows: dq;
 * contiguous dk, dv with narrow windows or with eight or more q heads per kv head: dk, dv,
 * from two CTAs per key tile, so the two-term sums are the same on every call).
 * Block-selected mode (ring_size 1) is supported: the selection is held
 * fixed ("AnnAttention", faiss_block_attention.py, which trains through the
 * gathered attention; no gradient reaches the indices), so the gradients are
 * those of attention under the union mask of the forward pass. */
bpa_status bpa_bwd(const bpa_attn_desc* desc, const void* o, const void* dout,
                   const float* m, const float* l, void* dq, void* dk, void* dv,
                   void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of workspace bpa_select_blocks needs (a multiple of 256), 0 if invalid. */
size_t bpa_select_workspace_size(int32_t B, int32_t S, int32_t H, int32_t d, int32_t block_size);

/* Exact top-n block selection.
 * Defined by "AnnAttention", faiss_block_attention.py, select_block (block
 * means as index keys, candidates strictly earlier than the query block,
 * indices sorted), made exact: per (b, h) the block sums
 * Qs[i] = sum of rows 32i..32i+31 of Q (likewise Ks[j]) are accumulated in
 * row order in float64; score(i, j) = sum_c Qs[i][c] * Ks[j][c] in channel
 * order, each step a float64 multiply then a float64 add (no fused
 * multiply-add).  Block i keeps the min(top_n, i) largest scores over
 * j < i (equal scores keep the lower j), written in ascending j and padded
 * with -1, to block_idx_out int32 [B, H, S/block_size, top_n].  Sums and
 * not means are compared; they rank identically.
 * q and k are [B, S, H, d] (dtype bpa_dtype) with (b, s, h) strides.
 * S % block_size == 0, S / block_size <= 4096, 1 <= top_n <= 64, d <= 512.
 * A NaN score (from non-finite inputs; the page does not rank one) ranks
 * below every number, NaN scores in block order. */
bpa_status bpa_select_blocks(const void* q, const void* k, int32_t dtype, int32_t B,
                             int32_t S, int32_t H, int32_t d, const int64_t q_strides[3],
                             const int64_t k_strides[3], int32_t block_size, int32_t top_n,
                             int32_t* block_idx_out, void* workspace,
                             size_t workspace_bytes, void* stream);

/* Block selection for callers that cannot provide device scratch memory.
 * (An addition of this library; the pages have no counterpart.)
 * Same inputs, output and arithmetic as bpa_select_blocks, minus the
 * workspace: the scratch is a fixed 16 MiB buffer compiled into the
 * library (a __device__ array that every GPU loading the library keeps
 * until the process exits).  It is for programs that must not call
 * cudaMalloc themselves: a plain host program without a device allocator,
 * where cudaMalloc could synchronise the device and stall other streams,
 * or an embedder that forbids device allocations after start-up.  This
 * entry point allocates nothing and calls no allocating routine.
 *   - Limit: problems whose bpa_select_workspace_size exceeds
 *     bpa_select_noalloc_max_bytes() (16 MiB; e.g. B*H*(S/block_size)*d
 *     up to about one million) are rejected with BPA_ERR_UNSUPPORTED
 *     before anything is launched; use bpa_select_blocks for them.
 *   - The first call on each device looks up the buffer's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture on that device.  The address is kept for the
 *     life of the process and does not survive cudaDeviceReset: do not call
 *     this entry point after resetting the device.
 *   - All calls share the one buffer, which keeps the last call's contents:
 *     each call clears the status word and overwrites every block sum it
 *     reads.  Calls whose kernels overlap on the GPU (different streams, or
 *     host threads without ordering between them) race on the buffer:
 *     order them on one stream.
 *   - Argument errors are reported exactly as bpa_select_blocks reports
 *     them, before the size limit is checked.  Errors come back through the
 *     returned code and bpa_last_error(); the selection kernels write no
 *     device-side status, so there is nothing for bpa_check to read here. */
size_t bpa_select_noalloc_max_bytes(void);
bpa_status bpa_select_blocks_noalloc(const void* q, const void* k, int32_t dtype, int32_t B,
                                     int32_t S, int32_t H, int32_t d,
                                     const int64_t q_strides[3], const int64_t k_strides[3],
                                     int32_t block_size, int32_t top_n,
                                     int32_t* block_idx_out, void* stream);

/* Reads the status word of a workspace used by an earlier call (blocking
 * copy; synchronise the stream first).  BPA_OK, BPA_ERR_TIMEOUT or
 * BPA_ERR_DEVICE_CHECK; BPA_ERR_CUDA if the copy itself fails. */
bpa_status bpa_check(const void* workspace);

/* Human-readable name of a status code (static storage). */
const char* bpa_status_string(bpa_status status);

/* Detail of the last error returned on this host thread (static storage,
 * overwritten by the next failing call; "" if none). */
const char* bpa_last_error(void);

/* BPA_VERSION of the library. */
int32_t bpa_version(void);

/* Instrumentation: the next bpa_fwd or bpa_bwd call made on this host
 * thread records the given CUDA events (cudaEvent_t values) on its stream
 * at its phase boundaries, then forgets them.  bpa_fwd: [0] before the
 * first kernel, [1] after the attention kernel(s) (every ring step), [2] at
 * the end (after the ring finalize).  bpa_bwd: [0] before the pre-pass,
 * [1] after it, [2] after the main kernel(s), [3] at the end.  Events past n
 * are not recorded; n <= 0 or events == NULL clears the hook.  Timing only:
 * nothing else changes. */
void bpa_set_phase_events(void* const* events, int32_t n);

/* Diagnostic for failure detection: launches one CTA whose bounded wait on a
 * barrier that nothing ever completes must give up after limit_ns
 * (0 < limit_ns <= 5e9) and record BPA_ERR_TIMEOUT in the workspace's status
 * word (read it with bpa_check after synchronising).  The same bounded-wait
 * routine guards every wait in the attention kernels.  Needs >= 256 bytes of
 * workspace.  This is not part of the pages' method. */
bpa_status bpa_debug_wait_timeout(void* workspace, size_t workspace_bytes, uint64_t limit_ns,
                                  void* stream);

#ifdef __cplusplus
}
#endif

#endif /* BPA_H */
