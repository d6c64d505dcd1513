// api.cu - the C ABI of libbpa (declared in include/bpa.h): argument checks,
// workspace layout, TMA descriptors and the launch sequence of each entry point.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stddef.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "bpa.h"
#include "bpa_internal.h"
#include "common.cuh"

using namespace bpa;

namespace {

thread_local char g_last_error[512] = "";

// phase-event hook (bpa_set_phase_events): consumed by the next fwd / bwd call
thread_local cudaEvent_t g_phase_events[8];
thread_local int g_phase_n = 0;

struct PhaseMarks {
    cudaEvent_t ev[8];
    int n = 0;
    PhaseMarks() {
        n = g_phase_n;
        for (int i = 0; i < n; ++i) ev[i] = g_phase_events[i];
        g_phase_n = 0;
    }
    void mark(int i, cudaStream_t s) const {
        if (i < n && ev[i]) cudaEventRecord(ev[i], s);
    }
};

bpa_status fail(bpa_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return st;
}

bpa_status cuda_fail(cudaError_t e, const char* what) {
    return fail(BPA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// NVTX range over a scope (header-only NVTX: free unless a profiler is attached), so that a
// timeline shows each call and each ring step; ncu can select kernels by them (--nvtx).
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    NvtxRange(const char* fmt, int i) {
        char buf[64];
        snprintf(buf, sizeof buf, fmt, i);
        nvtxRangePushA(buf);
    }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

constexpr size_t kHeader = 256;   // DevStatus

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---- descriptor validation ---------------------------------------------------
bpa_status make_problem(const bpa_attn_desc* d, Problem& P, bool need_qkv) {
    if (!d) return fail(BPA_ERR_INVALID_ARG, "desc is NULL");
    const size_t v1_size = offsetof(bpa_attn_desc, dv);          // version 1: no dv, o_strides
    const size_t v2_size = offsetof(bpa_attn_desc, seqlens_q);   // version 2: no sequence lengths
    const size_t v3_size = offsetof(bpa_attn_desc, sink);        // version 3: no sink
    const size_t v4_size = offsetof(bpa_attn_desc, deterministic);   // version 4: no determinism knob
    const size_t v5_size = offsetof(bpa_attn_desc, dropout_threshold);   // version 5: no dropout
    if (d->struct_size != sizeof(bpa_attn_desc) && d->struct_size != v1_size && d->struct_size != v2_size &&
        d->struct_size != v3_size && d->struct_size != v4_size && d->struct_size != v5_size)
        return fail(BPA_ERR_INVALID_ARG, "desc->struct_size is %u, expected %zu (or %zu, %zu, %zu, %zu, %zu)",
                    d->struct_size, sizeof(bpa_attn_desc), v5_size, v4_size, v3_size, v2_size, v1_size);
    const bool v2 = d->struct_size >= v2_size;
    const bool v3 = d->struct_size >= v3_size;
    const bool v4 = d->struct_size >= v4_size;
    const bool v5 = d->struct_size >= v5_size;
    const bool v6 = d->struct_size == sizeof(bpa_attn_desc);
    const bool varlen = v3 && (d->seqlens_q || d->seqlens_kv);
    if (d->dtype != BPA_BF16 && d->dtype != BPA_FP32)
        return fail(BPA_ERR_INVALID_ARG, "unknown dtype %d", d->dtype);
    if (d->B < 1 || d->S < 1 || d->Hq < 1 || d->Hkv < 1 || d->d < 1)
        return fail(BPA_ERR_INVALID_ARG, "B, S, Hq, Hkv, d must be >= 1");
    if (d->Hq % d->Hkv)
        return fail(BPA_ERR_INVALID_ARG, "Hq (%d) must be a multiple of Hkv (%d)", d->Hq, d->Hkv);
    if (d->d > 512) return fail(BPA_ERR_UNSUPPORTED, "head dim %d > 512", d->d);
    const int dv = v2 && d->dv ? d->dv : d->d;
    if (dv < 1) return fail(BPA_ERR_INVALID_ARG, "dv must be >= 1 (or 0 for d)");
    if (dv > 512) return fail(BPA_ERR_UNSUPPORTED, "value head dim %d > 512", dv);
    const bool own_os = v2 && (d->o_strides[0] | d->o_strides[1] | d->o_strides[2]) != 0;
    if (need_qkv && (!d->q || !d->k || !d->v)) return fail(BPA_ERR_INVALID_ARG, "q, k or v is NULL");
    if (d->window_left < -1 || d->window_right < -1)
        return fail(BPA_ERR_INVALID_ARG, "window bounds must be >= -1");
    const int n = d->ring_size;
    if (n < 1 || d->S % n) return fail(BPA_ERR_INVALID_ARG, "ring_size %d must divide S = %d", n, d->S);
    const int blk = d->S / n;
    if (d->query_chunk < 0 || d->key_chunk < 0 || (d->query_chunk && blk % d->query_chunk) ||
        (d->key_chunk && blk % d->key_chunk))
        return fail(BPA_ERR_INVALID_ARG, "query_chunk (%d) / key_chunk (%d) must divide S / ring_size = %d",
                    d->query_chunk, d->key_chunk, blk);
    for (int i = 0; i < 3; ++i)
        if (d->q_strides[i] < 0 || d->k_strides[i] < 0 || d->v_strides[i] < 0 || (own_os && d->o_strides[i] < 0))
            return fail(BPA_ERR_INVALID_ARG, "strides must be non-negative");
    if (d->bias)
        for (int i = 0; i < 4; ++i)
            if (d->bias_strides[i] < 0) return fail(BPA_ERR_INVALID_ARG, "bias strides must be >= 0");
    if (d->block_idx) {
        if (d->sel_block < 1 || d->S % d->sel_block)
            return fail(BPA_ERR_INVALID_ARG, "sel_block (%d) must divide S", d->sel_block);
        if (d->top_n < 1 || d->top_n > 64) return fail(BPA_ERR_INVALID_ARG, "top_n must be in [1, 64]");
        if (d->local_window < 0) return fail(BPA_ERR_INVALID_ARG, "local_window must be >= 0");
        if (n != 1) return fail(BPA_ERR_INVALID_ARG, "block-selected mode needs ring_size 1");
    }
    if (varlen && (n != 1 || d->block_idx))
        return fail(BPA_ERR_INVALID_ARG, "sequence lengths need ring_size 1 and no block selection");
    if (v4 && d->sink && n != 1) return fail(BPA_ERR_INVALID_ARG, "sink attention needs ring_size 1");
    if (v4 && d->dsink && !d->sink) return fail(BPA_ERR_INVALID_ARG, "dsink needs a sink");
    if (v5 && d->deterministic && n != 1) return fail(BPA_ERR_INVALID_ARG, "deterministic mode needs ring_size 1");
    if (v6 && d->dropout_reserved) return fail(BPA_ERR_INVALID_ARG, "dropout_reserved must be 0");
    P.B = d->B;
    P.S = d->S;
    P.Hq = d->Hq;
    P.Hkv = d->Hkv;
    P.G = d->Hq / d->Hkv;
    P.d = d->d;
    P.dv = dv;
    P.dtype = d->dtype;
    P.scale = d->scale > 0.f ? d->scale : 1.f / sqrtf(static_cast<float>(d->d));
    P.causal = d->causal != 0;
    P.wl = d->window_left;
    P.wr = d->window_right;
    P.q = d->q;
    P.k = d->k;
    P.v = d->v;
    for (int i = 0; i < 3; ++i) {
        P.qs[i] = d->q_strides[i];
        P.ks[i] = d->k_strides[i];
        P.vs[i] = d->v_strides[i];
        P.os[i] = own_os ? d->o_strides[i] : d->q_strides[i];
    }
    P.bias = d->bias;
    for (int i = 0; i < 4; ++i) P.bs[i] = d->bias ? d->bias_strides[i] : 0;
    P.ring_n = n;
    P.ring_blk = blk;
    P.block_idx = d->block_idx;
    P.seqlens_q = varlen ? d->seqlens_q : nullptr;
    P.seqlens_kv = varlen ? d->seqlens_kv : nullptr;
    P.bottom_right = v3 && d->bottom_right ? 1 : 0;
    P.sink = v4 ? d->sink : nullptr;
    P.dsink = v4 ? d->dsink : nullptr;
    P.det = v5 && d->deterministic ? 1 : 0;
    P.drop_thr = v6 ? d->dropout_threshold : 0u;
    P.drop_k0 = v6 ? static_cast<uint32_t>(d->dropout_seed) : 0u;
    P.drop_k1 = v6 ? static_cast<uint32_t>(d->dropout_seed >> 32) : 0u;
    P.sel_block = d->block_idx ? d->sel_block : 0;
    P.top_n = d->block_idx ? d->top_n : 0;
    P.local_window = d->block_idx ? d->local_window : 0;
    return BPA_OK;
}

// ---- workspace layout ------------------------------------------------------------
struct FwdLayout {
    size_t acc, total;
};
FwdLayout fwd_layout(const Problem& P) {
    FwdLayout L;
    L.acc = kHeader;
    size_t acc_bytes = P.ring_n > 1 ? round256(sizeof(float) * P.B * static_cast<size_t>(P.S) * P.Hq * P.dv) : 0;
    L.total = L.acc + acc_bytes;
    return L;
}

struct BwdLayout {
    int Spad;
    size_t D, lse, dq, dk, dv, total;
};
BwdLayout bwd_layout(const Problem& P) {
    BwdLayout L;
    L.Spad = (P.S + 63) / 64 * 64;
    const size_t rows = static_cast<size_t>(P.B) * P.Hq * L.Spad;
    L.D = kHeader;
    L.lse = L.D + round256(rows * sizeof(float));
    L.dq = L.lse + round256(rows * sizeof(float));
    // dQ accumulator [B, Hq, Spad / 4, d, 4]: four consecutive queries of one channel side by side;
    // deterministic mode: one per 128-key tile
    const size_t nkt = P.det ? (P.S + 127) / 128 : 1;
    const size_t nq = sizeof(float) * P.B * static_cast<size_t>(L.Spad) * P.Hq * P.d * nkt;
    const size_t nk = sizeof(float) * P.B * static_cast<size_t>(P.S) * P.Hkv * P.d;
    const size_t nv = sizeof(float) * P.B * static_cast<size_t>(P.S) * P.Hkv * P.dv;
    L.dk = L.dq + round256(nq);
    // float32 dK / dV: the ring's travelling carries, or the block-selected backward's accumulators
    const bool kv_acc = P.ring_n > 1 || P.block_idx;
    L.dv = L.dk + (kv_acc ? round256(nk) : 0);
    L.total = L.dv + (kv_acc ? round256(nv) : 0);
    return L;
}

bpa_status check_ws(void* ws, size_t have, size_t need) {
    if (!ws) return fail(BPA_ERR_WORKSPACE, "workspace is NULL (need %zu bytes)", need);
    if (reinterpret_cast<uintptr_t>(ws) & 255u) return fail(BPA_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    if (have < need) return fail(BPA_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", have, need);
    return BPA_OK;
}

// ---- TMA descriptors ----------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// BSHD bf16 tensor as a 4-D map (d, H, S, B); box = 64 channels x `rows` positions, 128-byte swizzle.
bool make_map(CUtensorMap* map, const void* base, int d, int H, int S, int B, const int64_t st[3], int rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(S),
                          static_cast<cuuint64_t>(B)};
    // a dimension of extent 1 never steps: give it any legal stride
    auto fix = [](int64_t s, int extent, int64_t fallback) { return extent == 1 ? fallback : s; };
    const int64_t sh = fix(st[2], H, d);
    const int64_t ss = fix(st[1], S, static_cast<int64_t>(d) * H);
    const int64_t sb = fix(st[0], B, static_cast<int64_t>(d) * H * S);
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(sh * 2), static_cast<cuuint64_t>(ss * 2),
                             static_cast<cuuint64_t>(sb * 2)};
    cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(rows), 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// The tensor-core kernels read through TMA: 16-byte aligned bases, strides in
// multiples of 8 elements.
bool tma_layout_ok(const Problem& P) {
    if (!aligned16(P.q) || !aligned16(P.k) || !aligned16(P.v)) return false;
    for (int i = 0; i < 3; ++i)
        if ((P.qs[i] | P.ks[i] | P.vs[i] | P.os[i]) & 7) return false;
    return true;
}

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

}  // namespace

namespace bpa {

bpa_status check_select_args(const void* q, const void* k, int32_t dtype, int32_t B, int32_t S, int32_t H,
                             int32_t d, const int64_t q_strides[3], const int64_t k_strides[3],
                             int32_t block_size, int32_t top_n, const int32_t* block_idx_out) {
    if (!q || !k || !q_strides || !k_strides || !block_idx_out)
        return fail(BPA_ERR_INVALID_ARG, "q, k, strides or block_idx_out is NULL");
    if (dtype != BPA_BF16 && dtype != BPA_FP32) return fail(BPA_ERR_INVALID_ARG, "unknown dtype %d", dtype);
    if (B < 1 || S < 1 || H < 1 || d < 1) return fail(BPA_ERR_INVALID_ARG, "B, S, H, d must be >= 1");
    if (d > 512) return fail(BPA_ERR_UNSUPPORTED, "head dim %d > 512", d);
    if (block_size < 1 || S % block_size)
        return fail(BPA_ERR_INVALID_ARG, "block_size (%d) must divide S (%d)", block_size, S);
    if (S / block_size > kSelectMaxBlocks)
        return fail(BPA_ERR_UNSUPPORTED, "%d blocks per sequence, more than %d", S / block_size, kSelectMaxBlocks);
    if (top_n < 1 || top_n > 64) return fail(BPA_ERR_INVALID_ARG, "top_n must be in [1, 64]");
    for (int i = 0; i < 3; ++i)
        if (q_strides[i] < 0 || k_strides[i] < 0) return fail(BPA_ERR_INVALID_ARG, "strides must be >= 0");
    return BPA_OK;
}

// Lets other translation units of the library report an error through bpa_last_error.
void set_last_error(const char* msg) { snprintf(g_last_error, sizeof g_last_error, "%s", msg); }
}  // namespace bpa

extern "C" {

int32_t bpa_version(void) { return BPA_VERSION; }

const char* bpa_last_error(void) { return g_last_error; }

const char* bpa_status_string(bpa_status st) {
    switch (st) {
        case BPA_OK: return "BPA_OK";
        case BPA_ERR_INVALID_ARG: return "BPA_ERR_INVALID_ARG";
        case BPA_ERR_UNSUPPORTED: return "BPA_ERR_UNSUPPORTED";
        case BPA_ERR_WORKSPACE: return "BPA_ERR_WORKSPACE";
        case BPA_ERR_CUDA: return "BPA_ERR_CUDA";
        case BPA_ERR_TIMEOUT: return "BPA_ERR_TIMEOUT";
        case BPA_ERR_DEVICE_CHECK: return "BPA_ERR_DEVICE_CHECK";
    }
    return "unknown bpa_status";
}

size_t bpa_workspace_size(int32_t op, const bpa_attn_desc* desc) {
    Problem P;
    if (make_problem(desc, P, false) != BPA_OK) return 0;
    if (op == BPA_OP_FWD) return fwd_layout(P).total;
    if (op == BPA_OP_BWD) return bwd_layout(P).total;
    fail(BPA_ERR_INVALID_ARG, "unknown op %d", op);
    return 0;
}

bpa_status bpa_fwd(const bpa_attn_desc* desc, void* o, float* m, float* l, void* workspace,
                   size_t workspace_bytes, void* stream) {
    const NvtxRange range("bpa_fwd");
    Problem P;
    bpa_status st = make_problem(desc, P, true);
    if (st != BPA_OK) return st;
    if (!o || !m || !l) return fail(BPA_ERR_INVALID_ARG, "o, m or l is NULL");
    const int n = P.ring_n;
    const int begin = desc->ring_step_begin, end = desc->ring_step_end ? desc->ring_step_end : n;
    if (begin < 0 || end > n || begin >= end)
        return fail(BPA_ERR_INVALID_ARG, "ring steps [%d, %d) outside [0, %d)", begin, end, n);
    const FwdLayout L = fwd_layout(P);
    if ((st = check_ws(workspace, workspace_bytes, L.total)) != BPA_OK) return st;
    cudaStream_t s = as_stream(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const PhaseMarks marks;
    cudaError_t e = cudaMemsetAsync(ws, 0, kHeader, s);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the status word");
    marks.mark(0, s);

    FwdArgs a;
    memset(&a, 0, sizeof a);
    a.P = P;
    a.o = o;
    a.m = m;
    a.l = l;
    a.status = reinterpret_cast<uint32_t*>(ws);
    // work-item counters of the tensor-core forward: words 2..63 of the (cleared) status
    // header, one per launch; a word is cleared again before it is reused
    uint32_t* counters = a.status + 2;
    constexpr int kCounters = static_cast<int>(kHeader / 4) - 2;
    a.sched = counters;

    if (P.block_idx) {
        // entries outside the contract are ignored by the kernels and reported in the status word
        if ((e = launch_check_blocks(P, a.status, s)) != cudaSuccess) return cuda_fail(e, "block index check");
        e = gather_supported(P) ? launch_gather_fwd(a, s) : launch_fwd_simt(a, s);
        marks.mark(1, s);
        marks.mark(2, s);
        return e == cudaSuccess ? BPA_OK : cuda_fail(e, "block-selected forward launch");
    }

    bool tc = fwd_tc_supported(P) && tma_layout_ok(P) && aligned16(o);
    CUtensorMap maps[3];
    if (tc) {
        tc = make_map(&maps[0], P.q, P.d, P.Hq, P.S, P.B, P.qs, 128) &&
             make_map(&maps[1], P.k, P.d, P.Hkv, P.S, P.B, P.ks, 128) &&
             make_map(&maps[2], P.v, P.dv, P.Hkv, P.S, P.B, P.vs, 128);
    }
    if (n == 1) {
        e = tc ? launch_fwd_tc(a, maps, s) : launch_fwd_simt(a, s);
        if (e == cudaSuccess && P.sink && (P.seqlens_q || P.seqlens_kv)) e = launch_pad_stats(a, s);
        marks.mark(1, s);
        marks.mark(2, s);
        return e == cudaSuccess ? BPA_OK : cuda_fail(e, "forward launch");
    }
    a.acc = reinterpret_cast<float*>(ws + L.acc);
    if (begin == 0 && (e = launch_ring_init(a, s)) != cudaSuccess) return cuda_fail(e, "ring carry init");
    for (int idx = begin; idx < end; ++idx) {
        const NvtxRange step("bpa_fwd ring step %d", idx);
        a.ring_idx = idx;
        const int li = idx - begin;
        a.sched = counters + li % kCounters;
        if (tc && li >= kCounters && (e = cudaMemsetAsync(a.sched, 0, sizeof(uint32_t), s)) != cudaSuccess)
            return cuda_fail(e, "clearing a work counter");
        e = tc ? launch_fwd_tc(a, maps, s) : launch_fwd_simt(a, s);
        if (e != cudaSuccess) return cuda_fail(e, "ring step launch");
    }
    marks.mark(1, s);
    if (end == n && (e = launch_ring_finalize(a, s)) != cudaSuccess) return cuda_fail(e, "ring finalize");
    marks.mark(2, s);
    return BPA_OK;
}

// SMs of the current device (cached per device; 1 if it cannot be read)
static int sm_count_current() {
    static int cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1) return 1;
    if (dev >= 0 && dev < 64) cached[dev] = sms;
    return sms;
}

bpa_status bpa_bwd(const bpa_attn_desc* desc, const void* o, const void* dout, const float* m, const float* l,
                   void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, void* stream) {
    const NvtxRange range("bpa_bwd");
    Problem P;
    bpa_status st = make_problem(desc, P, true);
    if (st != BPA_OK) return st;
    if (!o || !dout || !m || !l || !dq || !dk || !dv)
        return fail(BPA_ERR_INVALID_ARG, "o, dout, m, l, dq, dk or dv is NULL");
    const int n = P.ring_n;
    const int begin = desc->ring_step_begin, end = desc->ring_step_end ? desc->ring_step_end : n;
    if (begin != 0 || end != n)
        return fail(BPA_ERR_INVALID_ARG, "backward runs the whole ring sweep: steps must be [0, %d)", n);
    const BwdLayout L = bwd_layout(P);
    if ((st = check_ws(workspace, workspace_bytes, L.total)) != BPA_OK) return st;
    cudaStream_t s = as_stream(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const PhaseMarks marks;
    cudaError_t e = cudaMemsetAsync(ws, 0, kHeader, s);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the status word");
    marks.mark(0, s);

    BwdArgs a;
    memset(&a, 0, sizeof a);
    a.P = P;
    a.o = o;
    a.dout = dout;
    a.m = m;
    a.l = l;
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.Dvec = reinterpret_cast<float*>(ws + L.D);
    a.lse = reinterpret_cast<float*>(ws + L.lse);
    a.Spad = L.Spad;
    a.status = reinterpret_cast<uint32_t*>(ws);
    if (P.block_idx && (e = launch_check_blocks(P, a.status, s)) != cudaSuccess)
        return cuda_fail(e, "block index check");

    if (P.block_idx && !P.det && gather_supported(P) && aligned16(dout) && aligned16(dq) && aligned16(dk) && aligned16(dv)) {
        // gathered backward: dQ written per query block, dK / dV reduced into float32 accumulators
        a.dk_acc = reinterpret_cast<float*>(ws + L.dk);
        a.dv_acc = reinterpret_cast<float*>(ws + L.dv);
        if ((e = launch_bwd_pre(a, s)) != cudaSuccess || (P.dsink && (e = launch_sink_grad(a, s)) != cudaSuccess))
            return cuda_fail(e, "backward pre-pass");
        marks.mark(1, s);
        const size_t nk = sizeof(float) * P.B * static_cast<size_t>(P.S) * P.Hkv * P.d;
        const size_t nv = sizeof(float) * P.B * static_cast<size_t>(P.S) * P.Hkv * P.dv;
        if ((e = cudaMemsetAsync(a.dk_acc, 0, nk, s)) != cudaSuccess ||
            (e = cudaMemsetAsync(a.dv_acc, 0, nv, s)) != cudaSuccess)
            return cuda_fail(e, "clearing the dK / dV accumulators");
        if ((e = launch_gather_bwd(a, s)) != cudaSuccess) return cuda_fail(e, "block-selected backward launch");
        marks.mark(2, s);
        e = launch_cast_dkdv(a, s);
        marks.mark(3, s);
        return e == cudaSuccess ? BPA_OK : cuda_fail(e, "dK / dV cast");
    }
    // other block-selected problems run on the CUDA-core kernels, which visit only the selected blocks
    bool tc = !P.block_idx && bwd_tc_supported(P) && tma_layout_ok(P) && aligned16(o) && aligned16(dout) &&
              aligned16(dq) && aligned16(dk) && aligned16(dv);
    CUtensorMap maps[4];
    if (tc) {
        tc = make_map(&maps[0], P.q, P.d, P.Hq, P.S, P.B, P.qs, 64) &&
             make_map(&maps[1], P.k, P.d, P.Hkv, P.S, P.B, P.ks, 128) &&
             make_map(&maps[2], P.v, P.dv, P.Hkv, P.S, P.B, P.vs, 128) &&
             make_map(&maps[3], dout, P.dv, P.Hq, P.S, P.B, P.os, 64);
    }
    if (!tc) {
        if ((e = launch_bwd_pre(a, s)) != cudaSuccess || (P.dsink && (e = launch_sink_grad(a, s)) != cudaSuccess))
            return cuda_fail(e, "backward pre-pass");
        marks.mark(1, s);
        e = launch_bwd_simt(a, s);
        marks.mark(2, s);
        marks.mark(3, s);
        return e == cudaSuccess ? BPA_OK : cuda_fail(e, "backward launch");
    }
    // With contiguous, 16-byte aligned dk / dv the q heads of a group are split over two CTAs
    // per key tile, which add their dK, dV halves into dk, dv (zeroed by the pre-pass): exactly
    // two contributions per element, so the result does not depend on their order.
    const bool kv_dense = P.ks[2] == P.d && P.ks[1] == static_cast<int64_t>(P.Hkv) * P.d &&
                          P.ks[0] == static_cast<int64_t>(P.S) * P.Hkv * P.d && P.vs[2] == P.dv &&
                          P.vs[1] == static_cast<int64_t>(P.Hkv) * P.dv &&
                          P.vs[0] == static_cast<int64_t>(P.S) * P.Hkv * P.dv &&
                          ((reinterpret_cast<uintptr_t>(dk) | reinterpret_cast<uintptr_t>(dv)) & 15u) == 0;
    // ... and only where the halves fill the last wave better: ceil(2 c / sms) < 2 ceil(c / sms)
    // for c key-tile CTAs (measured: at B 1 of the sliding-window workload, 256 CTAs in two
    // waves either way, the split cost 8 %)
    const int sms = sm_count_current();
    const int64_t ctas = static_cast<int64_t>((P.S + 127) / 128) * P.Hkv * P.B;
    const bool fills = (2 * ctas + sms - 1) / sms < 2 * ((ctas + sms - 1) / sms);
    const int split_kv = kv_dense && fills && P.G % 2 == 0 && P.d % 8 == 0 && P.dv % 8 == 0 ? 2 : 1;
    if (n == 1 && bwd_band_supported(P)) {
        // band: the pre-pass zeroes dq, the main kernel adds dQ into it directly (dK, dV split
        // as below)
        a.dq_direct = 1;
        a.hsplit = split_kv;
        if ((e = launch_bwd_pre(a, s)) != cudaSuccess) return cuda_fail(e, "backward pre-pass");
        marks.mark(1, s);
        if ((e = launch_bwd_tc_band(a, maps, s)) != cudaSuccess) return cuda_fail(e, "backward launch");
        marks.mark(2, s);
        marks.mark(3, s);
        return BPA_OK;
    }
    a.dq_acc = reinterpret_cast<float*>(ws + L.dq);
    // (measured: with four q heads per group the half-length CTAs lost 8 %, with sixteen they
    // gained 4 %; the ring steps carry dK, dV in float32 instead)
    a.hsplit = n == 1 && P.G >= 8 ? split_kv : 1;
    if ((e = launch_bwd_pre(a, s)) != cudaSuccess || (P.dsink && (e = launch_sink_grad(a, s)) != cudaSuccess))
            return cuda_fail(e, "backward pre-pass");
    marks.mark(1, s);
    if (n == 1) {
        if ((e = launch_bwd_tc(a, maps, s)) != cudaSuccess) return cuda_fail(e, "backward launch");
    } else {
        a.dk_acc = reinterpret_cast<float*>(ws + L.dk);
        a.dv_acc = reinterpret_cast<float*>(ws + L.dv);
        const size_t nk = sizeof(float) * P.B * static_cast<size_t>(P.S) * P.Hkv * P.d;
        const size_t nv = sizeof(float) * P.B * static_cast<size_t>(P.S) * P.Hkv * P.dv;
        if ((e = cudaMemsetAsync(a.dk_acc, 0, nk, s)) != cudaSuccess ||
            (e = cudaMemsetAsync(a.dv_acc, 0, nv, s)) != cudaSuccess)
            return cuda_fail(e, "clearing the dK / dV carries");
        for (int idx = 0; idx < n; ++idx) {
            const NvtxRange step("bpa_bwd ring step %d", idx);
            a.ring_idx = idx;
            if ((e = launch_bwd_tc(a, maps, s)) != cudaSuccess) return cuda_fail(e, "ring backward step");
        }
    }
    marks.mark(2, s);
    e = P.det ? launch_dq_reduce(a, s) : launch_bwd_post(a, s);
    marks.mark(3, s);
    return e == cudaSuccess ? BPA_OK : cuda_fail(e, "backward post-pass");
}

size_t bpa_select_workspace_size(int32_t B, int32_t S, int32_t H, int32_t d, int32_t block_size) {
    if (B < 1 || S < 1 || H < 1 || d < 1 || block_size < 1 || S % block_size) return 0;
    const size_t sums = sizeof(double) * static_cast<size_t>(B) * H * (S / block_size) * d;
    return kHeader + 2 * round256(sums) + round256(sums / 2);
}

bpa_status bpa_select_blocks(const void* q, const void* k, int32_t dtype, int32_t B, int32_t S, int32_t H,
                             int32_t d, const int64_t q_strides[3], const int64_t k_strides[3],
                             int32_t block_size, int32_t top_n, int32_t* block_idx_out, void* workspace,
                             size_t workspace_bytes, void* stream) {
    bpa_status st = bpa::check_select_args(q, k, dtype, B, S, H, d, q_strides, k_strides, block_size, top_n,
                                           block_idx_out);
    if (st != BPA_OK) return st;
    const size_t need = bpa_select_workspace_size(B, S, H, d, block_size);
    st = check_ws(workspace, workspace_bytes, need);
    if (st != BPA_OK) return st;
    cudaStream_t s = as_stream(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    cudaError_t e = cudaMemsetAsync(ws, 0, kHeader, s);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the status word");
    SelectArgs a;
    memset(&a, 0, sizeof a);
    a.q = q;
    a.k = k;
    a.dtype = dtype;
    a.B = B;
    a.S = S;
    a.H = H;
    a.d = d;
    for (int i = 0; i < 3; ++i) {
        a.qs[i] = q_strides[i];
        a.ks[i] = k_strides[i];
    }
    a.block = block_size;
    a.top_n = top_n;
    a.out = block_idx_out;
    const size_t sums = sizeof(double) * static_cast<size_t>(B) * H * (S / block_size) * d;
    a.qsum = reinterpret_cast<double*>(ws + kHeader);
    a.ksum = reinterpret_cast<double*>(ws + kHeader + round256(sums));
    a.kt32 = reinterpret_cast<float*>(ws + kHeader + 2 * round256(sums));
    a.status = reinterpret_cast<uint32_t*>(ws);
    e = launch_select(a, s);
    return e == cudaSuccess ? BPA_OK : cuda_fail(e, "block selection launch");
}

bpa_status bpa_check(const void* workspace) {
    if (!workspace) return fail(BPA_ERR_INVALID_ARG, "workspace is NULL");
    DevStatus h;
    cudaError_t e = cudaMemcpy(&h, workspace, sizeof h, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "reading the status word");
    if (h.flags & ST_TIMEOUT) return fail(BPA_ERR_TIMEOUT, "a kernel wait gave up (site 0x%x)", h.where);
    if (h.flags & ST_CHECK) return fail(BPA_ERR_DEVICE_CHECK, "a device-side check failed (site 0x%x)", h.where);
    return BPA_OK;
}

void bpa_set_phase_events(void* const* events, int32_t n) {
    g_phase_n = 0;
    if (!events || n <= 0) return;
    if (n > 8) n = 8;
    for (int i = 0; i < n; ++i) g_phase_events[i] = static_cast<cudaEvent_t>(events[i]);
    g_phase_n = n;
}

// Diagnostic: launches one CTA whose bounded wait can never complete, so that
// the timeout path (status word, clean return) can be exercised on a GPU
// without hanging it.  limit_ns bounds the wait.
bpa_status bpa_debug_wait_timeout(void* workspace, size_t workspace_bytes, uint64_t limit_ns, void* stream) {
    bpa_status st = check_ws(workspace, workspace_bytes, kHeader);
    if (st != BPA_OK) return st;
    if (limit_ns == 0 || limit_ns > 5000000000ull) return fail(BPA_ERR_INVALID_ARG, "limit_ns must be in (0, 5e9]");
    cudaStream_t s = as_stream(stream);
    cudaError_t e = cudaMemsetAsync(workspace, 0, kHeader, s);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the status word");
    e = launch_wait_selftest(static_cast<uint32_t*>(workspace), limit_ns, s);
    return e == cudaSuccess ? BPA_OK : cuda_fail(e, "self-test launch");
}

}  // extern "C"
