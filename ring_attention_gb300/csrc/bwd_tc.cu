// bwd_tc.cu - blockwise attention backward on the 5th-generation tensor cores (bf16, d = 128).
//
// Recomputes the scores of every allowed (query tile, key tile) pair from
// the saved row statistics and accumulates the gradients ("bpt.py",
// _blockwise_attention_bwd / scan_kv_block):
//     P = exp(S - lse),  dP = dO V^T,  dS = P (dP - D),
//     dV += P^T dO,  dK += scale dS^T Q,  dQ += scale dS K
// One CTA owns one 128-key tile of one (batch, kv head) and walks every q
// head of the group and every 64-row query tile the mask allows, so dK and
// dV accumulate in TMEM for the whole group with no atomics; dQ partial
// tiles are added to a float32 accumulator in global memory.
// The scores are computed transposed (S^T = K Q^T, keys on the TMEM lanes),
// so that P^T and dS^T come out of the softmax warps already laid out as the
// A operands of the dV and dK products.
// TMEM (512 columns): S^T [0,64), dP^T x2 [64,192), dQ^T [192,256),
// dK [256,384), dV [384,512).  dP^T is double-buffered so that S^T and dP^T
// of tile it are computed while the softmax warps still work on tile it-1.
// Two softmax warpgroups split the 64 query columns of a tile (32 each).
// Once a warpgroup has read its 32 dP^T columns, it writes there its P^T
// (16 columns of bf16 pairs) and dS^T (16 columns), the TMEM A operands of
// the dV and dK products; dS^T also goes to shared memory, where it is the
// B operand of dQ^T.  The same warpgroup then drains its 32 columns of the
// previous tile's dQ^T (channels on the lanes) straight into a float32
// accumulator with coalesced 16-byte reductions.  The accumulator of one
// (batch, q head) is laid out [S'/4][128 channels][4 queries] (S' = S rounded
// up to 64), so a warp's reduction covers 512 contiguous bytes.
// Consecutive products into one TMEM accumulator wait on each other, so the
// independent S^T and dP^T products are issued interleaved (as are dV, dK).
// Roles (352 threads):
//   warps 0-3  query columns 0-31 of each tile, warps 4-7 columns 32-63;
//              thread (warp % 4) * 32 + lane owns key row / dQ channel of that TMEM lane;
//              at the end warps 0-3 write dK (scaled), warps 4-7 dV;
//   warp 8     TMA producer: K, V once; Q, dO (+ lse, D) per query tile;
//   warp 9     MMA issuer A: S^T and dP^T products; TMEM owner;
//   warp 10    MMA issuer B: dV, dK and dQ^T products.  Two issuers halve the per-thread
//              issue and wait chain; their shared resources are handed over by barriers
//              (a dP^T buffer returns to A once B's dV / dK have read its pairs; a Q / dO
//              stage is released by a commit from each).  Each issuer is a whole warp
//              running the loop with warp-uniform operands, one elected lane issuing.
#include <math.h>

#include <algorithm>

#include "bpa_internal.h"
#include "common.cuh"

namespace bpa {
namespace {

constexpr int D = 128;        // head dim
constexpr int BK = 128;       // keys per CTA
constexpr int BQ = 64;        // queries per tile
constexpr int NS = 4;         // Q / dO stages.  Measured: a second dS^T buffer (so that the softmax
                              // warps may write tile it while dQ^T(it - 1) still reads the other)
                              // made the backward slower, 8 % on the GQA causal workload (with three
                              // stages to make room) and 12 % on the MLA one (four stages)
constexpr int kThreads = 352;
constexpr int kSoftmax = 256;    // threads of the two softmax warpgroups

constexpr int SUBK = BK * 128;    // one 64-channel slab of the key tile
constexpr int SUBQ = BQ * 128;    // one 64-channel slab of a query tile
constexpr int OFF_K = 0;
// Shared-memory layout for value head dim DV (128, or 64 with q, k of 128: separate
// value head dims); V tiles and dO stages hold DV channels.
template <int DV>
struct BwdCfg {
    static constexpr int OFF_V = OFF_K + BK * D * 2;
    static constexpr int OFF_Q = OFF_V + BK * DV * 2;
    static constexpr int OFF_DO = OFF_Q + NS * BQ * D * 2;
    static constexpr int OFF_DS = OFF_DO + NS * BQ * DV * 2;   // dS^T [128 keys][64 q] bf16
    static constexpr int OFF_ST = OFF_DS + BK * BQ * 2;        // per stage: lse[64], D[64] float
    static constexpr int OFF_BAR = OFF_ST + NS * 512;
    static constexpr int SMEM = OFF_BAR + 256 + 1024;
    static constexpr int DO_BYTES = BQ * DV * 2;               // one dO stage
    static constexpr uint32_t IDESC_V = idesc_bf16_f32(BK, DV, 0, 1);   // dV: A from TMEM, B MN-major
    static_assert(SMEM <= 232448, "shared memory");
};

// barrier slots
constexpr int B_KV = 0, B_QF = 1, B_QE = 1 + NS, B_S = 1 + 2 * NS, B_SF = 2 + 2 * NS, B_DP = 3 + 2 * NS,
              B_DS = 5 + 2 * NS, B_DQF = 6 + 2 * NS, B_DQE = 7 + 2 * NS, B_PF = 8 + 2 * NS, B_KVD = 9 + 2 * NS,
              B_FIN = 10 + 2 * NS, B_PRF = 11 + 2 * NS /* x2 */, B_FINB = 13 + 2 * NS, NBAR = 14 + 2 * NS;
static_assert(8 * NBAR + 8 <= 256, "barrier area");

constexpr uint32_t IDESC_S = idesc_bf16_f32(BK, BQ, 0, 0);     // S^T, dP^T: both K-major
constexpr uint32_t IDESC_KV = idesc_bf16_f32(BK, D, 0, 1);     // dK: A from TMEM, B MN-major
constexpr uint32_t IDESC_Q = idesc_bf16_f32(D, BQ, 1, 1);      // dQ^T: both MN-major

struct Work {
    int b, hkv, k0;
    int q_lo, q_hi;      // query rows that may see this key tile (ring block included)
    int qt_lo, n_qt, n_it;
    int lk, off;         // valid keys of the batch entry, offset of the causal / window diagonal
    int g0, gn;          // q heads of the group this CTA walks: g0 .. g0 + gn - 1
};

// The work of key tile kt of (batch b, kv head hkv): the query rows that may see it.
__device__ __forceinline__ Work decode_tile_of(const BwdArgs& a, int b, int hkv, int kt) {
    const Problem& P = a.P;
    Work w;
    w.b = b;
    w.hkv = hkv;
    w.k0 = kt * BK;
    const Lens len = lens_of(P, w.b);   // full lengths unless the problem has sequence lengths
    w.lk = len.lk;
    w.off = len.off;
    const int k_last = min(w.k0 + BK - 1, len.lk - 1);
    int lo = 0, hi = w.k0 < len.lk ? len.lq - 1 : -1;
    if (a.dk_acc) {   // ring step: the query block that meets this key block now
        const int j = w.k0 / P.ring_blk;
        const int iq = (j + a.ring_idx) % P.ring_n;
        lo = iq * P.ring_blk;
        hi = lo + P.ring_blk - 1;
    }
    if (P.causal) lo = max(lo, w.k0 - w.off);
    if (P.wr >= 0) lo = max(lo, w.k0 - w.off - P.wr);
    if (P.wl >= 0) hi = min(hi, k_last - w.off + P.wl);
    w.q_lo = lo;
    w.q_hi = hi;
    w.qt_lo = lo / BQ;
    w.n_qt = lo <= hi ? hi / BQ - w.qt_lo + 1 : 0;
    w.g0 = 0;
    w.gn = P.G;
    w.n_it = w.n_qt * P.G;
    return w;
}

// Launch order: the lowest key tiles (most causal work) first, all (batch, kv head) groups
// interleaved.  Measured alternative: chunks of 4 or 8 groups at a time keep a group's Q / dO
// tiles and dQ accumulator rows in L2 (DRAM traffic 953 -> 426 / 534 MB per launch on the GQA
// causal workload) but balance the causal work worse (+5 % / +1.5 % time); the kernel is
// tensor-bound, so the interleaved order stays.
// With a head split, CTA pairs (2 r, 2 r + 1) share key tile r and take one half of the group's
// q heads each (the band backward: shorter, equal CTAs fill the last wave better).
__device__ __forceinline__ Work decode(const BwdArgs& a) {
    const Problem& P = a.P;
    const int hs = a.hsplit > 1 ? 2 : 1;
    int r = blockIdx.x / hs;
    const int half = blockIdx.x % hs;
    const int b = r % P.B;
    r /= P.B;
    const int hkv = r % P.Hkv;
    const int kt = r / P.Hkv;
    Work w = decode_tile_of(a, b, hkv, kt);
    w.gn = P.G / hs;
    w.g0 = half * w.gn;
    w.n_it = w.n_qt * w.gn;
    return w;
}

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint32_t* status) {
    int never = 0;
    mbar_wait(bar, parity, &never, status, 0xD1);
}

// DET: deterministic dQ slices; DROP: attention dropout; DQBF: the band backward's dQ added
// in bf16 pairs straight into dq.  Each is a separate instantiation, so that the default
// kernel's code stays as it is without the knobs.
template <int DV, bool DET, bool DROP, bool DQBF = false>
__global__ void __launch_bounds__(kThreads, 1)
    k_bwd_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
             const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
             const BwdArgs a) {
    using L = BwdCfg<DV>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const uint32_t sb = smem_u32(smem);
    const uint32_t bar0 = sb + L::OFF_BAR;
    auto BAR = [&](int i) { return bar0 + 8u * i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_BAR + 8 * NBAR);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const float* st_smem = reinterpret_cast<const float*>(smem + L::OFF_ST);

    const Problem& P = a.P;
    const Work W = decode(a);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(BAR(B_KV), 1);
        for (int s = 0; s < NS; ++s) {
            mbar_init(BAR(B_QF + s), 1);
            mbar_init(BAR(B_QE + s), 2);   // both MMA issuers read the stage
        }
        mbar_init(BAR(B_S), 1);
        mbar_init(BAR(B_SF), kSoftmax);
        mbar_init(BAR(B_DP + 0), 1);
        mbar_init(BAR(B_DP + 1), 1);
        mbar_init(BAR(B_DS), kSoftmax);
        mbar_init(BAR(B_DQF), 1);
        mbar_init(BAR(B_DQE), kSoftmax);
        mbar_init(BAR(B_PF), 1);
        mbar_init(BAR(B_KVD), 1);
        mbar_init(BAR(B_FIN), 1);
        mbar_init(BAR(B_FINB), 1);
        mbar_init(BAR(B_PRF + 0), 1);
        mbar_init(BAR(B_PRF + 1), 1);
        *abort_flag = (a.status && (*reinterpret_cast<volatile uint32_t*>(a.status) & ST_TIMEOUT)) ? 1 : 0;
        fence_mbar_init();
    }
    if (warp == 9) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tS = tmem, tDP = tmem + 64, tDQ = tmem + 192, tDK = tmem + 256, tDV = tmem + 384;
    const bool skip = *abort_flag != 0;
    const int n_it = skip ? 0 : W.n_it;

    // Query tiles from the last one down, the group's q heads innermost: the CTAs of one
    // (batch, kv head) then walk the same query tiles at about the same time, so a Q / dO
    // tile and its dQ accumulator rows are fetched once into L2 and shared.
    auto iter_head = [&](int it) { return W.hkv * P.G + W.g0 + it % W.gn; };
    auto iter_q0 = [&](int it) { return (W.qt_lo + W.n_qt - 1 - it / W.gn) * BQ; };

    if (warp == 8) {
        // ------------------------------------------------------------ producer
        if (lane == 0 && n_it > 0) {
            tma_prefetch(&tmQ);
            tma_prefetch(&tmK);
            tma_prefetch(&tmV);
            tma_prefetch(&tmDO);
            mbar_expect_tx(BAR(B_KV), BK * (D + DV) * 2);
            for (int sub = 0; sub < D / 64; ++sub)
                tma_load_4d(sb + OFF_K + sub * SUBK, &tmK, BAR(B_KV), sub * 64, W.hkv, W.k0, W.b);
            for (int sub = 0; sub < DV / 64; ++sub)
                tma_load_4d(sb + L::OFF_V + sub * SUBK, &tmV, BAR(B_KV), sub * 64, W.hkv, W.k0, W.b);
            int n_issued = 0;
            for (int it = 0; it < n_it; ++it) {
                const int st = it % NS, use = it / NS;
                if (use > 0 && !mbar_wait(BAR(B_QE + st), (use - 1) & 1, abort_flag, a.status, 0x40)) break;
                const int h = iter_head(it), q0 = iter_q0(it);
                mbar_expect_tx(BAR(B_QF + st), BQ * D * 2 + L::DO_BYTES + 512);
                for (int sub = 0; sub < D / 64; ++sub)
                    tma_load_4d(sb + L::OFF_Q + st * BQ * D * 2 + sub * SUBQ, &tmQ, BAR(B_QF + st), sub * 64, h,
                                q0, W.b);
                for (int sub = 0; sub < DV / 64; ++sub)
                    tma_load_4d(sb + L::OFF_DO + st * L::DO_BYTES + sub * SUBQ, &tmDO, BAR(B_QF + st), sub * 64,
                                h, q0, W.b);
                const int64_t row = (static_cast<int64_t>(W.b) * P.Hq + h) * a.Spad + q0;
                bulk_load(sb + L::OFF_ST + st * 512, a.lse + row, 256, BAR(B_QF + st));
                bulk_load(sb + L::OFF_ST + st * 512 + 256, a.Dvec + row, 256, BAR(B_QF + st));
                n_issued = it + 1;
            }
            drain_wait(BAR(B_KV), 0, a.status);
            for (int s = 0; s < NS; ++s) {
                const int uses = (n_issued - s + NS - 1) / NS;
                if (uses > 0) drain_wait(BAR(B_QF + s), (uses - 1) & 1, a.status);
            }
        }
    } else if (warp == 9) {
        // ------------------------------------------------------------ MMA issuer A: S^T, dP^T
        // The whole warp runs the loop with warp-uniform operands; one elected lane issues.
        if (n_it > 0) {
            bool ok = __all_sync(0xffffffffu, mbar_wait(BAR(B_KV), 0, abort_flag, a.status, 0x50));
            const uint64_t kd0 = sdesc_sw128(sb + OFF_K, 16, 1024), vd0 = sdesc_sw128(sb + L::OFF_V, 16, 1024);
            for (int it = 0; ok && it < n_it; ++it) {
                const int st = it % NS, buf = it & 1;
                if (!__all_sync(0xffffffffu, mbar_wait(BAR(B_QF + st), (it / NS) & 1, abort_flag, a.status, 0x51))) break;
                // S^T(it-1) has been read; the P^T / dS^T pairs of tile it-2 in this dP^T buffer
                // have been consumed by issuer B's dV / dK products
                if (it > 0 && !__all_sync(0xffffffffu, mbar_wait(BAR(B_SF), (it - 1) & 1, abort_flag, a.status, 0x54))) break;
                if (it > 1 && !__all_sync(0xffffffffu, mbar_wait(BAR(B_PRF + buf), ((it >> 1) - 1) & 1, abort_flag,
                                                                  a.status, 0x55)))
                    break;
                tc_fence_after();
                const uint64_t qd = sdesc_sw128(sb + L::OFF_Q + st * BQ * D * 2, 16, 1024);
                const uint64_t dod = sdesc_sw128(sb + L::OFF_DO + st * L::DO_BYTES, 16, 1024);
                // S^T and dP^T are independent accumulations: interleaved, each waits less on
                // its own previous step (dP^T contracts over DV channels, S^T over D)
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t offk = (kk >> 2) * SUBK + (kk & 3) * 32;
                    const uint32_t offq = (kk >> 2) * SUBQ + (kk & 3) * 32;
                    tc_mma_ss_w(tS, sdesc_advance(kd0, offk), sdesc_advance(qd, offq), IDESC_S, kk > 0);
                    if (kk < DV / 16)
                        tc_mma_ss_w(tDP + buf * BQ, sdesc_advance(vd0, offk), sdesc_advance(dod, offq), IDESC_S, kk > 0);
                }
                tc_commit_w(BAR(B_S));
                tc_commit_w(BAR(B_DP + buf));
                tc_commit_w(BAR(B_QE + st));   // this issuer's reads of the Q / dO stage
            }
            tc_commit_w(BAR(B_FIN));
            drain_wait(BAR(B_FIN), 0, a.status);
        }
    } else if (warp == 10) {
        // ------------------------------------------------------------ MMA issuer B: dV, dK, dQ^T
        if (n_it > 0) {
            const uint64_t kmn0 = sdesc_sw128(sb + OFF_K, SUBK, 1024);
            const uint64_t dsmn = sdesc_sw128(sb + L::OFF_DS, 16, 1024);
            for (int p = 0; p < n_it; ++p) {
                const int pst = p % NS, buf = p & 1;
                if (!__all_sync(0xffffffffu, mbar_wait(BAR(B_DS), p & 1, abort_flag, a.status, 0x52))) break;
                tc_fence_after();
                const uint64_t qmn = sdesc_sw128(sb + L::OFF_Q + pst * BQ * D * 2, SUBQ, 1024);
                const uint64_t domn = sdesc_sw128(sb + L::OFF_DO + pst * L::DO_BYTES, SUBQ, 1024);
                // bf16 pairs of query columns 16 kk .. 16 kk + 15: warpgroup kk / 2 wrote P^T at
                // columns 32 (kk / 2) + 8 (kk % 2) of the dP^T buffer and dS^T 16 columns further
                const uint32_t tPD = tDP + buf * BQ;
#pragma unroll
                for (int kk = 0; kk < BQ / 16; ++kk) {
                    const uint32_t acc = (p > 0 || kk > 0) ? 1u : 0u;
                    const uint32_t tp = tPD + (kk >> 1) * 32 + (kk & 1) * 8;
                    tc_mma_ts_w(tDV, tp, sdesc_advance(domn, kk * 2048), L::IDESC_V, acc);
                    tc_mma_ts_w(tDK, tp + 16, sdesc_advance(qmn, kk * 2048), IDESC_KV, acc);
                }
                tc_commit_w(BAR(B_PRF + buf));   // the pairs have been read: issuer A may reuse the buffer
                tc_commit_w(BAR(B_QE + pst));
                if (p > 0 && !__all_sync(0xffffffffu, mbar_wait(BAR(B_DQE), (p - 1) & 1, abort_flag, a.status, 0x53))) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk)
                    tc_mma_ss_w(tDQ, sdesc_advance(kmn0, kk * 2048), sdesc_advance(dsmn, kk * 2048), IDESC_Q, kk > 0);
                tc_commit_w(BAR(B_DQF));
                tc_commit_w(BAR(B_PF));
                if (p == n_it - 1) tc_commit_w(BAR(B_KVD));
            }
            tc_commit_w(BAR(B_FINB));
            drain_wait(BAR(B_FINB), 0, a.status);
        }
    } else {
        // ------------------------------------------------------------ P, dS, dQ (two warpgroups)
        const int wg = warp >> 2, quarter = warp & 3;
        const int r = quarter * 32 + lane;    // key row of S^T / dP^T, channel of dQ^T: the TMEM lane
        const int cq = wg * 32;               // this warpgroup's query columns of a tile
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const int k = W.k0 + r;
        int qmin = W.q_lo, qmax = min(W.q_hi, P.S - 1);
        if (P.causal) qmin = max(qmin, k - W.off);
        if (P.wr >= 0) qmin = max(qmin, k - W.off - P.wr);
        if (P.wl >= 0) qmax = min(qmax, k - W.off + P.wl);
        if (k >= W.lk) qmax = -1;
        const float sl2 = P.scale * kLog2e;
        bool aborted = false;

        // dQ^T of tile t, query columns cq .. cq+31, added to the accumulator [S'/4][128][4] of
        // its (batch, q head): four consecutive queries of this thread's channel are one 16-byte
        // reduction, and a warp's 32 channels are 512 contiguous bytes
        auto drain_dq = [&](int t) -> bool {
            if (!__all_sync(0xffffffffu, mbar_wait(BAR(B_DQF), t & 1, abort_flag, a.status, 0x70))) return false;
            tc_fence_after();
            uint32_t v[32];
            tmem_ld32(tDQ + cq + lane_base, v);
            tc_fence_before();
            mbar_arrive(BAR(B_DQE));
            if (DQBF) {
                // band backward: at most two key tiles add to any dq element, so bf16 pair
                // reductions straight into dq give an order-independent result.  Adjacent
                // lanes (channels r, r ^ 1) trade one value per two queries: the even lane
                // adds channels (r, r + 1) of query j, the odd lane those of query j + 1, so
                // a warp's reduction covers two 64-byte runs of dq.
                const int q0 = iter_q0(t) + cq;
                __nv_bfloat16* base = static_cast<__nv_bfloat16*>(a.dq) + W.b * P.qs[0] +
                                      static_cast<int64_t>(iter_head(t)) * P.qs[2] + (r & ~1);
                const bool odd = lane & 1;
#pragma unroll
                for (int jj = 0; jj < 32; jj += 2) {
                    const float mine0 = __uint_as_float(v[jj]), mine1 = __uint_as_float(v[jj + 1]);
                    const float got = __shfl_xor_sync(0xffffffffu, odd ? mine0 : mine1, 1);
                    const int q = q0 + jj + (odd ? 1 : 0);
                    const float lo = odd ? got : mine0, hi = odd ? mine1 : got;
                    if (q < P.S) red_add_bf16x2(base + static_cast<int64_t>(q) * P.qs[1], pack_bf16(lo * P.scale, hi * P.scale));
                }
                return true;
            }
            float* dst = a.dq_acc + (static_cast<int64_t>(W.b) * P.Hq + iter_head(t)) * a.Spad * D +
                         (static_cast<int64_t>((iter_q0(t) + cq) >> 2) * D + r) * 4;
            if (DET) {   // this key tile's own slice: written once, added in key order later
                dst += static_cast<int64_t>(W.k0 / BK) * P.B * P.Hq * a.Spad * D;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    *reinterpret_cast<float4*>(dst + j * (4 * D)) =
                        make_float4(__uint_as_float(v[4 * j]) * P.scale, __uint_as_float(v[4 * j + 1]) * P.scale,
                                    __uint_as_float(v[4 * j + 2]) * P.scale, __uint_as_float(v[4 * j + 3]) * P.scale);
                return true;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j)
                red_add_v4(dst + j * (4 * D), __uint_as_float(v[4 * j]) * P.scale,
                           __uint_as_float(v[4 * j + 1]) * P.scale, __uint_as_float(v[4 * j + 2]) * P.scale,
                           __uint_as_float(v[4 * j + 3]) * P.scale);
            return true;
        };

        for (int it = 0; it < n_it; ++it) {
            const int h = iter_head(it), q0 = iter_q0(it) + cq, st = it % NS, buf = it & 1;
            if (!__all_sync(0xffffffffu, mbar_wait(BAR(B_S), it & 1, abort_flag, a.status, 0x60))) {
                aborted = true;
                break;
            }
            tc_fence_after();
            float p[32];
            {
                uint32_t v[32];
                tmem_ld32(tS + cq + lane_base, v);
#pragma unroll
                for (int i = 0; i < 32; ++i) p[i] = __uint_as_float(v[i]) * sl2;
            }
            tc_fence_before();
            mbar_arrive(BAR(B_SF));   // S^T may be overwritten by the next tile
            // the lse / D of this tile came with the Q tile: observe that copy's barrier
            // (it cannot have moved on: the stage is refilled only after this tile's dS)
            if (!__all_sync(0xffffffffu, mbar_wait(BAR(B_QF + st), (it / NS) & 1, abort_flag, a.status, 0x64))) {
                aborted = true;
                break;
            }
            const float* lse = st_smem + st * 128 + cq;
            const float* Dq = st_smem + st * 128 + 64 + cq;
            if (P.bias) {
                const float* brow = P.bias + W.b * P.bs[0] + h * P.bs[1] + static_cast<int64_t>(min(k, P.S - 1)) * P.bs[3];
                if (P.bs[2] == 0) {   // the bias does not depend on the query: one value per key row
                    const float bk = brow[0] * kLog2e;
#pragma unroll
                    for (int c = 0; c < 32; ++c) p[c] += bk;
                } else {
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        const int q = min(q0 + c, P.S - 1);
                        p[c] = fmaf(brow[q * P.bs[2]], kLog2e, p[c]);
                    }
                }
            }
#pragma unroll
            for (int c = 0; c < 32; ++c) p[c] = ex2(p[c] - lse[c] * kLog2e);
            const bool edge = q0 < qmin || q0 + 31 > qmax;
            if (__any_sync(0xffffffffu, edge)) {
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const int q = q0 + c;
                    if (q < qmin || q > qmax) p[c] = 0.f;
                }
            }
            if constexpr (DROP) {   // dropped entries leave the softmax: P = 0, hence dS = 0
                const uint32_t keep = dropout_keep_q32(P.drop_thr, P.drop_k0, P.drop_k1, W.b, h, q0, k, lane);
#pragma unroll
                for (int c = 0; c < 32; ++c)
                    if (!((keep >> c) & 1u)) p[c] = 0.f;
            }
            // the dS^T buffer is free once the dQ product of the previous tile has read it
            if (it > 0 && !__all_sync(0xffffffffu, mbar_wait(BAR(B_PF), (it - 1) & 1, abort_flag, a.status, 0x61))) {
                aborted = true;
                break;
            }
            if (!__all_sync(0xffffffffu, mbar_wait(BAR(B_DP + buf), (it >> 1) & 1, abort_flag, a.status, 0x62))) {
                aborted = true;
                break;
            }
            tc_fence_after();
            // this warpgroup's 32 dP^T columns; once read, P^T pairs take the first 16 of them
            // and dS^T pairs the other 16
            const uint32_t tcol = tDP + buf * BQ + cq + lane_base;
            uint32_t ppk[16], dpk[16];
            {
                uint32_t v[32];
                tmem_ld32(tcol, v);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    ppk[i] = pack_bf16(p[2 * i], p[2 * i + 1]);
                    dpk[i] = pack_bf16(p[2 * i] * (__uint_as_float(v[2 * i]) - Dq[2 * i]),
                                       p[2 * i + 1] * (__uint_as_float(v[2 * i + 1]) - Dq[2 * i + 1]));
                }
            }
            tmem_st16_nowait(tcol, ppk);
            tmem_st16_nowait(tcol + 16, dpk);
            const uint32_t db = sb + L::OFF_DS;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
                st_shared_v4(db + sw128_offset(r, wg * 4 + cc), dpk[4 * cc], dpk[4 * cc + 1], dpk[4 * cc + 2],
                             dpk[4 * cc + 3]);
            tmem_st_wait();
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(BAR(B_DS));
            if (it > 0 && !drain_dq(it - 1)) {
                aborted = true;
                break;
            }
        }
        if (!aborted && n_it > 0 && !drain_dq(n_it - 1)) aborted = true;
        // ---- epilogue: warps 0-3 dK = scale * acc, warps 4-7 dV = acc
        if (!aborted && !skip) {
            if (n_it > 0) {
                if (!__all_sync(0xffffffffu, mbar_wait(BAR(B_KVD), 0, abort_flag, a.status, 0x63))) aborted = true;
                tc_fence_after();
            }
            if (!aborted) {
                const int kk = min(k, P.S - 1);
                const float f = wg == 0 ? P.scale : 1.f;
                const uint32_t tacc = wg == 0 ? tDK : tDV;
                __nv_bfloat16* out = wg == 0 ? static_cast<__nv_bfloat16*>(a.dk) + W.b * P.ks[0] +
                                                   static_cast<int64_t>(kk) * P.ks[1] + W.hkv * P.ks[2]
                                             : static_cast<__nv_bfloat16*>(a.dv) + W.b * P.vs[0] +
                                                   static_cast<int64_t>(kk) * P.vs[1] + W.hkv * P.vs[2];
                float* carry_base = wg == 0 ? a.dk_acc : a.dv_acc;
                const int ncol = wg == 0 ? D : DV;   // channels of dK / dV
                float* carry = carry_base
                                   ? carry_base + ((static_cast<int64_t>(W.b) * P.S + kk) * P.Hkv + W.hkv) * ncol
                                   : nullptr;
#pragma unroll 1
                for (int c = 0; c < ncol / 32; ++c) {
                    uint32_t v[32];
                    if (n_it > 0) {
                        tmem_ld32(tacc + c * 32 + lane_base, v);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = 0u;
                    }
                    if (k < P.S) {
                        if (carry) {
                            if (n_it > 0) {
                                float4* dst = reinterpret_cast<float4*>(carry + c * 32);
#pragma unroll
                                for (int i = 0; i < 8; ++i) {
                                    float4 x = dst[i];
                                    x.x += __uint_as_float(v[4 * i + 0]) * f;
                                    x.y += __uint_as_float(v[4 * i + 1]) * f;
                                    x.z += __uint_as_float(v[4 * i + 2]) * f;
                                    x.w += __uint_as_float(v[4 * i + 3]) * f;
                                    dst[i] = x;
                                }
                            }
                        } else {
                            uint32_t w[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                w[i] = pack_bf16(__uint_as_float(v[2 * i]) * f, __uint_as_float(v[2 * i + 1]) * f);
                            if (a.hsplit > 1) {
                                // two halves add into the zeroed dk / dv: 0 + x + y in either order
#pragma unroll
                                for (int i = 0; i < 16; ++i) red_add_bf16x2(out + c * 32 + 2 * i, w[i]);
                            } else if ((reinterpret_cast<uintptr_t>(out) & 31u) == 0) {   // whole 32-byte sectors
                                st_global_v8(out + c * 32, w);
                                st_global_v8(out + c * 32 + 16, w + 8);
                            } else {
                                uint4* dst = reinterpret_cast<uint4*>(out + c * 32);
#pragma unroll
                                for (int i = 0; i < 4; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
                            }
                        }
                    }
                }
            }
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int DV>
cudaError_t launch_dv(const BwdArgs& a, const CUtensorMap* maps, cudaStream_t s) {
    using L = BwdCfg<DV>;
    // the deterministic and dropout variants are separate instantiations: the default
    // kernel's code is left exactly as it is without the knobs
    static bool configured[4][64] = {};
    const int var = (a.P.det ? 1 : 0) | (a.P.drop_thr ? 2 : 0);
    void (*kern)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, BwdArgs) =
        var == 0 ? k_bwd_tc<DV, false, false>
                 : (var == 1 ? k_bwd_tc<DV, true, false> : (var == 2 ? k_bwd_tc<DV, false, true> : k_bwd_tc<DV, true, true>));
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !configured[var][dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) configured[var][dev] = true;
    }
    const int nkt = (a.P.S + BK - 1) / BK;
    const int grid = nkt * a.P.Hkv * a.P.B * (a.hsplit > 1 ? 2 : 1);
    kern<<<grid, kThreads, L::SMEM, s>>>(maps[0], maps[1], maps[2], maps[3], a);
    return cudaGetLastError();
}

// Deterministic mode: dQ = the sum of the key tiles' slices, in ascending key-tile order,
// cast to bf16.  One warp per (batch, q head, four query rows); a key tile's slice is read
// only if that tile's CTA visited the rows' 64-row query tile (the decoder above decides,
// as it did for the CTA), so unwritten slice rows are never read.
__global__ void k_dq_reduce(const BwdArgs a) {
    const Problem& P = a.P;
    const int lane = threadIdx.x & 31, even = (lane & 1) == 0;
    const int n4 = (P.S + 3) / 4, nkt = (P.S + BK - 1) / BK;
    const int64_t slice = static_cast<int64_t>(P.B) * P.Hq * a.Spad * D;
    const int64_t groups = static_cast<int64_t>(P.B) * P.Hq * n4;
    const int64_t wstride = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t gi = blockIdx.x * static_cast<int64_t>(blockDim.x >> 5) + (threadIdx.x >> 5); gi < groups;
         gi += wstride) {
        const int q4 = static_cast<int>(gi % n4);
        const int h = static_cast<int>((gi / n4) % P.Hq);
        const int b = static_cast<int>(gi / (static_cast<int64_t>(n4) * P.Hq));
        const int qt = q4 * 4 / BQ;
        const int64_t off = ((static_cast<int64_t>(b) * P.Hq + h) * (a.Spad / 4) + q4) * D * 4;
        float4 acc[D / 32];
#pragma unroll
        for (int g = 0; g < D / 32; ++g) acc[g] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int kt = 0; kt < nkt; ++kt) {
            const Work w = decode_tile_of(a, b, h / P.G, kt);
            if (qt < w.qt_lo || qt >= w.qt_lo + w.n_qt) continue;
            const float4* in = reinterpret_cast<const float4*>(a.dq_acc + kt * slice + off);
#pragma unroll
            for (int g = 0; g < D / 32; ++g) {
                const float4 x = in[g * 32 + lane];
                acc[g].x += x.x;
                acc[g].y += x.y;
                acc[g].z += x.z;
                acc[g].w += x.w;
            }
        }
        // lane = channel c0 + lane; its float4 holds queries 4 q4 .. 4 q4 + 3: even lanes write
        // rows 4 q4, 4 q4 + 1 and odd lanes rows 4 q4 + 2, + 3 as channel pairs
        const int qa = q4 * 4 + (even ? 0 : 2);
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.dq) + b * P.qs[0] + h * P.qs[2];
#pragma unroll
        for (int g = 0; g < D / 32; ++g) {
            const float4 x = acc[g];
            const float y0 = __shfl_xor_sync(0xffffffffu, even ? x.z : x.x, 1);
            const float y1 = __shfl_xor_sync(0xffffffffu, even ? x.w : x.y, 1);
            const int c = g * 32 + lane - (even ? 0 : 1);
            const uint32_t w0 = even ? pack_bf16(x.x, y0) : pack_bf16(y0, x.z);
            const uint32_t w1 = even ? pack_bf16(x.y, y1) : pack_bf16(y1, x.w);
            if (qa < P.S) *reinterpret_cast<uint32_t*>(out + static_cast<int64_t>(qa) * P.qs[1] + c) = w0;
            if (qa + 1 < P.S) *reinterpret_cast<uint32_t*>(out + static_cast<int64_t>(qa + 1) * P.qs[1] + c) = w1;
        }
    }
}

}  // namespace

cudaError_t launch_dq_reduce(const BwdArgs& a, cudaStream_t s) {
    const int64_t warps = static_cast<int64_t>(a.P.B) * a.P.Hq * ((a.P.S + 3) / 4);
    const int64_t blocks = std::min<int64_t>((warps + 7) / 8, 1 << 20);
    k_dq_reduce<<<static_cast<unsigned>(blocks), 256, 0, s>>>(a);
    return cudaGetLastError();
}

// Band backward: dQ reduced in bf16 pairs into dq (d = dv = 128).
cudaError_t launch_bwd_tc_band(const BwdArgs& a, const CUtensorMap* maps, cudaStream_t s) {
    using L = BwdCfg<128>;
    static bool configured[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !configured[dev]) {
        e = cudaFuncSetAttribute(k_bwd_tc<128, false, false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 L::SMEM);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) configured[dev] = true;
    }
    const int nkt = (a.P.S + BK - 1) / BK;
    const int grid = nkt * a.P.Hkv * a.P.B * (a.hsplit > 1 ? 2 : 1);
    k_bwd_tc<128, false, false, true><<<grid, kThreads, L::SMEM, s>>>(maps[0], maps[1], maps[2], maps[3], a);
    return cudaGetLastError();
}

bool bwd_band_supported(const Problem& P) {
    if (!bwd_tc_supported(P) || P.dv != D || P.ring_n != 1) return false;
    if (P.seqlens_q || P.seqlens_kv || P.sink || P.dsink || P.det || P.drop_thr) return false;
    // the vectorised pre-pass (which zeroes dq) indexes rows in 32 bits
    if (static_cast<int64_t>(P.B) * P.Hq * ((P.S + 63) / 64 * 64) >= (1ll << 31)) return false;
    // at most two key tiles may see any 64-row query tile (a window of at most one tile)
    for (int q0 = 0; q0 < P.S; q0 += BQ) {
        const int qb = q0 + BQ - 1 < P.S - 1 ? q0 + BQ - 1 : P.S - 1;
        int klo = 0, khi = P.S - 1;
        if (P.causal && qb < khi) khi = qb;
        if (P.wr >= 0 && qb + P.wr < khi) khi = qb + P.wr;
        if (P.wl >= 0 && q0 - P.wl > klo) klo = q0 - P.wl;
        if (klo <= khi && khi / BK - klo / BK + 1 > 2) return false;
    }
    return true;
}

bool bwd_tc_supported(const Problem& P) {
    if (P.dtype != BPA_BF16 || P.d != D || (P.dv != D && P.dv != 64) || P.block_idx) return false;
    if (P.ring_n > 1 && P.ring_blk % BK) return false;
    return true;
}

cudaError_t launch_bwd_tc(const BwdArgs& a, const CUtensorMap* maps, cudaStream_t s) {
    return a.P.dv == 64 ? launch_dv<64>(a, maps, s) : launch_dv<128>(a, maps, s);
}

}  // namespace bpa
