// fwd_tc.cuh - blockwise attention forward on the 5th-generation tensor cores (bf16; (d, dv) =
// (64, 64), (128, 128) or (128, 64)).
//
// Persistent: one CTA per SM (two for the one-tile variant) takes work items from a
// counter, heaviest first; an item is two 128-row query tiles: the same rows of two q heads
// of one kv head (even group sizes), else two consecutive row tiles of one (batch, q head).
// For each item the CTA walks the 128-key tiles the masks (and the batch entry's sequence
// lengths) allow, folding each into a running (max, numerator, denominator) carry per query
// row ("bpt.py", _blockwise_attention_fwd / scan_kv_block):
//     m' = max(m, rowmax S);  P = exp(S - m');  num = num * exp(m - m') + P V;
//     den = den * exp(m - m') + rowsum P
// Both query tiles share every K / V tile that is loaded.
// TMEM (512 columns): S0 [0,128), S1 [128,256), O0 [256,256+dv), O1 [384,384+dv).
// P (bf16, two per 32-bit column) is written back over the first 64 columns
// of its S tile and read from there by the P V product (A operand in TMEM).
// Roles (320 threads):
//   warps 0-3  softmax of query tile 0: thread t owns row t (TMEM lane t);
//   warps 4-7  softmax of query tile 1;
//   warp 8     TMA producer: Q0, Q1 once, then K / V tiles through their rings;
//   warp 9     MMA issuer (the whole warp runs the loop with warp-uniform operands, one
//              elected lane issues: cheaper per product than a lone lane), TMEM owner.  Issue order per key tile j:
//              [P0(j) ready] P0 V -> O0, S0(j+1) = Q0 K^T ; [P1(j) ready] P1 V -> O1,
//              S1(j+1): the tensor core works on one tile while the other tile's
//              softmax runs.  The products of a tile execute in issue order, so
//              when S_i(j+1) completes, P_i(j) V has consumed P_i(j) and O_i holds
//              every key tile up to j.
// The numerator is rescaled lazily: the reference max of a row only moves when
// its max grows by more than kTau (log2 units); exact in real arithmetic because
// numerator and denominator share the reference.
// Fully masked tiles are never visited (key ranges are cut by position); only
// tiles that straddle a mask edge apply the elementwise mask.
// The epilogue divides by the denominator (plus the sink term with sink attention) and
// stores O, m, l.
// Every wait is bounded (common.cuh); on a timeout the CTA drains its in-flight
// copies and MMAs, frees TMEM and returns.
#pragma once

#include <math.h>

#include <algorithm>

#include "bpa_internal.h"
#include "common.cuh"

namespace bpa {
namespace {

constexpr int BM = 128;       // query rows per tile
constexpr int BN = 128;       // keys per tile
constexpr float kTau = 8.f;   // lazy-rescale threshold, log2 units

// NQ query tiles per CTA.  NQ = 2: two softmax warpgroups share every K / V
// tile (long key ranges).  NQ = 1: a smaller CTA (192 threads, 256 TMEM
// columns, < 113 KB of shared memory) so that two run on an SM and one CTA's
// loads and stores overlap the other's products (short key ranges, e.g. a
// narrow sliding window).
// D: head dim of q, k; DV: head dim of v and the output (DV == D, or D = 128 with DV = 64).
template <int D, int DV, int NQ>
struct FwdCfg {
    static constexpr int kThreads = NQ * 128 + 64;
    static constexpr int kTmemCols = NQ * 256;
    static constexpr int kProducer = 4 * NQ, kMma = 4 * NQ + 1;   // warp indices
    // K and V flow through separate rings: K tile j is needed one product
    // earlier than V tile j, so it gets more stages where space allows.
    static constexpr int NSK = NQ == 2 ? (D == 128 ? 3 : 4) : (D == 128 ? 1 : 2);   // K stages
    static constexpr int NSV = NQ == 2 ? (DV == 128 ? 2 : (D == 128 ? 3 : 4)) : (DV == 128 ? 1 : 2);   // V stages
    static constexpr int Q_BYTES = BM * D * 2;     // one query tile
    static constexpr int KV_BYTES = BN * D * 2;    // one K tile
    static constexpr int V_BYTES = BN * DV * 2;    // one V tile
    static constexpr int SUB = 128 * 128;          // one 64-column slab of 128 rows
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + NQ * Q_BYTES;
    static constexpr int OFF_V = OFF_K + NSK * KV_BYTES;
    static constexpr int OFF_KB = OFF_V + NSV * V_BYTES;    // per K stage: the tile's 128 key-bias values
    static constexpr int OFF_BAR = OFF_KB + NSK * BN * 4;
    static constexpr int SMEM = OFF_BAR + 512 + 1024;   // + slack to align the base to 1024
    // barrier slots: Q full / empty; K full / empty, V full / empty; S, P, O full, O empty per
    // query tile; work item published / read (two slots)
    static constexpr int B_Q = 0, B_KF = 1, B_KE = 1 + NSK, B_VF = 1 + 2 * NSK, B_VE = 1 + 2 * NSK + NSV,
                         B_S = 1 + 2 * NSK + 2 * NSV, B_P = B_S + 2, B_O = B_S + 4, B_FIN = B_S + 6,
                         B_QE = B_S + 7, B_OE = B_S + 8, B_IF = B_S + 10, B_IE = B_S + 12, NBAR = B_S + 14;
    static_assert(8 * NBAR + 16 <= 512, "barrier area");
    static_assert(SMEM <= 232448, "shared memory");
    static constexpr uint32_t IDESC_S = idesc_bf16_f32(BM, BN, 0, 0);   // Q, K both K-major
    static constexpr uint32_t IDESC_PV = idesc_bf16_f32(BM, DV, 0, 1);   // P (TMEM), V MN-major
    static_assert(NQ == 2 || 2 * SMEM <= 233472, "two single-tile CTAs must fit an SM");
};

struct Tile {
    int b, h, hkv, q0;       // h, q0: head and first row of query tile 0
    int dh, dq;              // query tile 1: head h + dh, first row q0 + dq
    int rlo, rhi;            // key range of this launch (ring super-block or whole sequence)
    int kt0;                 // first key tile visited by the CTA
    int n;                   // key tiles visited by the CTA
    int lo[2], hi[2];        // per query tile: visited step range [lo, hi] (empty if lo > hi)
    int lq, off;             // valid query rows of the batch entry, offset of the causal / window diagonal
};

// The two query tiles of a work item are the same rows of two q heads that share a kv head
// when the group size is even (the tiles then see the same key tiles, so neither finishes
// alone, and a per-head key bias would differ between them, so none may be staged per key
// tile); otherwise two consecutive row tiles of one q head.
template <int NQ>
__host__ __device__ __forceinline__ bool head_pairs(const Problem& P) {
    return NQ == 2 && P.G % 2 == 0 && (P.bias == nullptr || P.bs[1] == 0);
}

template <int NQ>
__host__ __device__ __forceinline__ int fwd_items(const Problem& P) {
    return head_pairs<NQ>(P) ? ((P.S + BM - 1) / BM) * (P.Hq / 2) * P.B
                             : ((P.S + NQ * BM - 1) / (NQ * BM)) * P.Hq * P.B;
}

// Work item `item` (heaviest causal query rows first) -> its query tiles and key range.
template <int NQ>
__device__ __forceinline__ Tile decode_tile(const FwdArgs& a, int item) {
    const Problem& P = a.P;
    const bool hp = head_pairs<NQ>(P);
    const int per_g = hp ? P.G / 2 : P.G;   // items per (row block, batch entry, kv head)
    int r = item;
    const int gi = r % per_g;
    r /= per_g;
    Tile t;
    t.hkv = r % P.Hkv;
    r /= P.Hkv;
    t.b = r % P.B;
    if (hp) {
        const int qt = (P.S + BM - 1) / BM - 1 - r / P.B;   // heaviest (causal) rows first
        t.h = t.hkv * P.G + 2 * gi;
        t.q0 = qt * BM;
        t.dh = 1;
        t.dq = 0;
    } else {
        const int nqp = (P.S + NQ * BM - 1) / (NQ * BM);
        const int qp = nqp - 1 - r / P.B;
        t.h = t.hkv * P.G + gi;
        t.q0 = qp * NQ * BM;
        t.dh = 0;
        t.dq = BM;
    }
    const Lens len = lens_of(P, t.b);   // full lengths unless the problem has sequence lengths
    t.lq = len.lq;
    t.off = len.off;
    t.rlo = 0;
    t.rhi = len.lk - 1;
    if (a.acc) {
        const int i = t.q0 / P.ring_blk;
        const int j = ((i - a.ring_idx) % P.ring_n + P.ring_n) % P.ring_n;
        t.rlo = j * P.ring_blk;
        t.rhi = t.rlo + P.ring_blk - 1;
    }
    int ktlo[2] = {1, 1}, kthi[2] = {0, 0};
    int ulo = 1 << 30, uhi = -1;
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
        const int qa = t.q0 + i * t.dq, qb = min(qa + BM - 1, t.lq - 1);
        int lo = t.rlo, hi = t.rhi;
        if (qa >= t.lq) hi = -1;
        if (P.causal) hi = min(hi, qb + t.off);
        if (P.wr >= 0) hi = min(hi, qb + t.off + P.wr);
        if (P.wl >= 0) lo = max(lo, qa + t.off - P.wl);
        if (lo <= hi) {
            ktlo[i] = lo / BN;
            kthi[i] = hi / BN;
            ulo = min(ulo, ktlo[i]);
            uhi = max(uhi, kthi[i]);
        } else {
            ktlo[i] = 1;
            kthi[i] = 0;
        }
    }
    t.kt0 = uhi >= 0 ? ulo : 0;
    t.n = uhi >= 0 ? uhi - ulo + 1 : 0;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        t.lo[i] = ktlo[i] - t.kt0;
        t.hi[i] = kthi[i] - t.kt0;
    }
    return t;
}

// Sink attention: the sink logit sk (natural log units) joins a row's softmax max and
// denominator but brings no value vector.  From the row's sum lsum relative to m_used and
// its true max m_true (log2 units) returns (denominator relative to m_used, final max,
// final sum relative to the final max).  Out of line: it runs once per row and item.
__device__ __noinline__ float3 with_sink(float sk, float lsum, float m_used, float m_true) {
    const float s2 = sk * kLog2e;
    const float m_fin = fmaxf(m_true, s2);
    return make_float3(lsum + ex2(s2 - m_used), m_fin,
                       (m_true == -INFINITY ? 0.f : lsum * ex2(m_used - m_fin)) + ex2(s2 - m_fin));
}

// bounded wait that ignores the abort flag: used to drain in-flight work
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint32_t* status) {
    int never = 0;
    mbar_wait(bar, parity, &never, status, 0xD0);
}

// Softmax passes over one 128-column row of S in TMEM, specialised on whether
// an additive bias is present and whether the tile straddles a mask edge, so
// that interior tiles run branch-free.  Scores are in log2 units:
// x = S * scale * log2(e) + bias * log2(e), -inf where masked.
struct RowCtx {
    uint32_t tS;            // TMEM address of this thread's row of S
    float sl2;              // scale * log2(e)
    const float* bias_row;  // bias of this row (broadcast dims have stride 0)
    int64_t bs3;            // bias stride along keys
    const float* kbias;     // key-only bias: the tile's 128 values in shared memory
    int k0, kmin, kmax, S;  // first key of the tile, allowed keys of the row, length
    uint32_t keep[4];       // attention dropout: bit j of word j / 32 = key k0 + j kept
};

// BIAS: 0 none, 1 key-only bias staged in shared memory, 2 general bias read from global memory;
// DROP: dropped entries (attention dropout) leave the softmax like masked ones (used with EDGE)
template <int BIAS, bool EDGE, bool DROP = false>
__device__ __forceinline__ float score_at(const RowCtx& R, uint32_t raw, int i) {
    float x = __uint_as_float(raw) * R.sl2;
    if (BIAS == 1) x = fmaf(R.kbias[i], kLog2e, x);
    if (BIAS == 2) x = fmaf(R.bias_row[min(R.k0 + i, R.S - 1) * R.bs3], kLog2e, x);
    if (EDGE) x = (R.k0 + i < R.kmin || R.k0 + i > R.kmax) ? -INFINITY : x;
    if (DROP) x = ((R.keep[i >> 5] >> (i & 31)) & 1u) ? x : -INFINITY;
    return x;
}

// Two passes over the 128-column row of S.  S is read from TMEM twice rather
// than held in registers: 128 live scores do not fit the 168 registers a
// thread has with 10 warps.  Interior tiles use packed float32-pair
// arithmetic and a 3-input max.

// pass 1: the row max of the scores
template <int BIAS, bool EDGE, bool DROP = false>
__device__ __forceinline__ float row_max(const RowCtx& R) {
    float mt = -INFINITY;
    const uint64_t sl2x2 = f2_pack(R.sl2, R.sl2), l2e2 = f2_pack(kLog2e, kLog2e);
#pragma unroll
    for (int cc = 0; cc < BN / 64; ++cc) {
        uint32_t r[64];
        tmem_ld64(R.tS + cc * 64, r);
        if (BIAS == 1 && !EDGE) {
            float m2 = -INFINITY;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float4 bq = reinterpret_cast<const float4*>(R.kbias + cc * 64)[i];
                float x0, x1, x2, x3;
                f2_unpack(ffma2(f2_pack(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1])), sl2x2,
                                fmul2(f2_pack(bq.x, bq.y), l2e2)), x0, x1);
                f2_unpack(ffma2(f2_pack(__uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3])), sl2x2,
                                fmul2(f2_pack(bq.z, bq.w), l2e2)), x2, x3);
                m2 = fmax3(m2, x0, x1);
                m2 = fmax3(m2, x2, x3);
            }
            mt = fmaxf(mt, m2);
        } else if (!BIAS && !EDGE) {
            float m2 = -INFINITY;   // scale > 0: max of raw S, scaled once
#pragma unroll
            for (int i = 0; i < 32; ++i) m2 = fmax3(m2, __uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
            mt = fmaxf(mt, m2 * R.sl2);
        } else {
#pragma unroll
            for (int i = 0; i < 64; ++i) mt = fmaxf(mt, score_at<BIAS, EDGE, DROP>(R, r[i], cc * 64 + i));
        }
    }
    return mt;
}

// pass 2: P = exp2(x - mref) as bf16 pairs written over the first 64 columns
// of the row's S (chunk cc reads S columns [64cc, 64cc+64) and writes P
// columns [32cc, 32cc+32)); returns the row sum of P in float32
template <int BIAS, bool EDGE, bool DROP = false>
__device__ __forceinline__ float row_exp(const RowCtx& R, float mref) {
    uint64_t rs2 = 0;   // two float32 partial sums
    const uint64_t sl2x2 = f2_pack(R.sl2, R.sl2), negm2 = f2_pack(-mref, -mref);
#pragma unroll
    for (int cc = 0; cc < BN / 64; ++cc) {
        uint32_t r[64];
        tmem_ld64(R.tS + cc * 64, r);
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            uint64_t p2;
            if (BIAS == 1 && !EDGE) {
                const float2 bp = reinterpret_cast<const float2*>(R.kbias + cc * 64)[i];
                float x0, x1;   // S * scale_log2 + (bias * log2e - mref)
                f2_unpack(ffma2(f2_pack(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), sl2x2,
                                ffma2(f2_pack(bp.x, bp.y), f2_pack(kLog2e, kLog2e), negm2)),
                          x0, x1);
                p2 = f2_pack(ex2(x0), ex2(x1));
            } else if (!BIAS && !EDGE) {
                float x0, x1;
                f2_unpack(ffma2(f2_pack(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), sl2x2, negm2), x0, x1);
                p2 = f2_pack(ex2(x0), ex2(x1));
            } else {
                p2 = f2_pack(ex2(score_at<BIAS, EDGE, DROP>(R, r[2 * i], cc * 64 + 2 * i) - mref),
                             ex2(score_at<BIAS, EDGE, DROP>(R, r[2 * i + 1], cc * 64 + 2 * i + 1) - mref));
            }
            rs2 = fadd2(rs2, p2);
            float p0, p1;
            f2_unpack(p2, p0, p1);
            pk[i] = pack_bf16(p0, p1);
        }
        tmem_st32(R.tS + cc * 32, pk);
    }
    float a, b;
    f2_unpack(rs2, a, b);
    return a + b;
}

// One pass over the row for tiles after the first: P = exp2(x - mref) for the
// reference the row already has, kept in registers as bf16 pairs (pk[i] holds
// columns 2i, 2i+1), together with the tile max `mt` and the row sum of P.  The
// caller writes pk over S only when no row of the warp has to move its
// reference (mt > reference + kTau); otherwise it recomputes P with row_exp.
template <int BIAS, bool EDGE, bool DROP = false>
__device__ __forceinline__ float row_exp_1p(const RowCtx& R, float mref, uint32_t (&pk)[BN / 2], float& mt) {
    uint64_t ra = 0, rb = 0;   // two chains of float32 pair sums (even / odd pairs)
    float ma = -INFINITY, mb = -INFINITY;   // and of maxima
    const uint64_t sl2x2 = f2_pack(R.sl2, R.sl2), negm2 = f2_pack(-mref, -mref);
#pragma unroll
    for (int cc = 0; cc < BN / 32; ++cc) {
        uint32_t cur[32];
        tmem_ld32(R.tS + cc * 32, cur);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int col = cc * 32 + 2 * i;
            const float s0 = __uint_as_float(cur[2 * i]), s1 = __uint_as_float(cur[2 * i + 1]);
            float x0, x1;   // x - mref
            float& mx = (i & 1) ? mb : ma;
            if (!BIAS && !EDGE) {
                mx = fmax3(mx, s0, s1);   // scale > 0: max of raw S, scaled once
                f2_unpack(ffma2(f2_pack(s0, s1), sl2x2, negm2), x0, x1);
            } else if (BIAS == 1 && !EDGE) {
                const float2 bp = *reinterpret_cast<const float2*>(R.kbias + col);
                f2_unpack(ffma2(f2_pack(s0, s1), sl2x2, ffma2(f2_pack(bp.x, bp.y), f2_pack(kLog2e, kLog2e), negm2)),
                          x0, x1);
                mx = fmax3(mx, x0, x1);
            } else {
                x0 = score_at<BIAS, EDGE, DROP>(R, cur[2 * i], col) - mref;
                x1 = score_at<BIAS, EDGE, DROP>(R, cur[2 * i + 1], col + 1) - mref;
                mx = fmax3(mx, x0, x1);
            }
            const uint64_t p2 = f2_pack(ex2(x0), ex2(x1));
            if (i & 1)
                rb = fadd2(rb, p2);
            else
                ra = fadd2(ra, p2);
            float p0, p1;
            f2_unpack(p2, p0, p1);
            pk[cc * 16 + i] = pack_bf16(p0, p1);
        }
    }
    const float mx = fmaxf(ma, mb);
    mt = (!BIAS && !EDGE) ? mx * R.sl2 : mx + mref;
    float a0, a1, b0, b1;
    f2_unpack(ra, a0, a1);
    f2_unpack(rb, b0, b1);
    return (a0 + a1) + (b0 + b1);
}

// DROP: the attention-dropout instantiation (a separate kernel, so that the softmax of the
// one without dropout keeps its registers)
template <int D, int DV, int NQ, bool DROP>
__global__ void __launch_bounds__(FwdCfg<D, DV, NQ>::kThreads, NQ == 1 ? 2 : 1)
    k_fwd_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
             const __grid_constant__ CUtensorMap tmV, const FwdArgs a) {
    using C = FwdCfg<D, DV, NQ>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const uint32_t sb = smem_u32(smem);
    const uint32_t bar0 = sb + C::OFF_BAR;
    auto BAR = [&](int i) { return bar0 + 8u * i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + 8 * C::NBAR);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const Problem& P = a.P;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int* item_slot = reinterpret_cast<volatile int*>(tmem_slot + 2);   // two slots
    const int n_items = fwd_items<NQ>(P);

    if (threadIdx.x == 0) {
        mbar_init(BAR(C::B_Q), 1);
        mbar_init(BAR(C::B_QE), 1);
        for (int s = 0; s < C::NSK; ++s) {
            mbar_init(BAR(C::B_KF + s), 1);
            mbar_init(BAR(C::B_KE + s), 1);
        }
        for (int s = 0; s < C::NSV; ++s) {
            mbar_init(BAR(C::B_VF + s), 1);
            mbar_init(BAR(C::B_VE + s), 1);
        }
        for (int i = 0; i < NQ; ++i) {
            mbar_init(BAR(C::B_S + i), 1);
            mbar_init(BAR(C::B_P + i), 128);
            mbar_init(BAR(C::B_O + i), 1);
            mbar_init(BAR(C::B_OE + i), 128);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(BAR(C::B_IF + s), 1);
            mbar_init(BAR(C::B_IE + s), 2 + 4 * NQ);   // V lane, MMA lane, one lane per softmax warp
        }
        mbar_init(BAR(C::B_FIN), 1);
        // a CTA that starts after another one gave up does no work
        *abort_flag = (a.status && (*reinterpret_cast<volatile uint32_t*>(a.status) & ST_TIMEOUT)) ? 1 : 0;
        fence_mbar_init();
    }
    if (warp == C::kMma) {
        tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const bool skip = *abort_flag != 0;
    // a bias that does not depend on the query row (and is contiguous along keys)
    // is staged per key tile in shared memory by the producer
    const bool key_bias = P.bias && P.bs[2] == 0 && P.bs[3] == 1 && (P.S % BN) == 0 &&
                          ((reinterpret_cast<uintptr_t>(P.bias) | ((P.bs[0] | P.bs[1]) * 4)) & 15) == 0;

    // Work items are handed out dynamically (heaviest first): producer lane 0 takes the next
    // one from the global counter and publishes it in slot k % 2; every other role reads it.
    // A value >= n_items ends the loop.  Items whose tiles see no key carry no barrier phases.
    auto read_item = [&](int k, bool arrive) -> int {
        const int sl = k & 1;
        if (!mbar_wait(BAR(C::B_IF + sl), (k >> 1) & 1, abort_flag, a.status, 0x0F)) return n_items;
        const int item = item_slot[sl];
        __syncwarp(__activemask());
        if (arrive) mbar_arrive(BAR(C::B_IE + sl));
        return item;
    };

    if (warp == C::kProducer) {
        // ------------------------------------------------------------ producer
        // lane 0 fetches the work items and streams Q and the K ring (plus the staged key
        // bias), lane 1 the V ring: two independent loops, so no stage count can order them
        // into a wait cycle.  Ring positions continue across items.
        if (lane == 0) {
            tma_prefetch(&tmQ);
            tma_prefetch(&tmK);
            int kw = 0, gk = 0;
            for (int k = 0;; ++k) {
                if (k >= 2 && !mbar_wait(BAR(C::B_IE + (k & 1)), ((k >> 1) - 1) & 1, abort_flag, a.status, 0x0E)) break;
                int item = skip ? n_items : static_cast<int>(atomicAdd(a.sched, 1u));
                if (item > n_items) item = n_items;
                item_slot[k & 1] = item;
                mbar_arrive(BAR(C::B_IF + (k & 1)));
                if (item >= n_items) break;
                const Tile T = decode_tile<NQ>(a, item);
                if (T.n == 0) continue;
                // Q buffers are free once the previous item's S products are done
                if (kw > 0 && !mbar_wait(BAR(C::B_QE), (kw - 1) & 1, abort_flag, a.status, 0x12)) break;
                mbar_expect_tx(BAR(C::B_Q), NQ * C::Q_BYTES);
                for (int i = 0; i < NQ; ++i)
                    for (int sub = 0; sub < D / 64; ++sub)
                        tma_load_4d(sb + C::OFF_Q + i * C::Q_BYTES + sub * C::SUB, &tmQ, BAR(C::B_Q), sub * 64,
                                    T.h + i * T.dh, T.q0 + i * T.dq, T.b);
                ++kw;
                const float* kbias_src = key_bias ? P.bias + T.b * P.bs[0] + T.h * P.bs[1] : nullptr;
                bool ok = true;
                for (int j = 0; j < T.n; ++j, ++gk) {
                    const int st = gk % C::NSK, use = gk / C::NSK;
                    if (use > 0 && !mbar_wait(BAR(C::B_KE + st), (use - 1) & 1, abort_flag, a.status, 0x10)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(BAR(C::B_KF + st), C::KV_BYTES + (key_bias ? BN * 4 : 0));
                    if (key_bias)
                        bulk_load(sb + C::OFF_KB + st * BN * 4, kbias_src + (T.kt0 + j) * BN, BN * 4, BAR(C::B_KF + st));
                    for (int sub = 0; sub < D / 64; ++sub)
                        tma_load_4d(sb + C::OFF_K + st * C::KV_BYTES + sub * C::SUB, &tmK, BAR(C::B_KF + st), sub * 64,
                                    T.hkv, (T.kt0 + j) * BN, T.b);
                }
                if (!ok) break;
            }
            // drain: every copy issued must land before the CTA may exit
            if (kw > 0) drain_wait(BAR(C::B_Q), (kw - 1) & 1, a.status);
            for (int s = 0; s < C::NSK; ++s) {
                const int uses = (gk - s + C::NSK - 1) / C::NSK;
                if (uses > 0) drain_wait(BAR(C::B_KF + s), (uses - 1) & 1, a.status);
            }
        } else if (lane == 1) {
            tma_prefetch(&tmV);
            int gv = 0;
            for (int k = 0;; ++k) {
                const int item = read_item(k, true);
                if (item >= n_items) break;
                const Tile T = decode_tile<NQ>(a, item);
                bool ok = true;
                for (int j = 0; j < T.n; ++j, ++gv) {
                    const int st = gv % C::NSV, use = gv / C::NSV;
                    if (use > 0 && !mbar_wait(BAR(C::B_VE + st), (use - 1) & 1, abort_flag, a.status, 0x11)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(BAR(C::B_VF + st), C::V_BYTES);
                    for (int sub = 0; sub < DV / 64; ++sub)
                        tma_load_4d(sb + C::OFF_V + st * C::V_BYTES + sub * C::SUB, &tmV, BAR(C::B_VF + st), sub * 64,
                                    T.hkv, (T.kt0 + j) * BN, T.b);
                }
                if (!ok) break;
            }
            for (int s = 0; s < C::NSV; ++s) {
                const int uses = (gv - s + C::NSV - 1) / C::NSV;
                if (uses > 0) drain_wait(BAR(C::B_VF + s), (uses - 1) & 1, a.status);
            }
        }
    } else if (warp == C::kMma) {
        // ------------------------------------------------------------ MMA issuer
        {   // the whole warp runs the loop with warp-uniform operands; one elected lane issues
            int np[2] = {0, 0};       // products P_i V consumed per query tile (P barrier phases)
            int kw = 0, gk = 0, gv = 0;
            bool ok = true;
            for (int k = 0; ok; ++k) {
                const int item = __shfl_sync(0xffffffffu, read_item(k, lane == 0), 0);   // warp-uniform
                if (item >= n_items) break;
                const Tile T = decode_tile<NQ>(a, item);
                const int n = T.n;
                if (n == 0) continue;
                auto active = [&](int i, int j) { return j >= T.lo[i] && j <= T.hi[i]; };
                // descriptors are built once per tile and advanced by immediates
                auto issue_s = [&](int i, int j) {
                    const int st = (gk + j) % C::NSK;
                    const uint64_t qd = sdesc_sw128(sb + C::OFF_Q + i * C::Q_BYTES, 16, 1024);
                    const uint64_t kd = sdesc_sw128(sb + C::OFF_K + st * C::KV_BYTES, 16, 1024);
                    const uint32_t d_tmem = tmem + i * BN;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (kk >> 2) * C::SUB + (kk & 3) * 32;
                        tc_mma_ss_w(d_tmem, sdesc_advance(qd, off), sdesc_advance(kd, off), C::IDESC_S, kk > 0);
                    }
                    tc_commit_w(BAR(C::B_S + i));
                };
                auto issue_pv = [&](int i, int j, bool first) {
                    const int st = (gv + j) % C::NSV;
                    const uint64_t vd = sdesc_sw128(sb + C::OFF_V + st * C::V_BYTES, C::SUB, 1024);
                    const uint32_t t_p = tmem + i * BN, t_o = tmem + NQ * BN + i * 128;
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk)
                        tc_mma_ts_w(t_o, t_p + kk * 8, sdesc_advance(vd, kk * 2048), C::IDESC_PV,
                                  (!first || kk > 0) ? 1u : 0u);
                };
                auto wait_k = [&](int j) -> bool {
                    const int pos = gk + j;
                    return __all_sync(0xffffffffu, mbar_wait(BAR(C::B_KF + pos % C::NSK), (pos / C::NSK) & 1, abort_flag, a.status, 0x22)) != 0;
                };
                // O_i of the previous item must have been read by its epilogue before this
                // item's first P_i V overwrites it (waited once per item, in order)
                bool oe_seen[2] = {kw == 0, kw == 0};
                auto wait_oe = [&](int i) -> bool {
                    if (oe_seen[i]) return true;
                    oe_seen[i] = true;
                    return __all_sync(0xffffffffu, mbar_wait(BAR(C::B_OE + i), (kw - 1) & 1, abort_flag, a.status, 0x25)) != 0;
                };
                ok = __all_sync(0xffffffffu, mbar_wait(BAR(C::B_Q), kw & 1, abort_flag, a.status, 0x20)) && wait_k(0);
                if (!ok) break;
                tc_fence_after();
                // the S tiles still hold the previous item's P; its P V products were issued first
                for (int i = 0; i < NQ; ++i)
                    if (active(i, 0)) issue_s(i, 0);
                if (n == 1) tc_commit_w(BAR(C::B_QE));
                int pv_item[2] = {0, 0};
                for (int j = 0; ok && j < n; ++j) {
                    const bool next = j + 1 < n;
                    // every K / V copy is observed here, so a stage is never refilled while a copy is in flight
                    const int vpos = gv + j;
                    if (!__all_sync(0xffffffffu, mbar_wait(BAR(C::B_VF + vpos % C::NSV), (vpos / C::NSV) & 1, abort_flag, a.status, 0x23))) {
                        ok = false;
                        break;
                    }
                    bool k_ready = false;
                    const int last = active(NQ - 1, j) ? NQ - 1 : 0;   // last query tile active at step j
                    bool k_released = false;
                    for (int i = 0; i < NQ; ++i) {
                        if (active(i, j)) {
                            if (!__all_sync(0xffffffffu, mbar_wait(BAR(C::B_P + i), np[i] & 1, abort_flag, a.status, 0x24)) || !wait_oe(i)) {
                                ok = false;
                                break;
                            }
                            // every softmax of step j is done (S(j) and the staged bias are no longer
                            // read): release K_j's stage before S(j+1) may need a free one
                            if (i == last) {
                                tc_commit_w(BAR(C::B_KE + (gk + j) % C::NSK));
                                k_released = true;
                            }
                            tc_fence_after();
                            issue_pv(i, j, pv_item[i] == 0);
                            ++np[i];
                            ++pv_item[i];
                            if (j == T.hi[i]) tc_commit_w(BAR(C::B_O + i));
                        }
                        if (next && active(i, j + 1)) {
                            if (!k_ready) {
                                if (!wait_k(j + 1)) {
                                    ok = false;
                                    break;
                                }
                                k_ready = true;
                                tc_fence_after();
                            }
                            issue_s(i, j + 1);
                        }
                    }
                    if (!ok) break;
                    if (next && !k_ready && !wait_k(j + 1)) {
                        ok = false;
                        break;
                    }
                    if (j + 2 == n) tc_commit_w(BAR(C::B_QE));   // every S of this item is issued
                    if (!k_released) tc_commit_w(BAR(C::B_KE + (gk + j) % C::NSK));   // (a step no tile used)
                    tc_commit_w(BAR(C::B_VE + vpos % C::NSV));   // V_j is no longer read
                }
                if (!ok) break;
                // a query tile without keys in this item still completes its O phase
                for (int i = 0; i < NQ; ++i) {
                    if (T.lo[i] > T.hi[i]) {
                        if (!wait_oe(i)) {
                            ok = false;
                            break;
                        }
                        tc_commit_w(BAR(C::B_O + i));
                    }
                }
                gk += n;
                gv += n;
                ++kw;
            }
            // drain: all MMAs issued by this thread complete before TMEM is freed
            tc_commit_w(BAR(C::B_FIN));
            drain_wait(BAR(C::B_FIN), 0, a.status);
        }
    } else {
        // ------------------------------------------------------------ softmax (rows)
        const int qt = warp >> 2;             // query tile of this warpgroup
        const int t = threadIdx.x & 127;      // row within the tile == TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + qt * BN + lane_base, tO = tmem + NQ * BN + qt * 128 + lane_base;
        const float sl2 = P.scale * kLog2e;
        bool aborted = false;
        int cs = 0, kw = 0, gk = 0;           // S_qt tiles seen, items with work, K ring position
        for (int k = 0; !aborted; ++k) {
            const int item = read_item(k, lane == 0);
            if (item >= n_items) break;
            const Tile T = decode_tile<NQ>(a, item);
            const int q = T.q0 + qt * T.dq + t;
            const int h = T.h + qt * T.dh;        // q head of this warpgroup's tile
            int kmin = T.rlo, kmax = min(T.rhi, P.S - 1);
            if (P.causal) kmax = min(kmax, q + T.off);
            if (P.wr >= 0) kmax = min(kmax, q + T.off + P.wr);
            if (P.wl >= 0) kmin = max(kmin, q + T.off - P.wl);
            if (q >= T.lq) kmax = -1;             // padding row: nothing allowed
            const float* bias_row =
                P.bias ? P.bias + T.b * P.bs[0] + h * P.bs[1] + static_cast<int64_t>(min(q, P.S - 1)) * P.bs[2]
                       : nullptr;
            float m_used = -INFINITY, m_true = -INFINITY, lsum = 0.f;
            const int jlo = T.lo[qt], jhi = T.n > 0 ? T.hi[qt] : -1;
            int c = 0;                            // tiles of this item so far
            for (int j = jlo; j <= jhi; ++j, ++c, ++cs) {
            const int k0 = (T.kt0 + j) * BN;
            if (!__all_sync(0xffffffffu, mbar_wait(BAR(C::B_S + qt), cs & 1, abort_flag, a.status, 0x30))) {
                aborted = true;
                break;
            }
            tc_fence_after();
            const bool edge = __any_sync(0xffffffffu, k0 < kmin || k0 + BN - 1 > kmax);
            const int kpos = gk + j;   // position of K_j in the K ring
            const float* kb_tile = reinterpret_cast<const float*>(smem + C::OFF_KB + (kpos % C::NSK) * BN * 4);
            // the staged key bias arrived with K_j: observe that copy's barrier (the stage
            // cannot be refilled before this warpgroup's P(j) arrival)
            if (key_bias && !__all_sync(0xffffffffu, mbar_wait(BAR(C::B_KF + kpos % C::NSK), (kpos / C::NSK) & 1, abort_flag,
                                                               a.status, 0x34))) {
                aborted = true;
                break;
            }
            RowCtx R{tS, sl2, bias_row, P.bs[3], kb_tile, k0, kmin, kmax, P.S, {0u, 0u, 0u, 0u}};
            // mode = bias kind (0 none, 1 staged key bias, 2 general) * 2 + edge; with attention
            // dropout 6 + bias kind (every tile masked elementwise)
            int mode = (bias_row ? (key_bias ? 2 : 4) : 0) | (edge ? 1 : 0);
            if constexpr (DROP) {
#pragma unroll
                for (int w = 0; w < 4; ++w)
                    R.keep[w] = dropout_keep32(P.drop_thr, P.drop_k0, P.drop_k1, T.b, h, q, k0 + 32 * w);
                mode = 6 + (bias_row ? (key_bias ? 1 : 2) : 0);
            }
            // after the first tile: one pass with the reference the row already has, P kept in
            // registers; stored if no row of the warp has to move its reference
            if (c > 0) {
                const float mref0 = m_used == -INFINITY ? 0.f : m_used;
                float mt1, rs1;
                uint32_t pk[BN / 2];
                if constexpr (DROP) {
                    switch (mode) {
                        case 6: rs1 = row_exp_1p<0, true, true>(R, mref0, pk, mt1); break;
                        case 7: rs1 = row_exp_1p<1, true, true>(R, mref0, pk, mt1); break;
                        default: rs1 = row_exp_1p<2, true, true>(R, mref0, pk, mt1); break;
                    }
                } else switch (mode) {
                    case 0: rs1 = row_exp_1p<0, false>(R, mref0, pk, mt1); break;
                    case 1: rs1 = row_exp_1p<0, true>(R, mref0, pk, mt1); break;
                    case 2: rs1 = row_exp_1p<1, false>(R, mref0, pk, mt1); break;
                    case 3: rs1 = row_exp_1p<1, true>(R, mref0, pk, mt1); break;
                    case 4: rs1 = row_exp_1p<2, false>(R, mref0, pk, mt1); break;
                    default: rs1 = row_exp_1p<2, true>(R, mref0, pk, mt1); break;
                }
                if (!__any_sync(0xffffffffu, mt1 > m_used + kTau)) {
                    m_true = fmaxf(m_true, mt1);
                    tmem_st64(tS, pk);
                    lsum += rs1;
                    tc_fence_before();
                    mbar_arrive(BAR(C::B_P + qt));
                    continue;
                }
            }
            // first tile, or a warp where some row moves its reference: two passes
            float mt;
            if constexpr (DROP) {
                switch (mode) {
                    case 6: mt = row_max<0, true, true>(R); break;
                    case 7: mt = row_max<1, true, true>(R); break;
                    default: mt = row_max<2, true, true>(R); break;
                }
            } else switch (mode) {
                case 0: mt = row_max<0, false>(R); break;
                case 1: mt = row_max<0, true>(R); break;
                case 2: mt = row_max<1, false>(R); break;
                case 3: mt = row_max<1, true>(R); break;
                case 4: mt = row_max<2, false>(R); break;
                default: mt = row_max<2, true>(R); break;
            }
            m_true = fmaxf(m_true, mt);
            // lazy rescale: the reference max only moves when the tile max exceeds it by kTau
            float fac = 1.f;
            bool o_resc = false;
            if (mt > m_used + kTau) {
                fac = m_used == -INFINITY ? 0.f : ex2(m_used - mt);
                o_resc = c > 0 && m_used != -INFINITY;
                m_used = mt;
                lsum *= fac;
            }
            if (__any_sync(0xffffffffu, o_resc)) {
                // S(j) is complete, so every earlier P V has been added to O
                const float f = o_resc ? fac : 1.f;
#pragma unroll 1
                for (int cc = 0; cc < DV / 32; ++cc) {
                    uint32_t r[32];
                    tmem_ld32(tO + cc * 32, r);
#pragma unroll
                    for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * f);
                    tmem_st32(tO + cc * 32, r);
                }
            }
            const float mref = m_used == -INFINITY ? 0.f : m_used;
            float rs;
            if constexpr (DROP) {
                switch (mode) {
                    case 6: rs = row_exp<0, true, true>(R, mref); break;
                    case 7: rs = row_exp<1, true, true>(R, mref); break;
                    default: rs = row_exp<2, true, true>(R, mref); break;
                }
            } else switch (mode) {
                case 0: rs = row_exp<0, false>(R, mref); break;
                case 1: rs = row_exp<0, true>(R, mref); break;
                case 2: rs = row_exp<1, false>(R, mref); break;
                case 3: rs = row_exp<1, true>(R, mref); break;
                case 4: rs = row_exp<2, false>(R, mref); break;
                default: rs = row_exp<2, true>(R, mref); break;
            }
            lsum += rs;
            tc_fence_before();
            mbar_arrive(BAR(C::B_P + qt));
            }
            if (aborted) break;
            if (T.n > 0) {
                // the MMA issuer completes one O phase per item and query tile
                if (!__all_sync(0xffffffffu, mbar_wait(BAR(C::B_O + qt), kw & 1, abort_flag, a.status, 0x33))) {
                    aborted = true;
                    break;
                }
                tc_fence_after();
            }

            // -------------------------------------------------------- epilogue
            const int qc = min(q, P.S - 1);
            const int64_t mi = (static_cast<int64_t>(T.b) * P.Hq + h) * P.S + qc;
            const bool has_work = jlo <= jhi;
            // with a sink every row takes it here; padding rows of variable-length problems get
            // their m, l reset by a pass after the kernel (their O is 0 either way), which keeps
            // the row length out of the live registers
            const bool sink_row = P.sink != nullptr;
            if (!aborted && has_work) {
                tc_fence_after();
                // statistics relative to the true row max
                const float rel = m_true == -INFINITY ? 0.f : ex2(m_used - m_true);
                float l_true = lsum * rel;
                float m_fin = m_true;
                float den = lsum;   // softmax denominator relative to m_used
                if (sink_row) {
                    const float3 r = with_sink(__ldg(P.sink + h), lsum, m_used, m_true);
                    den = r.x;
                    m_fin = r.y;
                    l_true = r.z;
                }
                const float m_nat = m_fin * kLn2;
                if (!a.acc) {
                    const float inv = den > 0.f ? 1.f / den : 0.f;
                    __nv_bfloat16* O = static_cast<__nv_bfloat16*>(a.o) + T.b * P.os[0] +
                                       static_cast<int64_t>(qc) * P.os[1] + h * P.os[2];
                    // whole 32-byte sectors per store where the row allows (fewer, full-sector writes)
                    const bool al32 = (reinterpret_cast<uintptr_t>(O) & 31u) == 0;
    #pragma unroll 1
                    for (int cc = 0; cc < DV / 32; ++cc) {
                        uint32_t r[32];
                        tmem_ld32(tO + cc * 32, r);
                        if (q < P.S) {
                            uint32_t w[16];
    #pragma unroll
                            for (int i = 0; i < 16; ++i)
                                w[i] = pack_bf16(__uint_as_float(r[2 * i]) * inv, __uint_as_float(r[2 * i + 1]) * inv);
                            if (al32) {
                                st_global_v8(O + cc * 32, w);
                                st_global_v8(O + cc * 32 + 16, w + 8);
                            } else {
                                uint4* dst = reinterpret_cast<uint4*>(O + cc * 32);
    #pragma unroll
                                for (int v4 = 0; v4 < 4; ++v4) dst[v4] = make_uint4(w[4 * v4], w[4 * v4 + 1], w[4 * v4 + 2], w[4 * v4 + 3]);
                            }
                        }
                    }
                    if (q < P.S) {
                        a.m[mi] = m_nat;
                        a.l[mi] = l_true;
                    }
                } else {
                    // merge into the ring carry: (m_c, l_c, acc) with (m_nat, l_true, O * rel)
                    float mc = -INFINITY, lc = 0.f;
                    if (q < P.S) {
                        mc = a.m[mi];
                        lc = a.l[mi];
                    }
                    const float mn = fmaxf(mc, m_nat);
                    const float fa = mc == -INFINITY ? 0.f : ex2((mc - mn) * kLog2e);
                    const float fb = m_nat == -INFINITY ? 0.f : ex2((m_nat - mn) * kLog2e) * rel;
                    float* Cr = a.acc + ((static_cast<int64_t>(T.b) * P.S + qc) * P.Hq + h) * DV;
    #pragma unroll 1
                    for (int cc = 0; cc < DV / 32; ++cc) {
                        uint32_t r[32];
                        tmem_ld32(tO + cc * 32, r);
                        if (q < P.S && mn != -INFINITY) {
                            float4* dst = reinterpret_cast<float4*>(Cr + cc * 32);
    #pragma unroll
                            for (int v4 = 0; v4 < 8; ++v4) {
                                float4 x = dst[v4];
                                x.x = x.x * fa + __uint_as_float(r[v4 * 4 + 0]) * fb;
                                x.y = x.y * fa + __uint_as_float(r[v4 * 4 + 1]) * fb;
                                x.z = x.z * fa + __uint_as_float(r[v4 * 4 + 2]) * fb;
                                x.w = x.w * fa + __uint_as_float(r[v4 * 4 + 3]) * fb;
                                dst[v4] = x;
                            }
                        }
                    }
                    if (q < P.S && mn != -INFINITY) {
                        a.m[mi] = mn;
                        a.l[mi] = lc * fa + lsum * fb;
                    }
                }
            } else if (!aborted && !has_work && !a.acc && q < P.S) {
                // no key allowed for this tile: O = 0, m = -inf, l = 0 (with a sink: m = sink, l = 1)
                __nv_bfloat16* O = static_cast<__nv_bfloat16*>(a.o) + T.b * P.os[0] +
                                   static_cast<int64_t>(q) * P.os[1] + h * P.os[2];
                for (int cc = 0; cc < DV; cc += 8) *reinterpret_cast<uint4*>(O + cc) = make_uint4(0, 0, 0, 0);
                a.m[mi] = sink_row ? __ldg(P.sink + h) : -INFINITY;   // only the sink: m = sink, l = 1
                a.l[mi] = sink_row ? 1.f : 0.f;
            }

            if (T.n > 0) {
                // O_qt has been read: the next item's first P V may overwrite it
                tc_fence_before();
                mbar_arrive(BAR(C::B_OE + qt));
                ++kw;
                gk += T.n;
            }
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == C::kMma) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int D, int DV, int NQ, bool DROP>
cudaError_t launch(const FwdArgs& a, const CUtensorMap* maps, cudaStream_t s) {
    using C = FwdCfg<D, DV, NQ>;
    static bool configured[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !configured[dev]) {
        e = cudaFuncSetAttribute(k_fwd_tc<D, DV, NQ, DROP>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) configured[dev] = true;
    }
    // persistent CTAs (one per SM, two for single-tile CTAs) take work items from a counter
    static int sm_count[64] = {};
    int sms = dev >= 0 && dev < 64 ? sm_count[dev] : 0;
    if (sms <= 0) {
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) sm_count[dev] = sms;
    }
    const int64_t items = fwd_items<NQ>(a.P);
    const int grid = static_cast<int>(std::min<int64_t>(items, static_cast<int64_t>(sms) * (NQ == 1 ? 2 : 1)));
    k_fwd_tc<D, DV, NQ, DROP><<<grid, C::kThreads, C::SMEM, s>>>(maps[0], maps[1], maps[2], a);
    return cudaGetLastError();
}

// Key tiles one 128-row query tile visits at most (window and causal bounds).
int key_tiles_per_query_tile(const Problem& P) {
    const int64_t left = P.wl >= 0 ? P.wl : P.S, right = P.causal ? 0 : (P.wr >= 0 ? P.wr : P.S);
    const int64_t span = std::min<int64_t>(P.S, left + right + BM);
    return static_cast<int>((span + BN - 1) / BN) + 1;
}

// Short key ranges take the single-tile CTAs (two per SM); a ring block must hold whole CTAs.
bool fwd_single_tile(const Problem& P) {
    return key_tiles_per_query_tile(P) <= 4 || P.S <= BM || (P.ring_n > 1 && P.ring_blk % (2 * BM));
}

}  // namespace

// The attention-dropout instantiations (fwd_tc_drop.cu).
cudaError_t launch_fwd_tc_dropout(const FwdArgs& a, const CUtensorMap* maps, cudaStream_t s, bool single);

}  // namespace bpa
