// fwd_band.cu - blockwise attention forward for narrow key bands (sliding windows) with
// grouped heads, on the 5th-generation tensor cores (bf16, d = dv = 64 or 128).
//
// A sliding window of at most one tile ("JAX: Single-GPU Attention with TransformerEngine",
// section 1, _make_causal_swa_mask, e.g. window (128, 0)) lets each 128-row query tile see
// at most two 128-key tiles, so per (query tile, head) there is little tensor work and the
// pass is bound by reading Q and writing O.  The general forward (fwd_tc.cuh) spends most
// of such a pass between work items; this kernel is shaped for the band instead:
//   - Work is a static, contiguous share of the (batch, kv head, query tile, head pair)
//     sequence per CTA (one CTA per SM, balanced to one head pair), so no counter and no
//     mailbox: every role walks the same sequence.
//   - The key / value tiles of a (batch, kv head, query tile) stay in shared memory while
//     the G q heads of the group pass through; moving to the next query tile keeps the tile
//     both windows share and loads only the new one.
//   - Query tiles stream through a ring of per-head stages, so the next heads' loads are in
//     flight while the current ones are computed.
//   - Two softmax warpgroups take alternate heads (the two heads of a pair): the tensor core
//     works on one head while the other's softmax and epilogue run.
//   - A head's whole band (both key tiles, 256 keys) is scored at once, so its softmax is one
//     max pass and one exponential pass with the exact row max as the reference: the fold
//     of "bpt.py" scan_kv_block over the band's key blocks, with nothing to rescale.
// TMEM (512 columns): region i = [256 i, 256 i + 256) belongs to warpgroup i: S_i (one or two
// 128-column tiles), then P_i as bf16 pairs over its first 128 columns (read by the P V
// product from TMEM) and O_i in its columns [128, 128 + d), over scores already read.
// Roles (320 threads): warps 0-3 / 4-7 softmax of the pair's first / second head (thread =
// row = TMEM lane), warp 8 TMA producer (lane 0), warp 9 MMA issuer and TMEM owner.
// Every wait is bounded; on a timeout the CTA drains its copies and products, frees TMEM
// and returns.
#include "fwd_tc.cuh"

namespace bpa {
namespace {

template <int D>
struct BandCfg {
    static constexpr int kThreads = 320;
    static constexpr int kProducer = 8, kMma = 9;
    static constexpr int NSQ = D == 128 ? 3 : 6;     // query-tile stages (one head each)
    static constexpr int Q_BYTES = BM * D * 2;
    static constexpr int KV_BYTES = BN * D * 2;
    static constexpr int SUB = 128 * 128;            // one 64-column slab of 128 rows
    static constexpr int OFF_K = 0;                  // two key-tile slots (key tile kt in slot kt % 2)
    static constexpr int OFF_V = OFF_K + 2 * KV_BYTES;
    static constexpr int OFF_Q = OFF_V + 2 * KV_BYTES;
    static constexpr int OFF_BAR = OFF_Q + NSQ * Q_BYTES;
    static constexpr int SMEM = OFF_BAR + 256 + 1024;   // + slack to align the base to 1024
    // barriers: K / V slot full / empty; Q stage full / empty; per softmax warpgroup S ready,
    // P ready, O complete, O drained; final drain
    static constexpr int B_KVF = 0, B_KVE = 2, B_QF = 4, B_QE = 4 + NSQ, B_S = 4 + 2 * NSQ, B_P = B_S + 2,
                         B_O = B_S + 4, B_OE = B_S + 6, B_FIN = B_S + 8, NBAR = B_S + 9;
    static_assert(8 * NBAR + 16 <= 256, "barrier area");
    static_assert(SMEM <= 232448, "shared memory");
    static constexpr uint32_t IDESC_S = idesc_bf16_f32(BM, BN, 0, 0);   // Q, K both K-major
    static constexpr uint32_t IDESC_PV = idesc_bf16_f32(BM, D, 0, 1);   // P (TMEM), V MN-major
};

// One head pair of the sequence: batch entry, kv head, query tile and the pair's first q head.
// Walked incrementally (no 64-bit division per step: the sequence is (b, kv head, query
// tile, pair) with the pair innermost).
struct BandPair {
    int b, hkv, qt, hp;
    int64_t group;    // (batch, kv head, query tile) index
    __device__ __forceinline__ int h0(const Problem& P) const { return hkv * P.G + 2 * hp; }
    __device__ __forceinline__ void init(const Problem& P, int nqt, int64_t u) {
        const int hpg = P.G / 2;
        group = u / hpg;
        hp = static_cast<int>(u % hpg);
        qt = static_cast<int>(group % nqt);
        const int64_t t = group / nqt;
        hkv = static_cast<int>(t % P.Hkv);
        b = static_cast<int>(t / P.Hkv);
    }
    __device__ __forceinline__ void next(const Problem& P, int nqt) {
        if (++hp < P.G / 2) return;
        hp = 0;
        ++group;
        if (++qt < nqt) return;
        qt = 0;
        if (++hkv < P.Hkv) return;
        hkv = 0;
        ++b;
    }
};

// Key tiles query tile qt sees: lo .. lo + n - 1 (the causal / window bounds of its rows).
__host__ __device__ __forceinline__ void band_tiles(int S, int causal, int wl, int wr, int qt, int& lo, int& n) {
    const int q0 = qt * BM, qb = (q0 + BM - 1 < S - 1) ? q0 + BM - 1 : S - 1;
    int klo = 0, khi = S - 1;
    if (causal && qb < khi) khi = qb;
    if (wr >= 0 && qb + wr < khi) khi = qb + wr;
    if (wl >= 0 && q0 - wl > klo) klo = q0 - wl;
    if (klo > khi) {
        lo = 0;
        n = 0;
        return;
    }
    lo = klo / BN;
    n = khi / BN - lo + 1;
}

// Two per-slot (or per-warpgroup) values kept in registers: indexed by branches, not by
// an address, so that no local-memory array is needed.
template <typename T>
struct Two {
    T v0, v1;
    __device__ __forceinline__ T get(int i) const { return i ? v1 : v0; }
    __device__ __forceinline__ void set(int i, T x) {
        if (i) v1 = x;
        else v0 = x;
    }
};

// Slot-resident key tiles: a key tile is identified by (batch, kv head, tile).
__device__ __forceinline__ int64_t tile_key(const Problem& P, int b, int hkv, int kt, int nkt) {
    return (static_cast<int64_t>(b) * P.Hkv + hkv) * nkt + kt;
}

// Softmax passes over one row of the band's scores (one or two 128-key tiles), 32 columns at
// a time (few live registers: a warp runs one chunk after the other).  A chunk whose keys lie
// outside every row of the warp is skipped (its P columns are written as zeros); a chunk
// inside every row's range needs no mask; the others take a per-row bit mask of allowed keys.
// The allowed range [kmin, kmax] of a row never moves left as the row grows, so lane 0 and
// lane 31 hold the warp's extreme bounds and a chunk's kind needs no vote.  The maxima and
// sums run as two independent chains.  Scores are in log2 units, x = S * scale * log2(e).
struct BandRow {
    uint32_t tS;            // TMEM address of this thread's row of S (and of P over it)
    float sl2;              // scale * log2(e)
    int k0, kmin, kmax;     // first key of the band, allowed keys of the row
    int nch;                // 32-column chunks of S (4 per key tile)
    int lo_any, hi_any;     // warp-uniform: the union of the warp's rows' ranges
    int lo_all, hi_all;     // and their intersection
};

__device__ __forceinline__ BandRow band_row(uint32_t tS, float sl2, int k0, int kmin, int kmax, int nch) {
    BandRow R{tS, sl2, k0, kmin, kmax, nch, 0, 0, 0, 0};
    R.lo_any = __shfl_sync(0xffffffffu, kmin, 0);
    R.hi_any = __shfl_sync(0xffffffffu, kmax, 31);
    R.lo_all = __shfl_sync(0xffffffffu, kmin, 31);
    R.hi_all = __shfl_sync(0xffffffffu, kmax, 0);
    return R;
}

// 0: every key of chunk cc is outside every row's range, 1: inside every row's range,
// 2: mixed (warp-uniform)
__device__ __forceinline__ int chunk_kind(const BandRow& R, int cc) {
    const int a = R.k0 + 32 * cc, z = a + 31;
    if (z < R.lo_any || a > R.hi_any) return 0;
    if (a >= R.lo_all && z <= R.hi_all) return 1;
    return 2;
}

// bit i set: key a + i is allowed for this row
__device__ __forceinline__ uint32_t row_bits(const BandRow& R, int a) {
    const int lo = max(R.kmin - a, 0), hi = min(R.kmax - a, 31);
    if (hi < lo) return 0u;
    const uint32_t upto = hi == 31 ? 0xffffffffu : ((1u << (hi + 1)) - 1u);
    return upto & ~((1u << lo) - 1u);
}

// pass 1: the row max (log2 units; -inf if the row allows no key of the band)
__device__ __forceinline__ float band_row_max(const BandRow& R) {
    float m0 = -INFINITY, m1 = -INFINITY;   // of raw S (scale > 0: scaled once at the end)
#pragma unroll 1
    for (int cc = 0; cc < R.nch; ++cc) {
        const int kind = chunk_kind(R, cc);
        if (kind == 0) continue;
        uint32_t r[32];
        tmem_ld32(R.tS + cc * 32, r);
        if (kind == 1) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                m0 = fmax3(m0, __uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]));
                m1 = fmax3(m1, __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
            }
        } else {
            const uint32_t bits = row_bits(R, R.k0 + 32 * cc);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                m0 = fmaxf(m0, (bits >> (2 * i)) & 1u ? __uint_as_float(r[2 * i]) : -INFINITY);
                m1 = fmaxf(m1, (bits >> (2 * i + 1)) & 1u ? __uint_as_float(r[2 * i + 1]) : -INFINITY);
            }
        }
    }
    return fmaxf(m0, m1) * R.sl2;
}

// pass 2: P = exp2(x - mref) as bf16 pairs over the first 16 nch columns of the row (chunk
// cc reads S columns [32cc, 32cc + 32) and writes P columns [16cc, 16cc + 16), which were
// read by this or an earlier chunk); returns the row sum of P
__device__ __forceinline__ float band_row_exp(const BandRow& R, float mref) {
    const uint64_t sl2x2 = f2_pack(R.sl2, R.sl2), negm2 = f2_pack(-mref, -mref);
    uint64_t ra = 0, rb = 0;   // two chains of float32 pair sums
#pragma unroll 1
    for (int cc = 0; cc < R.nch; ++cc) {
        const int kind = chunk_kind(R, cc);
        uint32_t pk[16];
        if (kind == 0) {
#pragma unroll
            for (int i = 0; i < 16; ++i) pk[i] = 0u;
        } else {
            uint32_t r[32];
            tmem_ld32(R.tS + cc * 32, r);
            const uint32_t bits = kind == 1 ? 0xffffffffu : row_bits(R, R.k0 + 32 * cc);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                float x0, x1;
                f2_unpack(ffma2(f2_pack(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), sl2x2, negm2), x0,
                          x1);
                x0 = (bits >> (2 * i)) & 1u ? x0 : -INFINITY;
                x1 = (bits >> (2 * i + 1)) & 1u ? x1 : -INFINITY;
                const uint64_t p2 = f2_pack(ex2(x0), ex2(x1));
                if (i & 1)
                    rb = fadd2(rb, p2);
                else
                    ra = fadd2(ra, p2);
                float p0, p1;
                f2_unpack(p2, p0, p1);
                pk[i] = pack_bf16(p0, p1);
            }
        }
        tmem_st16_nowait(R.tS + cc * 16, pk);
    }
    tmem_st_wait();
    float a0, a1, b0, b1;
    f2_unpack(ra, a0, a1);
    f2_unpack(rb, b0, b1);
    return (a0 + a1) + (b0 + b1);
}

template <int D>
__global__ void __launch_bounds__(BandCfg<D>::kThreads, 1)
    k_fwd_band(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const FwdArgs a) {
    using C = BandCfg<D>;
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
    const int nqt = (P.S + BM - 1) / BM, nkt = (P.S + BN - 1) / BN;
    const int64_t total = static_cast<int64_t>(P.B) * P.Hkv * nqt * (P.G / 2);
    const int64_t u0 = total * blockIdx.x / gridDim.x, u1 = total * (blockIdx.x + 1) / gridDim.x;

    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(BAR(C::B_KVF + s), 1);
            mbar_init(BAR(C::B_KVE + s), 1);
        }
        for (int s = 0; s < C::NSQ; ++s) {
            mbar_init(BAR(C::B_QF + s), 1);
            mbar_init(BAR(C::B_QE + s), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(BAR(C::B_S + i), 1);
            mbar_init(BAR(C::B_P + i), 128);
            mbar_init(BAR(C::B_O + i), 1);
            mbar_init(BAR(C::B_OE + i), 128);
        }
        mbar_init(BAR(C::B_FIN), 1);
        // a CTA that starts after another one gave up does no work
        *abort_flag = (a.status && (*reinterpret_cast<volatile uint32_t*>(a.status) & ST_TIMEOUT)) ? 1 : 0;
        fence_mbar_init();
    }
    if (warp == C::kMma) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const bool skip = *abort_flag != 0;
    const int64_t uend = skip ? u0 : u1;

    if (warp == C::kProducer) {
        // ------------------------------------------------------------ producer (lane 0)
        // K / V tiles when the (batch, kv head, query tile) changes and a needed tile is not
        // resident; the two query tiles of every pair through the stage ring.  A slot is
        // refilled only after the MMA issuer released its previous tile (one release per
        // occupancy, so at most one release is ever outstanding per slot).
        if (lane == 0) {
            tma_prefetch(&tmQ);
            tma_prefetch(&tmK);
            tma_prefetch(&tmV);
            Two<int64_t> res{-1, -1};
            Two<int> loads{0, 0};
            int64_t prev_group = -1;
            int qpos = 0;
            bool ok = true;
            BandPair T;
            T.init(P, nqt, u0);
            for (int64_t u = u0; ok && u < uend; ++u, T.next(P, nqt)) {
                // the pair's two query tiles first: they never wait on a key-tile release
                for (int i = 0; i < 2; ++i, ++qpos) {
                    const int st = qpos % C::NSQ, use = qpos / C::NSQ;
                    if (use > 0 && !mbar_wait(BAR(C::B_QE + st), (use - 1) & 1, abort_flag, a.status, 0x81)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(BAR(C::B_QF + st), C::Q_BYTES);
                    for (int sub = 0; sub < D / 64; ++sub)
                        tma_load_4d(sb + C::OFF_Q + st * C::Q_BYTES + sub * C::SUB, &tmQ, BAR(C::B_QF + st), sub * 64,
                                    T.h0(P) + i, T.qt * BM, T.b);
                }
                if (!ok || T.group == prev_group) continue;
                prev_group = T.group;
                int lo, n;
                band_tiles(P.S, P.causal, P.wl, P.wr, T.qt, lo, n);
                for (int j = 0; j < n; ++j) {
                    const int kt = lo + j, s = kt & 1;
                    const int64_t key = tile_key(P, T.b, T.hkv, kt, nkt);
                    if (res.get(s) == key) continue;
                    if (loads.get(s) > 0 &&
                        !mbar_wait(BAR(C::B_KVE + s), (loads.get(s) - 1) & 1, abort_flag, a.status, 0x80)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(BAR(C::B_KVF + s), 2 * C::KV_BYTES);
                    for (int sub = 0; sub < D / 64; ++sub) {
                        tma_load_4d(sb + C::OFF_K + s * C::KV_BYTES + sub * C::SUB, &tmK, BAR(C::B_KVF + s), sub * 64,
                                    T.hkv, kt * BN, T.b);
                        tma_load_4d(sb + C::OFF_V + s * C::KV_BYTES + sub * C::SUB, &tmV, BAR(C::B_KVF + s), sub * 64,
                                    T.hkv, kt * BN, T.b);
                    }
                    res.set(s, key);
                    loads.set(s, loads.get(s) + 1);
                }
            }
            // drain: every copy issued must land before the CTA may exit
            for (int s = 0; s < 2; ++s)
                if (loads.get(s) > 0) drain_wait(BAR(C::B_KVF + s), (loads.get(s) - 1) & 1, a.status);
            for (int st = 0; st < C::NSQ; ++st) {
                const int uses = (qpos - st + C::NSQ - 1) / C::NSQ;
                if (uses > 0) drain_wait(BAR(C::B_QF + st), (uses - 1) & 1, a.status);
            }
        }
    } else if (warp == C::kMma) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs the loop with warp-uniform operands; one elected lane issues.
        // Per pair (heads t0 = 2p, t1 = 2p + 1 of the CTA's sequence, warpgroups 0, 1):
        //   [region i drained]  S_i = Q_i [K_lo .. K_lo+n-1]^T  (one N = 128 product per key tile)
        //   [P_i ready]         O_i = P_i [V_lo .. V_lo+n-1]
        // for i = 0, 1.  Region i holds S_i, then P_i over its first 128 columns and O_i in
        // columns [128, 128 + d): P_i V reads P_i and writes O_i over scores the softmax has read.
        Two<int64_t> res{-1, -1};
        Two<int> loads{0, 0};
        Two<int> seen{0, 0};           // slot loads whose arrival has been observed
        int64_t prev_group = -1;
        int qpos = 0, pair = 0;
        bool ok = true;
        int lo = 0, n = 0;
        BandPair T;
        T.init(P, nqt, u0);
        for (int64_t u = u0; ok && u < uend; ++u, ++pair, T.next(P, nqt)) {
            if (T.group != prev_group) {
                prev_group = T.group;
                band_tiles(P.S, P.causal, P.wl, P.wr, T.qt, lo, n);
                for (int j = 0; j < n; ++j) {
                    const int kt = lo + j, s = kt & 1;
                    const int64_t key = tile_key(P, T.b, T.hkv, kt, nkt);
                    if (res.get(s) != key) {
                        res.set(s, key);
                        loads.set(s, loads.get(s) + 1);
                    }
                }
            }
            // The last pair of its group releases each slot whose tile the next group does not
            // keep, right after the last product that reads it.
            BandPair N = T;
            N.next(P, nqt);
            Two<bool> release{false, false};
            if (u + 1 < uend && N.group != T.group) {
                int nlo, nn;
                band_tiles(P.S, P.causal, P.wl, P.wr, N.qt, nlo, nn);
                for (int j = 0; j < n; ++j) {
                    bool kept = false;
                    for (int jj = 0; jj < nn; ++jj)
                        kept = kept || tile_key(P, N.b, N.hkv, nlo + jj, nkt) == tile_key(P, T.b, T.hkv, lo + j, nkt);
                    release.set(j, !kept);
                }
            }
            // key tile j has landed (each load is observed once, before its first product)
            auto ensure_tile = [&](int j) -> bool {
                const int s = (lo + j) & 1;
                while (seen.get(s) < loads.get(s)) {
                    if (!__all_sync(0xffffffffu, mbar_wait(BAR(C::B_KVF + s), seen.get(s) & 1, abort_flag, a.status, 0x90)))
                        return false;
                    seen.set(s, seen.get(s) + 1);
                }
                return true;
            };
            const Two<int> stq{qpos % C::NSQ, (qpos + 1) % C::NSQ};
            for (int i = 0; ok && i < 2; ++i) {
                ok = __all_sync(0xffffffffu,
                                mbar_wait(BAR(C::B_QF + stq.get(i)), ((qpos + i) / C::NSQ) & 1, abort_flag, a.status, 0x91 + i));
                for (int j = 0; ok && j < n; ++j) ok = ensure_tile(j);
                // the previous pair's epilogue must have read O_i before S_i overwrites region i
                if (ok && pair > 0)
                    ok = __all_sync(0xffffffffu, mbar_wait(BAR(C::B_OE + i), (pair - 1) & 1, abort_flag, a.status, 0x94));
                if (!ok) break;
                tc_fence_after();
                const uint64_t qd = sdesc_sw128(sb + C::OFF_Q + stq.get(i) * C::Q_BYTES, 16, 1024);
                for (int j = 0; j < n; ++j) {
                    const uint64_t kd = sdesc_sw128(sb + C::OFF_K + ((lo + j) & 1) * C::KV_BYTES, 16, 1024);
                    const uint32_t d_tmem = tmem + i * 256 + j * BN;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (kk >> 2) * C::SUB + (kk & 3) * 32;
                        tc_mma_ss_w(d_tmem, sdesc_advance(qd, off), sdesc_advance(kd, off), C::IDESC_S, kk > 0);
                    }
                }
                tc_commit_w(BAR(C::B_S + i));
                tc_commit_w(BAR(C::B_QE + stq.get(i)));   // the head's only score product
            }
            for (int i = 0; ok && i < 2; ++i) {
                ok = __all_sync(0xffffffffu, mbar_wait(BAR(C::B_P + i), pair & 1, abort_flag, a.status, 0x93));
                if (!ok) break;
                tc_fence_after();
                const uint32_t t_r = tmem + i * 256;
                for (int j = 0; j < n; ++j) {
                    const uint64_t vd = sdesc_sw128(sb + C::OFF_V + ((lo + j) & 1) * C::KV_BYTES, C::SUB, 1024);
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk)
                        tc_mma_ts_w(t_r + 128, t_r + j * (BN / 2) + kk * 8, sdesc_advance(vd, kk * 2048), C::IDESC_PV,
                                    (j > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit_w(BAR(C::B_O + i));
            }
            if (ok)
                for (int j = 0; j < n; ++j)
                    if (release.get(j)) tc_commit_w(BAR(C::B_KVE + ((lo + j) & 1)));
            qpos += 2;
        }
        // drain: all MMAs issued by this warp complete before TMEM is freed
        tc_commit_w(BAR(C::B_FIN));
        drain_wait(BAR(C::B_FIN), 0, a.status);
    } else {
        // ------------------------------------------------------------ softmax (rows)
        const int wg = warp >> 2;             // head of the pair taken by this warpgroup
        const int t = threadIdx.x & 127;      // row within the query tile == TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + wg * 256 + lane_base, tO = tS + 128;
        const float sl2 = P.scale * kLog2e;
        bool aborted = false;
        int pair = 0;
        BandPair T;
        T.init(P, nqt, u0);
        for (int64_t u = u0; !aborted && u < uend; ++u, ++pair, T.next(P, nqt)) {
            const int h = T.h0(P) + wg;
            const int q = T.qt * BM + t;
            int lo, n;
            band_tiles(P.S, P.causal, P.wl, P.wr, T.qt, lo, n);
            int kmin = 0, kmax = P.S - 1;
            if (P.causal) kmax = min(kmax, q);
            if (P.wr >= 0) kmax = min(kmax, q + P.wr);
            if (P.wl >= 0) kmin = max(kmin, q - P.wl);
            if (!__all_sync(0xffffffffu, mbar_wait(BAR(C::B_S + wg), pair & 1, abort_flag, a.status, 0xA0))) {
                aborted = true;
                break;
            }
            tc_fence_after();
            // the whole band in one S: two passes, the row max, then P with it as the reference
            const BandRow R = band_row(tS, sl2, lo * BN, kmin, kmax, n * (BN / 32));
            const float mt = band_row_max(R);
            const float lsum = band_row_exp(R, mt == -INFINITY ? 0.f : mt);
            tc_fence_before();
            mbar_arrive(BAR(C::B_P + wg));
            // ------------------------------------------------------------ epilogue
            if (!__all_sync(0xffffffffu, mbar_wait(BAR(C::B_O + wg), pair & 1, abort_flag, a.status, 0xA1))) {
                aborted = true;
                break;
            }
            tc_fence_after();
            const int qc = min(q, P.S - 1);
            const int64_t mi = (static_cast<int64_t>(T.b) * P.Hq + h) * P.S + qc;
            const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
            __nv_bfloat16* O = static_cast<__nv_bfloat16*>(a.o) + T.b * P.os[0] + static_cast<int64_t>(qc) * P.os[1] +
                               h * P.os[2];
            const bool al32 = (reinterpret_cast<uintptr_t>(O) & 31u) == 0;
#pragma unroll 1
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t r[32];
                tmem_ld32(tO + cc * 32, r);
                if (cc == D / 32 - 1) {
                    // every column of O_wg has been read: the next pair's S may overwrite the region
                    tc_fence_before();
                    mbar_arrive(BAR(C::B_OE + wg));
                }
                if (q < P.S) {
                    uint32_t w[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        w[i] = pack_bf16(__uint_as_float(r[2 * i]) * inv, __uint_as_float(r[2 * i + 1]) * inv);
                    if (al32) {   // whole 32-byte sectors per store
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
                a.m[mi] = mt == -INFINITY ? -INFINITY : mt * kLn2;
                a.l[mi] = lsum;
            }
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == C::kMma) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int D>
cudaError_t launch_band(const FwdArgs& a, const CUtensorMap* maps, cudaStream_t s) {
    using C = BandCfg<D>;
    static bool configured[64] = {};
    static int sm_count[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !configured[dev]) {
        e = cudaFuncSetAttribute(k_fwd_band<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) configured[dev] = true;
    }
    int sms = dev >= 0 && dev < 64 ? sm_count[dev] : 0;
    if (sms <= 0) {
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) sm_count[dev] = sms;
    }
    const Problem& P = a.P;
    const int nqt = (P.S + BM - 1) / BM;
    const int64_t pairs = static_cast<int64_t>(P.B) * P.Hkv * nqt * (P.G / 2);
    const int grid = static_cast<int>(std::min<int64_t>(pairs, sms));
    k_fwd_band<D><<<grid, C::kThreads, C::SMEM, s>>>(maps[0], maps[1], maps[2], a);
    return cudaGetLastError();
}

}  // namespace

bool fwd_band_supported(const Problem& P) {
    if (P.dtype != BPA_BF16 || P.d != P.dv || (P.d != 64 && P.d != 128)) return false;
    if (P.ring_n != 1 || P.block_idx || P.seqlens_q || P.seqlens_kv || P.bias || P.sink || P.drop_thr) return false;
    if (P.G % 2) return false;
    // every query tile must see one or two key tiles (a window of at most one tile)
    const int nqt = (P.S + BM - 1) / BM;
    for (int qt = 0; qt < nqt; ++qt) {
        int lo, n;
        band_tiles(P.S, P.causal, P.wl, P.wr, qt, lo, n);
        if (n < 1 || n > 2) return false;
    }
    return true;
}

cudaError_t launch_fwd_band(const FwdArgs& a, const CUtensorMap* maps, cudaStream_t s) {
    return a.P.d == 128 ? launch_band<128>(a, maps, s) : launch_band<64>(a, maps, s);
}

}  // namespace bpa
