// fwd_tc.cu - blockwise attention forward on the 5th-generation tensor cores (bf16, d = 64 / 128).
//
// One CTA owns one 128-row query tile of one (batch, q head) and walks the
// 128-key tiles its mask allows, folding each into a running
// (max, numerator, denominator) carry ("bpt.py", _blockwise_attention_fwd /
// scan_kv_block):
//     m' = max(m, rowmax S);  P = exp(S - m');  num = num * exp(m - m') + P V;
//     den = den * exp(m - m') + rowsum P
// Roles (192 threads):
//   warps 0-3  softmax: thread t owns query row t (TMEM lane t); reads S from
//              TMEM, applies scale / bias / mask, keeps the row statistics,
//              writes P (bf16) to shared memory, rescales O when needed;
//   warp 4     TMA producer: Q once, then K / V tiles through an NS-stage ring;
//   warp 5     MMA issuer (one thread): S = Q K^T into a double-buffered TMEM
//              tile, O += P V into a TMEM accumulator; owns the TMEM allocation.
// The numerator is rescaled lazily: the reference max only moves when a row's
// max grows by more than kTau (log2 units), which is exact in real arithmetic
// because numerator and denominator share the reference.
// Fully masked tiles are never visited (the key range is cut by position);
// only tiles that straddle a mask edge apply the elementwise mask.
// Every wait is bounded (see common.cuh); on a timeout the CTA drains its
// in-flight copies and MMAs, frees TMEM and returns.
#include <math.h>

#include "bpa_internal.h"
#include "common.cuh"

namespace bpa {
namespace {

constexpr int BM = 128;       // query rows per tile
constexpr int BN = 128;       // keys per tile
constexpr float kTau = 8.f;   // lazy-rescale threshold, log2 units
constexpr int kThreads = 192;

template <int D>
struct FwdCfg {
    static constexpr int NS = D == 128 ? 2 : 4;    // K/V pipeline stages
    static constexpr int Q_BYTES = BM * D * 2;
    static constexpr int KV_BYTES = BN * D * 2;
    static constexpr int P_BYTES = BM * BN * 2;
    static constexpr int SUB = 128 * 128;          // one 64-column slab of 128 rows
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + Q_BYTES;
    static constexpr int OFF_V = OFF_K + NS * KV_BYTES;
    static constexpr int OFF_P = OFF_V + NS * KV_BYTES;
    static constexpr int OFF_BAR = OFF_P + 2 * P_BYTES;
    static constexpr int SMEM = OFF_BAR + 256 + 1024;   // + slack to align the base to 1024
    // barrier slots
    static constexpr int B_Q = 0, B_K = 1, B_V = 1 + NS, B_E = 1 + 2 * NS, B_S = 1 + 3 * NS,
                         B_P = 3 + 3 * NS, B_PV = 5 + 3 * NS, B_FIN = 7 + 3 * NS,
                         NBAR = 8 + 3 * NS;
    static constexpr uint32_t IDESC_S = idesc_bf16_f32(BM, BN, 0, 0);   // Q, K both K-major
    static constexpr uint32_t IDESC_PV = idesc_bf16_f32(BM, D, 0, 1);   // P K-major, V MN-major
};

struct Tile {
    int b, h, hkv, q0, kt_lo, n_kv;
    int rlo, rhi;   // key range of this launch (ring super-block or whole sequence)
};

__device__ __forceinline__ Tile decode_tile(const FwdArgs& a) {
    const Problem& P = a.P;
    const int nqt = (P.S + BM - 1) / BM;
    int r = blockIdx.x;
    const int gi = r % P.G;
    r /= P.G;
    Tile t;
    t.hkv = r % P.Hkv;
    r /= P.Hkv;
    t.b = r % P.B;
    const int qt = nqt - 1 - r / P.B;   // heaviest (causal) tiles first
    t.h = t.hkv * P.G + gi;
    t.q0 = qt * BM;
    const int q_last = min(t.q0 + BM - 1, P.S - 1);
    t.rlo = 0;
    t.rhi = P.S - 1;
    if (a.acc) {
        const int i = t.q0 / P.ring_blk;
        const int j = ((i - a.ring_idx) % P.ring_n + P.ring_n) % P.ring_n;
        t.rlo = j * P.ring_blk;
        t.rhi = t.rlo + P.ring_blk - 1;
    }
    int lo = t.rlo, hi = t.rhi;
    if (P.causal) hi = min(hi, q_last);
    if (P.wr >= 0) hi = min(hi, q_last + P.wr);
    if (P.wl >= 0) lo = max(lo, t.q0 - P.wl);
    t.kt_lo = lo / BN;
    t.n_kv = lo <= hi ? hi / BN - t.kt_lo + 1 : 0;
    return t;
}

// bounded wait that ignores the abort flag: used to drain in-flight work
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint32_t* status) {
    int never = 0;
    mbar_wait(bar, parity, &never, status, 0xD0);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    k_fwd_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
             const __grid_constant__ CUtensorMap tmV, const FwdArgs a) {
    using C = FwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const uint32_t sb = smem_u32(smem);
    const uint32_t bar0 = sb + C::OFF_BAR;
    auto BAR = [&](int i) { return bar0 + 8u * i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + 8 * C::NBAR);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const Problem& P = a.P;
    const Tile T = decode_tile(a);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(BAR(C::B_Q), 1);
        for (int s = 0; s < C::NS; ++s) {
            mbar_init(BAR(C::B_K + s), 1);
            mbar_init(BAR(C::B_V + s), 1);
            mbar_init(BAR(C::B_E + s), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(BAR(C::B_S + i), 1);
            mbar_init(BAR(C::B_P + i), 128);
            mbar_init(BAR(C::B_PV + i), 1);
        }
        mbar_init(BAR(C::B_FIN), 1);
        // a CTA that starts after another one gave up does no work
        *abort_flag = (a.status && (*reinterpret_cast<volatile uint32_t*>(a.status) & ST_TIMEOUT)) ? 1 : 0;
        fence_mbar_init();
    }
    if (warp == 5) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tS0 = tmem, tO = tmem + 256;
    const int n_kv = *abort_flag ? 0 : T.n_kv;
    const bool skip = *abort_flag != 0;

    if (warp == 4) {
        // ------------------------------------------------------------ producer
        if (lane == 0 && n_kv > 0) {
            tma_prefetch(&tmQ);
            tma_prefetch(&tmK);
            tma_prefetch(&tmV);
            mbar_expect_tx(BAR(C::B_Q), C::Q_BYTES);
            for (int sub = 0; sub < D / 64; ++sub)
                tma_load_4d(sb + C::OFF_Q + sub * C::SUB, &tmQ, BAR(C::B_Q), sub * 64, T.h, T.q0, T.b);
            int n_issued = 0;   // tiles whose loads were issued
            for (int j = 0; j < n_kv; ++j) {
                const int st = j % C::NS, use = j / C::NS;
                if (use > 0 && !mbar_wait(BAR(C::B_E + st), (use - 1) & 1, abort_flag, a.status, 0x10))
                    break;
                const int k0 = (T.kt_lo + j) * BN;
                mbar_expect_tx(BAR(C::B_K + st), C::KV_BYTES);
                for (int sub = 0; sub < D / 64; ++sub)
                    tma_load_4d(sb + C::OFF_K + st * C::KV_BYTES + sub * C::SUB, &tmK, BAR(C::B_K + st),
                                sub * 64, T.hkv, k0, T.b);
                mbar_expect_tx(BAR(C::B_V + st), C::KV_BYTES);
                for (int sub = 0; sub < D / 64; ++sub)
                    tma_load_4d(sb + C::OFF_V + st * C::KV_BYTES + sub * C::SUB, &tmV, BAR(C::B_V + st),
                                sub * 64, T.hkv, k0, T.b);
                n_issued = j + 1;
            }
            // drain: every copy issued must land before the CTA may exit
            drain_wait(BAR(C::B_Q), 0, a.status);
            for (int s = 0; s < C::NS; ++s) {
                const int uses = (n_issued - s + C::NS - 1) / C::NS;   // loads issued into stage s
                if (uses > 0) {
                    drain_wait(BAR(C::B_K + s), (uses - 1) & 1, a.status);
                    drain_wait(BAR(C::B_V + s), (uses - 1) & 1, a.status);
                }
            }
        }
    } else if (warp == 5) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && n_kv > 0) {
            auto issue_s = [&](int j) {
                const int st = j % C::NS;
                const uint32_t q_base = sb + C::OFF_Q, k_base = sb + C::OFF_K + st * C::KV_BYTES;
                const uint32_t d_tmem = tS0 + (j & 1) * BN;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * C::SUB + (kk & 3) * 32;
                    tc_mma_ss(d_tmem, sdesc_sw128(q_base + off, 16, 1024),
                              sdesc_sw128(k_base + off, 16, 1024), C::IDESC_S, kk > 0);
                }
                tc_commit(BAR(C::B_S + (j & 1)));
            };
            bool ok = mbar_wait(BAR(C::B_Q), 0, abort_flag, a.status, 0x20) &&
                      mbar_wait(BAR(C::B_K), 0, abort_flag, a.status, 0x21);
            if (ok) {
                tc_fence_after();
                issue_s(0);
            }
            for (int j = 0; ok && j < n_kv; ++j) {
                if (j + 1 < n_kv) {
                    const int st1 = (j + 1) % C::NS;
                    if (!mbar_wait(BAR(C::B_K + st1), ((j + 1) / C::NS) & 1, abort_flag, a.status, 0x22))
                        break;
                    tc_fence_after();
                    issue_s(j + 1);
                }
                const int st = j % C::NS;
                if (!mbar_wait(BAR(C::B_V + st), (j / C::NS) & 1, abort_flag, a.status, 0x23)) break;
                if (!mbar_wait(BAR(C::B_P + (j & 1)), (j >> 1) & 1, abort_flag, a.status, 0x24)) break;
                tc_fence_after();
                const uint32_t p_base = sb + C::OFF_P + (j & 1) * C::P_BYTES;
                const uint32_t v_base = sb + C::OFF_V + st * C::KV_BYTES;
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    const uint64_t ad = sdesc_sw128(p_base + (kk >> 2) * C::SUB + (kk & 3) * 32, 16, 1024);
                    const uint64_t bd = sdesc_sw128(v_base + kk * 2048, C::SUB, 1024);
                    tc_mma_ss(tO, ad, bd, C::IDESC_PV, (j > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(BAR(C::B_E + st));
                tc_commit(BAR(C::B_PV + (j & 1)));
            }
            // drain: all MMAs issued by this thread complete before TMEM is freed
            tc_commit(BAR(C::B_FIN));
            drain_wait(BAR(C::B_FIN), 0, a.status);
        }
    } else {
        // ------------------------------------------------------------ softmax (rows)
        const int t = threadIdx.x;            // row within the tile == TMEM lane
        const int q = T.q0 + t;
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        int kmin = T.rlo, kmax = min(T.rhi, P.S - 1);
        if (P.causal) kmax = min(kmax, q);
        if (P.wr >= 0) kmax = min(kmax, q + P.wr);
        if (P.wl >= 0) kmin = max(kmin, q - P.wl);
        if (q >= P.S) kmax = -1;              // padding row: nothing allowed
        const float sl2 = P.scale * kLog2e;
        const float* bias_row =
            P.bias ? P.bias + T.b * P.bs[0] + T.h * P.bs[1] + static_cast<int64_t>(min(q, P.S - 1)) * P.bs[2]
                   : nullptr;
        float m_used = -INFINITY, m_true = -INFINITY, lsum = 0.f;
        bool aborted = false;
        for (int j = 0; j < n_kv; ++j) {
            const int bsel = j & 1;
            const int k0 = (T.kt_lo + j) * BN;
            if (!__all_sync(0xffffffffu, mbar_wait(BAR(C::B_S + bsel), (j >> 1) & 1, abort_flag, a.status, 0x30))) {
                aborted = true;
                break;
            }
            tc_fence_after();
            float s[BN];
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(tS0 + bsel * BN + c * 32 + lane_base, r);
#pragma unroll
                for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(r[i]) * sl2;
            }
            if (bias_row) {
#pragma unroll
                for (int i = 0; i < BN; ++i) {
                    const int k = min(k0 + i, P.S - 1);
                    s[i] = fmaf(bias_row[k * P.bs[3]], kLog2e, s[i]);
                }
            }
            const bool edge = k0 < kmin || k0 + BN - 1 > kmax;
            if (__any_sync(0xffffffffu, edge)) {
#pragma unroll
                for (int i = 0; i < BN; ++i) {
                    const int k = k0 + i;
                    if (k < kmin || k > kmax) s[i] = -INFINITY;
                }
            }
            float mt = -INFINITY;
#pragma unroll
            for (int i = 0; i < BN; ++i) mt = fmaxf(mt, s[i]);
            m_true = fmaxf(m_true, mt);
            float fac = 1.f;
            bool o_resc = false;
            if (mt > m_used + kTau) {
                fac = m_used == -INFINITY ? 0.f : ex2(m_used - mt);
                o_resc = j > 0 && m_used != -INFINITY;
                m_used = mt;
                lsum *= fac;
            }
            if (__any_sync(0xffffffffu, o_resc)) {
                // O must hold every earlier P V before it is rescaled
                if (!__all_sync(0xffffffffu, mbar_wait(BAR(C::B_PV + ((j - 1) & 1)), ((j - 1) >> 1) & 1,
                                                       abort_flag, a.status, 0x31))) {
                    aborted = true;
                    break;
                }
                tc_fence_after();
                const float f = o_resc ? fac : 1.f;
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld32(tO + c * 32 + lane_base, r);
#pragma unroll
                    for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * f);
                    tmem_st32(tO + c * 32 + lane_base, r);
                }
            }
            const float mref = m_used == -INFINITY ? 0.f : m_used;
            float rs = 0.f;
#pragma unroll
            for (int i = 0; i < BN; ++i) {
                s[i] = ex2(s[i] - mref);
                rs += s[i];
            }
            lsum += rs;
            // the P buffer is free once the P V that read it two tiles ago is done
            if (j >= 2 && !__all_sync(0xffffffffu, mbar_wait(BAR(C::B_PV + bsel), ((j - 2) >> 1) & 1,
                                                              abort_flag, a.status, 0x32))) {
                aborted = true;
                break;
            }
            const uint32_t p_base = sb + C::OFF_P + bsel * C::P_BYTES;
#pragma unroll
            for (int cc = 0; cc < BN / 8; ++cc) {
                const uint32_t addr = p_base + (cc >> 3) * C::SUB + sw128_offset(t, cc & 7);
                st_shared_v4(addr, pack_bf16(s[cc * 8 + 0], s[cc * 8 + 1]),
                             pack_bf16(s[cc * 8 + 2], s[cc * 8 + 3]),
                             pack_bf16(s[cc * 8 + 4], s[cc * 8 + 5]),
                             pack_bf16(s[cc * 8 + 6], s[cc * 8 + 7]));
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(BAR(C::B_P + bsel));
        }

        // ------------------------------------------------------------ epilogue
        const int64_t mi = (static_cast<int64_t>(T.b) * P.Hq + T.h) * P.S + q;
        if (!aborted && n_kv > 0 &&
            __all_sync(0xffffffffu, mbar_wait(BAR(C::B_PV + ((n_kv - 1) & 1)), ((n_kv - 1) >> 1) & 1,
                                              abort_flag, a.status, 0x33))) {
            tc_fence_after();
            // statistics relative to the true row max
            const float rel = m_true == -INFINITY ? 0.f : ex2(m_used - m_true);
            const float l_true = lsum * rel;
            const float m_nat = m_true * kLn2;
            if (!a.acc) {
                const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
                __nv_bfloat16* O = static_cast<__nv_bfloat16*>(a.o) + T.b * P.qs[0] +
                                   static_cast<int64_t>(q) * P.qs[1] + T.h * P.qs[2];
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld32(tO + c * 32 + lane_base, r);
                    if (q < P.S) {
                        uint4* dst = reinterpret_cast<uint4*>(O + c * 32);
#pragma unroll
                        for (int v4 = 0; v4 < 4; ++v4) {
                            uint4 w;
                            w.x = pack_bf16(__uint_as_float(r[v4 * 8 + 0]) * inv, __uint_as_float(r[v4 * 8 + 1]) * inv);
                            w.y = pack_bf16(__uint_as_float(r[v4 * 8 + 2]) * inv, __uint_as_float(r[v4 * 8 + 3]) * inv);
                            w.z = pack_bf16(__uint_as_float(r[v4 * 8 + 4]) * inv, __uint_as_float(r[v4 * 8 + 5]) * inv);
                            w.w = pack_bf16(__uint_as_float(r[v4 * 8 + 6]) * inv, __uint_as_float(r[v4 * 8 + 7]) * inv);
                            dst[v4] = w;
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
                float* Cr = a.acc + ((static_cast<int64_t>(T.b) * P.S + q) * P.Hq + T.h) * D;
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld32(tO + c * 32 + lane_base, r);
                    if (q < P.S && mn != -INFINITY) {
                        float4* dst = reinterpret_cast<float4*>(Cr + c * 32);
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
        } else if (!aborted && !skip && n_kv == 0 && !a.acc && q < P.S) {
            // no key allowed for this tile: O = 0, m = -inf, l = 0
            __nv_bfloat16* O = static_cast<__nv_bfloat16*>(a.o) + T.b * P.qs[0] +
                               static_cast<int64_t>(q) * P.qs[1] + T.h * P.qs[2];
            for (int c = 0; c < D; c += 8) *reinterpret_cast<uint4*>(O + c) = make_uint4(0, 0, 0, 0);
            a.m[mi] = -INFINITY;
            a.l[mi] = 0.f;
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int D>
cudaError_t launch(const FwdArgs& a, const CUtensorMap* maps, cudaStream_t s) {
    using C = FwdCfg<D>;
    static bool configured[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !configured[dev]) {
        e = cudaFuncSetAttribute(k_fwd_tc<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) configured[dev] = true;
    }
    const int nqt = (a.P.S + BM - 1) / BM;
    const int grid = nqt * a.P.Hq * a.P.B;
    k_fwd_tc<D><<<grid, kThreads, C::SMEM, s>>>(maps[0], maps[1], maps[2], a);
    return cudaGetLastError();
}

}  // namespace

bool fwd_tc_supported(const Problem& P) {
    if (P.dtype != BPA_BF16 || (P.d != 64 && P.d != 128) || P.block_idx) return false;
    if (P.ring_n > 1 && P.ring_blk % BM) return false;
    return true;
}

cudaError_t launch_fwd_tc(const FwdArgs& a, const CUtensorMap* maps, cudaStream_t s) {
    return a.P.d == 128 ? launch<128>(a, maps, s) : launch<64>(a, maps, s);
}

}  // namespace bpa
