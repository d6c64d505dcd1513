// fwd_tc.cu - the forward tensor-core kernel's instantiations without attention dropout
// and the dispatch between its variants (the kernel itself is in fwd_tc.cuh).
#include "fwd_tc.cuh"

namespace bpa {

bool fwd_tc_supported(const Problem& P) {
    if (P.dtype != BPA_BF16 || (P.d != 64 && P.d != 128) || P.block_idx) return false;
    if (P.dv != P.d && !(P.d == 128 && P.dv == 64)) return false;
    if (P.ring_n > 1 && P.ring_blk % BM) return false;
    return true;
}

cudaError_t launch_fwd_tc(const FwdArgs& a, const CUtensorMap* maps, cudaStream_t s) {
    const Problem& P = a.P;
    // short key ranges: single-tile CTAs, two per SM; a ring block must hold whole CTAs
    if (fwd_band_supported(P)) return launch_fwd_band(a, maps, s);
    const bool single = fwd_single_tile(P);
    if (P.drop_thr) return launch_fwd_tc_dropout(a, maps, s, single);
    if (P.d == 128 && P.dv == 64) return single ? launch<128, 64, 1, false>(a, maps, s) : launch<128, 64, 2, false>(a, maps, s);
    if (P.d == 128) return single ? launch<128, 128, 1, false>(a, maps, s) : launch<128, 128, 2, false>(a, maps, s);
    return single ? launch<64, 64, 1, false>(a, maps, s) : launch<64, 64, 2, false>(a, maps, s);
}

}  // namespace bpa
