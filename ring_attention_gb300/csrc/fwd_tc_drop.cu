// fwd_tc_drop.cu - the forward tensor-core kernel's attention-dropout instantiations (a
// translation unit of their own, so that the library's parts compile in parallel).
#include "fwd_tc.cuh"

namespace bpa {

cudaError_t launch_fwd_tc_dropout(const FwdArgs& a, const CUtensorMap* maps, cudaStream_t s, bool single) {
    const Problem& P = a.P;
    if (P.d == 128 && P.dv == 64) return single ? launch<128, 64, 1, true>(a, maps, s) : launch<128, 64, 2, true>(a, maps, s);
    if (P.d == 128) return single ? launch<128, 128, 1, true>(a, maps, s) : launch<128, 128, 2, true>(a, maps, s);
    return single ? launch<64, 64, 1, true>(a, maps, s) : launch<64, 64, 2, true>(a, maps, s);
}

}  // namespace bpa
