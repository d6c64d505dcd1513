// bwd_tc.cu - blockwise attention backward on the 5th-generation tensor cores.
#include "bpa_internal.h"
#include "common.cuh"

namespace bpa {

bool bwd_tc_supported(const Problem&) { return false; }

cudaError_t launch_bwd_tc(const BwdArgs&, const CUtensorMap*, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace bpa
