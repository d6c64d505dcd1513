// gather.cu - block-selected attention forward over gathered key blocks.
#include "bpa_internal.h"
#include "common.cuh"

namespace bpa {

bool gather_supported(const Problem&) { return false; }

cudaError_t launch_gather_fwd(const FwdArgs&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace bpa
