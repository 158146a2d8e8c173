// Tensor-core (tcgen05) kernels: placeholder until the sm_103a pipeline lands.
#include "internal.h"

namespace sa {

size_t tc_workspace_bytes(const Problem &, const TcConfig &) { return 0; }

cudaError_t launch_tc(const Problem &, const TcConfig &, void *, size_t, cudaStream_t, int *launches) {
    *launches = 0;
    return cudaErrorNotSupported;
}

}  // namespace sa
