// Tensor-core (tcgen05) gradient kernel for sm_103a.
#include "tnd_internal.h"

namespace tnd {

bool grad_tc_supported(int, int) { return false; }

cudaError_t launch_grad_tc(const GradArgs &, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace tnd
