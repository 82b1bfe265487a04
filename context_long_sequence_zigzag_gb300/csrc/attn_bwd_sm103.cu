// attn_bwd_sm103.cu — tensor-core backward (tcgen05).  Until it is enabled,
// tc_bwd_supported() reports false and the backward runs on the CUDA-core
// kernels in simple_kernels.cu.
#include "internal.h"

namespace cpattn {

bool tc_bwd_supported(int32_t, int32_t) { return false; }

cudaError_t launch_tc_bwd(const AttnArgs&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace cpattn
