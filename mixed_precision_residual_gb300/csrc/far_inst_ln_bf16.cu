// Instantiations and launcher of the LayerNorm kernels for activations in bf16.
#include "far_kernels.cuh"

namespace far {

cudaError_t launch_ln_act_bf16(int wd, bool residual, const Launch& L) {
  switch (wd) {
    case FAR_BF16: return launch_ln<FAR_BF16, FAR_BF16>(residual, L);
    case FAR_F32: return launch_ln<FAR_BF16, FAR_F32>(residual, L);
    default: return cudaErrorInvalidValue;  // the pair is rejected before any launch
  }
}

}  // namespace far
