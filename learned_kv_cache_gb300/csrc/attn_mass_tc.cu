// Tensor-core (tcgen05 / TMEM / TMA) row-LSE and future-attention-mass passes.
#include "kvp_common.cuh"
#include "kvp_launch.h"

namespace kvp {

bool tc_supported(int, AttnShape) { return false; }
size_t fam_tc_workspace_size(AttnShape, int) { return 0; }
cudaError_t launch_lse_tc(const void*, const void*, int, AttnShape, float, float*, int*, cudaStream_t) {
  return cudaErrorNotSupported;
}
cudaError_t launch_fam_tc(const void*, const void*, const float*, int, AttnShape, float, int, float*,
                          void*, size_t, int*, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace kvp
