// Tensor-core attention (placeholder until the tcgen05 kernel lands).
#include "kernels.cuh"
namespace sa {
bool attend_tc_supported(const AttnArgs&) { return false; }
cudaError_t launch_attend_tc(const AttnArgs&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace sa
