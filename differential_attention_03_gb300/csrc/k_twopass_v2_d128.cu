#include "twopass_inst.cuh"
namespace da {
cudaError_t launch_twopass_v2_d128(const TwoPassParams& p, int grid, cudaStream_t s) {
  return launch_twopass<128, 128, true, kEpiV2, 5>(p, grid, s);
}
}  // namespace da
