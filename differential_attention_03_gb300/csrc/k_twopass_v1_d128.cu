#include "twopass_inst.cuh"
namespace da {
cudaError_t launch_twopass_v1_d128(const TwoPassParams& p, int grid, cudaStream_t s) {
  return launch_twopass<128, 256, false, kEpiRmsNorm, 4>(p, grid, s);
}
}  // namespace da
