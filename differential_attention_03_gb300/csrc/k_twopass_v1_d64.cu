#include "twopass_inst.cuh"
namespace da {
cudaError_t launch_twopass_v1_d64(const TwoPassParams& p, int grid, cudaStream_t s) {
  return launch_twopass<64, 128, false, kEpiRmsNorm, 12>(p, grid, s);
}
}  // namespace da
