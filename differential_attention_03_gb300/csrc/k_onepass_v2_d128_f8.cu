#include "onepass_inst.cuh"
namespace da {
cudaError_t launch_onepass_v2_d128_f8(const TwoPassParams& p, int grid, cudaStream_t s) {
  return launch_onepass<128, true, kEpiV2, 4, false, false, false, true>(p, grid, s);
}
}  // namespace da
