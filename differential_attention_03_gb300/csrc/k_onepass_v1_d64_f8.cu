#include "onepass_inst.cuh"
namespace da {
cudaError_t launch_onepass_v1_d64_f8(const TwoPassParams& p, int grid, bool persistent, cudaStream_t s) {
  return persistent ? launch_onepass<64, false, kEpiRmsNorm, 7, true, true, false, true>(p, grid, s)
                    : launch_onepass<64, false, kEpiRmsNorm, 7, true, false, false, true>(p, grid, s);
}
}  // namespace da
