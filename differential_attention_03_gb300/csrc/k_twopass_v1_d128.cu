#include "twopass_inst.cuh"
namespace da {
cudaError_t launch_twopass_v1_d128(const TwoPassParams& p, const ItemPlan& plan, int grid, bool persistent,
                                  cudaStream_t s) {
  return persistent ? launch_twopass<128, 256, false, kEpiRmsNorm, 4, true>(p, plan, grid, s)
                    : launch_twopass<128, 256, false, kEpiRmsNorm, 4, false>(p, plan, grid, s);
}
}  // namespace da
