// Launchers of the training forward: the one-sweep kernel with SAVE (the
// output plus each row's lse_1, lse_2 and normalised map outputs O_1, O_2).
#include "onepass_inst.cuh"
namespace da {
cudaError_t launch_onepass_v1_d64_save(const TwoPassParams& p, int grid, bool persistent, cudaStream_t s) {
  return persistent ? launch_onepass<64, false, kEpiRmsNorm, 7, true, true, false, false, true>(p, grid, s)
                    : launch_onepass<64, false, kEpiRmsNorm, 7, true, false, false, false, true>(p, grid, s);
}
cudaError_t launch_onepass_v2_d128_save(const TwoPassParams& p, int grid, cudaStream_t s) {
  return launch_onepass<128, true, kEpiV2, 4, false, false, false, false, true>(p, grid, s);
}
}  // namespace da
