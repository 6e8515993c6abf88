// Launchers of the tensor-core backward: the statistics pass (the one-sweep
// forward with its STATS epilogue) and the dK/dV/dQ kernel.
#include "bwd_prep.cuh"
#include "bwd_tc.cuh"
#include "launch.h"
#include "onepass_inst.cuh"

namespace da {

cudaError_t launch_bwd_stats(const TwoPassParams& p, bool v2, int grid, cudaStream_t s) {
  return v2 ? launch_onepass<128, true, kEpiV2, 4, false, false, true>(p, grid, s)
            : launch_onepass<64, false, kEpiRmsNorm, 7, true, false, true>(p, grid, s);
}

template <bool V2>
static cudaError_t launch_bwd_tc_t(const BwdTcParams& p, int grid, cudaStream_t s) {
  using C = BwdTcCfg<V2>;
  cudaError_t e = cudaFuncSetAttribute(bwd_tc_kernel<V2>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  bwd_tc_kernel<V2><<<grid, C::NTHREADS, C::SMEM_BYTES, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_bwd_tc(const BwdTcParams& p, bool v2, int grid, cudaStream_t s) {
  return v2 ? launch_bwd_tc_t<true>(p, grid, s) : launch_bwd_tc_t<false>(p, grid, s);
}

cudaError_t launch_bwd_prep(const BwdPrepParams& p, bool v2, int grid, cudaStream_t s) {
  if (v2)
    bwd_prep_kernel<true><<<grid, kPrepWarps * 32, 0, s>>>(p);
  else
    bwd_prep_kernel<false><<<grid, kPrepWarps * 32, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace da
