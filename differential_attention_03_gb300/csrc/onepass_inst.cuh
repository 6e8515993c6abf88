// Shared body of the one-sweep launcher translation units.
#pragma once

#include "launch.h"
#include "onepass.cuh"

namespace da {

template <int D, bool SHARED_K, int EPI, int NSLOT, bool PSM, bool PERSIST, bool STATS = false, bool F8 = false,
          bool SAVE = false>
cudaError_t launch_onepass(const TwoPassParams& p, int grid, cudaStream_t s) {
  using C = OnePassCfg<D, SHARED_K, EPI, NSLOT, PSM, PERSIST, STATS, F8, SAVE>;
  auto kern = onepass_fwd_kernel<D, SHARED_K, EPI, NSLOT, PSM, PERSIST, STATS, F8, SAVE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  kern<<<grid, C::NTHREADS, C::SMEM_BYTES, s>>>(p);
  return cudaGetLastError();
}

}  // namespace da
