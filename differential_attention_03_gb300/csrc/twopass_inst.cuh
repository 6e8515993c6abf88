// Shared body of the per-instantiation launcher translation units.
#pragma once

#include "launch.h"
#include "twopass.cuh"

namespace da {

template <int D, int DV, bool SHARED_K, int EPI, int NSLOT, bool PERSIST, bool F8 = false>
cudaError_t launch_twopass(const TwoPassParams& p, const ItemPlan& plan, int grid, cudaStream_t s) {
  using C = TwoPassCfg<D, DV, SHARED_K, EPI, NSLOT, PERSIST, F8>;
  auto kern = twopass_fwd_kernel<D, DV, SHARED_K, EPI, NSLOT, PERSIST, F8>;
  // The attribute is per function and per device; setting it again is cheap
  // and keeps this free of per-device bookkeeping.
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  kern<<<grid, C::NTHREADS, C::SMEM_BYTES, s>>>(p, plan);
  return cudaGetLastError();
}

}  // namespace da
