// Launcher of the projection GEMM (one persistent CTA per SM).
#include "gemm.cuh"
#include "launch.h"

namespace da {

cudaError_t launch_gemm_bf16(const GemmParams& p, int grid, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(gemm_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       GemmCfg::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  gemm_bf16_kernel<<<grid, GemmCfg::NTHREADS, GemmCfg::SMEM_BYTES, s>>>(p);
  return cudaGetLastError();
}

}  // namespace da
