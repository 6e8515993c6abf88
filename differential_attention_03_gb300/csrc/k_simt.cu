#include "launch.h"
#include "simt.cuh"
namespace da {
cudaError_t launch_simt_f32(const SimtParams& p, cudaStream_t s) {
  const long long nqb = (p.n + kSimtRows - 1) / kSimtRows;
  const long long blocks = nqb * p.B * p.units_per_batch;
  const int smem = simt_smem_floats(p.d, p.dv) * 4;
  cudaError_t e =
      cudaFuncSetAttribute(simt_fwd_f32_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  simt_fwd_f32_kernel<false><<<static_cast<unsigned>(blocks), kSimtWarps * 32, smem, s>>>(p, SimtBwdExtra{});
  return cudaGetLastError();
}
cudaError_t launch_simt_bwd_rows(const SimtParams& p, const SimtBwdExtra& x, cudaStream_t s) {
  const long long nqb = (p.n + kSimtRows - 1) / kSimtRows;
  const long long blocks = nqb * p.B * p.units_per_batch;
  const int smem = simt_smem_floats(p.d, p.dv) * 4;
  cudaError_t e =
      cudaFuncSetAttribute(simt_fwd_f32_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  simt_fwd_f32_kernel<true><<<static_cast<unsigned>(blocks), kSimtWarps * 32, smem, s>>>(p, x);
  return cudaGetLastError();
}
cudaError_t launch_lambda_reparam(const float* lq1, const float* lk1, const float* lq2, const float* lk2,
                                  int dim, float lambda_init, float* out, cudaStream_t s) {
  lambda_reparam_kernel<<<1, 32, 0, s>>>(lq1, lk1, lq2, lk2, dim, lambda_init, out);
  return cudaGetLastError();
}
cudaError_t launch_wait_selftest(unsigned long long budget_cycles, int* status, cudaStream_t s) {
  wait_timeout_selftest_kernel<<<1, 32, 0, s>>>(budget_cycles, status);
  return cudaGetLastError();
}
}  // namespace da
