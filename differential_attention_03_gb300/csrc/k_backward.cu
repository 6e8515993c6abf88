// Launchers of the fp32 DIFF V1 backward sweeps (dK/dV, dQ) and the
// dlambda/dgamma reduction; the row pass before them is launched from k_simt.cu.
#include "backward.cuh"
#include "launch.h"

namespace da {

static_assert(kBwdThreads == kSimtWarps * 32, "stage_rows assumes the SIMT CTA size");

cudaError_t launch_backward_f32(const BwdParams& p, cudaStream_t s) {
  cudaError_t e;
  const long long nblk = (p.n + kBwdBlk - 1) / kBwdBlk;
  const unsigned grid = static_cast<unsigned>(nblk * p.B * p.units);
  const int smem = bwd_smem_floats(p.d, p.dvw) * 4;
  e = cudaFuncSetAttribute(bwd_dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  bwd_dkdv_kernel<<<static_cast<unsigned>(nblk * p.B * p.heads_kv), kBwdThreads, smem, s>>>(p);
  bwd_dq_kernel<<<grid, kBwdThreads, smem, s>>>(p);
  const int nred = p.v2 ? p.n_logit_outs : 1 + (p.dgamma != nullptr ? p.dvw : 0);
  if (nred > 0) bwd_reduce_kernel<<<nred, kBwdThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_bwd_reduce(const BwdParams& p, cudaStream_t s) {
  const int nred = p.v2 ? p.n_logit_outs : 1 + (p.dgamma != nullptr ? p.dvw : 0);
  if (nred > 0) bwd_reduce_kernel<<<nred, kBwdThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_lambda_reparam_bwd(const float* lq1, const float* lk1, const float* lq2, const float* lk2,
                                      int dim, const float* dlambda, float* dlq1, float* dlk1, float* dlq2,
                                      float* dlk2, cudaStream_t s) {
  lambda_reparam_bwd_kernel<<<1, 32, 0, s>>>(lq1, lk1, lq2, lk2, dim, dlambda, dlq1, dlk1, dlq2, dlk2);
  return cudaGetLastError();
}

}  // namespace da
