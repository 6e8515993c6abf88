// Host-side launchers of the kernel instantiations (one translation unit each,
// so that they compile in parallel).  Each returns the cudaError_t of the launch.
#pragma once

#include <cuda_runtime.h>

#include "params.h"

namespace da {
struct DecodeParams;
struct BwdParams;
struct SimtBwdExtra;
struct GemmParams;
struct BwdTcParams;
struct BwdPrepParams;
}

namespace da {

// V1, d = 128, value width 256: two sweeps, one accumulator.
// plan: the persistent form's per-CTA item lists (plan.count == 0: snake order).
cudaError_t launch_twopass_v1_d128(const TwoPassParams& p, const ItemPlan& plan, int grid, bool persistent,
                                   cudaStream_t s);
// The same with e4m3 queries and keys (QK^T on kind::f8f6f4 MMAs; P.V in bf16).
cudaError_t launch_twopass_v1_d128_f8(const TwoPassParams& p, const ItemPlan& plan, int grid, bool persistent,
                                      cudaStream_t s);
// V1, d = 64, value width 128: one sweep, two online-softmax states.
cudaError_t launch_onepass_v1_d64(const TwoPassParams& p, int grid, bool persistent, cudaStream_t s);
// V2, d = 128 (query/key/value width 128), one K/V head per query-head pair: one sweep.
cudaError_t launch_onepass_v2_d128(const TwoPassParams& p, int grid, cudaStream_t s);
// The same with e4m3 queries and keys (tm_q1 / tm_k1 over bytes; scale_log2 carries their scales).
cudaError_t launch_onepass_v2_d128_f8(const TwoPassParams& p, int grid, cudaStream_t s);
// V1, d = 64, e4m3 queries and keys (each Q/K map {H d bytes, 1, n, B} with 128-byte boxes).
cudaError_t launch_onepass_v1_d64_f8(const TwoPassParams& p, int grid, bool persistent, cudaStream_t s);
// The training forward (SAVE): the output plus lse_r and O_r of every row (see TwoPassParams).
cudaError_t launch_onepass_v1_d64_save(const TwoPassParams& p, int grid, bool persistent, cudaStream_t s);
cudaError_t launch_onepass_v2_d128_save(const TwoPassParams& p, int grid, cudaStream_t s);

cudaError_t launch_simt_f32(const SimtParams& p, cudaStream_t s);
// V1 decode (one query per sequence over a key/value cache), d in {64, 128}:
// p.nsplit clusters of `cs` CTAs (1..8) over the keys of each of the `units` (batch, head)
// pairs (with p.nsplit > 1 the states go through p.ws to a combine kernel).  k8: e4m3 key caches.
cudaError_t launch_decode_v1(const DecodeParams& p, int d, bool k8, int units, int cs, cudaStream_t s);
// V2 decode, d = 128: head pairs over their shared KV head (one key tile for both queries).
cudaError_t launch_decode_v2_d128(const DecodeParams& p, bool k8, int units, int cs, cudaStream_t s);
// fp32 V1 backward: the row pass (per-row statistics, dO, dgamma shares), then the
// dK/dV and dQ sweeps and the dlambda/dgamma reduction (3 kernels).
cudaError_t launch_simt_bwd_rows(const SimtParams& p, const SimtBwdExtra& x, cudaStream_t s);
cudaError_t launch_backward_f32(const BwdParams& p, cudaStream_t s);
cudaError_t launch_lambda_reparam_bwd(const float* lq1, const float* lk1, const float* lq2, const float* lk2,
                                      int dim, const float* dlambda, float* dlq1, float* dlk1, float* dlq2,
                                      float* dlk2, cudaStream_t s);
cudaError_t launch_lambda_reparam(const float* lq1, const float* lk1, const float* lq2, const float* lk2,
                                  int dim, float lambda_init, float* out, cudaStream_t s);
// Tensor-core backward (bf16; V1 d = 64, V2 d = 128): the statistics pass
// (one-sweep forward, one item per CTA, grid = items) and the dK/dV/dQ kernel
// (grid = B * heads_kv * key tiles).
cudaError_t launch_bwd_stats(const TwoPassParams& p, bool v2, int grid, cudaStream_t s);
// The same per-row results from a training forward's saved statistics (CUDA cores; 128 rows a CTA).
cudaError_t launch_bwd_prep(const BwdPrepParams& p, bool v2, int grid, cudaStream_t s);
cudaError_t launch_bwd_tc(const BwdTcParams& p, bool v2, int grid, cudaStream_t s);
// The fp32 backward's reduction of the dlambda / dlogit and dgamma shares alone.
cudaError_t launch_bwd_reduce(const BwdParams& p, cudaStream_t s);
// Projection GEMM C = A B^T (bf16, fp32 accumulation), `grid` persistent CTAs.
cudaError_t launch_gemm_bf16(const GemmParams& p, int grid, cudaStream_t s);
cudaError_t launch_wait_selftest(unsigned long long budget_cycles, int* status, cudaStream_t s);

}  // namespace da
