// Parameter block of the tensor-core backward's dK/dV/dQ kernel (bwd_tc.cuh),
// shared with the host API.
#pragma once

#include <cuda.h>

namespace da {

struct BwdTcParams {
  CUtensorMap tm_q1, tm_q2;  // bf16 queries (V2: one map over q, heads 2g and 2g + 1)
  CUtensorMap tm_k1, tm_k2;  // bf16 keys (V2: tm_k2 unused)
  CUtensorMap tm_v;          // bf16 values
  CUtensorMap tm_do;         // bf16 dO [B, n, units, 128] (V1: from the statistics pass; V2: dy)
  CUtensorMap tm_dq1;        // fp32 dQ_1 (V2: dq, heads 2g and 2g + 1): boxes of 32 columns x 128 rows, reduce-add
  CUtensorMap tm_dq2;        // fp32 dQ_2 (V1 only)
  const float* row;          // [6][rows]: lse_1, lse_2, Delta_1, Delta_2, share, coefficient
  const float* lambda;       // V1: c_2 = -lambda
  float* dq1;                // fp32, zero on entry: V1 [B, n, H, d]; V2 dq [B, n, Hq, d] (dq2 == dq1)
  float* dq2;
  float* dk1;                // fp32: V1 [B, n, H, d]; V2 dk [B, n, Hkv, d]
  float* dk2;                // V1 only
  float* dv;                 // fp32 [B, n, heads_kv, 128]
  float scale_log2, scale;   // softmax scale x log2(e); softmax scale
  int B, n, causal;
  int heads_kv, units, group;  // units: V1 H, V2 Hq / 2 (rows of the statistics); group: V2 Hq / Hkv
  int num_tiles;               // 128-row tiles of n
  long long rows;              // B * units * n
  int* status;
};

}  // namespace da
