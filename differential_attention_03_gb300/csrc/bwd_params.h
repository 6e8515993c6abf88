// Parameters of the fp32 backward passes (V1 and V2): the extra arguments of
// the row pass (simt_fwd_f32_kernel<true>) and those of the dK/dV and dQ
// sweeps and the reduction (backward.cuh).
#pragma once

#include "params.h"

namespace da {

// Row pass: dy and where the per-row results go.
struct SimtBwdExtra {
  const float* dy;       // V1: [B, n, H, dv]; V2: [B, n, Hq / 2, d]
  float* ws_do;          // [B * units * n][dv]: dO, the gradient of the pre-norm output (V2: dy)
  float* ws_row;         // [6][B * units * n]: lse_1, lse_2, D_1, D_2, dlambda / dlogit share, coefficient
  float* ws_dgamma;      // V1: [CTAs][dv], each CTA's share of dgamma
  float* dlogits_dense;  // V2 with a per-token logit stride: dlogit of (b, t, pair) at b sb + t st + pair
};

struct BwdParams {
  const float* q1;  // V1: [B, n, H, d]; V2: q [B, n, Hq, d] (q1 == q2)
  const float* q2;
  const float* k1;  // V1: [B, n, H, d]; V2: k [B, n, Hkv, d] (k1 == k2)
  const float* k2;
  const float* v;       // V1: [B, n, H, dv]; V2: [B, n, Hkv, d]
  const float* dO;      // [B * units * n][dv] (row pass)
  const float* row;     // [6][B * units * n]: lse_1, lse_2, D_1, D_2, dlambda / dlogit share, coefficient
  const float* dgp;     // [n_row_ctas][dv]: dgamma shares (V1 row pass)
  const float* dlam_parts;  // V1: [n_row_ctas] dlambda shares of whole CTAs, or nullptr (then the rows' shares)
  const float* lambda;  // V1 device scalar
  float* dq1;           // V1: [B, n, H, d]; V2: dq [B, n, Hq, d] (dq1 == dq2)
  float* dq2;
  float* dk1;  // V1: [B, n, H, d]; V2: dk [B, n, Hkv, d] (dK_1 + dK_2 of every pair of the group)
  float* dk2;
  float* dv;       // like v
  float* dlambda;  // V1 device scalar
  float* dgamma;   // V1 [dv] or nullptr
  float* dlogits;  // V2, logit shared by a sequence's tokens: dlogit of (b, pair) at b sb + pair
  long long sb;    // (sb = 0: one logit per pair for every sequence)
  float scale;
  int B, n, d, dvw, causal, v2;
  int heads_q, heads_kv, units, group;  // units: V1 heads, V2 head pairs per sequence; group = Hq / Hkv
  long long rows;                       // B * units * n
  int n_row_ctas;
  int n_logit_outs;  // V2: dlogits entries the reduction writes (0: none)
};

}  // namespace da
