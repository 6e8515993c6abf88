// Kernel parameter blocks shared by the launchers and the host API.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

namespace da {

enum : int { kEpiRmsNorm = 0, kEpiV2 = 1 };

struct TwoPassParams {
  CUtensorMap tm_q1;  // 4-D maps over BSHD tensors: dims {W, heads, n, B}
  CUtensorMap tm_q2;
  CUtensorMap tm_k1;
  CUtensorMap tm_k2;
  CUtensorMap tm_v;
  __nv_bfloat16* out;       // [B, n, units_per_batch, DV]
  const float* lambda;      // V1: device scalar lambda
  const float* gamma;       // V1: [DV] or nullptr
  const float* lam_logits;  // V2: logit of (b, t, g) at b*sb + t*st + g
  long long sb, st;
  float scale_log2;  // softmax scale * log2(e) (map 1; both maps unless e4m3 inputs)
  float norm_mult;   // V1: 1 - lambda_init
  float eps;         // V1: RMSNorm epsilon
  int B, n, causal;
  int units_per_batch;  // V1: H; V2: Hq / 2
  int group;            // V2: query heads per KV head
  int num_q_tiles;   // query tiles per unit in this launch: [q_tile_begin, q_tile_begin + num_q_tiles)
  int order;  // 0: unit-major tile order, 1: query-tile-major
  int* status;
  CUtensorMap tm_out;  // output [B, n, units_per_batch, DV] for TMA stores
  // Backward statistics (one-sweep kernel with STATS): dy in, per-row results
  // out; row r = (b * units_per_batch + u) * n + t.
  const __nv_bfloat16* dy;  // [B, n, units_per_batch, DV]
  __nv_bfloat16* dO;        // V1: [B, n, units_per_batch, DV], the gradient of the pre-norm output
  float* row;               // [6][rows]: lse_1, lse_2, Delta_1, Delta_2, lambda / logit share, coefficient
  float* dgp;               // V1: [gridDim.x][DV], each CTA's share of dgamma
  float* dlam_part;         // V1: [gridDim.x], each CTA's share of dlambda
  float* dlogits_dense;     // V2, one logit per token: dlogit of (b, t, pair) at b sb + t st + pair
  long long rows;           // B * units_per_batch * n
  // Training forward (one-sweep kernel with SAVE): besides the output, each
  // row's lse_1, lse_2 (to row[ri], row[rows + ri]) and its normalised map
  // outputs O_1, O_2 in bf16, each laid out [B units_per_batch][128-row
  // tiles][4 blocks of 32 channels][128 rows][32 channels].
  __nv_bfloat16* o1_save;
  __nv_bfloat16* o2_save;
  float scale2_log2;  // e4m3 queries and keys only: map 2's softmax scale, with its dequantisation scales
  int q_tile_begin;   // first query tile (0 unless a causal forward is run over token chunks)
};

// Work plan of a persistent launch, computed on the host: CTA c takes the
// items items[first[c]] .. items[first[c + 1] - 1] in that order (indices of
// the unit-major item map).  count == 0: no plan (the snake order).  Passed
// by value as a second kernel parameter, so a launch needs no device memory
// or shared state for it.
constexpr int kPlanMaxCtas = 256, kPlanMaxItems = 4096;
struct ItemPlan {
  int count;  // CTAs with a list (the launch's grid), or 0
  unsigned short first[kPlanMaxCtas + 1];
  unsigned short items[kPlanMaxItems];
};

// What work item `idx` of a tcgen05 launch computes: batch b, unit u (V1:
// head; V2: query-head pair), its query heads and K/V head, query tile qt
// (first row q0).  Items are ordered heaviest causal first: unit-major keeps
// all query tiles of one unit together (its K/V stream shared in L2),
// query-tile-major runs the heaviest tiles of every unit first.
struct TileCoord {
  int b, u, hq1, hq2, hk, qt, q0;
};

template <int EPI>
__device__ __forceinline__ TileCoord tile_coord(const TwoPassParams& p, int idx) {
  const int units = p.B * p.units_per_batch;
  int unit, qt;
  if (p.order == 0) {
    unit = idx / p.num_q_tiles;
    qt = p.num_q_tiles - 1 - idx % p.num_q_tiles;
  } else {
    qt = p.num_q_tiles - 1 - idx / units;
    unit = idx % units;
  }
  TileCoord c;
  c.b = unit / p.units_per_batch;
  c.u = unit % p.units_per_batch;
  if (EPI == kEpiRmsNorm) {
    c.hq1 = c.hq2 = c.hk = c.u;
  } else {
    c.hq1 = 2 * c.u;
    c.hq2 = 2 * c.u + 1;
    c.hk = c.hq1 / p.group;
  }
  c.qt = qt + p.q_tile_begin;
  c.q0 = c.qt * 128;
  return c;
}

struct SimtParams {
  const float* q1;  // V1: [B, n, H, d]; V2: q [B, n, Hq, d] (q1 == q2)
  const float* q2;
  const float* k1;  // V1: [B, n, H, d]; V2: k [B, n, Hkv, d] (k1 == k2)
  const float* k2;
  const float* v;   // V1: [B, n, H, 2d]; V2: [B, n, Hkv, d]
  float* out;       // [B, n, units_per_batch, dv]
  const float* lambda;      // V1 device scalar
  const float* gamma;       // V1 [dv] or nullptr
  const float* lam_logits;  // V2
  long long sb, st;
  float scale, norm_mult, eps;
  int B, n, d, dv, causal, v2;
  int heads_q, heads_kv, units_per_batch, group;
  long long rows_total;
};

constexpr int kSimtMaxD = 128;
constexpr int kSimtMaxVPerLane = 8;  // value width <= 256
constexpr int kSimtWarps = 8;
constexpr int kSimtRows = 8;   // query rows per CTA (one per warp)
constexpr int kSimtKeys = 32;  // keys per shared-memory tile

}  // namespace da
