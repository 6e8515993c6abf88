// fp32 backward passes of the multi-head DIFF V1 and V2 forwards on CUDA cores.
//
// The forward (per batch b, head h; c = 1/sqrt d; causal or not):
//   A_r = softmax(c Q_r K_r^T),  O = (A_1 - lambda A_2) V,
//   y = (1 - lambda_init) gamma O / rms(O)
// ("Differential Transformer" glossary page, "How differential attention
// works"; news article section "差分注意力" for the lambda re-parameterisation
// and the per-head RMSNorm).  The pages give no backward; it is the chain rule
// of that forward:
//   dO from dy through the RMSNorm (row pass: simt_fwd_f32_kernel<true>),
//   dV = A_1^T dO - lambda A_2^T dO,
//   dS_1 = A_1 (dO V^T - D_1),  dS_2 = A_2 (-lambda dO V^T - D_2),
//   dQ_r = c dS_r K_r,  dK_r = c dS_r^T Q_r,
//   dlambda = -sum dO . A_2 V,  dgamma = sum (1 - lambda_init) (O / rms(O)) dy,
// with D_r = rowsum(A_r dA_r) from the row pass.  The maps are recomputed
// from the row pass's log-sum-exps, a 32 x 32 block at a time, never stored.
// DIFF V2 (DIFF V2 analysis page, "2. 커스텀 커널 제거" and "GQA와의 호환성"):
// map 1 / map 2 are query heads 2g / 2g + 1 over their shared KV head, the
// coefficient is the row's s = sigmoid(logit) instead of lambda, there is no
// norm (dO = dy), dK and dV sum over every pair of the KV head's group, and
// dlogit = -s (1 - s) dO . A_2 V.
//
//   bwd_dkdv_kernel: one CTA per (b, h, 32 keys); sweeps the query blocks that
//     see those keys; dV, dK_1, dK_2 of its keys in registers.
//   bwd_dq_kernel:   one CTA per (b, h, 32 queries); sweeps the key blocks the
//     queries see; dQ_1, dQ_2 in registers.
//   bwd_reduce_kernel: dlambda and dgamma from the row pass's shares, in a
//     fixed order (deterministic).
// Both sweeps use the same 32 x 32 block step: warp w takes query rows
// 4w .. 4w + 3 of the block and lane j its key j (scores and dO . v_j as
// dot products over shared-memory rows; with d % 32 == 0 as float4 reads,
// each of the lane's key-row reads serving the warp's four query rows),
// writes P = A_1 - lambda A_2, dS_1 and dS_2 to shared memory; then every
// thread accumulates its outputs from them (float4 reads of its channel
// slice when d % 32 == 0).
#pragma once

#include "bounds.cuh"
#include "bwd_params.h"
#include "stage.cuh"

#undef DA_BOUNDS_FILE
#define DA_BOUNDS_FILE 9

namespace da {

constexpr int kBwdBlk = 32;  // queries and keys per block step
constexpr int kBwdThreads = 256;
constexpr int kBwdMaxCV = 32;  // value channels a thread accumulates (dv <= 256)
constexpr int kBwdMaxCK = 16;  // key/query channels a thread accumulates (d <= 128)

// Row pitches of the shared-memory tiles.  d % 32 == 0 ("fast"): d + 4, so
// that rows start on 16 bytes and the float4 reads of eight consecutive lanes
// (rows j .. j + 7) fall on 32 different banks; else d + 1 (odd: a lane per
// row reads scalars without conflicts).
__host__ __device__ constexpr bool bwd_fast(int d) { return d % 32 == 0; }
__host__ __device__ constexpr int bwd_pitch(int w, bool fast) { return fast ? w + 4 : w + 1; }

// Shared-memory floats of both sweeps: K_1, K_2, V, Q_1, Q_2, dO tiles, three
// 32 x 33 blocks (P, dS_1, dS_2) and five row statistics.
__host__ __device__ constexpr int bwd_smem_floats(int d, int dv) {
  return 4 * kBwdBlk * bwd_pitch(d, bwd_fast(d)) + 2 * kBwdBlk * bwd_pitch(dv, bwd_fast(d)) +
         3 * kBwdBlk * (kBwdBlk + 1) + 5 * kBwdBlk;
}

struct BwdSmem {
  float *k1, *k2, *v, *q1, *q2, *dO, *P, *S1, *S2, *st;
  int dp, dvp;  // row pitches (floats)
  __device__ BwdSmem(float* sm, int d, int dv) {
    dp = bwd_pitch(d, bwd_fast(d));
    dvp = bwd_pitch(dv, bwd_fast(d));
    k1 = sm;
    k2 = k1 + kBwdBlk * dp;
    v = k2 + kBwdBlk * dp;
    q1 = v + kBwdBlk * dvp;
    q2 = q1 + kBwdBlk * dp;
    dO = q2 + kBwdBlk * dp;
    P = dO + kBwdBlk * dvp;
    S1 = P + kBwdBlk * (kBwdBlk + 1);
    S2 = S1 + kBwdBlk * (kBwdBlk + 1);
    st = S2 + kBwdBlk * (kBwdBlk + 1);  // [5][32]: lse_1, lse_2, D_1, D_2, coefficient of the query block
  }
};

// Stages the query block [q0, q0 + 32) of row unit `unit` (V1: (b, h); V2: (b, pair)):
// Q_1 (head hq1), Q_2 (head hq2), dO rows and the statistics.
__device__ __forceinline__ void bwd_stage_queries(const BwdParams& p, const BwdSmem& s, int b, int hq1, int hq2,
                                                  long long unit, int q0, bool vec) {
  const int d = p.d, dv = p.dvw;
  const size_t qrow = static_cast<size_t>(p.heads_q) * d;
  const float* qb = p.q1 + static_cast<size_t>(b) * p.n * qrow;
  const long long unit_row0 = unit * p.n;
  stage_rows(s.q1, s.dp, qb + static_cast<size_t>(hq1) * d, qrow, q0, p.n, d, kBwdBlk, vec);
  stage_rows(s.q2, s.dp, (p.q2 + static_cast<size_t>(b) * p.n * qrow) + static_cast<size_t>(hq2) * d, qrow, q0,
             p.n, d, kBwdBlk, vec);
  stage_rows(s.dO, s.dvp, p.dO + unit_row0 * dv, dv, q0, p.n, dv, kBwdBlk, (dv & 3) == 0);
  if (threadIdx.x < 5 * kBwdBlk) {
    const int k = threadIdx.x / kBwdBlk, i = threadIdx.x % kBwdBlk;
    const int slot = k < 4 ? k : 5;  // lse_1, lse_2, D_1, D_2, coefficient
    s.st[threadIdx.x] = (q0 + i < p.n) ? p.row[slot * p.rows + unit_row0 + q0 + i] : 0.f;
  }
}

// Stages the key block [k0, k0 + 32) of KV head hk: K_1, K_2 (V1 only; V2 reads K_1 twice), V rows.
__device__ __forceinline__ void bwd_stage_keys(const BwdParams& p, const BwdSmem& s, int b, int hk, int k0,
                                               bool vec) {
  const int d = p.d, dv = p.dvw;
  const size_t krow = static_cast<size_t>(p.heads_kv) * d, vrow = static_cast<size_t>(p.heads_kv) * dv;
  stage_rows(s.k1, s.dp, p.k1 + static_cast<size_t>(b) * p.n * krow + static_cast<size_t>(hk) * d, krow, k0, p.n,
             d, kBwdBlk, vec);
  if (!p.v2)
    stage_rows(s.k2, s.dp, p.k2 + static_cast<size_t>(b) * p.n * krow + static_cast<size_t>(hk) * d, krow, k0,
               p.n, d, kBwdBlk, vec);
  stage_rows(s.v, s.dvp, p.v + static_cast<size_t>(b) * p.n * vrow + static_cast<size_t>(hk) * dv, vrow, k0, p.n,
             dv, kBwdBlk, vec);
}

// The 32 x 32 block step: P = A_1 - coef A_2, dS_1, dS_2 for queries
// [q0, q0 + 32) and keys [k0, k0 + 32) into shared memory (0 where masked).
// coef is lambda (V1) or the row's sigmoid(logit) (V2).
__device__ __forceinline__ float dot4(float4 a, float4 b, float acc) {
  acc = fmaf(a.x, b.x, acc);
  acc = fmaf(a.y, b.y, acc);
  acc = fmaf(a.z, b.z, acc);
  return fmaf(a.w, b.w, acc);
}

__device__ __forceinline__ float4 ld4(const float* a) { return *reinterpret_cast<const float4*>(a); }

__device__ __forceinline__ void bwd_block_step(const BwdParams& p, const BwdSmem& s, int q0, int k0, float lam) {
  constexpr int RW = kBwdBlk / (kBwdThreads / 32);  // query rows per warp
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = p.d, dv = p.dvw, dp = s.dp, dvp = s.dvp;
  const int key = k0 + lane;
  const float* k2s = p.v2 ? s.k1 : s.k2;
  float s1v[RW], s2v[RW], dpvv[RW];
#pragma unroll
  for (int r = 0; r < RW; ++r) s1v[r] = s2v[r] = dpvv[r] = 0.f;
  if (bwd_fast(d)) {
    // Each float4 of this lane's key (and value) row is read once and used
    // for the warp's four query rows (broadcast float4 reads).
    for (int e = 0; e < d; e += 4) {
      const float4 ka = ld4(s.k1 + lane * dp + e), kb = ld4(k2s + lane * dp + e);
#pragma unroll
      for (int r = 0; r < RW; ++r) {
        const int i = warp * RW + r;
        s1v[r] = dot4(ld4(s.q1 + i * dp + e), ka, s1v[r]);
        s2v[r] = dot4(ld4(s.q2 + i * dp + e), kb, s2v[r]);
      }
    }
    for (int c = 0; c < dv; c += 4) {
      const float4 vv = ld4(s.v + lane * dvp + c);
#pragma unroll
      for (int r = 0; r < RW; ++r) dpvv[r] = dot4(ld4(s.dO + (warp * RW + r) * dvp + c), vv, dpvv[r]);
    }
  } else {
#pragma unroll
    for (int r = 0; r < RW; ++r) {
      const int i = warp * RW + r;
      for (int e = 0; e < d; ++e) {
        s1v[r] = fmaf(s.q1[i * dp + e], s.k1[lane * dp + e], s1v[r]);
        s2v[r] = fmaf(s.q2[i * dp + e], k2s[lane * dp + e], s2v[r]);
      }
      for (int c = 0; c < dv; ++c) dpvv[r] = fmaf(s.dO[i * dvp + c], s.v[lane * dvp + c], dpvv[r]);
    }
  }
#pragma unroll
  for (int r = 0; r < RW; ++r) {
    const int i = warp * RW + r, t = q0 + i;
    const bool valid = t < p.n && key < p.n && (!p.causal || key <= t);
    const float coef = p.v2 ? s.st[4 * kBwdBlk + i] : lam;
    const float s1 = s1v[r], s2 = s2v[r], dpv = dpvv[r];
    const float p1 = valid ? expf(s1 * p.scale - s.st[i]) : 0.f;
    const float p2 = valid ? expf(s2 * p.scale - s.st[kBwdBlk + i]) : 0.f;
    s.P[i * (kBwdBlk + 1) + lane] = p1 - coef * p2;
    s.S1[i * (kBwdBlk + 1) + lane] = p1 * (dpv - s.st[2 * kBwdBlk + i]);
    s.S2[i * (kBwdBlk + 1) + lane] = p2 * (-coef * dpv - s.st[3 * kBwdBlk + i]);
  }
}

__device__ __forceinline__ bool bwd_vec(const BwdParams& p) {
  return ((p.d & 3) == 0) && ((reinterpret_cast<uintptr_t>(p.q1) | reinterpret_cast<uintptr_t>(p.q2) |
                               reinterpret_cast<uintptr_t>(p.k1) | reinterpret_cast<uintptr_t>(p.k2) |
                               reinterpret_cast<uintptr_t>(p.v)) & 15u) == 0;
}

// dV, dK_1, dK_2 of 32 keys of one KV head (V1: head h; V2: KV head, over
// every head pair of its group): thread (warp w, lane j) owns key k0 + j and
// the channel slices w * cv .. w * cv + cv - 1 (value) and w * ck .. (key).
__global__ void __launch_bounds__(kBwdThreads) bwd_dkdv_kernel(const BwdParams p) {
  extern __shared__ float sm[];
  const BwdSmem s(sm, p.d, p.dvw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nblk = (p.n + kBwdBlk - 1) / kBwdBlk;
  const int kb = blockIdx.x % nblk, kvu = blockIdx.x / nblk;
  const int b = kvu / p.heads_kv, hk = kvu % p.heads_kv, k0 = kb * kBwdBlk;
  const int d = p.d, dv = p.dvw, dp = s.dp, dvp = s.dvp;
  const int cv = (dv + 7) / 8, ck = (d + 7) / 8;
  const bool vec = bwd_vec(p), fast = bwd_fast(d);
  const float lam = p.v2 ? 0.f : *p.lambda;
  // Query-head pairs reading this KV head: V1 the head itself; V2 pairs
  // hk * group / 2 .. (hk + 1) * group / 2 - 1.
  const int g0 = p.v2 ? hk * (p.group / 2) : hk, g1 = p.v2 ? g0 + p.group / 2 : hk + 1;
  bwd_stage_keys(p, s, b, hk, k0, vec);
  float av[kBwdMaxCV], a1[kBwdMaxCK], a2[kBwdMaxCK];
#pragma unroll
  for (int k = 0; k < kBwdMaxCV; ++k) av[k] = 0.f;
#pragma unroll
  for (int k = 0; k < kBwdMaxCK; ++k) a1[k] = a2[k] = 0.f;
  for (int g = g0; g < g1; ++g) {
    const int hq1 = p.v2 ? 2 * g : g, hq2 = p.v2 ? 2 * g + 1 : g;
    const long long unit = static_cast<long long>(b) * p.units + g;
    for (int qb = p.causal ? kb : 0; qb < nblk; ++qb) {
      const int q0 = qb * kBwdBlk;
      __syncthreads();  // the previous block's reads are done
      bwd_stage_queries(p, s, b, hq1, hq2, unit, q0, vec);
      __syncthreads();
      bwd_block_step(p, s, q0, k0, lam);
      __syncthreads();
      for (int i = 0; i < kBwdBlk; ++i) {
        const float w = s.P[i * (kBwdBlk + 1) + lane];
        const float e1 = s.S1[i * (kBwdBlk + 1) + lane];
        const float e2 = s.S2[i * (kBwdBlk + 1) + lane];
        if (fast) {  // cv, ck multiples of 4: float4 broadcast reads of the warp's channel slices
#pragma unroll
          for (int k = 0; k < kBwdMaxCV; k += 4) {
            if (k < cv) {
              const float4 o = ld4(s.dO + i * dvp + warp * cv + k);
              av[k] = fmaf(w, o.x, av[k]);
              av[k + 1] = fmaf(w, o.y, av[k + 1]);
              av[k + 2] = fmaf(w, o.z, av[k + 2]);
              av[k + 3] = fmaf(w, o.w, av[k + 3]);
            }
          }
#pragma unroll
          for (int k = 0; k < kBwdMaxCK; k += 4) {
            if (k < ck) {
              const float4 qa = ld4(s.q1 + i * dp + warp * ck + k), qb = ld4(s.q2 + i * dp + warp * ck + k);
              a1[k] = fmaf(e1, qa.x, a1[k]);
              a1[k + 1] = fmaf(e1, qa.y, a1[k + 1]);
              a1[k + 2] = fmaf(e1, qa.z, a1[k + 2]);
              a1[k + 3] = fmaf(e1, qa.w, a1[k + 3]);
              a2[k] = fmaf(e2, qb.x, a2[k]);
              a2[k + 1] = fmaf(e2, qb.y, a2[k + 1]);
              a2[k + 2] = fmaf(e2, qb.z, a2[k + 2]);
              a2[k + 3] = fmaf(e2, qb.w, a2[k + 3]);
            }
          }
          continue;
        }
#pragma unroll
        for (int k = 0; k < kBwdMaxCV; ++k) {
          const int c = warp * cv + k;
          if (k < cv && c < dv) av[k] = fmaf(w, s.dO[i * dvp + c], av[k]);
        }
#pragma unroll
        for (int k = 0; k < kBwdMaxCK; ++k) {
          const int c = warp * ck + k;
          if (k < ck && c < d) {
            a1[k] = fmaf(e1, s.q1[i * dp + c], a1[k]);
            a2[k] = fmaf(e2, s.q2[i * dp + c], a2[k]);
          }
        }
      }
    }
  }
  const int key = k0 + lane;
  if (key < p.n && DA_BOUNDS_V(b < p.B && hk < p.heads_kv, key)) {
    const size_t kr = (static_cast<size_t>(b) * p.n + key) * p.heads_kv + hk;
#pragma unroll
    for (int k = 0; k < kBwdMaxCV; ++k) {
      const int c = warp * cv + k;
      if (k < cv && c < dv) p.dv[kr * dv + c] = av[k];
    }
#pragma unroll
    for (int k = 0; k < kBwdMaxCK; ++k) {
      const int c = warp * ck + k;
      if (k < ck && c < d) {
        if (p.v2) {
          p.dk1[kr * d + c] = p.scale * (a1[k] + a2[k]);  // both query heads read this key
        } else {
          p.dk1[kr * d + c] = p.scale * a1[k];
          p.dk2[kr * d + c] = p.scale * a2[k];
        }
      }
    }
  }
}

// dQ_1, dQ_2 of 32 queries of one row unit (V1: head h; V2: the pair's two
// query heads): thread (warp w, lane i) owns query q0 + i and the channel
// slice w * ck .. w * ck + ck - 1.
__global__ void __launch_bounds__(kBwdThreads) bwd_dq_kernel(const BwdParams p) {
  extern __shared__ float sm[];
  const BwdSmem s(sm, p.d, p.dvw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nblk = (p.n + kBwdBlk - 1) / kBwdBlk;
  const int qb = nblk - 1 - blockIdx.x % nblk;  // heaviest causal blocks first
  const int unit = blockIdx.x / nblk;
  const int b = unit / p.units, g = unit % p.units, q0 = qb * kBwdBlk;
  const int hq1 = p.v2 ? 2 * g : g, hq2 = p.v2 ? 2 * g + 1 : g;
  const int hk = p.v2 ? (2 * g) / p.group : g;
  const int d = p.d, dp = s.dp;
  const int ck = (d + 7) / 8;
  const bool vec = bwd_vec(p), fast = bwd_fast(d);
  const float lam = p.v2 ? 0.f : *p.lambda;
  const float* k2s = p.v2 ? s.k1 : s.k2;
  bwd_stage_queries(p, s, b, hq1, hq2, unit, q0, vec);
  float a1[kBwdMaxCK], a2[kBwdMaxCK];
#pragma unroll
  for (int k = 0; k < kBwdMaxCK; ++k) a1[k] = a2[k] = 0.f;
  const int kb_end = p.causal ? qb : nblk - 1;
  for (int kb = 0; kb <= kb_end; ++kb) {
    const int k0 = kb * kBwdBlk;
    __syncthreads();  // the previous block's reads are done
    bwd_stage_keys(p, s, b, hk, k0, vec);
    __syncthreads();
    bwd_block_step(p, s, q0, k0, lam);
    __syncthreads();
    for (int j = 0; j < kBwdBlk; ++j) {
      const float e1 = s.S1[lane * (kBwdBlk + 1) + j];
      const float e2 = s.S2[lane * (kBwdBlk + 1) + j];
      if (fast) {  // ck a multiple of 4: float4 broadcast reads of the key rows' channel slice
#pragma unroll
        for (int k = 0; k < kBwdMaxCK; k += 4) {
          if (k < ck) {
            const float4 ka = ld4(s.k1 + j * dp + warp * ck + k), kb = ld4(k2s + j * dp + warp * ck + k);
            a1[k] = fmaf(e1, ka.x, a1[k]);
            a1[k + 1] = fmaf(e1, ka.y, a1[k + 1]);
            a1[k + 2] = fmaf(e1, ka.z, a1[k + 2]);
            a1[k + 3] = fmaf(e1, ka.w, a1[k + 3]);
            a2[k] = fmaf(e2, kb.x, a2[k]);
            a2[k + 1] = fmaf(e2, kb.y, a2[k + 1]);
            a2[k + 2] = fmaf(e2, kb.z, a2[k + 2]);
            a2[k + 3] = fmaf(e2, kb.w, a2[k + 3]);
          }
        }
        continue;
      }
#pragma unroll
      for (int k = 0; k < kBwdMaxCK; ++k) {
        const int c = warp * ck + k;
        if (k < ck && c < d) {
          a1[k] = fmaf(e1, s.k1[j * dp + c], a1[k]);
          a2[k] = fmaf(e2, k2s[j * dp + c], a2[k]);
        }
      }
    }
  }
  const int t = q0 + lane;
  if (t < p.n && DA_BOUNDS_V(b < p.B && hq1 < p.heads_q && hq2 < p.heads_q, t)) {
    const size_t qr = (static_cast<size_t>(b) * p.n + t) * p.heads_q;
#pragma unroll
    for (int k = 0; k < kBwdMaxCK; ++k) {
      const int c = warp * ck + k;
      if (k < ck && c < d) {
        p.dq1[(qr + hq1) * d + c] = p.scale * a1[k];
        p.dq2[(qr + hq2) * d + c] = p.scale * a2[k];
      }
    }
  }
}

// Fixed-order reductions of the row pass's shares, one CTA per output.  V1:
// CTA 0 dlambda = sum of every row's share; CTA 1 + c dgamma[c] = sum of the
// row-pass CTAs' shares.  V2 (logits shared by a sequence's tokens): dlogit of
// (b, pair) = sum over the tokens (and the sequences when sb = 0) of the
// rows' shares.
__global__ void __launch_bounds__(kBwdThreads) bwd_reduce_kernel(const BwdParams p) {
  __shared__ float red[kBwdThreads];
  const float* share = p.row + 4 * p.rows;
  float a = 0.f;
  int g = 0, b0 = 0, b1 = 0;
  const bool dgamma_cta = !p.v2 && blockIdx.x > 0;
  if (dgamma_cta) {
    const int c = static_cast<int>(blockIdx.x) - 1;
    for (int k = threadIdx.x; k < p.n_row_ctas; k += kBwdThreads) a += p.dgp[static_cast<size_t>(k) * p.dvw + c];
  } else if (p.v2) {
    g = p.sb == 0 ? static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x) % p.units;
    b0 = p.sb == 0 ? 0 : static_cast<int>(blockIdx.x) / p.units;
    b1 = p.sb == 0 ? p.B : b0 + 1;
    for (int b = b0; b < b1; ++b) {
      const float* sr = share + (static_cast<long long>(b) * p.units + g) * p.n;
      for (int t = threadIdx.x; t < p.n; t += kBwdThreads) a += sr[t];
    }
  } else if (p.dlam_parts != nullptr) {
    for (int k = threadIdx.x; k < p.n_row_ctas; k += kBwdThreads) a += p.dlam_parts[k];
  } else {
    for (long long r = threadIdx.x; r < p.rows; r += kBwdThreads) a += share[r];
  }
  red[threadIdx.x] = a;
  __syncthreads();
  for (int w = kBwdThreads / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x != 0) return;
  if (p.v2) {
    if (DA_BOUNDS_V(b0 < p.B && g < p.units, g)) p.dlogits[static_cast<long long>(b0) * p.sb + g] = red[0];
  } else if (dgamma_cta)
    DA_STORE(p.dgamma, blockIdx.x - 1, p.dvw, red[0]);
  else
    *p.dlambda = red[0];
}

// Gradients of lambda = exp(<lq1, lk1>) - exp(<lq2, lk2>) + lambda_init with
// respect to the four vectors, given dlambda (device scalar); one warp.
__global__ void lambda_reparam_bwd_kernel(const float* lq1, const float* lk1, const float* lq2, const float* lk2,
                                          int dim, const float* dlambda, float* dlq1, float* dlk1, float* dlq2,
                                          float* dlk2) {
  float a = 0.f, c = 0.f;
  for (int i = threadIdx.x; i < dim; i += 32) {
    a = fmaf(lq1[i], lk1[i], a);
    c = fmaf(lq2[i], lk2[i], c);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, off);
    c += __shfl_xor_sync(0xffffffffu, c, off);
  }
  const float g = *dlambda, e1 = g * expf(a), e2 = g * expf(c);
  for (int i = threadIdx.x; i < dim; i += 32) {
    dlq1[i] = e1 * lk1[i];
    dlk1[i] = e1 * lq1[i];
    dlq2[i] = -e2 * lk2[i];
    dlk2[i] = -e2 * lq2[i];
  }
}

}  // namespace da
