// fp32 differential-attention forward on CUDA cores (any sm), plus the lambda
// re-parameterisation kernel and the bounded-wait self-test kernel.
//
// The fp32 workload needs 1e-4 agreement after the per-head RMSNorm, which
// tf32 tensor-core operands (10-bit mantissa) cannot hold; this kernel keeps
// every product and sum in fp32 FFMA and calls expf.
//
// One CTA owns 8 query rows of one (batch, unit); each warp owns one row.  Key
// tiles of 32 keys (K1, K2, V) are staged in shared memory (K rows padded to
// d + 1 floats so that lane = key reads are conflict-free).  Per tile a lane
// scores its key against the warp's rows for both maps, the two online
// (max, sum) states are updated with warp shuffles, and every lane
// accumulates its value channels (lane + 32 c) of O1 and O2.  Epilogue:
// O1 / l1 - c O2 / l2, then the V1 per-head RMSNorm x (1 - lambda_init).
//
// With BWD (V1 only) the same sweep is the backward pass's row pass: the
// epilogue writes, per query row, the maps' log-sum-exps, dO (the gradient
// of the pre-norm output, through the RMSNorm), D_r = rowsum(A_r * dA_r) and
// the row's share of dlambda, and per CTA its share of dgamma (the dK/dV and
// dQ sweeps are in backward.cuh).
#pragma once

#include "bwd_params.h"
#include "params.h"
#include "ptx.cuh"
#include "stage.cuh"

#undef DA_BOUNDS_FILE
#define DA_BOUNDS_FILE 8

namespace da {


// Key-row pitch in shared memory: d + 4 when d % 32 == 0 (16-byte rows, and
// the float4 reads of eight consecutive lanes fall on 32 different banks),
// else d + 1 (odd: a lane per row reads scalars without conflicts).
__host__ __device__ constexpr int simt_kpitch(int d) { return d % 32 == 0 ? d + 4 : d + 1; }

// Shared-memory floats the kernel needs for query/key width d and value width dv.
__host__ __device__ constexpr int simt_smem_floats(int d, int dv) {
  return 2 * kSimtRows * d + 2 * kSimtKeys * simt_kpitch(d) + kSimtKeys * dv;
}

template <bool BWD>
__global__ void __launch_bounds__(kSimtWarps * 32) simt_fwd_f32_kernel(const SimtParams p, const SimtBwdExtra x) {
  extern __shared__ float sm[];
  constexpr int R = kSimtRows / kSimtWarps;  // query rows per warp
  constexpr int NC = kSimtMaxVPerLane;       // value channels per lane (lane + 32 c)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = p.d, dv = p.dv, dp = simt_kpitch(d);
  float* sq1 = sm;
  float* sq2 = sq1 + kSimtRows * d;
  float* sk1 = sq2 + kSimtRows * d;
  float* sk2 = sk1 + kSimtKeys * dp;
  float* sv = sk2 + kSimtKeys * dp;

  const int nqb = (p.n + kSimtRows - 1) / kSimtRows;
  const int unit = blockIdx.x / nqb;
  const int qb = nqb - 1 - static_cast<int>(blockIdx.x % nqb);  // heaviest causal blocks first
  const int u = unit % p.units_per_batch, b = unit / p.units_per_batch;
  int hq1, hq2, hk;
  if (p.v2) {
    hq1 = 2 * u;
    hq2 = 2 * u + 1;
    hk = hq1 / p.group;
  } else {
    hq1 = hq2 = hk = u;
  }
  const int q0 = qb * kSimtRows;
  const size_t qrow = static_cast<size_t>(p.heads_q) * d;
  const size_t krow = static_cast<size_t>(p.heads_kv) * d;
  const size_t vrow = static_cast<size_t>(p.heads_kv) * dv;
  const float* gq1 = p.q1 + (static_cast<size_t>(b) * p.n) * qrow + static_cast<size_t>(hq1) * d;
  const float* gq2 = p.q2 + (static_cast<size_t>(b) * p.n) * qrow + static_cast<size_t>(hq2) * d;
  const float* gk1 = p.k1 + (static_cast<size_t>(b) * p.n) * krow + static_cast<size_t>(hk) * d;
  const float* gk2 = p.k2 + (static_cast<size_t>(b) * p.n) * krow + static_cast<size_t>(hk) * d;
  const float* gv = p.v + (static_cast<size_t>(b) * p.n) * vrow + static_cast<size_t>(hk) * dv;

  // Every load of a tile is issued before any of them is consumed, so a tile
  // costs one memory round trip (16-byte loads when rows allow it).
  const bool vec = ((d & 3) == 0) && ((reinterpret_cast<uintptr_t>(p.q1) | reinterpret_cast<uintptr_t>(p.q2) |
                                       reinterpret_cast<uintptr_t>(p.k1) | reinterpret_cast<uintptr_t>(p.k2) |
                                       reinterpret_cast<uintptr_t>(p.v)) & 15u) == 0;
  stage_rows(sq1, d, gq1, qrow, q0, p.n, d, kSimtRows, vec);
  stage_rows(sq2, d, gq2, qrow, q0, p.n, d, kSimtRows, vec);

  float m1[R], l1[R], m2[R], l2[R], o1[R][NC], o2[R][NC];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    m1[r] = m2[r] = -INFINITY;
    l1[r] = l2[r] = 0.f;
#pragma unroll
    for (int c = 0; c < NC; ++c) o1[r][c] = o2[r][c] = 0.f;
  }
  const int kend = p.causal ? min(p.n, q0 + kSimtRows) : p.n;
  for (int k0 = 0; k0 < kend; k0 += kSimtKeys) {
    __syncthreads();
    stage_rows(sk1, dp, gk1, krow, k0, p.n, d, kSimtKeys, vec);
    stage_rows(sk2, dp, gk2, krow, k0, p.n, d, kSimtKeys, vec);
    stage_rows(sv, dv, gv, vrow, k0, p.n, dv, kSimtKeys, vec);
    __syncthreads();
    const int key = k0 + lane;  // this lane's key in the tile
    float pr1[R], pr2[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int row = warp * R + r, t = q0 + row;
      float s1 = 0.f, s2 = 0.f;
      if (d % 32 == 0) {  // float4 reads, the same products in the same order
        for (int e = 0; e < d; e += 4) {
          const float4 a1 = *reinterpret_cast<const float4*>(sq1 + row * d + e);
          const float4 b1 = *reinterpret_cast<const float4*>(sk1 + lane * dp + e);
          const float4 a2 = *reinterpret_cast<const float4*>(sq2 + row * d + e);
          const float4 b2 = *reinterpret_cast<const float4*>(sk2 + lane * dp + e);
          s1 = fmaf(a1.w, b1.w, fmaf(a1.z, b1.z, fmaf(a1.y, b1.y, fmaf(a1.x, b1.x, s1))));
          s2 = fmaf(a2.w, b2.w, fmaf(a2.z, b2.z, fmaf(a2.y, b2.y, fmaf(a2.x, b2.x, s2))));
        }
      } else {
        for (int e = 0; e < d; ++e) {
          s1 = fmaf(sq1[row * d + e], sk1[lane * dp + e], s1);
          s2 = fmaf(sq2[row * d + e], sk2[lane * dp + e], s2);
        }
      }
      const bool vis = key < p.n && (!p.causal || key <= t);
      s1 = vis ? s1 * p.scale : -INFINITY;
      s2 = vis ? s2 * p.scale : -INFINITY;
      float mx1 = s1, mx2 = s2;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        mx2 = fmaxf(mx2, __shfl_xor_sync(0xffffffffu, mx2, off));
      }
      const float n1 = fmaxf(m1[r], mx1), n2 = fmaxf(m2[r], mx2);
      // A row sees at least key 0 in the first tile, so n1, n2 are finite.
      const float f1 = expf(m1[r] - n1), f2 = expf(m2[r] - n2);
      pr1[r] = expf(s1 - n1);
      pr2[r] = expf(s2 - n2);
      float sum1 = pr1[r], sum2 = pr2[r];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        sum1 += __shfl_xor_sync(0xffffffffu, sum1, off);
        sum2 += __shfl_xor_sync(0xffffffffu, sum2, off);
      }
      l1[r] = l1[r] * f1 + sum1;
      l2[r] = l2[r] * f2 + sum2;
      m1[r] = n1;
      m2[r] = n2;
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        o1[r][c] *= f1;
        o2[r][c] *= f2;
      }
    }
    const int cnt = min(kSimtKeys, kend - k0);
    for (int kk = 0; kk < cnt; ++kk) {
      float vv[NC];
#pragma unroll
      for (int c = 0; c < NC; ++c) vv[c] = (lane + 32 * c < dv) ? sv[kk * dv + lane + 32 * c] : 0.f;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float w1 = __shfl_sync(0xffffffffu, pr1[r], kk);
        const float w2 = __shfl_sync(0xffffffffu, pr2[r], kk);
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          o1[r][c] = fmaf(w1, vv[c], o1[r][c]);
          o2[r][c] = fmaf(w2, vv[c], o2[r][c]);
        }
      }
    }
  }

  if constexpr (BWD) {
    static_assert(R == 1, "one query row per warp");
    // Backward row pass.  V1, with m = 1 - lambda_init, O_r = A_r V, O = O_1 - lambda O_2,
    // Oh = O / rms(O), g = m gamma dy:
    //   dO = (g - Oh mean(g Oh)) / rms(O);  D_1 = dO . O_1;  D_2 = -lambda dO . O_2;
    //   dlambda_row = -dO . O_2;  dgamma += m Oh dy.
    // V2 (no norm, s = sigmoid(logit) of the row): dO = dy;  D_1 = dO . O_1;
    //   D_2 = -s dO . O_2;  dlogit_row = -s (1 - s) dO . O_2.
    // Row slots: lse_1, lse_2, D_1, D_2, dlambda / dlogit share, coefficient (lambda or s).
    __syncthreads();  // every warp is done with the key tiles: sk1 now stages dgamma rows
    float* sdg = sk1;  // [kSimtWarps][dv] (32 (d + 1) >= 8 dv floats; sk2 follows)
    const int t = q0 + warp;
    const long long R_rows = p.rows_total;
    if (t < p.n) {  // warp-uniform
      const float coef =
          p.v2 ? 1.f / (1.f + expf(-p.lam_logits[b * p.sb + static_cast<long long>(t) * p.st + u])) : *p.lambda;
      const float a1 = 1.f / l1[0], a2 = 1.f / l2[0];
      float o1n[NC], o2n[NC], y[NC], ss = 0.f;
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        o1n[c] = o1[0][c] * a1;
        o2n[c] = o2[0][c] * a2;
        y[c] = o1n[c] - coef * o2n[c];
        if (lane + 32 * c < dv) ss = fmaf(y[c], y[c], ss);
      }
      const long long ri = (static_cast<long long>(b) * p.units_per_batch + u) * p.n + t;
      const float* dyrow = x.dy + ((static_cast<size_t>(b) * p.n + t) * p.units_per_batch + u) * dv;
      float dOv[NC];
      if (p.v2) {
#pragma unroll
        for (int c = 0; c < NC; ++c) dOv[c] = (lane + 32 * c < dv) ? dyrow[lane + 32 * c] : 0.f;
      } else {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        const float rinv = rsqrtf(ss / dv + p.eps);
        float g[NC], oh[NC], gs = 0.f;
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          const int col = lane + 32 * c;
          g[c] = oh[c] = 0.f;
          if (col < dv) {
            const float dyc = dyrow[col];
            g[c] = p.norm_mult * (p.gamma != nullptr ? p.gamma[col] : 1.f) * dyc;
            oh[c] = y[c] * rinv;
            gs = fmaf(g[c], oh[c], gs);
            sdg[warp * dv + col] = p.norm_mult * oh[c] * dyc;
          }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) gs += __shfl_xor_sync(0xffffffffu, gs, off);
        const float gmean = gs / dv;
#pragma unroll
        for (int c = 0; c < NC; ++c) dOv[c] = (g[c] - oh[c] * gmean) * rinv;
      }
      float dd1 = 0.f, dd2 = 0.f;
      float* dorow = x.ws_do + ri * dv;
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        const int col = lane + 32 * c;
        if (col < dv) {
          DA_STORE(dorow, col, (R_rows - ri) * dv, dOv[c]);
          dd1 = fmaf(dOv[c], o1n[c], dd1);
          dd2 = fmaf(dOv[c], o2n[c], dd2);
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        dd1 += __shfl_xor_sync(0xffffffffu, dd1, off);
        dd2 += __shfl_xor_sync(0xffffffffu, dd2, off);
      }
      if (lane == 0 && DA_BOUNDS_V(ri >= 0 && ri < R_rows && b < p.B && t < p.n && u < p.units_per_batch, ri)) {
        const float share = p.v2 ? -coef * (1.f - coef) * dd2 : -dd2;
        x.ws_row[ri] = m1[0] + logf(l1[0]);
        x.ws_row[R_rows + ri] = m2[0] + logf(l2[0]);
        x.ws_row[2 * R_rows + ri] = dd1;
        x.ws_row[3 * R_rows + ri] = -coef * dd2;
        x.ws_row[4 * R_rows + ri] = share;
        x.ws_row[5 * R_rows + ri] = coef;
        if (x.dlogits_dense != nullptr)  // V2 with one logit per token: its gradient directly
          x.dlogits_dense[b * p.sb + static_cast<long long>(t) * p.st + u] = share;
      }
    } else if (!p.v2) {
      for (int col = lane; col < dv; col += 32) sdg[warp * dv + col] = 0.f;
    }
    __syncthreads();
    if (!p.v2) {
      for (int col = threadIdx.x; col < dv; col += kSimtWarps * 32) {
        float a = 0.f;
#pragma unroll
        for (int w = 0; w < kSimtWarps; ++w) a += sdg[w * dv + col];
        DA_STORE(x.ws_dgamma, static_cast<size_t>(blockIdx.x) * dv + col, static_cast<size_t>(gridDim.x) * dv, a);
      }
    }
  } else {
  // ---- epilogue: out = O1 / l1 - c O2 / l2 (then the V1 norm)
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int t = q0 + warp * R + r;
    if (t >= p.n) continue;  // warp-uniform
    float coef;
    if (p.v2) {
      coef = 1.f / (1.f + expf(-p.lam_logits[b * p.sb + static_cast<long long>(t) * p.st + u]));
    } else {
      coef = *p.lambda;
    }
    const float a1 = 1.f / l1[r], a2 = coef / l2[r];
    float y[NC];
    float ss = 0.f;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      y[c] = o1[r][c] * a1 - o2[r][c] * a2;
      if (lane + 32 * c < dv) ss = fmaf(y[c], y[c], ss);
    }
    float rinv = 1.f;
    if (!p.v2) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
      rinv = p.norm_mult * rsqrtf(ss / dv + p.eps);
    }
    float* orow = p.out + ((static_cast<size_t>(b) * p.n + t) * p.units_per_batch + u) * dv;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const int col = lane + 32 * c;
      if (col < dv) {
        float v = y[c] * rinv;
        if (!p.v2 && p.gamma != nullptr) v *= p.gamma[col];
        if (DA_BOUNDS_V(b < p.B && u < p.units_per_batch, t)) orow[col] = v;
      }
    }
  }
  }  // !BWD
}

// lambda = exp(<lq1, lk1>) - exp(<lq2, lk2>) + lambda_init, one warp.
__global__ void lambda_reparam_kernel(const float* lq1, const float* lk1, const float* lq2, const float* lk2,
                                      int dim, float lambda_init, float* out) {
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
  if (threadIdx.x == 0) *out = expf(a) - expf(c) + lambda_init;
}

// Self-test of the bounded wait: one thread waits on an mbarrier that nothing
// arrives on; the wait must run out and record the timeout status.
__global__ void wait_timeout_selftest_kernel(unsigned long long budget_cycles, int* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const AbortState ab{&flag, status};
    mbar_wait(&bar, 0, ab, budget_cycles);
  }
}

}  // namespace da
