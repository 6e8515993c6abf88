// fp32 differential-attention forward on CUDA cores (any sm), plus the lambda
// re-parameterisation kernel and the bounded-wait self-test kernel.
//
// The fp32 workload needs 1e-4 agreement after the per-head RMSNorm, which
// tf32 tensor-core operands (10-bit mantissa) cannot hold; this kernel keeps
// every product and sum in fp32 FFMA.
//
// One warp owns one (batch, unit, query) row:
//   sweep 1  lanes split the visible keys; each lane computes full dot
//            products q1.k1_j, q2.k2_j and keeps a running (max, sum) per map;
//            the 32 partial states are merged with shuffles;
//   sweep 2  each lane forms p_j = e1_j / l1 - c e2_j / l2 for its keys;
//            the p_j are broadcast and every lane accumulates its value
//            channels (lane + 32 i) of O = sum_j p_j v_j;
//   epilogue V1: (1 - lambda_init) * gamma * O / sqrt(mean(O^2) + eps);
//            V2: O.
#pragma once

#include "params.h"
#include "ptx.cuh"

namespace da {


__global__ void __launch_bounds__(kSimtWarps * 32) simt_fwd_f32_kernel(const SimtParams p) {
  __shared__ float qs[kSimtWarps][2][kSimtMaxD];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long r = static_cast<long long>(blockIdx.x) * kSimtWarps + warp;
  if (r >= p.rows_total) return;
  const int t = static_cast<int>(r % p.n);
  const long long bu = r / p.n;
  const int u = static_cast<int>(bu % p.units_per_batch);
  const int b = static_cast<int>(bu / p.units_per_batch);
  int hq1, hq2, hk;
  if (p.v2) {
    hq1 = 2 * u;
    hq2 = 2 * u + 1;
    hk = hq1 / p.group;
  } else {
    hq1 = hq2 = hk = u;
  }
  const int d = p.d, dv = p.dv;
  const float* q1 = p.q1 + ((static_cast<size_t>(b) * p.n + t) * p.heads_q + hq1) * d;
  const float* q2 = p.q2 + ((static_cast<size_t>(b) * p.n + t) * p.heads_q + hq2) * d;
  for (int c = lane; c < d; c += 32) {
    qs[warp][0][c] = q1[c];
    qs[warp][1][c] = q2[c];
  }
  __syncwarp();
  const int kend = p.causal ? t + 1 : p.n;
  const size_t kstride = static_cast<size_t>(p.heads_kv) * d;
  const size_t vstride = static_cast<size_t>(p.heads_kv) * dv;
  const float* k1 = p.k1 + (static_cast<size_t>(b) * p.n * p.heads_kv + hk) * d;
  const float* k2 = p.k2 + (static_cast<size_t>(b) * p.n * p.heads_kv + hk) * d;
  const float* vb = p.v + (static_cast<size_t>(b) * p.n * p.heads_kv + hk) * dv;

  // ---- sweep 1: per-lane running max / sum, then merged across the warp
  float m1 = -INFINITY, l1 = 0.f, m2 = -INFINITY, l2 = 0.f;
  for (int j = lane; j < kend; j += 32) {
    const float* a = k1 + j * kstride;
    const float* c = k2 + j * kstride;
    float s1 = 0.f, s2 = 0.f;
    for (int e = 0; e < d; ++e) {
      s1 = fmaf(qs[warp][0][e], a[e], s1);
      s2 = fmaf(qs[warp][1][e], c[e], s2);
    }
    s1 *= p.scale;
    s2 *= p.scale;
    float mn = fmaxf(m1, s1);
    l1 = l1 * expf(m1 - mn) + expf(s1 - mn);
    m1 = mn;
    mn = fmaxf(m2, s2);
    l2 = l2 * expf(m2 - mn) + expf(s2 - mn);
    m2 = mn;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float om1 = __shfl_xor_sync(0xffffffffu, m1, off), ol1 = __shfl_xor_sync(0xffffffffu, l1, off);
    const float om2 = __shfl_xor_sync(0xffffffffu, m2, off), ol2 = __shfl_xor_sync(0xffffffffu, l2, off);
    float mn = fmaxf(m1, om1);
    if (mn != -INFINITY) {
      l1 = l1 * expf(m1 - mn) + ol1 * expf(om1 - mn);
      m1 = mn;
    }
    mn = fmaxf(m2, om2);
    if (mn != -INFINITY) {
      l2 = l2 * expf(m2 - mn) + ol2 * expf(om2 - mn);
      m2 = mn;
    }
  }
  float coef;
  if (p.v2) {
    const float lg = p.lam_logits[b * p.sb + static_cast<long long>(t) * p.st + u];
    coef = 1.f / (1.f + expf(-lg));
  } else {
    coef = *p.lambda;
  }
  const float inv1 = 1.f / l1, c2 = coef / l2;

  // ---- sweep 2: O = sum_j p_j v_j, channels lane + 32 i
  float o[kSimtMaxVPerLane];
#pragma unroll
  for (int i = 0; i < kSimtMaxVPerLane; ++i) o[i] = 0.f;
  for (int j0 = 0; j0 < kend; j0 += 32) {
    const int j = j0 + lane;
    float pj = 0.f;
    if (j < kend) {
      const float* a = k1 + j * kstride;
      const float* c = k2 + j * kstride;
      float s1 = 0.f, s2 = 0.f;
      for (int e = 0; e < d; ++e) {
        s1 = fmaf(qs[warp][0][e], a[e], s1);
        s2 = fmaf(qs[warp][1][e], c[e], s2);
      }
      pj = expf(s1 * p.scale - m1) * inv1 - expf(s2 * p.scale - m2) * c2;
    }
    const int cnt = min(32, kend - j0);
    for (int jj = 0; jj < cnt; ++jj) {
      const float w = __shfl_sync(0xffffffffu, pj, jj);
      const float* vr = vb + (j0 + jj) * vstride;
#pragma unroll
      for (int i = 0; i < kSimtMaxVPerLane; ++i) {
        const int c = lane + 32 * i;
        if (c < dv) o[i] = fmaf(w, vr[c], o[i]);
      }
    }
  }

  // ---- epilogue
  float rinv = 1.f;
  if (!p.v2) {
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < kSimtMaxVPerLane; ++i)
      if (lane + 32 * i < dv) ss = fmaf(o[i], o[i], ss);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    rinv = p.norm_mult * rsqrtf(ss / dv + p.eps);
  }
  float* orow = p.out + ((static_cast<size_t>(b) * p.n + t) * p.units_per_batch + u) * dv;
#pragma unroll
  for (int i = 0; i < kSimtMaxVPerLane; ++i) {
    const int c = lane + 32 * i;
    if (c < dv) {
      float y = o[i] * rinv;
      if (!p.v2 && p.gamma != nullptr) y *= p.gamma[c];
      orow[c] = y;
    }
  }
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
__global__ void wait_timeout_selftest_kernel(unsigned long long budget_ns, int* status) {
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
    mbar_wait(&bar, 0, ab, budget_ns);
  }
}

}  // namespace da
