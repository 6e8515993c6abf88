// Per-row preparation of the tensor-core backward from a training forward's
// saved statistics (CUDA cores, memory-bound).
//
// The training forward (one-sweep kernel with SAVE) keeps, per row, lse_1,
// lse_2 and the normalised map outputs O_1, O_2 (bf16).  From them and dy
// this kernel writes what the statistics pass would, without recomputing
// the attention:
//   V1 (per-head RMSNorm, "Differential Transformer" glossary page, "How
//   differential attention works"; news article section "差分注意力"):
//     O = O_1 - lambda O_2,  r = (mean O^2 + eps)^-1/2,  G = m gamma dy
//     (m = 1 - lambda_init),  dO = r G - (r^3 / DV) (G . O) O  (bf16);
//     Delta_1 = dO . O_1,  Delta_2 = -lambda dO . O_2,  share = -dO . O_2
//     (the row's dL/dlambda),  coefficient lambda; dgamma share of a row
//     m dy O r per channel.
//   V2 (DIFF V2 analysis page, "2. 커스텀 커널 제거"): s = sigmoid(logit),
//     dO = dy;  Delta_1 = dy . O_1,  Delta_2 = -s dy . O_2,
//     share = -s (1 - s) dy . O_2 (the row's dL/dlogit),  coefficient s.
// The dot products use the identity dO . X = r G . X - (r^3 / DV)(G . O)(O . X)
// so that each row needs one pass over its channels.  One warp per row, 4
// channels per lane; a CTA of 8 warps takes 128 consecutive rows (BSHD
// order) and writes one dgamma / dlambda partial, so the reduction that
// follows sums them in a fixed order.
#pragma once

#include <cuda_bf16.h>

#include "ptx.cuh"

#undef DA_BOUNDS_FILE
#define DA_BOUNDS_FILE 10

namespace da {

struct BwdPrepParams {
  const __nv_bfloat16* dy;  // [B, n, units, 128]
  const __nv_bfloat16* o1;  // saved O_1: [B units][128-row tiles][4 channel blocks][128 rows][32 channels]
  const __nv_bfloat16* o2;  // saved O_2, same layout
  const float* lse;         // saved [2][rows]: lse_1, lse_2 (row ri = (b units + u) n + t)
  const float* lambda;      // V1: device scalar
  const float* gamma;       // V1: [128] or nullptr
  const float* lam_logits;  // V2: logit of (b, t, u) at b sb + t st + u
  long long sb, st;
  float norm_mult, eps;     // V1
  int B, n, units;
  long long rows;           // B * units * n
  __nv_bfloat16* dO;        // V1 out: [B, n, units, 128]
  float* row;               // out [6][rows]: lse_1, lse_2, Delta_1, Delta_2, share, coefficient
  float* dgp;               // V1 out: [gridDim.x][128] dgamma partials
  float* dlam_part;         // V1 out: [gridDim.x] dlambda partials
  float* dlogits_dense;     // V2, one logit per token: dlogit of (b, t, u) at b sb + t st + u, or nullptr
};

constexpr int kPrepWarps = 8;
constexpr int kPrepRowsPerWarp = 16;
constexpr int kPrepRowsPerCta = kPrepWarps * kPrepRowsPerWarp;  // 128
constexpr int kPrepIlp = 4;  // rows whose loads a warp issues together

__device__ __forceinline__ void bf16x4_to_f32(uint2 w, float (&f)[4]) {
  f[0] = __uint_as_float(w.x << 16);
  f[1] = __uint_as_float(w.x & 0xffff0000u);
  f[2] = __uint_as_float(w.y << 16);
  f[3] = __uint_as_float(w.y & 0xffff0000u);
}

template <bool V2>
__global__ void __launch_bounds__(kPrepWarps * 32, 3) bwd_prep_kernel(const __grid_constant__ BwdPrepParams p) {
  constexpr int DV = 128;
  __shared__ float sdg[kPrepWarps][DV];
  __shared__ float sdl[kPrepWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c0 = 4 * lane;
  float gam[4] = {1.f, 1.f, 1.f, 1.f};
  if (!V2 && p.gamma != nullptr)
#pragma unroll
    for (int e = 0; e < 4; ++e) gam[e] = p.gamma[c0 + e];
  const float lam = V2 ? 0.f : *p.lambda;
  float dg[4] = {0.f, 0.f, 0.f, 0.f}, dl = 0.f;
  // Rows in groups of kPrepIlp: every load of a group is issued before the
  // first row's arithmetic, so each warp keeps several rows' reads in flight.
  for (int j0 = 0; j0 < kPrepRowsPerWarp; j0 += kPrepIlp) {
    const long long ob = static_cast<long long>(blockIdx.x) * kPrepRowsPerCta + warp * kPrepRowsPerWarp + j0;
    if (ob >= p.rows) break;  // warp-uniform
    // (batch, token, unit) of the group's rows: the first by division, the next by stepping the unit
    // (32-bit: rows < 2^31); ri = the row's index in the statistics arrays.
    long long ris[kPrepIlp];
    int bs[kPrepIlp], ts[kPrepIlp], us[kPrepIlp];
    {
      int u = static_cast<int>(ob) % p.units;
      const int bt = static_cast<int>(ob) / p.units;
      int t = bt % p.n, b = bt / p.n;
#pragma unroll
      for (int jj = 0; jj < kPrepIlp; ++jj) {
        if (jj > 0 && ++u == p.units) {
          u = 0;
          if (++t == p.n) {
            t = 0;
            ++b;
          }
        }
        bs[jj] = b;
        ts[jj] = t;
        us[jj] = u;
        ris[jj] = (static_cast<long long>(b) * p.units + u) * p.n + t;
      }
    }
    uint2 wdy[kPrepIlp], wo1[kPrepIlp], wo2[kPrepIlp];
    float lse_v[kPrepIlp];  // lanes 0, 1: lse_1, lse_2 of the row
    const int ntiles = (p.n + 127) / 128;
#pragma unroll
    for (int jj = 0; jj < kPrepIlp; ++jj) {
      const bool in = ob + jj < p.rows;
      const long long o = in ? ob + jj : ob;
      // this lane's 4 channels c0 .. c0 + 3: block c0 / 32 of the row's tile
      const long long so =
          ((((static_cast<long long>(bs[jj]) * p.units + us[jj]) * ntiles + ts[jj] / 128) * 4 + (c0 >> 5)) * 128 +
           ts[jj] % 128) * 32 + (c0 & 31);
      wdy[jj] = *reinterpret_cast<const uint2*>(p.dy + o * DV + c0);
      wo1[jj] = *reinterpret_cast<const uint2*>(p.o1 + so);
      wo2[jj] = *reinterpret_cast<const uint2*>(p.o2 + so);
      lse_v[jj] = (lane < 2 && in) ? p.lse[lane * p.rows + ris[jj]] : 0.f;
    }
#pragma unroll
  for (int jj = 0; jj < kPrepIlp; ++jj) {
    const long long o = ob + jj;
    if (o >= p.rows) break;  // warp-uniform
    const int u = us[jj], t = ts[jj], b = bs[jj];
    const long long ri = ris[jj];
    float dy[4], x1[4], x2[4];
    bf16x4_to_f32(wdy[jj], dy);
    bf16x4_to_f32(wo1[jj], x1);
    bf16x4_to_f32(wo2[jj], x2);
    float delta1, delta2, share, coef;
    if constexpr (!V2) {
      // partial sums: O.O, G.O, G.O_1, G.O_2, O.O_1, O.O_2
      float ov[4], gv[4], s[6] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        ov[e] = fmaf(-lam, x2[e], x1[e]);
        gv[e] = p.norm_mult * gam[e] * dy[e];
        s[0] = fmaf(ov[e], ov[e], s[0]);
        s[1] = fmaf(gv[e], ov[e], s[1]);
        s[2] = fmaf(gv[e], x1[e], s[2]);
        s[3] = fmaf(gv[e], x2[e], s[3]);
        s[4] = fmaf(ov[e], x1[e], s[4]);
        s[5] = fmaf(ov[e], x2[e], s[5]);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1)
#pragma unroll
        for (int k = 0; k < 6; ++k) s[k] += __shfl_xor_sync(0xffffffffu, s[k], off);
      const float r = rsqrtf(s[0] * (1.f / DV) + p.eps);
      const float k3 = r * r * r * (1.f / DV) * s[1];
      uint32_t w[2];
#pragma unroll
      for (int e = 0; e < 4; e += 2) {
        const float d0 = fmaf(r, gv[e], -k3 * ov[e]), d1 = fmaf(r, gv[e + 1], -k3 * ov[e + 1]);
        w[e >> 1] = pack_bf16x2(d0, d1);
        dg[e] = fmaf(dy[e] * p.norm_mult, ov[e] * r, dg[e]);
        dg[e + 1] = fmaf(dy[e + 1] * p.norm_mult, ov[e + 1] * r, dg[e + 1]);
      }
      DA_STORE(reinterpret_cast<uint2*>(p.dO), (o * DV + c0) / 4, p.rows * DV / 4, make_uint2(w[0], w[1]));
      const float dOO1 = fmaf(r, s[2], -k3 * s[4]), dOO2 = fmaf(r, s[3], -k3 * s[5]);
      delta1 = dOO1;
      delta2 = -lam * dOO2;
      share = -dOO2;
      coef = lam;
      dl += share;
    } else {
      float s1 = 0.f, s2 = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        s1 = fmaf(dy[e], x1[e], s1);
        s2 = fmaf(dy[e], x2[e], s2);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        s1 += __shfl_xor_sync(0xffffffffu, s1, off);
        s2 += __shfl_xor_sync(0xffffffffu, s2, off);
      }
      const long long li = b * p.sb + static_cast<long long>(t) * p.st + u;
      const float sg = 1.f / (1.f + expf(-p.lam_logits[li]));
      delta1 = s1;
      delta2 = -sg * s2;
      share = -sg * (1.f - sg) * s2;
      coef = sg;
      if (lane == 0 && p.dlogits_dense != nullptr) p.dlogits_dense[li] = share;
    }
    // lanes 0-5 write the row's six values (every lane holds the reduced ones)
    if (lane < 6 && DA_BOUNDS_V(ri >= 0 && ri < p.rows, ri)) {
      const float val = lane < 2 ? lse_v[jj] : (lane == 2 ? delta1 : lane == 3 ? delta2 : lane == 4 ? share : coef);
      p.row[lane * p.rows + ri] = val;
    }
  }
  }
  if constexpr (!V2) {
#pragma unroll
    for (int e = 0; e < 4; ++e) sdg[warp][c0 + e] = dg[e];
    if (lane == 0) sdl[warp] = dl;
    __syncthreads();
    if (threadIdx.x < DV) {
      float a = 0.f;
#pragma unroll
      for (int w = 0; w < kPrepWarps; ++w) a += sdg[w][threadIdx.x];
      DA_STORE(p.dgp, static_cast<long long>(blockIdx.x) * DV + threadIdx.x, static_cast<long long>(gridDim.x) * DV, a);
    }
    if (threadIdx.x == 0) {
      float a = 0.f;
#pragma unroll
      for (int w = 0; w < kPrepWarps; ++w) a += sdl[w];
      DA_STORE(p.dlam_part, blockIdx.x, gridDim.x, a);
    }
  }
}

}  // namespace da
