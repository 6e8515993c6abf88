// Two-sweep differential-attention forward on tcgen05 tensor cores (sm_103a).
//
// What it computes (per (batch, unit, 128-query tile)):
//   map r in {1, 2}:  A_r = softmax(Q_r K_r^T * scale)            (masked)
//   O   = (A_1 - c * A_2) V                                        one accumulator
//   V1: out = (1 - lambda_init) * gamma * O / sqrt(mean(O^2) + eps), c = lambda
//   V2: out = O, c = sigmoid(logit[b, t, pair]), Q_1/Q_2 = query heads 2g/2g+1
//       sharing one K/V head.
// ("Differential Transformer" glossary page, "How differential attention
// works"; DIFF V2 analysis page, sections on the DiffAttn operator, the V2
// code and GQA pairing; news article section "差分注意力" for the per-head
// RMSNorm and (1 - lambda_init).)
//
// Why two sweeps: the combined weights A_1 - c A_2 need the final row maxima
// and sums of both maps.  Sweep 1 computes S_1, S_2 tile by tile and keeps
// only (m_r, l_r) per row.  Sweep 2 recomputes S_1, S_2 and forms the signed
// weights P = 2^(s1*k - M1) - sign(c) 2^(s2*k - M2) (with the 1/l_r and |c|
// folded into M_r), so ONE P.V product serves both maps.  With a value width
// of 2d this costs exactly the tensor flops of the one-sweep form
// (4d + 4d + 4d per query-key pair against 4d + 8d) and needs one fp32
// accumulator instead of two, which is what lets d = 128 / V = 256 fit the
// 512 TMEM columns of an SM; it also removes every rescale of O.
//
// Roles (384 threads, one CTA per SM):
//   warp 0      TMA producer: Q_1, Q_2 once; K_1, K_2 (+ V in sweep 2) per
//               64-key tile into a STAGES-deep ring of shared memory.
//   warp 1      TMEM allocator and single-thread tcgen05.mma issuer.
//   warps 4-11  two warpgroups; thread = one query row (TMEM lane).
//               Sweep 1: warpgroup r keeps the statistics of map r.
//               Sweep 2: warpgroup w owns key columns [32w, 32w+32) of both
//               maps, writes its bf16 P into TMEM over its own S_1 columns.
//               Epilogue: warpgroup w normalises/stores channels of half w.
// TMEM (512 columns x 128 lanes, fp32): O at [0, DV); S stage s at
// DV + 128 s: S_1 in [0, 64), S_2 in [64, 128) of the stage; P of stage s
// (bf16 pairs) at stage columns [0, 16) and [32, 48).
#pragma once

#include <cuda_bf16.h>

#include "params.h"
#include "ptx.cuh"

namespace da {


template <int D, int DV, bool SHARED_K, int EPI, int STAGES>
struct TwoPassCfg {
  static constexpr int BM = 128;  // queries per CTA (TMEM lanes)
  static constexpr int BN = 64;   // keys per tile
  static constexpr int NTHREADS = 384;
  static constexpr int QB = D / 64;  // 128-byte swizzle boxes across a Q/K row
  static constexpr int VB = DV / 64;
  static constexpr int Q_TILE = BM * D * 2;
  static constexpr int K_TILE = BN * D * 2;
  static constexpr int V_TILE = BN * DV * 2;
  static constexpr int NK = SHARED_K ? 1 : 2;
  static constexpr int STAGE = NK * K_TILE + V_TILE;
  static constexpr int OFF_Q1 = 0;
  static constexpr int OFF_Q2 = Q_TILE;
  static constexpr int OFF_STAGES = 2 * Q_TILE;
  static constexpr int OFF_BARS = OFF_STAGES + STAGES * STAGE;
  static constexpr int NBARS = 2 + 2 * STAGES + 4;
  static constexpr int OFF_MISC = OFF_BARS + NBARS * 8;
  static constexpr int OFF_STATS = ((OFF_MISC + 16) + 15) / 16 * 16;
  static constexpr int STATS_BYTES = 6 * 128 * 4;  // m[2][128], l[2][128], ss[2][128]
  static constexpr int SMEM_BYTES = OFF_STATS + STATS_BYTES + 1024;  // + 1 KB alignment slack
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t TM_O = 0;
  static constexpr uint32_t TM_S = DV;
  static constexpr uint32_t IDESC_QK = idesc_bf16(BM, BN, false, false);
  static constexpr uint32_t IDESC_PV = idesc_bf16(BM, DV, false, true);
  static_assert(D == 64 || D == 128, "query/key width");
  static_assert(DV % 64 == 0 && DV <= 256 && DV + 256 <= 512, "value width");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
};

template <int D, int DV, bool SHARED_K, int EPI, int STAGES>
__global__ void __launch_bounds__(384, 1) twopass_fwd_kernel(const __grid_constant__ TwoPassParams p) {
  using C = TwoPassCfg<D, DV, SHARED_K, EPI, STAGES>;
  constexpr int BM = C::BM, BN = C::BN;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BARS);
  uint64_t* q_full = bars + 0;
  uint64_t* o_full = bars + 1;
  uint64_t* kv_full = bars + 2;
  uint64_t* kv_empty = bars + 2 + STAGES;
  uint64_t* s_full = bars + 2 + 2 * STAGES;
  uint64_t* s_free = s_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  float* stat_m = reinterpret_cast<float*>(smem + C::OFF_STATS);
  float* stat_l = stat_m + 256;
  float* stat_ss = stat_m + 512;

  // ---- which tile this CTA owns
  const int units = p.B * p.units_per_batch;
  int unit, qt;
  if (p.order == 0) {
    unit = blockIdx.x / p.num_q_tiles;
    qt = p.num_q_tiles - 1 - static_cast<int>(blockIdx.x % p.num_q_tiles);
  } else {
    qt = p.num_q_tiles - 1 - static_cast<int>(blockIdx.x / units);
    unit = blockIdx.x % units;
  }
  const int b = unit / p.units_per_batch;
  const int u = unit % p.units_per_batch;
  int hq1, hq2, hk;
  if (EPI == kEpiRmsNorm) {
    hq1 = hq2 = hk = u;
  } else {
    hq1 = 2 * u;
    hq2 = 2 * u + 1;
    hk = hq1 / p.group;
  }
  const int q0 = qt * BM;
  const int kv_end = p.causal ? min(p.n, q0 + BM) : p.n;
  const int T = (kv_end + BN - 1) / BN;  // key tiles per sweep (>= 1)
  const int NI = 2 * T;

  // ---- set-up
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(o_full, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&s_free[s], 8);  // one arrival per softmax warp
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const AbortState ab{abort_flag, p.status};

  if (warp == 0) {
    // =============================================================== producer
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q1);
      tma_prefetch_desc(&p.tm_q2);
      tma_prefetch_desc(&p.tm_k1);
      if (!SHARED_K) tma_prefetch_desc(&p.tm_k2);
      tma_prefetch_desc(&p.tm_v);
      mbar_arrive_expect_tx(q_full, 2 * C::Q_TILE);
      for (int bx = 0; bx < C::QB; ++bx) {
        tma_load_4d(smem + C::OFF_Q1 + bx * BM * 128, &p.tm_q1, q_full, bx * 64, hq1, q0, b);
        tma_load_4d(smem + C::OFF_Q2 + bx * BM * 128, &p.tm_q2, q_full, bx * 64, hq2, q0, b);
      }
      int issued = 0;
      for (int it = 0; it < NI; ++it) {
        const int st = it % STAGES;
        const uint32_t use = static_cast<uint32_t>(it / STAGES);
        if (use > 0 && !mbar_wait(&kv_empty[st], (use - 1) & 1u, ab)) break;
        const bool sweep2 = it >= T;
        const int j = sweep2 ? it - T : it;
        uint8_t* stage = smem + C::OFF_STAGES + st * C::STAGE;
        mbar_arrive_expect_tx(&kv_full[st], C::NK * C::K_TILE + (sweep2 ? C::V_TILE : 0));
        for (int bx = 0; bx < C::QB; ++bx)
          tma_load_4d(stage + bx * BN * 128, &p.tm_k1, &kv_full[st], bx * 64, hk, j * BN, b);
        if (!SHARED_K)
          for (int bx = 0; bx < C::QB; ++bx)
            tma_load_4d(stage + C::K_TILE + bx * BN * 128, &p.tm_k2, &kv_full[st], bx * 64, hk, j * BN, b);
        if (sweep2)
          for (int bx = 0; bx < C::VB; ++bx)
            tma_load_4d(stage + C::NK * C::K_TILE + bx * BN * 128, &p.tm_v, &kv_full[st], bx * 64, hk, j * BN,
                        b);
        issued = it + 1;
      }
      if (*ab.flag) {
        // Aborted: let the copies already issued land before the CTA exits.
        mbar_wait_drain(q_full, 0, kWaitBudgetNs);
        for (int it = (issued > STAGES ? issued - STAGES : 0); it < issued; ++it)
          mbar_wait_drain(&kv_full[it % STAGES], static_cast<uint32_t>(it / STAGES) & 1u, kWaitBudgetNs);
      }
    }
  } else if (warp == 1) {
    // =============================================================== MMA issuer
    if (lane == 0) {
      const uint32_t sQ1 = smem_u32(smem + C::OFF_Q1);
      const uint32_t sQ2 = smem_u32(smem + C::OFF_Q2);
      const uint32_t sStages = smem_u32(smem + C::OFF_STAGES);
      bool ok = mbar_wait(q_full, 0, ab);
      tc_fence_after();

      auto issue_qk = [&](int it) -> bool {
        const int st = it % STAGES;
        if (!mbar_wait(&kv_full[st], static_cast<uint32_t>(it / STAGES) & 1u, ab)) return false;
        tc_fence_after();
        const int s = it & 1;
        const uint32_t dS1 = tmem + C::TM_S + 128u * s;
        const uint32_t dS2 = dS1 + 64u;
        const uint32_t k1 = sStages + st * C::STAGE;
        const uint32_t k2 = SHARED_K ? k1 : k1 + C::K_TILE;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t oq = (k >> 2) * (BM * 128) + (k & 3) * 32;
          const uint32_t ok_ = (k >> 2) * (BN * 128) + (k & 3) * 32;
          mma_ss(dS1, sdesc_sw128(sQ1 + oq, 16, 1024), sdesc_sw128(k1 + ok_, 16, 1024), C::IDESC_QK, k > 0);
        }
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t oq = (k >> 2) * (BM * 128) + (k & 3) * 32;
          const uint32_t ok_ = (k >> 2) * (BN * 128) + (k & 3) * 32;
          mma_ss(dS2, sdesc_sw128(sQ2 + oq, 16, 1024), sdesc_sw128(k2 + ok_, 16, 1024), C::IDESC_QK, k > 0);
        }
        tc_commit(&s_full[s]);
        return true;
      };

      if (ok) ok = issue_qk(0);
      for (int it = 0; ok && it < NI; ++it) {
        if (it + 1 < NI) {
          // S stage (it+1)&1 was last used by iteration it-1; a sweep-1
          // iteration releases it here, a sweep-2 one was awaited before its PV.
          if (it >= 1 && it - 1 < T) {
            if (!mbar_wait(&s_free[(it - 1) & 1], static_cast<uint32_t>((it - 1) >> 1) & 1u, ab)) break;
          }
          if (!issue_qk(it + 1)) break;
        }
        if (it >= T) {
          const int s = it & 1;
          if (!mbar_wait(&s_free[s], static_cast<uint32_t>(it >> 1) & 1u, ab)) break;
          tc_fence_after();
          const int st = it % STAGES;
          const int j = it - T;
          const uint32_t vb = sStages + st * C::STAGE + C::NK * C::K_TILE;
          const uint32_t aP = tmem + C::TM_S + 128u * s;
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            const uint32_t acol = (kk < 2) ? kk * 8 : 32 + (kk - 2) * 8;
            mma_ts(tmem + C::TM_O, aP + acol, sdesc_sw128(vb + kk * 2048, BN * 128, 1024), C::IDESC_PV,
                   (j > 0 || kk > 0) ? 1u : 0u);
          }
        }
        tc_commit(&kv_empty[it % STAGES]);
      }
      tc_commit(o_full);
      if (*ab.flag) mbar_wait_drain(o_full, 0, kWaitBudgetNs);
    }
  } else if (warp >= 4) {
    // =============================================================== softmax + epilogue
    const int wg = (warp - 4) >> 2;
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const int t = q0 + row;
    const uint32_t tl = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const float sc = p.scale_log2;
    const int lim = p.causal ? min(t + 1, p.n) : p.n;  // keys j < lim are visible

    // ---- sweep 1: running max / sum of map (wg + 1)
    float m = -INFINITY, l = 0.f;
    for (int it = 0; it < T; ++it) {
      const int s = it & 1;
      mbar_wait(&s_full[s], static_cast<uint32_t>(it >> 1) & 1u, ab);
      __syncwarp();
      tc_fence_after();
      uint32_t r0[32], r1[32];
      const uint32_t ta = tl + C::TM_S + 128u * s + 64u * wg;
      tmem_ld32(ta, r0);
      tmem_ld32(ta + 32, r1);
      tmem_ld_wait2(r0, r1);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[s]);
      __syncwarp();
      const int nvis = lim - it * BN;
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        if (c >= nvis) r0[c] = __float_as_uint(-INFINITY);
        if (c + 32 >= nvis) r1[c] = __float_as_uint(-INFINITY);
        mx = fmaxf(mx, fmaxf(__uint_as_float(r0[c]), __uint_as_float(r1[c])));
      }
      const float m_new = fmaxf(m, mx * sc);
      const float base = (m_new == -INFINITY) ? 0.f : m_new;
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        s0 += ex2(fmaf(__uint_as_float(r0[c]), sc, -base));
        s1 += ex2(fmaf(__uint_as_float(r1[c]), sc, -base));
      }
      l = l * ex2(m - base) + (s0 + s1);
      m = m_new;
    }

    // ---- exchange the statistics of the two maps
    stat_m[wg * 128 + row] = m;
    stat_l[wg * 128 + row] = l;
    __syncwarp();
    named_bar_sync(1, 256);
    const float m1 = stat_m[row], l1 = stat_l[row];
    const float m2 = stat_m[128 + row], l2 = stat_l[128 + row];
    float coef;
    if (EPI == kEpiRmsNorm) {
      coef = *p.lambda;
    } else {
      const float lg = (t < p.n) ? p.lam_logits[b * p.sb + static_cast<long long>(t) * p.st + u] : 0.f;
      coef = 1.f / (1.f + expf(-lg));
    }
    // P = 2^(s1*sc - M1) + neg2 * 2^(s2*sc - M2),  M1 = m1 + log2 l1,
    // M2 = m2 + log2 l2 - log2 |coef|,  neg2 = -sign(coef).
    const float M1 = m1 + log2f(l1);
    const float acoef = fabsf(coef);
    const float M2 = (acoef > 0.f) ? m2 + log2f(l2) - log2f(acoef) : INFINITY;
    const float neg2 = (coef >= 0.f) ? -1.f : 1.f;

    // ---- sweep 2: signed combined weights -> TMEM (bf16) for the P.V MMA
    for (int it = T; it < NI; ++it) {
      const int s = it & 1;
      const int j = it - T;
      mbar_wait(&s_full[s], static_cast<uint32_t>(it >> 1) & 1u, ab);
      __syncwarp();
      tc_fence_after();
      uint32_t a[32], c2[32];
      const uint32_t ts = tl + C::TM_S + 128u * s;
      tmem_ld32(ts + 32u * wg, a);
      tmem_ld32(ts + 64u + 32u * wg, c2);
      tmem_ld_wait2(a, c2);
      const int nvis = lim - (j * BN + 32 * wg);
      uint32_t pk[16];
#pragma unroll
      for (int c = 0; c < 32; c += 2) {
        float p0 = fmaf(neg2, ex2(fmaf(__uint_as_float(c2[c]), sc, -M2)),
                        ex2(fmaf(__uint_as_float(a[c]), sc, -M1)));
        float p1 = fmaf(neg2, ex2(fmaf(__uint_as_float(c2[c + 1]), sc, -M2)),
                        ex2(fmaf(__uint_as_float(a[c + 1]), sc, -M1)));
        if (c >= nvis) p0 = 0.f;
        if (c + 1 >= nvis) p1 = 0.f;
        pk[c >> 1] = pack_bf16x2(p0, p1);
      }
      tmem_st16(ts + 32u * wg, pk);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[s]);
      __syncwarp();
    }

    // ---- epilogue
    mbar_wait(o_full, 0, ab);
    __syncwarp();
    tc_fence_after();
    constexpr int HALF = DV / 2;
    const uint32_t to = tl + C::TM_O + wg * HALF;
    __nv_bfloat16* orow =
        p.out + ((static_cast<size_t>(b) * p.n + t) * p.units_per_batch + u) * DV + wg * HALF;
    float rinv = 1.f;
    if (EPI == kEpiRmsNorm) {
      float ss = 0.f;
#pragma unroll
      for (int ch = 0; ch < HALF / 32; ++ch) {
        uint32_t r[32];
        tmem_ld32(to + 32 * ch, r);
        tmem_ld_wait(r);
#pragma unroll
        for (int c = 0; c < 32; ++c) ss = fmaf(__uint_as_float(r[c]), __uint_as_float(r[c]), ss);
      }
      stat_ss[wg * 128 + row] = ss;
      __syncwarp();
      named_bar_sync(1, 256);
      const float tot = stat_ss[row] + stat_ss[128 + row];
      rinv = p.norm_mult * rsqrtf(tot * (1.f / DV) + p.eps);
    }
#pragma unroll
    for (int ch = 0; ch < HALF / 32; ++ch) {
      uint32_t r[32];
      tmem_ld32(to + 32 * ch, r);
      tmem_ld_wait(r);
      if (t < p.n) {
        uint32_t w[16];
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          float y0 = __uint_as_float(r[c]) * rinv;
          float y1 = __uint_as_float(r[c + 1]) * rinv;
          if (EPI == kEpiRmsNorm && p.gamma != nullptr) {
            const int col = wg * HALF + ch * 32 + c;
            y0 *= __ldg(p.gamma + col);
            y1 *= __ldg(p.gamma + col + 1);
          }
          w[c >> 1] = pack_bf16x2(y0, y1);
        }
        uint4* dst = reinterpret_cast<uint4*>(orow + ch * 32);
#pragma unroll
        for (int v = 0; v < 4; ++v) dst[v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
      }
    }
  }

  // ---- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace da
