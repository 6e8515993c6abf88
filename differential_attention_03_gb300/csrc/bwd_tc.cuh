// Backward of the differential-attention operator on tcgen05 tensor cores
// (bf16 operands, fp32 accumulation; sm_103a): DIFF V1 with d = 64 (value
// width 128) and DIFF V2 with d = 128 (query-head pairs over a KV head).
//
// The forward ("Differential Transformer" glossary page, "How differential
// attention works"; DIFF V2 analysis page, V2 code and GQA pairing) per unit:
//   A_r = softmax(Q_r K_r^T * scale),  O = (A_1 + c_2 A_2) V,   c_2 = -lambda
//   (V1) or -sigmoid(logit of the query row) (V2).
// Its gradients given dO (the gradient of O; for V1 after the per-head norm),
// with dP = dO V^T:
//   dS_r = A_r (c_r dP - Delta_r),  Delta_r = c_r dO . (A_r V)  (c_1 = 1)
//   dV   = (A_1 + c_2 A_2)^T dO,  dK_r = scale dS_r^T Q_r,  dQ_r = scale dS_r K_r.
// A statistics pass (the one-sweep forward with its STATS epilogue) has
// written per query row lse_r (the log2-domain log-sum-exp), Delta_r, c_2
// and, for V1, dO; the maps are recomputed here tile by tile, never stored.
//
// One CTA owns (batch, KV unit, 128-key tile) and walks the query tiles that
// see its keys (and, for V2, every head pair of the KV head's group).  The
// keys sit on the TMEM lanes: S_r^T = K_r Q_r^T and dP^T = V dO^T are
// 128 keys x 128 queries, so thread = key row in the softmax warps, and the
// dV, dK accumulators (keys x channels) stay in TMEM for the whole CTA.
//   TMEM: dV [0, 128), dK_1 [128, 128 + d) and dK_2 (V1) / dK (V2) up to 256,
//         S [256, 384) (S_1^T, then S_2^T, then Pc^T as bf16 pairs and dQ_1),
//         dP [384, 512) (dP^T, then dQ_2).
//   warp 0      TMA: K_1, K_2 (or K) and V once; per query tile Q_1, Q_2, dO.
//   warp 1      MMAs S_1^T, S_2^T, dK (dS^T Q), dQ_2 = dS_2 K_2.
//   warp 2      MMAs dP^T, dV += Pc^T dO (Pc^T from TMEM), dQ_1 = dS_1 K_1.
//               (dQ_1 follows dV in the same warp, so it overwrites Pc^T only
//               after dV has read it: MMAs of one thread run in order.)
//   warps 4-11  two warpgroups, thread = key row; warpgroup h takes query
//               columns [64 h, +64): phase 1 P_1, dS_1 (kept: P_1 as bf16
//               pairs in registers, dS_1^T to shared memory); phase 2 P_2,
//               dS_2, Pc = P_1 + c_2 P_2 (Pc^T to TMEM over S_2^T); then the
//               tile's dQ (thread = query row): scaled and added to the fp32
//               dQ in global memory with vector atomics.
// dS^T tiles are bf16 [128 keys][128 queries] in two 64-query boxes (128-byte
// rows, 128-byte swizzle): K-major A of dK += dS^T Q, and read as the
// M-major A of dQ = dS K.  Every wait is bounded (abort flag, status word).
#pragma once

#include <cuda_bf16.h>

#include "bwd_tc_params.h"
#include "ptx.cuh"

namespace da {



template <bool V2>
struct BwdTcCfg {
  static constexpr int D = V2 ? 128 : 64;
  static constexpr int DV = 128;
  static constexpr int NK = V2 ? 1 : 2;  // key tiles held (K_1, K_2 or the shared K)
  static constexpr int NTHREADS = 384;
  static constexpr int KT = 128 * D * 2;  // a 128-row query or key tile
  static constexpr int VT = 128 * DV * 2;
  static constexpr int ST = 128 * 128 * 2;  // a dS^T tile
  static constexpr int OFF_K1 = 0;
  static constexpr int OFF_K2 = OFF_K1 + KT;
  static constexpr int OFF_V = OFF_K1 + NK * KT;
  static constexpr int OFF_Q1 = OFF_V + VT;
  static constexpr int OFF_Q2 = OFF_Q1 + KT;
  static constexpr int OFF_DO = OFF_Q2 + KT;
  static constexpr int OFF_DS1 = OFF_DO + VT;
  static constexpr int OFF_DS2 = OFF_DS1 + ST;
  static constexpr int OFF_ST = OFF_DS2 + ST;  // float [5][128]: lse_1, lse_2, Delta_1, Delta_2, c_2 of the tile's queries
  static constexpr int OFF_BARS = OFF_ST + 5 * 128 * 4;
  static constexpr int NBARS = 13;
  static constexpr int OFF_MISC = OFF_BARS + NBARS * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16;  // the base is 1024-byte aligned (checked)
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t TM_DV = 0, TM_DK1 = 128, TM_DK2 = 128 + D, TM_S = 256, TM_DP = 384;
  static constexpr uint32_t TM_PC = TM_S;                    // Pc^T: 128 queries as 64 columns of bf16 pairs
  static constexpr uint32_t TM_DQ1 = V2 ? TM_S : TM_S + 64;  // V1: beside Pc^T; V2: over it, after dV
  static constexpr uint32_t TM_DQ2 = TM_DP;
  static constexpr uint32_t IDESC_S = idesc_bf16(128, 128, false, false);  // S^T = K Q^T, dP^T = V dO^T
  static constexpr uint32_t IDESC_DV = idesc_bf16(128, DV, false, true);   // dV += Pc^T dO
  static constexpr uint32_t IDESC_DK = idesc_bf16(128, D, false, true);    // dK += dS^T Q
  static constexpr uint32_t IDESC_DQ = idesc_bf16(128, D, true, true);     // dQ = dS K
  static_assert(SMEM_BYTES <= 232448, "shared memory");
  static_assert(V2 || TM_DK2 + D <= TM_S, "TMEM layout");
};

__device__ __forceinline__ void bf16x2_unpack(uint32_t w, float& lo, float& hi) {
  lo = __uint_as_float(w << 16);
  hi = __uint_as_float(w & 0xffff0000u);
}

template <bool V2>
__global__ void __launch_bounds__(384, 1) bwd_tc_kernel(const __grid_constant__ BwdTcParams p) {
  using C = BwdTcCfg<V2>;
  constexpr int D = C::D, DV = C::DV;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BARS);
  uint64_t* kv_full = bars + 0;   // K and V of the CTA landed
  uint64_t* q_full = bars + 1;    // Q_1, Q_2, dO of the query tile landed
  uint64_t* q_empty = bars + 2;   // both MMA warps' last reads of the tile's Q_1, Q_2, dO done (2)
  uint64_t* s_full = bars + 3;    // S_1^T, then S_2^T, in the S columns (twice per tile)
  uint64_t* dp_full = bars + 4;   // dP^T in the dP columns
  uint64_t* s1_free = bars + 5;   // the softmax warps have loaded S_1^T (8)
  uint64_t* p1_ready = bars + 6;  // dS_1^T in shared memory (8)
  uint64_t* p2_ready = bars + 7;  // dS_2^T in shared memory, Pc^T in TMEM, dP^T loaded (8)
  uint64_t* dq_full = bars + 8;   // dQ_1, dQ_2 of the tile complete (2)
  uint64_t* dq_free = bars + 9;   // the softmax warps have read dQ_1, dQ_2 (8)
  uint64_t* acc_done = bars + 10; // every MMA of the CTA complete (2)
  uint64_t* mma_done = bars + 11; // [2] abort drain of each MMA warp
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  float* sst = reinterpret_cast<float*>(smem + C::OFF_ST);

  // The 128-byte swizzled tiles need a 1024-byte aligned base.
  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicCAS(p.status, 0, kStatusSmemAlign);
    return;
  }

  // ---- work of this CTA: key tile jt of KV unit hk of batch b; heaviest (jt = 0) first
  const int units_kv = p.B * p.heads_kv;
  const int jt = static_cast<int>(blockIdx.x) / units_kv;
  const int ukv = static_cast<int>(blockIdx.x) % units_kv;
  const int b = ukv / p.heads_kv, hk = ukv % p.heads_kv;
  const int j0 = jt * 128;
  const int i_first = p.causal ? jt : 0;
  const int nq = p.num_tiles - i_first;      // query tiles per pair
  const int npairs = V2 ? p.group / 2 : 1;   // head pairs reading this KV head
  const int nsteps = nq * npairs;
  // step s: pair s / nq, query tile i_first + s % nq
  auto step_pair = [&](int s) { return V2 ? hk * (p.group / 2) + s / nq : hk; };  // unit index (rows of the statistics)
  auto step_tile = [&](int s) { return i_first + s % nq; };

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    mbar_init(q_full, 1);
    mbar_init(q_empty, 2);
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    mbar_init(s1_free, 8);
    mbar_init(p1_ready, 8);
    mbar_init(p2_ready, 8);
    mbar_init(dq_full, 2);
    mbar_init(dq_free, 8);
    mbar_init(acc_done, 2);
    mbar_init(&mma_done[0], 1);
    mbar_init(&mma_done[1], 1);
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
    // ================================================================ producer
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q1);
      tma_prefetch_desc(&p.tm_k1);
      tma_prefetch_desc(&p.tm_v);
      tma_prefetch_desc(&p.tm_do);
      mbar_arrive_expect_tx(kv_full, C::NK * C::KT + C::VT);
      for (int bx = 0; bx < D / 64; ++bx) {
        tma_load_4d(smem + C::OFF_K1 + bx * 16384, &p.tm_k1, kv_full, bx * 64, hk, j0, b);
        if (!V2) tma_load_4d(smem + C::OFF_K2 + bx * 16384, &p.tm_k2, kv_full, bx * 64, hk, j0, b);
      }
      for (int bx = 0; bx < DV / 64; ++bx) tma_load_4d(smem + C::OFF_V + bx * 16384, &p.tm_v, kv_full, bx * 64, hk, j0, b);
      int loaded = 0;
      for (int s = 0; s < nsteps; ++s) {
        if (s > 0 && !mbar_wait(q_empty, static_cast<uint32_t>(s - 1) & 1u, ab)) break;
        const int u = step_pair(s), q0 = step_tile(s) * 128;
        const int hq1 = V2 ? 2 * u : u, hq2 = V2 ? 2 * u + 1 : u;
        mbar_arrive_expect_tx(q_full, 2 * C::KT + C::VT);
        for (int bx = 0; bx < D / 64; ++bx) {
          tma_load_4d(smem + C::OFF_Q1 + bx * 16384, &p.tm_q1, q_full, bx * 64, hq1, q0, b);
          tma_load_4d(smem + C::OFF_Q2 + bx * 16384, V2 ? &p.tm_q1 : &p.tm_q2, q_full, bx * 64, hq2, q0, b);
        }
        for (int bx = 0; bx < DV / 64; ++bx) tma_load_4d(smem + C::OFF_DO + bx * 16384, &p.tm_do, q_full, bx * 64, u, q0, b);
        ++loaded;
      }
      if (*ab.flag) {
        // Aborted: the copies already issued land before the CTA exits.
        mbar_wait_drain(kv_full, 0, kWaitBudgetCycles);
        if (loaded > 0) mbar_wait_drain(q_full, static_cast<uint32_t>(loaded - 1) & 1u, kWaitBudgetCycles);
      }
    }
  } else if (warp == 1 || warp == 2) {
    // ================================================================ MMA issuers
    const int mw = warp - 1;
    auto waitp = [&](uint64_t* bar, uint32_t parity) -> bool {
      const bool r = __all_sync(0xffffffffu, mbar_wait(bar, parity, ab));
      tc_fence_after();
      return r;
    };
    auto kdesc = [&](int off) { return sdesc_sw128(smem_u32(smem + off), 16, 1024); };     // K-major tile
    auto mdesc = [&](int off) { return sdesc_sw128(smem_u32(smem + off), 16384, 1024); };  // M/N-major tile
    // K-major k-step k (16 elements of K): 64-element box k / 4, 32 bytes (k % 4) into its rows
    auto kstep = [](int k) { return static_cast<uint64_t>(((k >> 2) * 16384 + (k & 3) * 32) >> 4); };
    // M/N-major k-step k: 16 rows of 128 bytes further
    auto mstep = [](int k) { return static_cast<uint64_t>((k * 2048) >> 4); };
    const uint64_t dK1 = kdesc(C::OFF_K1), dK2 = kdesc(V2 ? C::OFF_K1 : C::OFF_K2), dV = kdesc(C::OFF_V);
    const uint64_t dQ1 = kdesc(C::OFF_Q1), dQ2 = kdesc(C::OFF_Q2), dDO = kdesc(C::OFF_DO);
    const uint64_t mQ1 = mdesc(C::OFF_Q1), mQ2 = mdesc(C::OFF_Q2), mDO = mdesc(C::OFF_DO);
    const uint64_t mK1 = mdesc(C::OFF_K1), mK2 = mdesc(V2 ? C::OFF_K1 : C::OFF_K2);
    const uint64_t kS1 = kdesc(C::OFF_DS1), kS2 = kdesc(C::OFF_DS2), mS1 = mdesc(C::OFF_DS1), mS2 = mdesc(C::OFF_DS2);
    bool ok = waitp(kv_full, 0);
    for (int s = 0; ok && s < nsteps; ++s) {
      const uint32_t ph = static_cast<uint32_t>(s) & 1u;
      if (!waitp(q_full, ph) || (s > 0 && !waitp(dq_free, ph ^ 1u))) {
        ok = false;
        break;
      }
      if (mw == 0) {
        // S_1^T = K_1 Q_1^T, then (once the softmax has loaded it) S_2^T = K_2 Q_2^T
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          mma_ss_elect(tmem + C::TM_S, dK1 + kstep(k), dQ1 + kstep(k), C::IDESC_S, k > 0 ? 1u : 0u);
        tc_commit_elect(s_full);
        if (!waitp(s1_free, ph)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          mma_ss_elect(tmem + C::TM_S, dK2 + kstep(k), dQ2 + kstep(k), C::IDESC_S, k > 0 ? 1u : 0u);
        tc_commit_elect(s_full);
        const uint32_t acc0 = s > 0 ? 1u : 0u;
        if (!V2) {
          // dK_1 += dS_1^T Q_1 while the softmax works on map 2
          if (!waitp(p1_ready, ph)) {
            ok = false;
            break;
          }
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma_ss_elect(tmem + C::TM_DK1, kS1 + kstep(k), mQ1 + mstep(k), C::IDESC_DK, (acc0 | k) ? 1u : 0u);
        }
        if (!waitp(p2_ready, ph)) {
          ok = false;
          break;
        }
        if (V2) {
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma_ss_elect(tmem + C::TM_DK1, kS1 + kstep(k), mQ1 + mstep(k), C::IDESC_DK, (acc0 | k) ? 1u : 0u);
#pragma unroll
          for (int k = 0; k < 8; ++k) mma_ss_elect(tmem + C::TM_DK1, kS2 + kstep(k), mQ2 + mstep(k), C::IDESC_DK, 1u);
        } else {
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma_ss_elect(tmem + C::TM_DK2, kS2 + kstep(k), mQ2 + mstep(k), C::IDESC_DK, (acc0 | k) ? 1u : 0u);
        }
        tc_commit_elect(q_empty);
        // dQ_2 = dS_2 K_2 over the dP columns (the softmax has loaded dP^T)
#pragma unroll
        for (int k = 0; k < 8; ++k) mma_ss_elect(tmem + C::TM_DQ2, mS2 + mstep(k), mK2 + mstep(k), C::IDESC_DQ, k > 0 ? 1u : 0u);
        tc_commit_elect(dq_full);
      } else {
        // dP^T = V dO^T
#pragma unroll
        for (int k = 0; k < DV / 16; ++k)
          mma_ss_elect(tmem + C::TM_DP, dV + kstep(k), dDO + kstep(k), C::IDESC_S, k > 0 ? 1u : 0u);
        tc_commit_elect(dp_full);
        if (!waitp(p2_ready, ph)) {
          ok = false;
          break;
        }
        // dV += Pc^T dO, Pc^T from TMEM (k-step k: queries 16 k .. 16 k + 15 = pair columns 8 k .. 8 k + 7)
        const uint32_t acc0 = s > 0 ? 1u : 0u;
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_ts_elect(tmem + C::TM_DV, tmem + C::TM_PC + 8u * k, mDO + mstep(k), C::IDESC_DV, (acc0 | k) ? 1u : 0u);
        tc_commit_elect(q_empty);
        // dQ_1 = dS_1 K_1 (after dV in this warp's order: it may overwrite Pc^T)
#pragma unroll
        for (int k = 0; k < 8; ++k) mma_ss_elect(tmem + C::TM_DQ1, mS1 + mstep(k), mK1 + mstep(k), C::IDESC_DQ, k > 0 ? 1u : 0u);
        tc_commit_elect(dq_full);
      }
    }
    if (ok) tc_commit_elect(acc_done);
    tc_commit_elect(&mma_done[mw]);
    if (*ab.flag) mbar_wait_drain(&mma_done[mw], 0, kWaitBudgetCycles);
    __syncwarp();
  } else if (warp >= 4) {
    // ================================================================ softmax, dQ, epilogue
    const int h = (warp - 4) >> 2;  // query columns [64 h, +64)
    const int wq = warp & 3;        // TMEM lane quarter
    const int kr = wq * 32 + lane;  // key row (softmax) / query row (dQ)
    const uint32_t tl = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const int key = j0 + kr;
    const bool key_ok = key < p.n;
    const float sc = p.scale_log2;
    const float lam_c2 = V2 ? 0.f : -*p.lambda;
    const int t256 = threadIdx.x - 128;
    uint8_t* const ds1_row = smem + C::OFF_DS1 + h * 16384 + kr * 128;
    uint8_t* const ds2_row = smem + C::OFF_DS2 + h * 16384 + kr * 128;
    // These warps meet at named barriers, so none leaves the loop early: after
    // an abort every wait returns at once and the remaining steps run through
    // (their results are not used).
    for (int s = 0; s < nsteps; ++s) {
      const uint32_t ph = static_cast<uint32_t>(s) & 1u;
      const int u = step_pair(s), q0 = step_tile(s) * 128;
      // ---- the statistics of the tile's 128 queries -> shared memory
      named_bar_sync(1, 256);  // everyone is done with the previous tile's
      const long long r0 = (static_cast<long long>(b) * p.units + u) * p.n + q0;
      for (int idx = t256; idx < 5 * 128; idx += 256) {
        const int a = idx >> 7, qq = idx & 127;
        const bool in = q0 + qq < p.n;
        float v;
        if (a < 4)
          v = in ? p.row[a * p.rows + r0 + qq] : (a < 2 ? INFINITY : 0.f);
        else
          v = V2 ? (in ? -p.row[5 * p.rows + r0 + qq] : 0.f) : lam_c2;
        sst[idx] = v;
      }
      named_bar_sync(1, 256);
      const float* lse1 = sst + 64 * h;
      const float* lse2 = lse1 + 128;
      const float* del1 = lse1 + 256;
      const float* del2 = lse1 + 384;
      const float* cf2 = lse1 + 512;
      const int qbase = q0 + 64 * h;  // first query of this thread's columns
      auto visible = [&](int cidx) {
        const int tq = qbase + cidx;
        return key_ok && tq < p.n && (!p.causal || key <= tq);
      };
      // ---- phase 1: P_1, dS_1 = P_1 (dP - Delta_1)
      mbar_wait(s_full, 0, ab);
      mbar_wait(dp_full, ph, ab);
      __syncwarp();
      tc_fence_after();
      uint32_t sv[2][32];
      tmem_ld32(tl + C::TM_S + 64u * h, sv[0]);
      tmem_ld32(tl + C::TM_S + 64u * h + 32u, sv[1]);
      tmem_ld_wait2(sv[0], sv[1]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s1_free);  // S_2^T may overwrite the S columns
      __syncwarp();
      uint32_t p1k[32];  // P_1 of the 64 columns as bf16 pairs
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        uint32_t dp[32];
        tmem_ld32(tl + C::TM_DP + 64u * h + 32u * q, dp);
        tmem_ld_wait(dp);
        uint32_t dsk[16];
#pragma unroll
        for (int cc = 0; cc < 32; cc += 2) {
          const int c0 = 32 * q + cc;
          const float pa = visible(c0) ? ex2(fmaf(__uint_as_float(sv[q][cc]), sc, -lse1[c0])) : 0.f;
          const float pb = visible(c0 + 1) ? ex2(fmaf(__uint_as_float(sv[q][cc + 1]), sc, -lse1[c0 + 1])) : 0.f;
          const float da = pa * (__uint_as_float(dp[cc]) - del1[c0]);
          const float db = pb * (__uint_as_float(dp[cc + 1]) - del1[c0 + 1]);
          p1k[16 * q + (cc >> 1)] = pack_bf16x2(pa, pb);
          dsk[cc >> 1] = pack_bf16x2(da, db);
        }
        // 16-byte chunk 4 q + v of the row (queries 8 (4 q + v) ..), swizzled by the row
#pragma unroll
        for (int v = 0; v < 4; ++v)
          *reinterpret_cast<uint4*>(ds1_row + (((4 * q + v) ^ (kr & 7)) << 4)) =
              make_uint4(dsk[4 * v], dsk[4 * v + 1], dsk[4 * v + 2], dsk[4 * v + 3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(p1_ready);
      __syncwarp();
      // ---- phase 2: P_2, dS_2 = P_2 (c_2 dP - Delta_2), Pc = P_1 + c_2 P_2
      mbar_wait(s_full, 1, ab);
      __syncwarp();
      tc_fence_after();
      tmem_ld32(tl + C::TM_S + 64u * h, sv[0]);
      tmem_ld32(tl + C::TM_S + 64u * h + 32u, sv[1]);
      tmem_ld_wait2(sv[0], sv[1]);
      // Pc^T overwrites S columns [0, 64): both warpgroups must have loaded S_2^T first.
      tc_fence_before();
      named_bar_sync(2, 256);
      tc_fence_after();
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        uint32_t dp[32];
        tmem_ld32(tl + C::TM_DP + 64u * h + 32u * q, dp);
        tmem_ld_wait(dp);
        uint32_t dsk[16], pck[16];
#pragma unroll
        for (int cc = 0; cc < 32; cc += 2) {
          const int c0 = 32 * q + cc;
          const float pa = visible(c0) ? ex2(fmaf(__uint_as_float(sv[q][cc]), sc, -lse2[c0])) : 0.f;
          const float pb = visible(c0 + 1) ? ex2(fmaf(__uint_as_float(sv[q][cc + 1]), sc, -lse2[c0 + 1])) : 0.f;
          const float ca = cf2[c0], cb2 = cf2[c0 + 1];
          const float da = pa * fmaf(ca, __uint_as_float(dp[cc]), -del2[c0]);
          const float db = pb * fmaf(cb2, __uint_as_float(dp[cc + 1]), -del2[c0 + 1]);
          float p1a, p1b;
          bf16x2_unpack(p1k[16 * q + (cc >> 1)], p1a, p1b);
          dsk[cc >> 1] = pack_bf16x2(da, db);
          pck[cc >> 1] = pack_bf16x2(fmaf(ca, pa, p1a), fmaf(cb2, pb, p1b));
        }
#pragma unroll
        for (int v = 0; v < 4; ++v)
          *reinterpret_cast<uint4*>(ds2_row + (((4 * q + v) ^ (kr & 7)) << 4)) =
              make_uint4(dsk[4 * v], dsk[4 * v + 1], dsk[4 * v + 2], dsk[4 * v + 3]);
        tmem_st16(tl + C::TM_PC + 32u * h + 16u * q, pck);
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p2_ready);
      __syncwarp();
      // ---- dQ of the tile: thread = query row kr; warpgroup h reads dQ_(h+1)
      const bool dq_ok = __all_sync(0xffffffffu, mbar_wait(dq_full, ph, ab));
      tc_fence_after();
      {
        const int tq = q0 + kr;
        const int head = V2 ? 2 * u + h : u;
        float* dst = (h == 0 ? p.dq1 : p.dq2) +
                     ((static_cast<long long>(b) * p.n + tq) * (V2 ? 2 * p.units : p.units) + head) * D;
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t r[32];
          tmem_ld32(tl + (h == 0 ? C::TM_DQ1 : C::TM_DQ2) + 32u * ch, r);
          tmem_ld_wait(r);
          if (dq_ok && tq < p.n) {
#pragma unroll
            for (int v = 0; v < 8; ++v)
              atomicAdd(reinterpret_cast<float4*>(dst + 32 * ch + 4 * v),
                        make_float4(__uint_as_float(r[4 * v]) * p.scale, __uint_as_float(r[4 * v + 1]) * p.scale,
                                    __uint_as_float(r[4 * v + 2]) * p.scale, __uint_as_float(r[4 * v + 3]) * p.scale));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dq_free);
      __syncwarp();
    }
    // ---- epilogue: dV and dK of the CTA's keys (thread = key row); warpgroup h
    // writes dV columns [64 h, +64) and dK_(h+1) (V1) / dK columns [64 h, +64) (V2).
    if (__all_sync(0xffffffffu, mbar_wait(acc_done, 0, ab))) {
      tc_fence_after();
      const long long krow = static_cast<long long>(b) * p.n + key;
      float* dvp = p.dv + (krow * p.heads_kv + hk) * DV + 64 * h;
      float* dkp = V2 ? p.dk1 + (krow * p.heads_kv + hk) * D + 64 * h : (h == 0 ? p.dk1 : p.dk2) + (krow * p.heads_kv + hk) * D;
      const uint32_t tk = V2 ? C::TM_DK1 + 64u * h : (h == 0 ? C::TM_DK1 : C::TM_DK2);
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        uint32_t r[32], g[32];
        tmem_ld32(tl + C::TM_DV + 64u * h + 32u * ch, r);
        tmem_ld32(tl + tk + 32u * ch, g);
        tmem_ld_wait2(r, g);
        if (key_ok) {
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            reinterpret_cast<float4*>(dvp + 32 * ch)[v] =
                make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]), __uint_as_float(r[4 * v + 2]),
                            __uint_as_float(r[4 * v + 3]));
            reinterpret_cast<float4*>(dkp + 32 * ch)[v] =
                make_float4(__uint_as_float(g[4 * v]) * p.scale, __uint_as_float(g[4 * v + 1]) * p.scale,
                            __uint_as_float(g[4 * v + 2]) * p.scale, __uint_as_float(g[4 * v + 3]) * p.scale);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace da
