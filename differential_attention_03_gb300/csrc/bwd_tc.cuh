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
//   warps 3-18  four warpgroups, thread = key row; warpgroup h takes query
//               columns [32 h, +32): phase 1 P_1, dS_1 (dS_1^T to shared
//               memory, P_1 kept as bf16 pairs in registers); phase 2 P_2,
//               dS_2, Pc = P_1 + c_2 P_2 (Pc^T to TMEM over S_2^T); then the
//               tile's dQ (thread = query row): scaled, staged in the dS^T
//               buffers and added to the fp32 dQ in global memory by TMA bulk
//               reduce-adds; the next step's row statistics are fetched
//               meanwhile.  (V1 issues the dQ MMAs before dV and dK, so dQ is
//               read out while they run.)
// dS^T tiles are bf16 [128 keys][128 queries] in two 64-query boxes (128-byte
// rows, 128-byte swizzle): K-major A of dK += dS^T Q, and read as the
// M-major A of dQ = dS K.  Every wait is bounded (abort flag, status word).
#pragma once

#include <cuda_bf16.h>

#include <type_traits>

#include "bwd_tc_params.h"
#include "ptx.cuh"

#undef DA_BOUNDS_FILE
#define DA_BOUNDS_FILE 7

namespace da {



template <bool V2>
struct BwdTcCfg {
  static constexpr int D = V2 ? 128 : 64;
  static constexpr int DV = 128;
  static constexpr int NK = V2 ? 1 : 2;  // key tiles held (K_1, K_2 or the shared K)
  static constexpr int NTHREADS = 608;  // warp 0 TMA, warps 1-2 MMA, warps 3-18 softmax
  static constexpr int KT = 128 * D * 2;  // a 128-row query or key tile
  static constexpr int VT = 128 * DV * 2;
  static constexpr int ST = 128 * 128 * 2;  // a dS^T tile
  static constexpr int OFF_K1 = 0;
  static constexpr int OFF_K2 = OFF_K1 + KT;
  static constexpr int OFF_V = OFF_K1 + NK * KT;
  static constexpr int OFF_Q1 = OFF_V + VT;
  static constexpr int OFF_Q2 = OFF_Q1 + KT;
  static constexpr int OFF_DO = OFF_Q2 + KT;
  // dO of the next query tile loads while the current one is in use (V1; V2 has no room for it).
  static constexpr int NDO = V2 ? 1 : 2;
  static constexpr int OFF_DS1 = OFF_DO + NDO * VT;
  static constexpr int OFF_DS2 = OFF_DS1 + ST;
  static constexpr int OFF_ST = OFF_DS2 + ST;  // float [5][128]: lse_1, lse_2, Delta_1, Delta_2, c_2 of the tile's queries
  static constexpr int OFF_BARS = OFF_ST + 5 * 128 * 4;
  static constexpr int NBARS = 20;
  static constexpr int OFF_MISC = OFF_BARS + NBARS * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16;  // the base is 1024-byte aligned (checked)
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t TM_DV = 0, TM_DK1 = 128, TM_DK2 = 128 + D, TM_S = 256, TM_DP = 384;
  // Pc^T as bf16 pairs over S_2^T, each warpgroup over its own S columns: queries [32 h, +32) at
  // pair columns TM_S + 32 h + [0, 16), so k-step k (16 queries) of dV reads TM_S + 32 (k / 2) + 8 (k % 2).
  static constexpr uint32_t TM_PC = TM_S;
  static constexpr uint32_t TM_DQ1 = V2 ? TM_S : TM_DP + 64;  // V2: over Pc^T, after dV; V1: beside dQ_2
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
__global__ void __launch_bounds__(608, 1) bwd_tc_kernel(const __grid_constant__ BwdTcParams p) {
  using C = BwdTcCfg<V2>;
  constexpr int D = C::D, DV = C::DV;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BARS);
  uint64_t* kv_full = bars + 0;    // K and V of the CTA landed
  uint64_t* q1_full = bars + 1;    // Q_1 of the step landed
  uint64_t* q2_full = bars + 2;    // Q_2 of the step landed
  uint64_t* do_full = bars + 3;    // [2] dO of the step landed in buffer s % NDO
  uint64_t* q1_empty = bars + 5;   // the MMAs reading Q_1 (S_1^T, dK of map 1) done
  uint64_t* q2_empty = bars + 6;   // the MMAs reading Q_2 (S_2^T, dK of map 2) done
  uint64_t* do_empty = bars + 7;   // [2] the MMAs reading dO buffer b (dP^T, dV) done
  uint64_t* s_full = bars + 9;     // S_1^T, then S_2^T, in the S columns (twice per step)
  uint64_t* dp_full = bars + 10;   // dP^T in the dP columns
  uint64_t* s1_free = bars + 11;   // the softmax warps have loaded S_1^T (16)
  uint64_t* p1_ready = bars + 12;  // dS_1^T in shared memory (16)
  uint64_t* p2_ready = bars + 13;  // dS_2^T in shared memory, Pc^T in TMEM, dP^T loaded (16)
  uint64_t* dq_full = bars + 14;   // dQ_1, dQ_2 of the step complete (2)
  uint64_t* dq_free = bars + 15;   // the softmax warps have read dQ_1, dQ_2 (16)
  uint64_t* acc_done = bars + 16;  // every MMA of the CTA complete (2)
  uint64_t* mma_done = bars + 17;  // [2] abort drain of each MMA warp
  uint64_t* ds_done = bars + 19;   // every MMA of the step reading dS^T, Pc^T complete (2)
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
    mbar_init(q1_full, 1);
    mbar_init(q2_full, 1);
    mbar_init(q1_empty, 1);
    mbar_init(q2_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&do_full[i], 1);
      mbar_init(&do_empty[i], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    mbar_init(s1_free, 16);
    mbar_init(p1_ready, 16);
    mbar_init(p2_ready, 16);
    mbar_init(dq_full, 2);
    mbar_init(dq_free, 16);
    mbar_init(acc_done, 2);
    mbar_init(&mma_done[0], 1);
    mbar_init(&mma_done[1], 1);
    mbar_init(ds_done, 2);
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
      if (DA_BOUNDS_V(j0 < p.n && b < p.B && hk < p.heads_kv, j0)) {
        for (int bx = 0; bx < D / 64; ++bx) {
          tma_load_4d(smem + C::OFF_K1 + bx * 16384, &p.tm_k1, kv_full, bx * 64, hk, j0, b);
          if (!V2) tma_load_4d(smem + C::OFF_K2 + bx * 16384, &p.tm_k2, kv_full, bx * 64, hk, j0, b);
        }
        for (int bx = 0; bx < DV / 64; ++bx)
          tma_load_4d(smem + C::OFF_V + bx * 16384, &p.tm_v, kv_full, bx * 64, hk, j0, b);
      }
      // Per step: Q_1 (released mid-step by map 1's dK), Q_2 (released by map 2's dK) and dO (released
      // by dV; with two buffers the next step's loads during this one).
      int nq1 = 0, nq2 = 0, ndo[2] = {0, 0};
      bool ok = true;
      auto load_q = [&](int st_, int r) {  // r = 0: Q_1, 1: Q_2
        int& cnt = r == 0 ? nq1 : nq2;
        if (cnt > 0 && !mbar_wait(r == 0 ? q1_empty : q2_empty, static_cast<uint32_t>(cnt - 1) & 1u, ab)) {
          ok = false;
          return;
        }
        const int u = step_pair(st_), q0 = step_tile(st_) * 128;
        const int hq = V2 ? 2 * u + r : u;
        uint64_t* bar = r == 0 ? q1_full : q2_full;
        mbar_arrive_expect_tx(bar, C::KT);
        if (!DA_BOUNDS_V(q0 < p.n && b < p.B && hq < (V2 ? 2 : 1) * p.units, q0)) {
          ok = false;
          return;
        }
        for (int bx = 0; bx < D / 64; ++bx)
          tma_load_4d(smem + (r == 0 ? C::OFF_Q1 : C::OFF_Q2) + bx * 16384, (V2 || r == 0) ? &p.tm_q1 : &p.tm_q2,
                      bar, bx * 64, hq, q0, b);
        ++cnt;
      };
      auto load_do = [&](int st_) {
        const int db = st_ % C::NDO;
        if (ndo[db] > 0 && !mbar_wait(&do_empty[db], static_cast<uint32_t>(ndo[db] - 1) & 1u, ab)) {
          ok = false;
          return;
        }
        const int u = step_pair(st_), q0 = step_tile(st_) * 128;
        mbar_arrive_expect_tx(&do_full[db], C::VT);
        if (!DA_BOUNDS_V(q0 < p.n && b < p.B && u < p.units, q0)) {
          ok = false;
          return;
        }
        for (int bx = 0; bx < DV / 64; ++bx)
          tma_load_4d(smem + C::OFF_DO + db * C::VT + bx * 16384, &p.tm_do, &do_full[db], bx * 64, u, q0, b);
        ++ndo[db];
      };
      for (int s = 0; ok && s < nsteps; ++s) {
        // In the order the tiles are released: V1 dO (double-buffered) first, V2 Q_1 first.
        if (V2) {
          load_q(s, 0);
          if (ok) load_do(s);
        } else {
          load_do(s);
          if (ok) load_q(s, 0);
        }
        if (ok) load_q(s, 1);
      }
      if (*ab.flag) {
        // Aborted: the copies already issued land before the CTA exits.
        mbar_wait_drain(kv_full, 0, kWaitBudgetCycles);
        if (nq1 > 0) mbar_wait_drain(q1_full, static_cast<uint32_t>(nq1 - 1) & 1u, kWaitBudgetCycles);
        if (nq2 > 0) mbar_wait_drain(q2_full, static_cast<uint32_t>(nq2 - 1) & 1u, kWaitBudgetCycles);
        for (int i = 0; i < 2; ++i)
          if (ndo[i] > 0) mbar_wait_drain(&do_full[i], static_cast<uint32_t>(ndo[i] - 1) & 1u, kWaitBudgetCycles);
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
      if (mw == 0) {
        // S_1^T = K_1 Q_1^T; once the softmax has loaded it, S_2^T = K_2 Q_2^T (same columns)
        if (!waitp(q1_full, ph) || (s > 0 && (!waitp(dq_free, ph ^ 1u) || !waitp(ds_done, ph ^ 1u)))) {
          ok = false;
          break;
        }
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          mma_ss_elect(tmem + C::TM_S, dK1 + kstep(k), dQ1 + kstep(k), C::IDESC_S, k > 0 ? 1u : 0u);
        tc_commit_elect(s_full);
        if (!waitp(s1_free, ph) || !waitp(q2_full, ph)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          mma_ss_elect(tmem + C::TM_S, dK2 + kstep(k), dQ2 + kstep(k), C::IDESC_S, k > 0 ? 1u : 0u);
        tc_commit_elect(s_full);
        // dK += dS_1^T Q_1 while the softmax works on map 2; Q_1 is then free for the next step.
        if (!waitp(p1_ready, ph)) {
          ok = false;
          break;
        }
        const uint32_t acc0 = s > 0 ? 1u : 0u;
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_ss_elect(tmem + C::TM_DK1, kS1 + kstep(k), mQ1 + mstep(k), C::IDESC_DK, (acc0 | k) ? 1u : 0u);
        tc_commit_elect(q1_empty);
        if (!waitp(p2_ready, ph)) {
          ok = false;
          break;
        }
        // dQ_2 = dS_2 K_2 over the dP columns (the softmax has loaded dP^T), first: the softmax
        // warps read it out while dK accumulates.
#pragma unroll
        for (int k = 0; k < 8; ++k) mma_ss_elect(tmem + C::TM_DQ2, mS2 + mstep(k), mK2 + mstep(k), C::IDESC_DQ, k > 0 ? 1u : 0u);
        tc_commit_elect(dq_full);
        // dK of map 2: V1 its own accumulator, V2 the shared K's
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_ss_elect(tmem + (V2 ? C::TM_DK1 : C::TM_DK2), kS2 + kstep(k), mQ2 + mstep(k), C::IDESC_DK,
                       (V2 || acc0 || k) ? 1u : 0u);
        tc_commit_elect(q2_empty);
        tc_commit_elect(ds_done);
      } else {
        // dP^T = V dO^T
        const int db = s % C::NDO;
        const uint64_t dbo = static_cast<uint64_t>((db * C::VT) >> 4);
        if (!waitp(&do_full[db], static_cast<uint32_t>(s / C::NDO) & 1u) || (s > 0 && !waitp(dq_free, ph ^ 1u))) {
          ok = false;
          break;
        }
#pragma unroll
        for (int k = 0; k < DV / 16; ++k)
          mma_ss_elect(tmem + C::TM_DP, dV + kstep(k), dDO + dbo + kstep(k), C::IDESC_S, k > 0 ? 1u : 0u);
        tc_commit_elect(dp_full);
        if (!waitp(p2_ready, ph)) {
          ok = false;
          break;
        }
        // dV += Pc^T dO, Pc^T from TMEM, and dQ_1 = dS_1 K_1: V1 dQ_1 first (its columns are in the
        // dP buffer), V2 after dV (dQ_1 overwrites Pc^T; MMAs of one thread run in order).
        const uint32_t acc0 = s > 0 ? 1u : 0u;
        auto dq1_mmas = [&]() {
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma_ss_elect(tmem + C::TM_DQ1, mS1 + mstep(k), mK1 + mstep(k), C::IDESC_DQ, k > 0 ? 1u : 0u);
          tc_commit_elect(dq_full);
        };
        if (!V2) dq1_mmas();
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_ts_elect(tmem + C::TM_DV, tmem + C::TM_PC + 32u * (k >> 1) + 8u * (k & 1), mDO + dbo + mstep(k),
                       C::IDESC_DV, (acc0 | k) ? 1u : 0u);
        tc_commit_elect(&do_empty[db]);
        if (V2) dq1_mmas();
        tc_commit_elect(ds_done);
      }
    }
    if (ok) tc_commit_elect(acc_done);
    tc_commit_elect(&mma_done[mw]);
    if (*ab.flag) mbar_wait_drain(&mma_done[mw], 0, kWaitBudgetCycles);
    __syncwarp();
  } else {
    // ================================================================ softmax, dQ, epilogue
    // Four warpgroups (warps 3-18): warpgroup h takes query columns [32 h, +32) of the step in two
    // 16-column parts; thread = key row (TMEM lane quarter warp % 4).
    const int h = (warp - 3) >> 2;
    const int wq = warp & 3;
    const int kr = wq * 32 + lane;  // key row (softmax) / query row (dQ)
    const uint32_t tl = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const int key = j0 + kr;
    const bool key_ok = key < p.n;
    const float sc = p.scale_log2;
    const float lam_c2 = V2 ? 0.f : -*p.lambda;
    const int t512 = threadIdx.x - 96;
    const bool lead = (t512 & 127) == 0;  // issues the warpgroup's bulk reduce-adds
    // The warpgroup's 32 columns in the dS^T tiles: 64-query box h / 2, 16-byte chunks 4 (h % 2) .. + 3.
    uint8_t* const ds1_row = smem + C::OFF_DS1 + (h >> 1) * 16384 + kr * 128;
    uint8_t* const ds2_row = smem + C::OFF_DS2 + (h >> 1) * 16384 + kr * 128;
    const int chunk0 = 4 * (h & 1);
    // These warps meet at named barriers, so none leaves the loop early: after an abort every wait
    // returns at once and the remaining steps run through (their results are not used).
    // The statistics of a step's 128 queries (lse_1, lse_2, Delta_1, Delta_2, c_2): each of the 512
    // threads fetches up to two of the 640 values, for the next step while the current one ends.
    auto fetch_stats = [&](int st_, float (&v)[2]) {
      const int u_ = step_pair(st_), q0_ = step_tile(st_) * 128;
      const long long r0 = (static_cast<long long>(b) * p.units + u_) * p.n + q0_;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int idx = t512 + 512 * e;
        const int a = idx >> 7, qq = idx & 127;
        const bool in = q0_ + qq < p.n;
        float x = 0.f;
        if (idx < 5 * 128) {
          if (a < 4)
            x = in ? p.row[a * p.rows + r0 + qq] : (a < 2 ? INFINITY : 0.f);
          else
            x = V2 ? (in ? -p.row[5 * p.rows + r0 + qq] : 0.f) : lam_c2;
        }
        v[e] = x;
      }
    };
    float pre[2];
    fetch_stats(0, pre);
    // dQ_2's last reduce-add of a step is issued one phase later (pend_*: its column, head and first
    // query; pend_col < 0: none), after the next step's first phase has passed its barrier, so that
    // dQ_1's reduce-add, whose staging the next phase 1 overwrites, has the L2's reduction bandwidth
    // to itself; phase 2 waits for dQ_2's read before it overwrites that staging.
    int pend_col = -1, pend_head = 0, pend_q0 = 0;
    auto issue_pending = [&]() {
      if (lead && h >= 2 && pend_col >= 0) {
        tma_reduce_add_4d(V2 ? &p.tm_dq1 : &p.tm_dq2, smem + C::OFF_DS2 + (h & 1) * 16384, pend_col, pend_head,
                          pend_q0, b);
        bulk_commit_group();
        pend_col = -1;
      }
    };
    for (int s = 0; s < nsteps; ++s) {
      const uint32_t ph = static_cast<uint32_t>(s) & 1u;
      const int u = step_pair(s), q0 = step_tile(s) * 128;
      // ---- the step's statistics -> shared memory (fetched during the previous step); the first
      // barrier: every thread is done with the previous step's.
      named_bar_sync(1, 512);
      // Layout: (lse_1, Delta_1) pairs of the 128 queries, then (lse_2, Delta_2) pairs, then c_2.
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int idx = t512 + 512 * e;
        if (idx < 5 * 128) {
          const int a = idx >> 7, qq = idx & 127;
          const int pos = a == 4 ? 512 + qq : (a & 1) * 256 + 2 * qq + (a >> 1);
          sst[pos] = pre[e];
        }
      }
      named_bar_sync(1, 512);
      const float4* st1 = reinterpret_cast<const float4*>(sst) + 16 * h;        // (lse_1, Delta_1) x 2 columns
      const float4* st2 = reinterpret_cast<const float4*>(sst + 256) + 16 * h;  // (lse_2, Delta_2) x 2 columns
      const float* cf2 = sst + 512 + 32 * h;
      const int qbase = q0 + 32 * h;  // first query of this thread's columns
      // Every key of the tile precedes every query (or no mask applies) and no row is past n: no
      // per-column mask (every step except the diagonal and ragged ones).
      const bool full = (!p.causal || q0 > j0) && q0 + 128 <= p.n && j0 + 128 <= p.n;
      auto visible = [&](int cidx) {
        const int tq = qbase + cidx;
        return key_ok && tq < p.n && (!p.causal || key <= tq);
      };
      const uint64_t sc2 = f2pack(sc, sc);
      // The two phases, compiled with and without the per-column mask (a branch in every column pair
      // of the unrolled loops would split them into short blocks).
      auto phases = [&](auto full_tag) {
        constexpr bool FULL = decltype(full_tag)::value;
        // P of columns c0, c0 + 1 (x = s sc - lse, exp2), with their Delta pair.
        auto probs = [&](uint32_t sa, uint32_t sb, const float4& st, int c0, uint64_t& del) -> uint64_t {
          float xa, xb;
          f2unpack(fma2(f2pack(__uint_as_float(sa), __uint_as_float(sb)), sc2, f2pack(-st.x, -st.z)), xa, xb);
          float pa = ex2(xa), pb = ex2(xb);
          if constexpr (!FULL) {
            if (!visible(c0)) pa = 0.f;
            if (!visible(c0 + 1)) pb = 0.f;
          }
          del = f2pack(-st.y, -st.w);
          return f2pack(pa, pb);
        };
        // ---- phase 1: P_1, dS_1 = P_1 (dP - Delta_1); dS_1^T to its buffer, P_1 kept as bf16 pairs.
        uint32_t p1k[16];
        mbar_wait(s_full, 0, ab);
        mbar_wait(dp_full, ph, ab);
        __syncwarp();
        tc_fence_after();
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          uint32_t sv[16], dp[16];
          tmem_ld16(tl + C::TM_S + 32u * h + 16u * q, sv);
          tmem_ld16(tl + C::TM_DP + 32u * h + 16u * q, dp);
          tmem_ld_wait16x2(sv, dp);
          if (q == 1) {  // every S_1^T column of the thread is loaded: S_2^T may overwrite them
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(s1_free);
            __syncwarp();
          }
          uint32_t dsk[8];
#pragma unroll
          for (int cc = 0; cc < 16; cc += 2) {
            const int c0 = 16 * q + cc;
            uint64_t del;
            const uint64_t pp = probs(sv[cc], sv[cc + 1], st1[c0 >> 1], c0, del);
            const uint64_t ds = mul2(pp, add2(f2pack(__uint_as_float(dp[cc]), __uint_as_float(dp[cc + 1])), del));
            float pa, pb, xa, xb;
            f2unpack(pp, pa, pb);
            f2unpack(ds, xa, xb);
            p1k[8 * q + (cc >> 1)] = pack_bf16x2(pa, pb);
            dsk[cc >> 1] = pack_bf16x2(xa, xb);
          }
          if (q == 0) {
            // The dS_1^T buffer staged the previous step's dQ_1: its reduce-adds must have read it.
            if (lead && h < 2) bulk_wait_read_all();
            named_bar_sync(1, 512);
            issue_pending();  // the previous step's deferred dQ_2 reduce-add
          }
          // 16-byte chunks chunk0 + 2 q + v of the row, swizzled by the row
#pragma unroll
          for (int v = 0; v < 2; ++v)
            *reinterpret_cast<uint4*>(ds1_row + (((chunk0 + 2 * q + v) ^ (kr & 7)) << 4)) =
                make_uint4(dsk[4 * v], dsk[4 * v + 1], dsk[4 * v + 2], dsk[4 * v + 3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(p1_ready);
        __syncwarp();
        // ---- phase 2: P_2, dS_2 = P_2 (c_2 dP - Delta_2), Pc = P_1 + c_2 P_2.  Pc^T of the part goes
        // over this thread's own, already loaded, S_2^T columns: no other thread reads them.
        mbar_wait(s_full, 1, ab);
        // The dS_2^T buffer staged the previous step's dQ_2: its reduce-adds must have read it (they
        // have had all of phase 1).
        if (lead && h >= 2) bulk_wait_read_all();
        named_bar_sync(2, 512);
        __syncwarp();
        tc_fence_after();
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          uint32_t sv[16], dp[16];
          tmem_ld16(tl + C::TM_S + 32u * h + 16u * q, sv);
          tmem_ld16(tl + C::TM_DP + 32u * h + 16u * q, dp);
          tmem_ld_wait16x2(sv, dp);
          uint32_t dsk[8], pck[8];
#pragma unroll
          for (int cc = 0; cc < 16; cc += 2) {
            const int c0 = 16 * q + cc;
            uint64_t del;
            const uint64_t pp = probs(sv[cc], sv[cc + 1], st2[c0 >> 1], c0, del);
            const uint64_t c2 = V2 ? f2pack(cf2[c0], cf2[c0 + 1]) : f2pack(lam_c2, lam_c2);
            const uint64_t ds = mul2(pp, fma2(c2, f2pack(__uint_as_float(dp[cc]), __uint_as_float(dp[cc + 1])), del));
            float p1a, p1b;
            bf16x2_unpack(p1k[8 * q + (cc >> 1)], p1a, p1b);
            float xa, xb, ya, yb;
            f2unpack(ds, xa, xb);
            f2unpack(fma2(c2, pp, f2pack(p1a, p1b)), ya, yb);
            dsk[cc >> 1] = pack_bf16x2(xa, xb);
            pck[cc >> 1] = pack_bf16x2(ya, yb);
          }
#pragma unroll
          for (int v = 0; v < 2; ++v)
            *reinterpret_cast<uint4*>(ds2_row + (((chunk0 + 2 * q + v) ^ (kr & 7)) << 4)) =
                make_uint4(dsk[4 * v], dsk[4 * v + 1], dsk[4 * v + 2], dsk[4 * v + 3]);
          tmem_st8(tl + C::TM_PC + 32u * h + 8u * q, pck);
        }
        tmem_st_wait();
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p2_ready);
        __syncwarp();
      };
      if (full)
        phases(std::true_type{});
      else
        phases(std::false_type{});
      if (s + 1 < nsteps) fetch_stats(s + 1, pre);  // consumed at the top of the next step
      // ---- dQ of the step: thread = query row kr.  Warpgroup h takes dQ_(h / 2 + 1), columns
      // [(d / 2) (h % 2), +d / 2), 32 a round: scaled and staged as one 128-byte swizzled fp32 box
      // (128 rows x 32 columns) in its quarter of the dS^T buffers (free once the step's MMAs reading
      // them are done), then added to the fp32 dQ in global memory by a TMA bulk reduce-add (rows
      // past n are dropped).
      const bool dq_ok = __all_sync(0xffffffffu, mbar_wait(dq_full, ph, ab));
      tc_fence_after();
      {
        const int map = h >> 1;
        const uint32_t tdq = tl + (map == 0 ? C::TM_DQ1 : C::TM_DQ2);
        uint8_t* const stg = smem + (map == 0 ? C::OFF_DS1 : C::OFF_DS2) + (h & 1) * 16384;
        const CUtensorMap* dqmap = (V2 || map == 0) ? &p.tm_dq1 : &p.tm_dq2;
        const int head = V2 ? 2 * u + map : u;
        constexpr int ROUNDS = D / 64;
#pragma unroll
        for (int rd = 0; rd < ROUNDS; ++rd) {
          const int col0 = (D / 2) * (h & 1) + 32 * rd;
          uint32_t r[32];
          tmem_ld32(tdq + static_cast<uint32_t>(col0), r);
          tmem_ld_wait(r);
          if (rd == ROUNDS - 1) {  // dQ is in registers: the next step's MMAs may overwrite its columns
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dq_free);
            __syncwarp();
          }
          if (rd == 0) {
            // The MMAs reading this map's dS^T buffer are done: for dS_1 (dK_1 and dQ_1) dq_full
            // already implies it (each MMA warp's commit covers its earlier MMAs); dS_2 is also read
            // by dK_2, issued after dQ_2.
            if (map == 1) mbar_wait(ds_done, ph, ab);
            __syncwarp();
          } else {
            if (lead) bulk_wait_read_all();  // the previous round's reduce-add has read the staging
            named_bar_sync(3 + h, 128);
          }
          uint8_t* const srow = stg + kr * 128;
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *reinterpret_cast<float4*>(srow + ((j ^ (kr & 7)) << 4)) =
                make_float4(__uint_as_float(r[4 * j]) * p.scale, __uint_as_float(r[4 * j + 1]) * p.scale,
                            __uint_as_float(r[4 * j + 2]) * p.scale, __uint_as_float(r[4 * j + 3]) * p.scale);
          fence_proxy_async_smem();
          named_bar_sync(3 + h, 128);
          if (lead && dq_ok &&
              DA_BOUNDS_V(col0 % 4 == 0 && col0 < D && q0 < p.n && b < p.B && head < (V2 ? 2 : 1) * p.units, col0)) {
            if (map == 1 && rd == ROUNDS - 1) {
              pend_col = col0;
              pend_head = head;
              pend_q0 = q0;
            } else {
              tma_reduce_add_4d(dqmap, stg, col0, head, q0, b);
              bulk_commit_group();
            }
          }
        }
      }
    }
    issue_pending();
    if (lead) bulk_wait_all();  // the dQ reduce-adds have completed
    // ---- epilogue: dV and dK of the CTA's keys (thread = key row); warpgroup h writes dV columns
    // [32 h, +32) and dK columns [32 h, +32) of (dK_1 | dK_2) (V1) or of dK (V2).
    if (__all_sync(0xffffffffu, mbar_wait(acc_done, 0, ab))) {
      tc_fence_after();
      const long long krow = static_cast<long long>(b) * p.n + key;
      float* dvp = p.dv + (krow * p.heads_kv + hk) * DV + 32 * h;
      float* dkp = V2 ? p.dk1 + (krow * p.heads_kv + hk) * D + 32 * h
                      : (h < 2 ? p.dk1 : p.dk2) + (krow * p.heads_kv + hk) * D + 32 * (h & 1);
      const uint32_t tk = V2 ? C::TM_DK1 + 32u * h : (h < 2 ? C::TM_DK1 : C::TM_DK2) + 32u * (h & 1);
      uint32_t r[32], g[32];
      tmem_ld32(tl + C::TM_DV + 32u * h, r);
      tmem_ld32(tl + tk, g);
      tmem_ld_wait2(r, g);
      if (key_ok && DA_BOUNDS_V(krow < static_cast<long long>(p.B) * p.n && hk < p.heads_kv, krow)) {
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          reinterpret_cast<float4*>(dvp)[v] = make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                                          __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
          reinterpret_cast<float4*>(dkp)[v] =
              make_float4(__uint_as_float(g[4 * v]) * p.scale, __uint_as_float(g[4 * v + 1]) * p.scale,
                          __uint_as_float(g[4 * v + 2]) * p.scale, __uint_as_float(g[4 * v + 3]) * p.scale);
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
