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
// Tiles are 128 queries x 128 keys: every QK^T MMA is M128 N128 K16, the
// narrowest shape that runs at the full tensor rate on this part (N = 64 reads
// the Q operand from shared memory twice as often per flop and runs at 2/3).
//
// Pipelining.  Each hand-off between the MMA thread and the softmax warps
// costs several hundred cycles (commit -> mbarrier -> wake, and back), so no
// MMA may wait on the softmax of the tile just before it:
//   sweep 1  the O accumulator is not used yet, so all 512 TMEM columns form a
//            ring of four 128-column S buffers (S_1(j) in buffer 2j % 4, S_2(j)
//            in (2j+1) % 4); the MMA thread runs up to two tiles ahead.
//   sweep 2  P goes to shared memory (128-byte swizzled, the A operand of an
//            SS MMA), so S_1 / S_2 buffers are released as soon as the softmax
//            has loaded them: per tile the MMA issues QK2(j+1), QK1(j+1), then
//            PV(j), and the softmax of tile j+1 overlaps PV(j).
//
// Persistent variant (template flag PERSIST; else one CTA per item): one CTA
// per SM walks a list of work items, heaviest first, dealt out in "snake"
// order over the CTAs (round k: items k G .. k G + G - 1, reversed on odd
// rounds).  Ring fills, S-buffer uses and sweep-2 tile phases run on across
// items, so the next item's Q and K tiles load during the current item's last
// tiles and epilogue; q_free (both MMA warps' last QK^T of an item done)
// guards the Q buffer, o_free (every softmax warp done with O and the S_1
// buffer) guards the TMEM columns the next item's first MMAs write.
//
// Roles (640 threads, one CTA per SM):
//   warp 0      TMA producer: Q_1, Q_2 once, then K_1 / K_2 / V tiles into a
//               ring of NSLOT equal slots, in exactly the order warp 1
//               consumes them; a slot is released by a tcgen05.commit after
//               the last MMA reading it.
//   warp 1      TMEM allocator; issues the map-1 MMAs (S_1) and P.V.
//   warp 2      issues the map-2 MMAs (S_2).  (One warp cannot issue an MMA
//               faster than every ~100 cycles; an N = 128 MMA runs in 64.)
//   warps 4-19  four softmax warpgroups; thread = one query row (TMEM lane).
//               Sweep 1: warpgroup w keeps running (max, sum) of map w/2 over
//               key columns [64 (w%2), +64) of each tile.
//               Sweep 2: warpgroup w owns key columns [32 w, +32) of both
//               maps and writes its bf16 P into shared memory.
//               Epilogue: warpgroup w normalises/stores channels [w DV/4, +DV/4).
// TMEM (512 columns x 128 lanes, fp32): sweep 1: four S buffers at 0, 128,
// 256, 384; sweep 2: O at [0, DV), A (S_1) at [DV, DV+128), B (S_2) at
// [DV+128, DV+256).  Between the sweeps the per-warpgroup statistics travel
// through columns [0, 8); the epilogue's sums of squares through A.
#pragma once

#include <cuda_bf16.h>

#include "params.h"
#include "ptx.cuh"

#undef DA_BOUNDS_FILE
#define DA_BOUNDS_FILE 3

namespace da {

template <int D, int DV, bool SHARED_K, int EPI, int NSLOT, bool PERSIST, bool F8 = false>
struct TwoPassCfg {
  static constexpr int BM = 128;   // queries per CTA (TMEM lanes)
  static constexpr int BN = 128;   // keys per tile
  static constexpr int NSMWG = 4;  // softmax warpgroups
  static constexpr int NTHREADS = (4 + 4 * NSMWG) * 32;
  // F8: Q_1, Q_2, K_1, K_2 arrive as e4m3 bytes (one byte an element, a
  // whole d = 128 row in one 128-byte box); V and P stay bf16.
  static constexpr int QK_ES = F8 ? 1 : 2;  // bytes of a query/key element
  static constexpr int QB = D * QK_ES / 128;  // 128-byte swizzle boxes across a Q/K row
  static constexpr int VB = DV / 64;
  static constexpr int Q_TILE = BM * D * QK_ES;
  static constexpr int K_TILE = BN * D * QK_ES;
  static constexpr int V_TILE = BN * DV * 2;
  static constexpr int P_TILE = BM * BN * 2;  // bf16 P, two 64-key boxes
  static constexpr int SLOT = BN * D * 2;  // a bf16 key tile (an e4m3 one fills half)
  static constexpr int VF = V_TILE / SLOT;  // slots per V tile
  static constexpr int VKEYS = BN / VF;     // keys per V slot
  static constexpr int OFF_Q1 = 0;
  static constexpr int OFF_Q2 = Q_TILE;
  static constexpr int OFF_P = 2 * Q_TILE;
  static constexpr int OFF_RING = OFF_P + P_TILE;
  static constexpr int OFF_BARS = OFF_RING + NSLOT * SLOT;
  static constexpr int NBARS = 3 * NSLOT + 22;
  static constexpr int OFF_MISC = OFF_BARS + NBARS * 8;
  static constexpr int OFF_GAMMA = OFF_MISC + 16;            // float [DV] RMSNorm weight (V1)
  static constexpr int SMEM_BYTES = OFF_GAMMA + DV * 4 + 1024;  // + 1 KB alignment slack
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t TM_O = 0;
  static constexpr uint32_t TM_A = DV;
  static constexpr uint32_t TM_B = DV + 128;
  static constexpr uint32_t IDESC_QK = F8 ? idesc_e4m3(BM, BN) : idesc_bf16(BM, BN, false, false);
  static constexpr int QK_STEPS = F8 ? D / 32 : D / 16;  // MMAs per QK^T tile (32 bytes of K each)
  static constexpr uint32_t IDESC_PV = idesc_bf16(BM, DV, false, true);
  static_assert(D == 64 || D == 128, "query/key width");
  static_assert(!F8 || D == 128, "e4m3 queries and keys: d = 128 (one 128-byte box a row)");
  static_assert(DV == 256, "sweep-1 buffer ring assumes O spans two 128-column buffers");
  static_assert(V_TILE % SLOT == 0 && (VF == 1 || VF == 2), "value tile split");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
  static_assert(NSLOT >= VF + 2, "ring depth");
  static_assert(!SHARED_K, "the two MMA warps consume separate K_1 / K_2 fills");
  // Output staging per softmax warpgroup: 128 rows x 32 channels (64-byte
  // rows) in a quarter of the P buffer.
  static constexpr int STG_BYTES = BM * 64;
  static_assert(4 * STG_BYTES <= P_TILE && (DV / 4) % 32 == 0, "output staging");
  static constexpr int MAX_ITEMS = PERSIST ? 0x7fffffff : 1;  // work items per CTA
  static constexpr int FILLS_PER_TILE = 4 + VF;               // ring fills of an item with T key tiles: T * this
};

// Merge two partial softmax states (max in the scaled log2 domain, sum).
__device__ __forceinline__ void merge_state(float& m, float& l, float m2, float l2) {
  const float mn = fmaxf(m, m2);
  if (mn == -INFINITY) return;
  l = l * ex2(m - mn) + l2 * ex2(m2 - mn);
  m = mn;
}

// Running (max, sum) of 64 scores of one row (scaled log2 domain); columns at
// or beyond nvis are masked out.
__device__ __forceinline__ void row_stats64(uint32_t (&r0)[32], uint32_t (&r1)[32], int nvis, float sc, float& m,
                                            float& l) {
  if (nvis < 64) {
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      if (c >= nvis) r0[c] = __float_as_uint(-INFINITY);
      if (c + 32 >= nvis) r1[c] = __float_as_uint(-INFINITY);
    }
  }
  float t[22];
#pragma unroll
  for (int c = 0; c < 10; ++c)
    t[c] = max3(__uint_as_float(r0[3 * c]), __uint_as_float(r0[3 * c + 1]), __uint_as_float(r0[3 * c + 2]));
  t[10] = max3(__uint_as_float(r0[30]), __uint_as_float(r0[31]), __uint_as_float(r1[0]));
#pragma unroll
  for (int c = 0; c < 10; ++c)
    t[11 + c] = max3(__uint_as_float(r1[3 * c + 1]), __uint_as_float(r1[3 * c + 2]), __uint_as_float(r1[3 * c + 3]));
  t[21] = __uint_as_float(r1[31]);
#pragma unroll
  for (int c = 0; c < 7; ++c) t[c] = max3(t[3 * c], t[3 * c + 1], t[3 * c + 2]);
  t[7] = t[21];
  const float mx = max3(max3(t[0], t[1], t[2]), max3(t[3], t[4], t[5]), fmaxf(t[6], t[7]));
  const float m_new = fmaxf(m, mx * sc);
  const float base = (m_new == -INFINITY) ? 0.f : m_new;
  const uint64_t sc2 = f2pack(sc, sc);
  const uint64_t nb2 = f2pack(-base, -base);
  uint64_t acc0 = 0, acc1 = 0;
#pragma unroll
  for (int c = 0; c < 32; c += 2) {
    float a0, a1, b0, b1;
    f2unpack(fma2(f2pack(__uint_as_float(r0[c]), __uint_as_float(r0[c + 1])), sc2, nb2), a0, a1);
    f2unpack(fma2(f2pack(__uint_as_float(r1[c]), __uint_as_float(r1[c + 1])), sc2, nb2), b0, b1);
    acc0 = add2(acc0, f2pack(ex2(a0), ex2(a1)));
    acc1 = add2(acc1, f2pack(ex2(b0), ex2(b1)));
  }
  float s0, s1;
  f2unpack(add2(acc0, acc1), s0, s1);
  l = l * ex2(m - base) + (s0 + s1);
  m = m_new;
}

template <int D, int DV, bool SHARED_K, int EPI, int NSLOT, bool PERSIST, bool F8 = false>
__global__ void __launch_bounds__(640, 1)
    twopass_fwd_kernel(const __grid_constant__ TwoPassParams p, const __grid_constant__ ItemPlan plan) {
  using C = TwoPassCfg<D, DV, SHARED_K, EPI, NSLOT, PERSIST, F8>;
  constexpr int BM = C::BM, BN = C::BN;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BARS);
  uint64_t* full = bars;              // [2][NSLOT] ring slot loaded, one barrier per consuming warp
  uint64_t* empty = full + 2 * NSLOT; // [NSLOT] ring slot released by the MMAs
  uint64_t* q_full = empty + NSLOT;   // Q of the item landed
  uint64_t* o_full = q_full + 1;      // every PV of the item completed
  uint64_t* s1_full = o_full + 1;     // [4] sweep 1: S written into TMEM buffer b
  uint64_t* s1_free = s1_full + 4;    // [4] sweep 1: the map's 8 warps have loaded buffer b
  uint64_t* a2_full = s1_free + 4;    // sweep 2: S_1 of the tile in A
  uint64_t* b2_full = a2_full + 1;    // sweep 2: S_2 of the tile in B
  uint64_t* a2_free = b2_full + 1;    // sweep 2: every softmax warp has loaded A
  uint64_t* b2_free = a2_free + 1;    // sweep 2: every softmax warp has loaded B
  uint64_t* p_ready = b2_free + 1;    // sweep 2: P of the tile in shared memory
  uint64_t* pv_done = p_ready + 1;    // sweep 2: PV of the tile completed (P buffer free)
  uint64_t* q_free = pv_done + 1;     // both maps' last QK^T of the item completed
  uint64_t* o_free = q_free + 1;      // every softmax warp is done with O and the A buffer
  uint64_t* mma_done = o_free + 1;    // [2] every MMA of warp 1 / warp 2 completed (abort drain)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  // ---- this CTA's work items: its list in the host's plan, else round k
  // takes item k G + blockIdx.x, or k G + G - 1 - blockIdx.x on odd rounds;
  // the list ends at the first one past the last item.
  const int nitems = p.num_q_tiles * p.B * p.units_per_batch;
  const int G = static_cast<int>(gridDim.x);
  auto item_of = [&](int k) -> int {
    if (PERSIST && plan.count > 0) {
      const int a = plan.first[blockIdx.x] + k;
      return a < plan.first[blockIdx.x + 1] ? static_cast<int>(plan.items[a]) : nitems;
    }
    return k * G + ((k & 1) ? (G - 1 - static_cast<int>(blockIdx.x)) : static_cast<int>(blockIdx.x));
  };
  auto tiles_of = [&](const TileCoord& c) -> int {
    const int kv_end = p.causal ? min(p.n, c.q0 + BM) : p.n;
    return (kv_end + BN - 1) / BN;  // key tiles per sweep (>= 1)
  };

  // ---- set-up
  if (threadIdx.x == 0) {
    for (int s = 0; s < NSLOT; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&full[NSLOT + s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(q_full, 1);
    mbar_init(o_full, 1);
    for (int i = 0; i < 4; ++i) {
      mbar_init(&s1_full[i], 1);
      mbar_init(&s1_free[i], 8);  // the 8 warps of the map that owns buffer i
    }
    mbar_init(a2_full, 1);
    mbar_init(b2_full, 1);
    mbar_init(a2_free, 4 * C::NSMWG);
    mbar_init(b2_free, 4 * C::NSMWG);
    mbar_init(p_ready, 4 * C::NSMWG);
    mbar_init(pv_done, 1);
    mbar_init(q_free, 2);
    mbar_init(o_free, 4 * C::NSMWG);
    mbar_init(&mma_done[0], 1);
    mbar_init(&mma_done[1], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  // The epilogue's per-channel weight, staged once (a scalar global load per
  // channel sat on the epilogue's critical path).
  float* sgamma = reinterpret_cast<float*>(smem + C::OFF_GAMMA);
  for (int i = threadIdx.x; i < DV; i += C::NTHREADS)
    sgamma[i] = (EPI == kEpiRmsNorm && p.gamma != nullptr) ? p.gamma[i] : 1.f;
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
      int fill = 0, qloads = 0;
      bool ok = true;
      // Each fill signals the `full` barrier of the warp that reads it (o = 0:
      // warp 1, K_1 and V; o = 1: warp 2, K_2), so every warp sees only its
      // own fills, in order, and its parity waits are exact.  For the abort
      // drain, bit s of `last_o` is the owner of slot s's latest fill and bit
      // (o NSLOT + s) of `par` the parity of owner o's latest fill in slot s
      // (register bit masks: this bookkeeping sits on the producer's path).
      static_assert(2 * NSLOT <= 32, "bit masks");
      uint32_t last_o = 0, par = 0;
      for (int k = 0; ok && k < C::MAX_ITEMS; ++k) {
        const int idx = item_of(k);
        if (idx >= nitems) break;
        const TileCoord c = tile_coord<EPI>(p, idx);
        const int T = tiles_of(c);
        // Q of the previous item is read by its QK^T until q_free.
        if (PERSIST && k > 0 && !mbar_wait(q_free, static_cast<uint32_t>(k - 1) & 1u, ab)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(q_full, 2 * C::Q_TILE);
        for (int bx = 0; bx < C::QB; ++bx) {
          // (bounds build: query heads of the maps, V1 units, V2 2 units)
          if (DA_BOUNDS(bx * 64 < D && c.b < p.B && c.q0 < p.n &&
                        c.hq2 < (EPI == kEpiV2 ? 2 : 1) * p.units_per_batch)) {
            tma_load_4d(smem + C::OFF_Q1 + bx * BM * 128, &p.tm_q1, q_full, bx * 64, c.hq1, c.q0, c.b);
            tma_load_4d(smem + C::OFF_Q2 + bx * BM * 128, &p.tm_q2, q_full, bx * 64, c.hq2, c.q0, c.b);
          }
        }
        ++qloads;
        // One slot fill: `nbox` boxes of [rows][64 columns] at key row `key0`.
        auto load = [&](const CUtensorMap* map, int key0, int rows, int nbox, int o) {
          if (!ok) return;
          const int s = fill % NSLOT;
          const uint32_t use = static_cast<uint32_t>(fill / NSLOT);
          if (use > 0 && !mbar_wait(&empty[s], (use - 1) & 1u, ab)) {
            ok = false;
            return;
          }
          uint64_t* bar = &full[o * NSLOT + s];
          uint8_t* dst = smem + C::OFF_RING + s * C::SLOT;
          mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nbox * rows * 128));
          for (int bx = 0; bx < nbox; ++bx)
            if (DA_BOUNDS(key0 < (p.n + 127) / 128 * 128 && c.b < p.B &&  // (a box past n reads zeros)
                          c.hk < (EPI == kEpiV2 ? 2 * p.units_per_batch / p.group : p.units_per_batch)))
              tma_load_4d(dst + bx * rows * 128, map, bar, bx * 64, c.hk, key0, c.b);
          last_o = (last_o & ~(1u << s)) | (static_cast<uint32_t>(o) << s);
          par ^= 1u << (o * NSLOT + s);  // now the parity after this fill; the fill's own is the flip of it
          ++fill;
        };
        auto load_k1 = [&](int j) { load(&p.tm_k1, j * BN, BN, C::QB, 0); };
        auto load_k2 = [&](int j) { load(&p.tm_k2, j * BN, BN, C::QB, 1); };
        // The fill order is exactly the MMA warps' consumption order.
        for (int j = 0; j < T; ++j) {  // sweep 1
          load_k1(j);
          load_k2(j);
        }
        load_k2(0);  // sweep 2
        load_k1(0);
        for (int j = 0; j < T; ++j) {
          if (j + 1 < T) {
            load_k2(j + 1);
            load_k1(j + 1);
          }
          for (int part = 0; part < C::VF; ++part) load(&p.tm_v, j * BN + part * C::VKEYS, C::VKEYS, C::VB, 0);
        }
      }
      if (*ab.flag) {
        // Aborted: let the copies already issued land before the CTA exits.
        if (qloads > 0) mbar_wait_drain(q_full, static_cast<uint32_t>(qloads - 1) & 1u, kWaitBudgetCycles);
        for (int i = 0; i < NSLOT && i < fill; ++i) {
          const int o = (last_o >> i) & 1;
          mbar_wait_drain(&full[o * NSLOT + i], ((par >> (o * NSLOT + i)) & 1u) ^ 1u, kWaitBudgetCycles);
        }
      }
    }
  } else if (warp == 1 || warp == 2) {
    // =============================================================== MMA issuers
    // One warp issues at most one tcgen05.mma every ~100 cycles, while an
    // M128 N128 K16 MMA executes in 64: two issuing warps keep the tensor
    // pipe full.  Warp 1 issues every map-1 MMA (S_1) and the P.V chain,
    // warp 2 every map-2 MMA (S_2).  Each warp runs its loop warp-uniformly
    // (descriptors stay in uniform registers) and issues from one elected
    // lane; tcgen05.commit tracks the MMAs of the issuing thread, so every
    // warp commits (and releases ring slots) for its own MMAs only.
    const int mw = warp - 1;  // 0: map 1 + P.V, 1: map 2
    // Descriptors are built once; a k-step or a ring slot only adds its byte
    // offset >> 4 to the start-address field (addresses stay below 256 KB, so
    // the 14-bit field never carries into the next one).
    const uint64_t dQ = sdesc_sw128(smem_u32(smem + (mw == 0 ? C::OFF_Q1 : C::OFF_Q2)), 16, 1024);
    const uint64_t dP = sdesc_sw128(smem_u32(smem + C::OFF_P), 16, 1024);
    const uint64_t dRingK = sdesc_sw128(smem_u32(smem + C::OFF_RING), 16, 1024);
    const uint64_t dRingV = sdesc_sw128(smem_u32(smem + C::OFF_RING), C::VKEYS * 128, 1024);
    const uint32_t tS2 = tmem + (mw == 0 ? C::TM_A : C::TM_B);  // this map's sweep-2 S buffer
    uint64_t* s2_full = (mw == 0) ? a2_full : b2_full;
    uint64_t* s2_free = (mw == 0) ? a2_free : b2_free;
    // Every wait returns the same verdict in all lanes and leaves the warp converged.
    auto waitp = [&](uint64_t* bar, uint32_t parity) -> bool {
      const bool r = __all_sync(0xffffffffu, mbar_wait(bar, parity, ab));
      tc_fence_after();
      return r;
    };
    // Ring fill f sits in slot f % NSLOT and signals this warp's own `full`
    // barrier of the slot; bit s of `ph` is the parity of this warp's next
    // fill in slot s (each warp acquires its fills in increasing order).
    uint32_t ph = 0;
    uint64_t* my_full = full + mw * NSLOT;
    auto acquire = [&](int f) -> bool {
      const int s = f % NSLOT;
      const uint32_t par = (ph >> s) & 1u;
      ph ^= 1u << s;
      return waitp(&my_full[s], par);
    };
    auto qk = [&](uint32_t dst, int f) {
      const uint64_t dk = dRingK + static_cast<uint64_t>(((f % NSLOT) * C::SLOT) >> 4);
#pragma unroll
      for (int k = 0; k < C::QK_STEPS; ++k) {
        // k-step k reads 32 bytes of each row: box k / 4, bytes 32 (k % 4) .. +31
        const uint64_t a = dQ + static_cast<uint64_t>((((k >> 2) * (BM * 128)) + (k & 3) * 32) >> 4);
        const uint64_t b = dk + static_cast<uint64_t>((((k >> 2) * (BN * 128)) + (k & 3) * 32) >> 4);
        if constexpr (F8)
          mma_ss_f8_elect(dst, a, b, C::IDESC_QK, k > 0 ? 1u : 0u);
        else
          mma_ss_elect(dst, a, b, C::IDESC_QK, k > 0 ? 1u : 0u);
      }
    };
    constexpr int PER_TILE = 2 + C::VF;
    uint32_t use_lo = 0, use_hi = 0;  // sweep-1 writes so far of buffers mw and mw + 2
    int fbase = 0;                    // ring fills of earlier items
    uint32_t g1 = 0;                  // key tiles of earlier items (each sweep)
    bool ok = true;
    for (int it = 0; ok && it < C::MAX_ITEMS; ++it) {
      const int idx = item_of(it);
      if (idx >= nitems) break;
      const int T = tiles_of(tile_coord<EPI>(p, idx));
      // Fill order of the producer within an item: sweep 1 K1(j) = 2j,
      // K2(j) = 2j + 1; sweep 2 K2(0) = 2T, K1(0) = 2T + 1, then per tile j:
      // K2(j+1), K1(j+1) (if j + 1 < T) and the VF parts of V(j).
      const int F2 = fbase + 2 * T;
      auto fill_k_next = [&](int j) { return F2 + 2 + PER_TILE * j + (mw == 0 ? 1 : 0); };  // K_map(j+1)
      auto fill_v = [&](int j, int part) { return F2 + 2 + PER_TILE * j + (j + 1 < T ? 2 : 0) + part; };
      ok = waitp(q_full, static_cast<uint32_t>(it) & 1u);
      if (PERSIST && it > 0) {
        // The previous item's epilogue reads O (buffers 0, 1) and A; o_free
        // follows it, and so every sweep-2 read of the S buffers 2 and 3.
        ok = ok && waitp(o_free, static_cast<uint32_t>(it - 1) & 1u);
      }
      // ---- sweep 1: S_map(j) (S index k = 2 (g1 + j) + mw) goes to TMEM buffer k % 4
      for (int j = 0; ok && j < T; ++j) {
        const uint32_t k = 2u * (g1 + static_cast<uint32_t>(j)) + static_cast<uint32_t>(mw);
        const int bb = static_cast<int>(k & 3u);
        uint32_t& use = (bb & 2) ? use_hi : use_lo;
        if (!acquire(fbase + 2 * j + mw)) {
          ok = false;
          break;
        }
        if (use > 0 && !waitp(&s1_free[bb], (use - 1) & 1u)) {  // read since its last write
          ok = false;
          break;
        }
        ++use;
        qk(tmem + 128u * bb, fbase + 2 * j + mw);
        tc_commit_elect(&s1_full[bb]);
        tc_commit_elect(&empty[(fbase + 2 * j + mw) % NSLOT]);
      }
      // ---- sweep 2: this map's S buffer is sweep-1 buffer mw + 2 (A or B)
      if (ok && use_hi > 0) ok = waitp(&s1_free[mw + 2], (use_hi - 1) & 1u);
      if (ok) {
        const int f = F2 + (mw == 0 ? 1 : 0);
        ok = acquire(f);
        if (ok) {
          qk(tS2, f);
          tc_commit_elect(s2_full);
          tc_commit_elect(&empty[f % NSLOT]);
          if (PERSIST && T == 1) tc_commit_elect(q_free);
        }
      }
      for (int j = 0; ok && j < T; ++j) {
        const uint32_t ph2 = (g1 + static_cast<uint32_t>(j)) & 1u;
        if (j + 1 < T) {
          const int f = fill_k_next(j);
          if (!acquire(f) || !waitp(s2_free, ph2)) {
            ok = false;
            break;
          }
          qk(tS2, f);
          tc_commit_elect(s2_full);
          tc_commit_elect(&empty[f % NSLOT]);
          if (PERSIST && j + 2 == T) tc_commit_elect(q_free);  // the item's last QK^T of this map
        }
        if (mw == 0) {
          bool got = true;
#pragma unroll
          for (int part = 0; part < C::VF; ++part) got = acquire(fill_v(j, part)) && got;
          if (!got || !waitp(p_ready, ph2)) {
            ok = false;
            break;
          }
#pragma unroll
          for (int part = 0; part < C::VF; ++part) {
            const uint64_t dv = dRingV + static_cast<uint64_t>(((fill_v(j, part) % NSLOT) * C::SLOT) >> 4);
#pragma unroll
            for (int kk = 0; kk < C::VKEYS / 16; ++kk) {
              const int kg = part * (C::VKEYS / 16) + kk;  // global k-step: keys 16 kg .. 16 kg + 15
              mma_ss_elect(tmem + C::TM_O,
                           dP + static_cast<uint64_t>((((kg >> 2) * (BM * 128)) + (kg & 3) * 32) >> 4),
                           dv + static_cast<uint64_t>(kk * (2048 >> 4)), C::IDESC_PV, (j > 0 || kg > 0) ? 1u : 0u);
            }
            // Each V part is released as soon as its own MMAs are done, so the
            // next tile's first part starts loading half a P.V earlier.
            if (part + 1 < C::VF) tc_commit_elect(&empty[fill_v(j, part) % NSLOT]);
          }
          tc_commit_elect(pv_done);
          tc_commit_elect(&empty[fill_v(j, C::VF - 1) % NSLOT]);
        }
      }
      if (!ok) break;
      if (mw == 0) tc_commit_elect(o_full);
      fbase += C::FILLS_PER_TILE * T;
      g1 += static_cast<uint32_t>(T);
    }
    tc_commit_elect(&mma_done[mw]);
    if (*ab.flag) mbar_wait_drain(&mma_done[mw], 0, kWaitBudgetCycles);
    __syncwarp();
  } else if (warp >= 4) {
    // =============================================================== softmax + epilogue
    const int wg = (warp - 4) >> 2;  // 0..3
    const int wq = warp & 3;         // TMEM lane quarter
    const int row = wq * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const int map = wg >> 1;
    const int half = wg & 1;
    // Softmax scale x log2(e) of each map; with e4m3 inputs each map's also
    // carries its query and key dequantisation scales.
    const float sc_a = p.scale_log2;
    const float sc_b = F8 ? p.scale2_log2 : p.scale_log2;
    const float sc = map == 0 ? sc_a : sc_b;
    const float lam = (EPI == kEpiRmsNorm) ? *p.lambda : 0.f;  // read once per CTA
    uint32_t g1 = 0;  // key tiles of earlier items (each sweep)

    for (int it = 0; it < C::MAX_ITEMS; ++it) {
      const int idx = item_of(it);
      if (idx >= nitems) break;
      const TileCoord c = tile_coord<EPI>(p, idx);
      const int T = tiles_of(c);
      const int t = c.q0 + row;
      const int lim = p.causal ? min(t + 1, p.n) : p.n;  // keys j < lim are visible

      // ---- sweep 1: running max / sum of map (wg / 2) over key columns [64 (wg % 2), +64)
      float m = -INFINITY, l = 0.f;
      uint32_t ready = 0;  // early test of this tile's barrier, made during the previous tile
      for (int j = 0; j < T; ++j) {
        const uint32_t k = 2u * (g1 + static_cast<uint32_t>(j)) + static_cast<uint32_t>(map);  // buffer k % 4, its (k / 4)-th write
        const int bb = static_cast<int>(k & 3u);
        if (!ready) mbar_wait(&s1_full[bb], (k >> 2) & 1u, ab);
        __syncwarp();
        tc_fence_after();
        uint32_t r0[32], r1[32];
        const uint32_t tbuf = tl + 128u * bb + 64u * half;
        tmem_ld32(tbuf, r0);
        tmem_ld32(tbuf + 32, r1);
        // The MMA warps run ahead: test the next tile's buffer now (its previous
        // phase, tile j - 1, has been consumed, so the test is exact).
        ready = (j + 1 < T) ? mbar_test(&s1_full[(k + 2) & 3u], ((k + 2) >> 2) & 1u) : 0u;
        tmem_ld_wait2(r0, r1);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s1_free[bb]);
        __syncwarp();
        row_stats64(r0, r1, lim - (j * BN + 64 * half), sc, m, l);
      }

      // ---- exchange the four partial states through TMEM columns [0, 8).
      // The other map may still be reading buffer 0 for its last tile, so all
      // sweep-1 reads finish first; the next writes to buffer 0 are this
      // item's PV (after every warp has read the exchange) and, after o_free,
      // the next item's S.
      // The previous item's output stores staged in P: their issuing threads
      // (lane 0 of each warpgroup's first warp) wait for the reads before
      // this barrier, which every sweep-2 write of P follows.
      if ((threadIdx.x & 127) == 0) bulk_wait_read_all();
      tc_fence_before();
      named_bar_sync(1, 128 * C::NSMWG);
      tc_fence_after();
      tmem_st2(tl + 2u * wg, __float_as_uint(m), __float_as_uint(l));
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      named_bar_sync(1, 128 * C::NSMWG);
      tc_fence_after();
      uint32_t ps[8];
      tmem_ld8_wait(tl, ps);
      float m1 = __uint_as_float(ps[0]), l1 = __uint_as_float(ps[1]);
      merge_state(m1, l1, __uint_as_float(ps[2]), __uint_as_float(ps[3]));
      float m2 = __uint_as_float(ps[4]), l2 = __uint_as_float(ps[5]);
      merge_state(m2, l2, __uint_as_float(ps[6]), __uint_as_float(ps[7]));
      float coef = lam;
      if (EPI == kEpiV2) {
        const float lg = (t < p.n) ? p.lam_logits[c.b * p.sb + static_cast<long long>(t) * p.st + c.u] : 0.f;
        coef = 1.f / (1.f + expf(-lg));
      }
      // P = 2^(s1*sc - M1) + neg2 * 2^(s2*sc - M2),  M1 = m1 + log2 l1,
      // M2 = m2 + log2 l2 - log2 |coef|,  neg2 = -sign(coef).
      const float M1 = m1 + log2f(l1);
      const float acoef = fabsf(coef);
      const float M2 = (acoef > 0.f) ? m2 + log2f(l2) - log2f(acoef) : INFINITY;
      const float neg2 = (coef >= 0.f) ? -1.f : 1.f;
      const uint64_t sc2a = f2pack(sc_a, sc_a), sc2b = f2pack(sc_b, sc_b);
      const uint64_t nM1 = f2pack(-M1, -M1), nM2 = f2pack(-M2, -M2), ng2 = f2pack(neg2, neg2);
      // This thread's P chunks: row `row`, keys [32 wg, +32) = 64-key box wg / 2,
      // 16-byte chunks 4 (wg % 2) .. 4 (wg % 2) + 3 of the 128-byte swizzled row.
      uint8_t* prow = smem + C::OFF_P + (wg >> 1) * (BM * 128) + row * 128;

      // ---- sweep 2: signed combined weights of key columns [32 wg, +32) -> shared memory (bf16)
      for (int j = 0; j < T; ++j) {
        const uint32_t g = g1 + static_cast<uint32_t>(j);  // sweep-2 tile, counted across items
        mbar_wait(b2_full, g & 1u, ab);
        __syncwarp();
        tc_fence_after();
        uint32_t r[32];
        tmem_ld32(tl + C::TM_B + 32u * wg, r);
        tmem_ld_wait(r);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(b2_free);
        __syncwarp();
        uint64_t e2[16];
#pragma unroll
        for (int cc = 0; cc < 16; ++cc) {
          float x0, x1;
          f2unpack(fma2(f2pack(__uint_as_float(r[2 * cc]), __uint_as_float(r[2 * cc + 1])), sc2b, nM2), x0, x1);
          e2[cc] = f2pack(ex2(x0), ex2(x1));
        }
        mbar_wait(a2_full, g & 1u, ab);
        __syncwarp();
        tc_fence_after();
        tmem_ld32(tl + C::TM_A + 32u * wg, r);
        tmem_ld_wait(r);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(a2_free);
        __syncwarp();
        const int nvis = lim - (j * BN + 32 * wg);
        uint32_t pk[16];
#pragma unroll
        for (int cc = 0; cc < 16; ++cc) {
          float x0, x1;
          f2unpack(fma2(f2pack(__uint_as_float(r[2 * cc]), __uint_as_float(r[2 * cc + 1])), sc2a, nM1), x0, x1);
          float p0, p1;
          f2unpack(fma2(e2[cc], ng2, f2pack(ex2(x0), ex2(x1))), p0, p1);
          if (2 * cc >= nvis) p0 = 0.f;
          if (2 * cc + 1 >= nvis) p1 = 0.f;
          pk[cc] = pack_bf16x2(p0, p1);
        }
        // PV of the previous tile (possibly of the previous item) must have
        // completed before its P is overwritten.
        if (g > 0) mbar_wait(pv_done, (g - 1) & 1u, ab);
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
          *reinterpret_cast<uint4*>(prow + (((4 * (wg & 1) + cc) ^ (row & 7)) << 4)) =
              make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_ready);
        __syncwarp();
      }

      // ---- epilogue: warpgroup wg owns output channels [wg * DV/4, +DV/4)
      constexpr int QW = DV / 4;
      mbar_wait(o_full, static_cast<uint32_t>(it) & 1u, ab);
      __syncwarp();
      tc_fence_after();
      const uint32_t to = tl + C::TM_O + wg * QW;
      float rinv = 1.f;
      if (EPI == kEpiRmsNorm) {
        float ss0 = 0.f, ss1 = 0.f;
#pragma unroll
        for (int ch = 0; ch < QW / 32; ++ch) {
          uint32_t rr[32];
          tmem_ld32(to + 32 * ch, rr);
          tmem_ld_wait(rr);
#pragma unroll
          for (int cc = 0; cc < 32; cc += 2) {
            ss0 = fmaf(__uint_as_float(rr[cc]), __uint_as_float(rr[cc]), ss0);
            ss1 = fmaf(__uint_as_float(rr[cc + 1]), __uint_as_float(rr[cc + 1]), ss1);
          }
        }
        // Every MMA of the item has completed and every read of A is done: A
        // carries the exchange (the next item writes it only after o_free).
        tmem_st1(tl + C::TM_A + wg, __float_as_uint(ss0 + ss1));
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        named_bar_sync(1, 128 * C::NSMWG);
        tc_fence_after();
        uint32_t q4[4];
        tmem_ld4_wait(tl + C::TM_A, q4);
        const float tot = (__uint_as_float(q4[0]) + __uint_as_float(q4[1])) +
                          (__uint_as_float(q4[2]) + __uint_as_float(q4[3]));
        rinv = p.norm_mult * rsqrtf(tot * (1.f / DV) + p.eps);
      }
      uint32_t w[QW / 2];
#pragma unroll
      for (int ch = 0; ch < QW / 32; ++ch) {
        uint32_t rr[32];
        tmem_ld32(to + 32 * ch, rr);
        tmem_ld_wait(rr);
#pragma unroll
        for (int cc = 0; cc < 32; cc += 2) {
          float y0 = __uint_as_float(rr[cc]) * rinv;
          float y1 = __uint_as_float(rr[cc + 1]) * rinv;
          if (EPI == kEpiRmsNorm) {
            const int col = wg * QW + ch * 32 + cc;
            y0 *= sgamma[col];
            y1 *= sgamma[col + 1];
          }
          w[ch * 16 + (cc >> 1)] = pack_bf16x2(y0, y1);
        }
      }
      if constexpr (PERSIST) {
        // O and A are no longer read: the next item's first MMAs may write them.
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(o_free);
        __syncwarp();
      }
      // The warpgroup's 128 x QW block goes out in 128 x 32 rounds through its
      // quarter of the P buffer (free from the item's last PV until the next
      // item's sweep 2; 64-byte rows, 64-byte swizzle: 16-byte chunk v of row
      // `row` at v ^ ((row / 2) % 4)), each round one TMA store, which drops
      // rows past n.  (Row stores from registers, one row per thread and rows
      // DV * units * 2 bytes apart, took ~7k cycles per item.)
      {
        uint8_t* const srow = smem + C::OFF_P + wg * C::STG_BYTES + row * 64;
#pragma unroll
        for (int rd = 0; rd < QW / 32; ++rd) {
          if (rd > 0) {
            if ((threadIdx.x & 127) == 0) bulk_wait_read_all();  // the previous round has read the staging
            named_bar_sync(2 + wg, 128);
          }
#pragma unroll
          for (int v = 0; v < 4; ++v)
            *reinterpret_cast<uint4*>(srow + ((v ^ ((row >> 1) & 3)) << 4)) =
                make_uint4(w[16 * rd + 4 * v], w[16 * rd + 4 * v + 1], w[16 * rd + 4 * v + 2], w[16 * rd + 4 * v + 3]);
          fence_proxy_async_smem();
          named_bar_sync(2 + wg, 128);
          if ((threadIdx.x & 127) == 0) {
            if (DA_BOUNDS(wg * QW + 32 * rd < DV && c.u < p.units_per_batch && c.q0 < p.n && c.b < p.B))
              tma_store_4d(&p.tm_out, smem + C::OFF_P + wg * C::STG_BYTES, wg * QW + 32 * rd, c.u, c.q0, c.b);
            bulk_commit_group();
          }
        }
      }
      g1 += static_cast<uint32_t>(T);
    }
  }

  // ---- teardown
  if (warp >= 4 && (warp & 3) == 0 && lane == 0) bulk_wait_all();  // output stores
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace da
