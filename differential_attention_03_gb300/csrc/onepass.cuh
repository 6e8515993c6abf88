// One-sweep differential-attention forward with two online-softmax states
// (tcgen05 tensor cores, TMA, mbarriers; sm_103a).  Used where the value
// width is 128: DIFF V1 with d = 64 (V = 2d = 128) and DIFF V2 with d = 128.
//
// What it computes (per (batch, unit, 128-query tile)):
//   O_r = sum_j exp(S_r[:, j] - m_r) V_j,  l_r = sum_j exp(S_r[:, j] - m_r),   r in {1, 2}
//   out = O_1 / l_1 - c * O_2 / l_2
//   V1: c = lambda, then (1 - lambda_init) * gamma * out / sqrt(mean(out^2) + eps)
//   V2: c = sigmoid(logit[b, t, pair]); Q_1/Q_2 are query heads 2g/2g+1 over one K/V head.
// ("Differential Transformer" glossary page, "How differential attention
// works"; DIFF V2 analysis page, DiffAttn operator, V2 code, GQA pairing;
// news article section "差分注意力" for the per-head RMSNorm.)
//
// Each K/V tile is loaded once and serves both maps.  TMEM (512 columns):
// O_1 [0, 128), O_2 [128, 256), A [256, 384) holds S_1, B [384, 512) S_2.
// P placement (template flag PSM):
//   PSM = false  P_r (bf16 pairs) overwrites S_r in TMEM and PV_r reads it
//                from there (TS MMA); per map the MMAs run PV_r(j) then
//                QK_r(j+1) into the buffer PV_r(j) has just read, so a map's
//                softmax and its MMAs alternate.
//   PSM = true   P_r goes to shared memory (128-byte swizzled, SS MMA), so
//                S_r is released as soon as the softmax has loaded it:
//                QK_r(j+1) runs during the softmax of tile j and only PV_r(j)
//                waits for P_r(j); a pv_done barrier guards the P buffer and
//                the rescale of O_r.
// Either way S_r(j+1) (or pv_done) being complete implies PV_r(j) is
// complete, so a rescale of O_r never races an MMA.
//
// Rescaling is conditional: a row keeps its reference maximum until the true
// maximum exceeds it by more than 2^8 (P then stays below 256, exact enough in
// bf16 and far from fp32 overflow); when any row of a warp must move, the warp
// rescales its rows of O_r and l_r.
//
// Persistent (template flag PERSIST; else one CTA per item): one CTA per SM
// walks a list of work items (batch, unit, query tile), heaviest first, dealt out in "snake" order (round k takes items
// k G .. k G + G - 1, reversed on odd rounds), which balances the causal
// triangle as well as a greedy scheduler without any shared counter.  The
// ring, the per-tile barriers and their phases run on across items, so the
// next item's Q and K tiles and its first QK^T overlap the epilogue of the
// current one: q_free (both MMA warps' last QK^T of an item done) guards the
// Q buffer, o_free (every softmax warp has read O) guards the accumulators.
//
// Roles (608 threads, one CTA per SM):
//   warp 0      TMA producer (Q once; then K_1, K_2 / K and V tiles into a ring
//               of NSLOT equal slots, in the order the MMA warps walk them).
//   warps 1, 2  MMA issuers for map 1 and map 2 (warp 1 also allocates TMEM).
//               One warp issues at most one tcgen05.mma about every 100
//               cycles and an N = 128 MMA runs in 64, so each map gets its
//               own issuer.  Both warps walk every ring fill, wait for it and
//               commit its release once (empty barriers count two
//               arrivals), also for the other map's K tiles, which they do
//               not read.
//   warps 3-18  four softmax warpgroups, two per map: warpgroup (r, h) owns
//               key columns [64 h, +64) of every tile of map r; thread = one
//               query row (TMEM lane 32 (warp % 4) + lane).  The two halves of
//               a row agree on the running maximum through shared memory (a
//               named barrier per map and tile), so both scale P alike and
//               take the same rescale decisions; their partial row sums are
//               added in the epilogue, where warpgroup (r, h) owns output
//               channels [32 (2 r + h), +32).  Two halves give four warps per
//               SM sub-partition to hide the latency of loads and exp2.
#pragma once

#include <cuda_bf16.h>

#include "params.h"
#include "ptx.cuh"

#undef DA_BOUNDS_FILE
#define DA_BOUNDS_FILE 4

namespace da {

template <int D, bool SHARED_K, int EPI, int NSLOT, bool PSM, bool PERSIST, bool STATS = false, bool F8 = false,
          bool SAVE = false>
struct OnePassCfg {
  static constexpr int BM = 128;
  static constexpr int BN = 128;
  static constexpr int DV = 128;
  static constexpr int NCTRL = 3;  // producer, two MMA warps
  static constexpr int NSMWG = 4;  // two softmax warpgroups per map
  static constexpr int NTHREADS = (NCTRL + 4 * NSMWG) * 32;
  // F8: queries and keys arrive as e4m3 bytes; V and P stay bf16.  At d = 128
  // a row is one 128-byte box (a key fill takes half a ring slot).  At d = 64
  // (WIDE) a row's 64 bytes are read as a 128-byte box that also holds the
  // next head's 64 bytes (zeros past the last head), so the tile keeps the
  // 128-byte-swizzled layout of every other QK^T operand; the MMAs read the
  // first 64 bytes of each row only.
  static constexpr int QK_ES = F8 ? 1 : 2;       // bytes of a query/key element
  static constexpr bool WIDE = F8 && D == 64;
  static constexpr int QK_ROW = WIDE ? 128 : D * QK_ES;  // bytes of a Q/K tile row in shared memory
  static constexpr int QB = QK_ROW / 128;        // 128-byte boxes across a Q/K row
  static constexpr int VB = DV / 64;
  static constexpr int Q_TILE = BM * QK_ROW;
  static constexpr int K_TILE = BN * QK_ROW;
  static constexpr int V_TILE = BN * DV * 2;
  static constexpr int SLOT = BN * D * 2;  // a bf16 key tile
  static constexpr int VF = V_TILE / SLOT;
  static constexpr int VKEYS = BN / VF;
  static constexpr int OFF_Q1 = 0;
  static constexpr int OFF_Q2 = Q_TILE;
  static constexpr int P_TILE = BM * BN * 2;  // one map's P (bf16) when it lives in shared memory
  static constexpr int OFF_P = 2 * Q_TILE;
  static constexpr int OFF_RING = OFF_P + (PSM ? 2 * P_TILE : 0);
  static constexpr int OFF_BARS = OFF_RING + NSLOT * SLOT;
  static constexpr int NBARS = 6 + 2 * NSLOT + 8;
  static constexpr int OFF_MISC = OFF_BARS + NBARS * 8;
  // Epilogue scratch alternates with the item parity: a map that runs ahead
  // into the next item's epilogue never overwrites values still being read.
  static constexpr int OFF_LP = (OFF_MISC + 16 + 15) / 16 * 16;  // float [2 items][4][128] partial row sums
  static constexpr int OFF_SS = OFF_LP + 8 * 128 * 4;             // float [2 items][4][128] partial sums of squares
  static constexpr int OFF_XM = OFF_SS + 8 * 128 * 4;             // float [2 tiles][2 maps][2 halves][128]
  static constexpr int OFF_GAMMA = OFF_XM + 8 * 128 * 4;         // float [DV] RMSNorm weight (V1)
  static constexpr int SMEM_BYTES = OFF_GAMMA + DV * 4 + 1024;    // + 1 KB alignment slack
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t TM_O1 = 0, TM_O2 = 128, TM_A = 256, TM_B = 384;
  static constexpr uint32_t IDESC_QK = F8 ? idesc_e4m3(BM, BN) : idesc_bf16(BM, BN, false, false);
  static constexpr int QK_STEPS = D * QK_ES / 32;  // MMAs per QK^T tile (32 bytes of each row each)
  static constexpr uint32_t IDESC_PV = idesc_bf16(BM, DV, false, true);
  static constexpr float RESCALE_THRESHOLD = 8.f;  // log2 units
  static constexpr int MAX_ITEMS = PERSIST ? 0x7fffffff : 1;  // work items per CTA
  static_assert(D == 64 || D == 128, "query/key width");
  static_assert(!F8 || (!STATS && ((D == 128 && SHARED_K) || (D == 64 && !SHARED_K))),
                "e4m3 queries and keys: the V2 forward at d = 128, the V1 forward at d = 64");
  static_assert(!SAVE || (!STATS && !F8), "the training forward saves the bf16 forward's statistics");
  static_assert(V_TILE % SLOT == 0 && (VF == 1 || VF == 2), "value tile split");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
  static_assert(NSLOT >= 4, "ring depth");
  // Output staging of the one-item form (128 rows x 32 channels, 64-byte
  // rows, 64-byte swizzle) for warpgroup (r, h): the first half of its P box
  // when P is in shared memory, else a quarter of the Q buffers.
  static constexpr int STG_BYTES = BM * 64;
  static_assert(PSM || 2 * Q_TILE >= 4 * STG_BYTES, "output staging in the Q buffers");
  // STATS (the backward's statistics pass): one item per CTA; after the
  // item's last MMA the Q buffers hold the epilogue's exchange of partial
  // row sums ([6][4][128] floats) and the per-warp dgamma sums.
  static_assert(!STATS || !PERSIST, "the statistics pass runs one item per CTA");
  static constexpr int XCH_FLOATS = 6 * 4 * 128;
  static_assert(!STATS || 2 * Q_TILE >= (XCH_FLOATS + 4 * 4 * 32 + 4) * 4, "statistics exchange in the Q buffers");
};

// 32 output channels of one row: y * rinv (* gamma), rounded to bf16 pairs.
template <bool GAMMA>
__device__ __forceinline__ void pack_out_row(const float (&y)[32], float rinv, const float* g, uint32_t (&wv)[16]) {
#pragma unroll
  for (int cc = 0; cc < 32; cc += 2) {
    float y0 = y[cc] * rinv, y1 = y[cc + 1] * rinv;
    if (GAMMA) {
      y0 *= g[cc];
      y1 *= g[cc + 1];
    }
    wv[cc >> 1] = pack_bf16x2(y0, y1);
  }
}

// Epilogue of the backward's statistics pass (one item per CTA, every MMA of
// it complete): instead of the output, each row's quantities the tensor-core
// backward needs.  Thread = row `row` (token t) x channels [32 cb, +32) of
// map `map` (its running maximum m_used); l1, l2 the final row sums, coef the
// second map's coefficient (V1 lambda, V2 sigmoid of the row's logit).  With
// O_r = O_r' / l_r the normalised map outputs and O = O_1 - coef O_2:
//   V1: y = m gamma O r,  r = (mean O^2 + eps)^-1/2,  m = 1 - lambda_init;
//       G = m gamma dy,  dO = r G - (r^3 / DV) (G . O) O   (bf16 to p.dO);
//       dgamma share = dy m O r (per channel, summed over the CTA's rows).
//   V2: dO = dy.
//   Delta_1 = dO . O_1,  Delta_2 = -coef dO . O_2 (the row sums of the softmax
//   gradients: dS_r = P_r (c_r dO V^T - Delta_r) with c_1 = 1, c_2 = -coef);
//   lse_r = m_r + log2 l_r (scaled log2 domain);  share: V1 dL/dlambda of the
//   row = -dO . O_2, V2 dL/dlogit = -s (1 - s) dO . O_2.
// The four channel blocks of a row add their partial dot products through
// the Q buffers (free once the item's MMAs are done).
template <class C, int EPI>
__device__ __forceinline__ void onepass_stats_epilogue(const TwoPassParams& p, const TileCoord& c, int t, int row,
                                                       int lane, int warp, int cb, int map, float l1, float l2,
                                                       float coef, float m_used, uint32_t tl, uint8_t* smem,
                                                       const float* sgamma) {
  constexpr int DV = C::DV;
  constexpr bool V1 = EPI == kEpiRmsNorm;
  constexpr int NX = V1 ? 6 : 2;  // partial sums exchanged per row
  const bool live = t < p.n;
  const long long orow = (static_cast<long long>(c.b) * p.n + t) * p.units_per_batch + c.u;
  const float il1 = 1.f / l1, il2 = 1.f / l2;
  const float mult = p.norm_mult;
  const uint4* dysrc = reinterpret_cast<const uint4*>(p.dy + orow * DV + 32 * cb);
  // One half (16 channels) of the block: O_1, O_2 from TMEM and dy, unpacked to fp32.
  auto load_half = [&](int hf, uint32_t (&x1)[16], uint32_t (&x2)[16], float (&dyh)[16]) {
    tmem_ld16(tl + C::TM_O1 + 32u * cb + 16u * hf, x1);
    tmem_ld16(tl + C::TM_O2 + 32u * cb + 16u * hf, x2);
    uint4 u[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
    if (live) {
      u[0] = dysrc[2 * hf];
      u[1] = dysrc[2 * hf + 1];
    }
#pragma unroll
    for (int v = 0; v < 2; ++v) {
      const uint32_t w[4] = {u[v].x, u[v].y, u[v].z, u[v].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        dyh[8 * v + 2 * e] = __uint_as_float(w[e] << 16);
        dyh[8 * v + 2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
      }
    }
    tmem_ld_wait16x2(x1, x2);
  };
  // Pass 1: partial dot products of the block (V1: ss, G.O, G.O1, G.O2, O.O1, O.O2; V2: dy.O1, dy.O2),
  // with O_r = O_r' / l_r, O = O_1 - coef O_2, G = m gamma dy.
  float part[6] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    uint32_t o1[16], o2[16];
    float dyh[16];
    load_half(hf, o1, o2, dyh);
#pragma unroll
    for (int cc = 0; cc < 16; ++cc) {
      const float x1 = __uint_as_float(o1[cc]) * il1, x2 = __uint_as_float(o2[cc]) * il2;
      if constexpr (V1) {
        const float o = fmaf(-coef, x2, x1);
        const float g = mult * sgamma[32 * cb + 16 * hf + cc] * dyh[cc];
        part[0] = fmaf(o, o, part[0]);
        part[1] = fmaf(g, o, part[1]);
        part[2] = fmaf(g, x1, part[2]);
        part[3] = fmaf(g, x2, part[3]);
        part[4] = fmaf(o, x1, part[4]);
        part[5] = fmaf(o, x2, part[5]);
      } else {
        part[0] = fmaf(dyh[cc], x1, part[0]);
        part[1] = fmaf(dyh[cc], x2, part[1]);
      }
    }
  }
  float* xch = reinterpret_cast<float*>(smem + C::OFF_Q1);  // [NX][4][128]
#pragma unroll
  for (int k = 0; k < NX; ++k) xch[(k * 4 + cb) * 128 + row] = part[k];
  named_bar_sync(1, 128 * C::NSMWG);
  float tot[6];
#pragma unroll
  for (int k = 0; k < NX; ++k)
    tot[k] = (xch[(k * 4) * 128 + row] + xch[(k * 4 + 1) * 128 + row]) +
             (xch[(k * 4 + 2) * 128 + row] + xch[(k * 4 + 3) * 128 + row]);
  float delta1, delta2, share;
  if constexpr (V1) {
    const float r = rsqrtf(tot[0] * (1.f / DV) + p.eps);
    const float k3 = r * r * r * (1.f / DV) * tot[1];
    const float dO1 = r * tot[2] - k3 * tot[4];  // dO . O_1
    const float dO2 = r * tot[3] - k3 * tot[5];  // dO . O_2
    delta1 = dO1;
    delta2 = -coef * dO2;
    share = -dO2;
    // Pass 2: dO of the block (bf16) and its dgamma shares, dg = dy m O r, each half summed over the
    // warp's 32 rows: lane l ends with channel l % 16 of the half (each butterfly step halves the
    // channels a lane holds and doubles the rows), the last step adds the two lane halves.
    float dgw[2];
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      uint32_t o1[16], o2[16];
      float dyh[16], dg[16];
      load_half(hf, o1, o2, dyh);
      uint32_t w[8];
#pragma unroll
      for (int cc = 0; cc < 16; cc += 2) {
        float ov[2], gv[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float x1 = __uint_as_float(o1[cc + e]) * il1, x2 = __uint_as_float(o2[cc + e]) * il2;
          ov[e] = fmaf(-coef, x2, x1);
          gv[e] = mult * sgamma[32 * cb + 16 * hf + cc + e] * dyh[cc + e];
          dg[cc + e] = live ? dyh[cc + e] * mult * ov[e] * r : 0.f;
        }
        w[cc >> 1] = pack_bf16x2(r * gv[0] - k3 * ov[0], r * gv[1] - k3 * ov[1]);
      }
      if (live && DA_BOUNDS_V(orow >= 0 && orow < p.rows, orow)) {
        uint4* dst = reinterpret_cast<uint4*>(p.dO + orow * DV + 32 * cb + 16 * hf);
        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
      }
#pragma unroll
      for (int sft = 8; sft >= 1; sft >>= 1) {
        const bool upper = (lane & sft) != 0;
#pragma unroll
        for (int j = 0; j < sft; ++j) {
          const float send = upper ? dg[j] : dg[j + sft];
          const float keep = upper ? dg[j + sft] : dg[j];
          dg[j] = keep + __shfl_xor_sync(0xffffffffu, send, sft);
        }
      }
      dgw[hf] = dg[0] + __shfl_xor_sync(0xffffffffu, dg[0], 16);  // channel 16 hf + lane % 16
    }
    // lanes 0..15 hold channels 0..15 (half 0) and 16..31 (half 1): lane l writes channel l
    const float mine = lane < 16 ? dgw[0] : dgw[1];
    float* wsum = xch + C::XCH_FLOATS;  // [4 channel blocks][4 warps][32], then [4 warps] dlambda sums
    wsum[(cb * 4 + (warp & 3)) * 32 + lane] = mine;
    if (cb == 0) {  // the rows' dlambda shares, summed over the warp's 32 rows
      float sh = live ? -dO2 : 0.f;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) sh += __shfl_xor_sync(0xffffffffu, sh, off);
      if (lane == 0) wsum[16 * 32 + (warp & 3)] = sh;
    }
    named_bar_sync(1, 128 * C::NSMWG);
    if ((warp & 3) == 0) {
      const float* ws = wsum + cb * 4 * 32;
      DA_STORE(p.dgp, static_cast<long long>(blockIdx.x) * DV + 32 * cb + lane, static_cast<long long>(gridDim.x) * DV,
               (ws[lane] + ws[32 + lane]) + (ws[64 + lane] + ws[96 + lane]));
      if (cb == 0 && lane == 0)
        DA_STORE(p.dlam_part, blockIdx.x, gridDim.x,
                 (wsum[16 * 32] + wsum[16 * 32 + 1]) + (wsum[16 * 32 + 2] + wsum[16 * 32 + 3]));
    }
  } else {
    delta1 = tot[0];
    delta2 = -coef * tot[1];
    share = -coef * (1.f - coef) * tot[1];
  }
  if (live) {
    const long long ri = (static_cast<long long>(c.b) * p.units_per_batch + c.u) * p.n + t;
    if (!DA_BOUNDS_V(ri >= 0 && ri < p.rows && c.b < p.B && t < p.n && c.u < p.units_per_batch, ri)) {
    } else if (cb == 0) {  // map 1's running maximum lives in its warpgroups
      p.row[ri] = m_used + log2f(l1);
      p.row[2 * p.rows + ri] = delta1;
      p.row[3 * p.rows + ri] = delta2;
      p.row[4 * p.rows + ri] = share;
      p.row[5 * p.rows + ri] = coef;
      if (!V1 && p.dlogits_dense != nullptr) p.dlogits_dense[c.b * p.sb + static_cast<long long>(t) * p.st + c.u] = share;
    } else if (cb == 2) {
      p.row[p.rows + ri] = m_used + log2f(l2);
    }
  }
  (void)map;
}

template <int D, bool SHARED_K, int EPI, int NSLOT, bool PSM, bool PERSIST, bool STATS = false, bool F8 = false,
          bool SAVE = false>
__global__ void __launch_bounds__(608, 1) onepass_fwd_kernel(const __grid_constant__ TwoPassParams p) {
  using C = OnePassCfg<D, SHARED_K, EPI, NSLOT, PSM, PERSIST, STATS, F8, SAVE>;
  constexpr int BM = C::BM, BN = C::BN, DV = C::DV;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BARS);
  uint64_t* q_full = bars + 0;       // Q of the item landed
  uint64_t* o_full = bars + 1;       // every PV of the item completed (both MMA warps)
  uint64_t* q_free = bars + 2;       // the item's last QK^T of both maps completed: Q may be replaced
  uint64_t* o_free = bars + 3;       // every softmax warp has read the item's O
  uint64_t* mma_done = bars + 4;     // [2] every MMA of an MMA warp completed (abort drain)
  uint64_t* full = bars + 6;
  uint64_t* empty = full + NSLOT;
  uint64_t* s_full = empty + NSLOT;  // [2]: S_r of the current tile in its buffer
  uint64_t* p_ready = s_full + 2;    // [2]: P_r of the current tile written
  uint64_t* s_free = p_ready + 2;    // [2]: (PSM) S_r loaded by the map's softmax warps
  uint64_t* pv_done = s_free + 2;    // [2]: (PSM) PV_r of the tile completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  float* lpart = reinterpret_cast<float*>(smem + C::OFF_LP);
  float* sspart = reinterpret_cast<float*>(smem + C::OFF_SS);
  float* xmax = reinterpret_cast<float*>(smem + C::OFF_XM);
  float* sgamma = reinterpret_cast<float*>(smem + C::OFF_GAMMA);

  // ---- this CTA's work items: round k takes item k G + blockIdx.x, or
  // k G + G - 1 - blockIdx.x on odd rounds; the list ends at the first one
  // past the last item (later rounds start further on).
  const int nitems = p.num_q_tiles * p.B * p.units_per_batch;
  const int G = static_cast<int>(gridDim.x);
  auto item_of = [&](int k) -> int {
    return k * G + ((k & 1) ? (G - 1 - static_cast<int>(blockIdx.x)) : static_cast<int>(blockIdx.x));
  };
  auto tiles_of = [&](const TileCoord& c) -> int {
    const int kv_end = p.causal ? min(p.n, c.q0 + BM) : p.n;
    return (kv_end + BN - 1) / BN;
  };

  // ---- set-up
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(o_full, 2);  // both MMA warps
    mbar_init(q_free, 2);  // both MMA warps
    mbar_init(o_free, 4 * C::NSMWG);
    mbar_init(&mma_done[0], 1);
    mbar_init(&mma_done[1], 1);
    for (int s = 0; s < NSLOT; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 2);  // both MMA warps release every fill
    }
    for (int r = 0; r < 2; ++r) {
      mbar_init(&s_full[r], 1);
      mbar_init(&p_ready[r], 8);  // the map's 8 softmax warps
      mbar_init(&s_free[r], 8);
      mbar_init(&pv_done[r], 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  // The epilogue's per-channel weight, staged once per CTA (a scalar global
  // load per channel and item sat on the epilogue's critical path).
  if (threadIdx.x < DV) sgamma[threadIdx.x] = (EPI == kEpiRmsNorm && p.gamma != nullptr) ? p.gamma[threadIdx.x] : 1.f;
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
            // (WIDE maps are {H d bytes, 1, n, B}: a head's row starts at byte h d)
            tma_load_4d(smem + C::OFF_Q1 + bx * BM * 128, &p.tm_q1, q_full, C::WIDE ? c.hq1 * D : bx * 64,
                        C::WIDE ? 0 : c.hq1, c.q0, c.b);
            tma_load_4d(smem + C::OFF_Q2 + bx * BM * 128, &p.tm_q2, q_full, C::WIDE ? c.hq2 * D : bx * 64,
                        C::WIDE ? 0 : c.hq2, c.q0, c.b);
          }
        }
        ++qloads;
        auto load = [&](const CUtensorMap* map, int key0, int rows, int nbox) {
          if (!ok) return;
          const int s = fill % NSLOT;
          const uint32_t use = static_cast<uint32_t>(fill / NSLOT);
          if (use > 0 && !mbar_wait(&empty[s], (use - 1) & 1u, ab)) {
            ok = false;
            return;
          }
          uint8_t* dst = smem + C::OFF_RING + s * C::SLOT;
          mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(nbox * rows * 128));
          for (int bx = 0; bx < nbox; ++bx)
            if (DA_BOUNDS(key0 < (p.n + 127) / 128 * 128 && c.b < p.B &&  // (a box past n reads zeros)
                          c.hk < (EPI == kEpiV2 ? 2 * p.units_per_batch / p.group : p.units_per_batch)))
              tma_load_4d(dst + bx * rows * 128, map, &full[s],
                          (C::WIDE && map != &p.tm_v) ? c.hk * D : bx * 64,
                          (C::WIDE && map != &p.tm_v) ? 0 : c.hk, key0, c.b);
          ++fill;
        };
        // The fill order is the order in which both MMA warps walk the ring.
        load(&p.tm_k1, 0, BN, C::QB);
        if (!SHARED_K) load(&p.tm_k2, 0, BN, C::QB);
        // PSM: the next tile's K before this tile's V (QK(j+1) is issued
        // before PV(j)); otherwise after it.
        for (int j = 0; j < T; ++j) {
          if (PSM && j + 1 < T) {
            load(&p.tm_k1, (j + 1) * BN, BN, C::QB);
            if (!SHARED_K) load(&p.tm_k2, (j + 1) * BN, BN, C::QB);
          }
          for (int part = 0; part < C::VF; ++part) load(&p.tm_v, j * BN + part * C::VKEYS, C::VKEYS, C::VB);
          if (!PSM && j + 1 < T) {
            load(&p.tm_k1, (j + 1) * BN, BN, C::QB);
            if (!SHARED_K) load(&p.tm_k2, (j + 1) * BN, BN, C::QB);
          }
        }
      }
      if (*ab.flag) {
        // Aborted: let the copies already issued land before the CTA exits.
        if (qloads > 0) mbar_wait_drain(q_full, static_cast<uint32_t>(qloads - 1) & 1u, kWaitBudgetCycles);
        for (int f = (fill > NSLOT ? fill - NSLOT : 0); f < fill; ++f)
          mbar_wait_drain(&full[f % NSLOT], static_cast<uint32_t>(f / NSLOT) & 1u, kWaitBudgetCycles);
      }
    }
  } else if (warp == 1 || warp == 2) {
    // =============================================================== MMA issuers
    // Warp 1 + r issues every MMA of map r + 1, warp-uniformly (descriptors
    // stay in uniform registers), each from one elected lane.
    const int r = warp - 1;
    const uint64_t dQ = sdesc_sw128(smem_u32(smem + (r == 0 ? C::OFF_Q1 : C::OFF_Q2)), 16, 1024);
    const uint64_t dRingK = sdesc_sw128(smem_u32(smem + C::OFF_RING), 16, 1024);
    const uint64_t dRingV = sdesc_sw128(smem_u32(smem + C::OFF_RING), C::VKEYS * 128, 1024);
    const uint64_t dP = sdesc_sw128(smem_u32(smem + C::OFF_P + r * C::P_TILE), 16, 1024);
    const uint32_t tS = tmem + (r == 0 ? C::TM_A : C::TM_B);
    const uint32_t tO = tmem + (r == 0 ? C::TM_O1 : C::TM_O2);
    // Every wait returns the same verdict in all lanes and leaves the warp converged.
    auto waitp = [&](uint64_t* bar, uint32_t parity) -> bool {
      const bool v = __all_sync(0xffffffffu, mbar_wait(bar, parity, ab));
      tc_fence_after();
      return v;
    };
    int fill = 0;  // next ring fill: slot fill % NSLOT, its (fill / NSLOT)-th use
    // Both warps wait on every fill in ring order, so each parity wait
    // follows the completion of the slot's previous phase and is exact.
    auto acquire_next = [&](int& s) -> bool {
      s = fill % NSLOT;
      const uint32_t use = static_cast<uint32_t>(fill / NSLOT);
      ++fill;
      return waitp(&full[s], use & 1u);
    };
    // A fill this map does not read is still awaited and then released: every
    // arrival on a slot's empty barrier then follows the issue of that fill,
    // so no warp can run ahead into the slot's next phase.
    auto skip_next = [&]() -> bool {
      int s;
      const bool v = acquire_next(s);
      tc_commit_elect(&empty[s]);
      return v;
    };
    auto qk = [&](int s) {
      const uint64_t dk = dRingK + static_cast<uint64_t>((s * C::SLOT) >> 4);
#pragma unroll
      for (int k = 0; k < C::QK_STEPS; ++k) {
        // k-step k reads 32 bytes of each row: box k / 4, bytes 32 (k % 4) .. +31
        const uint64_t a = dQ + static_cast<uint64_t>((((k >> 2) * (BM * 128)) + (k & 3) * 32) >> 4);
        const uint64_t b = dk + static_cast<uint64_t>((((k >> 2) * (BN * 128)) + (k & 3) * 32) >> 4);
        if constexpr (F8)
          mma_ss_f8_elect(tS, a, b, C::IDESC_QK, k > 0 ? 1u : 0u);
        else
          mma_ss_elect(tS, a, b, C::IDESC_QK, k > 0 ? 1u : 0u);
      }
    };
    // K fills of the tile with global index g (tiles counted across items):
    // K (shared) or K_1 then K_2.  With P in shared memory QK_r(g) only waits
    // until the softmax has loaded S_r(g-1).  After an item's last QK^T both
    // warps release the Q buffer.
    auto k_tile = [&](uint32_t g, bool last_of_item) -> bool {
      if (!SHARED_K && r == 1 && !skip_next()) return false;
      int s;
      if (!acquire_next(s)) return false;
      if (PSM && g > 0 && !waitp(&s_free[r], (g - 1) & 1u)) return false;
      qk(s);
      tc_commit_elect(&s_full[r]);
      tc_commit_elect(&empty[s]);
      if (PERSIST && last_of_item) tc_commit_elect(q_free);
      return SHARED_K || r == 1 || skip_next();
    };
    bool ok = true;
    uint32_t gt = 0;  // tiles of earlier items
    for (int k = 0; ok && k < C::MAX_ITEMS; ++k) {
      const int idx = item_of(k);
      if (idx >= nitems) break;
      const int T = tiles_of(tile_coord<EPI>(p, idx));
      if (!waitp(q_full, static_cast<uint32_t>(k) & 1u) || !k_tile(gt, T == 1)) {
        ok = false;
        break;
      }
      for (int j = 0; ok && j < T; ++j) {
        const uint32_t g = gt + static_cast<uint32_t>(j);
        if (PSM && j + 1 < T && !k_tile(g + 1, j + 2 == T)) {
          ok = false;
          break;
        }
        int sv[C::VF];
        bool got = true;
#pragma unroll
        for (int part = 0; part < C::VF; ++part) got = acquire_next(sv[part]) && got;
        if (!got || !waitp(&p_ready[r], g & 1u)) {
          ok = false;
          break;
        }
        // The first PV of an item overwrites O_r: the previous item's
        // epilogue must have read it.
        if (PERSIST && j == 0 && k > 0 && !waitp(o_free, static_cast<uint32_t>(k - 1) & 1u)) {
          ok = false;
          break;
        }
        // PV_r(j): P_r from shared memory (k-step kg: keys 16 kg .. 16 kg + 15 =
        // 64-key box kg / 4, 32-byte step kg % 4), or bf16 pairs in TMEM columns
        // 8 kg .. 8 kg + 7 of the S_r buffer.
#pragma unroll
        for (int part = 0; part < C::VF; ++part) {
          const uint64_t dv = dRingV + static_cast<uint64_t>((sv[part] * C::SLOT) >> 4);
#pragma unroll
          for (int kk = 0; kk < C::VKEYS / 16; ++kk) {
            const int kg = part * (C::VKEYS / 16) + kk;
            const uint64_t dvk = dv + static_cast<uint64_t>(kk * (2048 >> 4));
            const uint32_t acc = (j > 0 || kg > 0) ? 1u : 0u;
            if (PSM)
              mma_ss_elect(tO, dP + static_cast<uint64_t>((((kg >> 2) * (BM * 128)) + (kg & 3) * 32) >> 4), dvk,
                           C::IDESC_PV, acc);
            else
              mma_ts_elect(tO, tS + 8u * kg, dvk, C::IDESC_PV, acc);
          }
          // Each V part is released as soon as its own MMAs are done.
          if (part + 1 < C::VF) tc_commit_elect(&empty[sv[part]]);
        }
        if (PSM) tc_commit_elect(&pv_done[r]);
        tc_commit_elect(&empty[sv[C::VF - 1]]);
        if (!PSM && j + 1 < T && !k_tile(g + 1, j + 2 == T)) {
          ok = false;
          break;
        }
      }
      if (!ok) break;
      tc_commit_elect(o_full);
      gt += static_cast<uint32_t>(T);
    }
    tc_commit_elect(&mma_done[r]);
    if (*ab.flag) mbar_wait_drain(&mma_done[r], 0, kWaitBudgetCycles);
    __syncwarp();
  } else {
    // =============================================================== softmax + epilogue
    const int sw = warp - C::NCTRL;   // 0..15
    const int map = sw >> 3;          // map (map + 1)
    const int half = (sw >> 2) & 1;   // key columns [64 half, +64) of each tile
    const int wq = warp & 3;          // TMEM lane quarter
    const int row = wq * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    // softmax scale x log2(e) of this warp's map (e4m3 inputs: with that map's dequantisation scales)
    const float sc = (F8 && map) ? p.scale2_log2 : p.scale_log2;
    const uint32_t tS = tl + (map ? C::TM_B : C::TM_A);
    const uint32_t tOr = tl + (map ? C::TM_O2 : C::TM_O1);
    const uint64_t sc2 = f2pack(sc, sc);
    const int cb = 2 * map + half;  // epilogue: output channels [32 cb, +32)
    const float lam = (EPI == kEpiRmsNorm) ? *p.lambda : 0.f;  // read once per CTA
    uint32_t gt = 0;                // tiles of earlier items

    for (int k = 0; k < C::MAX_ITEMS; ++k) {
      const int idx = item_of(k);
      if (idx >= nitems) break;
      const TileCoord c = tile_coord<EPI>(p, idx);
      const int T = tiles_of(c);
      const int t = c.q0 + row;
      const int lim = p.causal ? min(t + 1, p.n) : p.n;
      float m_used = -INFINITY, l = 0.f;
      uint32_t ready = 0;  // (PSM) early test of this tile's barrier, made during the previous tile

      for (int j = 0; j < T; ++j) {
        const uint32_t g = gt + static_cast<uint32_t>(j);
        if (!ready) mbar_wait(&s_full[map], g & 1u, ab);
        __syncwarp();
        tc_fence_after();
        uint32_t x[2][32];
#pragma unroll
        for (int q = 0; q < 2; ++q) tmem_ld32(tS + 64u * half + 32u * q, x[q]);
        tmem_ld_wait2(x[0], x[1]);
        if constexpr (PSM) {
          // S_r is in registers: the next tile's QK^T may overwrite the buffer.
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&s_free[map]);
          __syncwarp();
        }
        const int nvis = lim - (j * BN + 64 * half);
        if (nvis < 64) {
#pragma unroll
          for (int q = 0; q < 2; ++q)
#pragma unroll
            for (int cc = 0; cc < 32; ++cc)
              if (32 * q + cc >= nvis) x[q][cc] = __float_as_uint(-INFINITY);
        }
        float mq[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          float tm[11];
#pragma unroll
          for (int cc = 0; cc < 10; ++cc)
            tm[cc] = max3(__uint_as_float(x[q][3 * cc]), __uint_as_float(x[q][3 * cc + 1]),
                          __uint_as_float(x[q][3 * cc + 2]));
          tm[10] = fmaxf(__uint_as_float(x[q][30]), __uint_as_float(x[q][31]));
          mq[q] = max3(max3(tm[0], tm[1], tm[2]), max3(tm[3], tm[4], tm[5]), max3(max3(tm[6], tm[7], tm[8]), tm[9], tm[10]));
        }
        // Row maximum of the whole tile: exchange with the other half.  The
        // buffer alternates with the (global) tile, so a half one tile ahead
        // never overwrites a value the other half has yet to read.
        float* xm = xmax + ((g & 1u) * 2 + map) * 256;
        const float pm = fmaxf(mq[0], mq[1]);
        xm[half * 128 + row] = pm;
        named_bar_sync(2 + map, 256);
        const float mx = fmaxf(pm, xm[(half ^ 1) * 128 + row]);
        const float m_new = fmaxf(m_used, mx * sc);
        const bool rescale = __any_sync(0xffffffffu, m_new > m_used + C::RESCALE_THRESHOLD);
        float factor = 1.f;
        if (rescale) {
          factor = ex2(m_used - m_new);  // 0 on the first tile of an item
          l *= factor;
          m_used = m_new;
        }
        const uint64_t nb2 = f2pack(-m_used, -m_used);
        uint64_t acc[2] = {0, 0};
        // P pairs are packed in place over score registers already consumed:
        // x[q][0..15] then hold key columns 64 half + 32 q .. + 31 as bf16 pairs.
#pragma unroll
        for (int q = 0; q < 2; ++q) {
#pragma unroll
          for (int cc = 0; cc < 32; cc += 2) {
            float a0, a1;
            f2unpack(fma2(f2pack(__uint_as_float(x[q][cc]), __uint_as_float(x[q][cc + 1])), sc2, nb2), a0, a1);
            const float p0 = ex2(a0), p1 = ex2(a1);
            acc[q] = add2(acc[q], f2pack(p0, p1));
            x[q][cc >> 1] = pack_bf16x2(p0, p1);
          }
        }
        float s0, s1;
        f2unpack(add2(acc[0], acc[1]), s0, s1);
        l += s0 + s1;
        if constexpr (PSM) {
          // QK_r(g+1) was issued once S_r(g) was loaded: test its barrier now,
          // off the critical path (phase g has been consumed: the test is exact).
          ready = (j + 1 < T) ? mbar_test(&s_full[map], (g + 1) & 1u) : 0u;
          // PV_r(g-1) must be complete before P_r is overwritten or O_r rescaled.
          if (g > 0) {
            mbar_wait(&pv_done[map], (g - 1) & 1u, ab);
            __syncwarp();
            tc_fence_after();
          }
          // Row `row` of P_r, keys [64 half, +64) = 64-key box `half`: 16-byte
          // chunk cc holds keys 8cc .. 8cc + 7 of the box, at position cc ^ (row % 8).
          uint8_t* prow = smem + C::OFF_P + map * C::P_TILE + half * (BM * 128) + row * 128;
#pragma unroll
          for (int cc = 0; cc < 8; ++cc)
            *reinterpret_cast<uint4*>(prow + ((cc ^ (row & 7)) << 4)) =
                make_uint4(x[cc >> 2][4 * (cc & 3)], x[cc >> 2][4 * (cc & 3) + 1], x[cc >> 2][4 * (cc & 3) + 2],
                           x[cc >> 2][4 * (cc & 3) + 3]);
          fence_proxy_async_smem();
        } else {
          // P of key columns 32 q' .. 32 q' + 31 (q' = 2 half + q) -> buffer
          // columns 16 q' .. 16 q' + 15 (this thread's own row; the S columns it
          // overwrites are its own and already loaded).
#pragma unroll
          for (int q = 0; q < 2; ++q)
            tmem_st16(tS + 32u * half + 16u * q, reinterpret_cast<const uint32_t(&)[16]>(x[q]));
        }
        if (rescale && j > 0) {
          // PV_r(j-1) is complete: awaited above (PSM), or issued by the same
          // warp before QK_r(j), whose commit of S_r(j) tracks all its MMAs.
          // This half rescales O_r columns [64 half, +64) of its rows.  (On an
          // item's first tile O_r still holds the previous item: PV_r(0)
          // overwrites it.)
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            uint32_t o[32];
            tmem_ld32(tOr + 64u * half + 32u * q, o);
            tmem_ld_wait(o);
#pragma unroll
            for (int cc = 0; cc < 32; ++cc) o[cc] = __float_as_uint(__uint_as_float(o[cc]) * factor);
            tmem_st32(tOr + 64u * half + 32u * q, o);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_ready[map]);
        __syncwarp();
      }

      // ---- epilogue: out = O_1 / l_1 - c O_2 / l_2; warpgroup (map, half)
      // owns channels [32 cb, +32).  The row sums are final after the last
      // tile; the persistent form exchanges them while the last PVs still
      // run (one CTA per item measured better with the exchange after o_full).
      float* lp = lpart + (k & 1) * 512;
      float l1 = 0.f, l2 = 0.f;
      auto exchange_l = [&]() {
        lp[cb * 128 + row] = l;
        named_bar_sync(1, 128 * C::NSMWG);
        l1 = lp[row] + lp[128 + row];
        l2 = lp[256 + row] + lp[384 + row];
      };
      if constexpr (PERSIST) exchange_l();
      mbar_wait(o_full, static_cast<uint32_t>(k) & 1u, ab);
      __syncwarp();
      tc_fence_after();
      if constexpr (!PERSIST) exchange_l();
      float coef = lam;
      if (EPI == kEpiV2) {
        const float lg = (t < p.n) ? p.lam_logits[c.b * p.sb + static_cast<long long>(t) * p.st + c.u] : 0.f;
        coef = 1.f / (1.f + expf(-lg));
      }
      if constexpr (STATS) {
        onepass_stats_epilogue<C, EPI>(p, c, t, row, lane, warp, cb, map, l1, l2, coef, m_used, tl, smem, sgamma);
        continue;
      }
      const float a1 = 1.f / l1, a2 = -coef / l2;
      float y[32];
      {
        uint32_t o1[32], o2[32];
        tmem_ld32(tl + C::TM_O1 + 32u * cb, o1);
        tmem_ld32(tl + C::TM_O2 + 32u * cb, o2);
        tmem_ld_wait2(o1, o2);
        if constexpr (PERSIST) {
          // O is in registers: the next item's first PV may overwrite it.
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(o_free);
          __syncwarp();
        }
        if constexpr (SAVE) {
          // Training forward: the row's normalised map outputs O_r = O_r' / l_r
          // (bf16, this warpgroup's 32 channels), packed and stored 8 channels
          // at a time alongside y, and, from the warpgroups that hold each
          // map's running maximum, lse_r = m_r + log2 l_r.  Saved layout:
          // [unit][128-row tile][channel block cb][row][32 channels], so the
          // warp's 32 rows of a block are 2 KB in a row.
          const bool live = t < p.n && DA_BOUNDS_V(c.b < p.B && c.u < p.units_per_batch, t);
          const long long blk =
              ((static_cast<long long>(c.b) * p.units_per_batch + c.u) * ((p.n + 127) / 128) + c.qt) * 4 + cb;
          const long long off = (blk * 128 + row) * 32;
          const float il2 = 1.f / l2;
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint32_t w1[4], w2[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int cc = 8 * v + 2 * e;
              const float x1a = __uint_as_float(o1[cc]) * a1, x1b = __uint_as_float(o1[cc + 1]) * a1;
              y[cc] = fmaf(__uint_as_float(o2[cc]), a2, x1a);
              y[cc + 1] = fmaf(__uint_as_float(o2[cc + 1]), a2, x1b);
              w1[e] = pack_bf16x2(x1a, x1b);
              w2[e] = pack_bf16x2(__uint_as_float(o2[cc]) * il2, __uint_as_float(o2[cc + 1]) * il2);
            }
            if (live) {
              reinterpret_cast<uint4*>(p.o1_save + off)[v] = make_uint4(w1[0], w1[1], w1[2], w1[3]);
              reinterpret_cast<uint4*>(p.o2_save + off)[v] = make_uint4(w2[0], w2[1], w2[2], w2[3]);
            }
          }
          if (live) {
            const long long ri = (static_cast<long long>(c.b) * p.units_per_batch + c.u) * p.n + t;
            if (cb == 0) p.row[ri] = m_used + log2f(l1);
            if (cb == 2) p.row[p.rows + ri] = m_used + log2f(l2);
          }
        } else {
#pragma unroll
          for (int cc = 0; cc < 32; ++cc) y[cc] = fmaf(__uint_as_float(o2[cc]), a2, __uint_as_float(o1[cc]) * a1);
        }
      }
      float rinv = 1.f;
      if (EPI == kEpiRmsNorm) {
        float ss0 = 0.f, ss1 = 0.f;
#pragma unroll
        for (int cc = 0; cc < 32; cc += 2) {
          ss0 = fmaf(y[cc], y[cc], ss0);
          ss1 = fmaf(y[cc + 1], y[cc + 1], ss1);
        }
        float* sp = sspart + (k & 1) * 512;
        sp[cb * 128 + row] = ss0 + ss1;
        __syncwarp();
        named_bar_sync(1, 128 * C::NSMWG);
        const float tot = (sp[row] + sp[128 + row]) + (sp[256 + row] + sp[384 + row]);
        rinv = p.norm_mult * rsqrtf(tot * (1.f / DV) + p.eps);
      }
      if constexpr (PERSIST) {
        // Row stores straight from registers: they drain while the next
        // item starts (staging them for a TMA store put a warpgroup barrier
        // and a proxy fence on the item transition, measured slower).
        if (t < p.n && DA_BOUNDS_V(c.b < p.B && c.u < p.units_per_batch, t)) {
          __nv_bfloat16* orow =
              p.out + ((static_cast<size_t>(c.b) * p.n + t) * p.units_per_batch + c.u) * DV + 32 * cb;
          uint32_t wv[16];
          pack_out_row<EPI == kEpiRmsNorm>(y, rinv, sgamma + 32 * cb, wv);
          uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
          for (int v = 0; v < 4; ++v) dst[v] = make_uint4(wv[4 * v], wv[4 * v + 1], wv[4 * v + 2], wv[4 * v + 3]);
        }
      } else {
        // One item per CTA: the warpgroup's 128 x 32 block goes through
        // shared memory (16-byte chunk v of row `row` at v ^ ((row / 2) % 4):
        // the 64-byte swizzle) and one TMA store, which drops rows past n
        // (row stores, one row per thread and 4 KB apart, queue up in the
        // load/store unit at the end of the CTA).  The staging is free: the
        // item's MMAs have completed (o_full) and no other item follows.
        uint32_t wv[16];
        pack_out_row<EPI == kEpiRmsNorm>(y, rinv, sgamma + 32 * cb, wv);
        uint8_t* const stg =
            smem + (PSM ? C::OFF_P + map * C::P_TILE + half * (BM * 128) : C::OFF_Q1 + cb * C::STG_BYTES);
        uint8_t* srow = stg + row * 64;
#pragma unroll
        for (int v = 0; v < 4; ++v)
          *reinterpret_cast<uint4*>(srow + ((v ^ ((row >> 1) & 3)) << 4)) =
              make_uint4(wv[4 * v], wv[4 * v + 1], wv[4 * v + 2], wv[4 * v + 3]);
        fence_proxy_async_smem();
        named_bar_sync(4 + cb, 128);
        if ((threadIdx.x & 127) == 96) {  // lane 0 of the warpgroup's first warp
          if (DA_BOUNDS(32 * cb < DV && c.u < p.units_per_batch && c.q0 < p.n && c.b < p.B))
            tma_store_4d(&p.tm_out, stg, 32 * cb, c.u, c.q0, c.b);
          bulk_commit_group();
        }
      }
      gt += static_cast<uint32_t>(T);
    }
  }

  // ---- teardown
  if (!PERSIST && warp >= C::NCTRL && (threadIdx.x & 127) == 96) bulk_wait_all();  // output store
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace da
