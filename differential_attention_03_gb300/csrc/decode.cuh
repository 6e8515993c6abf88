// One-token differential-attention decode over a key/value cache (CUDA
// cores, TMA, thread-block clusters with distributed shared memory; sm_103a).
//
// What it computes, per (batch b, head h), with L = lens[b] visible keys:
//   O_r = sum_{j < L} softmax_j(q_r . k_r[j] / sqrt d) v[j]          r = 1, 2
//   out = (1 - lambda_init) gamma (O_1 - lambda O_2) / sqrt(mean_c (O_1 - lambda O_2)^2 + eps)
// i.e. the DIFF V1 operator for the newest token of a causal sequence, whose
// keys and values sit in the cache ("Differential Transformer" glossary page,
// "How differential attention works"; news article section "差分注意力" for
// the per-head RMSNorm with the fixed (1 - lambda_init)).  L = 0 gives zeros.
// DIFF V2 (template flag V2; DIFF V2 analysis page, "2. 커스텀 커널 제거" and
// "GQA와의 호환성"): per (b, head pair g), query heads 2g and 2g + 1 over their
// shared KV head, out = O_1 - sigmoid(logit[b, g]) O_2, no norm; the key tile
// is then read once for both queries and V is d wide.
// Template flag K8: the key caches in FP8 (e4m3, one dequantisation scale per
// tensor, folded into the query), the values in bf16; 6 d bytes a key (V1)
// instead of 8 d.  The low-bit attention the glossary page's remark on
// smaller activation outliers points to, applied where the step is bound by
// the bytes it reads.
//
// The step is bound by HBM: every visible key's k_1, k_2 and v are read
// exactly once (V once for both maps), 8 d bytes per key, against ~12 d
// flops.  The design spends itself on bytes in flight on every SM, and on
// keeping the instructions a key costs low enough that issue never limits
// the stream:
//   * A cluster of CS CTAs per (b, h) (CS from 1 to 8, chosen by the host so
//     that the grid fills the GPU); CTA c streams keys [c C, c C + C) of
//     the cache (C a multiple of the stage size) through a ring of NST
//     stages filled by TMA (K_1, K_2 and V tiles of BK keys, 128-byte
//     swizzled rows; 32 KB a stage).
//   * Four warps per CTA, BK / 4 keys each per stage (16, or 8 at the
//     32-key stages of bf16 V1 d = 128).
//     A warp scores its keys with warp-wide MMAs (mma.sync: bf16 m16n8k16,
//     or e4m3 m16n8k32 for FP8 keys), transposed so that the keys are the
//     MMA's rows and the queries two of its eight columns: S^T = K [q_1 q_2].
//     Its online-softmax state per map (running maximum, row sums) is
//     rescaled only when the maximum grows, and the weights go back through
//     the tensor cores as O^T += V^T P^T (bf16 P, fp32 accumulation; V read
//     once for both maps by transposed ldmatrix loads).  Against scalar
//     FMAs this cuts the instructions a key costs about fourfold.  HBM stays
//     the bound (ncu: the tensor pipe active 17-27 % of the time, issue
//     22-34 %); instruction issue was the limit of the scalar form, measured
//     at 0.83-0.85 of the HBM copy with FP8 keys.
//   * The CTA merges its warps' states in shared memory; the cluster's CTAs
//     then merge theirs through distributed shared memory in CTA rank 0,
//     which applies the combine and the per-head RMSNorm and stores the row.
//     No global scratch.  With few (b, h) pairs the caller may pass a
//     workspace: then nsplit clusters share a pair's keys, rank 0 of each
//     writes the cluster's state there, and decode_combine_kernel merges the
//     nsplit states of a pair and finishes the row.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "params.h"
#include "ptx.cuh"

#undef DA_BOUNDS_FILE
#define DA_BOUNDS_FILE 5

namespace da {

struct DecodeParams {
  CUtensorMap tm_k1;  // V1: [B, n, H, d] key caches; V2: [B, n, Hkv, d]; boxes of 64 columns (K8: d bytes) x BK keys
  CUtensorMap tm_k2;  // (V1 only)
  CUtensorMap tm_v;   // V1: [B, n, H, 2d]; V2: [B, n, Hkv, d]
  const __nv_bfloat16* q1;  // V1: [B, H, d]; V2: q [B, Hq, d]
  const __nv_bfloat16* q2;  // V1: [B, H, d]; V2: unused
  const int* lens;          // [B] visible keys, or nullptr: n for every sequence
  const float* lambda;      // V1: device scalar
  const float* gamma;       // V1: [2d] or nullptr
  const float* lam_logits;  // V2: logit of pair g of sequence b at b * sb + g
  long long sb;
  __nv_bfloat16* out;       // V1: [B, H, 2d]; V2: [B, Hq / 2, d]
  float scale_log2;         // softmax scale * log2(e)
  float k1_scale, k2_scale; // K8: dequantisation scales of the e4m3 key caches (V2: k1_scale)
  float norm_mult;          // V1: 1 - lambda_init
  float eps;
  int B, H, n;  // H: V1 heads; V2 head pairs per sequence (Hq / 2)
  int group;    // V2: query heads per KV head
  int nsplit;   // clusters per (b, h); > 1: each writes its state to ws and a combine kernel finishes
  float* ws;    // [B * H][nsplit][2 (DV + 2)] partial states (nsplit > 1)
  int* status;
};

template <int D, bool V2 = false, bool K8 = false>
struct DecodeCfg {
  static constexpr int MAX_CS = 8;  // CTAs per (b, h) cluster: chosen at launch, at most this (16-CTA
                                    // clusters measured slower: 5.5 vs 6.2 TB/s at B8 H8 n32768 d128)
  // Warps per CTA: four.  A warp scores 16 keys of a stage (one MMA tile of rows); at the 32-key
  // stages of bf16 V1 d = 128 two warps share each 16 keys and split the value channels.
  static constexpr int NWARP = 4;
  static constexpr int NTHREADS = NWARP * 32;
  static constexpr int DV = V2 ? D : 2 * D;     // value width
  static constexpr int NKT = V2 ? 1 : 2;         // key tiles a stage holds (V2: one K for both queries)
  // Keys per stage: 64; bf16 V1 d = 128 (a 64 KB key row set) 32.  FP8 V1 d = 128 takes 64-key
  // stages of 48 KB in a two-stage ring: 1.00 of the HBM copy against 0.90 with 32-key stages of
  // 24 KB in four (B8 H8 n32768).
  static constexpr int BK = (V2 || D == 64 || K8) ? 64 : 32;
  static constexpr int WPG = NWARP / (BK / 16);  // warps per 16 keys (1, or 2 at d = 128), splitting the channels
  static constexpr int KS = K8 ? D / 32 : D / 16;  // MMA k-steps over the query/key width
  static constexpr int MT = (V2 ? D : 2 * D) / 16;  // 16-channel tiles of the value width
  static constexpr int KROW = K8 ? D : 128;  // bytes of a key row in one TMA box (bf16: 64 columns)
  static constexpr int QB = K8 ? 1 : D / 64;  // key boxes per row
  static constexpr int VB = DV / 64;
  static constexpr int K_BYTES = QB * BK * KROW, V_BYTES = VB * BK * 128;
  static constexpr int STAGE = NKT * K_BYTES + V_BYTES;  // 32 KB (K8: 24 KB; V1 K8 d = 128: 48 KB)
  static constexpr int NST = 98304 / STAGE;              // 96 KB of stages in flight
  static constexpr int PART_FLOATS = 2 * (DV + 2);  // per map: max, sum, DV channels
  static constexpr int OFF_BARS = NST * STAGE;
  static constexpr int OFF_FLAG = OFF_BARS + 2 * NST * 8;
  static constexpr int OFF_WARP = (OFF_FLAG + 16 + 15) / 16 * 16;  // float [NWARP][PART_FLOATS]
  static constexpr int OFF_PART = OFF_WARP + NWARP * PART_FLOATS * 4;  // float [PART_FLOATS]: the CTA's state
  static constexpr int OFF_RED = OFF_PART + PART_FLOATS * 4;           // float [NWARP]
  static constexpr int SMEM_BYTES = OFF_RED + NWARP * 4 + 1024;        // + 1 KB alignment slack
  static_assert(D == 64 || D == 128, "query/key width");
  static_assert(WPG >= 1 && WPG * (BK / 16) == NWARP && MT % WPG == 0, "warps tile the stage's keys and channels");
  static_assert(NST * STAGE == 98304, "stage ring");
  static_assert(STAGE % 1024 == 0 && K_BYTES % 1024 == 0, "swizzled boxes start on 1 KB");
  static_assert(!V2 || D == 128, "V2 decode: d = 128");
};

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Float at shared-memory address `a` of CTA `rank` of this cluster.
__device__ __forceinline__ float ld_cluster_f32(uint32_t a, uint32_t rank) {
  uint32_t ra;
  float v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
  return v;
}

// Warp-wide tensor-core operations of the decode loop (mma.sync: the step is bound by HBM, the
// MMAs only cut the instructions a key costs).  Fragment layouts are the PTX ISA's for
// m16n8k16 (bf16) and m16n8k32 (e4m3) with lane = 4 g + t: A rows g and g + 8, B column g,
// C rows g, g + 8 x columns 2 t, 2 t + 1.
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_e4m3_16832(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// One k-step of the score MMA: bf16 keys (16 dims) or e4m3 keys (32 dims).
template <bool K8>
__device__ __forceinline__ void mma_keys(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  if constexpr (K8)
    mma_e4m3_16832(c, a, b0, b1);
  else
    mma_bf16_16816(c, a, b0, b1);
}

// Two floats as bf16 (round to nearest even), lo in bits 0..15.
__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Finishes row (b, h) from its merged state (sums l1, l2; unnormalised
// outputs y1, y2 of this thread's channels threadIdx.x + t NTHREADS): the
// combine (V1: lambda, V2: sigmoid(logit)), V1's per-head RMSNorm, the store.
// Every thread of the CTA calls it (it holds a CTA barrier for V1).
template <int D, bool V2, int NTHREADS, int CPT>
__device__ __forceinline__ void decode_finish(const DecodeParams& p, int b, int h, float l1, float l2,
                                              const float (&y1)[CPT], const float (&y2)[CPT], float* red) {
  constexpr int DV = V2 ? D : 2 * D;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool has_ch = threadIdx.x < DV;
  const float coef = V2 ? 1.f / (1.f + expf(-p.lam_logits[b * p.sb + h])) : *p.lambda;
  const float a1 = (l1 > 0.f) ? 1.f / l1 : 0.f;
  const float a2 = (l2 > 0.f) ? -coef / l2 : 0.f;
  float y[CPT], ss = 0.f;
#pragma unroll
  for (int t = 0; t < CPT; ++t) {
    y[t] = has_ch ? fmaf(y2[t], a2, y1[t] * a1) : 0.f;
    ss = fmaf(y[t], y[t], ss);
  }
  float rinv = 1.f;
  if (!V2) {
#pragma unroll
    for (int x = 1; x < 32; x <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, x);
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < NTHREADS / 32; ++w) tot += red[w];
    rinv = p.norm_mult * rsqrtf(tot * (1.f / DV) + p.eps);
  }
  __nv_bfloat16* orow = p.out + (static_cast<size_t>(b) * p.H + h) * DV;
#pragma unroll
  for (int t = 0; t < CPT; ++t) {
    const int c = threadIdx.x + t * NTHREADS;
    if (!has_ch) break;
    const float g = (!V2 && p.gamma) ? p.gamma[c] : 1.f;
    if (DA_BOUNDS_V(b < p.B && h < p.H && c < DV, c)) orow[c] = __float2bfloat16_rn(y[t] * rinv * g);
  }
}

// Merges the nsplit cluster states of each (b, h) pair (one CTA per pair)
// written by decode_kernel into p.ws, and finishes the row.
template <int D, bool V2>
__global__ void __launch_bounds__(DecodeCfg<D, V2>::NTHREADS) decode_combine_kernel(const __grid_constant__ DecodeParams p) {
  using C = DecodeCfg<D, V2>;  // (the key type does not change the state layout)
  // Launched as a programmatic dependent of decode_kernel: its CTAs may be resident before that
  // grid ends; the states it reads are complete and visible after this wait.
  grid_dep_wait();
  constexpr int DV = C::DV;
  constexpr int CPT = DV > C::NTHREADS ? DV / C::NTHREADS : 1;
  __shared__ float red[C::NWARP];
  const int unit = blockIdx.x;
  const int b = unit / p.H, h = unit % p.H;
  const float* src = p.ws + static_cast<size_t>(unit) * p.nsplit * C::PART_FLOATS;
  float M1 = -INFINITY, M2 = -INFINITY;
  for (int r = 0; r < p.nsplit; ++r) {
    M1 = fmaxf(M1, src[r * C::PART_FLOATS]);
    M2 = fmaxf(M2, src[r * C::PART_FLOATS + 2]);
  }
  float l1 = 0.f, l2 = 0.f, y1[CPT], y2[CPT];
#pragma unroll
  for (int t = 0; t < CPT; ++t) y1[t] = y2[t] = 0.f;
  for (int r = 0; r < p.nsplit; ++r) {
    const float* sr = src + r * C::PART_FLOATS;
    const float f1 = (sr[0] == -INFINITY) ? 0.f : ex2(sr[0] - M1);
    const float f2 = (sr[2] == -INFINITY) ? 0.f : ex2(sr[2] - M2);
    l1 = fmaf(sr[1], f1, l1);
    l2 = fmaf(sr[3], f2, l2);
#pragma unroll
    for (int t = 0; t < CPT; ++t) {
      const int c = threadIdx.x + t * C::NTHREADS;
      if (c >= DV) break;
      y1[t] = fmaf(sr[4 + c], f1, y1[t]);
      y2[t] = fmaf(sr[4 + DV + c], f2, y2[t]);
    }
  }
  decode_finish<D, V2, C::NTHREADS, CPT>(p, b, h, l1, l2, y1, y2, red);
}

template <int D, bool V2, bool K8>
__global__ void __launch_bounds__(DecodeCfg<D, V2, K8>::NTHREADS, 2)
    decode_kernel(const __grid_constant__ DecodeParams p) {
  using C = DecodeCfg<D, V2, K8>;
  // Launched as a programmatic dependent of whatever kernel precedes it on the stream (which may
  // write the queries, the cache, the lengths or the output): nothing global is touched before
  // this wait, so only the launch overlaps that kernel's end.  The next dependent (the combine
  // kernel of the split form, or the next call's decode) may be scheduled now.
  grid_dep_launch_dependents();
  grid_dep_wait();
  constexpr int BK = C::BK, DV = C::DV, NST = C::NST;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BARS);
  uint64_t* empty = full + NST;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_FLAG);
  float* wpart = reinterpret_cast<float*>(smem + C::OFF_WARP);
  float* part = reinterpret_cast<float*>(smem + C::OFF_PART);
  float* red = reinterpret_cast<float*>(smem + C::OFF_RED);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t cs = cluster_nctarank();
  const int cluster = static_cast<int>(blockIdx.x / cs);
  const int unit = cluster / p.nsplit;  // (b, h), V2: (b, pair)
  const int split = cluster % p.nsplit;  // which share of the pair's keys this cluster takes
  const uint32_t rank = cluster_ctarank();
  const int b = unit / p.H, h = unit % p.H;
  // Heads: V1 head h for everything; V2 query heads 2h, 2h + 1 over KV head 2h / group.
  const int hk = V2 ? (2 * h) / p.group : h;
  const size_t q1_off = V2 ? (static_cast<size_t>(b) * 2 * p.H + 2 * h) * D : (static_cast<size_t>(b) * p.H + h) * D;
  const size_t q2_off = V2 ? q1_off + D : q1_off;
  int L = p.lens ? p.lens[b] : p.n;
  L = max(0, min(L, p.n));
  // This CTA's keys: [k_begin, k_end), a multiple of BK long except at L.
  const int nct = static_cast<int>(cs) * p.nsplit;  // CTAs sharing the pair's keys
  const int chunk = ((L + nct * BK - 1) / (nct * BK)) * BK;
  const int k_begin = min(L, (split * static_cast<int>(cs) + static_cast<int>(rank)) * chunk);
  const int k_end = min(L, k_begin + chunk);
  const int nblk = (k_end - k_begin + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], C::NWARP);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const AbortState ab{abort_flag, p.status};

  auto issue = [&](int i) {  // block i of this CTA into stage i % NST
    uint8_t* st = smem + (i % NST) * C::STAGE;
    const int key0 = k_begin + i * BK;
    mbar_arrive_expect_tx(&full[i % NST], C::STAGE);
    // (bounds build: KV heads V1 H, V2 2 H / group; the block starts inside the cache)
    if (!DA_BOUNDS_V(key0 < p.n && b < p.B && hk < (V2 ? 2 * p.H / p.group : p.H), key0)) return;
    for (int bx = 0; bx < C::QB; ++bx) {  // (K8: one box of D bytes a row)
      tma_load_4d(st + bx * BK * C::KROW, &p.tm_k1, &full[i % NST], bx * 64, hk, key0, b);
      if (!V2) tma_load_4d(st + C::K_BYTES + bx * BK * C::KROW, &p.tm_k2, &full[i % NST], bx * 64, hk, key0, b);
    }
    for (int bx = 0; bx < C::VB; ++bx)
      tma_load_4d(st + C::NKT * C::K_BYTES + bx * BK * 128, &p.tm_v, &full[i % NST], bx * 64, hk, key0, b);
  };
  int issued = 0;
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&p.tm_k1);
    tma_prefetch_desc(&p.tm_k2);
    tma_prefetch_desc(&p.tm_v);
    for (; issued < NST && issued < nblk; ++issued) issue(issued);
  }

  // ---- the operands that stay in registers: the queries as the B operand of the score MMAs.
  // Scores are computed transposed, S^T = K Q (16 keys x 8 columns per warp-wide MMA): column 0
  // collects map 1 (the K_1 MMA sees q_1 there and zeros elsewhere), column 1 map 2 (the K_2 MMA
  // sees q_2 there), so both maps land in one accumulator.  Lane (g, t) = (lane / 4, lane % 4)
  // holds column g of the B fragments.
  constexpr int KS = C::KS, WPG = C::WPG, MTW = C::MT / WPG;
  const int g = lane >> 2, tq = lane & 3;
  constexpr int NT = K8 ? 2 : 1;      // query terms (e4m3: hi and lo)
  uint32_t qa[NT][KS][2], qb[NT][KS][2];  // B fragments of the K_1 (V2: the shared K) and K_2 MMAs
  float qs1, qs2;                 // what turns column 0 / 1 of S^T into log2-domain scores
  if constexpr (!K8) {
    // bf16 queries as they are (m16n8k16: rows 2t, 2t + 1 and 2t + 8, 2t + 9 of column g).
    const uint32_t* w1 = reinterpret_cast<const uint32_t*>(p.q1 + q1_off);
    const uint32_t* w2 = reinterpret_cast<const uint32_t*>((V2 ? p.q1 : p.q2) + q2_off);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int w = 8 * ks + tq + 4 * j;  // 32-bit word: dims 16 ks + 8 j + 2 t, + 1
        const uint32_t a = w1[w], c = w2[w];
        qa[0][ks][j] = (g == 0) ? a : ((V2 && g == 1) ? c : 0u);
        qb[0][ks][j] = (!V2 && g == 1) ? c : 0u;
      }
    }
    qs1 = qs2 = p.scale_log2;
  } else {
    // e4m3 keys meet e4m3 queries (m16n8k32).  Each query row is scaled by a power of two that
    // puts its largest magnitude in [128, 256) and split into two e4m3 terms, hi = e4m3(x) and
    // lo = e4m3(x - hi): a bf16 value has eight significant bits and each term holds four, so
    // the pair is exact for every element down to 2^-10 of the row's largest (smaller ones
    // keep an absolute error below 2^-18 of it).  The two terms are two MMAs into the same
    // column: V1 q_1 in column 0 (the K_1 MMAs), q_2 in column 1 (the K_2 MMAs); V2 q_even in 0,
    // q_odd in 1.  Lane (g, t) holds dims 32 ks + 4 t .. + 3 and 32 ks + 16 + 4 t .. + 3 of
    // column g's row.
    const __nv_bfloat16* qv = (g & 1) ? ((V2 ? p.q1 : p.q2) + q2_off) : (p.q1 + q1_off);
    float x[KS][8];
    float amax = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const uint2 w = *reinterpret_cast<const uint2*>(qv + 32 * ks + 16 * j + 4 * tq);
        x[ks][4 * j] = bf16_lo(w.x);
        x[ks][4 * j + 1] = bf16_hi(w.x);
        x[ks][4 * j + 2] = bf16_lo(w.y);
        x[ks][4 * j + 3] = bf16_hi(w.y);
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(x[ks][e]));
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));  // the four lanes of a column hold its row
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const int bexp = (__float_as_int(amax) >> 23) & 0xff;  // amax in [2^(bexp - 127), 2^(bexp - 126))
    const int sh = (amax > 0.f) ? max(-100, min(100, 134 - bexp)) : 0;
    const float mul = __int_as_float((127 + sh) << 23), inv = __int_as_float((127 - sh) << 23);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        uint32_t whi = 0, wlo = 0;
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const float v0 = x[ks][4 * j + 2 * h2] * mul, v1 = x[ks][4 * j + 2 * h2 + 1] * mul;
          const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(make_float2(v0, v1), __NV_SATFINITE, __NV_E4M3);
          const float2 hf = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(hi, __NV_E4M3)));
          const __nv_fp8x2_storage_t lo =
              __nv_cvt_float2_to_fp8x2(make_float2(v0 - hf.x, v1 - hf.y), __NV_SATFINITE, __NV_E4M3);
          whi |= static_cast<uint32_t>(hi) << (16 * h2);
          wlo |= static_cast<uint32_t>(lo) << (16 * h2);
        }
        const bool in_a = V2 ? (g < 2) : (g == 0), in_b = !V2 && g == 1;
        qa[0][ks][j] = in_a ? whi : 0u;
        qa[NT - 1][ks][j] = in_a ? wlo : 0u;
        qb[0][ks][j] = in_b ? whi : 0u;
        qb[NT - 1][ks][j] = in_b ? wlo : 0u;
      }
    }
    // Column 0's row scale is lane 0's, column 1's lane 4's.
    qs1 = p.scale_log2 * p.k1_scale * __shfl_sync(0xffffffffu, inv, 0);
    qs2 = p.scale_log2 * (V2 ? p.k1_scale : p.k2_scale) * __shfl_sync(0xffffffffu, inv, 4);
  }

  // ---- the warp's 16 keys kb .. kb + 15 of every stage and its MTW 16-channel tiles from mt0;
  // ldmatrix rows of this lane (matrix mi = lane / 8, row mr = lane % 8): the score MMA's A = K
  // (keys x dims) takes keys + 8 for matrices 1 and 3, the P.V MMA's A = V^T (channels x keys, a
  // transposed load) keys + 8 for matrices 2 and 3.  (kb + 15 < BK: the warps tile the stage.)
  const int mi = lane >> 3, mr = lane & 7;
  const int kb = (warp / WPG) * 16, mt0 = (warp % WPG) * MTW;
  const int s_row = kb + mr + (mi & 1) * 8;
  const int v_row = kb + mr + (mi >> 1) * 8;

  constexpr float kRescaleLog2 = 8.f;  // how far a score may exceed the reference maximum
  float m1 = -INFINITY, m2 = -INFINITY, ls1 = 0.f, ls2 = 0.f;
  float o[MTW][4];  // O^T tiles: lanes t = 0 hold channel 16 (mt0 + mt) + g (+ 8) of map 1 ([0], [2]) and map 2 ([1], [3])
#pragma unroll
  for (int mt = 0; mt < MTW; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

  for (int i = 0; i < nblk; ++i) {
    const int s = i % NST;
    if (!mbar_wait(&full[s], static_cast<uint32_t>(i / NST) & 1u, ab)) break;
    const uint32_t st = smem_u32(smem + s * C::STAGE);
    // ---- scores S^T of the warp's 16 key rows (fp32 accumulation on the tensor cores), in four
    // independent accumulator chains: V1 (map, parity of the MMA), V2 the MMA's index % 4
    float acc[4][4];
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[c][0] = acc[c][1] = acc[c][2] = acc[c][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const int ch = 2 * ks + (mi >> 1);  // 16-byte chunk of the key row
      uint32_t off;
      if constexpr (K8)  // rows of D bytes: 128-byte swizzle (chunk ^ row % 8) or 64-byte (chunk ^ (row / 2) % 4)
        off = s_row * C::KROW + (((C::KROW == 128) ? (ch ^ (s_row & 7)) : (ch ^ ((s_row >> 1) & 3))) << 4);
      else  // boxes of 64 bf16 columns, 128-byte rows, 128-byte swizzle
        off = (ch >> 3) * BK * 128 + s_row * 128 + (((ch & 7) ^ (s_row & 7)) << 4);
      uint32_t a[4];
      ldsm_x4(a, st + off);
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const int u = ks * NT + t;
        mma_keys<K8>(acc[V2 ? (u & 3) : (u & 1)], a, qa[t][ks][0], qa[t][ks][1]);
      }
      if constexpr (!V2) {
        ldsm_x4(a, st + C::K_BYTES + off);
#pragma unroll
        for (int t = 0; t < NT; ++t) mma_keys<K8>(acc[2 + ((ks * NT + t) & 1)], a, qb[t][ks][0], qb[t][ks][1]);
      }
    }
    float sc[4];  // columns 0 (map 1) and 1 (map 2) of rows g ([0], [1]) and g + 8 ([2], [3])
    if constexpr (V2) {
#pragma unroll
      for (int j = 0; j < 4; ++j) sc[j] = (acc[0][j] + acc[1][j]) + (acc[2][j] + acc[3][j]);
    } else {
      sc[0] = acc[0][0] + acc[1][0];
      sc[1] = acc[2][1] + acc[3][1];
      sc[2] = acc[0][2] + acc[1][2];
      sc[3] = acc[2][3] + acc[3][3];
    }
    // Lanes t = 0 now hold key kb + g ([0] map 1, [1] map 2) and key kb + g + 8 ([2], [3]).
    const int key = k_begin + i * BK + kb + g;
    float s1a = sc[0] * qs1, s2a = sc[1] * qs2, s1b = sc[2] * qs1, s2b = sc[3] * qs2;
    if (key >= k_end) s1a = s2a = -INFINITY;  // past this CTA's keys or the length
    if (key + 8 >= k_end) s1b = s2b = -INFINITY;
    // ---- online softmax of the warp's keys.  The reference maxima m1, m2 move only when a score
    // exceeds them by more than 2^8 (log2 domain: weights up to 256, safe in bf16 and in the fp32
    // sums), found by one vote; only then is the tile maximum reduced over lanes t = 0 and
    // broadcast, so the rescale branches stay uniform across the warp.
    float x1 = fmaxf(s1a, s1b), x2 = fmaxf(s2a, s2b);
    if (__any_sync(0xffffffffu, tq == 0 && (x1 > m1 + kRescaleLog2 || x2 > m2 + kRescaleLog2))) {
#pragma unroll
      for (int x = 4; x < 32; x <<= 1) {
        x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, x));
        x2 = fmaxf(x2, __shfl_xor_sync(0xffffffffu, x2, x));
      }
      x1 = __shfl_sync(0xffffffffu, x1, 0);
      x2 = __shfl_sync(0xffffffffu, x2, 0);
    } else {
      x1 = m1;
      x2 = m2;
    }
    if (x1 > m1) {
      const float f = (m1 == -INFINITY) ? 0.f : ex2(m1 - x1);
      m1 = x1;
      ls1 *= f;
#pragma unroll
      for (int mt = 0; mt < MTW; ++mt) {
        o[mt][0] *= f;
        o[mt][2] *= f;
      }
    }
    if (x2 > m2) {
      const float f = (m2 == -INFINITY) ? 0.f : ex2(m2 - x2);
      m2 = x2;
      ls2 *= f;
#pragma unroll
      for (int mt = 0; mt < MTW; ++mt) {
        o[mt][1] *= f;
        o[mt][3] *= f;
      }
    }
    const float p1a = (s1a == -INFINITY) ? 0.f : ex2(s1a - m1), p1b = (s1b == -INFINITY) ? 0.f : ex2(s1b - m1);
    const float p2a = (s2a == -INFINITY) ? 0.f : ex2(s2a - m2), p2b = (s2b == -INFINITY) ? 0.f : ex2(s2b - m2);
    ls1 += p1a + p1b;  // (meaningful in lanes t = 0)
    ls2 += p2a + p2b;
    // ---- P^T as the B operand (keys x columns; column 0 map 1, column 1 map 2) in bf16: lane
    // (g, t) needs keys 2t, 2t + 1 (b0) and 2t + 8, 2t + 9 (b1) of its column, held by lanes 8t
    // and 8t + 4 as (key, key + 8) pairs.
    uint32_t b0, b1;
    {
      const uint32_t u = bf16x2_bits(p1a, p1b), w = bf16x2_bits(p2a, p2b);
      const uint32_t ua = __shfl_sync(0xffffffffu, u, 8 * tq), ub = __shfl_sync(0xffffffffu, u, 8 * tq + 4);
      const uint32_t wa = __shfl_sync(0xffffffffu, w, 8 * tq), wb = __shfl_sync(0xffffffffu, w, 8 * tq + 4);
      const uint32_t xa = (g == 1) ? wa : ua, xb = (g == 1) ? wb : ub;
      b0 = __byte_perm(xa, xb, 0x5410);
      b1 = __byte_perm(xa, xb, 0x7632);
    }
    // ---- O^T += V^T P^T over the warp's keys, 16 channels a tile
#pragma unroll
    for (int mt = 0; mt < MTW; ++mt) {
      const int ch = 2 * (mt0 + mt) + (mi & 1);  // 16-byte chunk (8 channels) of the value row
      const uint32_t off = C::NKT * C::K_BYTES + (ch >> 3) * BK * 128 + v_row * 128 + (((ch & 7) ^ (v_row & 7)) << 4);
      uint32_t a[4];
      ldsm_x4_trans(a, st + off);
      mma_bf16_16816(o[mt], a, b0, b1);
    }
    // ---- release the stage; thread 0 refills it once all the warps have
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    if (threadIdx.x == 0 && issued < nblk) {
      if (!mbar_wait(&empty[s], static_cast<uint32_t>(i / NST) & 1u, ab)) break;
      issue(issued);
      ++issued;
    }
  }
  if (threadIdx.x == 0 && *ab.flag) {
    // Aborted: let the copies already issued land before the CTA exits.
    for (int f = (issued > NST ? issued - NST : 0); f < issued; ++f)
      mbar_wait_drain(&full[f % NST], static_cast<uint32_t>(f / NST) & 1u, kWaitBudgetCycles);
  }

  // ---- merge the warps' states (shared memory), then the cluster's (rank 0)
#pragma unroll
  for (int x = 4; x < 32; x <<= 1) {  // row sums over lanes t = 0
    ls1 += __shfl_xor_sync(0xffffffffu, ls1, x);
    ls2 += __shfl_xor_sync(0xffffffffu, ls2, x);
  }
  float* wp = wpart + warp * C::PART_FLOATS;  // [m1, l1, m2, l2, o1[DV], o2[DV]]
  // (Warps that share keys have the same maxima and sums: the first of them reports the sums, and
  // each reports zeros for the channels the others hold.)
  if (lane == 0) {
    wp[0] = m1;
    wp[1] = (warp % WPG == 0) ? ls1 : 0.f;
    wp[2] = m2;
    wp[3] = (warp % WPG == 0) ? ls2 : 0.f;
  }
  if (tq == 0) {
#pragma unroll
    for (int mt = 0; mt < MTW; ++mt) {
      const int c0 = 16 * (mt0 + mt) + g;
      wp[4 + c0] = o[mt][0];
      wp[4 + c0 + 8] = o[mt][2];
      wp[4 + DV + c0] = o[mt][1];
      wp[4 + DV + c0 + 8] = o[mt][3];
    }
  }
  if constexpr (WPG > 1) {
    for (int c = lane; c < DV; c += 32) {
      if (c / (16 * MTW) == warp % WPG) continue;
      wp[4 + c] = 0.f;
      wp[4 + DV + c] = 0.f;
    }
  }
  __syncthreads();
  {
    float M1 = -INFINITY, M2 = -INFINITY;
    float fa[C::NWARP], fb[C::NWARP];
#pragma unroll
    for (int w = 0; w < C::NWARP; ++w) {
      M1 = fmaxf(M1, wpart[w * C::PART_FLOATS]);
      M2 = fmaxf(M2, wpart[w * C::PART_FLOATS + 2]);
    }
#pragma unroll
    for (int w = 0; w < C::NWARP; ++w) {
      const float mw1 = wpart[w * C::PART_FLOATS], mw2 = wpart[w * C::PART_FLOATS + 2];
      fa[w] = (mw1 == -INFINITY) ? 0.f : ex2(mw1 - M1);
      fb[w] = (mw2 == -INFINITY) ? 0.f : ex2(mw2 - M2);
    }
    for (int c = threadIdx.x; c < DV; c += C::NTHREADS) {
      float a = 0.f, e = 0.f;
#pragma unroll
      for (int w = 0; w < C::NWARP; ++w) {
        a = fmaf(wpart[w * C::PART_FLOATS + 4 + c], fa[w], a);
        e = fmaf(wpart[w * C::PART_FLOATS + 4 + DV + c], fb[w], e);
      }
      part[4 + c] = a;
      part[4 + DV + c] = e;
    }
    if (threadIdx.x == 0) {
      float l1 = 0.f, l2 = 0.f;
#pragma unroll
      for (int w = 0; w < C::NWARP; ++w) {
        l1 = fmaf(wpart[w * C::PART_FLOATS + 1], fa[w], l1);
        l2 = fmaf(wpart[w * C::PART_FLOATS + 3], fb[w], l2);
      }
      part[0] = M1;
      part[1] = l1;
      part[2] = M2;
      part[3] = l2;
    }
  }
  cluster_sync_all();  // every CTA's state is written (release / acquire across the cluster)

  if (rank == 0) {
    const uint32_t pa = smem_u32(part);
    float M1 = -INFINITY, M2 = -INFINITY;
    for (uint32_t r = 0; r < cs; ++r) {
      M1 = fmaxf(M1, ld_cluster_f32(pa, r));
      M2 = fmaxf(M2, ld_cluster_f32(pa + 8, r));
    }
    float l1 = 0.f, l2 = 0.f;
    constexpr int CPT = DV > C::NTHREADS ? DV / C::NTHREADS : 1;  // channels per thread: 1 or 2
    const bool has_ch = threadIdx.x < DV;                           // (V2: 128 channels, 256 threads)
    float y1[CPT], y2[CPT];
#pragma unroll
    for (int t = 0; t < CPT; ++t) y1[t] = y2[t] = 0.f;
    for (uint32_t r = 0; r < cs; ++r) {
      const float mr1 = ld_cluster_f32(pa, r), mr2 = ld_cluster_f32(pa + 8, r);
      const float f1 = (mr1 == -INFINITY) ? 0.f : ex2(mr1 - M1);
      const float f2 = (mr2 == -INFINITY) ? 0.f : ex2(mr2 - M2);
      l1 = fmaf(ld_cluster_f32(pa + 4, r), f1, l1);
      l2 = fmaf(ld_cluster_f32(pa + 12, r), f2, l2);
#pragma unroll
      for (int t = 0; t < CPT; ++t) {
        const int c = threadIdx.x + t * C::NTHREADS;
        if (!has_ch) break;
        y1[t] = fmaf(ld_cluster_f32(pa + 4 * (4 + c), r), f1, y1[t]);
        y2[t] = fmaf(ld_cluster_f32(pa + 4 * (4 + DV + c), r), f2, y2[t]);
      }
    }
    if (p.nsplit > 1) {
      // This cluster's state of the pair: the combine kernel finishes the row.
      float* dst = p.ws + (static_cast<size_t>(unit) * p.nsplit + split) * C::PART_FLOATS;
      if (!DA_BOUNDS_V(unit < p.B * p.H && split < p.nsplit, unit)) dst = nullptr;
      if (dst == nullptr) {
      } else if (threadIdx.x == 0) {
        dst[0] = M1;
        dst[1] = l1;
        dst[2] = M2;
        dst[3] = l2;
      }
#pragma unroll
      for (int t = 0; t < CPT; ++t) {
        const int c = threadIdx.x + t * C::NTHREADS;
        if (!has_ch || dst == nullptr) break;
        dst[4 + c] = y1[t];
        dst[4 + DV + c] = y2[t];
      }
    } else {
      decode_finish<D, V2, C::NTHREADS, CPT>(p, b, h, l1, l2, y1, y2, red);
    }
  }
  cluster_sync_all();  // rank 0 has read every CTA's state: they may exit
}

}  // namespace da
