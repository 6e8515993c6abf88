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
// flops.  So no tensor cores: the work is spread so that enough bytes are in
// flight on every SM.
//   * A cluster of CS CTAs per (b, h) (CS from 1 to 8, chosen by the host so
//     that the grid fills the GPU); CTA c streams keys [c C, c C + C) of
//     the cache (C a multiple of the stage size) through a ring of NST
//     stages filled by TMA (K_1, K_2 and V tiles of BK keys, 128-byte
//     swizzled rows; 32 KB a stage).
//   * NWARP warps per CTA (four; eight for V2 and for FP8 keys), BK / NWARP
//     keys each per stage; PARTS lanes share a key (PE = 32 or 16 products of
//     q . k each, combined by shuffles), so a warp scores its
//     keys in one pass; every warp keeps its own online-softmax state per map
//     (running maximum, per-lane partial sums, 2d / 32 output channels per
//     lane for each map), rescaled only when the maximum grows.  Products
//     and value accumulations run as packed f32x2 FMAs (two lanes of fp32
//     arithmetic per instruction), which halves the instructions a key costs.
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
  // Warps per CTA.  V2: eight, so that a stage is 64 keys (32 KB).  V1 with
  // FP8 keys at d = 64: eight (PE = 16 products a lane), so that two CTAs per
  // SM hide the latency of the longer per-byte instruction stream (a key is
  // 6 d bytes instead of 8 d for the same work).  At d = 128 (32-key stages)
  // eight warps would leave 4 keys a warp and 8 lanes a key: measured at half
  // the bandwidth of four warps, so V1 d = 128 keeps four.
  static constexpr int NWARP = (V2 || (K8 && D == 64)) ? 8 : 4;
  static constexpr int NTHREADS = NWARP * 32;
  static constexpr int DV = V2 ? D : 2 * D;     // value width
  static constexpr int NKT = V2 ? 1 : 2;         // key tiles a stage holds (V2: one K for both queries)
  static constexpr int BK = (V2 || D == 64) ? 64 : 32;  // keys per stage
  static constexpr int KW = BK / NWARP;         // keys per warp per stage
  static constexpr int PARTS = 32 / KW;         // lanes per key
  static constexpr int PE = D / PARTS;          // q . k products per lane (32, or 16 with FP8 keys in V1)
  static constexpr int KROW = K8 ? D : 128;  // bytes of a key row in one TMA box (bf16: 64 columns)
  static constexpr int QB = K8 ? 1 : D / 64;  // key boxes per row
  static constexpr int VB = DV / 64;
  static constexpr int K_BYTES = QB * BK * KROW, V_BYTES = VB * BK * 128;
  static constexpr int STAGE = NKT * K_BYTES + V_BYTES;  // 32 KB (K8: 24 KB)
  static constexpr int NST = 98304 / STAGE;              // 96 KB of stages in flight
  static constexpr int CH = DV / 32;  // output channels per lane and map
  static constexpr int PART_FLOATS = 2 * (DV + 2);  // per map: max, sum, DV channels
  static constexpr int OFF_BARS = NST * STAGE;
  static constexpr int OFF_FLAG = OFF_BARS + 2 * NST * 8;
  static constexpr int OFF_WARP = (OFF_FLAG + 16 + 15) / 16 * 16;  // float [NWARP][PART_FLOATS]
  static constexpr int OFF_PART = OFF_WARP + NWARP * PART_FLOATS * 4;  // float [PART_FLOATS]: the CTA's state
  static constexpr int OFF_RED = OFF_PART + PART_FLOATS * 4;           // float [NWARP]
  static constexpr int SMEM_BYTES = OFF_RED + NWARP * 4 + 1024;        // + 1 KB alignment slack
  static_assert(D == 64 || D == 128, "query/key width");
  static_assert((PE == 32 || PE == 16) && PARTS * KW == 32, "lane split");
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

// Four e4m3 values (bytes 0..3 of w, byte 0 first) to floats; exact (every
// e4m3 value is an f16 value).
__device__ __forceinline__ void e4m3x4_to_f32(uint32_t w, float (&f)[4]) {
  uint32_t h01, h23;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, lo;\n\tcvt.rn.f16x2.e4m3x2 %1, hi;\n\t}"
      : "=r"(h01), "=r"(h23)
      : "r"(w));
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&h01));
  const float2 c = __half22float2(*reinterpret_cast<const __half2*>(&h23));
  f[0] = a.x;
  f[1] = a.y;
  f[2] = c.x;
  f[3] = c.y;
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
  constexpr int BK = C::BK, KW = C::KW, PARTS = C::PARTS, DV = C::DV, CH = C::CH, NST = C::NST;
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

  // This lane's PE query products (pre-scaled into the log2 domain, and by
  // the key scale of an e4m3 key cache).
  constexpr int PE = C::PE;
  const int kk = lane / PARTS, prt = lane % PARTS;
  const float qs1 = K8 ? p.scale_log2 * p.k1_scale : p.scale_log2;
  const float qs2 = K8 ? p.scale_log2 * (V2 ? p.k1_scale : p.k2_scale) : p.scale_log2;
  uint64_t q1r[PE / 2], q2r[PE / 2];  // pairs of query products
  {
    const __nv_bfloat16* q1p = p.q1 + q1_off + prt * PE;
    const __nv_bfloat16* q2p = (V2 ? p.q1 : p.q2) + q2_off + prt * PE;
#pragma unroll
    for (int i = 0; i < PE; i += 8) {
      const uint4 a = *reinterpret_cast<const uint4*>(q1p + i);
      const uint4 c = *reinterpret_cast<const uint4*>(q2p + i);
      const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wc[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        q1r[i / 2 + e] = f2pack(bf16_lo(wa[e]) * qs1, bf16_hi(wa[e]) * qs1);
        q2r[i / 2 + e] = f2pack(bf16_lo(wc[e]) * qs2, bf16_hi(wc[e]) * qs2);
      }
    }
  }

  float m1 = -INFINITY, m2 = -INFINITY, ls1 = 0.f, ls2 = 0.f;
  uint64_t o1p[CH / 2], o2p[CH / 2];
#pragma unroll
  for (int c = 0; c < CH / 2; ++c) o1p[c] = o2p[c] = 0ull;
  // Byte offsets inside a stage that do not change: this lane's PE key
  // columns (box, first 16-byte chunk) and its CH value channels.
  const int kbox = (prt * PE) / 64, kchunk0 = ((prt * PE) % 64) / 8;
  const int vc0 = lane * CH, vbox = vc0 / 64, vbyte = (vc0 % 64) * 2;

  for (int i = 0; i < nblk; ++i) {
    const int s = i % NST;
    if (!mbar_wait(&full[s], static_cast<uint32_t>(i / NST) & 1u, ab)) break;
    const uint8_t* st = smem + s * C::STAGE;
    const int row = warp * KW + kk;  // this lane's key within the stage
    // ---- scores: PE products per lane, PARTS lanes per key
    uint64_t a1 = 0ull, a2 = 0ull, b1 = 0ull, b2 = 0ull;
    if constexpr (K8) {
      // PE e4m3 key values: 16-byte chunks (PE / 16) prt .. of the row
      // (128-byte rows: 128-byte swizzle, chunk ^ (row % 8); 64-byte rows:
      // 64-byte swizzle, chunk ^ ((row / 2) % 4)).
#pragma unroll
      for (int c = 0; c < PE / 16; ++c) {
        const int ch = (PE / 16) * prt + c;
        const int pch = (C::KROW == 128) ? (ch ^ (row & 7)) : (ch ^ ((row >> 1) & 3));
        const int off = row * C::KROW + (pch << 4);
        const uint4 a = *reinterpret_cast<const uint4*>(st + off);
        const uint4 e = V2 ? a : *reinterpret_cast<const uint4*>(st + C::K_BYTES + off);  // V2: one key tile
        const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, we[4] = {e.x, e.y, e.z, e.w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          float fa[4], fe[4];
          e4m3x4_to_f32(wa[t], fa);
          e4m3x4_to_f32(we[t], fe);
          a1 = fma2(q1r[8 * c + 2 * t], f2pack(fa[0], fa[1]), a1);
          b1 = fma2(q1r[8 * c + 2 * t + 1], f2pack(fa[2], fa[3]), b1);
          a2 = fma2(q2r[8 * c + 2 * t], f2pack(fe[0], fe[1]), a2);
          b2 = fma2(q2r[8 * c + 2 * t + 1], f2pack(fe[2], fe[3]), b2);
        }
      }
    } else {
#pragma unroll
      for (int c = 0; c < PE / 8; ++c) {
        const int off = kbox * BK * 128 + row * 128 + (((kchunk0 + c) ^ (row & 7)) << 4);
        const uint4 a = *reinterpret_cast<const uint4*>(st + off);
        const uint4 e = V2 ? a : *reinterpret_cast<const uint4*>(st + C::K_BYTES + off);  // V2: one key tile
        const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, we[4] = {e.x, e.y, e.z, e.w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          if (t & 1) {
            b1 = fma2(q1r[4 * c + t], f2pack(bf16_lo(wa[t]), bf16_hi(wa[t])), b1);
            b2 = fma2(q2r[4 * c + t], f2pack(bf16_lo(we[t]), bf16_hi(we[t])), b2);
          } else {
            a1 = fma2(q1r[4 * c + t], f2pack(bf16_lo(wa[t]), bf16_hi(wa[t])), a1);
            a2 = fma2(q2r[4 * c + t], f2pack(bf16_lo(we[t]), bf16_hi(we[t])), a2);
          }
        }
      }
    }
    float s1, s2;
    {
      const uint64_t t1 = add2(a1, b1), t2 = add2(a2, b2);
      float l, h;
      f2unpack(t1, l, h);
      s1 = l + h;
      f2unpack(t2, l, h);
      s2 = l + h;
    }
#pragma unroll
    for (int x = 1; x < PARTS; x <<= 1) {
      s1 += __shfl_xor_sync(0xffffffffu, s1, x);
      s2 += __shfl_xor_sync(0xffffffffu, s2, x);
    }
    if (k_begin + i * BK + row >= k_end) s1 = s2 = -INFINITY;  // past this CTA's keys or the length
    // ---- online softmax of this warp's keys
    float x1 = s1, x2 = s2;
#pragma unroll
    for (int x = PARTS; x < 32; x <<= 1) {
      x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, x));
      x2 = fmaxf(x2, __shfl_xor_sync(0xffffffffu, x2, x));
    }
    if (x1 > m1) {
      const float f = (m1 == -INFINITY) ? 0.f : ex2(m1 - x1);
      m1 = x1;
      ls1 *= f;
#pragma unroll
      for (int c = 0; c < CH / 2; ++c) o1p[c] = fma2(o1p[c], f2pack(f, f), 0ull);
    }
    if (x2 > m2) {
      const float f = (m2 == -INFINITY) ? 0.f : ex2(m2 - x2);
      m2 = x2;
      ls2 *= f;
#pragma unroll
      for (int c = 0; c < CH / 2; ++c) o2p[c] = fma2(o2p[c], f2pack(f, f), 0ull);
    }
    const float p1 = (s1 == -INFINITY) ? 0.f : ex2(s1 - m1);
    const float p2 = (s2 == -INFINITY) ? 0.f : ex2(s2 - m2);
    if (prt == 0) {
      ls1 += p1;
      ls2 += p2;
    }
    // ---- P.V: every lane accumulates its CH channels over the warp's keys
    const uint8_t* vb = st + C::NKT * C::K_BYTES + vbox * BK * 128;
#pragma unroll
    for (int k2 = 0; k2 < KW; ++k2) {
      const float w1 = __shfl_sync(0xffffffffu, p1, k2 * PARTS);
      const float w2 = __shfl_sync(0xffffffffu, p2, k2 * PARTS);
      const int r = warp * KW + k2;
      const uint8_t* vr = vb + r * 128 + ((((vbyte >> 4)) ^ (r & 7)) << 4) + (vbyte & 15);
      uint32_t vw[CH / 2];
      if constexpr (CH == 4) {
        const uint2 t = *reinterpret_cast<const uint2*>(vr);
        vw[0] = t.x;
        vw[1] = t.y;
      } else {
        const uint4 t = *reinterpret_cast<const uint4*>(vr);
        vw[0] = t.x;
        vw[1] = t.y;
        vw[2] = t.z;
        vw[3] = t.w;
      }
#pragma unroll
      for (int c = 0; c < CH / 2; ++c) {
        const uint64_t vp = f2pack(bf16_lo(vw[c]), bf16_hi(vw[c]));
        o1p[c] = fma2(f2pack(w1, w1), vp, o1p[c]);
        o2p[c] = fma2(f2pack(w2, w2), vp, o2p[c]);
      }
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
  for (int x = 1; x < 32; x <<= 1) {
    ls1 += __shfl_xor_sync(0xffffffffu, ls1, x);
    ls2 += __shfl_xor_sync(0xffffffffu, ls2, x);
  }
  float* wp = wpart + warp * C::PART_FLOATS;  // [m1, l1, m2, l2, o1[DV], o2[DV]]
  if (lane == 0) {
    wp[0] = m1;
    wp[1] = ls1;
    wp[2] = m2;
    wp[3] = ls2;
  }
#pragma unroll
  for (int c = 0; c < CH / 2; ++c) {
    float l, h;
    f2unpack(o1p[c], l, h);
    wp[4 + vc0 + 2 * c] = l;
    wp[4 + vc0 + 2 * c + 1] = h;
    f2unpack(o2p[c], l, h);
    wp[4 + DV + vc0 + 2 * c] = l;
    wp[4 + DV + vc0 + 2 * c + 1] = h;
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
