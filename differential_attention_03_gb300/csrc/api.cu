// C ABI of libdiffattn.so: argument validation, TMA descriptor encoding,
// kernel selection and launch, and the device status word.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <functional>
#include <mutex>
#include <queue>
#include <string>
#include <utility>
#include <vector>

#include "bwd_params.h"
#include "bwd_prep.cuh"
#include "bwd_tc_params.h"
#include "decode.cuh"
#include "gemm_params.h"
#include "diffattn.h"
#include "launch.h"

// Device status word (one per device that loads the library).  Kernels record
// DIFFATTN_ERR_TIMEOUT here when a bounded wait runs out.
__device__ int g_diffattn_status = 0;

#ifdef DIFFATTN_BOUNDS
namespace da {
namespace {
struct BoundsRegistry {
  std::mutex mu;
  BoundsReader readers[64];
  int count = 0;
};
BoundsRegistry& bounds_registry() {
  static BoundsRegistry r;
  return r;
}
}  // namespace
void bounds_register(BoundsReader reader) {
  BoundsRegistry& r = bounds_registry();
  std::lock_guard<std::mutex> lk(r.mu);
  if (r.count < 64) r.readers[r.count++] = reader;
}
}  // namespace da
#endif

namespace {

thread_local std::string t_last_error;
std::atomic<long long> g_launches{0};

diffattn_status fail(diffattn_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return s;
}

diffattn_status ok() {
  t_last_error.clear();
  return DIFFATTN_OK;
}

diffattn_status cuda_fail(cudaError_t e, const char* what) {
  return fail(DIFFATTN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;

// Device address of g_diffattn_status on the current device.
diffattn_status status_word(int** out) {
  static std::mutex mu;
  static int* ptrs[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(DIFFATTN_ERR_CUDA, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lk(mu);
  if (ptrs[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_diffattn_status);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status)");
    ptrs[dev] = static_cast<int*>(p);
  }
  *out = ptrs[dev];
  return DIFFATTN_OK;
}

// Number of SMs of the current device (cached per device); 0 if unknown.
int sm_count() {
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  int v = cache[dev].load();
  if (v > 0) return v;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v < 1) return 0;
  cache[dev].store(v);
  return v;
}

// Grid of a persistent kernel: one CTA per SM, never more CTAs than items.
long long persistent_grid(long long items) {
  const int sms = sm_count();
  return (sms > 0 && items > sms) ? sms : items;
}

// ---------------------------------------------------------------- TMA maps
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

diffattn_status get_encoder(EncodeTiledFn* fn) {
  static std::once_flag once;
  static EncodeTiledFn cached = nullptr;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
    if (err == cudaSuccess && q == cudaDriverEntryPointSuccess) cached = reinterpret_cast<EncodeTiledFn>(p);
  });
  if (cached == nullptr)
    return fail(DIFFATTN_ERR_CUDA, "cuTensorMapEncodeTiled unavailable (%s)", cudaGetErrorString(err));
  *fn = cached;
  return DIFFATTN_OK;
}

// 4-D map over a BSHD bf16 view [B, n, heads, W]: W columns of each head,
// heads `head_stride` elements apart, tokens `token_stride` elements apart
// (e.g. the query map of one attention head inside a fused projection
// output); box = `cols` columns x 1 head x `rows` tokens x 1 batch, the
// swizzle as wide as a box row (64 or 128 bytes); loads past n return zeros,
// stores past n are dropped.
diffattn_status make_map_view(CUtensorMap* m, const void* base, int B, int n, int heads, int W, long long head_stride,
                              long long token_stride, int cols, int rows) {
  EncodeTiledFn enc;
  diffattn_status s = get_encoder(&enc);
  if (s != DIFFATTN_OK) return s;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(W), static_cast<cuuint64_t>(heads),
                              static_cast<cuuint64_t>(n), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(head_stride) * 2, static_cast<cuuint64_t>(token_stride) * 2,
                                 static_cast<cuuint64_t>(token_stride) * n * 2};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(cols), 1, static_cast<cuuint32_t>(rows), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapSwizzle sw = (cols * 2 == 128) ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(DIFFATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
  return DIFFATTN_OK;
}

// 4-D map over a contiguous BSHD bf16 tensor [B, n, heads, W]; box = `cols`
// columns x 1 head x `rows` tokens x 1 batch, the swizzle as wide as a box row
// (64 or 128 bytes); loads past n return zeros, stores past n are dropped.
diffattn_status make_map_box(CUtensorMap* m, const void* base, int B, int n, int heads, int W, int cols, int rows) {
  return make_map_view(m, base, B, n, heads, W, W, static_cast<long long>(W) * heads, cols, rows);
}

// 2-D map over a row-major bf16 matrix [rows, cols] with row stride `ld`
// elements: box = 64 columns (128 bytes, 128-byte swizzle) x `box_rows` rows;
// loads past either edge return zeros.
diffattn_status make_map_2d(CUtensorMap* m, const void* base, long long rows, long long cols, long long ld,
                            int box_rows) {
  EncodeTiledFn enc;
  diffattn_status s = get_encoder(&enc);
  if (s != DIFFATTN_OK) return s;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(DIFFATTN_ERR_CUDA, "cuTensorMapEncodeTiled (2-D) failed (CUresult %d)", (int)r);
  return DIFFATTN_OK;
}

// 4-D map over a contiguous BSHD fp32 tensor [B, n, heads, W]: box = 32 columns
// (128 bytes, 128-byte swizzle) x 1 head x `rows` tokens x 1 batch (the
// tensor-core backward adds dQ tiles into it with TMA reduce-adds).
diffattn_status make_map_f32(CUtensorMap* m, const void* base, int B, int n, int heads, int W, int rows) {
  EncodeTiledFn enc;
  diffattn_status s = get_encoder(&enc);
  if (s != DIFFATTN_OK) return s;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(W), static_cast<cuuint64_t>(heads),
                              static_cast<cuuint64_t>(n), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(W) * 4, static_cast<cuuint64_t>(W) * heads * 4,
                                 static_cast<cuuint64_t>(W) * heads * n * 4};
  const cuuint32_t box[4] = {32, 1, static_cast<cuuint32_t>(rows), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(DIFFATTN_ERR_CUDA, "cuTensorMapEncodeTiled (f32) failed (CUresult %d)", (int)r);
  return DIFFATTN_OK;
}

// Load maps: 64-column boxes (128-byte rows, 128-byte swizzle).
diffattn_status make_map(CUtensorMap* m, const void* base, int B, int n, int heads, int W, int rows) {
  return make_map_box(m, base, B, n, heads, W, 64, rows);
}

// 4-D map over a BSHD byte tensor (e4m3 key cache) [B, n, heads, W], W of 64
// or 128: box = one full row of W bytes x `rows` tokens, swizzle W bytes wide.
diffattn_status make_map_u8(CUtensorMap* m, const void* base, int B, int n, int heads, int W, int rows) {
  EncodeTiledFn enc;
  diffattn_status s = get_encoder(&enc);
  if (s != DIFFATTN_OK) return s;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(W), static_cast<cuuint64_t>(heads),
                              static_cast<cuuint64_t>(n), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(W), static_cast<cuuint64_t>(W) * heads,
                                 static_cast<cuuint64_t>(W) * heads * n};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(W), 1, static_cast<cuuint32_t>(rows), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapSwizzle sw = (W == 128) ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(DIFFATTN_ERR_CUDA, "cuTensorMapEncodeTiled (u8) failed (CUresult %d)", (int)r);
  return DIFFATTN_OK;
}

// 4-D map over e4m3 codes [B, n, heads, W] viewed as {heads W bytes, 1, n, B}, boxes of 128 bytes x
// `rows`: a head's W = 64-byte row is read together with the next head's (zeros past the last one), so
// the box has the 128-byte swizzled rows the MMA operands use.
diffattn_status make_map_u8_wide(CUtensorMap* m, const void* base, int B, int n, int heads, int W, int rows) {
  EncodeTiledFn enc;
  diffattn_status s = get_encoder(&enc);
  if (s != DIFFATTN_OK) return s;
  const cuuint64_t row = static_cast<cuuint64_t>(W) * heads;
  const cuuint64_t dims[4] = {row, 1, static_cast<cuuint64_t>(n), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {row, row, row * static_cast<cuuint64_t>(n)};
  const cuuint32_t box[4] = {128, 1, static_cast<cuuint32_t>(rows), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(DIFFATTN_ERR_CUDA, "cuTensorMapEncodeTiled (u8, wide) failed (CUresult %d)", (int)r);
  return DIFFATTN_OK;
}

// Per-CTA item lists for a persistent launch of `units` units x `nqt` query
// tiles (tiles [qt0, qt0 + nqt) of each sequence), as indices of the
// unit-major item map.  The units are taken in groups whose K/V streams
// together stay within 32 MiB (so the group's streams stay in L2), the
// heaviest causal tile of every unit of a group first; each item goes to the
// CTA whose planned work ends first, an item counting as its key tiles plus a
// fixed cost of two tiles (greedy list scheduling, as a shared work counter
// would hand items out, without one).  Measured on B2 H12 n4096 d128 (96 MiB of
// K/V): query-tile-major order over all heads in the snake order reads 2.2x the
// input bytes from HBM and takes 0.243 ms; this plan with groups of 8 heads
// 0.231 ms (groups of 12: 0.236 ms and 1.1x the bytes; of 6: 0.238 ms).
// Returns false (plan.count = 0: the kernel's snake order) past the plan's size.
bool plan_items(da::ItemPlan& plan, int grid, long long units, int nqt, int qt0, int n, int causal,
                long long kv_unit_bytes) {
  plan.count = 0;
  const long long nitems = units * nqt;
  if (grid < 1 || grid > da::kPlanMaxCtas || nitems < 1 || nitems > da::kPlanMaxItems) return false;
  const long long budget = 32ll << 20;
  const long long ngroups = std::max(1ll, (units * kv_unit_bytes + budget - 1) / budget);
  const long long ug = (units + ngroups - 1) / ngroups;
  const int ntiles = (n + 127) / 128;
  thread_local std::vector<std::vector<unsigned short>> lists;
  lists.assign(static_cast<size_t>(grid), {});
  using Slot = std::pair<long long, int>;  // (planned end, CTA): the earliest end first, then the lowest CTA
  std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> free_at;
  for (int c = 0; c < grid; ++c) free_at.push({0ll, c});
  for (long long g0 = 0; g0 < units; g0 += ug) {
    const long long g1 = std::min(units, g0 + ug);
    for (int ql = nqt - 1; ql >= 0; --ql) {
      const int T = causal ? std::min(ntiles, qt0 + ql + 1) : ntiles;
      for (long long u = g0; u < g1; ++u) {
        const Slot f = free_at.top();
        free_at.pop();
        lists[static_cast<size_t>(f.second)].push_back(static_cast<unsigned short>(u * nqt + (nqt - 1 - ql)));
        free_at.push({f.first + T + 2, f.second});
      }
    }
  }
  int a = 0;
  for (int c = 0; c < grid; ++c) {
    plan.first[c] = static_cast<unsigned short>(a);
    for (unsigned short it : lists[static_cast<size_t>(c)]) plan.items[a++] = it;
  }
  plan.first[grid] = static_cast<unsigned short>(a);
  plan.count = grid;
  return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Tile order: unit-major keeps all query tiles of one head together so that its
// K/V stream is shared in L2; query-tile-major runs the heaviest causal tiles
// of every head first.  Unit-major is used once the K/V bytes of all units
// exceed what L2 keeps comfortably.
int pick_order(long long units, long long n, int kv_row_bytes) {
  const long long total = units * n * kv_row_bytes;
  return total > (96ll << 20) ? 0 : 1;
}

// Where the inputs of one bf16 forward live: BSHD views, each a base pointer
// with head and token strides in elements (contiguous tensors, or the
// columns of one head inside a fused projection output).
struct QKVViews {
  const void* q1;
  const void* q2;
  const void* k1;
  const void* k2;
  const void* v;
  long long q_head, q_tok;  // strides of q1, q2
  long long k_head, k_tok;  // strides of k1, k2
  long long v_head, v_tok;  // strides of v
};

// Fills a V1 tcgen05 launch around its input maps (already in p) and
// launches it: sc1 / sc2 are the two maps' softmax scales x log2(e); f8
// selects the kernel that reads e4m3 queries and keys.  `out` is a
// contiguous [B, n, H, 2d] tensor.
// Query tiles [qt0, qt0 + nqt) of every (batch, head) (nqt < 0: all of them).
diffattn_status launch_v1_tc(const char* fn, da::TwoPassParams& p, bool f8, int B, int H, int n, int d, float sc1,
                             float sc2, const float* lambda, float lambda_init, const float* gamma, float eps,
                             int causal, void* out, int* status, cudaStream_t s, int qt0 = 0, int nqt = -1) {
  const int dv = 2 * d;
  diffattn_status st;
  // Output stores: boxes of 128 tokens x 32 channels.
  if ((st = make_map_box(&p.tm_out, out, B, n, H, dv, 32, 128)) != DIFFATTN_OK) return st;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lambda = lambda;
  p.gamma = gamma;
  p.lam_logits = nullptr;
  p.scale_log2 = sc1;
  p.scale2_log2 = sc2;
  p.norm_mult = 1.f - lambda_init;
  p.eps = eps;
  p.B = B;
  p.n = n;
  p.causal = causal ? 1 : 0;
  p.units_per_batch = H;
  p.group = 1;
  p.num_q_tiles = nqt < 0 ? (n + 127) / 128 : nqt;
  p.q_tile_begin = qt0;
  p.order = pick_order(static_cast<long long>(B) * H, n, (2 * d + dv) * 2);
  p.status = status;
  const long long grid = static_cast<long long>(p.num_q_tiles) * B * H;
  if (grid > 0x7fffffffll) return fail(DIFFATTN_ERR_SHAPE, "%s: too many tiles", fn);
  // d = 64 (value width 128): one sweep with two online-softmax states fits
  // TMEM; d = 128 (value width 256) does not, and sweeps the keys twice.
  // Short items (up to 64 query tiles per head): one persistent CTA per SM,
  // so each item's start overlaps the previous one's end.  Long items: one
  // CTA per item (the fixed cost is small against them, and the hardware's
  // dynamic CTA scheduling balances them; measured faster).
  const bool persist = qt0 + p.num_q_tiles <= 64;  // (the last tile's item length decides)
  const int g = static_cast<int>(persist ? persistent_grid(grid) : grid);
  // d = 128 persistent: the host's item plan (unit-major item map) instead of the snake order.
  thread_local da::ItemPlan plan;
  plan.count = 0;
  if (persist && d == 128 &&
      plan_items(plan, g, static_cast<long long>(B) * H, p.num_q_tiles, qt0, n, causal,
                 static_cast<long long>(n) * (2 * d + dv) * 2))
    p.order = 0;
  // (p.o1_save set: the training forward, d = 64, which also saves each row's statistics)
  cudaError_t e = f8 ? ((d == 64) ? da::launch_onepass_v1_d64_f8(p, g, persist, s)
                                   : da::launch_twopass_v1_d128_f8(p, plan, g, persist, s))
                  : (d == 64) ? (p.o1_save ? da::launch_onepass_v1_d64_save(p, g, persist, s)
                                           : da::launch_onepass_v1_d64(p, g, persist, s))
                              : da::launch_twopass_v1_d128(p, plan, g, persist, s);
  if (e != cudaSuccess) return cuda_fail(e, fn);
  g_launches.fetch_add(1);
  return DIFFATTN_OK;
}

// DIFF V1 bf16 forward (tcgen05 kernels) on already validated views; `out`
// is a contiguous [B, n, H, 2d] tensor.
diffattn_status forward_v1_bf16(const char* fn, const QKVViews& x, int B, int H, int n, int d, const float* lambda,
                                float lambda_init, const float* gamma, float eps, int causal, void* out, int* status,
                                cudaStream_t s, int qt0 = 0, int nqt = -1) {
  const int dv = 2 * d;
  da::TwoPassParams p;
  memset(&p, 0, sizeof(p));
  diffattn_status st;
  // Query and key tiles are 128 rows; a value tile is split into two 64-row ring slots.
  if ((st = make_map_view(&p.tm_q1, x.q1, B, n, H, d, x.q_head, x.q_tok, 64, 128)) != DIFFATTN_OK) return st;
  if ((st = make_map_view(&p.tm_q2, x.q2, B, n, H, d, x.q_head, x.q_tok, 64, 128)) != DIFFATTN_OK) return st;
  if ((st = make_map_view(&p.tm_k1, x.k1, B, n, H, d, x.k_head, x.k_tok, 64, 128)) != DIFFATTN_OK) return st;
  if ((st = make_map_view(&p.tm_k2, x.k2, B, n, H, d, x.k_head, x.k_tok, 64, 128)) != DIFFATTN_OK) return st;
  if ((st = make_map_view(&p.tm_v, x.v, B, n, H, dv, x.v_head, x.v_tok, 64, 64)) != DIFFATTN_OK) return st;
  const float sc = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d)));
  return launch_v1_tc(fn, p, false, B, H, n, d, sc, sc, lambda, lambda_init, gamma, eps, causal, out, status, s, qt0,
                      nqt);
}

// The DIFF V2 forward (d = 128) on tensor maps of q (Hq heads) and k, v (Hkv
// heads) already in p (e4m3 q and k when f8); `out` is a contiguous
// [B, n, Hq / 2, d] tensor; scale_log2 = softmax scale x log2(e) (x the
// e4m3 dequantisation scales).
diffattn_status launch_v2_tc(const char* fn, da::TwoPassParams& p, bool f8, int B, int Hq, int Hkv, int n, int d,
                             const float* lam_logits, long long sb, long long st_, float scale_log2, int causal,
                             void* out, int* status, cudaStream_t s) {
  const int G = Hq / 2;
  diffattn_status st;
  if ((st = make_map_box(&p.tm_out, out, B, n, G, d, 32, 128)) != DIFFATTN_OK) return st;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lam_logits = lam_logits;
  p.sb = sb;
  p.st = st_;
  p.scale_log2 = scale_log2;
  p.scale2_log2 = scale_log2;  // (both maps score against the same key head with the same scale)
  p.norm_mult = 1.f;
  p.eps = 0.f;
  p.B = B;
  p.n = n;
  p.causal = causal ? 1 : 0;
  p.units_per_batch = G;
  p.group = Hq / Hkv;
  p.num_q_tiles = (n + 127) / 128;
  // K/V bytes per pair: the pairs of one KV head share its stream.
  p.order = pick_order(static_cast<long long>(B) * Hkv, n, 2 * d * 2);
  p.status = status;
  const long long grid = static_cast<long long>(p.num_q_tiles) * B * G;
  if (grid > 0x7fffffffll) return fail(DIFFATTN_ERR_SHAPE, "%s: too many tiles", fn);
  // V2 items are long (up to n / 128 key tiles): one CTA per item, so the
  // hardware's dynamic CTA scheduling balances them (measured faster here).
  cudaError_t e = f8 ? da::launch_onepass_v2_d128_f8(p, static_cast<int>(grid), s)
                  : p.o1_save ? da::launch_onepass_v2_d128_save(p, static_cast<int>(grid), s)
                              : da::launch_onepass_v2_d128(p, static_cast<int>(grid), s);
  if (e != cudaSuccess) return cuda_fail(e, fn);
  g_launches.fetch_add(1);
  return DIFFATTN_OK;
}

// DIFF V2 bf16 forward (d = 128) on already validated views of q (Hq heads)
// and k, v (Hkv heads); `out` is a contiguous [B, n, Hq / 2, d] tensor.
diffattn_status forward_v2_bf16(const char* fn, const QKVViews& x, int B, int Hq, int Hkv, int n, int d,
                                const float* lam_logits, long long sb, long long st_, float scale, int causal,
                                void* out, int* status, cudaStream_t s) {
  da::TwoPassParams p;
  memset(&p, 0, sizeof(p));
  diffattn_status st;
  if ((st = make_map_view(&p.tm_q1, x.q1, B, n, Hq, d, x.q_head, x.q_tok, 64, 128)) != DIFFATTN_OK) return st;
  p.tm_q2 = p.tm_q1;
  // Key and value tiles are 128 rows (one ring slot each).
  if ((st = make_map_view(&p.tm_k1, x.k1, B, n, Hkv, d, x.k_head, x.k_tok, 64, 128)) != DIFFATTN_OK) return st;
  p.tm_k2 = p.tm_k1;
  if ((st = make_map_view(&p.tm_v, x.v, B, n, Hkv, d, x.v_head, x.v_tok, 64, 128)) != DIFFATTN_OK) return st;
  return launch_v2_tc(fn, p, false, B, Hq, Hkv, n, d, lam_logits, sb, st_,
                      static_cast<float>(1.4426950408889634 * scale), causal, out, status, s);
}

}  // namespace

extern "C" {

float diffattn_lambda_init(int layer_index) {
  if (layer_index < 1) return NAN;
  return static_cast<float>(0.8 - 0.6 * std::exp(-0.3 * (layer_index - 1)));
}

diffattn_status lambda_reparam(const float* lq1, const float* lk1, const float* lq2, const float* lk2, int dim,
                               float lambda_init, float* lambda_out, void* stream) {
  if (!lq1 || !lk1 || !lq2 || !lk2 || !lambda_out) return fail(DIFFATTN_ERR_NULL, "lambda_reparam: NULL pointer");
  if (dim < 1) return fail(DIFFATTN_ERR_SHAPE, "lambda_reparam: dim must be >= 1 (got %d)", dim);
  cudaError_t e = da::launch_lambda_reparam(lq1, lk1, lq2, lk2, dim, lambda_init, lambda_out,
                                            static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "lambda_reparam launch");
  g_launches.fetch_add(1);
  return ok();
}

diffattn_status diffattn_forward(diffattn_dtype dt, int B, int H, int n, int d, const void* q1, const void* q2,
                                 const void* k1, const void* k2, const void* v, const float* lambda,
                                 float lambda_init, const float* gamma, float eps, int causal, void* out,
                                 void* stream) {
  if (dt != DIFFATTN_F32 && dt != DIFFATTN_BF16) return fail(DIFFATTN_ERR_DTYPE, "diffattn_forward: bad dtype %d", (int)dt);
  if (B < 0 || H < 0 || n < 0 || d < 1)
    return fail(DIFFATTN_ERR_SHAPE, "diffattn_forward: bad sizes B=%d H=%d n=%d d=%d", B, H, n, d);
  if (B == 0 || H == 0 || n == 0) return ok();
  if (!q1 || !q2 || !k1 || !k2 || !v || !lambda || !out)
    return fail(DIFFATTN_ERR_NULL, "diffattn_forward: NULL pointer");
  if (!std::isfinite(lambda_init)) return fail(DIFFATTN_ERR_SHAPE, "diffattn_forward: lambda_init not finite");
  if (eps <= 0.f) eps = 1e-5f;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int dv = 2 * d;
  int* status = nullptr;

  if (dt == DIFFATTN_F32) {
    if (d > da::kSimtMaxD) return fail(DIFFATTN_ERR_UNSUPPORTED, "diffattn_forward: f32 needs d <= 128 (got %d)", d);
    diffattn_status st = status_word(&status);
    if (st != DIFFATTN_OK) return st;
    da::SimtParams p{};
    p.q1 = static_cast<const float*>(q1);
    p.q2 = static_cast<const float*>(q2);
    p.k1 = static_cast<const float*>(k1);
    p.k2 = static_cast<const float*>(k2);
    p.v = static_cast<const float*>(v);
    p.out = static_cast<float*>(out);
    p.lambda = lambda;
    p.gamma = gamma;
    p.scale = 1.f / std::sqrt(static_cast<float>(d));
    p.norm_mult = 1.f - lambda_init;
    p.eps = eps;
    p.B = B;
    p.n = n;
    p.d = d;
    p.dv = dv;
    p.causal = causal ? 1 : 0;
    p.v2 = 0;
    p.heads_q = p.heads_kv = p.units_per_batch = H;
    p.group = 1;
    p.rows_total = static_cast<long long>(B) * H * n;
    cudaError_t e = da::launch_simt_f32(p, s);
    if (e != cudaSuccess) return cuda_fail(e, "diffattn_forward (f32) launch");
    g_launches.fetch_add(1);
    return ok();
  }

  // bf16: tcgen05 kernels
  if (d != 64 && d != 128) return fail(DIFFATTN_ERR_UNSUPPORTED, "diffattn_forward: bf16 needs d in {64, 128} (got %d)", d);
  if (!aligned16(q1) || !aligned16(q2) || !aligned16(k1) || !aligned16(k2) || !aligned16(v) || !aligned16(out))
    return fail(DIFFATTN_ERR_ALIGN, "diffattn_forward: bf16 tensors must be 16-byte aligned");
  diffattn_status st = status_word(&status);
  if (st != DIFFATTN_OK) return st;
  const long long Hd = static_cast<long long>(H) * d;
  const QKVViews x{q1, q2, k1, k2, v, d, Hd, d, Hd, dv, 2 * Hd};
  if ((st = forward_v1_bf16("diffattn_forward (bf16)", x, B, H, n, d, lambda, lambda_init, gamma, eps, causal, out,
                            status, s)) != DIFFATTN_OK)
    return st;
  return ok();
}

// ---------------------------------------------------------------- forward with e4m3 queries and keys
diffattn_status diffattn_forward_fp8qk(int B, int H, int n, int d, const void* q1, const void* q2, const void* k1,
                                       const void* k2, float q1_scale, float q2_scale, float k1_scale,
                                       float k2_scale, const void* v, const float* lambda, float lambda_init,
                                       const float* gamma, float eps, int causal, void* out, void* stream) {
  const char* fn = "diffattn_forward_fp8qk";
  if (B < 0 || H < 0 || n < 0 || d < 1)
    return fail(DIFFATTN_ERR_SHAPE, "%s: bad sizes B=%d H=%d n=%d d=%d", fn, B, H, n, d);
  if (d != 128 && d != 64) return fail(DIFFATTN_ERR_UNSUPPORTED, "%s: d = 64 or 128 only (got %d)", fn, d);
  if (B == 0 || H == 0 || n == 0) return ok();
  if (d == 64 && H < 2)  // (the 128-byte boxes span two heads' rows)
    return fail(DIFFATTN_ERR_UNSUPPORTED, "%s: d = 64 needs at least two heads (got H = %d)", fn, H);
  if (!q1 || !q2 || !k1 || !k2 || !v || !lambda || !out) return fail(DIFFATTN_ERR_NULL, "%s: NULL pointer", fn);
  if (!std::isfinite(lambda_init)) return fail(DIFFATTN_ERR_SHAPE, "%s: lambda_init not finite", fn);
  for (float sc : {q1_scale, q2_scale, k1_scale, k2_scale})
    if (!(std::isfinite(sc) && sc > 0.f)) return fail(DIFFATTN_ERR_SHAPE, "%s: scales must be finite and positive", fn);
  if (!aligned16(q1) || !aligned16(q2) || !aligned16(k1) || !aligned16(k2) || !aligned16(v) || !aligned16(out))
    return fail(DIFFATTN_ERR_ALIGN, "%s: tensors must be 16-byte aligned", fn);
  if (eps <= 0.f) eps = 1e-5f;
  int* status = nullptr;
  diffattn_status st = status_word(&status);
  if (st != DIFFATTN_OK) return st;
  const int dv = 2 * d;
  da::TwoPassParams p;
  memset(&p, 0, sizeof(p));
  // Query and key rows: d = 128, 128 bytes, one box (128-byte swizzle) of 128 rows a tile; d = 64, a
  // 128-byte box over this head's row and the next one's.  V: 64-row boxes (the ring's half slots).
  auto qk_map = [&](CUtensorMap* m, const void* base) {
    return d == 128 ? make_map_u8(m, base, B, n, H, d, 128) : make_map_u8_wide(m, base, B, n, H, d, 128);
  };
  if ((st = qk_map(&p.tm_q1, q1)) != DIFFATTN_OK) return st;
  if ((st = qk_map(&p.tm_q2, q2)) != DIFFATTN_OK) return st;
  if ((st = qk_map(&p.tm_k1, k1)) != DIFFATTN_OK) return st;
  if ((st = qk_map(&p.tm_k2, k2)) != DIFFATTN_OK) return st;
  if ((st = make_map_box(&p.tm_v, v, B, n, H, dv, 64, 64)) != DIFFATTN_OK) return st;
  // S_r = (q_scale_r k_scale_r) e4m3(q_r) e4m3(k_r)^T / sqrt(d): the scales fold into each map's exponent.
  const double c = 1.4426950408889634 / std::sqrt(static_cast<double>(d));
  const float sc1 = static_cast<float>(c * q1_scale * k1_scale), sc2 = static_cast<float>(c * q2_scale * k2_scale);
  if ((st = launch_v1_tc(fn, p, true, B, H, n, d, sc1, sc2, lambda, lambda_init, gamma, eps, causal, out, status,
                         static_cast<cudaStream_t>(stream))) != DIFFATTN_OK)
    return st;
  return ok();
}

// DIFF V2 forward with e4m3 queries and keys (d = 128): QK^T on kind::f8f6f4.
diffattn_status diffattn_v2_forward_fp8qk(int B, int Hq, int Hkv, int n, int d, const void* q, const void* k,
                                          float q_scale, float k_scale, const void* v, const float* lam_logits,
                                          long long sb, long long st_, float softmax_scale, int causal, void* out,
                                          void* stream) {
  const char* fn = "diffattn_v2_forward_fp8qk";
  if (B < 0 || Hq < 0 || Hkv < 1 || n < 0 || d < 1)
    return fail(DIFFATTN_ERR_SHAPE, "%s: bad sizes B=%d Hq=%d Hkv=%d n=%d d=%d", fn, B, Hq, Hkv, n, d);
  if (Hq % 2 != 0 || Hq % Hkv != 0 || (Hq / Hkv) % 2 != 0)
    return fail(DIFFATTN_ERR_SHAPE, "%s: need Hq even, Hq %% Hkv == 0 and Hq/Hkv even (Hq=%d Hkv=%d)", fn, Hq, Hkv);
  if (sb < 0 || st_ < 0) return fail(DIFFATTN_ERR_SHAPE, "%s: negative logit stride", fn);
  if (d != 128) return fail(DIFFATTN_ERR_UNSUPPORTED, "%s: d = 128 only (got %d)", fn, d);
  if (B == 0 || Hq == 0 || n == 0) return ok();
  if (!q || !k || !v || !lam_logits || !out) return fail(DIFFATTN_ERR_NULL, "%s: NULL pointer", fn);
  for (float sc : {q_scale, k_scale})
    if (!(std::isfinite(sc) && sc > 0.f)) return fail(DIFFATTN_ERR_SHAPE, "%s: scales must be finite and positive", fn);
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return fail(DIFFATTN_ERR_ALIGN, "%s: tensors must be 16-byte aligned", fn);
  const double scale = softmax_scale > 0.f ? softmax_scale : 1.0 / std::sqrt(static_cast<double>(d));
  int* status = nullptr;
  diffattn_status st = status_word(&status);
  if (st != DIFFATTN_OK) return st;
  da::TwoPassParams p;
  memset(&p, 0, sizeof(p));
  // Query and key rows are 128 bytes: one box (128-byte swizzle) of 128 rows a tile.
  if ((st = make_map_u8(&p.tm_q1, q, B, n, Hq, d, 128)) != DIFFATTN_OK) return st;
  p.tm_q2 = p.tm_q1;
  if ((st = make_map_u8(&p.tm_k1, k, B, n, Hkv, d, 128)) != DIFFATTN_OK) return st;
  p.tm_k2 = p.tm_k1;
  if ((st = make_map_box(&p.tm_v, v, B, n, Hkv, d, 64, 128)) != DIFFATTN_OK) return st;
  // S = (q_scale k_scale) e4m3(q) e4m3(k)^T x scale: both scales fold into the exponent.
  const float sc = static_cast<float>(1.4426950408889634 * scale * q_scale * k_scale);
  if ((st = launch_v2_tc(fn, p, true, B, Hq, Hkv, n, d, lam_logits, sb, st_, sc, causal, out, status,
                         static_cast<cudaStream_t>(stream))) != DIFFATTN_OK)
    return st;
  return ok();
}

// ---------------------------------------------------------------- host-buffer forward
namespace {

constexpr int kMaxChunks = 8;  // chunks per call (events per pipeline)

// Copy streams and events of the host-buffer forward, created once per device
// and reused by every call (enqueueing a call holds the mutex, so calls from
// several host threads do not interleave their event records).
struct HostPipe {
  std::mutex mu;
  bool ready = false;
  cudaStream_t in = nullptr, out = nullptr;
  cudaStream_t comp = nullptr;  // second compute stream: token chunks alternate between it and the caller's
  cudaEvent_t start = nullptr, last_out = nullptr;
  cudaEvent_t in_done[kMaxChunks] = {}, fwd_done[kMaxChunks] = {};
};

diffattn_status host_pipe(HostPipe** out) {
  static HostPipe pipes[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(DIFFATTN_ERR_CUDA, "device index %d out of range", dev);
  *out = &pipes[dev];
  return DIFFATTN_OK;
}

diffattn_status host_pipe_init(HostPipe& hp) {
  if (hp.ready) return DIFFATTN_OK;
  cudaError_t e = cudaStreamCreateWithFlags(&hp.in, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&hp.out, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&hp.comp, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.start, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.last_out, cudaEventDisableTiming);
  for (int c = 0; e == cudaSuccess && c < kMaxChunks; ++c) {
    e = cudaEventCreateWithFlags(&hp.in_done[c], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.fwd_done[c], cudaEventDisableTiming);
  }
  if (e != cudaSuccess) return cuda_fail(e, "diffattn_forward_host: stream/event creation");
  hp.ready = true;
  return DIFFATTN_OK;
}

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

size_t diffattn_forward_host_workspace(diffattn_dtype dt, int B, int H, int n, int d) {
  if ((dt != DIFFATTN_F32 && dt != DIFFATTN_BF16) || B < 0 || H < 0 || n < 0 || d < 1) return 0;
  const size_t es = dt == DIFFATTN_BF16 ? 2 : 4;
  const size_t qk = static_cast<size_t>(B) * n * H * d * es;  // one of q1, q2, k1, k2
  const size_t vo = 2 * qk;                                   // v or out
  return 4 * round256(qk) + 2 * round256(vo);
}

diffattn_status diffattn_forward_host(diffattn_dtype dt, int B, int H, int n, int d, const void* q1,
                                      const void* q2, const void* k1, const void* k2, const void* v,
                                      const float* lambda, float lambda_init, const float* gamma, float eps,
                                      int causal, void* out, void* workspace, size_t workspace_bytes,
                                      void* stream) {
  if (dt != DIFFATTN_F32 && dt != DIFFATTN_BF16)
    return fail(DIFFATTN_ERR_DTYPE, "diffattn_forward_host: bad dtype %d", (int)dt);
  if (B < 0 || H < 0 || n < 0 || d < 1)
    return fail(DIFFATTN_ERR_SHAPE, "diffattn_forward_host: bad sizes B=%d H=%d n=%d d=%d", B, H, n, d);
  if (B == 0 || H == 0 || n == 0) return ok();
  if (!q1 || !q2 || !k1 || !k2 || !v || !lambda || !out || !workspace)
    return fail(DIFFATTN_ERR_NULL, "diffattn_forward_host: NULL pointer");
  const size_t need = diffattn_forward_host_workspace(dt, B, H, n, d);
  if (workspace_bytes < need)
    return fail(DIFFATTN_ERR_SHAPE, "diffattn_forward_host: workspace of %zu bytes, %zu needed", workspace_bytes,
                need);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(DIFFATTN_ERR_ALIGN, "diffattn_forward_host: workspace not 256-byte aligned");
  HostPipe* hp = nullptr;
  diffattn_status st = host_pipe(&hp);
  if (st != DIFFATTN_OK) return st;
  std::lock_guard<std::mutex> lk(hp->mu);
  if ((st = host_pipe_init(*hp)) != DIFFATTN_OK) return st;

  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t es = dt == DIFFATTN_BF16 ? 2 : 4;
  const size_t qk_b = static_cast<size_t>(n) * H * d * es;  // bytes of one batch of q1 (q2, k1, k2)
  const size_t vo_b = 2 * qk_b;                             // bytes of one batch of v (out)
  const size_t qk = round256(qk_b * B), vo = round256(vo_b * B);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint8_t* const dq1 = ws;
  uint8_t* const dq2 = dq1 + qk;
  uint8_t* const dk1 = dq2 + qk;
  uint8_t* const dk2 = dk1 + qk;
  uint8_t* const dv = dk2 + qk;
  uint8_t* const dout = dv + vo;

  // The copies in wait for the caller's earlier work on `stream` (which
  // includes the copy out of the previous call on this workspace).
  cudaError_t e = cudaEventRecord(hp->start, s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->in, hp->start, 0);
  if (e != cudaSuccess) return cuda_fail(e, "diffattn_forward_host: stream ordering");

  // Few sequences of a causal bf16 forward: pipeline over token chunks instead
  // of batch chunks.  Chunk c holds tokens [t0, t1) of every sequence (128-row
  // tiles [c0, c1)); in BSHD those rows are contiguous per sequence.  The
  // queries of chunk c see only keys < t1, all copied in by chunks 0 .. c, so
  // its forward (query tiles [c0, c1) against the whole device buffer) starts
  // once its own copies are in, while the next chunk's copies run.  The
  // chunks' forwards write disjoint rows and depend only on copies, so they
  // alternate between the caller's stream and a second compute stream: the
  // next chunk's CTAs take the SMs that the previous launch's last CTAs leave
  // idle.  Each query tile's item is the same as in one launch over every
  // tile, so the results are identical to diffattn_forward's.
  const int ntiles = (n + 127) / 128;
  if (dt == DIFFATTN_BF16 && causal && B < 4 && ntiles >= 2) {
    if (d != 64 && d != 128)
      return fail(DIFFATTN_ERR_UNSUPPORTED, "diffattn_forward_host: bf16 needs d in {64, 128} (got %d)", d);
    if (!std::isfinite(lambda_init)) return fail(DIFFATTN_ERR_SHAPE, "diffattn_forward_host: lambda_init not finite");
    int* status = nullptr;
    if ((st = status_word(&status)) != DIFFATTN_OK) return st;
    if (eps <= 0.f) eps = 1e-5f;
    const size_t qrow = static_cast<size_t>(H) * d * es, vrow = 2 * qrow;  // bytes of one token's row
    const long long Hd = static_cast<long long>(H) * d;
    const QKVViews x{dq1, dq2, dk1, dk2, dv, d, Hd, d, Hd, 2 * d, 2 * Hd};
    const int nchunk = ntiles < kMaxChunks ? ntiles : kMaxChunks;
    const uint8_t* hsrc[5] = {static_cast<const uint8_t*>(q1), static_cast<const uint8_t*>(q2),
                              static_cast<const uint8_t*>(k1), static_cast<const uint8_t*>(k2),
                              static_cast<const uint8_t*>(v)};
    uint8_t* const ddst[5] = {dq1, dq2, dk1, dk2, dv};
    for (int c = 0; c < nchunk; ++c) {
      const int c0 = static_cast<int>(static_cast<long long>(ntiles) * c / nchunk);
      const int c1 = static_cast<int>(static_cast<long long>(ntiles) * (c + 1) / nchunk);
      const size_t t0 = static_cast<size_t>(c0) * 128, t1 = std::min(static_cast<size_t>(n), static_cast<size_t>(c1) * 128);
      for (int b = 0; b < B && e == cudaSuccess; ++b) {
        const size_t r0 = static_cast<size_t>(b) * n + t0;
        for (int tsr = 0; tsr < 5 && e == cudaSuccess; ++tsr) {
          const size_t rb = tsr == 4 ? vrow : qrow;
          e = cudaMemcpyAsync(ddst[tsr] + r0 * rb, hsrc[tsr] + r0 * rb, (t1 - t0) * rb, cudaMemcpyHostToDevice,
                              hp->in);
        }
      }
      // (the second compute stream sees the caller's earlier work, lambda
      // included, through the copy stream, which waited for it at `start`)
      const cudaStream_t sc = (c & 1) ? hp->comp : s;
      if (e == cudaSuccess) e = cudaEventRecord(hp->in_done[c], hp->in);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(sc, hp->in_done[c], 0);
      if (e != cudaSuccess) return cuda_fail(e, "diffattn_forward_host: copy in");
      if ((st = forward_v1_bf16("diffattn_forward_host", x, B, H, n, d, lambda, lambda_init, gamma, eps, causal, dout,
                                status, sc, c0, c1 - c0)) != DIFFATTN_OK)
        return st;
      e = cudaEventRecord(hp->fwd_done[c], sc);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->out, hp->fwd_done[c], 0);
      for (int b = 0; b < B && e == cudaSuccess; ++b) {
        const size_t r0 = static_cast<size_t>(b) * n + t0;
        e = cudaMemcpyAsync(static_cast<uint8_t*>(out) + r0 * vrow, dout + r0 * vrow, (t1 - t0) * vrow,
                            cudaMemcpyDeviceToHost, hp->out);
      }
      if (e != cudaSuccess) return cuda_fail(e, "diffattn_forward_host: copy out");
    }
    e = cudaEventRecord(hp->last_out, hp->out);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, hp->last_out, 0);
    if (e != cudaSuccess) return cuda_fail(e, "diffattn_forward_host: stream ordering");
    return ok();
  }

  const int nchunk = B < kMaxChunks ? B : kMaxChunks;
  for (int c = 0; c < nchunk; ++c) {
    const int b0 = static_cast<int>(static_cast<long long>(B) * c / nchunk);
    const int b1 = static_cast<int>(static_cast<long long>(B) * (c + 1) / nchunk);
    const size_t oq = qk_b * b0, ov = vo_b * b0;
    const size_t nq = qk_b * (b1 - b0), nv = vo_b * (b1 - b0);
    const uint8_t* hq1 = static_cast<const uint8_t*>(q1);
    const uint8_t* hq2 = static_cast<const uint8_t*>(q2);
    const uint8_t* hk1 = static_cast<const uint8_t*>(k1);
    const uint8_t* hk2 = static_cast<const uint8_t*>(k2);
    const uint8_t* hv = static_cast<const uint8_t*>(v);
    // One cudaMemcpyAsync per tensor of the chunk, on the copy-in stream.
    e = cudaMemcpyAsync(dq1 + oq, hq1 + oq, nq, cudaMemcpyHostToDevice, hp->in);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dq2 + oq, hq2 + oq, nq, cudaMemcpyHostToDevice, hp->in);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dk1 + oq, hk1 + oq, nq, cudaMemcpyHostToDevice, hp->in);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dk2 + oq, hk2 + oq, nq, cudaMemcpyHostToDevice, hp->in);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dv + ov, hv + ov, nv, cudaMemcpyHostToDevice, hp->in);
    if (e == cudaSuccess) e = cudaEventRecord(hp->in_done[c], hp->in);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, hp->in_done[c], 0);
    if (e != cudaSuccess) return cuda_fail(e, "diffattn_forward_host: copy in");
    // The forward of the chunk on the caller's stream.
    st = diffattn_forward(dt, b1 - b0, H, n, d, dq1 + oq, dq2 + oq, dk1 + oq, dk2 + oq, dv + ov, lambda, lambda_init,
                          gamma, eps, causal, dout + ov, stream);
    if (st != DIFFATTN_OK) return st;
    // Its output back on the copy-out stream.
    e = cudaEventRecord(hp->fwd_done[c], s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->out, hp->fwd_done[c], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(static_cast<uint8_t*>(out) + ov, dout + ov, nv, cudaMemcpyDeviceToHost, hp->out);
    if (e != cudaSuccess) return cuda_fail(e, "diffattn_forward_host: copy out");
  }
  // The caller's stream resumes once every output byte is back in host memory.
  e = cudaEventRecord(hp->last_out, hp->out);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s, hp->last_out, 0);
  if (e != cudaSuccess) return cuda_fail(e, "diffattn_forward_host: stream ordering");
  return ok();
}

// CTAs per (batch, head) cluster of the decode kernels: the smallest power of
// two that gives at least two waves of two CTAs per SM, at most 8 and at most
// one CTA per four stages of keys.
static int decode_cluster_size(long long units, int n, int bk) {
  const int sms = sm_count() > 0 ? sm_count() : 148;
  const long long want = 4ll * sms;
  const int max_by_keys = std::max(1, n / (4 * bk));
  int cs = 1;
  while (cs < da::DecodeCfg<64>::MAX_CS && units * cs < want && cs * 2 <= max_by_keys) cs *= 2;
  return cs;
}

// Clusters per (batch, head) when a workspace is given: as many as keep the
// grid within one wave of two CTAs per SM (so that pairs too few to fill the
// GPU with one cluster each still do), at most kMaxSplit, each CTA keeping at
// least four stages of keys.
constexpr int kMaxSplit = 8;
static int decode_split(long long units, int cs, int n, int bk) {
  const int sms = sm_count() > 0 ? sm_count() : 148;
  int ns = static_cast<int>(std::min<long long>(kMaxSplit, (2ll * sms) / std::max<long long>(1, units * cs)));
  ns = std::max(1, std::min(ns, n / (4 * bk * cs)));
  return ns;
}

// Partial-state floats of one cluster: two maps x (maximum, sum, dv channels).
static size_t decode_part_floats(int dv) { return 2 * (static_cast<size_t>(dv) + 2); }

size_t diffattn_decode_workspace(int B, int H, int d) {
  if (B < 0 || H < 0 || d < 1) return 0;
  return static_cast<size_t>(B) * H * kMaxSplit * decode_part_floats(2 * d) * sizeof(float);
}

size_t diffattn_v2_decode_workspace(int B, int Hq, int d) {
  if (B < 0 || Hq < 0 || d < 1) return 0;
  return static_cast<size_t>(B) * (Hq / 2) * kMaxSplit * decode_part_floats(d) * sizeof(float);
}

// V1 decode with bf16 (k8 false) or e4m3 (k8 true, scales k1_scale, k2_scale) key caches.
static diffattn_status decode_v1(const char* fn, diffattn_dtype dt, int B, int H, int n, int d, const void* q1,
                                 const void* q2, const void* k1, const void* k2, bool k8, float k1_scale,
                                 float k2_scale, const void* v, const int* lens, const float* lambda,
                                 float lambda_init, const float* gamma, float eps, void* out, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  if (dt != DIFFATTN_F32 && dt != DIFFATTN_BF16) return fail(DIFFATTN_ERR_DTYPE, "%s: bad dtype %d", fn, (int)dt);
  if (B < 0 || H < 0 || n < 0 || d < 1)
    return fail(DIFFATTN_ERR_SHAPE, "%s: bad sizes B=%d H=%d n=%d d=%d", fn, B, H, n, d);
  if (B == 0 || H == 0) return ok();
  if (!q1 || !q2 || !k1 || !k2 || !v || !lambda || !out) return fail(DIFFATTN_ERR_NULL, "%s: NULL pointer", fn);
  if (dt != DIFFATTN_BF16 || (d != 64 && d != 128))
    return fail(DIFFATTN_ERR_UNSUPPORTED, "%s: bf16 with d in {64, 128} only (got dtype %d, d=%d)", fn, (int)dt,
                d);
  if (!std::isfinite(lambda_init)) return fail(DIFFATTN_ERR_SHAPE, "%s: lambda_init not finite", fn);
  if (k8 && !(std::isfinite(k1_scale) && std::isfinite(k2_scale) && k1_scale > 0.f && k2_scale > 0.f))
    return fail(DIFFATTN_ERR_SHAPE, "%s: key scales must be finite and positive", fn);
  if (!aligned16(q1) || !aligned16(q2) || !aligned16(k1) || !aligned16(k2) || !aligned16(v) || !aligned16(out))
    return fail(DIFFATTN_ERR_ALIGN, "%s: tensors must be 16-byte aligned", fn);
  const long long units = static_cast<long long>(B) * H;
  if (units * da::DecodeCfg<64>::MAX_CS * kMaxSplit > 0x7fffffffll)
    return fail(DIFFATTN_ERR_SHAPE, "%s: too many (batch, head) pairs", fn);
  if (workspace != nullptr) {
    const size_t need = diffattn_decode_workspace(B, H, d);
    if (workspace_bytes < need)
      return fail(DIFFATTN_ERR_SHAPE, "%s: workspace of %zu bytes, %zu needed (or pass NULL)", fn, workspace_bytes,
                  need);
    if ((reinterpret_cast<uintptr_t>(workspace) & 3u) != 0)
      return fail(DIFFATTN_ERR_ALIGN, "%s: workspace must be 4-byte aligned", fn);
  }
  if (eps <= 0.f) eps = 1e-5f;
  int* status = nullptr;
  diffattn_status st = status_word(&status);
  if (st != DIFFATTN_OK) return st;
  da::DecodeParams p;
  memset(&p, 0, sizeof(p));
  // keys per stage (= TMA box rows) of the kernel that runs
  const int bk = k8 ? ((d == 64) ? da::DecodeCfg<64, false, true>::BK : da::DecodeCfg<128, false, true>::BK)
                    : ((d == 64) ? da::DecodeCfg<64>::BK : da::DecodeCfg<128>::BK);
  const int nn = n > 0 ? n : 1;  // an empty cache still needs a valid map (no key is read)
  if (k8) {
    if ((st = make_map_u8(&p.tm_k1, k1, B, nn, H, d, bk)) != DIFFATTN_OK) return st;
    if ((st = make_map_u8(&p.tm_k2, k2, B, nn, H, d, bk)) != DIFFATTN_OK) return st;
  } else {
    if ((st = make_map(&p.tm_k1, k1, B, nn, H, d, bk)) != DIFFATTN_OK) return st;
    if ((st = make_map(&p.tm_k2, k2, B, nn, H, d, bk)) != DIFFATTN_OK) return st;
  }
  p.k1_scale = k1_scale;
  p.k2_scale = k2_scale;
  if ((st = make_map(&p.tm_v, v, B, nn, H, 2 * d, bk)) != DIFFATTN_OK) return st;
  p.q1 = static_cast<const __nv_bfloat16*>(q1);
  p.q2 = static_cast<const __nv_bfloat16*>(q2);
  p.lens = lens;
  p.lambda = lambda;
  p.gamma = gamma;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d)));
  p.norm_mult = 1.f - lambda_init;
  p.eps = eps;
  p.B = B;
  p.H = H;
  p.n = n;
  p.status = status;
  const int cs = decode_cluster_size(units, n, bk);
  p.nsplit = 1;
  if (workspace != nullptr) {
    p.nsplit = decode_split(units, cs, n, bk);
    p.ws = static_cast<float*>(workspace);
  }
  cudaError_t e = da::launch_decode_v1(p, d, k8, static_cast<int>(units), cs, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, fn);
  g_launches.fetch_add(1);
  return ok();
}

diffattn_status diffattn_decode(diffattn_dtype dt, int B, int H, int n, int d, const void* q1, const void* q2,
                                const void* k1, const void* k2, const void* v, const int* lens,
                                const float* lambda, float lambda_init, const float* gamma, float eps, void* out,
                                void* workspace, size_t workspace_bytes, void* stream) {
  return decode_v1("diffattn_decode", dt, B, H, n, d, q1, q2, k1, k2, false, 1.f, 1.f, v, lens, lambda, lambda_init,
                   gamma, eps, out, workspace, workspace_bytes, stream);
}

// ---------------------------------------------------------------- decode with no allocation
}  // extern "C"

// Scratch of diffattn_decode_noalloc: the partial softmax states of the
// clusters that share a (batch, head) pair's keys, the same data a caller's
// workspace holds for diffattn_decode.  A fixed array in the library's device
// image: every GPU that loads the library keeps these 4 MiB until the process
// exits.  Host code may not use the name as an address (it is a host-side
// stand-in); decode_noalloc_scratch() looks the device address up.
constexpr size_t kDecodeScratchBytes = size_t(4) << 20;
static __device__ __align__(256) float g_decode_noalloc_scratch[kDecodeScratchBytes / sizeof(float)];

namespace {

// Device address of the scratch on the current device, looked up once per
// device (the first call on a device does it, with that device current).
diffattn_status decode_noalloc_scratch(void** out) {
  static std::mutex mu;
  static void* ptrs[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(DIFFATTN_ERR_CUDA, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lk(mu);
  if (ptrs[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(decode scratch)");
    ptrs[dev] = p;
  }
  *out = ptrs[dev];
  return DIFFATTN_OK;
}

}  // namespace

extern "C" {

diffattn_status diffattn_decode_noalloc(diffattn_dtype dt, int B, int H, int n, int d, const void* q1,
                                        const void* q2, const void* k1, const void* k2, const void* v,
                                        const int* lens, const float* lambda, float lambda_init,
                                        const float* gamma, float eps, void* out, void* stream) {
  const char* fn = "diffattn_decode_noalloc";
  // Only calls that reach a launch need the scratch; every other call gets
  // diffattn_decode's own answer (an argument error, or nothing to do).
  void* scratch = nullptr;
  if (dt == DIFFATTN_BF16 && B > 0 && H > 0 && n >= 0 && (d == 64 || d == 128)) {
    const size_t need = diffattn_decode_workspace(B, H, d);
    if (need > kDecodeScratchBytes)
      return fail(DIFFATTN_ERR_SHAPE,
                  "%s: B*H = %lld (batch, head) pairs need %zu bytes of scratch, more than the %zu it has "
                  "(at most %zu pairs at d = %d); call diffattn_decode with a NULL workspace instead (it "
                  "allocates nothing, and that many pairs fill the GPU without splitting)",
                  fn, static_cast<long long>(B) * H, need, kDecodeScratchBytes,
                  kDecodeScratchBytes / diffattn_decode_workspace(1, 1, d), d);
    diffattn_status st = decode_noalloc_scratch(&scratch);
    if (st != DIFFATTN_OK) return st;
  }
  return decode_v1(fn, dt, B, H, n, d, q1, q2, k1, k2, false, 1.f, 1.f, v, lens, lambda, lambda_init, gamma, eps,
                   out, scratch, scratch ? kDecodeScratchBytes : 0, stream);
}

diffattn_status diffattn_decode_fp8k(int B, int H, int n, int d, const void* q1, const void* q2, const void* k1,
                                     const void* k2, float k1_scale, float k2_scale, const void* v,
                                     const int* lens, const float* lambda, float lambda_init, const float* gamma,
                                     float eps, void* out, void* workspace, size_t workspace_bytes, void* stream) {
  return decode_v1("diffattn_decode_fp8k", DIFFATTN_BF16, B, H, n, d, q1, q2, k1, k2, true, k1_scale, k2_scale, v,
                   lens, lambda, lambda_init, gamma, eps, out, workspace, workspace_bytes, stream);
}

// V2 decode with a bf16 (k8 false) or e4m3 (k8 true, scale k_scale) key cache.
static diffattn_status decode_v2(const char* fn, diffattn_dtype dt, int B, int Hq, int Hkv, int n, int d,
                                 const void* q, const void* k, bool k8, float k_scale, const void* v,
                                 const int* lens, const float* lam_logits, long long sb, float softmax_scale,
                                 void* out, void* workspace, size_t workspace_bytes, void* stream) {
  if (dt != DIFFATTN_F32 && dt != DIFFATTN_BF16)
    return fail(DIFFATTN_ERR_DTYPE, "%s: bad dtype %d", fn, (int)dt);
  if (B < 0 || Hq < 0 || Hkv < 1 || n < 0 || d < 1)
    return fail(DIFFATTN_ERR_SHAPE, "%s: bad sizes B=%d Hq=%d Hkv=%d n=%d d=%d", fn, B, Hq, Hkv, n, d);
  if (Hq % 2 != 0 || Hq % Hkv != 0 || (Hq / Hkv) % 2 != 0)
    return fail(DIFFATTN_ERR_SHAPE, "%s: need Hq even, Hq %% Hkv == 0 and Hq/Hkv even (Hq=%d Hkv=%d)", fn,
                Hq, Hkv);
  if (sb < 0) return fail(DIFFATTN_ERR_SHAPE, "%s: negative logit stride", fn);
  if (B == 0 || Hq == 0) return ok();
  if (k8 && !(std::isfinite(k_scale) && k_scale > 0.f))
    return fail(DIFFATTN_ERR_SHAPE, "%s: key scale must be finite and positive", fn);
  if (!q || !k || !v || !lam_logits || !out) return fail(DIFFATTN_ERR_NULL, "%s: NULL pointer", fn);
  if (dt != DIFFATTN_BF16 || d != 128)
    return fail(DIFFATTN_ERR_UNSUPPORTED, "%s: bf16 with d = 128 only (got dtype %d, d=%d)", fn, (int)dt,
                d);
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return fail(DIFFATTN_ERR_ALIGN, "%s: tensors must be 16-byte aligned", fn);
  const int G = Hq / 2;
  const long long units = static_cast<long long>(B) * G;
  if (units * da::DecodeCfg<128, true>::MAX_CS * kMaxSplit > 0x7fffffffll)
    return fail(DIFFATTN_ERR_SHAPE, "%s: too many (batch, pair) units", fn);
  if (workspace != nullptr) {
    const size_t need = diffattn_v2_decode_workspace(B, Hq, d);
    if (workspace_bytes < need)
      return fail(DIFFATTN_ERR_SHAPE, "%s: workspace of %zu bytes, %zu needed (or pass NULL)", fn, workspace_bytes,
                  need);
    if ((reinterpret_cast<uintptr_t>(workspace) & 3u) != 0)
      return fail(DIFFATTN_ERR_ALIGN, "%s: workspace must be 4-byte aligned", fn);
  }
  int* status = nullptr;
  diffattn_status st = status_word(&status);
  if (st != DIFFATTN_OK) return st;
  da::DecodeParams p;
  memset(&p, 0, sizeof(p));
  const int bk = k8 ? da::DecodeCfg<128, true, true>::BK : da::DecodeCfg<128, true>::BK;  // keys per stage (box rows)
  const int nn = n > 0 ? n : 1;  // an empty cache still needs a valid map (no key is read)
  if ((st = k8 ? make_map_u8(&p.tm_k1, k, B, nn, Hkv, d, bk) : make_map(&p.tm_k1, k, B, nn, Hkv, d, bk)) !=
      DIFFATTN_OK)
    return st;
  p.k1_scale = p.k2_scale = k_scale;
  if ((st = make_map(&p.tm_v, v, B, nn, Hkv, d, bk)) != DIFFATTN_OK) return st;
  p.tm_k2 = p.tm_k1;
  p.q1 = static_cast<const __nv_bfloat16*>(q);
  p.q2 = p.q1;
  p.lens = lens;
  p.lam_logits = lam_logits;
  p.sb = sb;
  p.out = static_cast<__nv_bfloat16*>(out);
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.f / std::sqrt(static_cast<float>(d));
  p.scale_log2 = static_cast<float>(1.4426950408889634 * scale);
  p.norm_mult = 1.f;
  p.B = B;
  p.H = G;
  p.n = n;
  p.group = Hq / Hkv;
  p.status = status;
  const int cs = decode_cluster_size(units, n, bk);
  p.nsplit = 1;
  if (workspace != nullptr) {
    p.nsplit = decode_split(units, cs, n, bk);
    p.ws = static_cast<float*>(workspace);
  }
  cudaError_t e = da::launch_decode_v2_d128(p, k8, static_cast<int>(units), cs, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, fn);
  g_launches.fetch_add(1);
  return ok();
}

diffattn_status diffattn_v2_decode(diffattn_dtype dt, int B, int Hq, int Hkv, int n, int d, const void* q,
                                   const void* k, const void* v, const int* lens, const float* lam_logits,
                                   long long sb, float softmax_scale, void* out, void* workspace,
                                   size_t workspace_bytes, void* stream) {
  return decode_v2("diffattn_v2_decode", dt, B, Hq, Hkv, n, d, q, k, false, 1.f, v, lens, lam_logits, sb,
                   softmax_scale, out, workspace, workspace_bytes, stream);
}

diffattn_status diffattn_v2_decode_fp8k(int B, int Hq, int Hkv, int n, int d, const void* q, const void* k,
                                        float k_scale, const void* v, const int* lens, const float* lam_logits,
                                        long long sb, float softmax_scale, void* out, void* workspace,
                                        size_t workspace_bytes, void* stream) {
  return decode_v2("diffattn_v2_decode_fp8k", DIFFATTN_BF16, B, Hq, Hkv, n, d, q, k, true, k_scale, v, lens,
                   lam_logits, sb, softmax_scale, out, workspace, workspace_bytes, stream);
}

diffattn_status diffattn_v2_forward(diffattn_dtype dt, int B, int Hq, int Hkv, int n, int d, const void* q,
                                    const void* k, const void* v, const float* lam_logits, long long sb,
                                    long long st_, float softmax_scale, int causal, void* out, void* stream) {
  if (dt != DIFFATTN_F32 && dt != DIFFATTN_BF16) return fail(DIFFATTN_ERR_DTYPE, "diffattn_v2_forward: bad dtype %d", (int)dt);
  if (B < 0 || Hq < 0 || Hkv < 1 || n < 0 || d < 1)
    return fail(DIFFATTN_ERR_SHAPE, "diffattn_v2_forward: bad sizes B=%d Hq=%d Hkv=%d n=%d d=%d", B, Hq, Hkv, n, d);
  if (Hq % 2 != 0 || Hq % Hkv != 0 || (Hq / Hkv) % 2 != 0)
    return fail(DIFFATTN_ERR_SHAPE, "diffattn_v2_forward: need Hq even, Hq %% Hkv == 0 and Hq/Hkv even (Hq=%d Hkv=%d)",
                Hq, Hkv);
  if (sb < 0 || st_ < 0) return fail(DIFFATTN_ERR_SHAPE, "diffattn_v2_forward: negative logit stride");
  if (B == 0 || Hq == 0 || n == 0) return ok();
  if (!q || !k || !v || !lam_logits || !out) return fail(DIFFATTN_ERR_NULL, "diffattn_v2_forward: NULL pointer");
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.f / std::sqrt(static_cast<float>(d));
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* status = nullptr;
  diffattn_status st = status_word(&status);
  if (st != DIFFATTN_OK) return st;
  const int G = Hq / 2;

  if (dt == DIFFATTN_F32) {
    if (d > da::kSimtMaxD) return fail(DIFFATTN_ERR_UNSUPPORTED, "diffattn_v2_forward: f32 needs d <= 128");
    da::SimtParams p{};
    p.q1 = p.q2 = static_cast<const float*>(q);
    p.k1 = p.k2 = static_cast<const float*>(k);
    p.v = static_cast<const float*>(v);
    p.out = static_cast<float*>(out);
    p.lam_logits = lam_logits;
    p.sb = sb;
    p.st = st_;
    p.scale = scale;
    p.norm_mult = 1.f;
    p.eps = 0.f;
    p.B = B;
    p.n = n;
    p.d = d;
    p.dv = d;
    p.causal = causal ? 1 : 0;
    p.v2 = 1;
    p.heads_q = Hq;
    p.heads_kv = Hkv;
    p.units_per_batch = G;
    p.group = Hq / Hkv;
    p.rows_total = static_cast<long long>(B) * G * n;
    cudaError_t e = da::launch_simt_f32(p, s);
    if (e != cudaSuccess) return cuda_fail(e, "diffattn_v2_forward (f32) launch");
    g_launches.fetch_add(1);
    return ok();
  }

  if (d != 128) return fail(DIFFATTN_ERR_UNSUPPORTED, "diffattn_v2_forward: bf16 needs d = 128 (got %d)", d);
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return fail(DIFFATTN_ERR_ALIGN, "diffattn_v2_forward: bf16 tensors must be 16-byte aligned");
  const long long Hqd = static_cast<long long>(Hq) * d, Hkvd = static_cast<long long>(Hkv) * d;
  const QKVViews x{q, q, k, k, v, d, Hqd, d, Hkvd, d, Hkvd};
  if ((st = forward_v2_bf16("diffattn_v2_forward (bf16)", x, B, Hq, Hkv, n, d, lam_logits, sb, st_, scale, causal,
                            out, status, s)) != DIFFATTN_OK)
    return st;
  return ok();
}

// ---------------------------------------------------------------- projections and the attention layer
}  // extern "C"

namespace {

constexpr int kGemmGroupM = 16;  // row blocks per group of the persistent tile walk

// C = A B^T on the tensor cores.  A [M, K] (row stride lda), B [N, K] (row
// stride ldb) bf16; columns [0, n_main) of C go to `c` in bf16 (row stride
// ldc), columns [n_main, N) to `c2` in fp32 (row stride ldc2).  Arguments
// validated by the caller (K >= 1, strides and pointers 16-byte aligned).
diffattn_status gemm_bf16(const char* fn, const void* a, long long lda, const void* b, long long ldb, int M, int N,
                          int K, void* c, long long ldc, int n_main, float* c2, long long ldc2, int* status,
                          cudaStream_t s) {
  da::GemmParams p;
  memset(&p, 0, sizeof(p));
  diffattn_status st;
  if ((st = make_map_2d(&p.tm_a, a, M, K, lda, da::kGemmBM)) != DIFFATTN_OK) return st;
  if ((st = make_map_2d(&p.tm_b, b, N, K, ldb, da::kGemmBN)) != DIFFATTN_OK) return st;
  p.c = static_cast<__nv_bfloat16*>(c);
  p.c2 = c2;
  p.ldc = ldc;
  p.ldc2 = ldc2;
  p.M = M;
  p.N = N;
  p.K = K;
  p.n_main = n_main;
  p.tiles_m = (M + da::kGemmBM - 1) / da::kGemmBM;
  p.tiles_n = (N + da::kGemmBN - 1) / da::kGemmBN;
  p.group_m = kGemmGroupM;
  p.status = status;
  const long long tiles = static_cast<long long>(p.tiles_m) * p.tiles_n;
  if (tiles > 0x7fffffffll) return fail(DIFFATTN_ERR_SHAPE, "%s: too many output tiles", fn);
  cudaError_t e = da::launch_gemm_bf16(p, static_cast<int>(persistent_grid(tiles)), s);
  if (e != cudaSuccess) return cuda_fail(e, fn);
  g_launches.fetch_add(1);
  return DIFFATTN_OK;
}

// Byte offset of element `elems` of a bf16 buffer.
const void* bf16_at(const void* base, long long elems) { return static_cast<const uint8_t*>(base) + 2 * elems; }

}  // namespace

extern "C" {

diffattn_status diffattn_projection(int M, int N, int K, const void* a, const void* w, void* c, void* stream) {
  const char* fn = "diffattn_projection";
  if (M < 0 || N < 0 || K < 1) return fail(DIFFATTN_ERR_SHAPE, "%s: bad sizes M=%d N=%d K=%d", fn, M, N, K);
  if (M == 0 || N == 0) return ok();
  if (!a || !w || !c) return fail(DIFFATTN_ERR_NULL, "%s: NULL pointer", fn);
  if (K % 8 != 0 || N % 8 != 0)
    return fail(DIFFATTN_ERR_SHAPE, "%s: K and N must be multiples of 8 (16-byte rows; got K=%d N=%d)", fn, K, N);
  if (!aligned16(a) || !aligned16(w) || !aligned16(c)) return fail(DIFFATTN_ERR_ALIGN, "%s: 16-byte alignment", fn);
  int* status = nullptr;
  diffattn_status st = status_word(&status);
  if (st != DIFFATTN_OK) return st;
  if ((st = gemm_bf16(fn, a, K, w, K, M, N, K, c, N, N, nullptr, 0, status, static_cast<cudaStream_t>(stream))) !=
      DIFFATTN_OK)
    return st;
  return ok();
}

size_t diffattn_layer_workspace(int B, int n, int H, int d) {
  if (B < 0 || n < 0 || H < 0 || d < 1) return 0;
  const size_t M = static_cast<size_t>(B) * n, Hd = static_cast<size_t>(H) * d;
  return round256(M * 6 * Hd * 2) + round256(M * 2 * Hd * 2) + 256;
}

diffattn_status diffattn_layer_forward(int B, int n, int D, int H, int d, const void* x, const void* w_qkv,
                                       const void* w_o, const float* lq1, const float* lk1, const float* lq2,
                                       const float* lk2, float lambda_init, const float* gamma, float eps,
                                       int causal, void* out, void* workspace, size_t workspace_bytes,
                                       void* stream) {
  const char* fn = "diffattn_layer_forward";
  if (B < 0 || n < 0 || D < 1 || H < 1 || d < 1)
    return fail(DIFFATTN_ERR_SHAPE, "%s: bad sizes B=%d n=%d D=%d H=%d d=%d", fn, B, n, D, H, d);
  if (d != 64 && d != 128) return fail(DIFFATTN_ERR_UNSUPPORTED, "%s: d must be 64 or 128 (got %d)", fn, d);
  if (D % 8 != 0) return fail(DIFFATTN_ERR_SHAPE, "%s: D must be a multiple of 8 (got %d)", fn, D);
  if (B == 0 || n == 0) return ok();
  if (!x || !w_qkv || !w_o || !lq1 || !lk1 || !lq2 || !lk2 || !out || !workspace)
    return fail(DIFFATTN_ERR_NULL, "%s: NULL pointer", fn);
  if (!std::isfinite(lambda_init)) return fail(DIFFATTN_ERR_SHAPE, "%s: lambda_init not finite", fn);
  if (!aligned16(x) || !aligned16(w_qkv) || !aligned16(w_o) || !aligned16(out))
    return fail(DIFFATTN_ERR_ALIGN, "%s: x, w_qkv, w_o and out must be 16-byte aligned", fn);
  const size_t need = diffattn_layer_workspace(B, n, H, d);
  if (workspace_bytes < need)
    return fail(DIFFATTN_ERR_SHAPE, "%s: workspace of %zu bytes, %zu needed", fn, workspace_bytes, need);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(DIFFATTN_ERR_ALIGN, "%s: workspace not 256-byte aligned", fn);
  const long long M = static_cast<long long>(B) * n, Hd = static_cast<long long>(H) * d;
  if (M > 0x7fffffffll || 6 * Hd > 0x7fffffffll) return fail(DIFFATTN_ERR_SHAPE, "%s: too large", fn);
  if (eps <= 0.f) eps = 1e-5f;
  int* status = nullptr;
  diffattn_status st = status_word(&status);
  if (st != DIFFATTN_OK) return st;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* qkv = ws;                                                      // [M, 6 H d]: q | k | v per token
  void* y = ws + round256(static_cast<size_t>(M) * 6 * Hd * 2);        // [M, 2 H d]: normalised heads
  float* lam = reinterpret_cast<float*>(static_cast<uint8_t*>(y) + round256(static_cast<size_t>(M) * 2 * Hd * 2));
  // 1. X [W^Q | W^K | W^V]: per token the 2d columns of head i of each
  //    projection hold Q_1 (first d) and Q_2 (last d), K_1 and K_2, and V.
  if ((st = gemm_bf16(fn, x, D, w_qkv, D, static_cast<int>(M), static_cast<int>(6 * Hd), D, qkv, 6 * Hd,
                      static_cast<int>(6 * Hd), nullptr, 0, status, s)) != DIFFATTN_OK)
    return st;
  // 2. lambda from its four vectors (one warp).
  cudaError_t e = da::launch_lambda_reparam(lq1, lk1, lq2, lk2, d, lambda_init, lam, s);
  if (e != cudaSuccess) return cuda_fail(e, "diffattn_layer_forward: lambda_reparam launch");
  g_launches.fetch_add(1);
  // 3. the operator with the per-head norm, reading the projections in place
  //    through strided tensor maps.
  const QKVViews v{qkv, bf16_at(qkv, d), bf16_at(qkv, 2 * Hd), bf16_at(qkv, 2 * Hd + d), bf16_at(qkv, 4 * Hd),
                   2 * d, 6 * Hd, 2 * d, 6 * Hd, 2 * d, 6 * Hd};
  if ((st = forward_v1_bf16(fn, v, B, H, static_cast<int>(n), d, lam, lambda_init, gamma, eps, causal, y, status,
                            s)) != DIFFATTN_OK)
    return st;
  // 4. Concat(heads) W^O.
  if ((st = gemm_bf16(fn, y, 2 * Hd, w_o, 2 * Hd, static_cast<int>(M), D, static_cast<int>(2 * Hd), out, D, D,
                      nullptr, 0, status, s)) != DIFFATTN_OK)
    return st;
  return ok();
}

size_t diffattn_v2_layer_workspace(int B, int n, int Hq, int Hkv, int d) {
  if (B < 0 || n < 0 || Hq < 0 || Hkv < 0 || d < 1) return 0;
  const size_t M = static_cast<size_t>(B) * n, G = static_cast<size_t>(Hq) / 2;
  const size_t nq = (static_cast<size_t>(Hq) + 2 * static_cast<size_t>(Hkv)) * d;
  return round256(M * nq * 2) + round256(M * G * 4) + round256(M * G * d * 2);
}

diffattn_status diffattn_v2_layer_forward(int B, int n, int D, int Hq, int Hkv, int d, const void* x,
                                          const void* w_qkvl, const void* w_o, int causal, void* out,
                                          void* workspace, size_t workspace_bytes, void* stream) {
  const char* fn = "diffattn_v2_layer_forward";
  if (B < 0 || n < 0 || D < 1 || Hq < 2 || Hkv < 1 || d < 1)
    return fail(DIFFATTN_ERR_SHAPE, "%s: bad sizes B=%d n=%d D=%d Hq=%d Hkv=%d d=%d", fn, B, n, D, Hq, Hkv, d);
  if (Hq % 2 != 0 || Hq % Hkv != 0 || (Hq / Hkv) % 2 != 0)
    return fail(DIFFATTN_ERR_SHAPE, "%s: need Hq even, Hq %% Hkv == 0 and Hq/Hkv even (Hq=%d Hkv=%d)", fn, Hq, Hkv);
  if (d != 128) return fail(DIFFATTN_ERR_UNSUPPORTED, "%s: d must be 128 (got %d)", fn, d);
  if (D % 8 != 0) return fail(DIFFATTN_ERR_SHAPE, "%s: D must be a multiple of 8 (got %d)", fn, D);
  if (B == 0 || n == 0) return ok();
  if (!x || !w_qkvl || !w_o || !out || !workspace) return fail(DIFFATTN_ERR_NULL, "%s: NULL pointer", fn);
  if (!aligned16(x) || !aligned16(w_qkvl) || !aligned16(w_o) || !aligned16(out))
    return fail(DIFFATTN_ERR_ALIGN, "%s: x, w_qkvl, w_o and out must be 16-byte aligned", fn);
  const size_t need = diffattn_v2_layer_workspace(B, n, Hq, Hkv, d);
  if (workspace_bytes < need)
    return fail(DIFFATTN_ERR_SHAPE, "%s: workspace of %zu bytes, %zu needed", fn, workspace_bytes, need);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(DIFFATTN_ERR_ALIGN, "%s: workspace not 256-byte aligned", fn);
  const long long M = static_cast<long long>(B) * n, G = Hq / 2;
  const long long nq = (static_cast<long long>(Hq) + 2ll * Hkv) * d;
  if (M > 0x7fffffffll || nq + G > 0x7fffffffll) return fail(DIFFATTN_ERR_SHAPE, "%s: too large", fn);
  int* status = nullptr;
  diffattn_status st = status_word(&status);
  if (st != DIFFATTN_OK) return st;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* qkv = ws;                                                                   // [M, (Hq + 2 Hkv) d]
  float* logits = reinterpret_cast<float*>(ws + round256(static_cast<size_t>(M) * nq * 2));  // [M, Hq / 2] fp32
  void* y = reinterpret_cast<uint8_t*>(logits) + round256(static_cast<size_t>(M) * G * 4);   // [M, Hq / 2 d]
  // 1. X [W^Q | W^K | W^V | W^lambda]: q, k, v in bf16, the pairs' lambda logits in fp32.
  if ((st = gemm_bf16(fn, x, D, w_qkvl, D, static_cast<int>(M), static_cast<int>(nq + G), D, qkv, nq,
                      static_cast<int>(nq), logits, G, status, s)) != DIFFATTN_OK)
    return st;
  // 2. the V2 operator, per token and pair logits (strides n G, G).
  const QKVViews v{qkv, qkv, bf16_at(qkv, static_cast<long long>(Hq) * d), bf16_at(qkv, static_cast<long long>(Hq) * d),
                   bf16_at(qkv, (static_cast<long long>(Hq) + Hkv) * d), d, nq, d, nq, d, nq};
  const float scale = 1.f / std::sqrt(static_cast<float>(d));
  if ((st = forward_v2_bf16(fn, v, B, Hq, Hkv, static_cast<int>(n), d, logits, static_cast<long long>(n) * G, G, scale,
                            causal, y, status, s)) != DIFFATTN_OK)
    return st;
  // 3. Concat(pairs) W^O.
  if ((st = gemm_bf16(fn, y, G * d, w_o, G * d, static_cast<int>(M), D, static_cast<int>(G * d), out, D, D, nullptr,
                      0, status, s)) != DIFFATTN_OK)
    return st;
  return ok();
}

// ---- backward on the tensor cores (bf16 inputs, fp32 gradients)
}  // extern "C"

namespace {

// V1 (d = 64): statistics pass, dK/dV/dQ kernel, reduction of dlambda and dgamma.
// A training forward's saved statistics: lse [2][rows] fp32, then O_1 and O_2
// in bf16, each in 128-token tiles: [units of all batches][tiles][4 channel
// blocks][128 rows][32 channels] (the layout the forward's epilogue writes
// with whole 64-byte rows per thread), 256-byte aligned parts.  `units` =
// batches x heads (V1) or head pairs (V2); `n` tokens.
struct SavedFwd {
  const float* lse;
  const __nv_bfloat16* o1;
  const __nv_bfloat16* o2;
};

size_t saved_fwd_bytes(size_t units, size_t n, size_t dv) {
  const size_t rows = units * n, padded = units * ((n + 127) / 128) * 128;
  return round256(2 * rows * 4) + 2 * round256(padded * dv * 2);
}

SavedFwd saved_fwd_views(const void* saved, size_t units, size_t n, size_t dv) {
  const size_t rows = units * n, padded = units * ((n + 127) / 128) * 128;
  const uint8_t* b = static_cast<const uint8_t*>(saved);
  SavedFwd v;
  v.lse = reinterpret_cast<const float*>(b);
  v.o1 = reinterpret_cast<const __nv_bfloat16*>(b + round256(2 * rows * 4));
  v.o2 = reinterpret_cast<const __nv_bfloat16*>(b + round256(2 * rows * 4) + round256(padded * dv * 2));
  return v;
}

diffattn_status backward_v1_tc(int B, int H, int n, const void* q1, const void* q2, const void* k1, const void* k2,
                               const void* v, const float* lambda, float lambda_init, const float* gamma, float eps,
                               int causal, const void* dy, void* dq1, void* dq2, void* dk1, void* dk2, void* dv,
                               float* dlambda, float* dgamma, uint8_t* ws, int* status, cudaStream_t s,
                               const SavedFwd* saved = nullptr) {
  const char* fn = saved ? "diffattn_backward_saved" : "diffattn_backward (bf16)";
  constexpr int d = 64, dv_w = 128;
  const size_t R = static_cast<size_t>(B) * H * n;
  const int nt = (n + 127) / 128;
  const long long stats_grid = static_cast<long long>(nt) * B * H;
  if (stats_grid > 0x7fffffffll) return fail(DIFFATTN_ERR_SHAPE, "%s: too many tiles", fn);
  __nv_bfloat16* ws_do = reinterpret_cast<__nv_bfloat16*>(ws);
  float* ws_row = reinterpret_cast<float*>(ws + round256(R * dv_w * 2));
  float* ws_dg = reinterpret_cast<float*>(ws + round256(R * dv_w * 2) + round256(6 * R * 4));
  float* ws_dl = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ws_dg) +
                                          round256(static_cast<size_t>(stats_grid) * dv_w * 4));
  const float sc = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d)));
  diffattn_status st;
  // 1. statistics: the forward's maps, dy in; lse, Delta, shares, dO and dgamma shares out
  da::TwoPassParams p;
  memset(&p, 0, sizeof(p));
  if ((st = make_map(&p.tm_q1, q1, B, n, H, d, 128)) != DIFFATTN_OK) return st;
  if ((st = make_map(&p.tm_q2, q2, B, n, H, d, 128)) != DIFFATTN_OK) return st;
  if ((st = make_map(&p.tm_k1, k1, B, n, H, d, 128)) != DIFFATTN_OK) return st;
  if ((st = make_map(&p.tm_k2, k2, B, n, H, d, 128)) != DIFFATTN_OK) return st;
  if ((st = make_map(&p.tm_v, v, B, n, H, dv_w, 64)) != DIFFATTN_OK) return st;
  p.lambda = lambda;
  p.gamma = gamma;
  p.scale_log2 = sc;
  p.scale2_log2 = sc;
  p.norm_mult = 1.f - lambda_init;
  p.eps = eps;
  p.B = B;
  p.n = n;
  p.causal = causal ? 1 : 0;
  p.units_per_batch = H;
  p.group = 1;
  p.num_q_tiles = nt;
  p.order = pick_order(static_cast<long long>(B) * H, n, (2 * d + dv_w) * 2);
  p.status = status;
  p.dy = static_cast<const __nv_bfloat16*>(dy);
  p.dO = ws_do;
  p.row = ws_row;
  p.dgp = ws_dg;
  p.dlam_part = ws_dl;
  p.rows = static_cast<long long>(R);
  cudaError_t e = cudaMemsetAsync(dq1, 0, R * d * 4, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(dq2, 0, R * d * 4, s);
  if (e != cudaSuccess) return cuda_fail(e, "diffattn_backward: clearing dq");
  int row_ctas = static_cast<int>(stats_grid);
  if (saved) {  // the per-row results from the saved statistics instead of a second forward
    da::BwdPrepParams q{};
    q.dy = p.dy;
    q.o1 = saved->o1;
    q.o2 = saved->o2;
    q.lse = saved->lse;
    q.lambda = lambda;
    q.gamma = gamma;
    q.norm_mult = 1.f - lambda_init;
    q.eps = eps;
    q.B = B;
    q.n = n;
    q.units = H;
    q.rows = static_cast<long long>(R);
    q.dO = ws_do;
    q.row = ws_row;
    q.dgp = ws_dg;
    q.dlam_part = ws_dl;
    row_ctas = static_cast<int>((R + da::kPrepRowsPerCta - 1) / da::kPrepRowsPerCta);  // <= stats_grid
    if ((e = da::launch_bwd_prep(q, false, row_ctas, s)) != cudaSuccess) return cuda_fail(e, fn);
  } else if ((e = da::launch_bwd_stats(p, false, static_cast<int>(stats_grid), s)) != cudaSuccess) {
    return cuda_fail(e, fn);
  }
  // 2. dK, dV, dQ
  da::BwdTcParams t;
  memset(&t, 0, sizeof(t));
  if ((st = make_map(&t.tm_q1, q1, B, n, H, d, 128)) != DIFFATTN_OK) return st;
  if ((st = make_map(&t.tm_q2, q2, B, n, H, d, 128)) != DIFFATTN_OK) return st;
  if ((st = make_map(&t.tm_k1, k1, B, n, H, d, 128)) != DIFFATTN_OK) return st;
  if ((st = make_map(&t.tm_k2, k2, B, n, H, d, 128)) != DIFFATTN_OK) return st;
  if ((st = make_map(&t.tm_v, v, B, n, H, dv_w, 128)) != DIFFATTN_OK) return st;
  if ((st = make_map(&t.tm_do, ws_do, B, n, H, dv_w, 128)) != DIFFATTN_OK) return st;
  if ((st = make_map_f32(&t.tm_dq1, dq1, B, n, H, d, 128)) != DIFFATTN_OK) return st;
  if ((st = make_map_f32(&t.tm_dq2, dq2, B, n, H, d, 128)) != DIFFATTN_OK) return st;
  t.row = ws_row;
  t.lambda = lambda;
  t.dq1 = static_cast<float*>(dq1);
  t.dq2 = static_cast<float*>(dq2);
  t.dk1 = static_cast<float*>(dk1);
  t.dk2 = static_cast<float*>(dk2);
  t.dv = static_cast<float*>(dv);
  t.scale_log2 = sc;
  t.scale = 1.f / std::sqrt(static_cast<float>(d));
  t.B = B;
  t.n = n;
  t.causal = causal ? 1 : 0;
  t.heads_kv = H;
  t.units = H;
  t.group = 1;
  t.num_tiles = nt;
  t.rows = static_cast<long long>(R);
  t.status = status;
  if ((e = da::launch_bwd_tc(t, false, static_cast<int>(stats_grid), s)) != cudaSuccess) return cuda_fail(e, fn);
  // 3. dlambda and dgamma in a fixed order
  da::BwdParams r{};
  r.row = ws_row;
  r.dgp = ws_dg;
  r.dlam_parts = ws_dl;
  r.dlambda = dlambda;
  r.dgamma = dgamma;
  r.B = B;
  r.n = n;
  r.d = d;
  r.dvw = dv_w;
  r.v2 = 0;
  r.units = H;
  r.rows = static_cast<long long>(R);
  r.n_row_ctas = row_ctas;
  if ((e = da::launch_bwd_reduce(r, s)) != cudaSuccess) return cuda_fail(e, fn);
  g_launches.fetch_add(4);
  return DIFFATTN_OK;
}

// V2 (d = 128): statistics pass (dlogits of per-token logits written there), dK/dV/dQ
// kernel, reduction of the logit gradients shared by tokens.
diffattn_status backward_v2_tc(int B, int Hq, int Hkv, int n, const void* q, const void* k, const void* v,
                               const float* lam_logits, long long sb, long long st_, float scale, int causal,
                               const void* dy, void* dq, void* dk, void* dv, float* dlogits, bool dense, uint8_t* ws,
                               int* status, cudaStream_t s, const SavedFwd* saved = nullptr) {
  const char* fn = saved ? "diffattn_v2_backward_saved" : "diffattn_v2_backward (bf16)";
  constexpr int d = 128;
  const int G = Hq / 2;
  const size_t R = static_cast<size_t>(B) * G * n;
  const int nt = (n + 127) / 128;
  const long long stats_grid = static_cast<long long>(nt) * B * G;
  const long long tc_grid = static_cast<long long>(nt) * B * Hkv;
  if (stats_grid > 0x7fffffffll) return fail(DIFFATTN_ERR_SHAPE, "%s: too many tiles", fn);
  float* ws_row = reinterpret_cast<float*>(ws);
  const float sc = static_cast<float>(1.4426950408889634 * scale);
  diffattn_status st;
  da::TwoPassParams p;
  memset(&p, 0, sizeof(p));
  if ((st = make_map(&p.tm_q1, q, B, n, Hq, d, 128)) != DIFFATTN_OK) return st;
  p.tm_q2 = p.tm_q1;
  if ((st = make_map(&p.tm_k1, k, B, n, Hkv, d, 128)) != DIFFATTN_OK) return st;
  p.tm_k2 = p.tm_k1;
  if ((st = make_map(&p.tm_v, v, B, n, Hkv, d, 128)) != DIFFATTN_OK) return st;
  p.lam_logits = lam_logits;
  p.sb = sb;
  p.st = st_;
  p.scale_log2 = sc;
  p.scale2_log2 = sc;
  p.norm_mult = 1.f;
  p.B = B;
  p.n = n;
  p.causal = causal ? 1 : 0;
  p.units_per_batch = G;
  p.group = Hq / Hkv;
  p.num_q_tiles = nt;
  p.order = pick_order(static_cast<long long>(B) * Hkv, n, 2 * d * 2);
  p.status = status;
  p.dy = static_cast<const __nv_bfloat16*>(dy);
  p.row = ws_row;
  p.dlogits_dense = dense ? dlogits : nullptr;
  p.rows = static_cast<long long>(R);
  cudaError_t e = cudaMemsetAsync(dq, 0, static_cast<size_t>(B) * n * Hq * d * 4, s);
  if (e != cudaSuccess) return cuda_fail(e, "diffattn_v2_backward: clearing dq");
  if (saved) {  // the per-row results from the saved statistics instead of a second forward
    da::BwdPrepParams q{};
    q.dy = p.dy;
    q.o1 = saved->o1;
    q.o2 = saved->o2;
    q.lse = saved->lse;
    q.lam_logits = lam_logits;
    q.sb = sb;
    q.st = st_;
    q.B = B;
    q.n = n;
    q.units = G;
    q.rows = static_cast<long long>(R);
    q.row = ws_row;
    q.dlogits_dense = p.dlogits_dense;
    const int row_ctas = static_cast<int>((R + da::kPrepRowsPerCta - 1) / da::kPrepRowsPerCta);
    if ((e = da::launch_bwd_prep(q, true, row_ctas, s)) != cudaSuccess) return cuda_fail(e, fn);
  } else if ((e = da::launch_bwd_stats(p, true, static_cast<int>(stats_grid), s)) != cudaSuccess) {
    return cuda_fail(e, fn);
  }
  da::BwdTcParams t;
  memset(&t, 0, sizeof(t));
  if ((st = make_map(&t.tm_q1, q, B, n, Hq, d, 128)) != DIFFATTN_OK) return st;
  t.tm_q2 = t.tm_q1;
  if ((st = make_map(&t.tm_k1, k, B, n, Hkv, d, 128)) != DIFFATTN_OK) return st;
  t.tm_k2 = t.tm_k1;
  if ((st = make_map(&t.tm_v, v, B, n, Hkv, d, 128)) != DIFFATTN_OK) return st;
  if ((st = make_map(&t.tm_do, dy, B, n, G, d, 128)) != DIFFATTN_OK) return st;
  if ((st = make_map_f32(&t.tm_dq1, dq, B, n, Hq, d, 128)) != DIFFATTN_OK) return st;
  t.tm_dq2 = t.tm_dq1;
  t.row = ws_row;
  t.dq1 = t.dq2 = static_cast<float*>(dq);
  t.dk1 = static_cast<float*>(dk);
  t.dv = static_cast<float*>(dv);
  t.scale_log2 = sc;
  t.scale = scale;
  t.B = B;
  t.n = n;
  t.causal = causal ? 1 : 0;
  t.heads_kv = Hkv;
  t.units = G;
  t.group = Hq / Hkv;
  t.num_tiles = nt;
  t.rows = static_cast<long long>(R);
  t.status = status;
  if ((e = da::launch_bwd_tc(t, true, static_cast<int>(tc_grid), s)) != cudaSuccess) return cuda_fail(e, fn);
  int launches = 3;
  if (!dense) {
    da::BwdParams r{};
    r.row = ws_row;
    r.dlogits = dlogits;
    r.sb = sb;
    r.B = B;
    r.n = n;
    r.d = d;
    r.dvw = d;
    r.v2 = 1;
    r.units = G;
    r.rows = static_cast<long long>(R);
    r.n_logit_outs = sb == 0 ? G : B * G;
    if ((e = da::launch_bwd_reduce(r, s)) != cudaSuccess) return cuda_fail(e, fn);
    ++launches;
  }
  g_launches.fetch_add(launches);
  return DIFFATTN_OK;
}

}  // namespace

extern "C" {

// ---- backward (fp32, V1)
static size_t bwd_rows(int B, int H, int n) { return static_cast<size_t>(B) * H * n; }
constexpr size_t kBwdRowSlots = 6;  // per row: lse_1, lse_2, D_1, D_2, dlambda / dlogit share, coefficient
static size_t bwd_row_ctas(int B, int H, int n) {
  return static_cast<size_t>(B) * H * ((static_cast<size_t>(n) + da::kSimtRows - 1) / da::kSimtRows);
}

size_t diffattn_backward_workspace(int B, int H, int n, int d) {
  if (B < 0 || H < 0 || n < 0 || d < 1) return 0;
  const size_t R = bwd_rows(B, H, n), dv = 2 * static_cast<size_t>(d);
  return round256(R * dv * 4) + round256(kBwdRowSlots * R * 4) + round256(bwd_row_ctas(B, H, n) * dv * 4);
}

diffattn_status diffattn_backward(diffattn_dtype dt, int B, int H, int n, int d, const void* q1, const void* q2,
                                  const void* k1, const void* k2, const void* v, const float* lambda,
                                  float lambda_init, const float* gamma, float eps, int causal, const void* dy,
                                  void* dq1, void* dq2, void* dk1, void* dk2, void* dv, float* dlambda,
                                  float* dgamma, void* workspace, size_t workspace_bytes, void* stream) {
  if (dt != DIFFATTN_F32 && dt != DIFFATTN_BF16)
    return fail(DIFFATTN_ERR_DTYPE, "diffattn_backward: bad dtype %d", (int)dt);
  if (B < 0 || H < 0 || n < 0 || d < 1)
    return fail(DIFFATTN_ERR_SHAPE, "diffattn_backward: bad sizes B=%d H=%d n=%d d=%d", B, H, n, d);
  if ((dt == DIFFATTN_F32 && d > da::kSimtMaxD) || (dt == DIFFATTN_BF16 && d != 64))
    return fail(DIFFATTN_ERR_UNSUPPORTED, "diffattn_backward: f32 with d <= 128 or bf16 with d = 64 (got dtype %d, d=%d)",
                (int)dt, d);
  if (!dlambda) return fail(DIFFATTN_ERR_NULL, "diffattn_backward: NULL dlambda");
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int dvw = 2 * d;
  if (B == 0 || H == 0 || n == 0) {  // no rows: dlambda = 0, dgamma = 0
    cudaError_t e = cudaMemsetAsync(dlambda, 0, sizeof(float), s);
    if (e == cudaSuccess && dgamma) e = cudaMemsetAsync(dgamma, 0, dvw * sizeof(float), s);
    if (e != cudaSuccess) return cuda_fail(e, "diffattn_backward: clearing dlambda / dgamma");
    return ok();
  }
  if (!q1 || !q2 || !k1 || !k2 || !v || !lambda || !dy || !dq1 || !dq2 || !dk1 || !dk2 || !dv || !workspace)
    return fail(DIFFATTN_ERR_NULL, "diffattn_backward: NULL pointer");
  if (!std::isfinite(lambda_init)) return fail(DIFFATTN_ERR_SHAPE, "diffattn_backward: lambda_init not finite");
  const size_t need = diffattn_backward_workspace(B, H, n, d);
  if (workspace_bytes < need)
    return fail(DIFFATTN_ERR_SHAPE, "diffattn_backward: workspace of %zu bytes, need %zu", workspace_bytes, need);
  if (!aligned16(workspace)) return fail(DIFFATTN_ERR_ALIGN, "diffattn_backward: workspace must be 16-byte aligned");
  const long long nqb8 = (static_cast<long long>(n) + da::kSimtRows - 1) / da::kSimtRows;
  if (static_cast<long long>(B) * H * nqb8 > 0x7fffffffll)
    return fail(DIFFATTN_ERR_SHAPE, "diffattn_backward: too many (batch, head, row block) units");
  if (eps <= 0.f) eps = 1e-5f;
  if (dt == DIFFATTN_BF16) {
    if (!aligned16(q1) || !aligned16(q2) || !aligned16(k1) || !aligned16(k2) || !aligned16(v) || !aligned16(dy) ||
        !aligned16(dq1) || !aligned16(dq2) || !aligned16(dk1) || !aligned16(dk2) || !aligned16(dv))
      return fail(DIFFATTN_ERR_ALIGN, "diffattn_backward: bf16 path needs 16-byte aligned tensors");
    int* status = nullptr;
    diffattn_status st = status_word(&status);
    if (st != DIFFATTN_OK) return st;
    if ((st = backward_v1_tc(B, H, n, q1, q2, k1, k2, v, lambda, lambda_init, gamma, eps, causal, dy, dq1, dq2, dk1,
                             dk2, dv, dlambda, dgamma, static_cast<uint8_t*>(workspace), status, s)) != DIFFATTN_OK)
      return st;
    return ok();
  }
  const size_t R = bwd_rows(B, H, n);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* ws_do = reinterpret_cast<float*>(ws);
  float* ws_row = reinterpret_cast<float*>(ws + round256(R * dvw * 4));
  float* ws_dg = reinterpret_cast<float*>(ws + round256(R * dvw * 4) + round256(kBwdRowSlots * R * 4));

  da::SimtParams rp{};
  rp.q1 = static_cast<const float*>(q1);
  rp.q2 = static_cast<const float*>(q2);
  rp.k1 = static_cast<const float*>(k1);
  rp.k2 = static_cast<const float*>(k2);
  rp.v = static_cast<const float*>(v);
  rp.lambda = lambda;
  rp.gamma = gamma;
  rp.scale = 1.f / std::sqrt(static_cast<float>(d));
  rp.norm_mult = 1.f - lambda_init;
  rp.eps = eps;
  rp.B = B;
  rp.n = n;
  rp.d = d;
  rp.dv = dvw;
  rp.causal = causal ? 1 : 0;
  rp.v2 = 0;
  rp.heads_q = rp.heads_kv = rp.units_per_batch = H;
  rp.group = 1;
  rp.rows_total = static_cast<long long>(R);
  da::SimtBwdExtra rx{};
  rx.dy = static_cast<const float*>(dy);
  rx.ws_do = ws_do;
  rx.ws_row = ws_row;
  rx.ws_dgamma = ws_dg;

  da::BwdParams p{};
  p.q1 = rp.q1;
  p.q2 = rp.q2;
  p.k1 = rp.k1;
  p.k2 = rp.k2;
  p.v = rp.v;
  p.dO = ws_do;
  p.row = ws_row;
  p.dgp = ws_dg;
  p.lambda = lambda;
  p.dq1 = static_cast<float*>(dq1);
  p.dq2 = static_cast<float*>(dq2);
  p.dk1 = static_cast<float*>(dk1);
  p.dk2 = static_cast<float*>(dk2);
  p.dv = static_cast<float*>(dv);
  p.dlambda = dlambda;
  p.dgamma = dgamma;
  p.scale = rp.scale;
  p.B = B;
  p.n = n;
  p.d = d;
  p.dvw = dvw;
  p.causal = rp.causal;
  p.v2 = 0;
  p.heads_q = p.heads_kv = p.units = H;
  p.group = 1;
  p.rows = static_cast<long long>(R);
  p.n_row_ctas = static_cast<int>(bwd_row_ctas(B, H, n));
  cudaError_t e = da::launch_simt_bwd_rows(rp, rx, s);
  if (e == cudaSuccess) e = da::launch_backward_f32(p, s);
  if (e != cudaSuccess) return cuda_fail(e, "diffattn_backward launch");
  g_launches.fetch_add(4);
  return ok();
}

size_t diffattn_v2_backward_workspace(int B, int Hq, int n, int d) {
  if (B < 0 || Hq < 0 || n < 0 || d < 1) return 0;
  const size_t R = bwd_rows(B, Hq / 2, n);
  return round256(R * static_cast<size_t>(d) * 4) + round256(kBwdRowSlots * R * 4);
}

diffattn_status diffattn_v2_backward(diffattn_dtype dt, int B, int Hq, int Hkv, int n, int d, const void* q,
                                     const void* k, const void* v, const float* lam_logits, long long sb,
                                     long long st, float softmax_scale, int causal, const void* dy, void* dq,
                                     void* dk, void* dv, float* dlogits, void* workspace, size_t workspace_bytes,
                                     void* stream) {
  if (dt != DIFFATTN_F32 && dt != DIFFATTN_BF16)
    return fail(DIFFATTN_ERR_DTYPE, "diffattn_v2_backward: bad dtype %d", (int)dt);
  if (B < 0 || Hq < 0 || Hkv < 1 || n < 0 || d < 1)
    return fail(DIFFATTN_ERR_SHAPE, "diffattn_v2_backward: bad sizes B=%d Hq=%d Hkv=%d n=%d d=%d", B, Hq, Hkv, n, d);
  if (Hq % 2 != 0 || Hq % Hkv != 0 || (Hq / Hkv) % 2 != 0)
    return fail(DIFFATTN_ERR_SHAPE, "diffattn_v2_backward: need Hq even, Hq %% Hkv == 0 and Hq/Hkv even");
  if (sb < 0 || st < 0) return fail(DIFFATTN_ERR_SHAPE, "diffattn_v2_backward: negative logit stride");
  if ((dt == DIFFATTN_F32 && d > da::kSimtMaxD) || (dt == DIFFATTN_BF16 && d != 128))
    return fail(DIFFATTN_ERR_UNSUPPORTED,
                "diffattn_v2_backward: f32 with d <= 128 or bf16 with d = 128 (got dtype %d, d=%d)", (int)dt, d);
  const int G = Hq / 2;
  const bool dense = st == G && sb == static_cast<long long>(n) * G;  // one logit per token and pair
  if (!dense && !(st == 0 && (sb == 0 || sb == G)))
    return fail(DIFFATTN_ERR_UNSUPPORTED,
                "diffattn_v2_backward: logit strides (sb, st) must be (n*Hq/2, Hq/2), (Hq/2, 0) or (0, 0)");
  if (B == 0 || Hq == 0 || n == 0) {  // no rows: a logit shared by tokens gets a zero gradient
    const size_t shared = dense ? 0 : (sb == 0 ? static_cast<size_t>(G) : static_cast<size_t>(B) * G);
    if (shared > 0 && dlogits != nullptr) {
      cudaError_t e = cudaMemsetAsync(dlogits, 0, shared * sizeof(float), static_cast<cudaStream_t>(stream));
      if (e != cudaSuccess) return cuda_fail(e, "diffattn_v2_backward: clearing dlogits");
    }
    return ok();
  }
  if (!q || !k || !v || !lam_logits || !dy || !dq || !dk || !dv || !dlogits || !workspace)
    return fail(DIFFATTN_ERR_NULL, "diffattn_v2_backward: NULL pointer");
  const size_t need = diffattn_v2_backward_workspace(B, Hq, n, d);
  if (workspace_bytes < need)
    return fail(DIFFATTN_ERR_SHAPE, "diffattn_v2_backward: workspace of %zu bytes, need %zu", workspace_bytes,
                need);
  if (!aligned16(workspace))
    return fail(DIFFATTN_ERR_ALIGN, "diffattn_v2_backward: workspace must be 16-byte aligned");
  const long long nqb8 = (static_cast<long long>(n) + da::kSimtRows - 1) / da::kSimtRows;
  if (static_cast<long long>(B) * G * nqb8 > 0x7fffffffll)
    return fail(DIFFATTN_ERR_SHAPE, "diffattn_v2_backward: too many (batch, pair, row block) units");
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.f / std::sqrt(static_cast<float>(d));
  if (dt == DIFFATTN_BF16) {
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dy) || !aligned16(dq) || !aligned16(dk) ||
        !aligned16(dv))
      return fail(DIFFATTN_ERR_ALIGN, "diffattn_v2_backward: bf16 path needs 16-byte aligned tensors");
    int* status = nullptr;
    diffattn_status stt = status_word(&status);
    if (stt != DIFFATTN_OK) return stt;
    if ((stt = backward_v2_tc(B, Hq, Hkv, n, q, k, v, lam_logits, sb, st, scale, causal, dy, dq, dk, dv, dlogits, dense,
                              static_cast<uint8_t*>(workspace), status, s)) != DIFFATTN_OK)
      return stt;
    return ok();
  }
  const size_t R = bwd_rows(B, G, n);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* ws_do = reinterpret_cast<float*>(ws);
  float* ws_row = reinterpret_cast<float*>(ws + round256(R * d * 4));

  da::SimtParams rp{};
  rp.q1 = rp.q2 = static_cast<const float*>(q);
  rp.k1 = rp.k2 = static_cast<const float*>(k);
  rp.v = static_cast<const float*>(v);
  rp.lam_logits = lam_logits;
  rp.sb = sb;
  rp.st = st;
  rp.scale = scale;
  rp.norm_mult = 1.f;
  rp.eps = 1e-5f;
  rp.B = B;
  rp.n = n;
  rp.d = d;
  rp.dv = d;
  rp.causal = causal ? 1 : 0;
  rp.v2 = 1;
  rp.heads_q = Hq;
  rp.heads_kv = Hkv;
  rp.units_per_batch = G;
  rp.group = Hq / Hkv;
  rp.rows_total = static_cast<long long>(R);
  da::SimtBwdExtra rx{};
  rx.dy = static_cast<const float*>(dy);
  rx.ws_do = ws_do;
  rx.ws_row = ws_row;
  rx.dlogits_dense = dense ? dlogits : nullptr;

  da::BwdParams p{};
  p.q1 = p.q2 = rp.q1;
  p.k1 = p.k2 = rp.k1;
  p.v = rp.v;
  p.dO = ws_do;
  p.row = ws_row;
  p.dq1 = p.dq2 = static_cast<float*>(dq);
  p.dk1 = p.dk2 = static_cast<float*>(dk);
  p.dv = static_cast<float*>(dv);
  p.dlogits = dlogits;
  p.sb = sb;
  p.scale = scale;
  p.B = B;
  p.n = n;
  p.d = d;
  p.dvw = d;
  p.causal = rp.causal;
  p.v2 = 1;
  p.heads_q = Hq;
  p.heads_kv = Hkv;
  p.units = G;
  p.group = Hq / Hkv;
  p.rows = static_cast<long long>(R);
  p.n_logit_outs = dense ? 0 : (sb == 0 ? G : B * G);
  cudaError_t e = da::launch_simt_bwd_rows(rp, rx, s);
  if (e == cudaSuccess) e = da::launch_backward_f32(p, s);
  if (e != cudaSuccess) return cuda_fail(e, "diffattn_v2_backward launch");
  g_launches.fetch_add(dense ? 3 : 4);
  return ok();
}

// ---- training forward (saves each row's statistics) and the backward from them
size_t diffattn_forward_saved_bytes(int B, int H, int n, int d) {
  if (B < 0 || H < 0 || n < 0 || d < 1) return 0;
  return saved_fwd_bytes(static_cast<size_t>(B) * H, static_cast<size_t>(n), 2 * static_cast<size_t>(d));
}

size_t diffattn_v2_forward_saved_bytes(int B, int Hq, int n, int d) {
  if (B < 0 || Hq < 0 || n < 0 || d < 1) return 0;
  return saved_fwd_bytes(static_cast<size_t>(B) * (Hq / 2), static_cast<size_t>(n), static_cast<size_t>(d));
}

// Checks shared by the training entry points: bf16 tensors 16-byte aligned, the saved buffer's size and alignment.
static diffattn_status check_saved(const char* fn, const void* saved, size_t saved_bytes, size_t need) {
  if (!saved) return fail(DIFFATTN_ERR_NULL, "%s: NULL saved buffer", fn);
  if (saved_bytes < need) return fail(DIFFATTN_ERR_SHAPE, "%s: saved buffer of %zu bytes, need %zu", fn, saved_bytes, need);
  if ((reinterpret_cast<uintptr_t>(saved) & 255u) != 0) return fail(DIFFATTN_ERR_ALIGN, "%s: saved buffer not 256-byte aligned", fn);
  return DIFFATTN_OK;
}

diffattn_status diffattn_forward_train(int B, int H, int n, int d, const void* q1, const void* q2, const void* k1,
                                       const void* k2, const void* v, const float* lambda, float lambda_init,
                                       const float* gamma, float eps, int causal, void* out, void* saved,
                                       size_t saved_bytes, void* stream) {
  const char* fn = "diffattn_forward_train";
  if (B < 0 || H < 0 || n < 0 || d < 1) return fail(DIFFATTN_ERR_SHAPE, "%s: bad sizes B=%d H=%d n=%d d=%d", fn, B, H, n, d);
  if (d != 64) return fail(DIFFATTN_ERR_UNSUPPORTED, "%s: d = 64 only (got %d)", fn, d);
  if (B == 0 || H == 0 || n == 0) return ok();
  if (!q1 || !q2 || !k1 || !k2 || !v || !lambda || !out) return fail(DIFFATTN_ERR_NULL, "%s: NULL pointer", fn);
  if (!std::isfinite(lambda_init)) return fail(DIFFATTN_ERR_SHAPE, "%s: lambda_init not finite", fn);
  if (!aligned16(q1) || !aligned16(q2) || !aligned16(k1) || !aligned16(k2) || !aligned16(v) || !aligned16(out))
    return fail(DIFFATTN_ERR_ALIGN, "%s: tensors must be 16-byte aligned", fn);
  const size_t R = static_cast<size_t>(B) * H * n;
  diffattn_status st = check_saved(fn, saved, saved_bytes, diffattn_forward_saved_bytes(B, H, n, d));
  if (st != DIFFATTN_OK) return st;
  if (eps <= 0.f) eps = 1e-5f;
  int* status = nullptr;
  if ((st = status_word(&status)) != DIFFATTN_OK) return st;
  const SavedFwd sv = saved_fwd_views(saved, static_cast<size_t>(B) * H, static_cast<size_t>(n), 2 * d);
  const long long Hd = static_cast<long long>(H) * d;
  da::TwoPassParams p;
  memset(&p, 0, sizeof(p));
  if ((st = make_map_view(&p.tm_q1, q1, B, n, H, d, d, Hd, 64, 128)) != DIFFATTN_OK) return st;
  if ((st = make_map_view(&p.tm_q2, q2, B, n, H, d, d, Hd, 64, 128)) != DIFFATTN_OK) return st;
  if ((st = make_map_view(&p.tm_k1, k1, B, n, H, d, d, Hd, 64, 128)) != DIFFATTN_OK) return st;
  if ((st = make_map_view(&p.tm_k2, k2, B, n, H, d, d, Hd, 64, 128)) != DIFFATTN_OK) return st;
  if ((st = make_map_view(&p.tm_v, v, B, n, H, 2 * d, 2 * d, 2 * Hd, 64, 64)) != DIFFATTN_OK) return st;
  p.row = const_cast<float*>(sv.lse);
  p.rows = static_cast<long long>(R);
  p.o1_save = const_cast<__nv_bfloat16*>(sv.o1);
  p.o2_save = const_cast<__nv_bfloat16*>(sv.o2);
  const float sc = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d)));
  if ((st = launch_v1_tc(fn, p, false, B, H, n, d, sc, sc, lambda, lambda_init, gamma, eps, causal, out, status,
                         static_cast<cudaStream_t>(stream))) != DIFFATTN_OK)
    return st;
  return ok();
}

diffattn_status diffattn_backward_saved(int B, int H, int n, int d, const void* q1, const void* q2, const void* k1,
                                        const void* k2, const void* v, const float* lambda, float lambda_init,
                                        const float* gamma, float eps, int causal, const void* dy, const void* saved,
                                        size_t saved_bytes, void* dq1, void* dq2, void* dk1, void* dk2, void* dv,
                                        float* dlambda, float* dgamma, void* workspace, size_t workspace_bytes,
                                        void* stream) {
  const char* fn = "diffattn_backward_saved";
  if (B < 0 || H < 0 || n < 0 || d < 1) return fail(DIFFATTN_ERR_SHAPE, "%s: bad sizes B=%d H=%d n=%d d=%d", fn, B, H, n, d);
  if (d != 64) return fail(DIFFATTN_ERR_UNSUPPORTED, "%s: d = 64 only (got %d)", fn, d);
  if (!dlambda) return fail(DIFFATTN_ERR_NULL, "%s: NULL dlambda", fn);
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (B == 0 || H == 0 || n == 0) {  // no rows: dlambda = 0, dgamma = 0
    cudaError_t e = cudaMemsetAsync(dlambda, 0, sizeof(float), s);
    if (e == cudaSuccess && dgamma) e = cudaMemsetAsync(dgamma, 0, 2 * d * sizeof(float), s);
    if (e != cudaSuccess) return cuda_fail(e, "diffattn_backward_saved: clearing dlambda / dgamma");
    return ok();
  }
  if (!q1 || !q2 || !k1 || !k2 || !v || !lambda || !dy || !dq1 || !dq2 || !dk1 || !dk2 || !dv || !workspace)
    return fail(DIFFATTN_ERR_NULL, "%s: NULL pointer", fn);
  if (!std::isfinite(lambda_init)) return fail(DIFFATTN_ERR_SHAPE, "%s: lambda_init not finite", fn);
  const size_t need = diffattn_backward_workspace(B, H, n, d);
  if (workspace_bytes < need) return fail(DIFFATTN_ERR_SHAPE, "%s: workspace of %zu bytes, need %zu", fn, workspace_bytes, need);
  if (!aligned16(workspace) || !aligned16(q1) || !aligned16(q2) || !aligned16(k1) || !aligned16(k2) || !aligned16(v) ||
      !aligned16(dy) || !aligned16(dq1) || !aligned16(dq2) || !aligned16(dk1) || !aligned16(dk2) || !aligned16(dv))
    return fail(DIFFATTN_ERR_ALIGN, "%s: tensors and workspace must be 16-byte aligned", fn);
  diffattn_status st = check_saved(fn, saved, saved_bytes, diffattn_forward_saved_bytes(B, H, n, d));
  if (st != DIFFATTN_OK) return st;
  const long long nqb = (static_cast<long long>(n) + 127) / 128;
  if (static_cast<long long>(B) * H * nqb > 0x7fffffffll || static_cast<long long>(B) * H * n > 0x7fffffffll)
    return fail(DIFFATTN_ERR_SHAPE, "%s: too many rows", fn);
  if (eps <= 0.f) eps = 1e-5f;
  int* status = nullptr;
  if ((st = status_word(&status)) != DIFFATTN_OK) return st;
  const SavedFwd sv = saved_fwd_views(saved, static_cast<size_t>(B) * H, static_cast<size_t>(n), 2 * d);
  if ((st = backward_v1_tc(B, H, n, q1, q2, k1, k2, v, lambda, lambda_init, gamma, eps, causal, dy, dq1, dq2, dk1, dk2,
                           dv, dlambda, dgamma, static_cast<uint8_t*>(workspace), status, s, &sv)) != DIFFATTN_OK)
    return st;
  return ok();
}

diffattn_status diffattn_v2_forward_train(int B, int Hq, int Hkv, int n, int d, const void* q, const void* k,
                                          const void* v, const float* lam_logits, long long sb, long long st_,
                                          float softmax_scale, int causal, void* out, void* saved, size_t saved_bytes,
                                          void* stream) {
  const char* fn = "diffattn_v2_forward_train";
  if (B < 0 || Hq < 0 || Hkv < 1 || n < 0 || d < 1)
    return fail(DIFFATTN_ERR_SHAPE, "%s: bad sizes B=%d Hq=%d Hkv=%d n=%d d=%d", fn, B, Hq, Hkv, n, d);
  if (Hq % 2 != 0 || Hq % Hkv != 0 || (Hq / Hkv) % 2 != 0)
    return fail(DIFFATTN_ERR_SHAPE, "%s: need Hq even, Hq %% Hkv == 0 and Hq/Hkv even (Hq=%d Hkv=%d)", fn, Hq, Hkv);
  if (sb < 0 || st_ < 0) return fail(DIFFATTN_ERR_SHAPE, "%s: negative logit stride", fn);
  if (d != 128) return fail(DIFFATTN_ERR_UNSUPPORTED, "%s: d = 128 only (got %d)", fn, d);
  if (B == 0 || Hq == 0 || n == 0) return ok();
  if (!q || !k || !v || !lam_logits || !out) return fail(DIFFATTN_ERR_NULL, "%s: NULL pointer", fn);
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return fail(DIFFATTN_ERR_ALIGN, "%s: tensors must be 16-byte aligned", fn);
  const int G = Hq / 2;
  const size_t R = static_cast<size_t>(B) * G * n;
  diffattn_status st = check_saved(fn, saved, saved_bytes, diffattn_v2_forward_saved_bytes(B, Hq, n, d));
  if (st != DIFFATTN_OK) return st;
  int* status = nullptr;
  if ((st = status_word(&status)) != DIFFATTN_OK) return st;
  const SavedFwd sv = saved_fwd_views(saved, static_cast<size_t>(B) * G, static_cast<size_t>(n), d);
  const double scale = softmax_scale > 0.f ? softmax_scale : 1.0 / std::sqrt(static_cast<double>(d));
  da::TwoPassParams p;
  memset(&p, 0, sizeof(p));
  if ((st = make_map_box(&p.tm_q1, q, B, n, Hq, d, 64, 128)) != DIFFATTN_OK) return st;
  p.tm_q2 = p.tm_q1;
  if ((st = make_map_box(&p.tm_k1, k, B, n, Hkv, d, 64, 128)) != DIFFATTN_OK) return st;
  p.tm_k2 = p.tm_k1;
  if ((st = make_map_box(&p.tm_v, v, B, n, Hkv, d, 64, 128)) != DIFFATTN_OK) return st;
  p.row = const_cast<float*>(sv.lse);
  p.rows = static_cast<long long>(R);
  p.o1_save = const_cast<__nv_bfloat16*>(sv.o1);
  p.o2_save = const_cast<__nv_bfloat16*>(sv.o2);
  if ((st = launch_v2_tc(fn, p, false, B, Hq, Hkv, n, d, lam_logits, sb, st_,
                         static_cast<float>(1.4426950408889634 * scale), causal, out, status,
                         static_cast<cudaStream_t>(stream))) != DIFFATTN_OK)
    return st;
  return ok();
}

diffattn_status diffattn_v2_backward_saved(int B, int Hq, int Hkv, int n, int d, const void* q, const void* k,
                                           const void* v, const float* lam_logits, long long sb, long long st_,
                                           float softmax_scale, int causal, const void* dy, const void* saved,
                                           size_t saved_bytes, void* dq, void* dk, void* dv, float* dlogits,
                                           void* workspace, size_t workspace_bytes, void* stream) {
  const char* fn = "diffattn_v2_backward_saved";
  if (B < 0 || Hq < 0 || Hkv < 1 || n < 0 || d < 1)
    return fail(DIFFATTN_ERR_SHAPE, "%s: bad sizes B=%d Hq=%d Hkv=%d n=%d d=%d", fn, B, Hq, Hkv, n, d);
  if (Hq % 2 != 0 || Hq % Hkv != 0 || (Hq / Hkv) % 2 != 0)
    return fail(DIFFATTN_ERR_SHAPE, "%s: need Hq even, Hq %% Hkv == 0 and Hq/Hkv even", fn);
  if (sb < 0 || st_ < 0) return fail(DIFFATTN_ERR_SHAPE, "%s: negative logit stride", fn);
  if (d != 128) return fail(DIFFATTN_ERR_UNSUPPORTED, "%s: d = 128 only (got %d)", fn, d);
  const int G = Hq / 2;
  const bool dense = st_ == G && sb == static_cast<long long>(n) * G;
  if (!dense && !(st_ == 0 && (sb == 0 || sb == G)))
    return fail(DIFFATTN_ERR_UNSUPPORTED, "%s: logit strides (sb, st) must be (n*Hq/2, Hq/2), (Hq/2, 0) or (0, 0)", fn);
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (B == 0 || Hq == 0 || n == 0) {  // no rows: a logit shared by tokens gets a zero gradient
    const size_t shared = dense ? 0 : (sb == 0 ? static_cast<size_t>(G) : static_cast<size_t>(B) * G);
    if (shared > 0 && dlogits != nullptr) {
      cudaError_t e = cudaMemsetAsync(dlogits, 0, shared * sizeof(float), s);
      if (e != cudaSuccess) return cuda_fail(e, "diffattn_v2_backward_saved: clearing dlogits");
    }
    return ok();
  }
  if (!q || !k || !v || !lam_logits || !dy || !dq || !dk || !dv || !dlogits || !workspace)
    return fail(DIFFATTN_ERR_NULL, "%s: NULL pointer", fn);
  const size_t need = diffattn_v2_backward_workspace(B, Hq, n, d);
  if (workspace_bytes < need) return fail(DIFFATTN_ERR_SHAPE, "%s: workspace of %zu bytes, need %zu", fn, workspace_bytes, need);
  if (!aligned16(workspace) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dy) || !aligned16(dq) ||
      !aligned16(dk) || !aligned16(dv))
    return fail(DIFFATTN_ERR_ALIGN, "%s: tensors and workspace must be 16-byte aligned", fn);
  diffattn_status st = check_saved(fn, saved, saved_bytes, diffattn_v2_forward_saved_bytes(B, Hq, n, d));
  if (st != DIFFATTN_OK) return st;
  const long long nqb = (static_cast<long long>(n) + 127) / 128;
  if (static_cast<long long>(B) * G * nqb > 0x7fffffffll || static_cast<long long>(B) * G * n > 0x7fffffffll)
    return fail(DIFFATTN_ERR_SHAPE, "%s: too many rows", fn);
  int* status = nullptr;
  if ((st = status_word(&status)) != DIFFATTN_OK) return st;
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.f / std::sqrt(static_cast<float>(d));
  const SavedFwd sv = saved_fwd_views(saved, static_cast<size_t>(B) * G, static_cast<size_t>(n), d);
  if ((st = backward_v2_tc(B, Hq, Hkv, n, q, k, v, lam_logits, sb, st_, scale, causal, dy, dq, dk, dv, dlogits, dense,
                           static_cast<uint8_t*>(workspace), status, s, &sv)) != DIFFATTN_OK)
    return st;
  return ok();
}

diffattn_status lambda_reparam_backward(const float* lq1, const float* lk1, const float* lq2, const float* lk2,
                                        int dim, const float* dlambda, float* dlq1, float* dlk1, float* dlq2,
                                        float* dlk2, void* stream) {
  if (!lq1 || !lk1 || !lq2 || !lk2 || !dlambda || !dlq1 || !dlk1 || !dlq2 || !dlk2)
    return fail(DIFFATTN_ERR_NULL, "lambda_reparam_backward: NULL pointer");
  if (dim < 1) return fail(DIFFATTN_ERR_SHAPE, "lambda_reparam_backward: dim must be >= 1 (got %d)", dim);
  cudaError_t e = da::launch_lambda_reparam_bwd(lq1, lk1, lq2, lk2, dim, dlambda, dlq1, dlk1, dlq2, dlk2,
                                                static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "lambda_reparam_backward launch");
  g_launches.fetch_add(1);
  return ok();
}

diffattn_status diffattn_device_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int* status = nullptr;
  diffattn_status st = status_word(&status);
  if (st != DIFFATTN_OK) return st;
  int host = 0;
  e = cudaMemcpy(&host, status, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read status word");
  const int zero = 0;
  e = cudaMemcpy(status, &zero, sizeof(int), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e, "clear status word");
#ifdef DIFFATTN_BOUNDS
  {  // the bounds-check build: every translation unit's record (a failed check usually ends in a timeout too)
    da::BoundsRegistry& r = da::bounds_registry();
    std::lock_guard<std::mutex> lk(r.mu);
    long long failures = 0;
    int first[3] = {0, 0, 0};
    for (int i = 0; i < r.count; ++i) {
      int rec[3] = {0, 0, 0};
      const int n = r.readers[i](rec);
      if (n < 0) return fail(DIFFATTN_ERR_CUDA, "reading a bounds-check record failed");
      if (n > 0 && failures == 0) std::copy(rec, rec + 3, first);
      failures += n;
    }
    if (failures > 0)
      return fail(DIFFATTN_ERR_BOUNDS, "%lld bounds-check failures; first in file tag %d at line %d (value %d)",
                  failures, first[1] / 100000, first[1] % 100000, first[2]);
  }
#endif
  if (host == DIFFATTN_ERR_TIMEOUT) return fail(DIFFATTN_ERR_TIMEOUT, "a bounded in-kernel wait ran out");
  if (host != 0) return fail(DIFFATTN_ERR_CUDA, "device status word holds %d", host);
  return ok();
}

const char* diffattn_last_error(void) { return t_last_error.c_str(); }

#ifdef DIFFATTN_BOUNDS
namespace {
// Self-test of the checks: one thread stores through DA_STORE at index 5 with
// a limit of 4.  The store is skipped and recorded; were it not, it would
// still land inside this 8-element array.
__device__ int g_bounds_selftest[8];
__global__ void bounds_selftest_kernel() { DA_STORE(g_bounds_selftest, 5, 4, 1); }
}  // namespace
#endif

int diffattn_debug_item_plan(int grid, long long units, int nqt, int qt0, int n, int causal, long long kv_unit_bytes,
                             unsigned short* first, unsigned short* items) {
  if (!first || !items || units < 1 || nqt < 1 || n < 1) return 0;
  thread_local da::ItemPlan plan;
  if (!plan_items(plan, grid, units, nqt, qt0, n, causal, kv_unit_bytes)) return 0;
  for (int c = 0; c <= grid; ++c) first[c] = plan.first[c];
  for (int a = 0; a < plan.first[grid]; ++a) items[a] = plan.items[a];
  return plan.count;
}

diffattn_status diffattn_debug_bounds_selftest(void* stream) {
#ifdef DIFFATTN_BOUNDS
  bounds_selftest_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>();
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "diffattn_debug_bounds_selftest launch");
  g_launches.fetch_add(1);
  return ok();
#else
  (void)stream;
  return fail(DIFFATTN_ERR_UNSUPPORTED, "diffattn_debug_bounds_selftest: not the bounds-check build");
#endif
}

int diffattn_bounds_checked(void) {
#ifdef DIFFATTN_BOUNDS
  return 1;
#else
  return 0;
#endif
}

diffattn_status diffattn_debug_wait_timeout(long long budget_ns, void* stream) {
  if (budget_ns < 1 || budget_ns > 1000000000ll)
    return fail(DIFFATTN_ERR_SHAPE, "diffattn_debug_wait_timeout: budget must be in [1, 1e9] ns");
  int* status = nullptr;
  diffattn_status st = status_word(&status);
  if (st != DIFFATTN_OK) return st;
  // The in-kernel budget counts SM cycles; 2 cycles per nanosecond (the
  // clock is at most 2.07 GHz) makes the wait last at least about budget_ns.
  cudaError_t e = da::launch_wait_selftest(static_cast<unsigned long long>(budget_ns) * 2ull, status,
                                           static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "diffattn_debug_wait_timeout launch");
  g_launches.fetch_add(1);
  return ok();
}

long long diffattn_launch_count(void) { return g_launches.load(); }

}  // extern "C"
