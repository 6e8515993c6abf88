// Dense bf16 GEMM on tcgen05 tensor cores (sm_103a) for the projections
// around the differential-attention operator:
//
//   C[M, N] = A[M, K] . B[N, K]^T      (bf16 operands, fp32 accumulation)
//
// The attention layer ("Differential Transformer" news article, section
// "差分注意力"; DIFF V2 analysis page, section "5. 간소화된 λ 매개변수화")
// projects the tokens X by W^Q, W^K, W^V (and, for DIFF V2, the lambda logits
// by W^lambda) and the concatenated normalised heads by W^O.  Both are plain
// GEMMs with the weights stored as [out features, in features] (K-major, the
// same operand form as the attention kernels' keys).  Columns [0, n_main) of C
// are written in bf16 to `c` (row stride ldc); columns [n_main, N), if any,
// in fp32 to `c2` (row stride ldc2): the DIFF V2 lambda logits stay fp32 for
// the sigmoid.
//
// Shape: one CTA per SM, persistent over 128 x 256 output tiles taken in
// groups of `group_m` row blocks (so that neighbouring CTAs share A and B
// tiles in L2).  Every MMA is M128 N256 K16, which one issuing thread keeps
// at the full tensor rate.
//   warp 0      TMA producer: A (128 x 64) and B (256 x 64) boxes of each
//               64-wide K block into a STAGES-deep ring (128-byte swizzle).
//   warp 1      TMEM allocator and MMA issuer: per K block four K16 MMAs into
//               the tile's accumulator; commits release the ring slot and,
//               after the last K block, hand the accumulator to the epilogue.
//   warps 2-5   epilogue: thread = output row (TMEM lane); reads the 256 fp32
//               columns in 32-column chunks, rounds to bf16 and stores.
// TMEM: two 256-column accumulators, so the epilogue of tile i overlaps the
// main loop of tile i + 1.  Rows past M and columns past N are zero-filled
// by TMA on load and skipped on store.
#pragma once

#include <cuda_bf16.h>

#include "gemm_params.h"
#include "ptx.cuh"

#undef DA_BOUNDS_FILE
#define DA_BOUNDS_FILE 6

namespace da {

struct GemmCfg {
  static constexpr int BM = kGemmBM, BN = kGemmBN, BK = 64;
  static constexpr int STAGES = 4;
  static constexpr int NTHREADS = 192;
  static constexpr int A_BYTES = BM * BK * 2;  // 16 KB
  static constexpr int B_BYTES = BN * BK * 2;  // 32 KB
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int OFF_BARS = STAGES * STAGE_BYTES;
  static constexpr int NBARS = 2 * STAGES + 5;  // full, empty, acc_full[2], acc_empty[2], mma_done
  static constexpr int OFF_MISC = OFF_BARS + NBARS * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + alignment slack
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t IDESC = idesc_bf16(BM, BN, false, false);
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

// Tile t of the persistent walk -> (row block, column block), row blocks in
// groups of group_m so that the CTAs working at one time share operands.
__device__ __forceinline__ void gemm_tile(const GemmParams& p, int t, int& mb, int& nb) {
  const int per_group = p.group_m * p.tiles_n;
  const int g = t / per_group;
  const int first = g * p.group_m;
  const int gm = min(p.group_m, p.tiles_m - first);
  const int r = t - g * per_group;
  mb = first + r % gm;
  nb = r / gm;
}

__global__ void __launch_bounds__(GemmCfg::NTHREADS, 1) gemm_bf16_kernel(const __grid_constant__ GemmParams p) {
  using C = GemmCfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BARS);
  uint64_t* full = bars;                 // [STAGES] A and B of a K block landed
  uint64_t* empty = full + C::STAGES;    // [STAGES] the MMAs reading the slot completed
  uint64_t* acc_full = empty + C::STAGES;  // [2] every MMA of the tile completed
  uint64_t* acc_empty = acc_full + 2;      // [2] the epilogue has read the accumulator
  uint64_t* mma_done = acc_empty + 2;      // every MMA issued completed (abort drain)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int tiles = p.tiles_m * p.tiles_n;
  const int kblocks = (p.K + C::BK - 1) / C::BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 4);  // one arrival per epilogue warp
    }
    mbar_init(mma_done, 1);
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
      tma_prefetch_desc(&p.tm_a);
      tma_prefetch_desc(&p.tm_b);
      long long fill = 0;  // K blocks loaded so far (all tiles)
      bool ok = true;
      for (int t = blockIdx.x; ok && t < tiles; t += gridDim.x) {
        int mb, nb;
        gemm_tile(p, t, mb, nb);
        for (int kb = 0; kb < kblocks; ++kb, ++fill) {
          const int s = static_cast<int>(fill % C::STAGES);
          const long long use = fill / C::STAGES;
          if (use > 0 && !mbar_wait(&empty[s], static_cast<uint32_t>(use - 1) & 1u, ab)) {
            ok = false;
            break;
          }
          uint8_t* dst = smem + s * C::STAGE_BYTES;
          mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
          if (DA_BOUNDS(kb * C::BK < p.K && mb * C::BM < p.M && nb * C::BN < p.N)) {
            tma_load_2d(dst, &p.tm_a, &full[s], kb * C::BK, mb * C::BM);
            tma_load_2d(dst + C::A_BYTES, &p.tm_b, &full[s], kb * C::BK, nb * C::BN);
          }
        }
      }
      if (*ab.flag) {
        // Aborted: the copies already issued land before the CTA exits.
        for (long long f = (fill > C::STAGES ? fill - C::STAGES : 0); f < fill; ++f)
          mbar_wait_drain(&full[f % C::STAGES], static_cast<uint32_t>(f / C::STAGES) & 1u, kWaitBudgetCycles);
      }
    }
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    const uint64_t dA = sdesc_sw128(smem_u32(smem), 16, 1024);
    const uint64_t dB = sdesc_sw128(smem_u32(smem + C::A_BYTES), 16, 1024);
    auto waitp = [&](uint64_t* bar, uint32_t parity) -> bool {
      const bool r = __all_sync(0xffffffffu, mbar_wait(bar, parity, ab));
      tc_fence_after();
      return r;
    };
    long long fill = 0;
    int i = 0;  // tiles of this CTA so far
    bool ok = true;
    for (int t = blockIdx.x; ok && t < tiles; t += gridDim.x, ++i) {
      const int a = i & 1;
      // The epilogue of tile i - 2 has read this accumulator.
      if (i >= 2 && !waitp(&acc_empty[a], static_cast<uint32_t>((i >> 1) - 1) & 1u)) {
        ok = false;
        break;
      }
      const uint32_t dacc = tmem + static_cast<uint32_t>(a * C::BN);
      for (int kb = 0; kb < kblocks; ++kb, ++fill) {
        const int s = static_cast<int>(fill % C::STAGES);
        if (!waitp(&full[s], static_cast<uint32_t>(fill / C::STAGES) & 1u)) {
          ok = false;
          break;
        }
        const uint64_t so = static_cast<uint64_t>((s * C::STAGE_BYTES) >> 4);
#pragma unroll
        for (int k = 0; k < C::BK / 16; ++k)
          mma_ss_elect(dacc, dA + so + static_cast<uint64_t>((k * 32) >> 4), dB + so + static_cast<uint64_t>((k * 32) >> 4),
                       C::IDESC, (kb > 0 || k > 0) ? 1u : 0u);
        tc_commit_elect(&empty[s]);
      }
      if (!ok) break;
      tc_commit_elect(&acc_full[a]);
    }
    tc_commit_elect(mma_done);
    if (*ab.flag) mbar_wait_drain(mma_done, 0, kWaitBudgetCycles);
    __syncwarp();
  } else {
    // ================================================================ epilogue
    const int wq = warp & 3;  // TMEM lane quarter this warp may access
    const int row_in_tile = wq * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    int i = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++i) {
      int mb, nb;
      gemm_tile(p, t, mb, nb);
      const int a = i & 1;
      const bool got = mbar_wait(&acc_full[a], static_cast<uint32_t>(i >> 1) & 1u, ab);
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after();
      const int row = mb * C::BM + row_in_tile;
      const bool row_ok = row < p.M;
#pragma unroll 1
      for (int ch = 0; ch < C::BN / 32; ++ch) {
        uint32_t r[32];
        tmem_ld32(tl + static_cast<uint32_t>(a * C::BN + ch * 32), r);
        tmem_ld_wait(r);
        const int c0 = nb * C::BN + ch * 32;
        if (!row_ok || c0 >= p.N) {
          // nothing of this chunk to store (the loads above stay warp-wide)
        } else if (!DA_BOUNDS_V(row >= 0 && c0 >= 0, row)) {
        } else if (c0 + 32 <= p.n_main) {
          uint4* dst = reinterpret_cast<uint4*>(p.c + static_cast<long long>(row) * p.ldc + c0);
#pragma unroll
          for (int v = 0; v < 4; ++v)
            dst[v] = make_uint4(pack_bf16x2(__uint_as_float(r[8 * v + 0]), __uint_as_float(r[8 * v + 1])),
                                pack_bf16x2(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3])),
                                pack_bf16x2(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5])),
                                pack_bf16x2(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7])));
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int col = c0 + j;
            if (col < p.n_main)
              p.c[static_cast<long long>(row) * p.ldc + col] = __float2bfloat16_rn(__uint_as_float(r[j]));
            else if (col < p.N)
              p.c2[static_cast<long long>(row) * p.ldc2 + (col - p.n_main)] = __uint_as_float(r[j]);
          }
        }
      }
      // Every read of this accumulator is done: the MMAs of tile i + 2 may overwrite it.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[a]);
      __syncwarp();
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
