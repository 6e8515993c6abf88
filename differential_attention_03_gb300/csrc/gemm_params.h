// Parameter block of the projection GEMM, shared by its launcher and the host API.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

namespace da {

constexpr int kGemmBM = 128;  // output rows per tile (TMEM lanes)
constexpr int kGemmBN = 256;  // output columns per tile (one M128 N256 MMA)

struct GemmParams {
  CUtensorMap tm_a;  // A [M, K] bf16: dims {K, M}, box {64, 128}, 128-byte swizzle
  CUtensorMap tm_b;  // B [N, K] bf16: dims {K, N}, box {64, 256}, 128-byte swizzle
  __nv_bfloat16* c;  // columns [0, n_main): c[row * ldc + col]
  float* c2;         // columns [n_main, N): c2[row * ldc2 + col - n_main] (nullptr if n_main == N)
  long long ldc, ldc2;
  int M, N, K, n_main;
  int tiles_m, tiles_n, group_m;
  int* status;
};

}  // namespace da
