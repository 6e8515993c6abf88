// Shared-memory staging of row tiles, used by the fp32 forward and backward
// kernels (CTAs of kSimtWarps warps).
#pragma once

#include <cstdint>

#include "params.h"

namespace da {

// Copies rows [r0, r0 + nrows) x columns [0, width) of a strided global matrix
// into shared memory (row pitch `pitch` floats), zero past `nvalid` rows.
// With `vec` (width % 4 == 0, 16-byte aligned rows) it uses 16-byte loads.
// All loads of the thread are issued before any store, so the copy costs one
// memory round trip.
__device__ __forceinline__ void stage_rows(float* dst, int pitch, const float* src, size_t stride, int r0,
                                           int nvalid, int width, int nrows, bool vec) {
  constexpr int kMaxPerThread = 8;  // 32 rows x 256 floats / 4 per load / 256 threads
  if (vec) {
    const int w4 = width >> 2, total = nrows * w4;
    float4 buf[kMaxPerThread];
#pragma unroll
    for (int k = 0; k < kMaxPerThread; ++k) {
      const int i = threadIdx.x + k * kSimtWarps * 32;
      buf[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (i < total) {
        const int r = i / w4, c = (i % w4) * 4;
        if (r0 + r < nvalid) buf[k] = __ldg(reinterpret_cast<const float4*>(src + (r0 + r) * stride + c));
      }
    }
#pragma unroll
    for (int k = 0; k < kMaxPerThread; ++k) {
      const int i = threadIdx.x + k * kSimtWarps * 32;
      if (i < total) {
        const int r = i / w4, c = (i % w4) * 4;
        float* o = dst + r * pitch + c;
        o[0] = buf[k].x;
        o[1] = buf[k].y;
        o[2] = buf[k].z;
        o[3] = buf[k].w;
      }
    }
  } else {
    constexpr int kMaxScalar = 4 * kMaxPerThread;
    const int total = nrows * width;
    for (int base = 0; base < total; base += kMaxScalar * kSimtWarps * 32) {
      float buf[kMaxScalar];
#pragma unroll
      for (int k = 0; k < kMaxScalar; ++k) {
        const int i = base + threadIdx.x + k * kSimtWarps * 32;
        buf[k] = 0.f;
        if (i < total) {
          const int r = i / width, c = i % width;
          if (r0 + r < nvalid) buf[k] = __ldg(src + (r0 + r) * stride + c);
        }
      }
#pragma unroll
      for (int k = 0; k < kMaxScalar; ++k) {
        const int i = base + threadIdx.x + k * kSimtWarps * 32;
        if (i < total) dst[(i / width) * pitch + i % width] = buf[k];
      }
    }
  }
}

}  // namespace da
