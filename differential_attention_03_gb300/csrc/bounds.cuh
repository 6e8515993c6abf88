// Bounds-check build.  Compiled with -DDIFFATTN_BOUNDS (the library is then
// libdiffattn_bounds.so, selected at load time with DIFFATTN_DEBUG=1), every
// TMA coordinate, tensor-memory address and global store in the kernels is
// checked before the access is made.  A failed check skips the access and
// records (number of failures, first site, first value) in a device word of
// this translation unit; diffattn_device_status collects the words of every
// translation unit and reports DIFFATTN_ERR_BOUNDS.  A site is
// DA_BOUNDS_FILE * 100000 + source line (each kernel header defines
// DA_BOUNDS_FILE after its includes).  A skipped TMA load leaves its
// mbarrier short of bytes, so the bounded wait on it runs out and the kernel
// aborts as on a timeout; nothing hangs and nothing is written out of range.
// In the normal build DA_BOUNDS(cond) is `true` (cond is not evaluated) and
// the kernels are unchanged.
#pragma once

#include <cstdint>

#ifdef DIFFATTN_BOUNDS
#include <cuda_runtime.h>

namespace da {

// Reads this translation unit's record into out[0..2] (count, site, value),
// clears it and returns the count (-1 if the read failed).
using BoundsReader = int (*)(int* out);
// Registers a translation unit's reader (host side; defined with the C ABI).
void bounds_register(BoundsReader reader);

static __device__ int g_bounds_word[3];

static __device__ __noinline__ bool bounds_fail(int site, long long value) {
  if (atomicAdd(&g_bounds_word[0], 1) == 0) {
    g_bounds_word[1] = site;
    g_bounds_word[2] = static_cast<int>(value);
  }
  return false;
}

static int bounds_read_this_unit(int* out) {
  int h[3] = {0, 0, 0};
  if (cudaMemcpyFromSymbol(h, g_bounds_word, sizeof(h)) != cudaSuccess) return -1;
  if (h[0] != 0) {
    const int z[3] = {0, 0, 0};
    if (cudaMemcpyToSymbol(g_bounds_word, z, sizeof(z)) != cudaSuccess) return -1;
    out[0] = h[0];
    out[1] = h[1];
    out[2] = h[2];
  }
  return h[0];
}

static const bool g_bounds_registered = (bounds_register(&bounds_read_this_unit), true);

}  // namespace da

#ifndef DA_BOUNDS_FILE
#define DA_BOUNDS_FILE 0
#endif
#define DA_BOUNDS_V(cond, value) \
  ((cond) ? true : ::da::bounds_fail(DA_BOUNDS_FILE * 100000 + __LINE__, static_cast<long long>(value)))
#define DA_BOUNDS(cond) DA_BOUNDS_V(cond, 0)

#else
#define DA_BOUNDS_V(cond, value) true
#define DA_BOUNDS(cond) true
#endif

// Global store with an index check in the bounds-check build:
// base[idx] = v when 0 <= idx < limit (normal build: base[idx] = v).
#ifdef DIFFATTN_BOUNDS
#define DA_STORE(base, idx, limit, v)                                            \
  do {                                                                           \
    const long long da_i_ = static_cast<long long>(idx);                         \
    if (DA_BOUNDS_V(da_i_ >= 0 && da_i_ < static_cast<long long>(limit), da_i_)) \
      (base)[da_i_] = (v);                                                       \
  } while (0)
#else
#define DA_STORE(base, idx, limit, v) ((base)[idx] = (v))
#endif
