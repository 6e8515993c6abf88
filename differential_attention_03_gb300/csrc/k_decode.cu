// Launchers of the decode kernel (p.nsplit clusters of `cs` CTAs per (batch, head), then the
// combine kernel when p.nsplit > 1).
#include "decode.cuh"
#include "launch.h"

namespace da {

template <int D, bool V2, bool K8>
static cudaError_t launch_decode(const DecodeParams& p, int units, int cs, cudaStream_t s) {
  using C = DecodeCfg<D, V2, K8>;
  auto kern = decode_kernel<D, V2, K8>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(units) * static_cast<unsigned>(p.nsplit) * static_cast<unsigned>(cs), 1, 1);
  cfg.blockDim = dim3(C::NTHREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cs);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // a programmatic dependent of the previous kernel on the stream (the kernel waits first thing)
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, kern, p);
  if (e != cudaSuccess) return e;
  if (p.nsplit > 1) {  // merge the clusters' states of every (b, h) and finish the rows
    // (the combine kernel's own block size: the key type does not change its layout).  A
    // programmatic dependent launch: its CTAs are scheduled while the last clusters finish and
    // wait in grid_dep_wait() for the states, which hides the launch between the two kernels.
    cudaLaunchConfig_t cc = {};
    cc.gridDim = dim3(static_cast<unsigned>(units), 1, 1);
    cc.blockDim = dim3(DecodeCfg<D, V2>::NTHREADS, 1, 1);
    cc.dynamicSmemBytes = 0;
    cc.stream = s;
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cc.attrs = pdl;
    cc.numAttrs = 1;
    e = cudaLaunchKernelEx(&cc, decode_combine_kernel<D, V2>, p);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

cudaError_t launch_decode_v1(const DecodeParams& p, int d, bool k8, int units, int cs, cudaStream_t s) {
  if (k8) return d == 64 ? launch_decode<64, false, true>(p, units, cs, s) : launch_decode<128, false, true>(p, units, cs, s);
  return d == 64 ? launch_decode<64, false, false>(p, units, cs, s) : launch_decode<128, false, false>(p, units, cs, s);
}

cudaError_t launch_decode_v2_d128(const DecodeParams& p, bool k8, int units, int cs, cudaStream_t s) {
  return k8 ? launch_decode<128, true, true>(p, units, cs, s) : launch_decode<128, true, false>(p, units, cs, s);
}

}  // namespace da
