// Instantiations and dispatch of the tcgen05 decode kernel (draft trees up to
// 32 rows per KV head, head_dim 128, bf16): flat and cluster partitions.
#include "decode_tc.cuh"
#include "internal.h"

namespace da {

template <class F>
static cudaError_t with_tc_kernel(bool cluster, F&& f) {
  return cluster ? f(decode_tc_kernel<true>) : f(decode_tc_kernel<false>);
}

cudaError_t tc_prepare(const Choice& c, int cluster) {
  return with_tc_kernel(cluster > 0, [&](auto kern) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)c.smem);
    if (e == cudaSuccess && cluster > 8)
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return e;
  });
}

int tc_max_active_clusters(const Choice& c, int cluster) {
  int n = 0;
  const cudaError_t e = with_tc_kernel(true, [&](auto kern) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)cluster);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = c.smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
  });
  if (e != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t tc_launch(const Choice& c, const DecodeArgs& a, const CUtensorMap& mk,
                      const CUtensorMap& mv, const CUtensorMap& ms, cudaStream_t st) {
  return with_tc_kernel(c.cluster > 0, [&](auto kern) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(c.cluster > 0 ? (unsigned)(a.B * a.H_kv * c.cluster) : (unsigned)a.n_cta);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = c.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    int na = 1;
    if (c.cluster > 0) {
      attr[1].id = cudaLaunchAttributeClusterDimension;
      attr[1].val.clusterDim.x = (unsigned)c.cluster;
      attr[1].val.clusterDim.y = 1;
      attr[1].val.clusterDim.z = 1;
      na = 2;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, a, mk, mv, ms, c.stages);
  });
}

}  // namespace da
