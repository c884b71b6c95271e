// Instantiations and dispatch of the decode kernel's cluster partition: one
// thread-block cluster of CTAs per (sequence, KV head), the partials merged
// through distributed shared memory (see decode_kernel).
#include "decode.cuh"
#include "internal.h"

namespace da {

// Calls f(kernel) with the cluster-partition instance for (choice, dtype, d):
// the shared-step engines only (no turn-taking warp groups, no FP8 side cache).
template <class F>
static cudaError_t with_cluster_kernel(const Choice& c, int dtype, int d, F&& f) {
  using bf = __nv_bfloat16;
  if (c.side_f8 || c.pingpong) return cudaErrorInvalidValue;
  if (c.engine == DA_ENGINE_MMA) {
    if (dtype != DA_DTYPE_BF16) return cudaErrorInvalidValue;
#define DA_MMA(D, NT, SPLIT, RK) \
  if (d == D && c.rk == RK) return f(decode_kernel<bf, D, MmaEngine<D, NT, SPLIT>, 1, RK, true>);
    DA_MMA(128, 1, true, 8) DA_MMA(128, 2, true, 16) DA_MMA(128, 2, false, 32)
    DA_MMA(64, 1, true, 8) DA_MMA(64, 2, true, 16) DA_MMA(64, 2, false, 32)
#undef DA_MMA
    return cudaErrorInvalidValue;
  }
#define DA_CORE(T, D, RK)                                                                       \
  if (dtype == (sizeof(T) == 2 ? DA_DTYPE_BF16 : DA_DTYPE_FP32) && d == D && c.rk == RK) {       \
    if constexpr (RK <= 4)                                                                       \
      return f(decode_kernel<T, D, CoreEngine<T, D, RK, false>, kVariantCore, RK, true>);        \
    else                                                                                         \
      return f(decode_kernel<T, D, CoreEngineWide<T, D, RK>, kVariantCore, RK, true>);           \
  }
  DA_CORE(bf, 128, 1) DA_CORE(bf, 128, 2) DA_CORE(bf, 128, 4) DA_CORE(bf, 128, 8)
  DA_CORE(bf, 64, 1) DA_CORE(bf, 64, 2) DA_CORE(bf, 64, 4) DA_CORE(bf, 64, 8)
  DA_CORE(float, 128, 1) DA_CORE(float, 128, 2) DA_CORE(float, 128, 4) DA_CORE(float, 128, 8)
  DA_CORE(float, 64, 1) DA_CORE(float, 64, 2) DA_CORE(float, 64, 4) DA_CORE(float, 64, 8)
#undef DA_CORE
  return cudaErrorInvalidValue;
}

bool cluster_supported(const Choice& c, int dtype, int d) {
  if (c.engine == DA_ENGINE_TC05) return true;
  return with_cluster_kernel(c, dtype, d, [](auto) { return cudaSuccess; }) == cudaSuccess;
}

cudaError_t prepare_cluster(const Choice& c, int dtype, int d, int cluster) {
  if (c.engine == DA_ENGINE_TC05) return tc_prepare(c, cluster);
  return with_cluster_kernel(c, dtype, d, [&](auto kern) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)c.smem);
    if (e == cudaSuccess && cluster > 8)
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return e;
  });
}

int max_active_clusters(const Choice& c, int dtype, int d, int cluster) {
  if (c.engine == DA_ENGINE_TC05) return tc_max_active_clusters(c, cluster);
  int n = 0;
  const cudaError_t e = with_cluster_kernel(c, dtype, d, [&](auto kern) {
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

cudaError_t launch_cluster(const Choice& c, int dtype, int d, const DecodeArgs& a,
                           const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& ms,
                           cudaStream_t st) {
  if (c.engine == DA_ENGINE_TC05) return tc_launch(c, a, mk, mv, ms, st);
  return with_cluster_kernel(c, dtype, d, [&](auto kern) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(a.B * a.H_kv * c.cluster));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = c.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)c.cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, a, mk, mv, ms, c.stages);
  });
}

}  // namespace da
