// Instantiations and dispatch of the split-KV decode kernel.
#include "decode.cuh"
#include "internal.h"

namespace da {

bool choose_kernel(int dtype, int d, int rows, int batch, int max_smem, Choice* c) {
  const int es = dtype == DA_DTYPE_BF16 ? 2 : 4;
  if (rows <= 8) {
    c->engine = DA_ENGINE_CUDA_CORE;
    c->rk = rows <= 1 ? 1 : rows <= 2 ? 2 : rows <= 4 ? 4 : 8;
  } else if (rows <= 32 && dtype == DA_DTYPE_BF16) {
    c->engine = DA_ENGINE_MMA;
    c->rk = 32;
  } else {
    return false;
  }
  for (int s = 4; s >= 2; --s) {
    const Layout L = make_layout(c->engine, es, d, c->rk, s, batch);
    if ((int)L.total <= max_smem) {
      c->stages = s;
      c->smem = L.total;
      return true;
    }
  }
  return false;
}

// Calls f(kernel) with the decode kernel instance for (choice, dtype, d).
template <class F>
static cudaError_t with_kernel(const Choice& c, int dtype, int d, F&& f) {
  using bf = __nv_bfloat16;
  if (c.engine == DA_ENGINE_MMA) {
    if (dtype != DA_DTYPE_BF16) return cudaErrorInvalidValue;
    if (d == 128) return f(decode_kernel<bf, 128, MmaEngine<128>, 1, 32>);
    return f(decode_kernel<bf, 64, MmaEngine<64>, 1, 32>);
  }
#define DA_CORE(T, D, RK) \
  if (dtype == (sizeof(T) == 2 ? DA_DTYPE_BF16 : DA_DTYPE_FP32) && d == D && c.rk == RK) \
    return f(decode_kernel<T, D, CoreEngine<T, D, RK>, 0, RK>);
  DA_CORE(bf, 128, 1) DA_CORE(bf, 128, 2) DA_CORE(bf, 128, 4) DA_CORE(bf, 128, 8)
  DA_CORE(bf, 64, 1) DA_CORE(bf, 64, 2) DA_CORE(bf, 64, 4) DA_CORE(bf, 64, 8)
  DA_CORE(float, 128, 1) DA_CORE(float, 128, 2) DA_CORE(float, 128, 4) DA_CORE(float, 128, 8)
  DA_CORE(float, 64, 1) DA_CORE(float, 64, 2) DA_CORE(float, 64, 4) DA_CORE(float, 64, 8)
#undef DA_CORE
  return cudaErrorInvalidValue;
}

cudaError_t prepare_decode(const Choice& c, int dtype, int d) {
  return with_kernel(c, dtype, d, [&](auto kern) {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)c.smem);
  });
}

cudaError_t launch_decode(const Choice& c, int dtype, int d, const DecodeArgs& a,
                          const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& ms,
                          cudaStream_t st) {
  return with_kernel(c, dtype, d, [&](auto kern) {
    kern<<<a.n_cta, kThreads, c.smem, st>>>(a, mk, mv, ms, c.stages);
    return cudaGetLastError();
  });
}

}  // namespace da
