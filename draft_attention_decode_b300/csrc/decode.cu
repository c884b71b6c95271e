// Instantiations and dispatch of the split-KV decode kernel.
#include <type_traits>

#include "decode_tc.cuh"
#include "internal.h"

namespace da {

bool choose_kernel(int dtype, int d, int rows, int batch, int mode, int engine_hint, int stages,
                   int max_smem, bool side_f8, Choice* c) {
  const int es = dtype == DA_DTYPE_BF16 ? 2 : 4;
  // Automatic choice: 17..32 rows (draft trees over a GQA group) scanning a
  // long selection (full, FOLD, SharpDraft) go to the tcgen05 kernel; measured
  // on the ragged draft-tree workload it reads 0.90 of the copy bandwidth
  // there against 0.86 on mma.sync.  A window's single short piece per CTA
  // stays on mma.sync (0.55 against 0.46).
  if (engine_hint == 0 && dtype == DA_DTYPE_BF16 && d == 128 && rows > 16 && rows <= kTcRows &&
      !side_f8 && mode != DA_MODE_WINDOW && stages <= kTcMaxStages) {
    Choice t = *c;
    if (choose_kernel(dtype, d, rows, batch, mode, 3, stages, max_smem, side_f8, &t)) {
      *c = t;
      return true;
    }
  }
  if (engine_hint == 3) {
    // the tcgen05 kernel: bf16, head_dim 128, up to 32 rows, no FP8 side cache
    if (dtype != DA_DTYPE_BF16 || d != 128 || rows > kTcRows || side_f8) return false;
    if (stages > kTcMaxStages) return false;
    c->engine = DA_ENGINE_TC05;
    c->variant = kVariantTc;
    c->rk = kTcRows;
    c->pingpong = false;
    c->side_f8 = false;
    const int hi = stages > 0 ? stages : kTcMaxStages, lo = stages > 0 ? stages : 2;
    for (int s = hi; s >= lo; --s) {
      const TcLayout L = make_tc_layout(s, batch);
      if (tc_layout_check(L, s, batch) != 0) continue;
      if ((int)L.total <= max_smem) {
        c->stages = s;
        c->smem = L.total;
        return true;
      }
    }
    return false;
  }
  // Rows of one KV head that share every key: up to 4 stay on the FP32 pipes;
  // from 5 on, QK^T and PV are dense enough for an n8 tensor-core tile
  // (bf16 only).  An FP8 side cache goes to the tensor cores at any row count:
  // there its codes widen to f16 in one cvt per pair and feed the MMA, while
  // on the FP32 pipes the widening makes the far scan issue-bound.
  // engine_hint 1/2 forces the CUDA cores / tensor cores.
  bool mma = dtype == DA_DTYPE_BF16 && (rows > 4 || side_f8);
  if (engine_hint == 1) mma = false;
  if (engine_hint == 2) mma = true;
  c->pingpong = false;
  c->side_f8 = side_f8;
  // The FP8 side cache (FOLD): the turn-taking CUDA-core engine (<= 4 rows) or
  // the tensor-core engine, bf16, head_dim 128.
  if (side_f8 && (dtype != DA_DTYPE_BF16 || mode != DA_MODE_FOLD || (!mma && rows > 4)))
    return false;
  if (mma) {
    if (dtype != DA_DTYPE_BF16 || rows > 32) return false;
    c->engine = DA_ENGINE_MMA;
    c->variant = kVariantMma;
    c->rk = rows <= 8 ? 8 : rows <= 16 ? 16 : 32;
  } else {
    if (rows > 8) return false;
    c->engine = DA_ENGINE_CUDA_CORE;
    c->rk = rows <= 1 ? 1 : rows <= 2 ? 2 : rows <= 4 ? 4 : 8;
    c->variant = kVariantCore;
    // Turn-taking warp groups pay off on long selections (full, FOLD,
    // SharpDraft); a window's few pages per CTA keep all eight warps together.
    c->pingpong = c->rk <= 4 && mode != DA_MODE_WINDOW;
  }
  // Deepest pipeline that fits (a requested depth must fit as it is).
  const int s_hi = stages > 0 ? stages : (c->pingpong ? kMaxAutoStagesCore : kMaxAutoStages);
  const int s_lo = stages > 0 ? stages : 2;
  for (int s = s_hi; s >= s_lo; --s) {
    const Layout L = make_layout(c->variant, es, d, c->rk, s, batch);
    if (layout_check(L, c->variant, es, d, c->rk, s, batch) != 0) continue;
    if ((int)L.total <= max_smem) {
      c->stages = s;
      c->smem = L.total;
      return true;
    }
  }
  return false;
}

bool fit_cluster(Choice* c, int dtype, int d, int batch, int cluster, int stages, int max_smem) {
  c->cluster = cluster;
  if (c->engine == DA_ENGINE_TC05) return true;   // its partials stay in its own stages
  const int es = dtype == DA_DTYPE_BF16 ? 2 : 4;
  const int s_hi = stages > 0 ? stages : kMaxAutoStages, s_lo = stages > 0 ? stages : 2;
  for (int s = s_hi; s >= s_lo; --s) {
    const Layout L = make_layout(c->variant, es, d, c->rk, s, batch, cluster);
    if (layout_check(L, c->variant, es, d, c->rk, s, batch, cluster) != 0) continue;
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
  // The FP8 side-cache instances first: they take precedence over the engine's others.
  if (c.side_f8 && c.engine == DA_ENGINE_MMA) {
    if (dtype != DA_DTYPE_BF16) return cudaErrorInvalidValue;
#define DA_MMA_F8(D, NT, SPLIT, RK) \
  if (d == D && c.rk == RK) return f(decode_kernel<bf, D, MmaEngine<D, NT, SPLIT, true>, 1, RK>);
    DA_MMA_F8(128, 1, true, 8) DA_MMA_F8(128, 2, true, 16) DA_MMA_F8(128, 2, false, 32)
    DA_MMA_F8(64, 1, true, 8) DA_MMA_F8(64, 2, true, 16) DA_MMA_F8(64, 2, false, 32)
#undef DA_MMA_F8
    return cudaErrorInvalidValue;
  }
  if (c.engine == DA_ENGINE_MMA) {
    if (dtype != DA_DTYPE_BF16) return cudaErrorInvalidValue;
#define DA_MMA(D, NT, SPLIT, RK) \
  if (d == D && c.rk == RK) return f(decode_kernel<bf, D, MmaEngine<D, NT, SPLIT>, 1, RK>);
    DA_MMA(128, 1, true, 8) DA_MMA(128, 2, true, 16) DA_MMA(128, 2, false, 32)
    DA_MMA(64, 1, true, 8) DA_MMA(64, 2, true, 16) DA_MMA(64, 2, false, 32)
#undef DA_MMA
    return cudaErrorInvalidValue;
  }
  if (c.side_f8) {
    if (dtype != DA_DTYPE_BF16 || !c.pingpong) return cudaErrorInvalidValue;
#define DA_CORE_F8(D, RK)     \
  if (d == D && c.rk == RK) \
    return f(decode_kernel<bf, D, CoreEngine<bf, D, RK, true, true>, kVariantCore, RK>);
    DA_CORE_F8(128, 1) DA_CORE_F8(128, 2) DA_CORE_F8(128, 4)
    DA_CORE_F8(64, 1) DA_CORE_F8(64, 2) DA_CORE_F8(64, 4)
#undef DA_CORE_F8
    return cudaErrorInvalidValue;
  }
#define DA_CORE(T, D, RK)                                                                     \
  if (dtype == (sizeof(T) == 2 ? DA_DTYPE_BF16 : DA_DTYPE_FP32) && d == D && c.rk == RK) {       \
    if constexpr (RK <= 4) {                                                                     \
      if (c.pingpong)                                                                            \
        return f(decode_kernel<T, D, CoreEngine<T, D, RK, true>, kVariantCore, RK>);             \
      return f(decode_kernel<T, D, CoreEngine<T, D, RK, false>, kVariantCore, RK>);              \
    } else {                                                                                     \
      return f(decode_kernel<T, D, CoreEngineWide<T, D, RK>, kVariantCore, RK>);                 \
    }                                                                                            \
  }
  DA_CORE(bf, 128, 1) DA_CORE(bf, 128, 2) DA_CORE(bf, 128, 4) DA_CORE(bf, 128, 8)
  DA_CORE(bf, 64, 1) DA_CORE(bf, 64, 2) DA_CORE(bf, 64, 4) DA_CORE(bf, 64, 8)
  DA_CORE(float, 128, 1) DA_CORE(float, 128, 2) DA_CORE(float, 128, 4) DA_CORE(float, 128, 8)
  DA_CORE(float, 64, 1) DA_CORE(float, 64, 2) DA_CORE(float, 64, 4) DA_CORE(float, 64, 8)
#undef DA_CORE
  return cudaErrorInvalidValue;
}

cudaError_t prepare_decode(const Choice& c, int dtype, int d) {
  if (c.engine == DA_ENGINE_TC05) return tc_prepare(c, 0);
  return with_kernel(c, dtype, d, [&](auto kern) {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)c.smem);
  });
}

cudaError_t launch_decode(const Choice& c, int dtype, int d, const DecodeArgs& a,
                          const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& ms,
                          cudaStream_t st) {
  if (c.engine == DA_ENGINE_TC05) return tc_launch(c, a, mk, mv, ms, st);
  return with_kernel(c, dtype, d, [&](auto kern) {
    return launch_pdl(kern, dim3(a.n_cta), dim3(kThreads), c.smem, st, a, mk, mv, ms, c.stages);
  });
}

}  // namespace da
