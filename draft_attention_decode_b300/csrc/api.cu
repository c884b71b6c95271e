// The C ABI (include/draft_attn.h): host-side validation, plans, tensor-map
// encoding and launches.  No exceptions cross this boundary.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <mutex>
#include <new>

#include "internal.h"

// One status word per device; kernels OR DA_STATUS_* bits into it.
__device__ uint32_t g_da_status;

struct da_plan_s {
  da_params p;
  int device;
  int num_sms;
  int rows;
  da::Choice choice;
  size_t cnt_bytes;
  size_t ws_bytes;
  uint32_t* status;
  float2 turn_freq[64];   // theta^(-2i/d) / 2pi, split into hi + lo floats
  float scale_log2;
};

namespace {

constexpr int kAbiVersion = 101;

// FOLD's rotated-K ring: pages of sinks that keep their own slots.
int32_t ring_sink_pages(const da_params& p) {
  return p.n_sink > 0 ? (int32_t)(((int64_t)p.n_sink + da::kPage - 1) / da::kPage) : 0;
}

struct DeviceGuard {
  int prev = -1;
  bool ok = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) return;
    ok = (prev == dev) || cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D view of a cache array: rows = num_pages * H_kv * 64 tokens, columns =
// head_dim elements; box = 64 rows x 128 bytes with the 128-byte swizzle.
// pages: the cache array's page count (num_pages, or batch * k_ring_pages for
// FOLD's ring of rotated keys).
// fp8: the array holds one byte per element (FOLD's E4M3 side cache).
bool encode_cache_map(CUtensorMap* m, const void* base, const da_params& p, int64_t pages,
                      bool fp8 = false) {
  auto fn = encode_fn();
  if (!fn) return false;
  const int es = fp8 ? 1 : p.dtype == DA_DTYPE_BF16 ? 2 : 4;
  cuuint64_t gdim[2] = {(cuuint64_t)p.head_dim, (cuuint64_t)pages * p.num_kv_heads * da::kPage};
  cuuint64_t gstride[1] = {(cuuint64_t)p.head_dim * es};
  // fp8 rows of 64 bytes (head_dim 64) are copied whole and unswizzled
  const bool narrow = fp8 && p.head_dim * es < da::kSwizzleRow;
  cuuint32_t box[2] = {(cuuint32_t)(narrow ? p.head_dim : da::kSwizzleRow / es),
                       (cuuint32_t)da::kPage};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                  : p.dtype == DA_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                             : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                  2, const_cast<void*>(base), gdim, gstride, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE,
                  narrow ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

void fill_args(const da_plan_s* pl, da::DecodeArgs* a) {
  const da_params& p = pl->p;
  std::memset(a, 0, sizeof(*a));
  a->status = pl->status;
  a->B = p.batch;
  a->n_q = p.n_q;
  a->H_q = p.num_q_heads;
  a->H_kv = p.num_kv_heads;
  a->G = p.num_q_heads / p.num_kv_heads;
  a->R = pl->rows;
  a->max_pages = p.max_pages_per_seq;
  a->num_pages = p.num_pages;
  a->mode = p.mode;
  a->W = p.window;
  a->n_sink = (p.mode == DA_MODE_WINDOW || p.mode == DA_MODE_FOLD) ? p.n_sink : 0;
  a->n_tree = p.tree_size;
  a->alpha = p.alpha;
  a->far_mix = p.far_mix;
  a->far_kscale = p.side_fp8 == 1 ? p.side_scale : 1.f;
  a->beta = p.scale_slope;
  a->n_ref = p.scale_ref;
  a->scale_log2 = pl->scale_log2;
  a->n_cta = p.num_ctas;
  a->min_pages = p.min_pages_per_cta > 0 ? p.min_pages_per_cta : da::kMinPagesPerCta;
  a->k_ring = p.k_ring_pages;
  a->k_ring_sp = p.k_ring_pages > 0 ? ring_sink_pages(p) : 0;
  a->cluster = pl->choice.cluster;
  a->tables_ready = p.tables_ready == 1 && pl->choice.engine != DA_ENGINE_TC05;
  for (int i = 0; i < 64; ++i) a->turn_freq[i] = pl->turn_freq[i];
}

}  // namespace

namespace da {
bool plan_workspace_layout(const da_plan_s* pl, int* device, size_t* counter_bytes,
                           size_t* workspace_bytes) {
  if (!pl) return false;
  *device = pl->device;
  *counter_bytes = pl->cnt_bytes;
  *workspace_bytes = pl->ws_bytes;
  return true;
}
}  // namespace da

extern "C" {

int draft_attn_version(void) { return kAbiVersion; }

const char* draft_attn_error_string(int code) {
  switch (code) {
    case DA_OK: return "ok";
    case DA_ERR_INVALID_ARG: return "invalid argument";
    case DA_ERR_UNSUPPORTED: return "unsupported shape or parameter combination";
    case DA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case DA_ERR_CUDA: return "CUDA runtime error";
    case DA_ERR_DEVICE_FAULT: return "device status word reported a fault";
    default: return "unknown error";
  }
}

int draft_attn_check_params(const da_params* p) {
  if (!p) return DA_ERR_INVALID_ARG;
  if (p->batch < 1 || p->batch > da::kMaxBatch) return DA_ERR_INVALID_ARG;
  if (p->n_q < 1 || p->num_q_heads < 1 || p->num_kv_heads < 1) return DA_ERR_INVALID_ARG;
  if (p->num_q_heads % p->num_kv_heads != 0) return DA_ERR_INVALID_ARG;
  if (p->head_dim != 64 && p->head_dim != 128) return DA_ERR_INVALID_ARG;
  if (p->page_size != da::kPage) return DA_ERR_INVALID_ARG;
  if (p->num_pages < 1 || p->max_pages_per_seq < 1) return DA_ERR_INVALID_ARG;
  if ((int64_t)p->num_pages * p->num_kv_heads * da::kPage >= (int64_t)1 << 31)
    return DA_ERR_INVALID_ARG;
  // positions must stay below 2^24 (exact in FP32 for the RoPE angle)
  if ((int64_t)p->max_pages_per_seq * da::kPage > (int64_t)1 << 24) return DA_ERR_INVALID_ARG;
  if (p->dtype != DA_DTYPE_BF16 && p->dtype != DA_DTYPE_FP32) return DA_ERR_INVALID_ARG;
  if (p->mode < DA_MODE_FULL || p->mode > DA_MODE_SHARP) return DA_ERR_INVALID_ARG;
  if (!(p->rope_theta >= 0.0) || !std::isfinite(p->rope_theta)) return DA_ERR_INVALID_ARG;
  if (!(p->softmax_scale >= 0.f) || !std::isfinite(p->softmax_scale)) return DA_ERR_INVALID_ARG;
  if (p->num_ctas < 0 || p->num_ctas > 65535) return DA_ERR_INVALID_ARG;
  if (p->engine < 0 || p->engine > 3) return DA_ERR_INVALID_ARG;
  if (p->min_pages_per_cta < 0 || p->min_pages_per_cta > (1 << 20)) return DA_ERR_INVALID_ARG;
  if (p->stages != 0 && (p->stages < 2 || p->stages > 8)) return DA_ERR_INVALID_ARG;
  if (p->tree_size < 0 || p->tree_size > 64) return DA_ERR_INVALID_ARG;
  if (p->tree_size > 0 && (p->mode == DA_MODE_WINDOW || p->mode == DA_MODE_FOLD) &&
      p->tree_size > p->window)
    return DA_ERR_INVALID_ARG;
  if (p->tables_ready != 0 && p->tables_ready != 1) return DA_ERR_INVALID_ARG;
  if (p->cluster_ctas < -1 || p->cluster_ctas > 16) return DA_ERR_INVALID_ARG;
  if (p->cluster_ctas > 0 &&
      (p->mode != DA_MODE_WINDOW || p->num_ctas != 0 || p->min_pages_per_cta != 0))
    return DA_ERR_INVALID_ARG;
  if (p->side_fp8 != 0 && p->side_fp8 != 1) return DA_ERR_INVALID_ARG;
  if (p->side_fp8 == 1) {
    if (p->mode != DA_MODE_FOLD) return DA_ERR_INVALID_ARG;
    if (!(p->side_scale > 0.f) || !std::isfinite(p->side_scale)) return DA_ERR_INVALID_ARG;
  } else if (p->side_scale != 0.f) {
    return DA_ERR_INVALID_ARG;
  }
  if (p->k_ring_pages != 0) {   // FOLD's rotated K kept for the local keys only
    if (p->mode != DA_MODE_FOLD || p->window < 1) return DA_ERR_INVALID_ARG;
    if (p->n_sink < 0) return DA_ERR_INVALID_ARG;
    if (p->k_ring_pages < ring_sink_pages(*p) + (p->window + da::kPage - 1) / da::kPage + 1)
      return DA_ERR_INVALID_ARG;
    if ((int64_t)p->k_ring_pages * p->batch * p->num_kv_heads * da::kPage >= (int64_t)1 << 31)
      return DA_ERR_INVALID_ARG;
  }
  if (p->mode == DA_MODE_WINDOW || p->mode == DA_MODE_FOLD) {
    if (p->window < 1) return DA_ERR_INVALID_ARG;
  }
  if ((p->mode == DA_MODE_WINDOW || p->mode == DA_MODE_FOLD) && p->n_sink < 0)
    return DA_ERR_INVALID_ARG;
  if (p->mode == DA_MODE_FOLD) {
    if (!(p->alpha > 0.f) || !std::isfinite(p->alpha)) return DA_ERR_INVALID_ARG;
    if (!(p->far_mix >= 0.f && p->far_mix <= 1.f)) return DA_ERR_INVALID_ARG;
  }
  if (p->mode == DA_MODE_SHARP) {
    if (!(p->scale_slope >= 0.f) || !std::isfinite(p->scale_slope)) return DA_ERR_INVALID_ARG;
    if (p->scale_ref < 1) return DA_ERR_INVALID_ARG;
  }
  const int64_t rows = (int64_t)(p->num_q_heads / p->num_kv_heads) * p->n_q;
  if (rows > 32) return DA_ERR_UNSUPPORTED;
  if (rows > 8 && (p->dtype != DA_DTYPE_BF16 || p->engine == 1)) return DA_ERR_UNSUPPORTED;
  if (p->engine == 2 && p->dtype != DA_DTYPE_BF16) return DA_ERR_UNSUPPORTED;
  if (p->engine == 3 && (p->dtype != DA_DTYPE_BF16 || p->head_dim != 128 || p->side_fp8 == 1 ||
                         (p->stages != 0 && p->stages > 3)))
    return DA_ERR_UNSUPPORTED;
  // the FP8 side cache (bf16 caches): the tensor-core engine, or the
  // turn-taking CUDA-core engine up to 4 rows
  if (p->side_fp8 == 1 && (p->dtype != DA_DTYPE_BF16 || (p->engine == 1 && rows > 4)))
    return DA_ERR_UNSUPPORTED;
  return DA_OK;
}

int draft_attn_plan(const da_params* params, int device, da_plan_t* plan, size_t* workspace_bytes) {
  if (!plan) return DA_ERR_INVALID_ARG;
  *plan = nullptr;
  int rc = draft_attn_check_params(params);
  if (rc != DA_OK) return rc;
  DeviceGuard g(device);
  if (!g.ok) return DA_ERR_CUDA;
  int sms = 0, max_smem = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) !=
          cudaSuccess)
    return DA_ERR_CUDA;
  da_plan_s* pl = new (std::nothrow) da_plan_s();
  if (!pl) return DA_ERR_CUDA;
  pl->p = *params;
  pl->device = device;
  pl->num_sms = sms;
  pl->rows = (params->num_q_heads / params->num_kv_heads) * params->n_q;
  if (!da::choose_kernel(params->dtype, params->head_dim, pl->rows, params->batch, params->mode,
                         params->engine, params->stages, max_smem, params->side_fp8 == 1,
                         &pl->choice)) {
    delete pl;
    return DA_ERR_UNSUPPORTED;
  }
  if (pl->p.num_ctas == 0) pl->p.num_ctas = sms;  // one persistent CTA per SM
  // Window mode: one cluster of CTAs per (sequence, KV head) when asked for,
  // or, automatically, when every such cluster can be resident at once (the
  // selection of a window is short: its latency, not the grid's reach, is
  // what the partition has to minimise).
  pl->choice.cluster = 0;
  if (params->mode == DA_MODE_WINDOW && params->cluster_ctas != -1 &&
      da::cluster_supported(pl->choice, params->dtype, params->head_dim)) {
    const int64_t heads = (int64_t)params->batch * params->num_kv_heads;
    const int64_t pmax = ring_sink_pages(*params) + (params->window + da::kPage - 1) / da::kPage + 1;
    const int dt = params->dtype, hd = params->head_dim;
    da::Choice cc = pl->choice;
    int C = 0;
    if (params->cluster_ctas > 0) {
      if (!da::fit_cluster(&cc, dt, hd, params->batch, params->cluster_ctas, params->stages,
                           max_smem)) {
        delete pl;
        return DA_ERR_UNSUPPORTED;
      }
      C = params->cluster_ctas;
    } else if (params->num_ctas == 0 && params->min_pages_per_cta == 0 && heads <= sms) {
      int64_t c = sms / heads;
      c = c < 16 ? c : 16;
      c = c < pmax ? c : pmax;
      for (; c >= 1 && C == 0; --c) {
        da::Choice t = pl->choice;
        if (!da::fit_cluster(&t, dt, hd, params->batch, (int)c, params->stages, max_smem)) continue;
        if (da::prepare_cluster(t, dt, hd, (int)c) != cudaSuccess) {
          cudaGetLastError();
          continue;
        }
        if (da::max_active_clusters(t, dt, hd, (int)c) >= heads) {
          cc = t;
          C = (int)c;
        }
      }
      // The fewest CTAs whose longest stretch is as short as with C: the
      // same critical path, fewer partials to push and merge (33 pages: 9
      // CTAs of at most 4 pages instead of 10).
      if (C > 1) {
        const int64_t per = (pmax + C - 1) / C;
        const int c2 = (int)((pmax + per - 1) / per);
        da::Choice t = pl->choice;
        if (c2 < C && da::fit_cluster(&t, dt, hd, params->batch, c2, params->stages, max_smem) &&
            da::prepare_cluster(t, dt, hd, c2) == cudaSuccess) {
          cc = t;
          C = c2;
        } else {
          cudaGetLastError();
        }
      }
    }
    if (C > 0) {
      if (da::prepare_cluster(cc, dt, hd, C) != cudaSuccess) {
        delete pl;
        return DA_ERR_CUDA;
      }
      pl->choice = cc;
    }
  }
  const int d = params->head_dim;
  // workspace: per-(b, kv head) page counters, then the partial (m, l, o) slots
  pl->cnt_bytes = ((size_t)params->batch * params->num_kv_heads * 4 + 255) / 256 * 256;
  const size_t slots = (size_t)pl->p.num_ctas + (size_t)2 * params->batch * params->num_kv_heads;
  pl->ws_bytes = pl->cnt_bytes + slots * (size_t)da::slot_floats(pl->choice.rk, d) * sizeof(float);
  for (int i = 0; i < 64; ++i) {
    // turns per position, theta^(-2i/d) / 2pi, as hi + lo floats (rope_cos_sin);
    // theta = 0: NoPE, every angle is zero
    const double f = (i < d / 2 && params->rope_theta > 0.0)
                         ? std::pow(params->rope_theta, -2.0 * i / d) / (2.0 * M_PI)
                         : 0.0;
    const float hi = (float)f;
    pl->turn_freq[i] = make_float2(hi, (float)(f - (double)hi));
  }
  const double c = params->softmax_scale > 0.f ? (double)params->softmax_scale
                                               : 1.0 / std::sqrt((double)d);
  pl->scale_log2 = (float)(c * 1.4426950408889634074);  // log2(e)
  void* sp = nullptr;
  if (cudaGetSymbolAddress(&sp, g_da_status) != cudaSuccess ||
      da::prepare_decode(pl->choice, params->dtype, d) != cudaSuccess) {
    delete pl;
    return DA_ERR_CUDA;
  }
  pl->status = static_cast<uint32_t*>(sp);
  *plan = pl;
  if (workspace_bytes) *workspace_bytes = pl->ws_bytes;
  return DA_OK;
}

int draft_attn_plan_info(da_plan_t pl, da_plan_info* info) {
  if (!pl || !info) return DA_ERR_INVALID_ARG;
  std::memset(info, 0, sizeof(*info));
  info->num_ctas = pl->p.num_ctas;
  info->num_sms = pl->num_sms;
  info->rows_per_kv_head = pl->rows;
  info->kernel_rows = pl->choice.rk;
  info->engine = pl->choice.engine;
  info->stages = pl->choice.stages;
  info->smem_bytes = (int32_t)pl->choice.smem;
  info->cluster_ctas = pl->choice.cluster;
  if (pl->choice.cluster > 0)
    info->num_ctas = pl->p.batch * pl->p.num_kv_heads * pl->choice.cluster;
  info->workspace_bytes = pl->ws_bytes;
  return DA_OK;
}

void draft_attn_plan_destroy(da_plan_t pl) { delete pl; }

int draft_attn_append_kv(da_plan_t pl, const void* k_new, const void* v_new, const int32_t* pos,
                         int32_t batch, int32_t n_new, const int32_t* block_table, void* k_cache,
                         void* v_cache, void* k_side, void* stream) {
  if (!pl || batch < 0 || batch > pl->p.batch || n_new < 0) return DA_ERR_INVALID_ARG;
  if (pl->p.k_ring_pages > 0 && batch != pl->p.batch) return DA_ERR_INVALID_ARG;
  if (batch == 0 || n_new == 0) return DA_OK;
  if (!k_new || !v_new || !pos || !block_table || !k_cache || !v_cache) return DA_ERR_INVALID_ARG;
  if (pl->p.mode == DA_MODE_FOLD && !k_side) return DA_ERR_INVALID_ARG;
  DeviceGuard g(pl->device);
  if (!g.ok) return DA_ERR_CUDA;
  da::AppendArgs a;
  std::memset(&a, 0, sizeof(a));
  a.k = k_new;
  a.v = v_new;
  a.pos = pos;
  a.block_table = block_table;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.k_side = k_side;
  a.status = pl->status;
  a.B = batch;
  a.n_new = n_new;
  a.H_kv = pl->p.num_kv_heads;
  a.max_pages = pl->p.max_pages_per_seq;
  a.num_pages = pl->p.num_pages;
  a.k_ring = pl->p.k_ring_pages;
  a.k_ring_sp = pl->p.k_ring_pages > 0 ? ring_sink_pages(pl->p) : 0;
  a.side_f8 = pl->p.side_fp8;
  a.side_scale = pl->p.side_scale;
  for (int i = 0; i < 64; ++i) a.turn_freq[i] = pl->turn_freq[i];
  cudaError_t e = da::launch_append(pl->p.dtype, pl->p.head_dim, a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DA_OK : DA_ERR_CUDA;
}

int draft_attn_run(da_plan_t pl, const void* q, const int32_t* q_pos, const int32_t* ctx_lens,
                   const int32_t* block_table, const void* k_cache, const void* v_cache,
                   const void* k_side, void* out, void* workspace, size_t workspace_bytes,
                   void* stream) {
  return draft_attn_run_tree(pl, q, q_pos, ctx_lens, block_table, k_cache, v_cache, k_side,
                             nullptr, out, workspace, workspace_bytes, stream);
}

}  // extern "C"

namespace {

// Validation and argument set-up of an attention call, shared by the run and
// step entry points: everything that can fail on the host fails here, before
// any launch.
struct RunPrep {
  da::DecodeArgs a;
  CUtensorMap mk, mv, ms;
};

int prepare_run(da_plan_t pl, const void* q, const int32_t* q_pos, const int32_t* ctx_lens,
                const int32_t* block_table, const void* k_cache, const void* v_cache,
                const void* k_side, const uint64_t* tree_mask, void* out, void* workspace,
                size_t workspace_bytes, RunPrep* r) {
  if (!pl || !q || !q_pos || !ctx_lens || !block_table || !k_cache || !v_cache || !out ||
      !workspace)
    return DA_ERR_INVALID_ARG;
  const bool fold = pl->p.mode == DA_MODE_FOLD;
  if (fold && !k_side) return DA_ERR_INVALID_ARG;
  if (!aligned(workspace, 256) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      (k_side && !aligned(k_side, 16)))
    return DA_ERR_INVALID_ARG;
  if (workspace_bytes < pl->ws_bytes) return DA_ERR_WORKSPACE_TOO_SMALL;
  const int64_t k_pages = pl->p.k_ring_pages > 0 ? (int64_t)pl->p.k_ring_pages * pl->p.batch
                                                 : (int64_t)pl->p.num_pages;
  if (!encode_cache_map(&r->mk, k_cache, pl->p, k_pages) ||
      !encode_cache_map(&r->mv, v_cache, pl->p, pl->p.num_pages))
    return DA_ERR_CUDA;
  if (fold) {
    if (!encode_cache_map(&r->ms, k_side, pl->p, pl->p.num_pages, pl->p.side_fp8 == 1))
      return DA_ERR_CUDA;
  } else {
    r->ms = r->mk;
  }
  da::DecodeArgs& a = r->a;
  fill_args(pl, &a);
  a.q = q;
  a.q_pos = q_pos;
  a.ctx_lens = ctx_lens;
  a.block_table = block_table;
  a.tree_mask = pl->p.tree_size > 0 ? tree_mask : nullptr;
  a.out = out;
  a.cnt = static_cast<uint32_t*>(workspace);
  a.part = reinterpret_cast<float*>(static_cast<char*>(workspace) + pl->cnt_bytes);
  return DA_OK;
}

int launch_run(da_plan_t pl, const RunPrep& r, void* stream) {
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const cudaError_t e =
      pl->choice.cluster > 0
          ? da::launch_cluster(pl->choice, pl->p.dtype, pl->p.head_dim, r.a, r.mk, r.mv, r.ms, st)
          : da::launch_decode(pl->choice, pl->p.dtype, pl->p.head_dim, r.a, r.mk, r.mv, r.ms, st);
  return e == cudaSuccess ? DA_OK : DA_ERR_CUDA;
}

}  // namespace

extern "C" {

int draft_attn_run_tree(da_plan_t pl, const void* q, const int32_t* q_pos,
                        const int32_t* ctx_lens, const int32_t* block_table,
                        const void* k_cache, const void* v_cache, const void* k_side,
                        const uint64_t* tree_mask, void* out, void* workspace,
                        size_t workspace_bytes, void* stream) {
  if (!pl) return DA_ERR_INVALID_ARG;
  DeviceGuard g(pl->device);
  if (!g.ok) return DA_ERR_CUDA;
  RunPrep r;
  const int rc = prepare_run(pl, q, q_pos, ctx_lens, block_table, k_cache, v_cache, k_side,
                             tree_mask, out, workspace, workspace_bytes, &r);
  return rc != DA_OK ? rc : launch_run(pl, r, stream);
}

int draft_attn_step(da_plan_t pl, const void* k_new, const void* v_new, const int32_t* pos,
                    int32_t n_new, const void* q, const int32_t* q_pos, const int32_t* ctx_lens,
                    const int32_t* block_table, void* k_cache, void* v_cache, void* k_side,
                    const uint64_t* tree_mask, void* out, void* workspace,
                    size_t workspace_bytes, void* stream) {
  if (n_new < 0) return DA_ERR_INVALID_ARG;
  if (n_new > 32) return DA_ERR_UNSUPPORTED;
  if (!pl || (n_new > 0 && (!k_new || !v_new || !pos))) return DA_ERR_INVALID_ARG;
  DeviceGuard g(pl->device);
  if (!g.ok) return DA_ERR_CUDA;
  RunPrep r;
  int rc = prepare_run(pl, q, q_pos, ctx_lens, block_table, k_cache, v_cache, k_side, tree_mask,
                       out, workspace, workspace_bytes, &r);
  if (rc != DA_OK) return rc;
  if (pl->choice.cluster > 0 && pl->choice.engine != DA_ENGINE_TC05 && n_new > 0 &&
      n_new <= da::kMaxFusedNew) {
    // The cluster partition appends the tokens itself: one launch per step.
    r.a.k_new = k_new;
    r.a.v_new = v_new;
    r.a.new_pos = pos;
    r.a.k_cache_w = k_cache;
    r.a.v_cache_w = v_cache;
    r.a.n_new = n_new;
    r.a.inputs_ready = 0;
    return launch_run(pl, r, stream);
  }
  r.a.inputs_ready = n_new > 0 && pl->p.batch > 0;
  // The append runs first; the attention kernel is launched behind it with
  // programmatic dependent launch.  Its set-up, the block-table reads and the
  // query preparation overlap the append; only its first cache load waits
  // for the append to finish.
  rc = draft_attn_append_kv(pl, k_new, v_new, pos, pl->p.batch, n_new, block_table, k_cache,
                            v_cache, k_side, stream);
  return rc != DA_OK ? rc : launch_run(pl, r, stream);
}

int draft_attn_debug_gather(da_plan_t pl, const int32_t* q_pos, const int32_t* ctx_lens,
                            const int32_t* block_table, const uint64_t* tree_mask, int32_t b,
                            int32_t t, int32_t* positions,
                            int64_t* phys_slot, int32_t* key_rope_pos, int32_t* q_rope_pos,
                            int8_t* segment, int64_t capacity, int64_t* count, void* stream) {
  if (!pl || !q_pos || !ctx_lens || !block_table || !count || capacity < 0) return DA_ERR_INVALID_ARG;
  if (b < 0 || b >= pl->p.batch || t < 0 || t >= pl->p.n_q) return DA_ERR_INVALID_ARG;
  if (capacity > 0 && (!positions || !phys_slot || !key_rope_pos || !q_rope_pos || !segment))
    return DA_ERR_INVALID_ARG;
  DeviceGuard g(pl->device);
  if (!g.ok) return DA_ERR_CUDA;
  da::DecodeArgs a;
  fill_args(pl, &a);
  a.q_pos = q_pos;
  a.ctx_lens = ctx_lens;
  a.block_table = block_table;
  a.tree_mask = pl->p.tree_size > 0 ? tree_mask : nullptr;
  da::GatherOut o{positions, phys_slot, key_rope_pos, q_rope_pos, segment, capacity, count};
  return da::launch_gather(a, b, t, o, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? DA_OK
             : DA_ERR_CUDA;
}

int draft_attn_ring_size(int32_t window, int32_t n_sink, int32_t* n_ring, int32_t* n_sink_pages) {
  if (window < 1 || n_sink < 0 || !n_ring || !n_sink_pages) return DA_ERR_INVALID_ARG;
  const int64_t sp = ((int64_t)n_sink + da::kPage - 1) / da::kPage;
  const int64_t wp = ((int64_t)window + da::kPage - 1) / da::kPage + 1;
  if (sp + wp > INT32_MAX) return DA_ERR_INVALID_ARG;
  *n_sink_pages = (int32_t)sp;
  *n_ring = (int32_t)(sp + wp);
  return DA_OK;
}

int draft_attn_ring_block_table(int32_t* table, int64_t max_pages, const int32_t* ring_pages,
                                int32_t n_ring, int32_t n_sink_pages) {
  if (!table || !ring_pages || max_pages < 1 || n_sink_pages < 0 || n_ring <= n_sink_pages)
    return DA_ERR_INVALID_ARG;
  const int64_t cycle = n_ring - n_sink_pages;
  for (int64_t j = 0; j < max_pages; ++j)
    table[j] = j < n_sink_pages ? ring_pages[j] : ring_pages[n_sink_pages + (j - n_sink_pages) % cycle];
  return DA_OK;
}

int draft_attn_debug_wait_timeout(da_plan_t pl, void* stream) {
  if (!pl) return DA_ERR_INVALID_ARG;
  DeviceGuard g(pl->device);
  if (!g.ok) return DA_ERR_CUDA;
  return da::launch_wait_timeout(pl->status, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? DA_OK
             : DA_ERR_CUDA;
}

int draft_attn_get_status(da_plan_t pl, void* stream, uint32_t* bits) {
  if (!pl) return DA_ERR_INVALID_ARG;
  DeviceGuard g(pl->device);
  if (!g.ok) return DA_ERR_CUDA;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return DA_ERR_CUDA;
  uint32_t v = 0;
  if (cudaMemcpy(&v, pl->status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess)
    return DA_ERR_CUDA;
  if (v) {
    const uint32_t zero = 0;
    if (cudaMemcpy(pl->status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
      return DA_ERR_CUDA;
  }
  if (bits) *bits = v;
  return v ? DA_ERR_DEVICE_FAULT : DA_OK;
}

}  // extern "C"
