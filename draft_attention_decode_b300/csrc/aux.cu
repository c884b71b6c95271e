// KV append with RoPE, and the debug-gather hook.
#include "internal.h"

namespace da {

// ---------------------------------------------------------------------------
// KV append + RoPE.  One warp per (b, token, kv head); lane f handles the
// rotate-half pairs (f, f + d/2), f = lane, lane + 32.  Writes the rotated key
// to the K cache, the raw key to the FOLD side cache ("FOLD", review: the
// unrotated side cache) and the value to the V cache.  With side_f8 the side
// cache takes one byte per element: the E4M3 code of the float32 quotient
// k / side_scale (IEEE division), rounded to nearest even and saturated to
// the largest finite code by cvt's satfinite mode.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;   // lo's code in the low byte
}

template <typename T, int D>
__global__ void __launch_bounds__(256) append_kernel(const __grid_constant__ AppendArgs a) {
  // Wait for the predecessor first, then let the dependent start: a
  // dependent attention kernel (draft_attn_step) reads its inputs before its
  // own griddepcontrol.wait, relying on this order.
  grid_dep_wait();
  grid_dep_launch_dependents();
  const int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t total = (int64_t)a.B * a.n_new * a.H_kv;
  if (w >= total) return;
  const int h = (int)(w % a.H_kv);
  const int64_t bt_tok = w / a.H_kv;           // b * n_new + token
  const int b = (int)(bt_tok / a.n_new);
  // the token's K and V do not depend on where it goes: load them first
  const int64_t src = (bt_tok * a.H_kv + h) * D;
  const T* k = static_cast<const T*>(a.k) + src;
  const T* v = static_cast<const T*>(a.v) + src;
  T kx[D / 64], ky[D / 64], vx[D / 64], vy[D / 64];
#pragma unroll
  for (int u = 0; u < D / 64; ++u) {
    const int f = lane + 32 * u;
    kx[u] = k[f];
    ky[u] = k[f + D / 2];
    vx[u] = v[f];
    vy[u] = v[f + D / 2];
  }
  const int32_t pos = __ldg(a.pos + bt_tok);
  if (pos < 0) return;                          // padding token
  const int32_t pg = pos / kPage;
  if (pg >= a.max_pages) {
    if (lane == 0) atomicOr(a.status, DA_STATUS_BAD_POSITION);
    return;
  }
  const int32_t phys = __ldg(a.block_table + (int64_t)b * a.max_pages + pg);
  if (phys < 0 || phys >= a.num_pages) {
    if (lane == 0) atomicOr(a.status, DA_STATUS_BAD_PAGE);
    return;
  }
  const int64_t dst = (((int64_t)phys * a.H_kv + h) * kPage + (pos - pg * kPage)) * D;
  const int64_t kpage =
      a.k_ring > 0 ? (int64_t)b * a.k_ring + ring_slot(pg, a.k_ring, a.k_ring_sp) : phys;
  T* kc = static_cast<T*>(a.k_cache) + ((kpage * a.H_kv + h) * kPage + (pos - pg * kPage)) * D;
  T* vc = static_cast<T*>(a.v_cache) + dst;
  T* ks = (a.k_side && !a.side_f8) ? static_cast<T*>(a.k_side) + dst : nullptr;
  uint8_t* ks8 = (a.k_side && a.side_f8) ? static_cast<uint8_t*>(a.k_side) + dst : nullptr;
#pragma unroll
  for (int u = 0; u < D / 64; ++u) {
    const int f = lane + 32 * u;
    const float x = to_f32<T>(kx[u]), y = to_f32<T>(ky[u]);
    float c, s, xr, yr;
    rope_cos_sin(pos, a.turn_freq[f], c, s);
    rope_pair(x, y, c, s, xr, yr);
    kc[f] = from_f32<T>(xr);
    kc[f + D / 2] = from_f32<T>(yr);
    if (ks) {
      ks[f] = kx[u];
      ks[f + D / 2] = ky[u];
    }
    if (ks8) {
      const uint16_t c2 = e4m3x2(__fdiv_rn(x, a.side_scale), __fdiv_rn(y, a.side_scale));
      ks8[f] = (uint8_t)(c2 & 0xffu);
      ks8[f + D / 2] = (uint8_t)(c2 >> 8);
    }
    vc[f] = vx[u];
    vc[f + D / 2] = vy[u];
  }
}

cudaError_t launch_append(int dtype, int d, const AppendArgs& a, cudaStream_t st) {
  const int64_t warps = (int64_t)a.B * a.n_new * a.H_kv;
  if (warps == 0) return cudaSuccess;
  const int64_t blocks = (warps * 32 + 255) / 256;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const dim3 grid((unsigned)blocks);
  if (dtype == DA_DTYPE_BF16) {
    if (d == 128) return launch_pdl(append_kernel<__nv_bfloat16, 128>, grid, 256, 0, st, a);
    return launch_pdl(append_kernel<__nv_bfloat16, 64>, grid, 256, 0, st, a);
  }
  if (d == 128) return launch_pdl(append_kernel<float, 128>, grid, 256, 0, st, a);
  return launch_pdl(append_kernel<float, 64>, grid, 256, 0, st, a);
}

// ---------------------------------------------------------------------------
// Debug gather: the selection of query token t of sequence b, computed with
// the decode kernel's own routines (mode_ranges, fold_far_pos, phys_page).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) gather_kernel(const __grid_constant__ DecodeArgs a, int b,
                                                     int t, GatherOut o) {
  const int32_t L = clamp_ctx(__ldg(a.ctx_lens + b), a.max_pages, a.status);
  const int32_t p = __ldg(a.q_pos + b * a.n_q + t);
  const Ranges rg = mode_ranges(a.mode, L, a.W, a.n_sink);
  // the ranges in position order (they are disjoint): ord[0] < ord[1] < ord[2]
  int ord[kRanges] = {0, 1, 2};
  for (int i = 1; i < kRanges; ++i)
    for (int j = i; j > 0 && rg.lo(ord[j]) < rg.lo(ord[j - 1]); --j) {
      const int t = ord[j]; ord[j] = ord[j - 1]; ord[j - 1] = t;
    }
  int64_t cnt[kRanges];
  for (int i = 0; i < kRanges; ++i) {
    const int32_t k0 = rg.lo(ord[i]), k1 = rg.hi(ord[i]);
    cnt[i] = k1 > k0 ? k1 - k0 : 0;
  }
  const int64_t dense = cnt[0] + cnt[1] + cnt[2];
  // Draft-tree keys (the last `present` keys, all of them in the selection)
  // are kept only where the query's mask bit is set; they come last, so the
  // kept ones are compacted by a popcount of the lower bits.
  const bool masked = a.tree_mask != nullptr && a.n_tree > 0;
  const uint64_t m = masked ? (uint64_t)__ldg(reinterpret_cast<const unsigned long long*>(a.tree_mask) +
                                              b * a.n_q + t)
                            : ~0ull;
  const int32_t present = masked ? min(a.n_tree, L) : 0;
  const int32_t base = L - a.n_tree;              // position of tree token 0
  const int32_t lo_bit = a.n_tree - present;
  const uint64_t valid = present == 0 ? 0ull
                         : ((present >= 64 ? ~0ull : ((1ull << present) - 1)) << lo_bit);
  const int64_t n_before = dense - present;
  const int64_t total = n_before + __popcll(m & valid);
  if (blockIdx.x == 0 && threadIdx.x == 0) *o.count = total;
  const int32_t pf = fold_far_pos(L, a.W);
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < dense;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int oi = idx < cnt[0] ? 0 : (idx < cnt[0] + cnt[1] ? 1 : 2);
    const int rr = ord[oi];
    const int64_t before = oi == 0 ? 0 : (oi == 1 ? cnt[0] : cnt[0] + cnt[1]);
    const int32_t j = rg.lo(rr) + (int32_t)(idx - before);
    int64_t out = idx;
    if (idx >= n_before) {
      const int i = j - base;
      if (!((m >> i) & 1ull)) continue;
      out = n_before + __popcll(m & valid & ((1ull << i) - 1));
    }
    if (out >= o.capacity) continue;
    const bool far = range_is_far(a.mode, rr);
    const int32_t pg = j / kPage;
    const int32_t phys = phys_page(a.block_table, b, pg, a.max_pages, a.num_pages, a.status);
    o.positions[out] = j;
    o.phys_slot[out] = phys < 0 ? -1 : (int64_t)phys * kPage + (j - pg * kPage);
    o.key_rope_pos[out] = far ? pf : j;
    o.q_rope_pos[out] = far ? p - pf : p;
    o.segment[out] = far ? 1 : 0;
  }
}

cudaError_t launch_gather(const DecodeArgs& a, int b, int t, const GatherOut& o, cudaStream_t st) {
  gather_kernel<<<148, 256, 0, st>>>(a, b, t, o);
  return cudaGetLastError();
}

// The give-up path of the kernels' bounded wait: one warp waits, with the
// same mbar_wait, on an mbarrier that nothing ever arrives on.  After about
// 2^31 cycles the first thread to give up sets DA_STATUS_WAIT_TIMEOUT in the
// status word and raises the abort flag; the others then return at once.
__global__ void __launch_bounds__(32) wait_timeout_kernel(uint32_t* status) {
  __shared__ uint64_t bar;
  __shared__ int32_t abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  mbar_wait(&bar, 0u, status, &abort_flag);
}

cudaError_t launch_wait_timeout(uint32_t* status, cudaStream_t st) {
  wait_timeout_kernel<<<1, 32, 0, st>>>(status);
  return cudaGetLastError();
}

}  // namespace da
