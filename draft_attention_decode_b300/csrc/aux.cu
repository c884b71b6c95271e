// KV append with RoPE, the split combine pass, and the debug-gather hook.
#include "internal.h"

namespace da {

// ---------------------------------------------------------------------------
// KV append + RoPE.  One warp per (b, token, kv head); lane f handles the
// rotate-half pairs (f, f + d/2), f = lane, lane + 32.  Writes the rotated key
// to the K cache, the raw key to the FOLD side cache ("FOLD", review: the
// unrotated side cache) and the value to the V cache.
// ---------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(256) append_kernel(const __grid_constant__ AppendArgs a) {
  const int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t total = (int64_t)a.B * a.n_new * a.H_kv;
  if (w >= total) return;
  const int h = (int)(w % a.H_kv);
  const int64_t bt_tok = w / a.H_kv;           // b * n_new + token
  const int b = (int)(bt_tok / a.n_new);
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
  const int64_t src = (bt_tok * a.H_kv + h) * D;
  const int64_t dst = (((int64_t)phys * a.H_kv + h) * kPage + (pos - pg * kPage)) * D;
  const T* k = static_cast<const T*>(a.k) + src;
  const T* v = static_cast<const T*>(a.v) + src;
  T* kc = static_cast<T*>(a.k_cache) + dst;
  T* vc = static_cast<T*>(a.v_cache) + dst;
  T* ks = a.k_side ? static_cast<T*>(a.k_side) + dst : nullptr;
#pragma unroll
  for (int f = lane; f < D / 2; f += 32) {
    const T xr = k[f], yr = k[f + D / 2];
    const float x = to_f32<T>(xr), y = to_f32<T>(yr);
    float c, s;
    rope_cos_sin(pos, a.inv_freq[f], c, s);
    kc[f] = from_f32<T>(x * c - y * s);
    kc[f + D / 2] = from_f32<T>(y * c + x * s);
    if (ks) {
      ks[f] = xr;
      ks[f + D / 2] = yr;
    }
    vc[f] = v[f];
    vc[f + D / 2] = v[f + D / 2];
  }
}

cudaError_t launch_append(int dtype, int d, const AppendArgs& a, cudaStream_t st) {
  const int64_t warps = (int64_t)a.B * a.n_new * a.H_kv;
  if (warps == 0) return cudaSuccess;
  const int64_t blocks = (warps * 32 + 255) / 256;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const dim3 grid((unsigned)blocks);
  if (dtype == DA_DTYPE_BF16) {
    if (d == 128) append_kernel<__nv_bfloat16, 128><<<grid, 256, 0, st>>>(a);
    else append_kernel<__nv_bfloat16, 64><<<grid, 256, 0, st>>>(a);
  } else {
    if (d == 128) append_kernel<float, 128><<<grid, 256, 0, st>>>(a);
    else append_kernel<float, 64><<<grid, 256, 0, st>>>(a);
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Combine: for each (b, kv head) and query row, log-sum-exp merge of the
// pieces' partials of each softmax segment, then (FOLD) the far/local mix
// (1 - lambda_eff) o_loc + lambda_eff o_far, lambda_eff = 0 when the far
// memory is empty ("FOLD", abstract: separate control of the far memory's
// total weight).  One warp per row, lane owns d/32 dimensions.  CTAs whose
// page range is empty wrote no partial and are skipped.
// ---------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(256) combine_kernel(const __grid_constant__ DecodeArgs a, int RK) {
  constexpr int DPL = D / 32;
  const int b = blockIdx.x / a.H_kv, h = blockIdx.x - b * a.H_kv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t* pfx = a.pfx;
  const int64_t TP = (int64_t)pfx[2 * a.B] * a.H_kv;
  const int64_t slot_f = (int64_t)RK * (D + 2);
  const bool fold = a.mode == DA_MODE_FOLD;
  int64_t i0[2], i1[2], sq[2];
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    const int e = 2 * b + rr;
    const int32_t n = pfx[e + 1] - pfx[e];
    sq[rr] = (int64_t)e * a.H_kv + h;
    if (n == 0) {
      i0[rr] = 0;
      i1[rr] = -1;
    } else {
      const int64_t x0 = (int64_t)pfx[e] * a.H_kv + (int64_t)h * n;
      i0[rr] = cta_of(x0, TP, a.n_cta);
      i1[rr] = cta_of(x0 + n - 1, TP, a.n_cta);
    }
  }
  const float lam = (fold && pfx[2 * b + 1] > pfx[2 * b]) ? a.far_mix : 0.f;
  const int nseg = fold ? 2 : 1;
  for (int r = warp; r < a.R; r += 8) {
    float res[DPL];
#pragma unroll
    for (int e = 0; e < DPL; ++e) res[e] = 0.f;
    for (int seg = 0; seg < nseg; ++seg) {
      float M = -INFINITY;
      for (int rr = 0; rr < 2; ++rr) {
        if ((fold && rr == 0 ? 1 : 0) != seg) continue;
        for (int64_t i = i0[rr] + lane; i <= i1[rr]; i += 32)
          if (cta_begin(i, TP, a.n_cta) < cta_begin(i + 1, TP, a.n_cta))
            M = fmaxf(M, a.part[(i + sq[rr]) * slot_f + r]);
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      if (M == -INFINITY) continue;
      float O[DPL], Ls = 0.f;
#pragma unroll
      for (int e = 0; e < DPL; ++e) O[e] = 0.f;
      for (int rr = 0; rr < 2; ++rr) {
        if ((fold && rr == 0 ? 1 : 0) != seg) continue;
        for (int64_t i = i0[rr]; i <= i1[rr]; ++i) {
          if (cta_begin(i, TP, a.n_cta) == cta_begin(i + 1, TP, a.n_cta)) continue;
          const float* base = a.part + (i + sq[rr]) * slot_f;
          const float w = fast_exp2(base[r] - M);
          Ls += w * base[RK + r];
          const float* o = base + 2 * RK + (int64_t)r * D + lane * DPL;
#pragma unroll
          for (int e = 0; e < DPL; ++e) O[e] += w * o[e];
        }
      }
      const float wseg = fold ? (seg == 1 ? lam : 1.f - lam) : 1.f;
      if (Ls > 0.f) {
        const float inv = wseg / Ls;
#pragma unroll
        for (int e = 0; e < DPL; ++e) res[e] += O[e] * inv;
      }
    }
    const int t = r / a.G, j = r - t * a.G;
    T* out = static_cast<T*>(a.out) + ((int64_t)(b * a.n_q + t) * a.H_q + h * a.G + j) * D + lane * DPL;
#pragma unroll
    for (int e = 0; e < DPL; ++e) out[e] = from_f32<T>(res[e]);
  }
}

cudaError_t launch_combine(int dtype, int d, int rk, const DecodeArgs& a, cudaStream_t st) {
  const dim3 grid((unsigned)(a.B * a.H_kv));
  if (dtype == DA_DTYPE_BF16) {
    if (d == 128) combine_kernel<__nv_bfloat16, 128><<<grid, 256, 0, st>>>(a, rk);
    else combine_kernel<__nv_bfloat16, 64><<<grid, 256, 0, st>>>(a, rk);
  } else {
    if (d == 128) combine_kernel<float, 128><<<grid, 256, 0, st>>>(a, rk);
    else combine_kernel<float, 64><<<grid, 256, 0, st>>>(a, rk);
  }
  return cudaGetLastError();
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
  const int64_t n0 = rg.k1[0] > rg.k0[0] ? rg.k1[0] - rg.k0[0] : 0;
  const int64_t n1 = rg.k1[1] > rg.k0[1] ? rg.k1[1] - rg.k0[1] : 0;
  const int64_t total = n0 + n1;
  if (blockIdx.x == 0 && threadIdx.x == 0) *o.count = total;
  const int64_t lim = total < o.capacity ? total : o.capacity;
  const int32_t pf = fold_far_pos(L, a.W);
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < lim;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int rr = idx < n0 ? 0 : 1;
    const int32_t j = (rr ? rg.k0[1] : rg.k0[0]) + (int32_t)(idx < n0 ? idx : idx - n0);
    const bool far = range_is_far(a.mode, rr);
    const int32_t pg = j / kPage;
    const int32_t phys = phys_page(a.block_table, b, pg, a.max_pages, a.num_pages, a.status);
    o.positions[idx] = j;
    o.phys_slot[idx] = phys < 0 ? -1 : (int64_t)phys * kPage + (j - pg * kPage);
    o.key_rope_pos[idx] = far ? pf : j;
    o.q_rope_pos[idx] = far ? p - pf : p;
    o.segment[idx] = far ? 1 : 0;
  }
}

cudaError_t launch_gather(const DecodeArgs& a, int b, int t, const GatherOut& o, cudaStream_t st) {
  gather_kernel<<<148, 256, 0, st>>>(a, b, t, o);
  return cudaGetLastError();
}

}  // namespace da
