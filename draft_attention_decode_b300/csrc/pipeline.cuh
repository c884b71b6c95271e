// Split-KV decode pipeline shared by the two compute engines.
//
// One persistent CTA per SM: warp 8 is the producer, warps 0..7 consume.
// The CTA owns a contiguous stretch of the flat page line (see cta_begin in
// common.cuh).  For every page on it the producer translates the block table,
// then issues 2-D TMA loads of the page's K slab (from the rotated cache, or
// from the un-rotated side cache for FOLD far memory) and V slab into a ring
// of shared-memory stages, 128-byte swizzled.  The consumers run the online
// softmax over each page; at the end of each piece they merge their eight
// per-warp states and write one partial (m, l, o) per query row.
#pragma once

#include <type_traits>

#include "common.cuh"

namespace da {

enum : int { kFirst = 1, kLast = 2, kValid = 4 };

// Named barrier ids: 1 the consumer warps among themselves, 2 the end of the
// kernel (consumers arrive, the producer warp waits; see producer()).
constexpr int kEndBarrier = 2;

// Tree offset of a page with no draft-tree key under a mask.
constexpr int32_t kNoTree = -(1 << 30);

struct PageInfo {
  int32_t seq;    // piece id: piece_seq(mode, b, h, H_kv, range)
  int32_t lohi;   // first and one-past-last valid key in the page
  int32_t flags;
  int32_t toff;   // key k of the page is tree token k + toff (when in [0, 64))
};


// Shared-memory layout (host and device agree on it).
struct Layout {
  uint32_t stage_bytes, stages;
  uint32_t q_off, mo_off, ml_off, p_off, info_off, bar_off, invf_off, len_off, pfx_off, n0_off,
      n01_off, flag_off, tm_off, rm_off, recv_off, recv_slots, mbar_off, pnew_off, newpos_off,
      newkv_off, total;
};

__host__ __device__ inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

// Merge buffers hold `rm` rows per consumer warp: rk on the CUDA cores, 16
// on the tensor cores; the CUDA-core variant also keeps a per-warp
// probability buffer (used by the 5..8-row engine).
// recv_slots: cluster partition, the CTAs per cluster whose partials rank 0
// receives (0 for the flat partition).
__host__ __device__ inline Layout make_layout(int variant, int es, int d, int rk, int stages,
                                              int batch, int recv_slots = 0) {
  Layout L;
  L.stage_bytes = 2u * (uint32_t)(d * es / kSwizzleRow) * kBoxBytes;
  L.stages = stages;
  uint32_t off = L.stage_bytes * stages;
  const uint32_t ncw = (uint32_t)kConsumerWarps;
  const int rm = variant == kVariantMma ? 16 : rk;
  L.q_off = off;     off += align_up((uint32_t)rk * d * 4, 128);
  L.mo_off = off;    off += align_up(ncw * rm * d * 4, 128);
  L.ml_off = off;    off += align_up(ncw * rm * 8, 128);
  L.p_off = off;     off += variant == kVariantCore ? align_up(ncw * 9 * rk * 4, 128) : 0;
  L.info_off = off;  off += align_up((uint32_t)stages * sizeof(PageInfo), 128);
  L.bar_off = off;   off += align_up((uint32_t)stages * 16, 128);
  L.invf_off = off;  off += align_up((uint32_t)(d / 2) * 8, 128);   // float2 per pair
  L.len_off = off;   off += align_up((uint32_t)batch * 4, 128);
  L.pfx_off = off;   off += align_up((uint32_t)(batch + 1) * 4, 128);
  L.n0_off = off;    off += align_up((uint32_t)batch * 4, 128);
  L.n01_off = off;   off += align_up((uint32_t)batch * 4, 128);
  L.flag_off = off;  off += 128;
  L.tm_off = off;    off += align_up((uint32_t)rk * 8, 128);
  L.rm_off = off;    off += align_up((uint32_t)rk * 4, 128);
  L.recv_off = off;  L.recv_slots = (uint32_t)recv_slots;
  off += align_up((uint32_t)recv_slots * slot_floats(rk, d) * 4, 128);
  L.mbar_off = off;  off += recv_slots > 0 ? 128 : 0;   // the merge barrier
  // cluster partition, a fused draft step: per stage the new tokens the page
  // holds, the new positions, and the new tokens' keys (rotated) and values
  L.pnew_off = off;   off += recv_slots > 0 ? align_up((uint32_t)stages * 4, 128) : 0;
  L.newpos_off = off; off += recv_slots > 0 ? 128 : 0;
  L.newkv_off = off;  off += recv_slots > 0 ? align_up((uint32_t)kMaxFusedNew * 2 * d * es, 128) : 0;

  L.total = off + 1024;  // slack to align the dynamic base to 1024 bytes
  return L;
}

// Checks the alignment and extent of every region of a layout, as the
// kernels use them: the stage ring at the 1024-byte-aligned base, each stage
// a whole number of 1024-byte swizzle atoms (128-byte-swizzled TMA
// destinations); every other region 128-byte aligned (which covers the
// 8-byte mbarriers and uint64 masks and the 16-byte ld.shared.v4 / float4
// accesses), in order, large enough, without overlap, and the zero chunk of
// the flag block 16-byte aligned.  Returns 0, or the number of the first
// check that fails.  Host code runs it for every layout a plan may choose.
__host__ __device__ inline int layout_check(const Layout& L, int variant, int es, int d, int rk,
                                            int stages, int batch, int recv_slots = 0) {
  if ((int)L.recv_slots != recv_slots) return 3;
  if (L.stage_bytes == 0 || L.stage_bytes % 1024 != 0) return 1;
  if ((uint32_t)stages != L.stages) return 2;
  const uint32_t ncw = (uint32_t)kConsumerWarps;
  const uint32_t rm = variant == kVariantMma ? 16u : (uint32_t)rk;
  struct Region { uint32_t off, need; };
  const Region r[] = {
      {0, L.stage_bytes * (uint32_t)stages},
      {L.q_off, (uint32_t)rk * d * 4},
      {L.mo_off, ncw * rm * d * 4},
      {L.ml_off, ncw * rm * 8},
      {L.p_off, variant == kVariantCore ? ncw * 9 * (uint32_t)rk * 4 : 0u},
      {L.info_off, (uint32_t)stages * (uint32_t)sizeof(PageInfo)},
      {L.bar_off, (uint32_t)stages * 16},
      {L.invf_off, (uint32_t)(d / 2) * 8},
      {L.len_off, (uint32_t)batch * 4},
      {L.pfx_off, (uint32_t)(batch + 1) * 4},
      {L.n0_off, (uint32_t)batch * 4},
      {L.n01_off, (uint32_t)batch * 4},
      {L.flag_off, 80},
      {L.tm_off, (uint32_t)rk * 8},
      {L.rm_off, (uint32_t)rk * 4},
      {L.recv_off, L.recv_slots * (uint32_t)slot_floats(rk, d) * 4},
      {L.mbar_off, L.recv_slots ? 8u : 0u},
      {L.pnew_off, L.recv_slots ? (uint32_t)stages * 4 : 0u},
      {L.newpos_off, L.recv_slots ? (uint32_t)kMaxFusedNew * 4 : 0u},
      {L.newkv_off, L.recv_slots ? (uint32_t)(kMaxFusedNew * 2 * d * es) : 0u},
  };
  constexpr int n = sizeof(r) / sizeof(r[0]);
  for (int i = 1; i < n; ++i) {
    if (r[i].off % 128 != 0) return 10 + i;
    if (r[i].off < r[i - 1].off + r[i - 1].need) return 30 + i;
  }
  if ((L.flag_off + 64) % 16 != 0) return 50;
  if (L.total < r[n - 1].off + r[n - 1].need + 1024) return 51;
  if (es * d % kSwizzleRow != 0) return 52;
  return 0;
}

struct Smem {
  uint8_t* stage;       // stages x [K boxes | V boxes]
  float* q;             // [rk][d] rotated, scaled queries of the current piece
  float* mo;            // merge buffer for o (also the cos/sin table during prep)
  float2* ml;           // merge buffer for (m, l)
  float* p;             // CUDA-core engine: per-warp probabilities
  PageInfo* info;
  uint64_t* full;
  uint64_t* empty;
  float2* invf;         // turn frequencies (rope_cos_sin)
  int32_t* len;
  int32_t* pfx;         // [B + 1] pages per head of sequences before b
  int32_t* n0;          // [B] pages per head of range 0
  int32_t* n01;         // [B] pages per head of ranges 0 and 1
  int32_t* flag;        // broadcast of the merge ticket (word 0)
  volatile int32_t* abort;   // word 1 of the flag block: set when a wait gave up
  uint32_t zero16;      // shared address of 16 zero bytes (words 16..19 of the flag block)
  uint64_t* tmask;      // [rk] visible tree keys of each row of the current piece
  float* rmult;         // [rk] logit multiplier of each row of the current piece
  float* recv;          // cluster partition, rank 0: one partial slot per CTA of the cluster
  uint64_t* merge_bar;  // cluster partition, rank 0: every CTA's consumers arrive once filled
  uint32_t* pnew;       // fused step: [stages] bit j = the page holds new token j
  int32_t* newpos;      // fused step: [kMaxFusedNew] positions of the sequence's new tokens
  uint8_t* newkv;       // fused step: [kMaxFusedNew][2][d] rotated keys and values (cache dtype)
};

__device__ inline Smem carve(uint8_t* raw, const Layout& L) {
  uint32_t base = smem_u32(raw);
  uint8_t* p = raw + (align_up(base, 1024) - base);
  Smem s;
  s.stage = p;
  s.q = reinterpret_cast<float*>(p + L.q_off);
  s.mo = reinterpret_cast<float*>(p + L.mo_off);
  s.ml = reinterpret_cast<float2*>(p + L.ml_off);
  s.p = reinterpret_cast<float*>(p + L.p_off);
  s.info = reinterpret_cast<PageInfo*>(p + L.info_off);
  s.full = reinterpret_cast<uint64_t*>(p + L.bar_off);
  s.empty = s.full + L.stages;
  s.invf = reinterpret_cast<float2*>(p + L.invf_off);
  s.len = reinterpret_cast<int32_t*>(p + L.len_off);
  s.pfx = reinterpret_cast<int32_t*>(p + L.pfx_off);
  s.n0 = reinterpret_cast<int32_t*>(p + L.n0_off);
  s.n01 = reinterpret_cast<int32_t*>(p + L.n01_off);
  s.flag = reinterpret_cast<int32_t*>(p + L.flag_off);
  s.abort = s.flag + 1;
  s.zero16 = smem_u32(p + L.flag_off + 64);
  s.tmask = reinterpret_cast<uint64_t*>(p + L.tm_off);
  s.rmult = reinterpret_cast<float*>(p + L.rm_off);
  s.recv = reinterpret_cast<float*>(p + L.recv_off);
  s.merge_bar = reinterpret_cast<uint64_t*>(p + L.mbar_off);
  s.pnew = reinterpret_cast<uint32_t*>(p + L.pnew_off);
  s.newpos = reinterpret_cast<int32_t*>(p + L.newpos_off);
  s.newkv = p + L.newkv_off;
  return s;
}

// Prologue: context lengths and the page prefix over (b, range), computed
// identically by every CTA.  All threads take part.
template <int D, int ES, int NCW>
__device__ inline void prologue(const DecodeArgs& a, Smem& s, const Layout& L) {
  const int tid = threadIdx.x;
  grid_dep_launch_dependents();
  for (int i = tid; i < D / 2; i += blockDim.x) s.invf[i] = a.turn_freq[i];
  if (tid < 4) s.flag[16 + tid] = 0;
  if (tid == 0) *s.abort = 0;
  if (tid == 0) {
    for (uint32_t i = 0; i < L.stages; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], NCW);
    }
    fence_barrier_init();
  }
  // global memory from here on (the caches only after the producer's wait
  // when the inputs are known to be ready)
  if (!a.inputs_ready && !a.tables_ready) grid_dep_wait();
  for (int b = tid; b < a.B; b += blockDim.x)
    s.len[b] = clamp_ctx(__ldg(a.ctx_lens + b), a.max_pages, a.status);
  // Small query tensors are pulled into L2 now, while the lengths load: the
  // query preparation that follows then waits on L2, not on HBM.
  {
    const int64_t qbytes = (int64_t)a.B * a.n_q * a.H_q * D * ES;
    const int64_t pbytes = (int64_t)a.B * a.n_q * 4;
    if (qbytes <= (64 << 10))
      for (int64_t off = (int64_t)tid * 128; off < qbytes; off += (int64_t)blockDim.x * 128)
        prefetch_l2(static_cast<const char*>(a.q) + off);
    if (pbytes <= (16 << 10))
      for (int64_t off = (int64_t)tid * 128; off < pbytes; off += (int64_t)blockDim.x * 128)
        prefetch_l2(reinterpret_cast<const char*>(a.q_pos) + off);
  }
  __syncthreads();
  if (tid < 32) {
    const int lane = tid;
    int32_t carry = 0;
    for (int base = 0; base < a.B; base += 32) {
      const int b = base + lane;
      int32_t v = 0;
      if (b < a.B) {
        const Ranges r = mode_ranges(a.mode, s.len[b], a.W, a.n_sink);
        const int32_t n0 = range_pages(r.k0[0], r.k1[0]);
        const int32_t n01 = n0 + range_pages(r.k0[1], r.k1[1]);
        v = n01 + range_pages(r.k0[2], r.k1[2]);
        s.n0[b] = n0;
        s.n01[b] = n01;
      }

      int32_t inc = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int32_t t = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += t;
      }
      if (b < a.B) s.pfx[b] = carry + inc - v;
      carry += __shfl_sync(0xffffffffu, inc, 31);
    }
    if (lane == 0) s.pfx[a.B] = carry;
  }
  __syncthreads();
}

// Flat position -> (sequence b, head h, page k of the head's line, range r,
// page kr inside that range).
struct Where {
  int b, h, k, r, kr;
};
__device__ __forceinline__ Where locate(const Smem& s, int B, int H, int64_t x) {
  int lo = 0, hi = B - 1;  // largest b with pfx[b] * H <= x
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((int64_t)s.pfx[mid] * H <= x) lo = mid; else hi = mid - 1;
  }
  Where w;
  w.b = lo;
  const int64_t rel = x - (int64_t)s.pfx[lo] * H;
  const int32_t nb = s.pfx[lo + 1] - s.pfx[lo];
  w.h = (int)(rel / nb);
  w.k = (int)(rel - (int64_t)w.h * nb);
  const int32_t n0 = s.n0[lo], n01 = s.n01[lo];
  w.r = w.k < n0 ? 0 : (w.k < n01 ? 1 : 2);
  w.kr = w.k - (w.r == 0 ? 0 : (w.r == 1 ? n0 : n01));
  return w;
}

// Per-page fields the producer derives for flat position x.
struct PageFields {
  int32_t seq, lohi, flags, phys, far, h, toff, kphys;
  uint32_t newmask;   // fused step: the new tokens among the page's read keys
};

// Fields of page P (of range r of sequence b's KV head h), the page being
// the first or last of its piece as given.
__device__ __forceinline__ PageFields page_fields(const DecodeArgs& a, const Smem& s, int b, int h,
                                                  int32_t Lb, const Ranges& rg, int r, int kr,
                                                  bool first, bool last) {
  const bool fold = a.mode == DA_MODE_FOLD;
  const int32_t k0 = rg.lo(r), k1 = rg.hi(r);
  const int32_t P = k0 / kPage + kr;
  const int32_t pk0 = P * kPage;
  const int32_t lo = max(k0, pk0) - pk0, hi = min(k1, pk0 + kPage) - pk0;
  PageFields f;
  f.newmask = 0;
  f.h = h;
  f.seq = piece_seq(a.mode, b, h, a.H_kv, r);
  f.lohi = lo | (hi << 16);
  f.phys = phys_page(a.block_table, b, P, a.max_pages, a.num_pages, a.status);
  f.flags = (first ? kFirst : 0) | (last ? kLast : 0) | (f.phys >= 0 ? kValid : 0);
  f.far = (fold && r == 0) ? 1 : 0;
  f.kphys = (a.k_ring > 0 && !f.far) ? b * a.k_ring + ring_slot(P, a.k_ring, a.k_ring_sp) : f.phys;
  f.toff = kNoTree;
  if (a.tree_mask && a.n_tree > 0 && !f.far) {
    const int32_t t0 = Lb - a.n_tree;   // position of tree token 0
    if (pk0 + kPage > t0) f.toff = pk0 - t0;
  }
  return f;
}

// The producer warp: block-table translation and TMA issue for the CTA's
// stretch [xs, xe) of the page line.  ES = element bytes, NCB = 128-byte
// column boxes per row (head_dim * ES / 128).  F8: far keys come from an FP8
// side cache, one box of 64 rows x head_dim bytes per page, into the stage's
// first K box.  fields(x) gives the page fields of position x.
template <int ES, int NCB, bool F8, class Fields>
__device__ inline void producer_loop(const DecodeArgs& a, Smem& s, const Layout& L, int64_t xs,
                                     int64_t xe, const CUtensorMap* mk, const CUtensorMap* mv,
                                     const CUtensorMap* ms, Fields&& fields) {
  const int lane = threadIdx.x & 31;
  const uint64_t pol = kv_policy(a.mode);
  if (lane == 0) {
    prefetch_tmap(mk);
    prefetch_tmap(mv);
    if (a.mode == DA_MODE_FOLD) prefetch_tmap(ms);
  }
  uint32_t n = 0;        // pages armed so far (loads issued, or a plain arrive)
  bool stopped = false;
  for (int64_t base = xs; base < xe; base += 32) {
    const int64_t x = base + lane;
    int32_t seq = 0, lohi = 0, flags = 0, phys = -1, far = 0, h = 0, toff = kNoTree;
    int32_t kphys = -1;   // page of the K array (the ring slot of a FOLD local page)
    uint32_t newmask = 0;
    if (x < xe) {
      const PageFields f = fields(x);
      seq = f.seq; lohi = f.lohi; flags = f.flags; phys = f.phys; far = f.far; h = f.h;
      toff = f.toff; kphys = f.kphys; newmask = f.newmask;
    }
    const int cnt = (xe - base) < 32 ? (int)(xe - base) : 32;
    for (int j = 0; j < cnt; ++j) {
      const int32_t jseq = __shfl_sync(0xffffffffu, seq, j);
      const int32_t jlohi = __shfl_sync(0xffffffffu, lohi, j);
      const int32_t jflags = __shfl_sync(0xffffffffu, flags, j);
      const int32_t jphys = __shfl_sync(0xffffffffu, phys, j);
      const int32_t jfar = __shfl_sync(0xffffffffu, far, j);
      const int32_t jh = __shfl_sync(0xffffffffu, h, j);
      const int32_t jtoff = __shfl_sync(0xffffffffu, toff, j);
      const int32_t jkphys = __shfl_sync(0xffffffffu, kphys, j);
      const uint32_t jnew = __shfl_sync(0xffffffffu, newmask, j);
      int gave_up = 0;
      if (lane == 0) {
        const uint32_t st = n % L.stages;
        const uint32_t par = (n / L.stages) & 1u;
        if (n == 0 && (a.inputs_ready || a.tables_ready)) {   // the predecessor's writes land first
          grid_dep_wait();
          fence_proxy_async_global();
        }
        if (mbar_wait(&s.empty[st], par ^ 1u, a.status, s.abort)) {
          s.info[st] = PageInfo{jseq, jlohi, jflags, jtoff};
          if (L.recv_slots) s.pnew[st] = jnew;
          uint8_t* kdst = s.stage + st * L.stage_bytes;
          uint8_t* vdst = kdst + NCB * kBoxBytes;
          if (jflags & kValid) {
            const int32_t y = (jphys * a.H_kv + jh) * kPage;
            const int32_t yk = (jkphys * a.H_kv + jh) * kPage;
            if (F8 && jfar) {
              mbar_arrive_expect_tx(&s.full[st], NCB * kBoxBytes + kPage * (NCB * kSwizzleRow / ES));
              tma_load_2d(kdst, ms, 0, yk, &s.full[st], pol);
#pragma unroll
              for (int cb = 0; cb < NCB; ++cb)
                tma_load_2d(vdst + cb * kBoxBytes, mv, cb * (kSwizzleRow / ES), y, &s.full[st], pol);
            } else {
              mbar_arrive_expect_tx(&s.full[st], L.stage_bytes);
              const CUtensorMap* km = jfar ? ms : mk;
#pragma unroll
              for (int cb = 0; cb < NCB; ++cb) {
                tma_load_2d(kdst + cb * kBoxBytes, km, cb * (kSwizzleRow / ES), yk, &s.full[st], pol);
                tma_load_2d(vdst + cb * kBoxBytes, mv, cb * (kSwizzleRow / ES), y, &s.full[st], pol);
              }
            }
          } else {
            mbar_arrive(&s.full[st]);
          }
        } else {
          gave_up = 1;   // a wait gave up: issue nothing more
        }
      }
      if (__shfl_sync(0xffffffffu, gave_up, 0)) {
        stopped = true;
        break;
      }
      ++n;
      __syncwarp();
    }
    if (stopped) break;
  }
  // Every consumer warp arrives here once its page loop is over.  If any wait
  // of the CTA gave up, the copies this warp armed may still be in flight:
  // let them land (bounded) before the CTA, and its shared memory, goes away.
  // Only the last `stages` pages can be outstanding, one per stage.
  named_barrier(kEndBarrier, kConsumerThreads + 32);
  if (lane == 0 && *s.abort) {
    const uint32_t first = n > L.stages ? n - L.stages : 0u;
    for (uint32_t i = first; i < n; ++i) mbar_drain(&s.full[i % L.stages], (i / L.stages) & 1u);
  }
  __syncwarp();   // the warp leaves converged
}

// Flat partition: positions of the page line over every (sequence, KV head, range).
template <int ES, int NCB, bool F8>
__device__ inline void producer(const DecodeArgs& a, Smem& s, const Layout& L, int64_t xs,
                                int64_t xe, const CUtensorMap* mk, const CUtensorMap* mv,
                                const CUtensorMap* ms) {
  const bool fold = a.mode == DA_MODE_FOLD;
  producer_loop<ES, NCB, F8>(a, s, L, xs, xe, mk, mv, ms, [&](int64_t x) {
    const Where w = locate(s, a.B, a.H_kv, x);
    const Ranges rg = mode_ranges(a.mode, s.len[w.b], a.W, a.n_sink);
    const int32_t nb = s.pfx[w.b + 1] - s.pfx[w.b], n0 = s.n0[w.b];
    const bool first = x == xs || w.k == 0 || (fold && w.k == n0);
    const bool last = x == xe - 1 || w.k == nb - 1 || (fold && w.k == n0 - 1);
    return page_fields(a, s, w.b, w.h, s.len[w.b], rg, w.r, w.kr, first, last);
  });
}

// Cluster partition: pages [k_lo, k_hi) of sequence b's KV head h (context
// length Lb), numbered over the head's ranges, without the flat prefix.
template <int ES, int NCB, bool F8>
__device__ inline void producer_head(const DecodeArgs& a, Smem& s, const Layout& L, int b, int h,
                                     int32_t Lb, int64_t k_lo, int64_t k_hi, const CUtensorMap* mk,
                                     const CUtensorMap* mv, const CUtensorMap* ms) {
  const bool fold = a.mode == DA_MODE_FOLD;
  const Ranges rg = mode_ranges(a.mode, Lb, a.W, a.n_sink);
  const int32_t n0 = range_pages(rg.k0[0], rg.k1[0]);
  const int32_t n01 = n0 + range_pages(rg.k0[1], rg.k1[1]);
  const int32_t nb = n01 + range_pages(rg.k0[2], rg.k1[2]);
  producer_loop<ES, NCB, F8>(a, s, L, k_lo, k_hi, mk, mv, ms, [&](int64_t x) {
    const int32_t k = (int32_t)x;
    const int r = k < n0 ? 0 : (k < n01 ? 1 : 2);
    const int kr = k - (r == 0 ? 0 : (r == 1 ? n0 : n01));
    const bool first = x == k_lo || k == 0 || (fold && k == n0);
    const bool last = x == k_hi - 1 || k == nb - 1 || (fold && k == n0 - 1);
    PageFields f = page_fields(a, s, b, h, Lb, rg, r, kr, first, last);
    if (a.n_new > 0 && (f.flags & kValid)) {   // a fused step: new tokens this page reads
      const int32_t pk0 = (rg.lo(r) / kPage + kr) * kPage;
      const int32_t lo = pk0 + (f.lohi & 0xffff), hi = pk0 + (f.lohi >> 16);
      for (int j = 0; j < a.n_new; ++j) {
        const int32_t p = s.newpos[j];
        if (p >= lo && p < hi) f.newmask |= 1u << j;
      }
    }
    return f;
  });
}

// Cluster partition start: barriers (the stage ring, and the merge barrier
// that rank 0's consumers wait on: rank 0 arrives once, expecting the bytes
// the other CTAs' partials bring), the angle table, flags; a CTA barrier; and the
// arrival half of a cluster barrier, whose wait (cluster_wait, before a CTA
// first touches rank 0's shared memory) guarantees that rank 0 initialised
// its merge barrier.  Every thread of the CTA arrives here; only the
// consumers wait (the producer and idle warps exit, which the barrier allows).
template <int D, int NCW>
__device__ inline void cluster_start(const DecodeArgs& a, Smem& s, const Layout& L) {
  const int tid = threadIdx.x;
  grid_dep_launch_dependents();
  for (int i = tid; i < D / 2; i += blockDim.x) s.invf[i] = a.turn_freq[i];
  if (tid < 4) s.flag[16 + tid] = 0;
  if (tid == 0) {
    *s.abort = 0;
    for (uint32_t i = 0; i < L.stages; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], NCW);
    }
    mbar_init(s.merge_bar, 1);   // rank 0's expect-tx arrival; the other CTAs' bytes complete it
    fence_barrier_init();
  }
  __syncthreads();
  cluster_arrive();
}

}  // namespace da
