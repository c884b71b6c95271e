// Shared device helpers of the draft-attention kernels (sm_103a).
//
// Everything here is used by more than one kernel so that the decode kernels,
// the append kernel and the debug-gather hook take the same decisions: the
// mode's key ranges, the block-table translation, the RoPE angle.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "draft_attn.h"

namespace da {

constexpr int kPage = 64;            // tokens per page (the only page size built)
constexpr int kSwizzleRow = 128;     // bytes per row of a 128B-swizzled TMA box
constexpr int kBoxBytes = kPage * kSwizzleRow;  // one 64-row x 128-byte box
constexpr int kMaxBatch = 1024;
constexpr int kMaxFusedNew = 8;      // tokens per sequence one fused draft step may append
// Kernel variants (shared-memory layout): 0 CUDA cores, 1 tensor cores.
// Both run two consumer warpgroups plus one producer warpgroup (only its
// first warp works), launched at 168 registers per thread; the producer group
// gives registers back (setmaxnreg 40) so the consumers can hold 232:
// 128 * 40 + 256 * 232 = 384 * 168.
constexpr int kVariantCore = 0;
constexpr int kVariantMma = 1;
constexpr int kVariantTc = 2;     // the tcgen05 kernel (its own layout, decode_tc.cuh)
constexpr int kConsumerWarps = 8;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kThreads = kConsumerThreads + 128;
constexpr int kProducerRegs = 40;
constexpr int kConsumerRegs = 232;

// ---------------------------------------------------------------------------
// Parameters shared by the split-KV kernels and the combine pass.
// ---------------------------------------------------------------------------
struct DecodeArgs {
  const void* q;
  const int32_t* q_pos;
  const int32_t* ctx_lens;
  const int32_t* block_table;
  const uint64_t* tree_mask;  // [B][n_q] visible tree keys per query, or null (all)
  void* out;
  float* part;          // partial (m, l, o) slots
  uint32_t* cnt;        // per-(b, kv head) count of pages finished; the CTA that
                        // completes the count merges and resets it to zero
  uint32_t* status;
  int32_t B, n_q, H_q, H_kv, G, R;  // R = G * n_q rows per KV head
  int32_t max_pages, num_pages;
  int32_t mode, W, n_sink;
  int32_t n_tree;       // tree tokens at the end of each context
  float alpha, far_mix, beta;
  float far_kscale;     // far keys as stored times this are the keys (FP8 side cache scale, else 1)
  int32_t n_ref;
  float scale_log2;     // softmax scale * log2(e)
  int32_t n_cta;
  int32_t min_pages;    // split floor (pages per active CTA)
  // Nonzero when the previous kernel in the stream is this library's append
  // kernel (draft_attn_step): it waits for its own predecessor before it lets
  // this kernel start, so every input but the caches it writes may be read
  // before griddepcontrol.wait; only the producer's first cache load waits.
  int32_t inputs_ready;
  // Nonzero when the caller promises that ctx_lens, block_table and new_pos
  // were final before the previous kernel started: those are read (and the
  // producer translates its first pages) before griddepcontrol.wait; the
  // consumers still wait before they read queries, masks or new tokens, the
  // producer before its first cache load.
  int32_t tables_ready;
  int32_t k_ring;       // FOLD: rotated K of page P of sequence b at b * k_ring + ring_slot(P)
  int32_t k_ring_sp;    // pages of sinks at the head of each sequence's ring
  int32_t cluster;      // CTAs per cluster of the cluster partition (0: flat partition)
  // Cluster partition, one draft step in one launch: n_new tokens per
  // sequence to append (keys un-rotated, values, positions [B][n_new]) into
  // the caches k_cache_w / v_cache_w before they are attended; 0: none.
  const void* k_new;
  const void* v_new;
  const int32_t* new_pos;
  void* k_cache_w;
  void* v_cache_w;
  int32_t n_new;
  float2 turn_freq[64];  // theta^(-2i/d) / 2pi as hi + lo floats, i < d/2
};

// Partial slot of one piece: m[RK], l[RK], padding to a 16-byte boundary,
// then o[RK][D] (16-byte aligned, so the merge reads it as float4).
__host__ __device__ constexpr int slot_o_off(int rk) { return (2 * rk + 3) / 4 * 4; }
__host__ __device__ constexpr int slot_floats(int rk, int d) { return slot_o_off(rk) + rk * d; }

// ---------------------------------------------------------------------------
// Mode -> key ranges.  Three half-open ranges per sequence (empty ones are
// [x, x)); range 0 of FOLD is the far memory, everything else belongs to the
// main (local) softmax.
//   full / sharp : [0, L)                              "Windowed-MTP", Abstract
//   window       : [0, n_sink) u [L-W, L)  (merged into [0, L) when they touch)
//   fold         : far [s, L-W), local [0, s) u [L-W, L), s = min(n_sink, L-W)
//                  ("FOLD", abstract; the sinks, when given, are exact local
//                  keys, as in window mode)
// Ranges are disjoint; only FOLD with sinks lists them out of position order.
// ---------------------------------------------------------------------------
constexpr int kRanges = 3;
struct Ranges {
  int32_t k0[kRanges], k1[kRanges];
  __host__ __device__ __forceinline__ int32_t lo(int r) const {
    return r == 0 ? k0[0] : (r == 1 ? k0[1] : k0[2]);
  }
  __host__ __device__ __forceinline__ int32_t hi(int r) const {
    return r == 0 ? k1[0] : (r == 1 ? k1[1] : k1[2]);
  }
};

__host__ __device__ __forceinline__ Ranges mode_ranges(int mode, int32_t L, int32_t W,
                                                       int32_t n_sink) {
  Ranges r;
  r.k0[0] = 0; r.k1[0] = 0; r.k0[1] = L; r.k1[1] = L; r.k0[2] = L; r.k1[2] = L;
  if (L <= 0) { r.k0[1] = r.k1[1] = r.k0[2] = r.k1[2] = 0; return r; }
  int32_t ws = L - W > 0 ? L - W : 0;
  switch (mode) {
    case DA_MODE_WINDOW:
      if (n_sink > 0 && ws > n_sink) {
        r.k0[0] = 0; r.k1[0] = n_sink; r.k0[1] = ws; r.k1[1] = L;
      } else if (n_sink > 0) {
        r.k0[0] = 0; r.k1[0] = L;
      } else {
        r.k0[0] = ws; r.k1[0] = L;
      }
      break;
    case DA_MODE_FOLD: {
      const int32_t sk = n_sink < ws ? n_sink : ws;
      r.k0[0] = sk; r.k1[0] = ws; r.k0[1] = 0; r.k1[1] = sk; r.k0[2] = ws; r.k1[2] = L;
      break;
    }
    default:  // full, sharp
      r.k0[0] = 0; r.k1[0] = L;
      break;
  }
  return r;
}

__host__ __device__ __forceinline__ bool range_is_far(int mode, int r) {
  return mode == DA_MODE_FOLD && r == 0;
}

__host__ __device__ __forceinline__ int32_t range_pages(int32_t k0, int32_t k1) {
  return k1 > k0 ? (k1 + kPage - 1) / kPage - k0 / kPage : 0;
}

// FOLD's ring of rotated keys: slot of logical page P in a sequence's R
// pages.  The first sp pages (the sinks' pages) keep their own slots; later
// pages cycle through the other R - sp.
__host__ __device__ __forceinline__ int32_t ring_slot(int32_t P, int32_t R, int32_t sp) {
  return P < sp ? P : sp + (P - sp) % (R - sp);
}

// Shared virtual position of the FOLD far memory (the newest far token).
__host__ __device__ __forceinline__ int32_t fold_far_pos(int32_t L, int32_t W) {
  return L - W - 1;
}

// Number of keys the main softmax of a sequence sees (SharpDraft's |S|).
__host__ __device__ __forceinline__ int32_t visible_keys(int mode, int32_t L, int32_t W,
                                                        int32_t n_sink) {
  Ranges r = mode_ranges(mode, L, W, n_sink);
  int32_t n = 0;
  for (int i = 0; i < kRanges; ++i)
    if (!range_is_far(mode, i) && r.k1[i] > r.k0[i]) n += r.k1[i] - r.k0[i];
  return n;
}

// ---------------------------------------------------------------------------
// RoPE angle, in FP32 only.  Each frequency is kept as f = theta^(-2i/d) / 2pi
// (turns per position) split into two floats hi + lo (formed on the host in
// double: hi = f rounded, lo = f - hi rounded), so that pos * f is the angle in
// turns.  pos * hi is formed without error as the float pair th + te by an FMA
// (Dekker's TwoProduct: te = fma(pos, hi, -th)); the whole turns of th are
// dropped exactly, te and pos * lo are added, and CUDA's sincospif (which
// works in units of pi) takes twice the remaining fraction of a turn.  With
// |pos| < 2^24 (exact in float) the angle is within a few 1e-7 rad at every
// position, where a plain float product pos * inv_freq would be off by
// ~0.06 rad near 1M.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void rope_cos_sin(int32_t pos, float2 f, float& c, float& s) {
  const float p = (float)pos;
  const float th = __fmul_rn(p, f.x);
  const float te = __fmaf_rn(p, f.x, -th);
  const float t = __fadd_rn(th, -rintf(th)) + (te + p * f.y);
  sincospif(2.f * t, &s, &c);
}

// Rotate-half RoPE of one pair: (x cos - y sin, y cos + x sin), each with one
// product rounded and the other fused.  Every kernel that writes a rotated
// key uses this, so that a key appended by any of them is the same bits.
__device__ __forceinline__ void rope_pair(float x, float y, float c, float s, float& xr,
                                          float& yr) {
  xr = __fmaf_rn(x, c, -__fmul_rn(y, s));
  yr = __fmaf_rn(y, c, __fmul_rn(x, s));
}

// ---------------------------------------------------------------------------
// Block-table translation (PagedAttention layout).  Returns -1 and flags the
// status word when the entry is outside [0, num_pages).
// ---------------------------------------------------------------------------
__device__ __forceinline__ int32_t phys_page(const int32_t* bt, int32_t b, int32_t page,
                                             int32_t max_pages, int32_t num_pages,
                                             uint32_t* status) {
  if (page < 0 || page >= max_pages) {
    atomicOr(status, DA_STATUS_BAD_CTX_LEN);
    return -1;
  }
  int32_t p = __ldg(bt + (int64_t)b * max_pages + page);
  if (p < 0 || p >= num_pages) {
    atomicOr(status, DA_STATUS_BAD_PAGE);
    return -1;
  }
  return p;
}

// Context length clamped to what the block table can hold.
__device__ __forceinline__ int32_t clamp_ctx(int32_t L, int32_t max_pages, uint32_t* status) {
  int64_t cap = (int64_t)max_pages * kPage;
  if (L < 0 || (int64_t)L > cap) {
    atomicOr(status, DA_STATUS_BAD_CTX_LEN);
    return L < 0 ? 0 : (int32_t)cap;
  }
  return L;
}

// ---------------------------------------------------------------------------
// Flat work partition.  The pages of every (b, kv head) are laid end to end
// (b outer, then head, then ranges 0, 1, 2 in turn); with TP pages in all and
// n active CTAs, CTA i takes positions [floor(i*TP/n), floor((i+1)*TP/n)).
// n = min(grid, ceil(TP / min_pages)): a small selection (a window)
// goes to fewer, fuller CTAs, so that each (b, head) has few pieces to merge.
// A "piece" is the part of one (b, head, softmax segment) that one CTA covers
// (the ranges of window mode are one segment; FOLD's far range is one segment
// and its local ranges the other).  Its seq = (b * H_kv + head) * 2 + segment never decreases along
// the line, so slot = cta + seq is unique: every new piece advances the CTA,
// the seq, or both.
// ---------------------------------------------------------------------------
constexpr int kMaxAutoStages = 4;       // pipeline depth chosen when da_params.stages = 0
constexpr int kMaxAutoStagesCore = 6;   // the same for the CUDA-core engines (two warp
                                        // groups hold two steps, the producer fills more)
constexpr int kMinPagesPerCta = 1;   // default split floor (da_params.min_pages_per_cta = 0)

__host__ __device__ __forceinline__ int64_t cta_begin(int64_t i, int64_t TP, int64_t n) {
  return (i * TP) / n;
}
// The CTA whose (non-empty) range holds flat position x.
__host__ __device__ __forceinline__ int64_t cta_of(int64_t x, int64_t TP, int64_t n) {
  return ((x + 1) * n - 1) / TP;
}
__host__ __device__ __forceinline__ int64_t active_ctas(int64_t TP, int64_t grid,
                                                       int64_t min_pages) {
  const int64_t want = (TP + min_pages - 1) / min_pages;
  return want < 1 ? 1 : (want < grid ? want : grid);
}
// Piece id of (b, head, range); FOLD keeps its far range apart from the rest.
__host__ __device__ __forceinline__ int32_t piece_seq(int mode, int b, int h, int H, int range) {
  return (b * H + h) * 2 + (mode == DA_MODE_FOLD && range != 0 ? 1 : 0);
}
__host__ __device__ __forceinline__ bool seq_is_far(int mode, int32_t seq) {
  return mode == DA_MODE_FOLD && (seq & 1) == 0;
}

// ---------------------------------------------------------------------------
// PTX wrappers: mbarrier, TMA, register reallocation, misc.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait: gives up after ~2^31 SM cycles (about a second), sets the
// timeout status bit and the CTA's abort flag (a shared-memory word every
// waiting thread of the CTA polls) and returns false; a thread that sees the
// flag set by another gives up at once.  Never expected to trigger.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t* status,
                                          volatile int32_t* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (clock64() - t0 > (1ll << 31)) {
      atomicOr(status, DA_STATUS_WAIT_TIMEOUT);
      *abort = 1;
      return false;
    }
  }
}

// Bounded wait that ignores the abort flag (used to let copies already in
// flight land before a CTA that gave up exits); false after ~2^28 cycles.
__device__ __forceinline__ bool mbar_drain(uint64_t* bar, uint32_t parity) {
  long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > (1ll << 28)) return false;
  return true;
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// 2-D tiled TMA load of one 64-row x 128-byte box into shared memory,
// completing on `bar` (transaction bytes).  x is the element column (a
// multiple of 128 bytes here), y the row.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int32_t x,
                                            int32_t y, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// L2 policy for data read once (the KV stream of full, FOLD and SharpDraft
// attention): evict first.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// L2 policy for a window's keys, which the next draft step reads again (all
// but one token): normal eviction.
__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// The policy for the KV loads of `mode`.
__device__ __forceinline__ uint64_t kv_policy(int mode) {
  return mode == DA_MODE_WINDOW ? policy_evict_normal() : policy_evict_first();
}

template <int N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// Programmatic dependent launch.  Kernels are launched with programmatic
// stream serialisation: the next kernel in the stream may start while this one
// runs, but every kernel waits (grid_dep_wait) for its predecessor to finish
// and flush its writes before it reads or writes any global memory.
__device__ __forceinline__ void grid_dep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_dep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" :::);
}
// Orders global writes made visible to this thread (by the previous grid)
// before the TMA loads it issues next.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;"
               : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void named_barrier(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}
__device__ __forceinline__ void named_barrier_arrive(int id, int threads) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Thread-block clusters: rank of this CTA in its cluster, the cluster's size,
// the shared-memory address of the same location in CTA `rank`'s shared
// memory (distributed shared memory), loads from such addresses, and the
// cluster-wide barrier (release/acquire: shared-memory writes before it are
// visible to every CTA of the cluster after it).
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t dsmem_addr(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
__device__ __forceinline__ float dsmem_ld_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ float4 dsmem_ld_f32x4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr) : "memory");
  return v;
}
// Generic address of the same shared-memory location in CTA `rank` of the
// cluster (generic loads and stores reach it).
template <typename T>
__device__ __forceinline__ T* dsmem_ptr(T* local, uint32_t rank) {
  uint64_t r;
  asm volatile("mapa.u64 %0, %1, %2;" : "=l"(r) : "l"(reinterpret_cast<uint64_t>(local)), "r"(rank));
  return reinterpret_cast<T*>(r);
}
// Asynchronous stores into (possibly another cluster CTA's) shared memory at
// shared::cluster address `addr`; each completes `bar` (a shared::cluster
// mbarrier address in the same CTA as `addr`) with its byte count, which
// makes the data visible to a thread that sees the barrier's phase complete.
__device__ __forceinline__ void st_async_f32x4(uint32_t addr, float4 v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1,%2,%3,%4}, [%5];"
               ::"r"(addr), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(bar) : "memory");
}
__device__ __forceinline__ void st_async_f32(uint32_t addr, float v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];"
               ::"r"(addr), "f"(v), "r"(bar) : "memory");
}
// Arrive on the mbarrier at `local`'s place in CTA `rank`, releasing this
// thread's earlier writes (its distributed-shared-memory stores included) to
// the cluster.
__device__ __forceinline__ void mbar_arrive_remote(uint64_t* local, uint32_t rank) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];"
               ::"r"(dsmem_addr(smem_u32(local), rank)) : "memory");
}
// Bounded wait (as mbar_wait) that acquires at cluster scope: writes other
// CTAs released before their arrivals are visible after it.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, uint32_t* status,
                                                  volatile int32_t* abort) {
  long long t0 = 0;
  bool started = false;
  while (true) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    if (ok) return true;
    if (!started) {
      t0 = clock64();
      started = true;
    }
    if (*abort) return false;
    if (clock64() - t0 > (1ll << 31)) {
      atomicOr(status, DA_STATUS_WAIT_TIMEOUT);
      *abort = 1;
      return false;
    }
  }
}
// The two halves of the cluster barrier: every thread arrives once (release)
// and, before it depends on the other CTAs, waits once (acquire).
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}

// Address of element (row, byte offset) inside a stage buffer laid out as
// consecutive 64-row x 128-byte boxes with the 128-byte TMA swizzle: the
// 16-byte chunk index inside a row is XOR-ed with the row index mod 8.
__device__ __forceinline__ uint32_t swz_addr(uint32_t base, int row, int byte) {
  int box = byte >> 7;
  int chunk = (byte >> 4) & 7;
  return base + box * kBoxBytes + row * kSwizzleRow + ((chunk ^ (row & 7)) << 4) + (byte & 15);
}

// swz_addr of byte 32 ks + b0 (b0 < 32) of a row, from the address a0 of byte
// b0: inside a row, 16-byte chunk 2 ks' + (b0 / 16) sits at that chunk XOR the
// row's swizzle, i.e. a0's chunk XOR 2 ks', with ks' = ks mod 4 (bits 5-6 of
// the address, all zero in the 1024-byte-aligned stage base and row offset);
// every 4 steps move to the next 128-byte column box.
__device__ __forceinline__ uint32_t swz_step(uint32_t a0, int ks) {
  return (a0 ^ ((uint32_t)(ks & 3) << 5)) + (uint32_t)(ks >> 2) * kBoxBytes;
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

}  // namespace da
