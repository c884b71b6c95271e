// Split-KV decode on the 5th-generation tensor cores (tcgen05, sm_103a) for
// draft trees: up to 32 query rows per KV head (an 8-token tree over a GQA
// group of 4, or a 16-token block over 2), head_dim 128, bf16 caches.
//
// One step is two consecutive pages of a piece (128 keys), staged by TMA in
// one pipeline stage laid out as [K d0-63 | K d64-127 | V d0-63 | V d64-127],
// each part [page A rows 0-63 | page B rows 0-63] with the 128-byte swizzle,
// so that 128 keys are one M = 128 operand with 1024-byte row groups.
//
//  * QK^T as S^T = K Q^T: M = 128 keys, N = 32 query rows, K = 128 (eight
//    K = 16 MMAs).  A = the staged keys (K-major), B = the piece's rotated and
//    scaled queries (bf16, K-major, written by query preparation).  S^T
//    accumulates in TMEM: lane = key, column = query row.
//  * Softmax: thread t of a warp group owns key t of the step and reads its
//    32 scores with one tcgen05.ld.  The group keeps one reference maximum
//    per row, raised lazily (only when a visible score exceeds it by more
//    than 2^8: a barrier-wide vote, then an exact row maximum over the keys);
//    exponentials are taken against it, each thread sums its own key's
//    probabilities per row, and the sums are reduced once per piece.
//  * PV as O^T = V^T P^T: M = 128 dimensions, N = 32 rows, K = 128 keys.
//    A = the staged values read as dimension-major (MN-major), B = P^T
//    written by the softmax threads (one 64-byte row per key, MN-major with
//    the 64-byte swizzle).  O^T accumulates in TMEM: lane = dimension.
//    A raise rescales O^T in TMEM (tcgen05.ld / .st) before the next PV.
//
// Warps 0-3 and 4-7 are two softmax groups that take alternate steps, each
// with its own S^T and O^T in TMEM and its own P^T buffer; warp 8 issues the
// TMA loads, warp 9 (one elected thread) the MMAs; they meet on mbarriers:
//   full/empty (stage loaded / stage free: the PV's commit and a read of the
//   step's page information by each consumer warp), s_full (S^T ready),
//   s_free (S^T read), p_full (P^T written, invalid keys' values zeroed),
//   o_done (a PV finished), q_full (the piece's queries written).
// Keys outside a page's valid range may hold anything (NaN included): their
// scores are masked and their value rows zeroed in shared memory before the
// PV reads them.
#pragma once

#include "decode.cuh"

namespace da {

// ---------------------------------------------------------------------------
// tcgen05 wrappers.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {   // whole warp
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
               ::"r"(smem_u32(slot)), "r"(ncols) : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {   // whole warp
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// D (TMEM) = A B (+ D when acc), kind::f16 (bf16 operands, f32 accumulation).
__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}
// Arrives on `bar` once every tcgen05 operation this thread issued before has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Generic-proxy shared-memory writes of this thread, ordered before later
// async-proxy (tensor core) reads.
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// 32 lanes x 32 columns of 32 bits: thread i gets lane (lane base + i),
// columns col .. col + 31.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// 32 lanes x 16 columns (thread i: lane base + i, columns col .. col + 15).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};"
      ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
        "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]),
        "r"(r[14]), "r"(r[15])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// Scales 32 columns of TMEM (this warp's lanes) by the per-column factors f,
// 16 columns at a time.
__device__ __forceinline__ void tmem_scale32(uint32_t taddr, const float* f) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t v[16];
    tmem_ld16(taddr + 16u * h, v);
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * f[16 * h + i]);
    tmem_st16(taddr + 16u * h, v);
  }
}
// Float maximum over a warp's lanes by the integer reduction (the bits of a
// float map to an integer of the same order: negative values flipped).
__device__ __forceinline__ float warp_max(float x) {
  const int b = __float_as_int(x);
  const int key = b >= 0 ? b : b ^ 0x7fffffff;
  const int m = __reduce_max_sync(0xffffffffu, key);
  return __int_as_float(m >= 0 ? m : m ^ 0x7fffffff);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
      ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
        "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]),
        "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]),
        "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
        "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor: start address, leading and stride byte
// offsets (the canonical layouts' LBO / SBO), version 1, swizzle mode
// (0 none, 2 128-byte, 4 64-byte).
__device__ __forceinline__ uint64_t tc_desc(uint32_t addr, uint32_t lbo, uint32_t sbo,
                                            uint32_t swizzle) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | ((uint64_t)swizzle << 61);
}
// Instruction descriptor, kind::f16: f32 accumulator, bf16 A and B, each
// K-major (0) or MN-major (1), M x N.
__host__ __device__ constexpr uint32_t tc_idesc(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// OR of `pred` over the `threads` threads of named barrier `id` (all wait).
__device__ __forceinline__ bool barrier_or(int id, int threads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r) : "r"((uint32_t)pred), "r"(id), "r"(threads) : "memory");
  return r != 0;
}

// ---------------------------------------------------------------------------
// Shared-memory layout of the tcgen05 kernel.
// ---------------------------------------------------------------------------
constexpr int kTcRows = 32;            // query rows the kernel computes (N of both MMAs)
constexpr int kTcStageBytes = 65536;   // two pages of K and V, head_dim 128, bf16
constexpr int kTcMaxStages = 3;
constexpr uint32_t kTcCols = 128;      // TMEM: S^T A | S^T B | O^T A | O^T B
constexpr int kPair = 8;               // PageInfo flag: the step holds two pages
constexpr int kTcEndBarrier = 5;       // the MMA warp waits for the consumers before freeing TMEM
// Register split of this kernel (launched at 168 per thread): the producer
// warpgroup (TMA and MMA issue) keeps 56, the softmax warpgroups take 224
// (their scores, probabilities and row-sum shares): 128 * 56 + 256 * 224 =
// 64512 = 384 * 168.
constexpr int kTcProducerRegs = 56;
constexpr int kTcConsumerRegs = 224;
static_assert(128 * kTcProducerRegs + 256 * kTcConsumerRegs <= 384 * 168, "register split");

struct TcLayout {
  uint32_t stages, qb_off, pt_off, info_off, bar_off, invf_off, len_off, pfx_off, n0_off,
      n01_off, flag_off, tm_off, rm_off, red_off, mm_off, total;
};

__host__ __device__ inline TcLayout make_tc_layout(int stages, int batch) {
  TcLayout L;
  L.stages = stages;
  uint32_t off = (uint32_t)stages * kTcStageBytes;
  L.qb_off = off;   off += kTcRows * 256;                     // Q tile, bf16, 2 boxes
  L.pt_off = off;   off += 2 * 128 * kTcRows * 2;             // P^T of each group (16 KB);
                                                              // also query-prep scratch and
                                                              // the piece-end merge buffer
  L.info_off = off; off += align_up((uint32_t)stages * 2 * sizeof(PageInfo), 128);
  L.bar_off = off;  off += 512;                               // 16 mbarriers, the TMEM
                                                              // address slot
  L.invf_off = off; off += align_up(64 * 8, 128);
  L.len_off = off;  off += align_up((uint32_t)batch * 4, 128);
  L.pfx_off = off;  off += align_up((uint32_t)(batch + 1) * 4, 128);
  L.n0_off = off;   off += align_up((uint32_t)batch * 4, 128);
  L.n01_off = off;  off += align_up((uint32_t)batch * 4, 128);
  L.flag_off = off; off += 128;
  L.tm_off = off;   off += align_up(kTcRows * 8, 128);
  L.rm_off = off;   off += align_up(kTcRows * 4, 128);
  L.red_off = off;  off += 2 * 4 * kTcRows * 4;               // per group and warp, per row
  L.mm_off = off;   off += 4 * kTcRows * 4;                   // reference maxima and rescale
                                                              // factors of each group
  L.total = off + 1024;
  return L;
}

__host__ __device__ inline int tc_layout_check(const TcLayout& L, int stages, int batch) {
  if ((int)L.stages != stages) return 1;
  if (L.qb_off % 1024 || L.pt_off % 1024) return 2;         // swizzle atoms
  if (L.info_off % 128 || L.bar_off % 128 || L.invf_off % 128 || L.len_off % 128 ||
      L.pfx_off % 128 || L.n0_off % 128 || L.n01_off % 128 || L.flag_off % 128 ||
      L.tm_off % 128 || L.rm_off % 128 || L.red_off % 128 || L.mm_off % 128)
    return 3;
  if (L.pt_off < L.qb_off + kTcRows * 256 || L.info_off < L.pt_off + 16384) return 4;
  // barriers: full and empty per stage (kTcMaxStages each), eight per group
  // pair, q_full, drain; the TMEM slot after them, all before invf
  if (stages > kTcMaxStages) return 7;
  if (L.invf_off < L.bar_off + (2 * kTcMaxStages + 10) * 8 + 4) return 8;
  if (L.mm_off < L.red_off + 2 * 4 * kTcRows * 4) return 5;
  if (L.total < L.mm_off + 4 * kTcRows * 4 + 1024) return 5;
  if (batch < 1) return 6;
  return 0;
}

struct TcSmem {
  uint8_t* stage;
  uint8_t* qb;
  uint8_t* pt;
  PageInfo* info;
  uint64_t* full;    // [stages]
  uint64_t* empty;   // [stages]
  uint64_t* s_full;  // [2]
  uint64_t* s_free;  // [2]
  uint64_t* p_full;  // [2]
  uint64_t* o_done;  // [2]
  uint64_t* q_full;  // [1]
  uint64_t* drain;   // [1]
  uint32_t* tslot;
  float* red;        // [2][4][32]
  float* mref;       // [2][32] reference maxima of each group
  float* alpha;      // [2][32] rescale factors of a raise
};

// The Smem view the shared routines (prologue, producer helpers, query
// preparation, merges) use, pointed at this kernel's regions.
__device__ inline Smem tc_carve(uint8_t* raw, const TcLayout& L, TcSmem& t) {
  uint32_t base = smem_u32(raw);
  uint8_t* p = raw + (align_up(base, 1024) - base);
  t.stage = p;
  t.qb = p + L.qb_off;
  t.pt = p + L.pt_off;
  t.info = reinterpret_cast<PageInfo*>(p + L.info_off);
  uint64_t* b = reinterpret_cast<uint64_t*>(p + L.bar_off);
  t.full = b;
  t.empty = b + kTcMaxStages;
  t.s_full = b + 2 * kTcMaxStages;
  t.s_free = t.s_full + 2;
  t.p_full = t.s_free + 2;
  t.o_done = t.p_full + 2;
  t.q_full = t.o_done + 2;
  t.drain = t.q_full + 1;
  t.tslot = reinterpret_cast<uint32_t*>(t.drain + 1);
  t.red = reinterpret_cast<float*>(p + L.red_off);
  t.mref = reinterpret_cast<float*>(p + L.mm_off);
  t.alpha = t.mref + 2 * kTcRows;
  Smem s;
  s.stage = p;
  s.q = nullptr;
  s.mo = reinterpret_cast<float*>(t.pt);   // cos/sin scratch of query preparation
  s.ml = nullptr;
  s.p = nullptr;
  s.info = t.info;
  s.full = t.full;
  s.empty = t.empty;
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
  return s;
}

// ---------------------------------------------------------------------------
// Producer: the CTA's stretch [xs, xe) as steps of two pages (one when a page
// ends its piece), each step into one stage.
// ---------------------------------------------------------------------------
__device__ inline void tc_producer(const DecodeArgs& a, Smem& s, const TcSmem& t, uint32_t stages,
                                   int64_t xs, int64_t xe, const CUtensorMap* mk,
                                   const CUtensorMap* mv, const CUtensorMap* ms) {
  const int lane = threadIdx.x & 31;
  const uint64_t pol = kv_policy(a.mode);
  if (lane == 0) {
    prefetch_tmap(mk);
    prefetch_tmap(mv);
    if (a.mode == DA_MODE_FOLD) prefetch_tmap(ms);
  }
  const bool fold = a.mode == DA_MODE_FOLD;
  uint32_t n = 0;          // steps armed
  int half = 0;            // pages placed in the current step
  PageInfo first_info{0, 0, 0, kNoTree};
  bool stopped = false;
  bool waited_inputs = false;
  for (int64_t base = xs; base < xe && !stopped; base += 32) {
    const int64_t x = base + lane;
    int32_t seq = 0, lohi = 0, flags = 0, phys = -1, far = 0, h = 0, toff = kNoTree, kphys = -1;
    if (x < xe) {
      const Where w = locate(s, a.B, a.H_kv, x);
      const Ranges rg = mode_ranges(a.mode, s.len[w.b], a.W, a.n_sink);
      const int32_t k0 = rg.lo(w.r), k1 = rg.hi(w.r);
      const int32_t P = k0 / kPage + w.kr;
      const int32_t pk0 = P * kPage;
      const int32_t lo = max(k0, pk0) - pk0, hi = min(k1, pk0 + kPage) - pk0;
      const int32_t nb = s.pfx[w.b + 1] - s.pfx[w.b], n0 = s.n0[w.b];
      h = w.h;
      seq = piece_seq(a.mode, w.b, w.h, a.H_kv, w.r);
      lohi = lo | (hi << 16);
      phys = phys_page(a.block_table, w.b, P, a.max_pages, a.num_pages, a.status);
      const bool first = x == xs || w.k == 0 || (fold && w.k == n0);
      const bool last = x == xe - 1 || w.k == nb - 1 || (fold && w.k == n0 - 1);
      flags = (first ? kFirst : 0) | (last ? kLast : 0) | (phys >= 0 ? kValid : 0);
      far = (fold && w.r == 0) ? 1 : 0;
      kphys = (a.k_ring > 0 && !far) ? w.b * a.k_ring + ring_slot(P, a.k_ring, a.k_ring_sp) : phys;
      if (a.tree_mask && a.n_tree > 0 && !far) {
        const int32_t t0 = s.len[w.b] - a.n_tree;
        if (pk0 + kPage > t0) toff = pk0 - t0;
      }
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
      int gave_up = 0;
      if (lane == 0) {
        const uint32_t st = n % stages;
        if (!waited_inputs && a.inputs_ready) {   // the append kernel's writes land first
          grid_dep_wait();
          fence_proxy_async_global();
          waited_inputs = true;
        }
        bool ok = true;
        if (half == 0) ok = mbar_wait(&t.empty[st], ((n / stages) & 1u) ^ 1u, a.status, s.abort);
        if (ok) {
          uint8_t* sb = t.stage + (size_t)st * kTcStageBytes;
          if (jflags & kValid) {
            const int32_t y = (jphys * a.H_kv + jh) * kPage;
            const int32_t yk = (jkphys * a.H_kv + jh) * kPage;
            const CUtensorMap* km = jfar ? ms : mk;
            mbar_expect_tx(&t.full[st], 4 * kBoxBytes);
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) {
              tma_load_2d(sb + cb * 2 * kBoxBytes + half * kBoxBytes, km, cb * 64, yk, &t.full[st], pol);
              tma_load_2d(sb + 4 * kBoxBytes + cb * 2 * kBoxBytes + half * kBoxBytes, mv, cb * 64, y,
                          &t.full[st], pol);
            }
          }
          const PageInfo pi{jseq, jlohi, jflags, jtoff};
          if (half == 0 && !(jflags & kLast)) {
            first_info = pi;
            half = 1;
          } else {
            PageInfo i0 = half == 0 ? pi : first_info;
            PageInfo i1 = half == 0 ? PageInfo{jseq, 0, 0, kNoTree} : pi;
            if (half == 1) i0.flags |= kPair;
            t.info[2 * st] = i0;
            t.info[2 * st + 1] = i1;
            mbar_arrive(&t.full[st]);
            ++n;
            half = 0;
          }
        } else {
          gave_up = 1;
        }
      }
      if (__shfl_sync(0xffffffffu, gave_up, 0)) {
        stopped = true;
        break;
      }
      __syncwarp();
    }
  }
  n = __shfl_sync(0xffffffffu, n, 0);
  named_barrier(kEndBarrier, kConsumerThreads + 32);
  if (lane == 0 && *s.abort) {
    const uint32_t first = n > stages ? n - stages : 0u;
    for (uint32_t i = first; i < n; ++i) mbar_drain(&t.full[i % stages], (i / stages) & 1u);
  }
  __syncwarp();
}

// ---------------------------------------------------------------------------
// MMA issue (one thread).
// ---------------------------------------------------------------------------
struct TcTmem {
  uint32_t base;
  __device__ __forceinline__ uint32_t s(int g) const { return base + 32u * g; }
  __device__ __forceinline__ uint32_t o(int g) const { return base + 64u + 32u * g; }
};

__device__ __forceinline__ void tc_issue_qk(const TcSmem& t, const TcTmem& tm, uint32_t st, int g) {
  constexpr uint32_t id = tc_idesc(128, kTcRows, 0, 0);
  const uint32_t kb = smem_u32(t.stage) + st * kTcStageBytes;
  const uint32_t qb = smem_u32(t.qb);
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const uint64_t ad = tc_desc(kb + (ks >> 2) * 2 * kBoxBytes + (ks & 3) * 32, 16, 1024, 2);
    const uint64_t bd = tc_desc(qb + (ks >> 2) * (kTcRows * 128) + (ks & 3) * 32, 16, 1024, 2);
    tc_mma(tm.s(g), ad, bd, id, ks > 0);
  }
}

__device__ __forceinline__ void tc_issue_pv(const TcSmem& t, const TcTmem& tm, uint32_t st, int g,
                                            bool acc) {
  constexpr uint32_t id = tc_idesc(128, kTcRows, 1, 1);
  const uint32_t vb = smem_u32(t.stage) + st * kTcStageBytes + 4 * kBoxBytes;
  const uint32_t pb = smem_u32(t.pt) + g * (128 * kTcRows * 2);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint64_t ad = tc_desc(vb + kk * 2048, 2 * kBoxBytes, 1024, 2);
    const uint64_t bd = tc_desc(pb + kk * 1024, 8192, 512, 4);
    tc_mma(tm.o(g), ad, bd, id, (acc || kk > 0) ? 1u : 0u);
  }
}

// PV of group g's step in stage st, once its P^T is
// written (the group's c-th step); the commits release the stage and tell
// the group its P^T buffer is free.
__device__ __forceinline__ bool tc_pv_when_ready(const DecodeArgs& a, Smem& s, const TcSmem& t,
                                                 const TcTmem& tm, uint32_t st, int g, uint32_t c,
                                                 bool acc) {
  if (!mbar_wait(&t.p_full[g], c & 1u, a.status, s.abort)) return false;
  tc_fence_after();
  tc_issue_pv(t, tm, st, g, acc);
  tc_commit(&t.o_done[g]);
  tc_commit(&t.empty[st]);
  return true;
}

__device__ __forceinline__ void tc_mma_thread(const DecodeArgs& a, Smem& s, const TcSmem& t,
                                           const TcTmem& tm, uint32_t stages, int64_t xs,
                                           int64_t xe) {
  uint32_t u = 0, ng0 = 0, ng1 = 0, piece = 0;
  bool fresh0 = true, fresh1 = true;
  // the previous step's PV, issued after the next step's QK^T (its P^T is
  // being written meanwhile); bit 31 set = none pending
  uint32_t pend = 1u << 31;
  for (int64_t x = xs; x < xe;) {
    const uint32_t st = u % stages;
    if (!mbar_wait(&t.full[st], (u / stages) & 1u, a.status, s.abort)) break;
    const PageInfo ia = t.info[2 * st], ib = t.info[2 * st + 1];
    const int np = (ia.flags & kPair) ? 2 : 1;
    const bool last = (((np == 2) ? ib.flags : ia.flags) & kLast) != 0;
    if (ia.flags & kFirst) {
      if (!mbar_wait(t.q_full, piece & 1u, a.status, s.abort)) break;
      ++piece;
      fresh0 = fresh1 = true;
    }
    const int g = (int)(u & 1u);
    const uint32_t c = g ? ng1 : ng0;
    if (c > 0 && !mbar_wait(&t.s_free[g], (c - 1) & 1u, a.status, s.abort)) break;
    tc_fence_after();
    tc_issue_qk(t, tm, st, g);
    tc_commit(&t.s_full[g]);
    if (!(pend >> 31)) {
      // pend: stage (bits 0-7), group (8), count (9-29), accumulate (30)
      if (!tc_pv_when_ready(a, s, t, tm, pend & 0xffu, (int)((pend >> 8) & 1u),
                            (pend >> 9) & 0x1fffffu, ((pend >> 30) & 1u) != 0))
        break;
      pend = 1u << 31;
    }
    const bool acc = g ? !fresh1 : !fresh0;
    if (g) { fresh1 = false; ng1 = c + 1; } else { fresh0 = false; ng0 = c + 1; }
    if (last) {
      if (!tc_pv_when_ready(a, s, t, tm, st, g, c, acc)) break;
    } else {
      pend = st | ((uint32_t)g << 8) | ((c & 0x1fffffu) << 9) | ((uint32_t)acc << 30);
    }
    x += np;
    ++u;
  }
  // every MMA issued has completed before TMEM is released
  tc_commit(t.drain);
  mbar_drain(t.drain, 0);
}

// ---------------------------------------------------------------------------
// The kernel.
// ---------------------------------------------------------------------------
template <bool CLUSTER>
__global__ void __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ DecodeArgs a, const __grid_constant__ CUtensorMap mk,
                     const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap ms,
                     int stages_arg) {
  using T = __nv_bfloat16;
  constexpr int D = 128, RK = kTcRows, NCT = kConsumerThreads;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t stages = (uint32_t)stages_arg;
  const TcLayout L = make_tc_layout(stages_arg, a.B);
  TcSmem t;
  Smem s = tc_carve(smem_raw, L, t);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // barriers (the shared prologue initialises none of them: its stage count is 0)
  if (tid == 0) {
    for (uint32_t i = 0; i < stages; ++i) {
      mbar_init(&t.full[i], 1);
      mbar_init(&t.empty[i], 1 + kConsumerWarps);   // the PV's commit + each consumer warp
    }
    for (int g = 0; g < 2; ++g) {
      mbar_init(&t.s_full[g], 1);
      mbar_init(&t.s_free[g], 128);
      mbar_init(&t.p_full[g], 128);
      mbar_init(&t.o_done[g], 1);
    }
    mbar_init(t.q_full, NCT);
    mbar_init(t.drain, 1);
    fence_barrier_init();
  }
  if (warp == kConsumerWarps + 1) tmem_alloc(t.tslot, kTcCols);
  tc_fence_before();
  Layout pl{};        // the shared prologue's view: no stages of its own
  pl.stages = 0;
  prologue<D, 2, kConsumerWarps>(a, s, pl);
  tc_fence_after();
  const TcTmem tm{*t.tslot};

  int64_t xs, xe;
  int cb = 0, ch = 0;
  if constexpr (CLUSTER) {
    const uint32_t cr = cluster_rank(), cn = cluster_size();
    const int bh = (int)(blockIdx.x / cn);
    cb = bh / a.H_kv;
    ch = bh - cb * a.H_kv;
    const int64_t nb = s.pfx[cb + 1] - s.pfx[cb];
    const int64_t x0 = (int64_t)s.pfx[cb] * a.H_kv + (int64_t)ch * nb;
    xs = x0 + nb * cr / cn;
    xe = x0 + nb * (cr + 1) / cn;
  } else {
    const int64_t TP = (int64_t)s.pfx[a.B] * a.H_kv;
    const int64_t n_act = active_ctas(TP, a.n_cta, a.min_pages);
    xs = blockIdx.x < n_act ? cta_begin(blockIdx.x, TP, n_act) : 0;
    xe = blockIdx.x < n_act ? cta_begin(blockIdx.x + 1, TP, n_act) : 0;
  }

  if (warp >= kConsumerWarps) {
    regs_dec<kTcProducerRegs>();
    if (warp == kConsumerWarps) {
      tc_producer(a, s, t, stages, xs, xe, &mk, &mv, &ms);
    } else if (warp == kConsumerWarps + 1) {
      if (lane == 0) tc_mma_thread(a, s, t, tm, stages, xs, xe);
      __syncwarp();
      named_barrier(kTcEndBarrier, NCT + 32);   // the consumers have read TMEM for the last time
      tc_fence_after();
      tmem_dealloc(tm.base, kTcCols);
    }
    if constexpr (CLUSTER) {
      cluster_sync_all();
      cluster_sync_all();
    }
    return;
  }
  regs_inc<kTcConsumerRegs>();
  if constexpr (!CLUSTER) zero_empty<T, D, NCT>(a, s);
  const int grp = warp >> 2;                 // softmax group
  const int gt = tid & 127;                  // thread in the group = key of the step, or dimension
  const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
  float* const own_part = reinterpret_cast<float*>(t.stage);
  float* const mref = t.mref + grp * RK;     // the group's reference maxima (uniform)
  float* const alph = t.alpha + grp * RK;    // rescale factors of a raise
  bool wrote = false;

  uint32_t u = 0, ns[2] = {0u, 0u}, pages = 0;
  bool have[2] = {false, false};
  // this thread's share of its group's row sums: the probabilities of the
  // keys it owned in the group's steps of the piece (summed over the group's
  // threads at the piece's end)
  float lsum[RK];
#pragma unroll
  for (int r = 0; r < RK; ++r) lsum[r] = 0.f;
  int64_t x = xs;
  // Every consumer thread takes the same path through the loop (the steps'
  // page information is read from shared memory by all), so that the named
  // barriers inside it always meet; after a wait gave up the loop still runs
  // to its end, every later wait returning at once.
  while (x < xe) {
    const uint32_t st = u % stages;
    mbar_wait(&t.full[st], (u / stages) & 1u, a.status, s.abort);
    const PageInfo ia = t.info[2 * st], ib = t.info[2 * st + 1];
    __syncwarp();
    if (lane == 0) mbar_arrive(&t.empty[st]);
    const int np = (ia.flags & kPair) ? 2 : 1;
    const bool last = (((np == 2) ? ib.flags : ia.flags) & kLast) != 0;
    if (ia.flags & kFirst) {
      // a new piece: its queries (the previous piece's MMAs have all
      // completed: its end waited for its last PVs)
      prep_queries<T, D, RK, NCT, true, true>(a, s, ia.seq, t.qb);
      fence_async_smem();
      mbar_arrive(t.q_full);
      have[0] = have[1] = false;
#pragma unroll
      for (int r = 0; r < RK; ++r) lsum[r] = 0.f;
      if (gt < RK) mref[gt] = -INFINITY;
      named_barrier(1, NCT);
    }
    const int g = (int)(u & 1u);
    const uint32_t c = ns[g];
    if (grp == g) {
      // ---- softmax of this step: thread gt owns key gt ----
      const int pg = gt >> 6, k = gt & 63;
      const PageInfo ip = pg ? ib : ia;
      const bool page_ok = (ip.flags & kValid) && (pg == 0 || np == 2);
      const int lo = ip.lohi & 0xffff, hi = ip.lohi >> 16;
      const bool key_ok = page_ok && k >= lo && k < hi;
      bool ok = mbar_wait(&t.s_full[g], c & 1u, a.status, s.abort);
      float sc[RK];
      {
        uint32_t sr[RK];
        if (ok) {
          tc_fence_after();
          tmem_ld32(tm.s(g) + lane_off, sr);
          tc_fence_before();
        }
        mbar_arrive(&t.s_free[g]);
#pragma unroll
        for (int r = 0; r < RK; ++r) {
          bool vis = key_ok && ok;
          if (ip.toff != kNoTree) vis = vis && tree_visible(k, ip.toff, s.tmask[r]);
          sc[r] = vis ? __uint_as_float(sr[r]) : -INFINITY;
        }
      }
      bool need = false;
#pragma unroll
      for (int r = 0; r < RK; r += 4) {
        const float4 m4 = *reinterpret_cast<const float4*>(mref + r);
        need |= sc[r] > m4.x + 8.f;
        need |= sc[r + 1] > m4.y + 8.f;
        need |= sc[r + 2] > m4.z + 8.f;
        need |= sc[r + 3] > m4.w + 8.f;
      }
      // group-wide vote: a raise of the reference maxima (rare)
      if (barrier_or(3 + g, 128, need)) {
        // exact row maxima over the group's keys: per warp by one integer
        // reduction per row, then over the group's four warps
        float* red = t.red + g * 4 * RK;
#pragma unroll
        for (int r = 0; r < RK; ++r) {
          const float mx = warp_max(sc[r]);
          if (lane == 0) red[(warp & 3) * RK + r] = mx;
        }
        named_barrier(3 + g, 128);
        if (gt < RK) {
          const float mx = fmaxf(fmaxf(red[gt], red[RK + gt]), fmaxf(red[2 * RK + gt], red[3 * RK + gt]));
          const float mo = mref[gt];
          const float mn = fmaxf(mo, mx);
          alph[gt] = (mn == -INFINITY) ? 1.f : fast_exp2(mo - mn);   // 0 when mo = -inf
          mref[gt] = mn;
        }
        named_barrier(3 + g, 128);
        bool any_alpha = false;
#pragma unroll
        for (int r = 0; r < RK; ++r) any_alpha |= alph[r] != 1.f;
        if (any_alpha) {
#pragma unroll
          for (int r = 0; r < RK; ++r) lsum[r] *= alph[r];
        }
        if (have[g] && any_alpha) {
          // O^T holds this piece's earlier PVs: scale it (thread gt = dimension gt)
          ok = ok && mbar_wait(&t.o_done[g], (c - 1) & 1u, a.status, s.abort);
          if (ok) {
            tc_fence_after();
            tmem_scale32(tm.o(g) + lane_off, alph);
            tc_fence_before();
          }
        }
      }
      // this key's probabilities for every row, as bf16 pairs
      uint32_t pw[RK / 2];
#pragma unroll
      for (int r = 0; r < RK; r += 4) {
        const float4 m4 = *reinterpret_cast<const float4*>(mref + r);
        const float p0 = sc[r] > -INFINITY ? fast_exp2(sc[r] - m4.x) : 0.f;
        const float p1 = sc[r + 1] > -INFINITY ? fast_exp2(sc[r + 1] - m4.y) : 0.f;
        const float p2 = sc[r + 2] > -INFINITY ? fast_exp2(sc[r + 2] - m4.z) : 0.f;
        const float p3 = sc[r + 3] > -INFINITY ? fast_exp2(sc[r + 3] - m4.w) : 0.f;
        lsum[r] += p0;
        lsum[r + 1] += p1;
        lsum[r + 2] += p2;
        lsum[r + 3] += p3;
        pw[r / 2] = pack_bf16(p0, p1);
        pw[r / 2 + 1] = pack_bf16(p2, p3);
      }
      // the P^T buffer is free once this group's previous PV has completed
      if (c > 0) ok = mbar_wait(&t.o_done[g], (c - 1) & 1u, a.status, s.abort) && ok;
      // row gt of P^T: 64 bytes, 64-byte swizzle (16-byte chunk j at j ^ ((gt % 8) / 2))
      uint8_t* prow = t.pt + g * (128 * RK * 2) + (gt >> 3) * 512 + (gt & 7) * 64;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t off = (uint32_t)((j ^ ((gt & 7) >> 1)) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(smem_u32(prow + off)),
                     "r"(pw[4 * j]), "r"(pw[4 * j + 1]), "r"(pw[4 * j + 2]), "r"(pw[4 * j + 3])
                     : "memory");
      }
      if (!key_ok) {   // its value row may hold anything: zero it for the PV
        uint8_t* vrow = t.stage + (size_t)st * kTcStageBytes + 4 * kBoxBytes + pg * kBoxBytes + k * 128;
#pragma unroll
        for (int cbx = 0; cbx < 2; ++cbx)
#pragma unroll
          for (int j = 0; j < 8; ++j)
            asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};"
                         ::"r"(smem_u32(vrow + cbx * 2 * kBoxBytes + j * 16)), "r"(0u) : "memory");
      }
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&t.p_full[g]);
      if (!ok) *s.abort = 1;
    }
    have[g] = true;
    ns[g] = c + 1;
    if (last) {
      // ---- end of the piece: merge the two groups' states ----
      // The group's row sums first (their 32 registers are free before the
      // group's O^T is read): a reduce-scatter leaves lane r of each warp with
      // row r's sum over the warp's keys, which goes to the group's own part
      // of red (the other group may still use its part for a raise in its
      // last step); thread r of the group adds the four warps' after the
      // barrier below.
      float* const lred = t.red + grp * 4 * RK;
      static_assert(RK == 32, "one row per lane");
#pragma unroll
      for (int h = 16; h >= 1; h >>= 1) {
        const bool upper = (lane & h) != 0;
#pragma unroll
        for (int i = 0; i < h; ++i) {
          const float send = upper ? lsum[i] : lsum[i + h];
          const float keep = upper ? lsum[i + h] : lsum[i];
          lsum[i] = keep + __shfl_xor_sync(0xffffffffu, send, h);
        }
      }
      bool mine = have[grp];
      float oo[RK];
      if (mine) {
        const bool ok = mbar_wait(&t.o_done[grp], (ns[grp] - 1) & 1u, a.status, s.abort);
        uint32_t o[RK];
        if (ok) {
          tc_fence_after();
          tmem_ld32(tm.o(grp) + lane_off, o);
        }
#pragma unroll
        for (int r = 0; r < RK; ++r) oo[r] = ok ? __uint_as_float(o[r]) : 0.f;
        mine = ok;
      }
      lred[(warp & 3) * RK + lane] = mine ? lsum[0] : 0.f;
      if (gt < RK && !mine) mref[gt] = -INFINITY;
      // group A's o for the merge goes to the P^T region ([row][dim]): every
      // PV of the piece has completed, so the region is free
      float* mob = reinterpret_cast<float*>(t.pt);
      tc_fence_before();
      named_barrier(1, NCT);
      if (gt < RK) lred[gt] += lred[RK + gt] + lred[2 * RK + gt] + lred[3 * RK + gt];
      if (grp == 0) {
#pragma unroll
        for (int r = 0; r < RK; ++r) mob[r * D + gt] = oo[r];
      }
      named_barrier(1, NCT);
      if (grp == 1) {
        float* part = CLUSTER ? own_part
                              : a.part + ((int64_t)blockIdx.x + ia.seq) * slot_floats(RK, D);
        const float* ma = t.mref;
        const float* mb = t.mref + RK;
#pragma unroll
        for (int r = 0; r < RK; ++r) {
          const float M = fmaxf(ma[r], mb[r]);
          const float sa = ma[r] == -INFINITY ? 0.f : fast_exp2(ma[r] - M);
          const float sb = mb[r] == -INFINITY ? 0.f : fast_exp2(mb[r] - M);
          const float oa = mob[r * D + gt];
          part[slot_o_off(RK) + r * D + gt] = (sa > 0.f ? sa * oa : 0.f) + (sb > 0.f ? sb * oo[r] : 0.f);
          if (gt == 0) {
            const float la = t.red[r], lb = t.red[4 * RK + r];
            part[r] = M;
            part[RK + r] = (sa > 0.f ? sa * la : 0.f) + (sb > 0.f ? sb * lb : 0.f);
          }
        }
      }
      named_barrier(1, NCT);
      if constexpr (CLUSTER) {
        wrote = true;
      } else {
        ticket<T, D, RK, NCT>(a, s, ia.seq, pages + np);
      }
      pages = 0;
    } else {
      pages += np;
    }
    x += np;
    ++u;
  }
  named_barrier_arrive(kEndBarrier, NCT + 32);
  named_barrier_arrive(kTcEndBarrier, NCT + 32);
  if constexpr (CLUSTER) {
    if (!wrote || *s.abort) {
      for (int r = threadIdx.x; r < RK; r += NCT) {
        own_part[r] = -INFINITY;
        own_part[RK + r] = 0.f;
      }
    }
    cluster_sync_all();
    cluster_merge<T, D, RK, NCT>(a, cb, ch, smem_u32(own_part));
    cluster_sync_all();
  }
}

}  // namespace da
