// Split-KV decode kernel: the pipeline of pipeline.cuh driving one of three
// compute engines.
//
//  * CoreEngine (<= 4 query rows per KV head: one draft token over a small GQA
//    group).  QK^T and PV on the FP32 pipes with packed two-wide FMAs; no
//    tensor cores, since with this few rows the page read, not arithmetic, is
//    the bound.  Eight lanes share a key (16 dimensions each at d = 128), a
//    reduce-scatter butterfly leaves lane i with row i's score, and PV runs in
//    the same layout.  With PINGPONG (long selections) the consumer warps form
//    two groups that take alternate steps.
//  * CoreEngineWide (5..8 rows on the FP32 pipes: fp32 caches, or on
//    request).  QK^T as in CoreEngine; for PV every lane owns d/32 dimensions
//    of all rows.
//  * MmaEngine (5..32 rows: a GQA group of 8, or draft trees).  QK^T and PV as
//    bf16 m16n8k16 tensor-core MMAs with FP32 accumulation, keys on the M side
//    of QK^T (S^T = K Q^T) so that 8-row query tiles need no padding, P^T
//    moved into the PV operand layout with movmatrix.
//
// All keep an online softmax (m, l, o) per warp and query row, in the log2
// domain (the query is pre-scaled by softmax_scale * log2 e and by alpha or
// gamma), and merge the eight warps only at the end of a piece.
#pragma once

#include "pipeline.cuh"

namespace da {

// ---------------------------------------------------------------------------
// Query preparation for a piece: RoPE at the query position (or at
// q_pos - P_far for FOLD far memory, which equals rotating the keys at P_far:
// <R(p)q, R(P)k> = <R(p-P)q, k>), times the row's logit multiplier, into s.q
// [rk][d] as FP32, and each row's draft-tree mask into s.tmask.  Rows >= R
// are zero.  Consumer threads only.
// ---------------------------------------------------------------------------
// QB: the rows go to qtile instead, as bf16 in the 128-byte-swizzled K-major
// layout the tcgen05 engine's MMA reads (two [RK][64] boxes, dimensions 0-63
// then 64-127).
template <typename T, int D, int RK, int NCT, bool KSQ = true, bool QB = false>
__device__ inline void prep_queries(const DecodeArgs& a, Smem& s, int seq,
                                    uint8_t* qtile = nullptr) {
  const int tid = threadIdx.x;
  const int bh = seq >> 1, b = bh / a.H_kv, h = bh - b * a.H_kv;
  const int32_t L = s.len[b];
  const bool far = seq_is_far(a.mode, seq);
  const int32_t shift = far ? fold_far_pos(L, a.W) : 0;
  // Row masks and multipliers.  A tree key hidden from a row also leaves that
  // row's SharpDraft count |S| (every tree key lies in the main selection).
  if (tid < RK) {
    const int row = tid;
    uint64_t m = ~0ull;
    if (row < a.R && a.tree_mask && a.n_tree > 0)
      m = __ldg(reinterpret_cast<const unsigned long long*>(a.tree_mask) + b * a.n_q + row / a.G);
    s.tmask[row] = m;
    float mult = a.scale_log2;
    if (far) {
      // "FOLD", abstract: concentration factor; an FP8 side cache's scale
      // (unless the engine applies it to the scores: KSQ false)
      mult *= KSQ ? a.alpha * a.far_kscale : a.alpha;
    } else if (a.mode == DA_MODE_SHARP) {    // "SharpDraft", Abstract: query scaling
      int32_t n = visible_keys(a.mode, L, a.W, a.n_sink);
      if (a.tree_mask && a.n_tree > 0) {
        const int32_t present = min(a.n_tree, L);   // tree tokens that exist
        const uint64_t bits = (present >= 64 ? ~0ull : ((1ull << present) - 1))
                              << (a.n_tree - present);
        n -= present - __popcll(m & bits);
      }
      if (n > 0) mult *= fmaxf(1.f, 1.f + a.beta * logf((float)n / (float)a.n_ref));
    }
    s.rmult[row] = mult;
  }
  // The query elements this thread rotates are loaded first, so that their
  // latency overlaps the position loads and the angle table.
  constexpr int PER = (RK * (D / 2) + NCT - 1) / NCT;   // rotate-half pairs per thread
  const T* qb = static_cast<const T*>(a.q);
  float qx[PER], qy[PER];
#pragma unroll
  for (int u = 0; u < PER; ++u) {
    const int i = tid + u * NCT;
    const int row = i / (D / 2), f = i - row * (D / 2);
    qx[u] = qy[u] = 0.f;
    if (i < RK * (D / 2) && row < a.R) {
      const int t = row / a.G, j = row - t * a.G;
      const T* src = qb + ((int64_t)(b * a.n_q + t) * a.H_q + h * a.G + j) * D;
      qx[u] = to_f32<T>(src[f]);
      qy[u] = to_f32<T>(src[f + D / 2]);
    }
  }
  float2* cs = reinterpret_cast<float2*>(s.mo);
  for (int i = tid; i < a.n_q * (D / 2); i += NCT) {
    const int t = i / (D / 2), f = i - t * (D / 2);
    const int32_t p = __ldg(a.q_pos + b * a.n_q + t) - shift;
    float c, sn;
    rope_cos_sin(p, s.invf[f], c, sn);
    cs[i] = make_float2(c, sn);
  }
  named_barrier(1, NCT);
#pragma unroll
  for (int u = 0; u < PER; ++u) {
    const int i = tid + u * NCT;
    if (i < RK * (D / 2)) {
      const int row = i / (D / 2), f = i - row * (D / 2);
      float xr = 0.f, yr = 0.f;
      if (row < a.R) {
        const float2 c = cs[(row / a.G) * (D / 2) + f];
        const float mult = s.rmult[row];
        xr = (qx[u] * c.x - qy[u] * c.y) * mult;
        yr = (qy[u] * c.x + qx[u] * c.y) * mult;
      }
      if constexpr (QB) {
        // dims f and f + D/2 (D = 128: box 0 and box 1, same column)
        static_assert(D == 128, "tcgen05 query tile");
        const int byte = f * 2;
        const uint32_t off = (uint32_t)row * 128 + ((((byte >> 4) ^ row) & 7) << 4) + (byte & 15);
        *reinterpret_cast<__nv_bfloat16*>(qtile + off) = __float2bfloat16_rn(xr);
        *reinterpret_cast<__nv_bfloat16*>(qtile + RK * 128 + off) = __float2bfloat16_rn(yr);
      } else {
        s.q[row * D + f] = xr;
        s.q[row * D + f + D / 2] = yr;
      }
    }
  }
  named_barrier(1, NCT);
}

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

// Whether a row with tree mask m sees key `key` of a page whose key k is tree
// token k + toff (toff = kNoTree: no tree key under a mask in this page).
__device__ __forceinline__ bool tree_visible(int key, int toff, uint64_t m) {
  const int ti = key + toff;
  return (unsigned)ti >= 64u || ((m >> ti) & 1ull) != 0;
}

// Reduce-scatter of RK per-lane partial sums over the W lanes of a key group
// (lane bits below log2 W): afterwards lane ds holds the total for row
// ds & (RK-1).
template <int RK, int W>
__device__ __forceinline__ float reduce_scatter(float (&v)[RK], int ds) {
#pragma unroll
  for (int m = RK / 2; m >= 1; m >>= 1) {
    const bool up = (ds & m) != 0;
#pragma unroll
    for (int i = 0; i < m; ++i) {
      const float send = up ? v[i] : v[i + m];
      const float keep = up ? v[i + m] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
    }
  }
  float x = v[0];
#pragma unroll
  for (int m = RK; m < W; m <<= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
  return x;
}
template <int RK>
__device__ __forceinline__ float reduce_scatter8(float (&v)[RK], int ds) {
  return reduce_scatter<RK, 8>(v, ds);
}

template <typename T>
struct Chunk;  // one 16-byte shared-memory chunk as floats
// raw(): the 16 bytes as loaded; cvt(): those bytes as floats.
template <>
struct Chunk<__nv_bfloat16> {
  __device__ __forceinline__ static void raw(uint32_t addr, uint32_t (&w)[4]) {
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]) : "r"(addr));
  }
  __device__ __forceinline__ static void cvt(const uint32_t (&w)[4], float (&f)[8]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = bf16lo(w[i]);
      f[2 * i + 1] = bf16hi(w[i]);
    }
  }
  __device__ __forceinline__ static void load(uint32_t addr, float (&f)[8]) {
    uint32_t w[4];
    raw(addr, w);
    cvt(w, f);
  }
};
template <>
struct Chunk<float> {
  __device__ __forceinline__ static void raw(uint32_t addr, uint32_t (&w)[4]) {
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]) : "r"(addr));
  }
  __device__ __forceinline__ static void cvt(const uint32_t (&w)[4], float (&f)[4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) f[i] = __uint_as_float(w[i]);
  }
  __device__ __forceinline__ static void load(uint32_t addr, float (&f)[4]) {
    uint32_t w[4];
    raw(addr, w);
    cvt(w, f);
  }
};

// Four E4M3 codes (bytes of w, lowest first) as floats: two codes at a time
// to an f16 pair (every E4M3 value is an f16 value), then each f16 to f32.
__device__ __forceinline__ void e4m3x4_to_f32(uint32_t w, float& f0, float& f1, float& f2,
                                              float& f3) {
  asm("{\n\t.reg .b16 a, b, c0, c1, c2, c3;\n\t.reg .b32 h0, h1;\n\t"
      "mov.b32 {a, b}, %4;\n\t"
      "cvt.rn.f16x2.e4m3x2 h0, a;\n\t"
      "cvt.rn.f16x2.e4m3x2 h1, b;\n\t"
      "mov.b32 {c0, c1}, h0;\n\t"
      "mov.b32 {c2, c3}, h1;\n\t"
      "cvt.f32.f16 %0, c0;\n\t"
      "cvt.f32.f16 %1, c1;\n\t"
      "cvt.f32.f16 %2, c2;\n\t"
      "cvt.f32.f16 %3, c3;\n\t}"
      : "=f"(f0), "=f"(f1), "=f"(f2), "=f"(f3)
      : "r"(w));
}

// DPL consecutive elements (the PV slice of one lane) as floats.
template <typename T, int DPL>
__device__ __forceinline__ void load_slice(uint32_t addr, float (&f)[DPL]) {
  if constexpr (sizeof(T) == 2 && DPL == 4) {
    uint32_t w0, w1;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(w0), "=r"(w1) : "r"(addr));
    f[0] = bf16lo(w0); f[1] = bf16hi(w0); f[2] = bf16lo(w1); f[3] = bf16hi(w1);
  } else if constexpr (sizeof(T) == 2 && DPL == 2) {
    uint32_t w0;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w0) : "r"(addr));
    f[0] = bf16lo(w0); f[1] = bf16hi(w0);
  } else if constexpr (sizeof(T) == 4 && DPL == 4) {
    asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(f[0]), "=f"(f[1]), "=f"(f[2]), "=f"(f[3]) : "r"(addr));
  } else {
    static_assert(sizeof(T) == 4 && DPL == 2, "slice shape");
    asm volatile("ld.shared.v2.f32 {%0,%1}, [%2];" : "=f"(f[0]), "=f"(f[1]) : "r"(addr));
  }
}

// ---------------------------------------------------------------------------
// CUDA-core engine, 1..4 rows.  Without PINGPONG the eight consumer warps
// share every step (two consecutive pages of a piece, or one) and warp w owns
// keys 8w .. 8w+7 of each page.  With PINGPONG (the long selections of full,
// FOLD and SharpDraft) they form two groups of four that take turns: a group
// takes a whole step, the other group the next one, so each scheduler holds
// one warp of each group and one group's reductions and shuffles overlap the
// other's dot products; warp w of a group owns keys 16w .. 16w+15.  The eight
// lanes of key group kg (lane bits 3, 4) share key KPW w + kg + 4 ps on pass
// ps and lane ds (bits 0..2) owns D/8 of its
// dimensions, read as 16-byte chunks whose order is rotated by ds (no bank
// conflicts under the 128-byte swizzle).  QK^T: per-lane partial dots, then a
// reduce-scatter leaves lane ds with row ds's score.  PV runs in the same
// layout: the row probabilities of the lane's key come back by shuffle, the
// lane accumulates p * V over its own dimensions, and the key groups are
// summed only at the end of a piece.  The running maximum is raised lazily
// (only when a score exceeds it by more than 2^8): the result is exact for
// any reference value, and the accumulators are rescaled only a handful of
// times.
// With F8 (FOLD with an FP8 side cache) a far piece's keys are rows of D
// E4M3 codes: lane ds reads its DQ = D/8 dimensions DQ ds .. DQ ds + DQ - 1 in
// one load (d 128: a 16-byte chunk of a 128-byte row, row-rotated by the TMA
// swizzle, so the eight lanes of a key cover all 32 banks; d 64: 8 bytes of an
// unswizzled 64-byte row, four consecutive keys filling 256 contiguous bytes),
// and the piece's queries are laid out in that order (begin_far).
// ---------------------------------------------------------------------------
// Where a piece's partial (m[RK], l[RK], pad, o[RK][D], as floats) goes: plain
// stores through `p` (the workspace), or, on the cluster partition,
// asynchronous stores into rank 0's slot (shared::cluster address `sa`), each
// counted on rank 0's merge barrier (`bar`).  Offsets are in floats.
struct PartOut {
  float* p;
  uint32_t sa, bar;
  __device__ __forceinline__ void put4(int off, float4 v) const {
    if (bar) st_async_f32x4(sa + 4u * (uint32_t)off, v, bar);
    else *reinterpret_cast<float4*>(p + off) = v;
  }
  __device__ __forceinline__ void put1(int off, float v) const {
    if (bar) st_async_f32(sa + 4u * (uint32_t)off, v, bar);
    else p[off] = v;
  }
};
// Bytes a partial of RK rows sends to rank 0 (m, l and o; not the pad).
__host__ __device__ constexpr uint32_t part_bytes(int rk, int d) {
  return (uint32_t)(2 * rk + rk * d) * 4u;
}

template <typename T, int D, int RK, bool PINGPONG, bool F8 = false>
struct CoreEngine {
  static constexpr int NCW = kConsumerWarps;
  static constexpr int NCT = NCW * 32;
  static constexpr bool kPairs = true;         // takes two pages per step
  static constexpr bool kPingPong = PINGPONG;  // the two warp groups alternate steps
  static constexpr bool kSideF8 = F8;          // far keys as E4M3 codes
  static constexpr bool kFarScaleInQ = true;
  static constexpr int GW = PINGPONG ? NCW / 2 : NCW;   // warps sharing a step
  static constexpr int LPK = 8;                // lanes per key
  static constexpr int KG = 32 / LPK;          // key groups per pass
  static constexpr int KPW = 64 / GW;          // keys per warp and page
  static constexpr int PP = KPW / KG;          // passes per page
  static constexpr int ES = sizeof(T);
  static constexpr int DQ = D / LPK;           // dimensions per lane
  static constexpr int NCH = DQ * ES / 16;     // 16-byte chunks per lane (1, 2 or 4)
  static constexpr int EPC = 16 / ES;          // elements per chunk
  static constexpr float kLazy = 8.f;          // log2 headroom before a rescale
  static_assert(RK == 1 || RK == 2 || RK == 4, "rows");
  static_assert(NCH >= 1 && (NCH & (NCH - 1)) == 0, "chunks");
  static_assert(!F8 || (ES == 2 && PINGPONG), "FP8 side cache: bf16, turn-taking groups");

  float2 q2[RK][DQ / 2];
  float2 o2[RK][DQ / 2];
  float m_run, l_run;    // row ds & (RK-1): reference maximum, partial sum
  // Swizzled byte offsets of the lane's chunks on passes 0 and 1; pass ps adds
  // 1024 (ps / 2) bytes: its row is 8 further on and has the same swizzle.
  uint32_t off[2][NCH];
  uint32_t off8[2];      // F8: the lane's E4M3 codes on passes 0 and 1 (pass ps: + 8 D (ps / 2))
  int lane, warp, kg, ds;
  static_assert(KG == 4, "rows of passes ps and ps + 2 differ by 8");
  __device__ __forceinline__ uint32_t off_of(int ps, int i) const {
    return off[ps & 1][i] + (uint32_t)(ps >> 1) * (8 * kSwizzleRow);
  }

  __device__ __forceinline__ int chunk_of(int i) const {
    return ds * NCH + ((i + ((ds * NCH) >> 3)) & (NCH - 1));
  }
  // Dimension of element e of chunk slot i of this lane.
  __device__ __forceinline__ int dim_of(int i, int e) const { return chunk_of(i) * EPC + e; }

  __device__ __forceinline__ void init() {
    lane = threadIdx.x & 31;
    warp = threadIdx.x >> 5;
    kg = lane / LPK;
    ds = lane % LPK;
#pragma unroll
    for (int it = 0; it < 2; ++it)
#pragma unroll
      for (int i = 0; i < NCH; ++i)
        off[it][i] = swz_addr(0u, (warp & (GW - 1)) * KPW + kg + KG * it, chunk_of(i) * 16);
    if constexpr (F8) {
#pragma unroll
      for (int it = 0; it < 2; ++it) {
        const int row = (warp & (GW - 1)) * KPW + kg + KG * it;
        off8[it] = D == 128 ? swz_addr(0u, row, ds * 16) : (uint32_t)(row * D + ds * DQ);
      }
    }
  }

  // Step u (a pair or a single page) belongs to warp group u mod 2.
  __device__ __forceinline__ bool owns(uint32_t u) const {
    return !PINGPONG || (int)(u & 1u) == warp / GW;
  }

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int r = 0; r < RK; ++r)
#pragma unroll
      for (int e = 0; e < DQ / 2; ++e) o2[r][e] = make_float2(0.f, 0.f);
    m_run = -INFINITY;
    l_run = 0.f;
  }

  __device__ __forceinline__ void begin(const Smem& s) {
#pragma unroll
    for (int i = 0; i < NCH; ++i)
#pragma unroll
      for (int r = 0; r < RK; ++r)
#pragma unroll
        for (int e = 0; e < EPC / 2; ++e) {
          const int d0 = dim_of(i, 2 * e);
          q2[r][i * (EPC / 2) + e] = make_float2(s.q[r * D + d0], s.q[r * D + d0 + 1]);
        }
    reset();
  }

  // F8: a far piece takes its queries in the order of the lane's E4M3 codes
  // (slot i, pair e: dimensions DQ ds + EPC i + 2 e, + 1).
  __device__ __forceinline__ void begin_far(const Smem& s, bool far) {
    if (!far) {
      begin(s);
      return;
    }
#pragma unroll
    for (int i = 0; i < NCH; ++i)
#pragma unroll
      for (int r = 0; r < RK; ++r)
#pragma unroll
        for (int e = 0; e < EPC / 2; ++e) {
          const int d0 = ds * DQ + i * EPC + 2 * e;
          q2[r][i * (EPC / 2) + e] = make_float2(s.q[r * D + d0], s.q[r * D + d0 + 1]);
        }
    reset();
  }

  // NP consecutive pages of one piece: K/V stage addresses, valid key ranges
  // [lo, hi) inside each page and tree offsets.  FK: the keys are E4M3 rows.
  template <int NP, bool FK = false>
  __device__ __forceinline__ void pages(const Smem& s, const uint32_t (&kb)[NP],
                                        const uint32_t (&vb)[NP], const int (&lo)[NP],
                                        const int (&hi)[NP], const int (&toff)[NP]) {
    constexpr int NIT = PP * NP;
    // With 4 rows two passes share one reduce-scatter (8 values over the 8
    // lanes of a key group): lane ds then holds row ds & 3 of pass
    // 2 j + (ds >> 2), no lane duplicates another, and a lane keeps NIT / 2
    // scores.  Fewer rows keep one reduce-scatter per pass.
    constexpr bool PAIR = RK == 4;
    static_assert(!PAIR || (PP % 2 == 0), "paired passes stay inside a page");
    constexpr int NS = PAIR ? NIT / 2 : NIT;   // scores per lane
    const int kw = (warp & (GW - 1)) * KPW + kg;   // the lane's key on pass 0
    float sc[NS];
    // bit it: the key of pass it is inside [lo, hi) of its page (a mask in one
    // register rather than NIT predicates)
    uint32_t okm = 0;
    float vp[PAIR ? 2 * RK : 1];   // PAIR: the even pass's partial sums
#pragma unroll
    for (int it = 0; it < NIT; ++it) {
      const int pg = it / PP, ps = it % PP;
      const int key = kw + KG * ps;
      okm |= (key >= lo[pg] && key < hi[pg]) ? 1u << it : 0u;
      // With turn-taking groups, two accumulators per row (even and odd element
      // pairs) halve the chain of dependent FFMA2s behind each dot product
      // (FOLD 4 x 256K 694 -> 686 us; the shared-step window engine is faster
      // with one).
      constexpr int NA = PINGPONG ? 2 : 1;
      float2 acc[NA][RK];
#pragma unroll
      for (int u = 0; u < NA; ++u)
#pragma unroll
        for (int r = 0; r < RK; ++r) acc[u][r] = make_float2(0.f, 0.f);
      if constexpr (FK) {
        static_assert(NCH * EPC == DQ && (DQ == 16 || DQ == 8), "one load per lane and key");
        constexpr int NW = DQ / 4;   // 32-bit words of codes
        uint32_t w[NW];
        const uint32_t ka = kb[pg] + off8[ps & 1] + (uint32_t)(ps >> 1) * (8 * D);
        if constexpr (NW == 4)
          asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                       : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]) : "r"(ka));
        else
          asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(w[0]), "=r"(w[1]) : "r"(ka));
        float f[DQ];
#pragma unroll
        for (int j = 0; j < NW; ++j) e4m3x4_to_f32(w[j], f[4 * j], f[4 * j + 1], f[4 * j + 2], f[4 * j + 3]);
#pragma unroll
        for (int i = 0; i < NCH; ++i)
#pragma unroll
          for (int e = 0; e < EPC / 2; ++e) {
            const float2 kk = make_float2(f[i * EPC + 2 * e], f[i * EPC + 2 * e + 1]);
#pragma unroll
            for (int r = 0; r < RK; ++r)
              acc[e % NA][r] = ffma2(q2[r][i * (EPC / 2) + e], kk, acc[e % NA][r]);
          }
      } else {
#pragma unroll
        for (int i = 0; i < NCH; ++i) {
          float f[EPC];
          Chunk<T>::load(kb[pg] + off_of(ps, i), f);
#pragma unroll
          for (int e = 0; e < EPC / 2; ++e) {
            const float2 kk = make_float2(f[2 * e], f[2 * e + 1]);
#pragma unroll
            for (int r = 0; r < RK; ++r)
              acc[e % NA][r] = ffma2(q2[r][i * (EPC / 2) + e], kk, acc[e % NA][r]);
          }
        }
      }
      float v[RK];
#pragma unroll
      for (int r = 0; r < RK; ++r) {
        float2 t = acc[0][r];
        if constexpr (NA == 2) t = make_float2(t.x + acc[1][r].x, t.y + acc[1][r].y);
        v[r] = t.x + t.y;
      }
      if constexpr (PAIR) {
#pragma unroll
        for (int r = 0; r < RK; ++r) vp[(it & 1) * RK + r] = v[r];
        if (it & 1) sc[it >> 1] = reduce_scatter<2 * RK, LPK>(vp, ds);
      } else {
        const float sr = reduce_scatter<RK, LPK>(v, ds);
        sc[it] = ((okm >> it) & 1u) ? sr : -INFINITY;
      }
    }
    if constexpr (PAIR) {
#pragma unroll
      for (int j = 0; j < NS; ++j)
        if (!((okm >> (2 * j + ((ds & 4) ? 1 : 0))) & 1u)) sc[j] = -INFINITY;
    }
    // Draft-tree keys the row does not see (only pages that hold tree keys).
    bool has_tree = false;
#pragma unroll
    for (int pg = 0; pg < NP; ++pg) has_tree |= toff[pg] != kNoTree;
    if (has_tree) {
      const uint64_t tm = s.tmask[ds & (RK - 1)];
#pragma unroll
      for (int j = 0; j < NS; ++j) {
        const int it = PAIR ? 2 * j + (ds >> 2) : j;   // the pass of the lane's key
        if (!tree_visible(kw + KG * (it % PP), toff[(PAIR ? 2 * j : j) / PP], tm))
          sc[j] = -INFINITY;
      }
    }
    // Row maximum over the warp's keys (lanes holding the same row).
    float mx = sc[0];
#pragma unroll
    for (int j = 1; j < NS; ++j) mx = fmaxf(mx, sc[j]);
#pragma unroll
    for (int m = PAIR ? RK : LPK; m < 32; m <<= 1)
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
    const bool raise = mx > m_run + kLazy;
    if (__any_sync(0xffffffffu, raise)) {
      const float m_new = raise ? mx : m_run;
      const float al = raise ? fast_exp2(m_run - m_new) : 1.f;   // 0 when m_run = -inf
      l_run *= al;
      m_run = m_new;
#pragma unroll
      for (int r = 0; r < RK; ++r) {
        const float ar = __shfl_sync(0xffffffffu, al, (lane & ~(LPK - 1)) | r);
#pragma unroll
        for (int e = 0; e < DQ / 2; ++e) {
          o2[r][e].x *= ar;
          o2[r][e].y *= ar;
        }
      }
    }
    float p[NS];
#pragma unroll
    for (int j = 0; j < NS; ++j) {
      p[j] = sc[j] > -INFINITY ? fast_exp2(sc[j] - m_run) : 0.f;
      l_run += p[j];
    }
    // PV in the QK^T layout.  A key outside [lo, hi) may hold anything, NaN
    // included: it reads the zeroed chunk instead (its probability is 0).
#pragma unroll
    for (int it = 0; it < NIT; ++it) {
      const int pg = it / PP, ps = it % PP;
      float pr[RK];
#pragma unroll
      for (int r = 0; r < RK; ++r)
        pr[r] = PAIR ? __shfl_sync(0xffffffffu, p[it >> 1], (lane & ~(LPK - 1)) | r | ((it & 1) << 2))
                     : __shfl_sync(0xffffffffu, p[it], (lane & ~(LPK - 1)) | r);
#pragma unroll
      for (int i = 0; i < NCH; ++i) {
        float f[EPC];
        Chunk<T>::load(((okm >> it) & 1u) ? vb[pg] + off_of(ps, i) : s.zero16, f);
#pragma unroll
        for (int e = 0; e < EPC / 2; ++e) {
          const float2 vv = make_float2(f[2 * e], f[2 * e + 1]);
#pragma unroll
          for (int r = 0; r < RK; ++r)
            o2[r][i * (EPC / 2) + e] = ffma2(make_float2(pr[r], pr[r]), vv, o2[r][i * (EPC / 2) + e]);
        }
      }
    }
  }

  template <bool FK = false>
  __device__ __forceinline__ void page(const Smem& s, uint32_t kbase, uint32_t vbase, int lo, int hi,
                                       int toff) {
    const uint32_t kb[1] = {kbase}, vb[1] = {vbase};
    const int l[1] = {lo}, h[1] = {hi}, o[1] = {toff};
    pages<1, FK>(s, kb, vb, l, h, o);
  }

  // Sum the key groups, merge the consumer warps, write the piece's partial.
  // part: where the piece's partial (m[RK], l[RK], pad, o[RK][D]) goes (global or shared).
  __device__ __forceinline__ void finish(const Smem& s, const PartOut& part) {
    float lt = l_run;
    // with 4 rows lanes ds and ds ^ 4 hold one row's sums over different keys
#pragma unroll
    for (int m = RK == 4 ? RK : LPK; m < 32; m <<= 1) lt += __shfl_xor_sync(0xffffffffu, lt, m);
    if (kg == 0 && ds < RK) s.ml[warp * RK + ds] = make_float2(m_run, lt);
    // The four key groups' partial outputs, reduce-scattered over lane bits
    // 4 and 3: the lane's RK (D / 8) values, as float2 slots f = r (DQ / 2) + e,
    // halve twice, and key group kg is left with the totals of the quarter
    // of slots from kg (NV / 4) on, which it writes.
    constexpr int NV = RK * (DQ / 2);
    static_assert(NV % 4 == 0, "quarters");
    float2* const v = &o2[0][0];
    const bool b1 = (kg & 2) != 0, b0 = (kg & 1) != 0;
#pragma unroll
    for (int i = 0; i < NV / 2; ++i) {
      const float2 send = b1 ? v[i] : v[i + NV / 2];
      const float2 keep = b1 ? v[i + NV / 2] : v[i];
      v[i] = make_float2(keep.x + __shfl_xor_sync(0xffffffffu, send.x, 16),
                         keep.y + __shfl_xor_sync(0xffffffffu, send.y, 16));
    }
#pragma unroll
    for (int i = 0; i < NV / 4; ++i) {
      const float2 send = b0 ? v[i] : v[i + NV / 4];
      const float2 keep = b0 ? v[i + NV / 4] : v[i];
      v[i] = make_float2(keep.x + __shfl_xor_sync(0xffffffffu, send.x, 8),
                         keep.y + __shfl_xor_sync(0xffffffffu, send.y, 8));
    }
#pragma unroll
    for (int i = 0; i < NV / 4; ++i) {
      const int f = kg * (NV / 4) + i;
      const int r = f / (DQ / 2), e = f % (DQ / 2);
      *reinterpret_cast<float2*>(s.mo + (warp * RK + r) * D + dim_of(e / (EPC / 2), 2 * (e % (EPC / 2)))) = v[i];
    }
    named_barrier(1, NCT);
    for (int idx = threadIdx.x; idx < RK * D / 4; idx += NCT) {
      const int r = idx / (D / 4), d4 = idx - r * (D / 4);
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < NCW; ++w) M = fmaxf(M, s.ml[w * RK + r].x);
      float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
      float l = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < NCW; ++w) {
          const float2 ml = s.ml[w * RK + r];
          const float sc = fast_exp2(ml.x - M);
          const float4 v = *reinterpret_cast<const float4*>(s.mo + (w * RK + r) * D + 4 * d4);
          o.x = fmaf(sc, v.x, o.x);
          o.y = fmaf(sc, v.y, o.y);
          o.z = fmaf(sc, v.z, o.z);
          o.w = fmaf(sc, v.w, o.w);
          l = fmaf(sc, ml.y, l);
        }
      }
      part.put4(slot_o_off(RK) + r * D + 4 * d4, o);
      if (d4 == 0) {
        part.put1(r, M);
        part.put1(RK + r, l);
      }
    }
    named_barrier(1, NCT);
    reset();
  }
};

// ---------------------------------------------------------------------------
// CUDA-core engine for 5..8 rows (fp32 caches, or on request).  QK^T as in
// CoreEngine; PV with every lane owning d/32 dimensions of all rows and the
// probabilities passed through shared memory.
// ---------------------------------------------------------------------------
template <typename T, int D, int RK>
struct CoreEngineWide {
  static constexpr bool kPairs = false;
  static constexpr bool kPingPong = false;
  static constexpr bool kSideF8 = false;
  static constexpr bool kFarScaleInQ = true;
  static constexpr int NCW = 8;
  static constexpr int NCT = NCW * 32;
  static constexpr int ES = sizeof(T);
  static constexpr int DQ = D / 8;            // QK dims per lane
  static constexpr int NCH = DQ * ES / 16;    // 16-byte chunks per lane (1, 2 or 4)
  static constexpr int EPC = 16 / ES;         // elements per chunk
  static constexpr int DPL = D / 32;          // PV dims per lane
  static_assert(RK == 1 || RK == 2 || RK == 4 || RK == 8, "rows");
  static_assert(NCH >= 1 && (NCH & (NCH - 1)) == 0, "chunks");

  float2 q2[RK][DQ / 2];
  float2 o2[RK][DPL / 2];
  float m_run, l_run;
  int lane, warp, kg, ds;

  __device__ __forceinline__ void init() {
    lane = threadIdx.x & 31;
    warp = threadIdx.x >> 5;
    kg = lane >> 3;
    ds = lane & 7;
  }

  __device__ __forceinline__ bool owns(uint32_t) const { return true; }

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int r = 0; r < RK; ++r)
#pragma unroll
      for (int e = 0; e < DPL / 2; ++e) o2[r][e] = make_float2(0.f, 0.f);
    m_run = -INFINITY;
    l_run = 0.f;
  }

  __device__ __forceinline__ void begin(const Smem& s) {
    // The lane's QK dims, chunk order rotated by ds so that the eight lanes of
    // a key group hit eight different 16-byte bank groups.
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
      const int ic = (i + ((ds * NCH) >> 3)) & (NCH - 1);
      const int d0 = (ds * NCH + ic) * EPC;
#pragma unroll
      for (int r = 0; r < RK; ++r)
#pragma unroll
        for (int e = 0; e < EPC / 2; ++e)
          q2[r][i * (EPC / 2) + e] = make_float2(s.q[r * D + d0 + 2 * e], s.q[r * D + d0 + 2 * e + 1]);
    }
    reset();
  }

  __device__ __forceinline__ void pv_key(uint32_t vbase, const float* pw, int key, int j) {
    float v[DPL];
    load_slice<T, DPL>(swz_addr(vbase, key, lane * DPL * ES), v);
    float pj[RK];
    if constexpr (RK >= 4) {
#pragma unroll
      for (int r = 0; r < RK; r += 4) {
        const float4 x = *reinterpret_cast<const float4*>(pw + j * RK + r);
        pj[r] = x.x; pj[r + 1] = x.y; pj[r + 2] = x.z; pj[r + 3] = x.w;
      }
    } else {
#pragma unroll
      for (int r = 0; r < RK; ++r) pj[r] = pw[j * RK + r];
    }
#pragma unroll
    for (int r = 0; r < RK; ++r)
#pragma unroll
      for (int e = 0; e < DPL / 2; ++e)
        o2[r][e] = ffma2(make_float2(pj[r], pj[r]), make_float2(v[2 * e], v[2 * e + 1]), o2[r][e]);
  }

  __device__ __forceinline__ void page(const Smem& s, uint32_t kbase, uint32_t vbase, int lo, int hi,
                                       int toff) {
    const int wk0 = warp * 8;
    float sc[2];
#pragma unroll
    for (int it = 0; it < 2; ++it) {
      const int key = wk0 + kg + 4 * it;
      float2 acc[RK];
#pragma unroll
      for (int r = 0; r < RK; ++r) acc[r] = make_float2(0.f, 0.f);
#pragma unroll
      for (int i = 0; i < NCH; ++i) {
        const int ic = (i + ((ds * NCH) >> 3)) & (NCH - 1);
        float f[EPC];
        Chunk<T>::load(swz_addr(kbase, key, (ds * NCH + ic) * 16), f);
#pragma unroll
        for (int e = 0; e < EPC / 2; ++e) {
          const float2 kk = make_float2(f[2 * e], f[2 * e + 1]);
#pragma unroll
          for (int r = 0; r < RK; ++r) acc[r] = ffma2(q2[r][i * (EPC / 2) + e], kk, acc[r]);
        }
      }
      float v[RK];
#pragma unroll
      for (int r = 0; r < RK; ++r) v[r] = acc[r].x + acc[r].y;
      const float sr = reduce_scatter8<RK>(v, ds);
      sc[it] = (key >= lo && key < hi) ? sr : -INFINITY;
    }
    if (toff != kNoTree) {   // draft-tree keys the row does not see
      const uint64_t tm = s.tmask[ds & (RK - 1)];
#pragma unroll
      for (int it = 0; it < 2; ++it)
        if (!tree_visible(wk0 + kg + 4 * it, toff, tm)) sc[it] = -INFINITY;
    }
    // Online softmax for row ds & (RK-1) over the warp's 8 keys.
    float mx = fmaxf(sc[0], sc[1]);
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    const float m_new = fmaxf(m_run, mx);
    float alpha = 1.f, p0 = 0.f, p1 = 0.f;
    if (m_new != -INFINITY) {
      alpha = fast_exp2(m_run - m_new);
      p0 = fast_exp2(sc[0] - m_new);
      p1 = fast_exp2(sc[1] - m_new);
    }
    l_run = l_run * alpha + p0 + p1;
    m_run = m_new;
    float* pw = s.p + warp * 9 * RK;
    __syncwarp();
    if (ds < RK) {
      pw[kg * RK + ds] = p0;
      pw[(kg + 4) * RK + ds] = p1;
      if (kg == 0) pw[8 * RK + ds] = alpha;
    }
    __syncwarp();
    // PV over the warp's valid keys.
#pragma unroll
    for (int r = 0; r < RK; ++r) {
      const float al = pw[8 * RK + r];
#pragma unroll
      for (int e = 0; e < DPL / 2; ++e) {
        o2[r][e].x *= al;
        o2[r][e].y *= al;
      }
    }
    const int jlo = max(lo - wk0, 0), jhi = min(hi - wk0, 8);
    if (jlo == 0 && jhi == 8) {
#pragma unroll
      for (int j = 0; j < 8; ++j) pv_key(vbase, pw, wk0 + j, j);
    } else {
      for (int j = jlo; j < jhi; ++j) pv_key(vbase, pw, wk0 + j, j);
    }
  }

  // Merge the eight warps' states and write the piece's partial to `slot`.
  // part: where the piece's partial (m[RK], l[RK], pad, o[RK][D]) goes (global or shared).
  __device__ __forceinline__ void finish(const Smem& s, const PartOut& part) {
    float lt = l_run + __shfl_xor_sync(0xffffffffu, l_run, 8);
    lt += __shfl_xor_sync(0xffffffffu, lt, 16);
    if (kg == 0 && ds < RK) s.ml[warp * RK + ds] = make_float2(m_run, lt);
#pragma unroll
    for (int r = 0; r < RK; ++r)
#pragma unroll
      for (int e = 0; e < DPL / 2; ++e)
        *reinterpret_cast<float2*>(s.mo + (warp * RK + r) * D + lane * DPL + 2 * e) = o2[r][e];
    named_barrier(1, NCT);
    for (int idx = threadIdx.x; idx < RK * D / 4; idx += NCT) {
      const int r = idx / (D / 4), d4 = idx - r * (D / 4);
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < NCW; ++w) M = fmaxf(M, s.ml[w * RK + r].x);
      float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
      float l = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < NCW; ++w) {
          const float2 ml = s.ml[w * RK + r];
          const float sc = fast_exp2(ml.x - M);
          const float4 v = *reinterpret_cast<const float4*>(s.mo + (w * RK + r) * D + 4 * d4);
          o.x = fmaf(sc, v.x, o.x);
          o.y = fmaf(sc, v.y, o.y);
          o.z = fmaf(sc, v.z, o.z);
          o.w = fmaf(sc, v.w, o.w);
          l = fmaf(sc, ml.y, l);
        }
      }
      part.put4(slot_o_off(RK) + r * D + 4 * d4, o);
      if (d4 == 0) {
        part.put1(r, M);
        part.put1(RK + r, l);
      }
    }
    named_barrier(1, NCT);
    reset();
  }
};

// ---------------------------------------------------------------------------
// Tensor-core engine (bf16 only, 32 rows).  Warp w: key block kb = w & 3 (16
// keys of the page), row group rg = w >> 2 (16 query rows, two n8 tiles).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_f16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// Two E4M3 codes (low byte first) as an f16 pair, exactly.
__device__ __forceinline__ uint32_t e4m3x2_f16x2(uint32_t two_codes) {
  uint32_t r;
  asm("{\n\t.reg .b16 c;\n\tcvt.u16.u32 c, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, c;\n\t}"
      : "=r"(r) : "r"(two_codes));
  return r;
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// NT n8 tiles of query rows per warp.  Warp w takes key block kb = w & 3 (16
// of the page's 64 keys) and belongs to group grp = w >> 2.
//  * SPLIT_PAGES: the two groups take alternate pages and each holds all
//    RK = 8 NT rows (8 or 16 rows: one query token with a GQA group of 8, or
//    a small draft tree).
//  * otherwise: both groups work on every page, on row halves of
//    RK = 16 NT rows (32 rows: an 8-token draft tree over a GQA group of 4).
// With F8 (FOLD with an FP8 side cache) a far piece's QK^T is an f16 MMA:
// E4M3 codes widen exactly to f16 pairs, and the k order inside each k-step is
// permuted so that a thread's A elements are whole bytes of its own span of
// SP = D/4 bytes of the key row: logical k = 2t + j (+ 8 h) of k-step ks is
// dimension SP t + 4 ks + 2 h + j.  The queries take the same order (in f16)
// and the side cache's scale multiplies the scores.  Key rows are 128-byte
// swizzled (d 128) or 64-byte unswizzled (d 64).
template <int D, int NT, bool SPLIT_PAGES, bool F8 = false>
struct MmaEngine {
  static constexpr bool kPairs = false;
  static constexpr bool kPingPong = false;
  static constexpr bool kSideF8 = F8;
  static constexpr bool kFarScaleInQ = !F8;   // F8: the scale goes on the scores
  static_assert(D == 128 || D == 64, "head_dim");
  static constexpr int NCW = 8;
  static constexpr int NCT = NCW * 32;
  static constexpr int RK = SPLIT_PAGES ? 8 * NT : 16 * NT;
  static constexpr int RW = 8 * NT;   // rows per warp
  static constexpr int KS = D / 16;   // k-steps of QK^T, m-tiles of PV
  static_assert(RW <= 16, "merge buffer holds 16 rows per warp");
  uint32_t qf[KS][NT][2];
  float O[KS][NT][4];
  float m[NT][2], l[NT][2];
  float kscale;          // F8: the side cache's scale
  int lane, warp, kb, grp, g, t;

  __device__ __forceinline__ void init() {
    lane = threadIdx.x & 31;
    warp = threadIdx.x >> 5;
    kb = warp & 3;
    grp = warp >> 2;
    g = lane >> 2;
    t = lane & 3;
  }

  __device__ __forceinline__ bool owns(uint32_t n) const {
    return SPLIT_PAGES ? (int)(n & 1u) == grp : true;
  }

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int mt = 0; mt < KS; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 4; ++c) O[mt][nt][c] = 0.f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) { m[nt][cc] = -INFINITY; l[nt][cc] = 0.f; }
  }

  __device__ __forceinline__ void begin(const Smem& s) {
    const int row0 = SPLIT_PAGES ? 0 : grp * RW;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const float* qr = s.q + (row0 + 8 * nt + g) * D + 16 * ks + 2 * t;
        qf[ks][nt][0] = pack_bf16(qr[0], qr[1]);
        qf[ks][nt][1] = pack_bf16(qr[8], qr[9]);
      }
    reset();
  }

  // F8: a far piece's queries in f16, in the permuted k order.
  __device__ __forceinline__ void begin_far(const Smem& s, bool far) {
    if (!far) {
      begin(s);
      return;
    }
    const int row0 = SPLIT_PAGES ? 0 : grp * RW;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const float* qr = s.q + (row0 + 8 * nt + g) * D + (D / 4) * t + 4 * ks;
        qf[ks][nt][0] = pack_f16(qr[0], qr[1]);
        qf[ks][nt][1] = pack_f16(qr[2], qr[3]);
      }
    reset();
  }

  template <bool FK = false>
  __device__ __forceinline__ void page(const Smem& s, uint32_t kbase, uint32_t vbase, int lo, int hi,
                                       int toff) {
    const int key0 = 16 * kb;
    if (hi <= key0 || lo >= key0 + 16) return;
    float S[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int c = 0; c < 4; ++c) S[nt][c] = 0.f;
    if constexpr (FK) {
      // rows key0 + g and key0 + g + 8; bytes SP t .. SP t + SP - 1 (NC chunks)
      constexpr int NC = D / 64;
      uint32_t w[2][NC][4];
#pragma unroll
      for (int rh = 0; rh < 2; ++rh)
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          const int row = key0 + g + 8 * rh;
          const uint32_t ad = D == 128 ? swz_addr(kbase, row, (2 * t + c) * 16)
                                       : kbase + (uint32_t)(row * D + 16 * t);
          asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                       : "=r"(w[rh][c][0]), "=r"(w[rh][c][1]), "=r"(w[rh][c][2]), "=r"(w[rh][c][3])
                       : "r"(ad));
        }
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const uint32_t w0 = w[0][ks >> 2][ks & 3], w1 = w[1][ks >> 2][ks & 3];
        const uint32_t a[4] = {e4m3x2_f16x2(w0 & 0xffffu), e4m3x2_f16x2(w1 & 0xffffu),
                               e4m3x2_f16x2(w0 >> 16), e4m3x2_f16x2(w1 >> 16)};
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_f16(S[nt], a, qf[ks][nt][0], qf[ks][nt][1]);
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 4; ++c) S[nt][c] *= kscale;
    } else {
      const int krow = key0 + (lane & 7) + ((lane >> 3) & 1) * 8;
      const uint32_t ka0 = swz_addr(kbase, krow, (lane >> 4) * 16);   // k-step 0
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        uint32_t a[4];
        ldsm_x4(swz_step(ka0, ks), a);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_bf16(S[nt], a, qf[ks][nt][0], qf[ks][nt][1]);
      }
    }
    if (toff != kNoTree) {   // draft-tree keys a row does not see
      const int row0 = SPLIT_PAGES ? 0 : grp * RW;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const uint64_t m = s.tmask[row0 + 8 * nt + 2 * t + cc];
          if (!tree_visible(key0 + g, toff, m)) S[nt][cc] = -INFINITY;
          if (!tree_visible(key0 + g + 8, toff, m)) S[nt][cc + 2] = -INFINITY;
        }
    }
    const bool oka = (key0 + g >= lo) && (key0 + g < hi);
    const bool okb = (key0 + g + 8 >= lo) && (key0 + g + 8 < hi);
    float alpha[NT][2];
    uint32_t bp[NT][2];
    bool all_one = true;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float P[4];
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const float v0 = oka ? S[nt][cc] : -INFINITY;
        const float v1 = okb ? S[nt][cc + 2] : -INFINITY;
        float mx = fmaxf(v0, v1);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float mn = fmaxf(m[nt][cc], mx);
        float al = 1.f, p0 = 0.f, p1 = 0.f;
        if (mn != -INFINITY) {
          al = fast_exp2(m[nt][cc] - mn);
          p0 = fast_exp2(v0 - mn);
          p1 = fast_exp2(v1 - mn);
        }
        l[nt][cc] = l[nt][cc] * al + p0 + p1;
        m[nt][cc] = mn;
        alpha[nt][cc] = al;
        all_one &= (al == 1.f);
        P[cc] = p0;
        P[cc + 2] = p1;
      }
      bp[nt][0] = movm_t(pack_bf16(P[0], P[1]));
      bp[nt][1] = movm_t(pack_bf16(P[2], P[3]));
    }
    if (!__all_sync(0xffffffffu, all_one)) {
#pragma unroll
      for (int mt = 0; mt < KS; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          O[mt][nt][0] *= alpha[nt][0];
          O[mt][nt][1] *= alpha[nt][1];
          O[mt][nt][2] *= alpha[nt][0];
          O[mt][nt][3] *= alpha[nt][1];
        }
    }
    // Keys outside [lo, hi) may hold anything (NaN included): zero their V.
    uint32_t mask01 = 0xffffffffu, mask23 = 0xffffffffu;
    if (lo > key0 || hi < key0 + 16) {
      const int k2 = key0 + 2 * t;
      auto ok = [&](int k) { return k >= lo && k < hi; };
      mask01 = (ok(k2) ? 0x0000ffffu : 0u) | (ok(k2 + 1) ? 0xffff0000u : 0u);
      mask23 = (ok(k2 + 8) ? 0x0000ffffu : 0u) | (ok(k2 + 9) ? 0xffff0000u : 0u);
    }
    const int vrow = key0 + (lane & 7) + (lane >> 4) * 8;
    const uint32_t va0 = swz_addr(vbase, vrow, ((lane >> 3) & 1) * 16);   // m-tile 0
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
      uint32_t a[4];
      ldsm_x4_t(swz_step(va0, mt), a);
      a[0] &= mask01; a[1] &= mask01; a[2] &= mask23; a[3] &= mask23;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma_bf16(O[mt][nt], a, bp[nt][0], bp[nt][1]);
    }
  }

  // Merge the warps holding each row and write the piece's partial to `slot`.
  // part: where the piece's partial (m[RK], l[RK], pad, o[RK][D]) goes (global or shared).
  __device__ __forceinline__ void finish(const Smem& s, const PartOut& part) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        float lt = l[nt][cc];
        lt += __shfl_xor_sync(0xffffffffu, lt, 4);
        lt += __shfl_xor_sync(0xffffffffu, lt, 8);
        lt += __shfl_xor_sync(0xffffffffu, lt, 16);
        if (g == 0) s.ml[warp * 16 + 8 * nt + 2 * t + cc] = make_float2(m[nt][cc], lt);
      }
#pragma unroll
    for (int mt = 0; mt < KS; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int lr = 8 * nt + 2 * t;
        float* base = s.mo + (warp * 16) * D + 16 * mt + g;
        base[lr * D] = O[mt][nt][0];
        base[(lr + 1) * D] = O[mt][nt][1];
        base[lr * D + 8] = O[mt][nt][2];
        base[(lr + 1) * D + 8] = O[mt][nt][3];
      }
    named_barrier(1, NCT);
    constexpr int NW = SPLIT_PAGES ? 8 : 4;   // warps holding one row
    for (int idx = threadIdx.x; idx < RK * D / 4; idx += NCT) {
      const int r = idx / (D / 4), d4 = idx - r * (D / 4);
      const int w0 = SPLIT_PAGES ? 0 : (r / RW) * 4;
      const int lr = SPLIT_PAGES ? r : r % RW;
      float M = -INFINITY;
#pragma unroll
      for (int k = 0; k < NW; ++k) M = fmaxf(M, s.ml[(w0 + k) * 16 + lr].x);
      float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
      float lsum = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int k = 0; k < NW; ++k) {
          const int w = w0 + k;
          const float2 ml = s.ml[w * 16 + lr];
          const float sc = fast_exp2(ml.x - M);
          const float4 v = *reinterpret_cast<const float4*>(s.mo + (w * 16 + lr) * D + 4 * d4);
          o.x = fmaf(sc, v.x, o.x);
          o.y = fmaf(sc, v.y, o.y);
          o.z = fmaf(sc, v.z, o.z);
          o.w = fmaf(sc, v.w, o.w);
          lsum = fmaf(sc, ml.y, lsum);
        }
      }
      part.put4(slot_o_off(RK) + r * D + 4 * d4, o);
      if (d4 == 0) {
        part.put1(r, M);
        part.put1(RK + r, lsum);
      }
    }
    named_barrier(1, NCT);
    reset();
  }
};

// ---------------------------------------------------------------------------
// Split merge, fused into the decode kernel.  Every piece adds its page count
// to cnt[b, h]; the CTA whose addition completes the (b, h) total (all ranges)
// is the last writer, and merges all pieces' partials: per softmax segment a
// log-sum-exp merge, then for FOLD the far/local mix
// (1 - lambda_eff) o_loc + lambda_eff o_far with lambda_eff = 0 when the far
// memory is empty ("FOLD", abstract: the far memory's total weight is
// controlled separately).  No CTA ever waits for another.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int32_t seq_pages(const int32_t* pfx, int b) {
  return pfx[b + 1] - pfx[b];
}

// Running log-sum-exp merge state of one row and four dimensions.
struct MergeState {
  float m, l, o[4];
  __device__ __forceinline__ void init() {
    m = -INFINITY;
    l = 0.f;
    o[0] = o[1] = o[2] = o[3] = 0.f;
  }
  __device__ __forceinline__ void add(float pm, float pl, const float4& po) {
    if (pm == -INFINITY) return;
    const float mn = fmaxf(m, pm);
    const float so = fast_exp2(m - mn), sn = fast_exp2(pm - mn);   // so = 0 when m = -inf
    l = l * so + pl * sn;
    o[0] = o[0] * so + po.x * sn;
    o[1] = o[1] * so + po.y * sn;
    o[2] = o[2] * so + po.z * sn;
    o[3] = o[3] * so + po.w * sn;
    m = mn;
  }
  __device__ __forceinline__ void add(const MergeState& b) {
    add(b.m, b.l, make_float4(b.o[0], b.o[1], b.o[2], b.o[3]));
  }
  // Merge with the state of lane (lane ^ mask).
  __device__ __forceinline__ void add_xor(int mask) {
    MergeState b;
    b.m = __shfl_xor_sync(0xffffffffu, m, mask);
    b.l = __shfl_xor_sync(0xffffffffu, l, mask);
#pragma unroll
    for (int k = 0; k < 4; ++k) b.o[k] = __shfl_xor_sync(0xffffffffu, o[k], mask);
    add(b);
  }
};

// Folds the partials of pieces i0 .. i1 (every `step`-th, starting at i0) of
// one range into st; eight pieces' loads are in flight at a time.
template <int D, int RK>
__device__ __forceinline__ void merge_range(const DecodeArgs& a, int64_t i0, int64_t i1,
                                            int step, int64_t sq, int64_t TP, int64_t n_act,
                                            bool dense, int r, int c4, MergeState& st) {
  constexpr int64_t SF = slot_floats(RK, D);
  for (int64_t i = i0; i <= i1; i += 8 * step) {
    float mm[8], ll[8];
    float4 oo[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int64_t ii = i + (int64_t)u * step;
      mm[u] = -INFINITY;
      ll[u] = 0.f;
      oo[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (ii <= i1 && (dense || cta_begin(ii, TP, n_act) < cta_begin(ii + 1, TP, n_act))) {
        const float* base = a.part + (ii + sq) * SF;
        mm[u] = __ldcg(base + r);
        ll[u] = __ldcg(base + RK + r);
        oo[u] = __ldcg(reinterpret_cast<const float4*>(base + slot_o_off(RK) + r * D) + c4);
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) st.add(mm[u], ll[u], oo[u]);
  }
}

template <typename T>
__device__ __forceinline__ void store4(T* p, const float (&v)[4]);
template <>
__device__ __forceinline__ void store4<float>(float* p, const float (&v)[4]) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* p, const float (&v)[4]) {
  uint2 w;
  w.x = pack_bf16(v[0], v[1]);
  w.y = pack_bf16(v[2], v[3]);
  *reinterpret_cast<uint2*>(p) = w;
}

// Merge of every piece of (b, h).  Work items are (row, 4 dimensions); when
// there are fewer items than consumer threads, SPLIT adjacent lanes share an
// item, each folding every SPLIT-th piece, and combine by shuffles.
template <typename T, int D, int RK, int NCT>
__device__ inline void merge_sequence(const DecodeArgs& a, const Smem& s, int b, int h) {
  constexpr int C4 = D / 4;
  constexpr int ITEMS = RK * C4;
  constexpr int SPLIT = ITEMS >= NCT ? 1 : NCT / ITEMS;
  static_assert(SPLIT <= 32 && (SPLIT & (SPLIT - 1)) == 0, "split");
  const int64_t TP = (int64_t)s.pfx[a.B] * a.H_kv;
  const int64_t n_act = active_ctas(TP, a.n_cta, a.min_pages);
  const bool dense = TP >= n_act;            // then no CTA's stretch is empty
  const bool fold = a.mode == DA_MODE_FOLD;
  // Pieces of (b, h): FOLD keeps the far range (seq even) and the local range
  // (seq odd) apart; every other mode has one segment over the head's line.
  const int32_t nb = s.pfx[b + 1] - s.pfx[b];
  const int32_t n0 = fold ? s.n0[b] : nb;
  const int64_t x0 = (int64_t)s.pfx[b] * a.H_kv + (int64_t)h * nb;
  const int64_t seq0 = ((int64_t)b * a.H_kv + h) * 2;
  int64_t i0[2], i1[2], sq[2];
  const int64_t beg[2] = {x0, x0 + n0}, len[2] = {n0, nb - n0};
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    sq[rr] = seq0 + rr;
    if (len[rr] == 0) {
      i0[rr] = 0;
      i1[rr] = -1;
    } else {
      i0[rr] = cta_of(beg[rr], TP, n_act);
      i1[rr] = cta_of(beg[rr] + len[rr] - 1, TP, n_act);
    }
  }
  const float lam = (fold && n0 > 0) ? a.far_mix : 0.f;
  const int sub = threadIdx.x & (SPLIT - 1);
  for (int item = threadIdx.x / SPLIT; item < a.R * C4; item += NCT / SPLIT) {
    const int r = item / C4, c4 = item - r * C4;
    // s0: FOLD far memory, or the whole selection; s1: FOLD local window
    MergeState s0, s1;
    s0.init();
    s1.init();
    merge_range<D, RK>(a, i0[0] + sub, i1[0], SPLIT, sq[0], TP, n_act, dense, r, c4, s0);
    merge_range<D, RK>(a, i0[1] + sub, i1[1], SPLIT, sq[1], TP, n_act, dense, r, c4, s1);
#pragma unroll
    for (int mask = 1; mask < SPLIT; mask <<= 1) {
      s0.add_xor(mask);
      s1.add_xor(mask);
    }
    float res[4];
    if (fold) {
      // (1 - lambda_eff) o_loc + lambda_eff o_far ("FOLD", abstract)
#pragma unroll
      for (int k = 0; k < 4; ++k)
        res[k] = (s1.l > 0.f ? (1.f - lam) * s1.o[k] / s1.l : 0.f) +
                 (s0.l > 0.f ? lam * s0.o[k] / s0.l : 0.f);
    } else {
      s1.add(s0);                            // one softmax over both ranges
#pragma unroll
      for (int k = 0; k < 4; ++k) res[k] = s1.l > 0.f ? s1.o[k] / s1.l : 0.f;
    }
    if (sub == 0) {
      const int t = r / a.G, j = r - t * a.G;
      T* out = static_cast<T*>(a.out) + ((int64_t)(b * a.n_q + t) * a.H_q + h * a.G + j) * D + 4 * c4;
      store4<T>(out, res);
    }
  }
}

// After a piece's partial is written: take the ticket, merge when last.
template <typename T, int D, int RK, int NCT>
__device__ inline void ticket(const DecodeArgs& a, Smem& s, int seq, uint32_t pages) {
  const int bh = seq >> 1, b = bh / a.H_kv, h = bh - b * a.H_kv;
  uint32_t* c = a.cnt + (int64_t)bh;
  if (threadIdx.x == 0) {
    // Release: the partial the consumers wrote before the barrier in finish()
    // is visible before the count; acquire: when last, every other piece's
    // partial is visible to this CTA (its threads read after the barrier).
    const uint32_t total = (uint32_t)seq_pages(s.pfx, b);
    const uint32_t old = atom_add_acq_rel_gpu(c, pages);
    const int last = old + pages == total;
    if (last) atomicExch(c, 0u);  // every piece of (b, h) has arrived: ready for the next call
    s.flag[0] = last;
  }
  named_barrier(1, NCT);
  const int last = s.flag[0];
  named_barrier(1, NCT);
  if (last) merge_sequence<T, D, RK, NCT>(a, s, b, h);
}

// Cluster partition: merge of the partials the cluster's CTAs hold in their
// shared memory (at the same offset `local` in each), read through
// distributed shared memory.  Work items are (row, 4 dimensions), spread
// over the cluster's consumer threads; each loads every CTA's (m, l, o)
// before it merges, so the remote loads are in flight together.
template <typename T, int D, int RK, int NCT>
__device__ inline void cluster_merge(const DecodeArgs& a, int b, int h, uint32_t local) {
  constexpr int C4 = D / 4;
  constexpr int kMaxCluster = 16;
  const uint32_t cn = cluster_size(), cr = cluster_rank();
  uint32_t src[kMaxCluster];
#pragma unroll
  for (int k = 0; k < kMaxCluster; ++k) src[k] = dsmem_addr(local, (uint32_t)k < cn ? k : 0);
  for (int item = threadIdx.x * (int)cn + (int)cr; item < a.R * C4; item += NCT * (int)cn) {
    const int r = item / C4, c4 = item - r * C4;
    float mm[kMaxCluster], ll[kMaxCluster];
    float4 oo[kMaxCluster];
#pragma unroll
    for (int k = 0; k < kMaxCluster; ++k) {
      mm[k] = -INFINITY;
      ll[k] = 0.f;
      oo[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      if ((uint32_t)k < cn) {
        mm[k] = dsmem_ld_f32(src[k] + 4u * r);
        ll[k] = dsmem_ld_f32(src[k] + 4u * (RK + r));
        oo[k] = dsmem_ld_f32x4(src[k] + 4u * (slot_o_off(RK) + r * D + 4 * c4));
      }
    }
    MergeState st;
    st.init();
#pragma unroll
    for (int k = 0; k < kMaxCluster; ++k) st.add(mm[k], ll[k], oo[k]);
    float res[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) res[k] = st.l > 0.f ? st.o[k] / st.l : 0.f;
    const int t = r / a.G, j = r - t * a.G;
    T* out = static_cast<T*>(a.out) + ((int64_t)(b * a.n_q + t) * a.H_q + h * a.G + j) * D + 4 * c4;
    store4<T>(out, res);
  }
}

// Cluster partition, rank 0: merge of the partials every CTA of the cluster
// stored into this CTA's receive slots.  Work items are (row, 4 dimensions).
// The largest slot maximum is found first, so that the C slots' weights are
// independent and their sums form short chains instead of one dependent
// rescale after another.
template <typename T, int D, int RK, int NCT>
__device__ inline void recv_merge(const DecodeArgs& a, const Smem& s, int b, int h) {
  constexpr int C4 = D / 4;
  constexpr int SF = slot_floats(RK, D);
  constexpr int kMaxCluster = 16;
  const int cn = (int)cluster_size();
  for (int item = threadIdx.x; item < a.R * C4; item += NCT) {
    const int r = item / C4, c4 = item - r * C4;
    float mk[kMaxCluster];
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < kMaxCluster; ++k) {
      mk[k] = k < cn ? s.recv[k * SF + r] : -INFINITY;
      M = fmaxf(M, mk[k]);
    }
    float l = 0.f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY) {
#pragma unroll
      for (int k = 0; k < kMaxCluster; ++k) {
        if (k < cn && mk[k] != -INFINITY) {
          const float* slot = s.recv + k * SF;
          const float w = fast_exp2(mk[k] - M);
          const float4 v = *reinterpret_cast<const float4*>(slot + slot_o_off(RK) + r * D + 4 * c4);
          l = fmaf(w, slot[RK + r], l);
          o.x = fmaf(w, v.x, o.x);
          o.y = fmaf(w, v.y, o.y);
          o.z = fmaf(w, v.z, o.z);
          o.w = fmaf(w, v.w, o.w);
        }
      }
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const float res[4] = {o.x * inv, o.y * inv, o.z * inv, o.w * inv};
    const int t = r / a.G, j = r - t * a.G;
    T* out = static_cast<T*>(a.out) + ((int64_t)(b * a.n_q + t) * a.H_q + h * a.G + j) * D + 4 * c4;
    store4<T>(out, res);
  }
}

// Cluster partition, before the wait for the predecessor: L2 prefetches of
// the small inputs this CTA reads first (its sequence's context length, new
// positions and query positions, its KV head's query rows and new tokens).
// A prefetch returns nothing to the SM and L2 is the point of coherence, so
// the loads after the wait still see the predecessor's writes; they only
// find the lines closer.  One warp.
template <typename T, int D>
__device__ inline void prefetch_head_inputs(const DecodeArgs& a, int b, int h) {
  const int lane = threadIdx.x & 31;
  const char* const q = static_cast<const char*>(a.q);
  constexpr int ROWB = D * (int)sizeof(T);
  const int qlines = a.n_q * ((a.G * ROWB + 127) / 128);
  for (int i = lane; i < qlines; i += 32) {
    const int t = i / ((a.G * ROWB + 127) / 128), l = i - t * ((a.G * ROWB + 127) / 128);
    prefetch_l2(q + ((int64_t)(b * a.n_q + t) * a.H_q + h * a.G) * ROWB + l * 128);
  }
  if (a.n_new > 0) {
    const int nl = 2 * a.n_new * ((ROWB + 127) / 128);
    for (int i = lane; i < nl; i += 32) {
      const int kv = i & 1, rest = i >> 1;
      const int j = rest / ((ROWB + 127) / 128), l = rest - j * ((ROWB + 127) / 128);
      const char* src = static_cast<const char*>(kv ? a.v_new : a.k_new);
      prefetch_l2(src + ((int64_t)(b * a.n_new + j) * a.H_kv + h) * ROWB + l * 128);
    }
  }
  if (lane == 0) {
    prefetch_l2(a.ctx_lens + b);
    prefetch_l2(a.q_pos + (int64_t)b * a.n_q);
    if (a.n_new > 0) prefetch_l2(a.new_pos + (int64_t)b * a.n_new);
  }
}

// ---------------------------------------------------------------------------
// One launch per draft step (cluster partition): the step's new tokens are
// appended by the attention kernel itself.  A spare warp of every CTA writes
// its share of the new keys (rotated at their positions) and values of the
// cluster's (sequence, KV head) to the caches, as the append kernel would;
// the pages this step reads that hold a new token are loaded from the cache
// as they were and have the token's rows replaced in shared memory, from a
// copy the consumers computed at the start with the same arithmetic.  Keys
// and values are therefore bit-identical to an append followed by the call.
// ---------------------------------------------------------------------------
template <typename T, int D>
__device__ inline void fused_append(const DecodeArgs& a, const Smem& s, int b, int h, uint32_t cr,
                                    uint32_t cn) {
  const int lane = threadIdx.x & 31;
  for (int j = (int)cr; j < a.n_new; j += (int)cn) {
    const int32_t pos = s.newpos[j];
    if (pos < 0) continue;                          // padding
    const int32_t pg = pos / kPage;
    if (pg >= a.max_pages) {
      if (lane == 0) atomicOr(a.status, DA_STATUS_BAD_POSITION);
      continue;
    }
    const int32_t phys = __ldg(a.block_table + (int64_t)b * a.max_pages + pg);
    if (phys < 0 || phys >= a.num_pages) {
      if (lane == 0) atomicOr(a.status, DA_STATUS_BAD_PAGE);
      continue;
    }
    const int64_t src = ((int64_t)(b * a.n_new + j) * a.H_kv + h) * D;
    const int64_t dst = (((int64_t)phys * a.H_kv + h) * kPage + (pos - pg * kPage)) * D;
    const T* k = static_cast<const T*>(a.k_new) + src;
    const T* v = static_cast<const T*>(a.v_new) + src;
    T* kc = static_cast<T*>(a.k_cache_w) + dst;
    T* vc = static_cast<T*>(a.v_cache_w) + dst;
#pragma unroll
    for (int u = 0; u < D / 64; ++u) {
      const int f = lane + 32 * u;
      float c, sn, xr, yr;
      rope_cos_sin(pos, s.invf[f], c, sn);
      rope_pair(to_f32<T>(k[f]), to_f32<T>(k[f + D / 2]), c, sn, xr, yr);
      kc[f] = from_f32<T>(xr);
      kc[f + D / 2] = from_f32<T>(yr);
      vc[f] = v[f];
      vc[f + D / 2] = v[f + D / 2];
    }
  }
}

// Consumers: the rotated key and the value of every new token of sequence b,
// KV head h, into s.newkv (one consumer warp per token).
template <typename T, int D>
__device__ inline void stage_new_tokens(const DecodeArgs& a, const Smem& s, int b, int h) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp < a.n_new) {
    const int32_t pos = s.newpos[warp];
    if (pos >= 0) {
      const int64_t src = ((int64_t)(b * a.n_new + warp) * a.H_kv + h) * D;
      const T* k = static_cast<const T*>(a.k_new) + src;
      const T* v = static_cast<const T*>(a.v_new) + src;
      T* dk = reinterpret_cast<T*>(s.newkv) + (size_t)warp * 2 * D;
      T* dv = dk + D;
#pragma unroll
      for (int u = 0; u < D / 64; ++u) {
        const int f = lane + 32 * u;
        float c, sn, xr, yr;
        rope_cos_sin(pos, s.invf[f], c, sn);
        rope_pair(to_f32<T>(k[f]), to_f32<T>(k[f + D / 2]), c, sn, xr, yr);
        dk[f] = from_f32<T>(xr);
        dk[f + D / 2] = from_f32<T>(yr);
        dv[f] = v[f];
        dv[f + D / 2] = v[f + D / 2];
      }
    }
  }
  named_barrier(1, kConsumerThreads);
}

// Consumers, after stage st landed: the new tokens it holds replace their
// rows of the staged keys and values (128-byte swizzled boxes); every
// consumer thread reads the same mask, so the barrier is met by all or none.
template <typename T, int D, int NCT>
__device__ inline void patch_new_tokens(const Smem& s, const Layout& L, uint32_t st) {
  const uint32_t nm = s.pnew[st];
  if (nm == 0) return;
  constexpr int ROWB = D * (int)sizeof(T);       // bytes of one key or value row
  constexpr int NCB = ROWB / kSwizzleRow;        // 128-byte boxes per row
  constexpr int CPR = ROWB / 16;                 // 16-byte chunks per row
  if (threadIdx.x < 32) {
    uint8_t* kst = s.stage + st * L.stage_bytes;
    uint8_t* vst = kst + NCB * kBoxBytes;
    uint32_t m = nm;
    while (m) {
      const int j = __ffs(m) - 1;
      m &= m - 1;
      const int slot = s.newpos[j] & (kPage - 1);
      const uint8_t* src = s.newkv + (size_t)j * 2 * ROWB;
      for (int c = threadIdx.x; c < 2 * CPR; c += 32) {
        const int kv = c / CPR, cc = c - kv * CPR;
        const int box = cc >> 3, ch16 = cc & 7;
        uint8_t* dst = (kv ? vst : kst) + box * kBoxBytes + slot * kSwizzleRow +
                       ((ch16 ^ (slot & 7)) << 4);
        *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src + kv * ROWB + cc * 16);
      }
    }
  }
  named_barrier(1, NCT);
}

// Rows of (b, h) whose selection is empty get a zero output (nobody merges
// them); CTA (b * H_kv + h) mod n_cta writes it.
template <typename T, int D, int NCT>
__device__ inline void zero_empty(const DecodeArgs& a, const Smem& s) {
  for (int bh = blockIdx.x; bh < a.B * a.H_kv; bh += a.n_cta) {
    const int b = bh / a.H_kv, h = bh - b * a.H_kv;
    if (seq_pages(s.pfx, b) != 0) continue;
    for (int idx = threadIdx.x; idx < a.R * D; idx += NCT) {
      const int r = idx / D, dim = idx - r * D;
      const int t = r / a.G, j = r - t * a.G;
      static_cast<T*>(a.out)[((int64_t)(b * a.n_q + t) * a.H_q + h * a.G + j) * D + dim] =
          from_f32<T>(0.f);
    }
  }
}

// ---------------------------------------------------------------------------
// The kernel.
// ---------------------------------------------------------------------------
//
// Two partitions of the work:
//  * flat (CLUSTER false): one persistent CTA per SM takes an equal stretch
//    of the page line of every (sequence, KV head, range); pieces leave
//    partials in the workspace and the last CTA of each (sequence, KV head)
//    merges them (ticket, merge_sequence).
//  * cluster (CLUSTER true; one-segment modes whose selection is short, such
//    as window mode): one thread-block cluster of a.cluster CTAs per
//    (sequence, KV head).  CTA r of the cluster takes an equal r-th share of
//    that head's pages (one piece) and sends its partial into slot r of rank
//    0's shared memory by asynchronous stores that complete rank 0's merge
//    barrier by their byte count; rank 0 merges the slots and writes the
//    output: no workspace round trip and no ticket.
template <typename T, int D, class Engine, int VARIANT, int RK, bool CLUSTER = false>
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ DecodeArgs a, const __grid_constant__ CUtensorMap mk,
                  const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap ms,
                  int stages) {
  extern __shared__ uint8_t smem_raw[];
  constexpr int ES = sizeof(T);
  constexpr int NCB = D * ES / kSwizzleRow;
  constexpr int NCW = Engine::NCW;
  constexpr int NCT = NCW * 32;
  static_assert(NCW == kConsumerWarps, "consumer warps");
  static_assert(!CLUSTER || !Engine::kPingPong, "cluster partition: shared-step engines");
  static_assert(!CLUSTER || slot_floats(RK, D) * 4 <= 2 * (D * ES / kSwizzleRow) * kBoxBytes,
                "the partial fits in one pipeline stage");
  const Layout L = make_layout(VARIANT, ES, D, RK, stages, a.B, CLUSTER ? a.cluster : 0);
  Smem s = carve(smem_raw, L);
  int64_t xs, xe;
  int cb = 0, ch = 0;   // cluster partition: the cluster's (sequence, KV head)
  uint32_t cr = 0;      // and this CTA's rank in it
  int32_t Lb = 0;
  if constexpr (CLUSTER) {
    // No page prefix: the CTA knows its (sequence, KV head) from its cluster
    // and its pages from that one context length, read by every thread (the
    // load is issued first, so that its latency overlaps the set-up).
    cr = cluster_rank();
    const uint32_t cn = cluster_size();
    const int bh = (int)(blockIdx.x / cn);
    cb = bh / a.H_kv;
    ch = bh - cb * a.H_kv;
    // Inputs known to be ready (all but the caches behind this library's
    // append kernel; the context lengths, positions and block table when the
    // caller sets tables_ready) are read at once; otherwise the set-up overlaps
    // the predecessor's tail and every global access waits for it.
    const bool early = a.inputs_ready || a.tables_ready;
    int32_t Lraw = early ? __ldg(a.ctx_lens + cb) : 0;
    int32_t npos = 0;
    if (early && threadIdx.x < a.n_new) npos = __ldg(a.new_pos + cb * a.n_new + threadIdx.x);
    if (!a.inputs_ready && threadIdx.x < 32) prefetch_head_inputs<T, D>(a, cb, ch);
    cluster_start<D, NCW>(a, s, L);
    if (!early) {
      grid_dep_wait();
      Lraw = __ldg(a.ctx_lens + cb);
      if (threadIdx.x < a.n_new) npos = __ldg(a.new_pos + cb * a.n_new + threadIdx.x);
    }
    if (a.n_new > 0) {   // one launch for the draft step: the new tokens' positions
      if (threadIdx.x < a.n_new) s.newpos[threadIdx.x] = npos;
      __syncthreads();
    }
    Lb = clamp_ctx(Lraw, a.max_pages, a.status);
    s.len[cb] = Lb;   // query preparation reads it (every thread writes the same value)
    const Ranges rg = mode_ranges(a.mode, Lb, a.W, a.n_sink);
    const int64_t nb = range_pages(rg.k0[0], rg.k1[0]) + range_pages(rg.k0[1], rg.k1[1]) +
                       range_pages(rg.k0[2], rg.k1[2]);
    xs = nb * cr / cn;
    xe = nb * (cr + 1) / cn;
  } else {
    prologue<D, ES, NCW>(a, s, L);
    const int64_t TP = (int64_t)s.pfx[a.B] * a.H_kv;
    const int64_t n_act = active_ctas(TP, a.n_cta, a.min_pages);
    xs = blockIdx.x < n_act ? cta_begin(blockIdx.x, TP, n_act) : 0;
    xe = blockIdx.x < n_act ? cta_begin(blockIdx.x + 1, TP, n_act) : 0;
  }
  const int warp = threadIdx.x >> 5;
  if (warp >= NCW) {
    regs_dec<kProducerRegs>();
    if (warp == NCW) {
      if constexpr (CLUSTER)
        producer_head<ES, NCB, Engine::kSideF8>(a, s, L, cb, ch, Lb, xs, xe, &mk, &mv, &ms);
      else
        producer<ES, NCB, Engine::kSideF8>(a, s, L, xs, xe, &mk, &mv, &ms);
    } else if (CLUSTER && warp == NCW + 1 && a.n_new > 0) {
      if (a.tables_ready && !a.inputs_ready) grid_dep_wait();   // before the caches are written
      fused_append<T, D>(a, s, cb, ch, cr, cluster_size());
    }
    return;   // arrived at the cluster barrier in cluster_start; nothing to wait for
  }
  regs_inc<kConsumerRegs>();
  Engine eng;
  eng.init();
  if constexpr (!Engine::kFarScaleInQ) eng.kscale = a.far_kscale;
  // tables read early: the queries, masks, new tokens, the workspace and the
  // output wait for the previous kernel
  if (a.tables_ready && !a.inputs_ready) grid_dep_wait();
  if constexpr (!CLUSTER) zero_empty<T, D, NCT>(a, s);
  // cluster partition: this CTA's partial goes straight to its slot in rank
  // 0's shared memory, by asynchronous stores counted on rank 0's merge
  // barrier (rank 0 itself stores its own slot directly)
  PartOut cpart{nullptr, 0u, 0u};
  if constexpr (CLUSTER) {
    float* const own = s.recv + (size_t)cr * slot_floats(RK, D);
    if (cr == 0) {
      cpart.p = own;
    } else {
      cpart.sa = dsmem_addr(smem_u32(own), 0u);
      cpart.bar = dsmem_addr(smem_u32(s.merge_bar), 0u);
    }
  }
  bool wrote = false, cwaited = false;
  // A fused draft step: the new tokens' rotated keys and values, for pages
  // that hold them (patched into the staged copy before they are read).
  if constexpr (CLUSTER) {
    if (a.n_new > 0) stage_new_tokens<T, D>(a, s, cb, ch);
  }
  // The first piece's queries are prepared while its first pages load.
  if (xs < xe) {
    int32_t seq;
    if constexpr (CLUSTER) {
      seq = piece_seq(a.mode, cb, ch, a.H_kv, 0);   // one segment (no FOLD here)
    } else {
      const Where w = locate(s, a.B, a.H_kv, xs);
      seq = piece_seq(a.mode, w.b, w.h, a.H_kv, w.r);
    }
    prep_queries<T, D, RK, NCT, Engine::kFarScaleInQ>(a, s, seq);
    if constexpr (Engine::kSideF8) eng.begin_far(s, (seq & 1) == 0); else eng.begin(s);
  }
  const uint32_t base = smem_u32(s.stage);
  uint32_t n = 0, pages = 0;
  uint32_t unit = 0;   // steps taken (a pair or a single page): the ping-pong turn
  const bool long_stretch = !Engine::kPingPong || xe - xs >= 4;
  for (int64_t x = xs; x < xe;) {
    const uint32_t st = n % L.stages;
    if (!mbar_wait(&s.full[st], (n / L.stages) & 1u, a.status, s.abort)) break;
    const PageInfo inf = s.info[st];
    if constexpr (CLUSTER) {
      if (a.n_new > 0) patch_new_tokens<T, D, NCT>(s, L, st);
    }
    if ((inf.flags & kFirst) && x != xs) {
      prep_queries<T, D, RK, NCT, Engine::kFarScaleInQ>(a, s, inf.seq);
      if constexpr (Engine::kSideF8) eng.begin_far(s, (inf.seq & 1) == 0); else eng.begin(s);
    }
    const uint32_t kb0 = base + st * L.stage_bytes;
    const int lo0 = (inf.flags & kValid) ? (inf.lohi & 0xffff) : 0;
    const int hi0 = (inf.flags & kValid) ? (inf.lohi >> 16) : 0;
    const int to0 = inf.toff;
    bool last = (inf.flags & kLast) != 0;
    uint32_t taken = 1;
    if constexpr (Engine::kPairs) {
      // the next page belongs to the same piece unless this one ends it; a
      // short stretch goes page by page, so that both warp groups work
      if (!last && long_stretch) {
        const uint32_t st1 = (n + 1) % L.stages;
        if (!mbar_wait(&s.full[st1], ((n + 1) / L.stages) & 1u, a.status, s.abort)) break;
        const PageInfo inf1 = s.info[st1];
        if constexpr (CLUSTER) {
          if (a.n_new > 0) patch_new_tokens<T, D, NCT>(s, L, st1);
        }
        const uint32_t kb1 = base + st1 * L.stage_bytes;
        const uint32_t kb[2] = {kb0, kb1};
        const uint32_t vb[2] = {kb0 + NCB * kBoxBytes, kb1 + NCB * kBoxBytes};
        const int lo[2] = {lo0, (inf1.flags & kValid) ? (inf1.lohi & 0xffff) : 0};
        const int hi[2] = {hi0, (inf1.flags & kValid) ? (inf1.lohi >> 16) : 0};
        const int to[2] = {to0, inf1.toff};
        if (eng.owns(unit)) {
          if constexpr (Engine::kPingPong && sizeof(T) == 4) {   // fp32: a step per page
            const uint32_t k1[1] = {kb[0]}, v1[1] = {vb[0]}, k2[1] = {kb[1]}, v2[1] = {vb[1]};
            const int l1[1] = {lo[0]}, h1[1] = {hi[0]}, t1[1] = {to[0]};
            const int l2[1] = {lo[1]}, h2[1] = {hi[1]}, t2[1] = {to[1]};
            eng.template pages<1>(s, k1, v1, l1, h1, t1);
            eng.template pages<1>(s, k2, v2, l2, h2, t2);
          } else if constexpr (Engine::kSideF8) {   // FOLD: seq even = far memory
            if ((inf.seq & 1) == 0) eng.template pages<2, true>(s, kb, vb, lo, hi, to);
            else eng.template pages<2>(s, kb, vb, lo, hi, to);
          } else {
            eng.template pages<2>(s, kb, vb, lo, hi, to);
          }
        }
        __syncwarp();
        if ((threadIdx.x & 31) == 0) {
          mbar_arrive(&s.empty[st]);
          mbar_arrive(&s.empty[st1]);
        }
        taken = 2;
        last = (inf1.flags & kLast) != 0;
      }
    }
    if (taken == 1) {
      const bool mine = Engine::kPingPong ? eng.owns(unit) : eng.owns(n);
      if (hi0 > lo0 && mine) {
        if constexpr (Engine::kSideF8) {
          if ((inf.seq & 1) == 0) eng.template page<true>(s, kb0, kb0 + NCB * kBoxBytes, lo0, hi0, to0);
          else eng.page(s, kb0, kb0 + NCB * kBoxBytes, lo0, hi0, to0);
        } else {
          eng.page(s, kb0, kb0 + NCB * kBoxBytes, lo0, hi0, to0);
        }
      }
      __syncwarp();
      if ((threadIdx.x & 31) == 0) mbar_arrive(&s.empty[st]);
    }
    pages += taken;
    x += taken;
    n += taken;
    ++unit;
    if (last) {
      if constexpr (CLUSTER) {
        // rank 0 initialised its merge barrier before its cluster arrival
        cluster_wait();
        cwaited = true;
        eng.finish(s, cpart);   // the CTA's one piece
        wrote = true;
      } else {
        eng.finish(s, PartOut{a.part + ((int64_t)blockIdx.x + inf.seq) * slot_floats(RK, D), 0u, 0u});
        ticket<T, D, RK, NCT>(a, s, inf.seq, pages);
      }
      pages = 0;
    }
  }
  // The producer warp waits for this before it exits (it lets its copies
  // land first when a wait gave up).
  named_barrier_arrive(kEndBarrier, NCT + 32);
  if constexpr (CLUSTER) {
    if (!cwaited) cluster_wait();
    // A CTA with no pages (a selection shorter than the cluster) or whose wait
    // gave up before its piece's end sends an empty partial, so that every
    // CTA but rank 0 sends part_bytes to rank 0's barrier.
    if (!wrote) {
      for (int i = threadIdx.x; i < RK * D / 4; i += NCT)
        cpart.put4(slot_o_off(RK) + 4 * i, make_float4(0.f, 0.f, 0.f, 0.f));
      for (int r = threadIdx.x; r < RK; r += NCT) {
        cpart.put1(r, -INFINITY);
        cpart.put1(RK + r, 0.f);
      }
    }
    // Rank 0 expects the other CTAs' bytes on its merge barrier (a single
    // arrival) and merges once they have landed and its own consumers have
    // written its slot.  The other CTAs are done: nothing reads their shared
    // memory, and their stores carry registers, not shared memory.
    if (cr == 0) {
      if (threadIdx.x == 0) mbar_arrive_expect_tx(s.merge_bar, (cluster_size() - 1) * part_bytes(RK, D));
      named_barrier(1, NCT);
      if (mbar_wait_cluster(s.merge_bar, 0u, a.status, s.abort)) recv_merge<T, D, RK, NCT>(a, s, cb, ch);
    }
  }
}

}  // namespace da
