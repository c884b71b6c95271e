/*
 * draft_attn.h -- C ABI of the speculative-draft decode attention library.
 *
 * One data-parallel hot path: the attention of an MTP/NEXTN-style draft head
 * over a long, paged KV cache, in four modes:
 *
 *   DA_MODE_FULL    every key of the context (the "full-context draft-KV tax").
 *                   "Windowed-MTP: Removing the Full-Context Draft-KV Tax at
 *                   Million-Token Context", Abstract.
 *   DA_MODE_WINDOW  the last W keys plus the first n_sink keys (attention
 *                   sinks), so the draft's KV read stops growing with context.
 *                   Same page, Abstract.
 *   DA_MODE_FOLD    two softmaxes: the last W keys at their exact RoPE
 *                   positions, and every older key as far memory, read from
 *                   an unrotated side cache and rotated at one shared position
 *                   P_far = L - W - 1, its logits sharpened by alpha; the two
 *                   are mixed as (1 - far_mix) * local + far_mix * far
 *                   (far_mix counts only when the far memory is non-empty).
 *                   With n_sink > 0 the first n_sink keys join the local
 *                   softmax at their own positions, as the sinks of window
 *                   mode do, and the far memory starts after them (the
 *                   library's reading: the FOLD page names no sinks).
 *                   "FOLD: Position-Free Far Memory with Local Order for
 *                   Long-Context Speculative Decoding", summary and abstract.
 *   DA_MODE_SHARP   all keys, logits scaled by
 *                   gamma = max(1, 1 + scale_slope * ln(|S| / scale_ref)),
 *                   |S| the number of visible keys.  "SharpDraft: Accelerating
 *                   Long-Context Speculative Decoding with Cardinality-Aware
 *                   Query Scaling", Abstract.  (The page prints no formula;
 *                   this fixed-slope form is the one the library implements.)
 *
 * RoPE is rotate-half (pairs (x_i, x_{i+d/2}), inv_freq_i = theta^(-2i/d)),
 * after "RoFormer: Enhanced Transformer with Rotary Position Embedding", which
 * the Windowed-MTP page lists under "Builds on"; the paged cache follows
 * "Efficient Memory Management for Large Language Model Serving with
 * PagedAttention", listed there too.
 *
 * Layouts (row-major, element type = params.dtype for q, caches and out):
 *   q            [batch][n_q][num_q_heads][head_dim]
 *   out          [batch][n_q][num_q_heads][head_dim]
 *   k_new, v_new [batch][n_new][num_kv_heads][head_dim]
 *   k_cache, v_cache, k_side
 *                [num_pages][num_kv_heads][page_size][head_dim]
 *                k_cache holds keys rotated at their own positions, k_side
 *                the same keys un-rotated (FOLD only), v_cache the values.
 *                With side_fp8 = 1, k_side holds one byte per element: the
 *                FP8 E4M3 code of k / side_scale.  With k_ring_pages = R,
 *                k_cache is [batch * R][num_kv_heads][page_size][head_dim].
 *   block_table  int32 [batch][max_pages_per_seq]; logical page j of sequence
 *                b lives in physical page block_table[b][j].
 *   ctx_lens     int32 [batch]: keys 0 .. ctx_lens[b]-1 are visible.
 *   q_pos        int32 [batch][n_q]: RoPE position of each query token.
 * Query head h reads KV head h / (num_q_heads / num_kv_heads).
 *
 * Ownership: the caller allocates and owns every device buffer (q, caches,
 * block table, lengths, out and the workspace).  The library owns only the
 * opaque host-side plan and one 4-byte device status word per device.  All
 * device work is asynchronous on the given stream; no call allocates device
 * memory, and none synchronises except draft_attn_get_status.  Every pointer
 * argument of the run/append/gather calls is a DEVICE pointer unless stated
 * otherwise.
 *
 * Errors: every call returns DA_OK (0) or a negative DA_ERR_* code; nothing
 * throws or aborts across this ABI.  Faults found on the device (an invalid
 * block-table entry, a context length beyond the block table, a position out
 * of range) never trap: the affected keys are skipped, a bit is set in the
 * device status word, and draft_attn_get_status reports it.
 */
#ifndef DRAFT_ATTN_H
#define DRAFT_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
#define DA_OK                        0
#define DA_ERR_INVALID_ARG          -1  /* null pointer, bad size or parameter   */
#define DA_ERR_UNSUPPORTED          -2  /* valid, but no kernel for this shape   */
#define DA_ERR_WORKSPACE_TOO_SMALL  -3  /* workspace_bytes below the plan's need */
#define DA_ERR_CUDA                 -4  /* a CUDA runtime call or launch failed  */
#define DA_ERR_DEVICE_FAULT         -5  /* the device status word was non-zero   */

/* Device status bits (draft_attn_get_status). */
#define DA_STATUS_BAD_PAGE      1u  /* block-table entry outside [0, num_pages) */
#define DA_STATUS_BAD_CTX_LEN   2u  /* ctx_len < 0 or > max_pages_per_seq*page  */
#define DA_STATUS_BAD_POSITION  4u  /* append position beyond the block table   */
#define DA_STATUS_WAIT_TIMEOUT  8u  /* a pipeline wait gave up (never expected) */

typedef enum { DA_MODE_FULL = 0, DA_MODE_WINDOW = 1, DA_MODE_FOLD = 2, DA_MODE_SHARP = 3 } da_mode;
typedef enum { DA_DTYPE_BF16 = 0, DA_DTYPE_FP32 = 1 } da_dtype;

/* Kernel engines (da_plan_info.engine).  "Rows" are the query rows that share
 * one KV head: (num_q_heads / num_kv_heads) * n_q.  Automatic choice: up to 4
 * rows on the FP32 pipes; 5..32 rows (bf16) on the tensor cores, where the
 * rows fill n8 MMA tiles and QK^T / PV are dense contractions. */
#define DA_ENGINE_CUDA_CORE 0  /* <= 8 rows: FP32 FMA path                        */
#define DA_ENGINE_MMA       1  /* 5..32 rows, bf16: m16n8k16 tensor-core path     */
#define DA_ENGINE_TC05      2  /* <= 32 rows, bf16, head_dim 128: tcgen05 MMAs with
                                  TMEM accumulators (da_params.engine = 3)         */

typedef struct {
  double  rope_theta;        /* RoPE base theta, > 0; 0 = NoPE (no rotation)      */
  int32_t batch;             /* sequences, 1..1024                                 */
  int32_t n_q;               /* query tokens per sequence (draft-tree width)       */
  int32_t num_q_heads;       /* H_q, a multiple of num_kv_heads                    */
  int32_t num_kv_heads;      /* H_kv                                               */
  int32_t head_dim;          /* 64 or 128                                          */
  int32_t page_size;         /* tokens per page; must be 64                        */
  int32_t num_pages;         /* physical pages in each cache array                 */
  int32_t max_pages_per_seq; /* row length of the block table; at most 2^24 /
                                page_size, so every position is below 2^24       */
  int32_t dtype;             /* da_dtype of q, caches and out                      */
  int32_t mode;              /* da_mode                                            */
  int32_t window;            /* W (window, fold), >= 1                             */
  int32_t n_sink;            /* sink tokens (window, fold), >= 0; in FOLD the
                                first n_sink keys stay exact local keys and
                                leave the far memory (not with k_ring_pages)     */
  float   alpha;             /* FOLD far-logit concentration factor, > 0           */
  float   far_mix;           /* FOLD far-memory weight lambda in [0, 1]            */
  float   scale_slope;       /* SharpDraft slope beta, >= 0                        */
  int32_t scale_ref;         /* SharpDraft reference key count N_ref, >= 1         */
  float   softmax_scale;     /* logit scale c; 0 selects 1/sqrt(head_dim)          */
  int32_t num_ctas;          /* persistent CTAs; 0 = one per SM (tests vary this)  */
  int32_t engine;            /* 0 automatic, 1 CUDA cores (<= 8 rows), 2 tensor
                                cores (mma.sync, bf16 only), 3 tcgen05 tensor
                                cores (bf16, head_dim 128, no FP8 side cache);
                                see DA_ENGINE_*                                  */
  int32_t min_pages_per_cta; /* split floor: a call whose selection has P pages
                                (over all sequences and KV heads) runs on
                                min(num_ctas, ceil(P / this)) CTAs; 0 = default
                                (1)                                               */
  int32_t stages;            /* shared-memory pipeline depth in pages, 2..8;
                                0 = as deep as shared memory allows (<= 6 for
                                the CUDA-core engine outside window mode, <= 4
                                otherwise)                                       */
  int32_t tree_size;         /* draft-tree tokens at the end of each context,
                                0..64 (<= window in window and FOLD modes); the
                                per-query masks go to draft_attn_run_tree        */
  int32_t k_ring_pages;      /* FOLD only: 0, or R >= S + ceil(window / 64) + 1,
                                S = ceil(n_sink / 64) the sinks' pages.  The
                                rotated K cache then keeps only the local keys:
                                logical page P of sequence b lives at page
                                b * R + P for P < S, else at b * R + S +
                                ((P - S) mod (R - S)), of k_cache (batch * R
                                pages), while the side cache and the V cache stay
                                paged by the block table.  The far memory reads
                                the side cache only, so the unrotated keys are
                                the one full-length copy of K.  Appends then
                                cover every sequence (batch = params.batch), and
                                one call must not hold two positions of pages
                                >= S that are (R - S) * 64 apart (they would
                                share a slot).  draft_attn_ring_size(window,
                                n_sink) gives the smallest R.                    */
  int32_t side_fp8;          /* FOLD only: 0 = k_side in dtype; 1 = k_side as FP8
                                E4M3 codes (one byte per element) of the float32
                                quotient k / side_scale, rounded to nearest, ties
                                to even, saturating at +-448; the far memory reads
                                code value * side_scale.  Halves the side cache
                                against bf16 (the FOLD page gives no format for
                                it).  Needs bf16.  Runs on the tensor-core
                                engine unless engine = 1 forces the CUDA cores
                                (then at most 4 rows per KV head;
                                DA_ERR_UNSUPPORTED otherwise).                   */
  float   side_scale;        /* > 0 and finite with side_fp8 = 1, else 0           */
  int32_t cluster_ctas;      /* window mode: how the attention kernel splits the
                                work.  0 = automatic: when num_ctas and
                                min_pages_per_cta are 0 and one cluster per
                                (sequence, KV head) fits on the GPU at once, the
                                cluster partition (below): the largest size (up
                                to 16) at which every cluster is resident, cut to
                                the fewest CTAs that keep the most pages any CTA
                                scans the same; else the flat one;
                                -1 = always the flat partition (persistent CTAs
                                take equal stretches of every head's pages and
                                the last CTA of each head merges through the
                                workspace); 1..16 = the cluster partition with
                                that many CTAs per cluster: one thread-block
                                cluster per (sequence, KV head), each CTA an
                                equal share of that head's pages, the partial
                                results merged through distributed shared
                                memory.  Other modes: 0 or -1 (flat).          */
  int32_t tables_ready;      /* 0 or 1.  1 promises that ctx_lens, block_table and
                                draft_attn_step's pos hold their final values
                                before the kernel issued just before this call
                                on the stream starts (filled by the host, or by
                                work that completes before that kernel begins).
                                The attention kernel then reads them, and
                                translates the block table, before it waits
                                for that kernel (programmatic dependent launch);
                                queries, tree masks, new tokens and the caches
                                are still read only after the wait.  0: every
                                input is read after the wait.  The tcgen05
                                engine ignores it.                              */
} da_params;

typedef struct {
  int32_t num_ctas;          /* grid of the split-KV kernel                        */
  int32_t num_sms;
  int32_t rows_per_kv_head;  /* (num_q_heads / num_kv_heads) * n_q                 */
  int32_t kernel_rows;       /* rows the chosen kernel instance computes           */
  int32_t engine;            /* DA_ENGINE_*                                        */
  int32_t stages;            /* shared-memory pipeline depth (pages in flight)     */
  int32_t smem_bytes;        /* dynamic shared memory of the split-KV kernel       */
  int32_t cluster_ctas;      /* CTAs per cluster of the cluster partition (window
                                mode; the grid is batch * num_kv_heads clusters),
                                0 for the flat partition (grid num_ctas)         */
  size_t  workspace_bytes;   /* what draft_attn_run needs                          */
} da_plan_info;

typedef struct da_plan_s* da_plan_t;

/* Validates params on the host only (no CUDA call).  DA_OK, INVALID_ARG or
 * UNSUPPORTED. */
int draft_attn_check_params(const da_params* params);

/* Builds an immutable plan for `params` on CUDA device `device` and returns,
 * in *workspace_bytes, the size of the device workspace draft_attn_run needs.
 * The plan fixes the grid (one CTA per SM unless params->num_ctas is set) and
 * depends only on shapes, never on context lengths, so one plan serves every
 * draft step and can be captured in a CUDA graph.  Thread-safe after
 * creation.  Allocates no device memory. */
int draft_attn_plan(const da_params* params, int device, da_plan_t* plan,
                    size_t* workspace_bytes);

int draft_attn_plan_info(da_plan_t plan, da_plan_info* info);

void draft_attn_plan_destroy(da_plan_t plan);

/* KV append + RoPE: for every (b, token, kv head) with pos[b][token] >= 0,
 * writes RoPE(k_new, pos) to k_cache, k_new unchanged to k_side (when
 * k_side != NULL) and v_new to v_cache, at page
 * block_table[b][pos / page_size], slot pos % page_size.  Angles are formed
 * in FP32 from an exact product of the position and a two-float frequency
 * (error a few 1e-7 rad below 2^24), the rotation in FP32, the store rounds
 * to nearest even.  A negative position skips the token (padding for ragged batches).
 * batch may be below params.batch (pass a block_table offset by rows to
 * append to a subset), except with params.k_ring_pages, where row b of the
 * call is sequence b of the ring (batch must equal params.batch; pad with
 * negative positions).  k_side is required when params.mode is FOLD.
 * "FOLD ...", review (the unrotated side cache); Windowed-MTP, Abstract (the
 * draft KV grows by one token per draft step). */
int draft_attn_append_kv(da_plan_t plan, const void* k_new, const void* v_new,
                         const int32_t* pos, int32_t batch, int32_t n_new,
                         const int32_t* block_table, void* k_cache, void* v_cache,
                         void* k_side, void* stream);

/* Draft attention for every (b, query token, q head): the mode's key
 * selection, split-KV flash-decoding over the pages (one online softmax, two
 * for FOLD) in one persistent kernel, whose last CTA to finish a (sequence,
 * KV head) merges that pair's splits and writes out.  k_side may be NULL
 * unless the mode is FOLD.
 * workspace: device scratch of at least the plan's workspace_bytes, 256-byte
 * aligned.  It holds per-(sequence, KV head) page counters that must be zero
 * when a call starts: zero-fill the buffer once before its first use (every
 * call leaves the counters at zero again), and once more after a call that
 * reported DA_STATUS_WAIT_TIMEOUT.  Calls that share a workspace must not
 * overlap on the GPU. */
int draft_attn_run(da_plan_t plan, const void* q, const int32_t* q_pos,
                   const int32_t* ctx_lens, const int32_t* block_table,
                   const void* k_cache, const void* v_cache, const void* k_side,
                   void* out, void* workspace, size_t workspace_bytes, void* stream);

/* draft_attn_run for a draft tree (EAGLE-style dynamic trees, DFlash blocks:
 * drafters the FOLD and SharpDraft pages name).  The last params.tree_size
 * keys of every context are the tree's own tokens: key L - tree_size + i is
 * tree token i, appended at its slot position and rotated there.
 * tree_mask: DEVICE uint64 [batch][n_q]; bit i of tree_mask[b][t] says whether
 * query t of sequence b sees tree token i (its ancestors and itself).  Every
 * other selected key is seen as in draft_attn_run; SharpDraft's |S| counts the
 * keys the query sees.  tree_mask = NULL means every tree key is visible
 * (draft_attn_run is exactly that).  Bits at or above tree_size are ignored. */
int draft_attn_run_tree(da_plan_t plan, const void* q, const int32_t* q_pos,
                        const int32_t* ctx_lens, const int32_t* block_table,
                        const void* k_cache, const void* v_cache, const void* k_side,
                        const uint64_t* tree_mask, void* out, void* workspace,
                        size_t workspace_bytes, void* stream);

/* One draft step in one call: exactly draft_attn_append_kv(k_new, v_new,
 * pos, batch = params.batch, n_new) followed by draft_attn_run_tree, as the
 * draft head hands over its query and its new key/value together.  Every
 * argument of the attention is checked before anything is launched, so an
 * error leaves the caches untouched.  The attention kernel is launched behind
 * the append with programmatic dependent launch: its set-up overlaps the
 * append and its first global read waits for it.  n_new in 0..32 (0: no
 * append); ctx_lens already count the new tokens, as for draft_attn_run.
 * k_side is required in FOLD mode.  DA_ERR_UNSUPPORTED for n_new > 32. */
int draft_attn_step(da_plan_t plan, const void* k_new, const void* v_new, const int32_t* pos,
                    int32_t n_new, const void* q, const int32_t* q_pos, const int32_t* ctx_lens,
                    const int32_t* block_table, void* k_cache, void* v_cache, void* k_side,
                    const uint64_t* tree_mask, void* out, void* workspace,
                    size_t workspace_bytes, void* stream);

/* Ring-buffer draft KV for window mode ("Windowed-MTP ...", Abstract: the
 * draft KV outside the window is never read and can be reclaimed into a
 * compact ring).  Window mode reads only the sink positions and the last W
 * positions, so its pages can live in a ring: the first n_sink_pages logical
 * pages keep pages of their own, every later logical page j maps to ring slot
 * (j - n_sink_pages) mod (n_ring - n_sink_pages).  Appending position p then
 * overwrites a page that no window read will touch again, provided the ring
 * has at least draft_attn_ring_size() pages.  Both calls are host-only.
 *
 * draft_attn_ring_size: the smallest ring for window W and n_sink sinks:
 *   *n_sink_pages = ceil(n_sink / page_size), *n_ring = *n_sink_pages +
 *   ceil(W / page_size) + 1.  DA_ERR_INVALID_ARG for W < 1 or n_sink < 0.
 * draft_attn_ring_block_table: fills the HOST array table[0 .. max_pages-1]
 *   (one block-table row) from the HOST array ring_pages[0 .. n_ring-1] of
 *   physical page ids.  DA_ERR_INVALID_ARG for null pointers, max_pages < 1,
 *   n_sink_pages < 0 or n_ring <= n_sink_pages.  The mapping is only valid for
 *   window mode with the same W and n_sink (full, sharp and FOLD read every
 *   position). */
int draft_attn_ring_size(int32_t window, int32_t n_sink, int32_t* n_ring, int32_t* n_sink_pages);
int draft_attn_ring_block_table(int32_t* table, int64_t max_pages, const int32_t* ring_pages,
                                int32_t n_ring, int32_t n_sink_pages);

/* Size of the library-owned workspace that draft_attn_run_static uses
 * (8 MiB): enough for every shape up to 16 sequences x 8 KV heads x 32 rows
 * at head_dim 128 on 148 SMs.  Each GPU that loads the library keeps this much
 * device memory reserved until the process exits. */
#define DA_STATIC_WORKSPACE_BYTES (8u << 20)

/* draft_attn_run without a caller-supplied workspace, for callers that cannot
 * allocate device memory when they run the draft step (code that runs inside
 * another framework's allocator or memory pool, or a runtime that hands out
 * only the buffers it owns).  The scratch is a fixed array of
 * DA_STATIC_WORKSPACE_BYTES in the library's device image; the call itself
 * allocates nothing and calls no allocating routine.  The caller still passes
 * the inputs and out.  (The pages describe no such entry point; it exists for
 * deployment only.)
 *  - The first call on a device looks up the array's device address (with
 *    that device current) and caches it; make that first call before any
 *    stream capture.  A failed lookup is not cached (the call returns
 *    DA_ERR_CUDA and the next call tries again).
 *  - Returns DA_ERR_WORKSPACE_TOO_SMALL when the plan's workspace_bytes
 *    exceeds DA_STATIC_WORKSPACE_BYTES.
 *  - Every call shares the one array: each call first clears its counters
 *    on `stream`, and calls whose GPU work overlaps (different streams, or
 *    different threads) race and must be serialised by the caller.
 * Otherwise identical to draft_attn_run. */
int draft_attn_run_static(da_plan_t plan, const void* q, const int32_t* q_pos,
                          const int32_t* ctx_lens, const int32_t* block_table,
                          const void* k_cache, const void* v_cache, const void* k_side,
                          void* out, void* stream);

/* Test hook: the keys query token t of sequence b selects, computed by the
 * same device routines as draft_attn_run_tree (tree_mask: as there, may be
 * NULL).  Per key, ascending by position:
 * positions (int32), phys_slot = physical_page * page_size + slot (int64, -1
 * for an invalid block-table entry; the block table's page, where V and the
 * side cache live: with k_ring_pages a local key's rotated K sits in the
 * ring page given there), key_rope_pos (the position the key is
 * rotated at: its own, or P_far for FOLD far keys), q_rope_pos (the position
 * the kernel rotates the query by: q_pos, or q_pos - P_far for far keys) and
 * segment (0 main/local, 1 FOLD far).  At most `capacity` entries are written;
 * *count (device int64) receives the total. */
int draft_attn_debug_gather(da_plan_t plan, const int32_t* q_pos, const int32_t* ctx_lens,
                            const int32_t* block_table, const uint64_t* tree_mask, int32_t b,
                            int32_t t,
                            int32_t* positions, int64_t* phys_slot, int32_t* key_rope_pos,
                            int32_t* q_rope_pos, int8_t* segment, int64_t capacity,
                            int64_t* count, void* stream);

/* Test hook for the kernels' bounded waits: launches, on `stream`, one warp
 * that waits on an mbarrier nothing ever completes, with the same bounded wait
 * the attention kernels use.  After about 2^31 cycles (about a second) the
 * wait gives up and sets DA_STATUS_WAIT_TIMEOUT in the plan device's status
 * word, read with draft_attn_get_status; nothing faults and the context stays
 * usable.  Returns DA_ERR_INVALID_ARG for a NULL plan, DA_ERR_CUDA when the
 * launch fails. */
int draft_attn_debug_wait_timeout(da_plan_t plan, void* stream);

/* Synchronises `stream`, reads and clears the plan device's status word.
 * Returns DA_OK when it was zero, DA_ERR_DEVICE_FAULT otherwise; *bits (host
 * pointer, may be NULL) receives the DA_STATUS_* bits. */
int draft_attn_get_status(da_plan_t plan, void* stream, uint32_t* bits);

const char* draft_attn_error_string(int code);

/* ABI version (major * 100 + minor). */
int draft_attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DRAFT_ATTN_H */
