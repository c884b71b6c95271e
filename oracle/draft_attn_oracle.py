"""Plain float64 CPU oracle for speculative-draft decode attention.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or links
this module: only the tests, the smoke check and the benchmark's CPU-baseline
leg do.  It shares no code with the CUDA library (no kernels, headers, tables or
helpers); the only thing both sides share is the seeded input generator, which
holds none of the method's arithmetic.

What it computes, and where each piece comes from (sources are the web pages on
the subject, cited by title and section):

* "Windowed-MTP: Removing the Full-Context Draft-KV Tax at Million-Token
  Context", Abstract (arXiv):
    - ``full``: the MTP draft head attends over the entire KV cache at every
      draft step (the "draft-KV tax").
    - ``window``: a StreamingLLM-style sliding window of the last W tokens plus
      attention-sink tokens, applied to the draft's attention only.
  RoPE follows "RoFormer: Enhanced Transformer with Rotary Position Embedding",
  listed under that page's "Builds on"; sinks follow "Efficient Streaming
  Language Models with Attention Sinks", listed in the same place.
* "FOLD: Position-Free Far Memory with Local Order for Long-Context Speculative
  Decoding", summary, review and abstract:
    - ``fold``: exact positions inside a local window; every older key is a
      far-memory entry rotated at one shared virtual position from an unrotated
      side cache; a concentration factor alpha sharpens the far softmax, which
      is normalised separately from the local one, and the far memory's total
      weight is controlled separately (the mix weight lambda).
* "SharpDraft: Accelerating Long-Context Speculative Decoding with
  Cardinality-Aware Query Scaling", Abstract:
    - ``sharp``: the query is scaled by a fixed-slope closed-form function of
      the number of visible keys.

The pages print no formula for any of these.  The readings taken where they are
silent (all listed again in the design notes):

1. RoPE: rotate-half pairing (x_i, x_{i+d/2}), inv_freq_i = theta^(-2i/d),
   angle = pos * inv_freq_i, the whole head_dim rotated, no scaling.
2. Keys keep their original positions; a key at position j is stored rotated
   at j.  The query position p is an explicit input.
3. window: S = {0 <= j < min(n_sink, L)} union {max(0, L-W) <= j < L}.
4. fold: Loc = {max(0, L-W) <= j < L}, Far = {0 <= j < L-W}, shared far
   position P_far = L-W-1 (the newest far token).  With n_sink > 0 (FOLD
   combined with StreamingLLM-style sinks) the first n_sink keys join the
   local softmax at their exact positions: Loc = {j < min(n_sink, L)} union
   {max(0, L-W) <= j < L}, Far = {n_sink <= j < L-W}.  Far logits are
   alpha * c * <RoPE(q, p), RoPE(k_raw_j, P_far)>; two independent softmaxes;
   o = (1-lam_eff) o_loc + lam_eff o_far with lam_eff = lam if Far is non-empty
   else 0.  V is never rotated; far V comes from the main V cache.
5. sharp: S as in full; gamma = max(1, 1 + beta * ln(|S| / N_ref)); logits are
   gamma * c * <RoPE(q, p), K_rot_j>.
6. Grouped-query attention: query head h reads KV head h // (H_q / H_kv).
7. An empty selection gives a zero output.
8. NoPE: rope_theta = 0 means no rotation at all (keys and queries enter the
   dot product as stored), for the NoPE draft the Windowed-MTP abstract names.
9. Draft trees (EAGLE-style dynamic trees and DFlash blocks, which the FOLD
   and SharpDraft pages name as drafters): the last n_tree keys of a context
   are the tree's own tokens, key L-n_tree+i being tree token i at its own
   slot position.  A query sees the mode's selection with the tree keys
   restricted to those whose bit i is set in its mask (its ancestors and
   itself); SharpDraft's |S| counts the keys the query actually sees.
10. FP8 side cache (the FOLD page puts the side cache's size at up to 6 GiB
   and fixes no format; this is the library's option for shrinking it): the
   side cache may hold the unrotated keys as FP8 E4M3 codes of k_raw / s, s a
   positive per-tensor scale.  The quotient is formed in IEEE float32 (the
   precision the kernel decides the code in), then rounded to the nearest
   E4M3 value, ties to the even code, magnitudes at or above 448 saturating
   to 448.  Far keys are then code value * s.  E4M3 (the OCP 8-bit floating
   point format): 1 sign, 4 exponent (bias 7), 3 mantissa bits; exponent 0 is
   subnormal (m/8 * 2^-6); S.1111.111 is NaN; no infinities.

Arithmetic: float64 throughout (numpy).  Softmax is exp(s - max) / sum.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

MODES = ("full", "window", "fold", "sharp")

# Segment ids used in the selection lists: the main (local) softmax and the
# FOLD far-memory softmax.
SEG_LOCAL = 0
SEG_FAR = 1


@dataclass
class Params:
    """Mode hyper-parameters (names follow the pages: W, alpha, lambda, beta)."""

    mode: str = "full"
    window: int = 0          # W (window, fold)
    n_sink: int = 0          # attention-sink tokens (window, fold)
    alpha: float = 1.0       # FOLD concentration factor
    far_mix: float = 0.0     # FOLD far-memory weight lambda
    scale_slope: float = 0.0  # SharpDraft slope beta
    scale_ref: int = 4096     # SharpDraft reference cardinality N_ref
    rope_theta: float = 10000.0
    softmax_scale: float = 0.0  # 0 => 1/sqrt(d)
    n_tree: int = 0           # draft-tree tokens at the end of the context (reading 9)
    side_fp8_scale: float = 0.0  # > 0: FOLD side cache as E4M3 codes of k / s (reading 10)
    extra: dict = field(default_factory=dict)


# --------------------------------------------------------------------------
# RoPE ("RoFormer", listed under Windowed-MTP "Builds on"; reading 1)
# --------------------------------------------------------------------------

def rope_inv_freq(d: int, theta: float) -> np.ndarray:
    """inv_freq_i = theta^(-2i/d) for i < d/2, in float64.  theta = 0 selects
    NoPE (no positional rotation: every frequency is zero), the draft of the
    Mamba2-hybrid NoPE model in the Windowed-MTP abstract (reading 8)."""
    i = np.arange(d // 2, dtype=np.float64)
    if theta == 0:
        return np.zeros(d // 2)
    return np.power(np.float64(theta), -2.0 * i / d)


def rope_angles(pos, d: int, theta: float) -> np.ndarray:
    """angle[..., i] = pos * inv_freq_i (float64), pos of any integer shape."""
    pos = np.asarray(pos, dtype=np.float64)
    return pos[..., None] * rope_inv_freq(d, theta)


def rope(x, pos, theta: float) -> np.ndarray:
    """Rotate-half RoPE of ``x[..., d]`` at integer positions ``pos`` (broadcast
    against x's leading shape).  Pair (x_i, x_{i+d/2}) is rotated by angle_i:
        x'_i       = x_i cos a - x_{i+d/2} sin a
        x'_{i+d/2} = x_{i+d/2} cos a + x_i sin a
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    a = rope_angles(pos, d, theta)
    c, s = np.cos(a), np.sin(a)
    x1, x2 = x[..., : d // 2], x[..., d // 2:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


# --------------------------------------------------------------------------
# Key selection (Windowed-MTP Abstract; FOLD abstract; readings 3 and 4)
# --------------------------------------------------------------------------

def window_start(L: int, W: int) -> int:
    return max(0, L - W)


def fold_far_position(L: int, W: int) -> int:
    """Shared virtual position of the FOLD far memory: the newest far token."""
    return L - W - 1


def select_keys(mode: str, L: int, W: int = 0, n_sink: int = 0) -> dict:
    """Selected key positions per segment, ascending.

    Returns {"loc": positions of the main softmax, "far": FOLD far positions}.
    """
    if mode not in MODES:
        raise ValueError(mode)
    empty = np.zeros(0, dtype=np.int64)
    if mode in ("full", "sharp"):
        return {"loc": np.arange(L, dtype=np.int64), "far": empty}
    ws = window_start(L, W)
    if mode == "window":
        sinks = np.arange(min(n_sink, L), dtype=np.int64)
        recent = np.arange(ws, L, dtype=np.int64)
        return {"loc": np.union1d(sinks, recent).astype(np.int64), "far": empty}
    # fold: sinks, when given, join the local softmax (reading 4)
    sinks = np.arange(min(n_sink, L), dtype=np.int64)
    return {"loc": np.union1d(sinks, np.arange(ws, L, dtype=np.int64)).astype(np.int64),
            "far": np.arange(min(n_sink, max(0, L - W)), max(0, L - W), dtype=np.int64)}


def sharp_gamma(n_keys: int, beta: float, n_ref: int) -> float:
    """SharpDraft fixed-slope query scale (reading 5), float64."""
    if n_keys <= 0:
        return 1.0
    return max(1.0, 1.0 + beta * math.log(n_keys / n_ref))


def page_slot(positions, block_table_row, page_size: int = 64):
    """Paged-cache address of each logical position (PagedAttention, listed
    under Windowed-MTP "Builds on"): the position's page index selects an entry
    of the block table, the remainder is the slot inside that page.
    Returns (physical page, slot, physical_page * page_size + slot)."""
    positions = np.asarray(positions, dtype=np.int64)
    bt = np.asarray(block_table_row, dtype=np.int64)
    phys = bt[positions // page_size]
    slot = positions % page_size
    return phys, slot, phys * page_size + slot


def tree_filter(positions, L: int, n_tree: int, tree_mask):
    """Drops the tree keys (positions >= L - n_tree) whose bit is clear in
    tree_mask (an int; None keeps every key).  Reading 9."""
    positions = np.asarray(positions, dtype=np.int64)
    if tree_mask is None or n_tree <= 0:
        return positions
    base = L - n_tree
    keep = [j < base or (int(tree_mask) >> int(j - base)) & 1 == 1 for j in positions]
    return positions[np.asarray(keep, dtype=bool)] if positions.size else positions


def selection_list(mode: str, L: int, p: int, prm: Params, block_table_row=None,
                   page_size: int = 64, tree_mask=None) -> dict:
    """Per selected key: position, segment, the RoPE position its key is
    rotated at (j, or P_far for far keys), the position the query is rotated by
    when the key side is left as stored (p, or p - P_far for far keys, from
    <R(p)q, R(P)k> = <R(p-P)q, k>), and optionally the paged address.
    Sorted by position (positions are unique within one selection)."""
    sel = select_keys(mode, L, prm.window, prm.n_sink)
    loc = tree_filter(sel["loc"], L, prm.n_tree, tree_mask)
    far = tree_filter(sel["far"], L, prm.n_tree, tree_mask)
    pos = np.concatenate([far, loc])
    seg = np.concatenate([np.full(far.size, SEG_FAR, np.int8),
                          np.full(loc.size, SEG_LOCAL, np.int8)])
    if far.size:
        pf = fold_far_position(L, prm.window)
        key_rope = np.concatenate([np.full(far.size, pf, np.int64), loc])
        q_rope = np.concatenate([np.full(far.size, p - pf, np.int64),
                                 np.full(loc.size, p, np.int64)])
    else:
        key_rope = loc.copy()
        q_rope = np.full(loc.size, p, np.int64)
    order = np.argsort(pos, kind="stable")
    out = {"position": pos[order], "segment": seg[order],
           "key_rope_pos": key_rope[order], "q_rope_pos": q_rope[order]}
    if block_table_row is not None:
        _, _, flat = page_slot(out["position"], block_table_row, page_size)
        out["phys_slot"] = flat
    return out


# --------------------------------------------------------------------------
# Attention for one query row
# --------------------------------------------------------------------------

def _softmax(s: np.ndarray) -> np.ndarray:
    """exp(s - max) / sum over axis 0 (float64); empty input -> empty."""
    if s.shape[0] == 0:
        return s
    e = np.exp(s - s.max(axis=0, keepdims=True))
    return e / e.sum(axis=0, keepdims=True)


def _take(a, idx: np.ndarray):
    """a[idx] for the first axis; a view when idx is one contiguous run."""
    if idx.size and idx[-1] - idx[0] + 1 == idx.size:
        return a[int(idx[0]): int(idx[-1]) + 1]
    return np.asarray(a)[idx]


def _logits(q_rot: np.ndarray, k_raw: np.ndarray, key_pos, theta: float,
            chunk: int) -> np.ndarray:
    """s[j, r] = <q_rot[r], RoPE(k_raw[j], key_pos[j])> for every selected key,
    evaluated chunk by chunk over keys (each logit is computed on its own, so
    chunking does not change any value)."""
    n = k_raw.shape[0]
    out = np.empty((n, q_rot.shape[0]), dtype=np.float64)
    key_pos = np.broadcast_to(np.asarray(key_pos, dtype=np.int64), (n,))
    for a in range(0, n, chunk):
        b = min(n, a + chunk)
        kr = rope(np.asarray(k_raw[a:b], dtype=np.float64), key_pos[a:b], theta)
        out[a:b] = kr @ q_rot.T
    return out


def _weighted_sum(w: np.ndarray, v: np.ndarray, chunk: int) -> np.ndarray:
    """o[r] = sum_j w[j, r] v[j], accumulated in key order chunk by chunk."""
    o = np.zeros((w.shape[1], v.shape[1]), dtype=np.float64)
    for a in range(0, w.shape[0], chunk):
        b = min(w.shape[0], a + chunk)
        o += w[a:b].T @ np.asarray(v[a:b], dtype=np.float64)
    return o


def attend_group(q_rows, p: int, k_raw, v, L: int, prm: Params,
                 chunk: int = 1 << 16, return_weights: bool = False, tree_mask=None):
    """Attention of several query rows that share one query position p and one
    KV head.

    q_rows: [n_rows, d] un-rotated queries.  k_raw, v: [>= L, d] un-rotated keys
    and values of that KV head, indexed by logical position.  tree_mask: the
    query's visible tree keys (reading 9; None: all).  Returns o: [n_rows, d]
    float64 (and, optionally, the effective per-key weights).
    """
    q_rows = np.atleast_2d(np.asarray(q_rows, dtype=np.float64))
    n_rows, d = q_rows.shape
    c = prm.softmax_scale if prm.softmax_scale > 0 else 1.0 / math.sqrt(d)
    theta = prm.rope_theta
    q_rot = rope(q_rows, p, theta)
    sel = select_keys(prm.mode, L, prm.window, prm.n_sink)
    loc = tree_filter(sel["loc"], L, prm.n_tree, tree_mask)
    far = tree_filter(sel["far"], L, prm.n_tree, tree_mask)

    gamma = 1.0
    if prm.mode == "sharp":
        gamma = sharp_gamma(loc.size, prm.scale_slope, prm.scale_ref)

    # Local / main segment: keys rotated at their own positions.
    s_loc = gamma * c * _logits(q_rot, _take(k_raw, loc), loc, theta, chunk)
    w_loc = _softmax(s_loc)
    o_loc = (_weighted_sum(w_loc, _take(v, loc), chunk) if loc.size
             else np.zeros((n_rows, d)))

    if prm.mode != "fold":
        return (o_loc, {"loc": (loc, w_loc)}) if return_weights else o_loc

    # FOLD far memory: raw keys from the side cache rotated at one shared
    # position, logits sharpened by alpha, softmax normalised on its own.
    if far.size:
        pf = fold_far_position(L, prm.window)
        k_far = _take(k_raw, far)
        if prm.side_fp8_scale > 0:
            k_far = side_fp8_keys(k_far, prm.side_fp8_scale)
        f_far = prm.alpha * c * _logits(q_rot, k_far, pf, theta, chunk)
        w_far = _softmax(f_far)
        o_far = _weighted_sum(w_far, _take(v, far), chunk)
        lam = prm.far_mix
    else:
        w_far = np.zeros((0, n_rows))
        o_far = np.zeros((n_rows, d))
        lam = 0.0
    o = (1.0 - lam) * o_loc + lam * o_far
    if return_weights:
        return o, {"loc": (loc, (1.0 - lam) * w_loc), "far": (far, lam * w_far)}
    return o


def attend(q, q_pos, k_raw, v, ctx_lens, prm: Params, rows=None,
           chunk: int = 1 << 16, tree_masks=None) -> np.ndarray:
    """Draft attention for a batch.

    q: [B, n_q, H_q, d]; q_pos: [B, n_q]; k_raw[b], v[b]: [>= L_b, H_kv, d]
    (un-rotated keys and values by logical position, any float dtype; a list or
    an array); ctx_lens: [B].  ``rows`` optionally restricts the computation to
    a list of (b, t, h) query rows (others are left NaN).  tree_masks[b][t]:
    the visible tree keys of query t (reading 9).  Returns
    [B, n_q, H_q, d] float64.
    """
    q = np.asarray(q)
    B, n_q, H_q, d = q.shape
    H_kv = np.asarray(k_raw[0]).shape[1]
    G = H_q // H_kv
    out = np.full((B, n_q, H_q, d), np.nan)
    want = None if rows is None else {tuple(r) for r in rows}
    for b in range(B):
        L = int(ctx_lens[b])
        for t in range(n_q):
            p = int(q_pos[b][t])
            for g in range(H_kv):
                heads = [g * G + j for j in range(G)
                         if want is None or (b, t, g * G + j) in want]
                if not heads:
                    continue
                kb = np.asarray(k_raw[b])[:, g, :]
                vb = np.asarray(v[b])[:, g, :]
                tm = None if tree_masks is None else int(tree_masks[b][t])
                o = attend_group(q[b, t, heads, :], p, kb, vb, L, prm, chunk=chunk, tree_mask=tm)
                out[b, t, heads, :] = o
    return out


# --------------------------------------------------------------------------
# KV append (rotated cache, FOLD side cache, V cache)
# --------------------------------------------------------------------------

def append_rotated_keys(k_new, pos, theta: float) -> np.ndarray:
    """Keys as the rotated cache stores them: RoPE(k_raw, pos) in float64.
    k_new: [..., H_kv, d]; pos: [...] (one position per token)."""
    k = np.asarray(k_new, dtype=np.float64)
    pos = np.asarray(pos, dtype=np.int64)
    return rope(k, pos[..., None], theta)


# --------------------------------------------------------------------------
# FP8 E4M3 side cache (reading 10)
# --------------------------------------------------------------------------

E4M3_MAX = 448.0


def e4m3_value(code: int) -> float:
    """The value of one E4M3 code (0..255) from the format's fields."""
    sign = -1.0 if code & 0x80 else 1.0
    e, m = (code >> 3) & 0xF, code & 0x7
    if e == 15 and m == 7:
        return math.nan
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** -6
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def e4m3_encode(x) -> np.ndarray:
    """Codes of float32 values: nearest E4M3 value, ties to the even code,
    |x| >= 448 saturating to 448, the sign kept (so -0 and small negatives that
    round to zero give 0x80)."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    mags = np.array([e4m3_value(c) for c in range(0x7F)])     # codes 0..126, ascending
    a = np.minimum(np.abs(x), E4M3_MAX).ravel()
    hi = np.searchsorted(mags, a, side="left")                # first magnitude >= a
    hi = np.minimum(hi, 0x7E)
    lo = np.maximum(hi - 1, 0)
    d_lo, d_hi = a - mags[lo], mags[hi] - a
    code = np.where(d_lo < d_hi, lo, hi)
    tie = d_lo == d_hi
    code = np.where(tie, np.where(lo % 2 == 0, lo, hi), code)
    code = np.where(mags[hi] == a, hi, code)                  # exact values
    sign = np.signbit(x.ravel()).astype(np.int64) << 7
    return (code.astype(np.int64) | sign).astype(np.uint8).reshape(x.shape)


def e4m3_decode(codes) -> np.ndarray:
    table = np.array([e4m3_value(c) for c in range(256)])
    return table[np.asarray(codes, dtype=np.int64)]


def side_fp8_codes(k_raw, scale: float) -> np.ndarray:
    """The side cache's bytes for un-rotated keys k_raw: E4M3 codes of the
    float32 quotient k_raw / scale."""
    q = np.asarray(k_raw, dtype=np.float32) / np.float32(scale)
    return e4m3_encode(q)


def side_fp8_keys(k_raw, scale: float) -> np.ndarray:
    """Far keys as the FP8 side cache gives them back: code value * scale."""
    return e4m3_decode(side_fp8_codes(k_raw, scale)) * np.float64(np.float32(scale))


def round_to_bf16(x) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 value (ties to even),
    returned as float64.  bfloat16 has 8 mantissa bits (7 stored) and float32's
    exponent range; below 2^-126 the spacing is fixed at 2^-133."""
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros_like(x)
    nz = (x != 0) & np.isfinite(x)
    ax = np.abs(x[nz])
    e = np.floor(np.log2(ax))
    # guard log2 rounding at exact powers of two
    e = np.where(np.ldexp(1.0, e.astype(np.int64)) > ax, e - 1, e)
    e = np.where(np.ldexp(1.0, (e + 1).astype(np.int64)) <= ax, e + 1, e)
    e = np.maximum(e, -126.0)
    ulp = np.ldexp(1.0, (e - 7).astype(np.int64))
    out[nz] = np.rint(x[nz] / ulp) * ulp          # np.rint: half to even
    out[~np.isfinite(x)] = x[~np.isfinite(x)]
    return out
