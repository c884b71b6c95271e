"""Seeded synthetic inputs for draft-decode attention.

This module only draws numbers and lays them out: it holds none of the
method's arithmetic (no RoPE, no selection, no softmax).  The CUDA path and the
float64 oracle both take their inputs from here, so both see the same values.

Five workloads, named by what they are:

==================  ==========================================================
tiny_window_fp32    B=1, 1 query, 8/2 heads, d=64, fp32, context 4096 (keys at
                    positions 0..4095), query at 4096, theta=1e4, W=512 + 4
                    sinks; full and window.
mtp_draft_128k      B=1, 32/8 heads, d=128, bf16, context 131072, 64-token
                    pages with a shuffled block table, 4 draft steps that each
                    append one token then attend (query at the new token);
                    full and window (W=2048).
mtp_draft_1m        B=1, 64/8 heads, d=128, bf16, context 1,048,576, theta=1e6,
                    6 draft steps; full and window (W=4096 + 4 sinks).
fold_4x256k         B=4, 32/8 heads, d=128, bf16, contexts 262144, query at
                    position L; fold (W=2048, alpha=2, lambda=0.5), plus full
                    and window for reference.
ragged_tree_16x8    B=16, 8 draft-tree queries per sequence (query t at L+t),
                    32/8 heads, d=128, bf16, context lengths log-uniform in
                    [32768, 524288]; full, window (W=4096) and sharp
                    (beta=0.05, N_ref=4096).
==================  ==========================================================

Values are N(0, 1) float32 draws rounded (ties to even) to the storage dtype.
The block table is a seeded permutation of all physical pages.  Sub-seeds:
seed*16 + {1: q, 2: K, 3: V, 4: block table, 5: lengths}.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import numpy as np
import torch

PAGE = 64


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    n_q: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    dtype: str                      # "bf16" | "fp32"
    ctx: tuple                      # context length per sequence before drafting
    modes: tuple
    window: int = 0
    n_sink: int = 0
    rope_theta: float = 10000.0
    draft_steps: int = 0            # >0: append one token then attend, per step
    alpha: float = 1.0
    far_mix: float = 0.0
    scale_slope: float = 0.0
    scale_ref: int = 4096
    query_at: str = "after"         # "after": p = L + t ; "self": p = new token
    seed: int = 0
    mode_window: dict = field(default_factory=dict)  # per-mode W override

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    def window_for(self, mode: str) -> int:
        return self.mode_window.get(mode, self.window)

    def sinks_for(self, mode: str) -> int:
        return self.n_sink if mode == "window" else 0


def ragged_lengths(batch: int, lo: int, hi: int, seed: int) -> tuple:
    """round(exp(U[ln lo, ln hi])) per sequence, seeded."""
    rng = np.random.default_rng(seed * 16 + 5)
    u = rng.uniform(math.log(lo), math.log(hi), size=batch)
    return tuple(int(round(math.exp(x))) for x in u)


WORKLOADS = {
    "tiny_window_fp32": Workload(
        "tiny_window_fp32", 1, 1, 8, 2, 64, "fp32", (4096,), ("full", "window"),
        window=512, n_sink=4, rope_theta=1e4, seed=0),
    "mtp_draft_128k": Workload(
        "mtp_draft_128k", 1, 1, 32, 8, 128, "bf16", (131072,), ("full", "window"),
        window=2048, n_sink=0, rope_theta=1e4, draft_steps=4, query_at="self", seed=1),
    "mtp_draft_1m": Workload(
        "mtp_draft_1m", 1, 1, 64, 8, 128, "bf16", (1048576,), ("full", "window"),
        window=4096, n_sink=4, rope_theta=1e6, draft_steps=6, query_at="self", seed=2),
    "fold_4x256k": Workload(
        "fold_4x256k", 4, 1, 32, 8, 128, "bf16", (262144,) * 4,
        ("fold", "full", "window"), window=2048, alpha=2.0, far_mix=0.5,
        rope_theta=1e4, seed=3),
    "ragged_tree_16x8": Workload(
        "ragged_tree_16x8", 16, 8, 32, 8, 128, "bf16",
        ragged_lengths(16, 32768, 524288, 4), ("full", "window", "sharp"),
        window=4096, scale_slope=0.05, scale_ref=4096, rope_theta=1e4, seed=4),
}


def resized(wl: Workload, ctx) -> Workload:
    """Same workload with other context lengths (for reduced-size tests)."""
    if isinstance(ctx, int):
        ctx = (ctx,) * wl.batch
    return replace(wl, ctx=tuple(int(c) for c in ctx), batch=len(ctx))


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def randn(shape, dtype, device, seed: int) -> torch.Tensor:
    """N(0,1) float32 draws rounded to ``dtype``."""
    x = torch.randn(shape, generator=_gen(device, seed), device=device,
                    dtype=torch.float32)
    return x.to(dtype)


def block_table(capacity, seed: int, spare_pages: int = 0, page: int = PAGE,
                device="cpu"):
    """Block table [B, max_pages] int32 whose rows hold a seeded permutation of
    all physical pages (each sequence owns ceil(capacity_b / page) of them; the
    rest of each row is -1).  Returns (table, num_pages)."""
    need = [(int(c) + page - 1) // page for c in capacity]
    num_pages = sum(need) + spare_pages
    perm = torch.randperm(num_pages, generator=_gen("cpu", seed * 16 + 4))
    maxp = max(max(need), 1)
    bt = torch.full((len(need), maxp), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(need):
        bt[b, :n] = perm[off: off + n].to(torch.int32)
        off += n
    return bt.to(device), num_pages


@dataclass
class Case:
    """One workload instance.  ``k_raw[b]``/``v[b]``: [cap_b, H_kv, d] raw keys
    and values by logical position (cap_b = L_b + draft steps); ``q``: per draft
    step (or a single entry) [B, n_q, H_q, d]; ``q_pos``/``ctx_lens`` likewise."""
    wl: Workload
    k_raw: list
    v: list
    q: list
    q_pos: list
    ctx_lens: list
    block_table: torch.Tensor
    num_pages: int


def make_case(wl: Workload, device="cpu", seed=None) -> Case:
    seed = wl.seed if seed is None else seed
    dt = wl.torch_dtype
    steps = max(wl.draft_steps, 1)
    cap = [c + wl.draft_steps for c in wl.ctx]
    k_raw, v = [], []
    for b, c in enumerate(cap):
        k_raw.append(randn((c, wl.num_kv_heads, wl.head_dim), dt, device,
                           seed * 16 + 2 + 1000 * b))
        v.append(randn((c, wl.num_kv_heads, wl.head_dim), dt, device,
                       seed * 16 + 3 + 1000 * b))
    qs, qp, cl = [], [], []
    for s in range(steps):
        qs.append(randn((wl.batch, wl.n_q, wl.num_q_heads, wl.head_dim), dt, device,
                        seed * 16 + 1 + 7919 * s))
        if wl.draft_steps:
            L = [c + s + 1 for c in wl.ctx]           # the step's token is appended first
            p = [[c + s] * wl.n_q for c in wl.ctx]    # the query sits at that token
        else:
            L = list(wl.ctx)
            p = [[c + t for t in range(wl.n_q)] for c in wl.ctx]
        qp.append(torch.tensor(p, dtype=torch.int32, device=device))
        cl.append(torch.tensor(L, dtype=torch.int32, device=device))
    bt, npg = block_table(cap, seed, device=device)
    return Case(wl, k_raw, v, qs, qp, cl, bt, npg)
