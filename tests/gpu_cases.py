"""Shared set-up of the GPU parity tests: seeded inputs, paged caches filled
through the library's own append entry point, the float64 oracle on the same
values, and the tolerance check.

Tolerances: bf16 outputs max |err| <= 2e-2 and mean |err| <= 2e-3; fp32
outputs max |err| <= 1e-5 (both against the float64 oracle).
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle.draft_attn_oracle as orc
from draft_attention_decode_b300 import binding as B
from draft_attention_decode_b300 import workloads as WL

TOL = {"bf16": (2e-2, 2e-3), "fp32": (1e-5, 1e-6)}


class Setup:
    """One plan, its caches and the raw inputs they were filled from."""

    def __init__(self, *, batch, n_q, num_q_heads, num_kv_heads, head_dim, dtype, ctx,
                 mode="full", window=0, n_sink=0, alpha=1.0, far_mix=0.0, scale_slope=0.0,
                 scale_ref=4096, rope_theta=1e4, num_ctas=0, seed=0, extra_tokens=0,
                 spare_pages=3, q_pos=None, fill=True, engine=0, tree_size=0,
                 side_fp8_scale=0.0, cluster_ctas=0, tables_ready=0):
        self.dev = torch.device("cuda", 0)
        self.dtype = dtype
        tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
        self.ctx = [int(c) for c in ctx]
        cap = [c + extra_tokens for c in self.ctx]
        self.cap = cap
        self.k_raw = [WL.randn((max(c, 1), num_kv_heads, head_dim), tdt, self.dev,
                               seed * 16 + 2 + 1000 * b) for b, c in enumerate(cap)]
        self.v = [WL.randn((max(c, 1), num_kv_heads, head_dim), tdt, self.dev,
                           seed * 16 + 3 + 1000 * b) for b, c in enumerate(cap)]
        self.q = WL.randn((batch, n_q, num_q_heads, head_dim), tdt, self.dev, seed * 16 + 1)
        if q_pos is None:
            q_pos = [[c + t for t in range(n_q)] for c in self.ctx]
        self.q_pos = torch.tensor(q_pos, dtype=torch.int32, device=self.dev)
        self.ctx_lens = torch.tensor(self.ctx, dtype=torch.int32, device=self.dev)
        bt, npg = WL.block_table([max(c, 1) for c in cap], seed, spare_pages=spare_pages,
                                 device=self.dev)
        self.block_table = bt.contiguous()
        self.num_pages = npg
        self.da = B.DraftAttention(
            device=0, batch=batch, n_q=n_q, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
            head_dim=head_dim, num_pages=npg, max_pages_per_seq=bt.shape[1], dtype=dtype,
            mode=mode, window=window, n_sink=n_sink, alpha=alpha, far_mix=far_mix,
            scale_slope=scale_slope, scale_ref=scale_ref, rope_theta=rope_theta,
            num_ctas=num_ctas, engine=engine, tree_size=tree_size,
            side_fp8=1 if side_fp8_scale > 0 else 0, side_scale=side_fp8_scale,
            cluster_ctas=cluster_ctas, tables_ready=tables_ready)
        shape = (npg, num_kv_heads, WL.PAGE, head_dim)
        # NaN-filled so that a read of a slot nobody wrote shows up in the output
        self.k_cache = torch.full(shape, float("nan"), dtype=tdt, device=self.dev)
        self.v_cache = torch.full(shape, float("nan"), dtype=tdt, device=self.dev)
        if mode == "fold" and side_fp8_scale > 0:   # E4M3 codes; 0x7F is NaN
            self.k_side = torch.full(shape, 0x7F, dtype=torch.uint8, device=self.dev)
        elif mode == "fold":
            self.k_side = torch.full(shape, float("nan"), dtype=tdt, device=self.dev)
        else:
            self.k_side = None
        self.prm = orc.Params(mode=mode, window=window, n_sink=n_sink if mode in ("window", "fold") else 0,
                              alpha=alpha, far_mix=far_mix, scale_slope=scale_slope,
                              scale_ref=scale_ref, rope_theta=rope_theta, n_tree=tree_size,
                              side_fp8_scale=side_fp8_scale)
        if fill:
            for b, c in enumerate(self.ctx):
                self.append(b, 0, c)

    def append(self, b, start, stop):
        """Appends tokens start..stop-1 of sequence b through the library."""
        if stop <= start:
            return
        k = self.k_raw[b][start:stop].unsqueeze(0).contiguous()
        v = self.v[b][start:stop].unsqueeze(0).contiguous()
        pos = torch.arange(start, stop, dtype=torch.int32, device=self.dev).unsqueeze(0)
        self.da.append_kv(k, v, pos, self.block_table[b:b + 1], self.k_cache, self.v_cache,
                          self.k_side)

    def run(self, q=None, q_pos=None, ctx_lens=None, tree_mask=None):
        out = self.da.run(self.q if q is None else q, self.q_pos if q_pos is None else q_pos,
                          self.ctx_lens if ctx_lens is None else ctx_lens, self.block_table,
                          self.k_cache, self.v_cache, self.k_side, tree_mask=tree_mask)
        torch.cuda.synchronize()
        return out

    def status(self):
        return self.da.status()

    def oracle(self, groups=None, q=None, q_pos=None, ctx=None, tree_masks=None):
        """Float64 oracle output [B, n_q, H_q, d] (NaN outside `groups`, a list
        of (b, t, kv_head)); tree_masks[b][t]: the query's visible tree keys."""
        q = (self.q if q is None else q).float().cpu().numpy().astype(np.float64)
        qp = (self.q_pos if q_pos is None else q_pos).cpu().numpy()
        ctx = self.ctx if ctx is None else ctx
        Bn, n_q, H_q, d = q.shape
        H_kv = self.k_raw[0].shape[1]
        G = H_q // H_kv
        if groups is None:
            groups = [(b, t, g) for b in range(Bn) for t in range(n_q) for g in range(H_kv)]
        out = np.full(q.shape, np.nan)
        cache = {}
        for b, t, g in sorted(groups):
            L = int(ctx[b])
            if (b, g) not in cache:
                cache.clear()
                n = max(L, 1)
                cache[(b, g)] = (self.k_raw[b][:n, g].float().cpu().numpy(),
                                 self.v[b][:n, g].float().cpu().numpy())
            kb, vb = cache[(b, g)]
            heads = slice(g * G, (g + 1) * G)
            tm = None if tree_masks is None else int(tree_masks[b][t])
            out[b, t, heads] = orc.attend_group(q[b, t, heads], int(qp[b, t]), kb, vb, L,
                                                self.prm, tree_mask=tm)
        return out

    def close(self):
        self.da.close()


def compare(got, want, dtype, what=""):
    """Element-wise comparison of the GPU output with the oracle where the
    oracle was evaluated (non-NaN)."""
    g = got.float().cpu().numpy().astype(np.float64)
    m = ~np.isnan(want)
    assert m.any()
    assert np.isfinite(g[m]).all(), f"{what}: non-finite GPU output"
    err = np.abs(g[m] - want[m])
    tmax, tmean = TOL[dtype]
    assert err.max() <= tmax and err.mean() <= tmean, (
        f"{what}: max {err.max():.3g} (tol {tmax}), mean {err.mean():.3g} (tol {tmean})")
    return float(err.max()), float(err.mean())


def sample_groups(batch, n_q, H_kv, k, seed):
    rng = np.random.default_rng(seed)
    allg = [(b, t, g) for b in range(batch) for t in range(n_q) for g in range(H_kv)]
    idx = rng.choice(len(allg), size=min(k, len(allg)), replace=False)
    return [allg[i] for i in sorted(idx)]


def equal_up_to_one_rounding(a, b, atol=2.0 ** -17):
    """Element-wise |a - b| <= one bf16 ulp of the larger magnitude + atol: two
    kernels that compute the same attention with a different summation order
    (the CUDA-core engine with or without turn-taking warp groups, or another
    split of the keys over CTAs) hold FP32 results a few 1e-7 apart, which
    round to the same or an adjacent bf16 value; atol covers outputs near
    zero, where that FP32 difference is larger than a bf16 ulp of the result."""
    x = a.float().cpu().numpy().astype(np.float64)
    y = b.float().cpu().numpy().astype(np.float64)
    return bool((np.abs(x - y) <= bf16_ulp(np.maximum(np.abs(x), np.abs(y))) + atol).all())


def bf16_ulp(x):
    """Spacing of bfloat16 at |x| (normal range)."""
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    return np.ldexp(1.0, (np.floor(np.log2(ax)) - 7).astype(np.int64))


def gamma(n, beta, n_ref):
    return max(1.0, 1.0 + beta * math.log(n / n_ref)) if n > 0 else 1.0
