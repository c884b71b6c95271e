"""GPU parity at the five workloads' full sizes, in the launch configuration
the benchmark times (one persistent CTA per SM, the default plan).  Outputs
are compared element by element on sampled (sequence, query, KV head) groups
that the float64 oracle evaluates one by one; the selection of every sampled
query is compared bit-exact through the gather hook."""
import numpy as np
import pytest
import torch

import oracle.draft_attn_oracle as orc
from draft_attention_decode_b300 import binding as B
from draft_attention_decode_b300 import workloads as WL
from tests.gpu_cases import Setup, compare, sample_groups

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu(cuda_lib):
    yield


def _setup(wl, mode, **kw):
    return Setup(batch=wl.batch, n_q=wl.n_q, num_q_heads=wl.num_q_heads,
                 num_kv_heads=wl.num_kv_heads, head_dim=wl.head_dim, dtype=wl.dtype,
                 ctx=list(wl.ctx), mode=mode, window=wl.window_for(mode),
                 n_sink=wl.sinks_for(mode), alpha=wl.alpha, far_mix=wl.far_mix,
                 scale_slope=wl.scale_slope, scale_ref=wl.scale_ref, rope_theta=wl.rope_theta,
                 seed=wl.seed, extra_tokens=wl.draft_steps, **kw)


def _check_gather(s, b, t):
    L = int(s.ctx_lens[b])
    qp = int(s.q_pos[b, t])
    want = orc.selection_list(s.prm.mode, L, qp, s.prm, s.block_table[b].cpu().numpy(), 64)
    g = B.draft_attn_debug_gather(s.da.plan, s.q_pos, s.ctx_lens, s.block_table, b, t,
                                  capacity=want["position"].size)
    assert g["count"] == want["position"].size
    for k in ("position", "phys_slot", "key_rope_pos", "q_rope_pos", "segment"):
        assert np.array_equal(g[k].cpu().numpy().astype(np.int64), want[k].astype(np.int64)), k


@pytest.mark.parametrize("mode", ["full", "window"])
def test_tiny_window_fp32(mode):
    """B=1, 8/2 heads, d=64, fp32, keys 0..4095, query at 4096: every output."""
    wl = WL.WORKLOADS["tiny_window_fp32"]
    s = _setup(wl, mode)
    compare(s.run(), s.oracle(), "fp32", mode)
    _check_gather(s, 0, 0)
    assert s.status() == (B.DA_OK, 0)
    s.close()


def _draft_loop(wl, mode, check_steps, groups_per_step, seed):
    """Draft steps that each append one token then attend with the query at
    that token; checks the listed steps against the oracle."""
    s = _setup(wl, mode)
    L0 = wl.ctx[0]
    for step in range(wl.draft_steps):
        for b in range(wl.batch):
            s.append(b, L0 + step, L0 + step + 1)
        q = WL.randn(tuple(s.q.shape), s.q.dtype, s.dev, wl.seed * 16 + 1 + 7919 * step)
        q_pos = torch.full((wl.batch, wl.n_q), L0 + step, dtype=torch.int32, device=s.dev)
        lens = torch.full((wl.batch,), L0 + step + 1, dtype=torch.int32, device=s.dev)
        out = s.run(q=q, q_pos=q_pos, ctx_lens=lens)
        if step in check_steps:
            groups = sample_groups(wl.batch, wl.n_q, wl.num_kv_heads, groups_per_step,
                                   seed + step)
            want = s.oracle(groups, q=q, q_pos=q_pos, ctx=[L0 + step + 1] * wl.batch)
            compare(out, want, wl.dtype, f"{wl.name} {mode} step {step}")
            s.q_pos, s.ctx_lens = q_pos, lens
            _check_gather(s, 0, 0)
    assert s.status() == (B.DA_OK, 0)
    s.close()


@pytest.mark.parametrize("mode", ["full", "window"])
def test_mtp_draft_128k(mode):
    wl = WL.WORKLOADS["mtp_draft_128k"]
    _draft_loop(wl, mode, check_steps=(0, 1, 2, 3), groups_per_step=8 if mode == "window" else 3,
                seed=11)


@pytest.mark.parametrize("mode", ["full", "window"])
def test_mtp_draft_1m(mode):
    wl = WL.WORKLOADS["mtp_draft_1m"]
    _draft_loop(wl, mode, check_steps=(0, 5), groups_per_step=8 if mode == "window" else 2,
                seed=21)


@pytest.mark.parametrize("mode", ["fold", "full", "window"])
def test_fold_4x256k(mode):
    wl = WL.WORKLOADS["fold_4x256k"]
    s = _setup(wl, mode)
    out = s.run()
    groups = sample_groups(wl.batch, wl.n_q, wl.num_kv_heads, 4, 31)
    compare(out, s.oracle(groups), wl.dtype, f"fold_4x256k {mode}")
    _check_gather(s, 2, 0)
    assert s.status() == (B.DA_OK, 0)
    s.close()


@pytest.mark.parametrize("engine", ["auto", "cuda_core"])
def test_fold_4x256k_fp8_side_cache(engine):
    """The FOLD workload with its side cache as E4M3 codes (scale 1/64), in the
    configurations the benchmark times: the append writes the codes, sampled
    outputs match the oracle, which quantises the far keys the same way."""
    wl = WL.WORKLOADS["fold_4x256k"]
    s = _setup(wl, "fold", side_fp8_scale=1 / 64, engine=engine)
    assert s.da.info()["engine_name"] == ("mma" if engine == "auto" else "cuda_core")
    out = s.run()
    groups = sample_groups(wl.batch, wl.n_q, wl.num_kv_heads, 4, 37)
    compare(out, s.oracle(groups), wl.dtype, f"fold_4x256k fp8 {engine}")
    assert s.status() == (B.DA_OK, 0)
    s.close()


@pytest.mark.parametrize("mode", ["full", "window", "sharp"])
def test_ragged_tree_16x8(mode):
    wl = WL.WORKLOADS["ragged_tree_16x8"]
    s = _setup(wl, mode)
    info = s.da.info()
    # 32 rows: the tcgen05 engine scans the long selections, mma.sync the window
    assert info["engine_name"] == ("mma" if mode == "window" else "tc05")
    assert info["rows_per_kv_head"] == 32
    out = s.run()
    groups = sample_groups(wl.batch, wl.n_q, wl.num_kv_heads, 5, 41)
    # the shortest and the longest sequence always
    bmin, bmax = int(np.argmin(wl.ctx)), int(np.argmax(wl.ctx))
    groups += [(bmin, 7, 3), (bmax, 0, 5)]
    compare(out, s.oracle(sorted(set(groups))), wl.dtype, f"ragged {mode}")
    _check_gather(s, bmax, 7)
    assert s.status() == (B.DA_OK, 0)
    s.close()
