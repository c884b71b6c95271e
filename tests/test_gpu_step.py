"""draft_attn_step (append + attend in one call) on the GPU: the output and
every cache it writes are bit-identical to draft_attn_append_kv followed by
draft_attn_run(_tree), for every mode and engine, for tokens that the call
reads and tokens it does not, and a draft loop matches the oracle."""
import numpy as np
import pytest
import torch

from draft_attention_decode_b300 import binding as B
from draft_attention_decode_b300 import workloads as WL
from tests.gpu_cases import Setup, compare, sample_groups
from tests.test_gpu_tree import random_tree_masks

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu(cuda_lib):
    yield


def _same(a, b):
    return torch.equal(torch.isnan(a), torch.isnan(b)) and torch.equal(
        torch.nan_to_num(a.float()), torch.nan_to_num(b.float()))


MODES = [("full", {}), ("window", dict(window=300, n_sink=4)),
         ("fold", dict(window=200, alpha=2.0, far_mix=0.5)),
         ("sharp", dict(scale_slope=0.05, scale_ref=256))]


@pytest.mark.parametrize("mode,kw", MODES, ids=[m for m, _ in MODES])
@pytest.mark.parametrize("shape,n_new,visible,dtype", [
    ((32, 8, 1), 1, 1, "bf16"),          # a draft step, 4 rows (CUDA cores)
    ((64, 8, 1), 1, 1, "bf16"),          # 8 rows (tensor cores)
    ((32, 8, 8), 8, 8, "bf16"),          # a block of 8 drafted tokens, 32 rows
    ((32, 8, 1), 3, 1, "bf16"),          # two of the three tokens are past ctx_len
    ((8, 4, 1), 2, 2, "fp32"),
], ids=["r4", "r8", "r32", "unread", "fp32"])
def test_step_equals_append_then_run(mode, kw, shape, n_new, visible, dtype):
    h, hk, nq = shape
    L0 = [2000, 63, 777]
    s = Setup(batch=3, n_q=nq, num_q_heads=h, num_kv_heads=hk, head_dim=128, dtype=dtype,
              ctx=L0, mode=mode, extra_tokens=n_new, seed=23,
              q_pos=[[c + t for t in range(nq)] for c in L0], **kw)
    kc, vc = s.k_cache.clone(), s.v_cache.clone()
    ks = s.k_side.clone() if s.k_side is not None else None
    lens = torch.tensor([c + visible for c in L0], dtype=torch.int32, device=s.dev)
    k_new = torch.stack([s.k_raw[b][c:c + n_new] for b, c in enumerate(L0)]).contiguous()
    v_new = torch.stack([s.v[b][c:c + n_new] for b, c in enumerate(L0)]).contiguous()
    pos = torch.tensor([[c + j for j in range(n_new)] for c in L0], dtype=torch.int32,
                       device=s.dev)
    # reference: separate append and run
    s.da.append_kv(k_new, v_new, pos, s.block_table, s.k_cache, s.v_cache, s.k_side)
    want = s.run(ctx_lens=lens).clone()
    # one call
    got = s.da.step(k_new, v_new, pos, s.q, s.q_pos, lens, s.block_table, kc, vc, ks)
    torch.cuda.synchronize()
    assert torch.equal(got, want)
    assert _same(kc, s.k_cache) and _same(vc, s.v_cache)
    if ks is not None:
        assert _same(ks, s.k_side)
    assert s.status() == (B.DA_OK, 0)
    s.close()


@pytest.mark.parametrize("mode,kw", MODES, ids=[m for m, _ in MODES])
def test_step_with_tree_mask(mode, kw):
    L0 = [1500, 90]
    nq = 8
    s = Setup(batch=2, n_q=nq, num_q_heads=32, num_kv_heads=8, head_dim=128, dtype="bf16",
              ctx=L0, mode=mode, extra_tokens=nq, seed=29, tree_size=nq,
              q_pos=[[c + t for t in range(nq)] for c in L0], **kw)
    masks = torch.tensor(random_tree_masks(2, nq, 7).view(np.int64), device=s.dev)
    kc, vc = s.k_cache.clone(), s.v_cache.clone()
    ks = s.k_side.clone() if s.k_side is not None else None
    lens = torch.tensor([c + nq for c in L0], dtype=torch.int32, device=s.dev)
    k_new = torch.stack([s.k_raw[b][c:c + nq] for b, c in enumerate(L0)]).contiguous()
    v_new = torch.stack([s.v[b][c:c + nq] for b, c in enumerate(L0)]).contiguous()
    pos = torch.tensor([[c + j for j in range(nq)] for c in L0], dtype=torch.int32, device=s.dev)
    s.da.append_kv(k_new, v_new, pos, s.block_table, s.k_cache, s.v_cache, s.k_side)
    want = s.run(ctx_lens=lens, tree_mask=masks).clone()
    got = s.da.step(k_new, v_new, pos, s.q, s.q_pos, lens, s.block_table, kc, vc, ks,
                    tree_mask=masks)
    torch.cuda.synchronize()
    assert torch.equal(got, want)
    assert _same(kc, s.k_cache) and _same(vc, s.v_cache)
    s.close()


@pytest.mark.parametrize("mode", ["full", "window"])
def test_step_draft_loop_matches_oracle(mode):
    """Four draft steps at 20K context, each one call, against the oracle."""
    wl = WL.resized(WL.WORKLOADS["mtp_draft_128k"], 20000)
    s = Setup(batch=1, n_q=1, num_q_heads=32, num_kv_heads=8, head_dim=128, dtype="bf16",
              ctx=list(wl.ctx), mode=mode, window=2048, extra_tokens=4, seed=1)
    L0 = wl.ctx[0]
    for st in range(4):
        q = WL.randn(tuple(s.q.shape), s.q.dtype, s.dev, 16 + 1 + 7919 * st)
        pos = torch.tensor([[L0 + st]], dtype=torch.int32, device=s.dev)
        lens = torch.tensor([L0 + st + 1], dtype=torch.int32, device=s.dev)
        out = s.da.step(s.k_raw[0][None, L0 + st:L0 + st + 1].contiguous(),
                        s.v[0][None, L0 + st:L0 + st + 1].contiguous(), pos, q, pos, lens,
                        s.block_table, s.k_cache, s.v_cache)
        torch.cuda.synchronize()
        groups = sample_groups(1, 1, 8, 8, st)
        compare(out, s.oracle(groups, q=q, q_pos=pos, ctx=[L0 + st + 1]), "bf16",
                f"step {mode} {st}")
    assert s.status() == (B.DA_OK, 0)
    s.close()


def test_step_rejects_too_many_tokens():
    s = Setup(batch=1, n_q=1, num_q_heads=8, num_kv_heads=8, head_dim=128, dtype="bf16",
              ctx=[64], extra_tokens=40)
    k = s.k_raw[0][None, :33].contiguous()
    pos = torch.arange(33, dtype=torch.int32, device=s.dev)[None]
    with pytest.raises(B.DraftAttnError) as e:
        s.da.step(k, k, pos, s.q, s.q_pos, s.ctx_lens, s.block_table, s.k_cache, s.v_cache)
    assert e.value.code == B.DA_ERR_UNSUPPORTED
    s.close()


def test_step_error_leaves_cache_untouched():
    """A step whose attention arguments are invalid fails before the append
    is launched."""
    s = Setup(batch=1, n_q=1, num_q_heads=8, num_kv_heads=8, head_dim=128, dtype="bf16",
              ctx=[100], extra_tokens=1)
    kc = s.k_cache.clone()
    k = s.k_raw[0][None, 100:101].contiguous()
    pos = torch.tensor([[100]], dtype=torch.int32, device=s.dev)
    lens = torch.tensor([101], dtype=torch.int32, device=s.dev)
    out = torch.empty_like(s.q)
    with pytest.raises(B.DraftAttnError) as e:
        B.draft_attn_step(s.da.plan, k, k, pos, s.q, s.q_pos, lens, s.block_table, s.k_cache,
                          s.v_cache, None, out, s.da.workspace[:16], None, None)
    assert e.value.code == B.DA_ERR_WORKSPACE_TOO_SMALL
    torch.cuda.synchronize()
    assert _same(kc, s.k_cache)          # unwritten slots hold NaN
    s.close()


@pytest.mark.parametrize("mode,kw,cluster", [
    ("full", {}, 0), ("window", dict(window=300, n_sink=4), 0),
    ("window", dict(window=300, n_sink=4), -1), ("fold", dict(window=200, alpha=2.0, far_mix=0.5), 0)],
    ids=["full", "window-cluster", "window-flat", "fold"])
@pytest.mark.parametrize("shape", [(32, 8, 1), (64, 8, 1)], ids=["r4", "r8"])
def test_tables_ready_changes_nothing(mode, kw, cluster, shape):
    """tables_ready = 1 lets the attention kernel read the context lengths,
    positions and block table before it waits for the previous kernel.  A
    draft loop of back-to-back steps (each kernel may start while the one
    before it still appends and attends) gives outputs and caches bit-identical
    to the same loop without it."""
    h, hk, nq = shape
    L0 = [2000, 63, 777]
    steps = 4
    outs, caches = [], []
    for tr in (0, 1):
        s = Setup(batch=3, n_q=nq, num_q_heads=h, num_kv_heads=hk, head_dim=128, dtype="bf16",
                  ctx=L0, mode=mode, extra_tokens=steps, seed=31, cluster_ctas=cluster,
                  tables_ready=tr, **kw)
        qs = [WL.randn(tuple(s.q.shape), s.q.dtype, s.dev, 900 + st) for st in range(steps)]
        k_new = [torch.stack([s.k_raw[b][c + st:c + st + 1] for b, c in enumerate(L0)]).contiguous()
                 for st in range(steps)]
        v_new = [torch.stack([s.v[b][c + st:c + st + 1] for b, c in enumerate(L0)]).contiguous()
                 for st in range(steps)]
        pos = [torch.tensor([[c + st] for c in L0], dtype=torch.int32, device=s.dev)
               for st in range(steps)]
        lens = [torch.tensor([c + st + 1 for c in L0], dtype=torch.int32, device=s.dev)
                for st in range(steps)]
        res = [torch.empty_like(s.q) for _ in range(steps)]
        torch.cuda.synchronize()
        for st in range(steps):   # no host work or other kernel between the steps
            s.da.step(k_new[st], v_new[st], pos[st], qs[st], pos[st], lens[st], s.block_table,
                      s.k_cache, s.v_cache, s.k_side, out=res[st])
        torch.cuda.synchronize()
        assert s.status() == (B.DA_OK, 0)
        outs.append([r.clone() for r in res])
        caches.append((s.k_cache.clone(), s.v_cache.clone()))
        s.close()
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a, b)
    assert _same(caches[0][0], caches[1][0]) and _same(caches[0][1], caches[1][1])
