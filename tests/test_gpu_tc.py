"""The tcgen05 engine (draft_attention_decode_b300 engine "tc05": tensor-core
MMAs with TMEM accumulators, two pages per step) against the float64 oracle:
every mode, 1 to 32 query rows per KV head, ragged contexts (odd page counts,
partial pages, a single key, an empty context), draft-tree masks, both
partitions, split counts, FOLD with sinks and with its rotated keys in a
ring, and draft_attn_step."""
import numpy as np
import pytest
import torch

from draft_attention_decode_b300 import binding as B
from tests.gpu_cases import Setup, compare, sample_groups
from tests.test_gpu_tree import random_tree_masks

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu(cuda_lib):
    yield


MODES = [
    ("full", {}),
    ("window", dict(window=300, n_sink=4)),
    ("window_flat", dict(window=300, n_sink=4, cluster_ctas=-1)),
    ("fold", dict(window=200, alpha=2.0, far_mix=0.5)),
    ("fold_sinks", dict(window=200, n_sink=70, alpha=2.0, far_mix=0.5)),
    ("sharp", dict(scale_slope=0.05, scale_ref=256)),
]
# (num_q_heads, num_kv_heads, n_q): rows per KV head 32, 16, 8, 4, 1
SHAPES = [(32, 8, 8), (16, 8, 8), (32, 8, 2), (32, 8, 1), (8, 8, 1)]


@pytest.mark.parametrize("mode,kw", MODES, ids=[m for m, _ in MODES])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "h%d_%d_q%d" % s)
def test_tc_parity(mode, kw, shape):
    h, hk, nq = shape
    ctx = [1000, 64, 3001, 5, 0, 129]
    s = Setup(batch=len(ctx), n_q=nq, num_q_heads=h, num_kv_heads=hk, head_dim=128,
              dtype="bf16", ctx=ctx, mode=mode.split("_")[0], seed=7, engine="tc05", **kw)
    assert s.da.info()["engine_name"] == "tc05"
    compare(s.run(), s.oracle(), "bf16", f"tc05 {mode} {shape}")
    assert s.status() == (B.DA_OK, 0)
    s.close()


@pytest.mark.parametrize("num_ctas", [1, 7, 148, 300])
@pytest.mark.parametrize("mode", ["full", "fold"])
def test_tc_split_count(num_ctas, mode):
    s = Setup(batch=3, n_q=8, num_q_heads=32, num_kv_heads=8, head_dim=128, dtype="bf16",
              ctx=[5000, 130, 2047], mode=mode, window=1000, alpha=2.0, far_mix=0.5,
              num_ctas=num_ctas, seed=3, engine="tc05")
    compare(s.run(), s.oracle(), "bf16", f"tc05 {mode} ctas {num_ctas}")
    assert s.status() == (B.DA_OK, 0)
    s.close()


@pytest.mark.parametrize("mode,kw", [m for m in MODES if m[0] != "window_flat"],
                         ids=[m for m, _ in MODES if m != "window_flat"])
def test_tc_tree_masks(mode, kw):
    L0 = [2500, 40, 777]
    nq = 8
    ctx = [c + nq for c in L0]
    q_pos = [[c + t for t in range(nq)] for c in L0]
    s = Setup(batch=3, n_q=nq, num_q_heads=32, num_kv_heads=8, head_dim=128, dtype="bf16",
              ctx=ctx, q_pos=q_pos, mode=mode.split("_")[0], tree_size=nq, seed=19,
              engine="tc05", **kw)
    masks = random_tree_masks(3, nq, 5)
    tm = torch.tensor(masks.view(np.int64), device=s.dev)
    compare(s.run(tree_mask=tm), s.oracle(tree_masks=masks), "bf16", f"tc05 tree {mode}")
    assert s.status() == (B.DA_OK, 0)
    s.close()


def test_tc_rising_maxima():
    """Scores that keep rising along the context (no rotation: NoPE, so that
    a key's alignment with the query is what it was built to be): keys move
    from far against the query to near it, so each piece's reference maxima
    are raised many times and O^T is rescaled in TMEM between PVs; the
    winning scores stay small, so the bf16 query's rounding stays far below
    the tolerance."""
    d, L0 = 128, [4000, 900]
    s = Setup(batch=2, n_q=8, num_q_heads=32, num_kv_heads=8, head_dim=d, dtype="bf16",
              ctx=L0, mode="full", seed=5, engine="tc05", rope_theta=0.0, fill=False)
    qf = s.q.float()                                   # [B, n_q, H_q, d]
    for b, c in enumerate(L0):
        # per KV head: the mean direction of its 32 query rows
        qd = qf[b].reshape(8, 8, 4, d).permute(2, 0, 1, 3).reshape(8, 32, d).mean(1)
        qd = qd / qd.norm(dim=-1, keepdim=True)        # [H_kv, d]
        a = torch.linspace(-60.0, 0.0, c, device=s.dev)[:, None, None]
        k = 0.5 * s.k_raw[b][:c].float() + a * qd[None]
        s.k_raw[b][:c] = k.to(torch.bfloat16)
        s.append(b, 0, c)
    compare(s.run(), s.oracle(), "bf16", "tc05 rising maxima")
    assert s.status() == (B.DA_OK, 0)
    s.close()


def test_tc_matches_mma_engine_on_the_ragged_shape():
    """The ragged draft-tree shape (32 rows) at reduced contexts: the tcgen05
    engine and the mma.sync engine both match the oracle."""
    from draft_attention_decode_b300 import workloads as WL
    lens = [min(c, 40000) // 4 for c in WL.WORKLOADS["ragged_tree_16x8"].ctx]
    kw = dict(batch=16, n_q=8, num_q_heads=32, num_kv_heads=8, head_dim=128, dtype="bf16",
              ctx=lens, mode="sharp", scale_slope=0.05, scale_ref=4096, seed=4)
    a = Setup(engine="tc05", **kw)
    groups = sample_groups(16, 8, 8, 12, seed=2)
    ref = a.oracle(groups)
    compare(a.run(), ref, "bf16", "tc05 ragged")
    assert a.status() == (B.DA_OK, 0)
    a.close()


def test_tc_step_equals_append_then_run():
    L0 = [2000, 63, 777]
    nq = 8
    s = Setup(batch=3, n_q=nq, num_q_heads=32, num_kv_heads=8, head_dim=128, dtype="bf16",
              ctx=L0, mode="full", extra_tokens=nq, seed=23, engine="tc05",
              q_pos=[[c + t for t in range(nq)] for c in L0])
    kc, vc = s.k_cache.clone(), s.v_cache.clone()
    lens = torch.tensor([c + nq for c in L0], dtype=torch.int32, device=s.dev)
    k_new = torch.stack([s.k_raw[b][c:c + nq] for b, c in enumerate(L0)]).contiguous()
    v_new = torch.stack([s.v[b][c:c + nq] for b, c in enumerate(L0)]).contiguous()
    pos = torch.tensor([[c + j for j in range(nq)] for c in L0], dtype=torch.int32, device=s.dev)
    s.da.append_kv(k_new, v_new, pos, s.block_table, s.k_cache, s.v_cache, None)
    want = s.run(ctx_lens=lens).clone()
    got = s.da.step(k_new, v_new, pos, s.q, s.q_pos, lens, s.block_table, kc, vc, None)
    torch.cuda.synchronize()
    assert torch.equal(got, want)
    compare(got, s.oracle(ctx=[c + nq for c in L0]), "bf16", "tc05 step")
    assert s.status() == (B.DA_OK, 0)
    s.close()
