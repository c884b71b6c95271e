"""The largest sizes a plan accepts, on the GPU against the float64 oracle:
the largest batch (1024 sequences of ragged, mostly short contexts, some
empty) and the largest draft tree (a 64-bit ancestor mask over 64 tree tokens,
queried by its last 32 tokens, 32 rows per KV head).  Every output the oracle
is asked for matches it; the device status stays clean."""
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


MAX_BATCH = 1024


@pytest.mark.parametrize("mode,kw", [("full", {}), ("window", dict(window=96, n_sink=4)),
                                     ("fold", dict(window=64, alpha=2.0, far_mix=0.5))],
                         ids=["full", "window", "fold"])
@pytest.mark.parametrize("nq", [1, 8], ids=["rows4", "rows32"])
def test_largest_batch(mode, kw, nq):
    rng = np.random.default_rng(3)
    ctx = [int(c) for c in rng.integers(0, 300, size=MAX_BATCH)]
    ctx[0], ctx[1], ctx[-1] = 0, 1, 4096           # empty, one key, a longer one last
    s = Setup(batch=MAX_BATCH, n_q=nq, num_q_heads=32, num_kv_heads=8, head_dim=128,
              dtype="bf16", ctx=ctx, mode=mode, seed=61, **kw)
    out = s.run()
    groups = sample_groups(MAX_BATCH, nq, 8, 24, seed=5)
    groups += [(0, 0, 0), (1, nq - 1, 7), (MAX_BATCH - 1, 0, 3)]
    compare(out, s.oracle(sorted(set(groups))), "bf16", f"batch {MAX_BATCH} {mode} q{nq}")
    assert torch.count_nonzero(out[0]) == 0           # the empty context
    assert s.status() == (B.DA_OK, 0)
    s.close()


@pytest.mark.parametrize("mode,kw", [("full", {}), ("window", dict(window=300, n_sink=4)),
                                     ("sharp", dict(scale_slope=0.05, scale_ref=256))],
                         ids=["full", "window", "sharp"])
def test_largest_tree(mode, kw):
    """tree_size 64 (the mask's width) with 32 queries over 8 KV heads (32 rows
    per KV head): query t is tree token 32 + t and sees its ancestors among
    all 64 tree tokens."""
    tree, nq = 64, 32
    L0 = [1500, 7, 200]
    ctx = [c + tree for c in L0]
    q_pos = [[c + (tree - nq) + t for t in range(nq)] for c in L0]
    s = Setup(batch=len(L0), n_q=nq, num_q_heads=8, num_kv_heads=8, head_dim=128,
              dtype="bf16", ctx=ctx, q_pos=q_pos, mode=mode, tree_size=tree, seed=67, **kw)
    masks = random_tree_masks(len(L0), tree, 9)[:, tree - nq:]
    tm = torch.tensor(np.ascontiguousarray(masks).view(np.int64), device=s.dev)
    out = s.run(tree_mask=tm)
    compare(out, s.oracle(tree_masks=masks), "bf16", f"tree {tree} {mode}")
    assert s.status() == (B.DA_OK, 0)
    s.close()
