"""Draft-tree attention with intra-tree ancestor masks on the GPU against the
float64 oracle: the last tree_size keys of each context are the tree's
tokens, and each query sees only its ancestors among them (and itself).
Every engine and mode; the gather hook bit-exact under the mask; an
all-ones mask bit-identical to no mask; SharpDraft's per-query |S|."""
import numpy as np
import pytest
import torch

import oracle.draft_attn_oracle as orc
from draft_attention_decode_b300 import binding as B
from tests.gpu_cases import Setup, compare

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu(cuda_lib):
    yield


def random_tree_masks(batch, n_q, seed):
    """Per sequence a random tree over n_q tokens (token 0 the root, every other
    token's parent an earlier token); mask[t] = t and its ancestors."""
    rng = np.random.default_rng(seed)
    masks = np.zeros((batch, n_q), dtype=np.uint64)
    for b in range(batch):
        for t in range(n_q):
            par = -1 if t == 0 else int(rng.integers(0, t))
            masks[b, t] = (np.uint64(1) << np.uint64(t)) | (masks[b, par] if par >= 0 else 0)
    return masks


def _setup(shape, dtype, mode, kw, L0, seed=19, **extra):
    h, hk, nq = shape
    ctx = [c + nq for c in L0]                      # the tree's tokens are the last keys
    q_pos = [[c + t for t in range(nq)] for c in L0]
    return Setup(batch=len(L0), n_q=nq, num_q_heads=h, num_kv_heads=hk, head_dim=128,
                 dtype=dtype, ctx=ctx, q_pos=q_pos, mode=mode, tree_size=nq, seed=seed,
                 **kw, **extra)


MODES = [("full", {}), ("window", dict(window=300, n_sink=4)),
         ("fold", dict(window=200, alpha=2.0, far_mix=0.5)),
         ("fold_sinks", dict(window=200, n_sink=4, alpha=2.0, far_mix=0.5)),
         ("sharp", dict(scale_slope=0.05, scale_ref=256))]


@pytest.mark.parametrize("mode,kw", MODES, ids=[m for m, _ in MODES])
@pytest.mark.parametrize("shape,dtype", [((32, 8, 8), "bf16"), ((16, 8, 4), "bf16"),
                                         ((8, 8, 4), "bf16"), ((8, 8, 2), "bf16"),
                                         ((8, 8, 4), "fp32"), ((8, 4, 4), "fp32")],
                         ids=["r32", "r8", "r4", "r2", "r4f32", "r8f32"])
def test_tree_parity(mode, kw, shape, dtype):
    L0 = [2500, 40, 777]
    s = _setup(shape, dtype, mode.split("_")[0], kw, L0)
    masks = random_tree_masks(len(L0), shape[2], 5)
    tm = torch.tensor(masks.view(np.int64), device=s.dev)
    out = s.run(tree_mask=tm)
    compare(out, s.oracle(tree_masks=masks), dtype, f"tree {mode} {shape} {dtype}")
    # the selection, bit-exact, for every query of one sequence
    bt = s.block_table.cpu().numpy()
    for t in range(shape[2]):
        g = B.draft_attn_debug_gather(s.da.plan, s.q_pos, s.ctx_lens, s.block_table, 0, t,
                                      capacity=L0[0] + shape[2] + 8, tree_mask=tm)
        want = orc.selection_list(s.prm.mode, L0[0] + shape[2], int(s.q_pos[0, t]), s.prm, bt[0], 64,
                                  tree_mask=int(masks[0, t]))
        assert g["count"] == want["position"].size
        for k in ("position", "phys_slot", "key_rope_pos", "q_rope_pos", "segment"):
            np.testing.assert_array_equal(g[k].cpu().numpy().astype(np.int64),
                                          want[k].astype(np.int64), err_msg=k)
    assert s.status() == (B.DA_OK, 0)
    s.close()


@pytest.mark.parametrize("mode,kw", MODES, ids=[m for m, _ in MODES])
def test_all_ones_mask_is_no_mask(mode, kw):
    s = _setup((32, 8, 8), "bf16", mode.split("_")[0], kw, [3000, 100])
    ones = torch.full((2, 8), -1, dtype=torch.int64, device=s.dev)
    a = s.run(tree_mask=ones).clone()
    b = s.run()
    assert torch.equal(a, b)
    s.close()


def test_chain_tree_is_causal_block():
    """A chain (every token the parent of the next) is a causal block: each
    query sees the cache and the tree tokens up to itself -- the same as
    attention over a context that ends at that query's token."""
    L0 = [1000]
    s = _setup((8, 8, 4), "bf16", "full", {}, L0)
    chain = np.array([[(1 << (t + 1)) - 1 for t in range(4)]], dtype=np.uint64)
    out = s.run(tree_mask=torch.tensor(chain.view(np.int64), device=s.dev))
    prm = orc.Params("full", rope_theta=1e4)
    q = s.q.float().cpu().numpy()
    for t in range(4):
        L = L0[0] + t + 1
        want = np.stack([orc.attend_group(q[0, t, h:h + 1], L0[0] + t,
                                          s.k_raw[0][:L, h].float().cpu().numpy(),
                                          s.v[0][:L, h].float().cpu().numpy(), L, prm)[0]
                         for h in range(8)])
        full = np.full(tuple(s.q.shape), np.nan)
        full[0, t] = want
        compare(out, full, "bf16", f"chain t={t}")
    s.close()
