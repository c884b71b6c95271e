"""Window mode's cluster partition on the GPU: one thread-block cluster of C
CTAs per (sequence, KV head), each CTA an equal share of that head's pages,
the partial results merged through distributed shared memory.  Against the
float64 oracle at every cluster size (1 to 16, and more CTAs than pages),
every engine, both dtypes and head dims, with sinks, ragged and empty
contexts and draft-tree masks; equal to the flat partition up to one
rounding; and the plan's automatic choice."""
import numpy as np
import pytest
import torch

from draft_attention_decode_b300 import binding as B
from tests.gpu_cases import Setup, compare, equal_up_to_one_rounding, sample_groups
from tests.test_gpu_tree import random_tree_masks

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu(cuda_lib):
    yield


def _same(a, b):
    """Bit-equal, NaN slots (never-written cache slots) included."""
    return torch.equal(torch.isnan(a), torch.isnan(b)) and torch.equal(
        torch.nan_to_num(a.float()), torch.nan_to_num(b.float()))


# (num_q_heads, num_kv_heads, n_q): rows per KV head 1, 4, 8, 16, 32
SHAPES = [(8, 8, 1), (32, 8, 1), (64, 8, 1), (32, 8, 4), (32, 8, 8)]


@pytest.mark.parametrize("cluster", [1, 2, 3, 5, 8, 9, 10, 16])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "h%d_%d_q%d" % s)
@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("bf16", 64), ("fp32", 128)])
def test_cluster_parity(cluster, shape, dtype, d):
    h, hk, nq = shape
    if dtype == "fp32" and (h // hk) * nq > 8:
        pytest.skip("more than 8 rows per KV head is bf16-only (tensor cores)")
    # ragged: a window well inside the context, one shorter than it, a single
    # key, an empty context, and a window of exactly one page boundary
    ctx = [3001, 129, 1, 0, 1024]
    rows = (h // hk) * nq
    try:
        s = Setup(batch=len(ctx), n_q=nq, num_q_heads=h, num_kv_heads=hk, head_dim=d,
                  dtype=dtype, ctx=ctx, mode="window", window=300, n_sink=4,
                  cluster_ctas=cluster, seed=31)
    except B.DraftAttnError as e:
        # rank 0 keeps one partial per CTA of the cluster in shared memory:
        # a forced size whose partials cannot fit is refused
        rk = 8 if rows <= 8 and rows > 4 else (rows if rows <= 4 else (16 if rows <= 16 else 32))
        slot = (((2 * rk + 3) // 4) * 4 + rk * d) * 4
        assert e.code == B.DA_ERR_UNSUPPORTED and cluster * slot > 64 * 1024, (cluster, rows, d)
        pytest.skip(f"{cluster} partials of {rows} rows do not fit in shared memory")
    assert s.da.info()["cluster_ctas"] == cluster
    out = s.run()
    compare(out, s.oracle(), dtype, f"cluster {cluster} {shape} {dtype} d{d}")
    assert s.status() == (B.DA_OK, 0)
    s.close()


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "h%d_%d_q%d" % s)
@pytest.mark.parametrize("window,n_sink", [(2048, 0), (4096, 4), (129, 0), (64, 70)])
def test_cluster_equals_flat(shape, window, n_sink):
    """The same inputs through the automatic cluster partition and through
    the flat one: on the CUDA cores (FP32 throughout, only the summation
    order differs) equal up to one rounding of the result; on the tensor
    cores, whose probabilities are rounded to bf16 against each piece's own
    running maximum, within 2e-3 of each other; both match the oracle."""
    h, hk, nq = shape
    ctx = [20000, 5000, 2100]
    kw = dict(batch=3, n_q=nq, num_q_heads=h, num_kv_heads=hk, head_dim=128, dtype="bf16",
              ctx=ctx, mode="window", window=window, n_sink=n_sink, seed=41)
    a = Setup(cluster_ctas=0, **kw)
    assert a.da.info()["cluster_ctas"] >= 1
    b = Setup(cluster_ctas=-1, **kw)
    assert b.da.info()["cluster_ctas"] == 0
    oa, ob = a.run(), b.run()
    if (h // hk) * nq <= 4:
        assert equal_up_to_one_rounding(oa, ob)
    else:
        assert (oa.float() - ob.float()).abs().max().item() <= 2e-3
    groups = sample_groups(3, nq, hk, 6, seed=1)
    compare(oa, a.oracle(groups), "bf16", f"cluster auto {shape} W{window}")
    a.close()
    b.close()


@pytest.mark.parametrize("shape", [(32, 8, 8), (16, 8, 4), (8, 8, 4)], ids=["r32", "r8", "r4"])
@pytest.mark.parametrize("cluster", [1, 4, 16])
def test_cluster_tree_masks(shape, cluster):
    h, hk, nq = shape
    L0 = [2500, 40, 777]
    ctx = [c + nq for c in L0]
    q_pos = [[c + t for t in range(nq)] for c in L0]
    try:
        s = Setup(batch=3, n_q=nq, num_q_heads=h, num_kv_heads=hk, head_dim=128, dtype="bf16",
                  ctx=ctx, q_pos=q_pos, mode="window", window=300, n_sink=4, tree_size=nq,
                  cluster_ctas=cluster, seed=19)
    except B.DraftAttnError as e:
        # 32 rows x 16 CTAs: rank 0 cannot hold 16 partials of 16 KB
        assert e.code == B.DA_ERR_UNSUPPORTED and (h // hk) * nq * cluster > 256
        pytest.skip("the cluster's partials do not fit in shared memory")
    masks = random_tree_masks(3, nq, 5)
    tm = torch.tensor(masks.view(np.int64), device=s.dev)
    compare(s.run(tree_mask=tm), s.oracle(tree_masks=masks), "bf16", f"tree cluster {cluster}")
    assert s.status() == (B.DA_OK, 0)
    s.close()


def test_cluster_step_equals_append_then_run():
    """draft_attn_step on the cluster partition (its set-up overlaps the
    append): bit-identical to the append followed by the run."""
    L0 = [2000, 63, 777]
    s = Setup(batch=3, n_q=1, num_q_heads=32, num_kv_heads=8, head_dim=128, dtype="bf16",
              ctx=L0, mode="window", window=300, n_sink=4, extra_tokens=1, seed=23,
              q_pos=[[c] for c in L0])
    assert s.da.info()["cluster_ctas"] >= 1
    kc, vc = s.k_cache.clone(), s.v_cache.clone()
    lens = torch.tensor([c + 1 for c in L0], dtype=torch.int32, device=s.dev)
    k_new = torch.stack([s.k_raw[b][c:c + 1] for b, c in enumerate(L0)]).contiguous()
    v_new = torch.stack([s.v[b][c:c + 1] for b, c in enumerate(L0)]).contiguous()
    pos = torch.tensor([[c] for c in L0], dtype=torch.int32, device=s.dev)
    s.da.append_kv(k_new, v_new, pos, s.block_table, s.k_cache, s.v_cache, None)
    want = s.run(ctx_lens=lens).clone()
    got = s.da.step(k_new, v_new, pos, s.q, s.q_pos, lens, s.block_table, kc, vc, None)
    torch.cuda.synchronize()
    assert torch.equal(got, want)
    assert _same(kc, s.k_cache) and _same(vc, s.v_cache)
    compare(got, s.oracle(ctx=[c + 1 for c in L0]), "bf16", "cluster step")
    assert s.status() == (B.DA_OK, 0)
    s.close()


def test_cluster_automatic_choice():
    """The plan takes the cluster partition in window mode when one cluster
    per (sequence, KV head) fits on the GPU at once (at most 16 CTAs each,
    never more than the window has pages), and the flat one otherwise, in
    other modes, or when a flat-partition knob is set."""
    def info(**kw):
        base = dict(batch=1, n_q=1, num_q_heads=32, num_kv_heads=8, head_dim=128,
                    num_pages=4096, max_pages_per_seq=4096, mode="window", window=2048)
        base.update(kw)
        p = B.make_params(**base)
        plan, _ = B.draft_attn_plan(p, 0)
        try:
            return B.draft_attn_plan_info(plan)
        finally:
            B.draft_attn_plan_destroy(plan)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    i = info()
    assert 1 <= i["cluster_ctas"] <= 16 and i["num_ctas"] == 8 * i["cluster_ctas"]
    assert info(window=64)["cluster_ctas"] <= 2            # two pages at most
    assert info(batch=(sms // 8) + 1)["cluster_ctas"] == 0  # more heads than SMs
    assert info(mode="full")["cluster_ctas"] == 0
    assert info(num_ctas=64)["cluster_ctas"] == 0
    assert info(cluster_ctas=-1)["cluster_ctas"] == 0
    assert info(cluster_ctas=3)["cluster_ctas"] == 3
    # The fewest CTAs for the longest stretch: one CTA fewer would lengthen it
    # (a window of W keys plus sinks spans at most ceil(W / 64) + 1 pages, and
    # one more for the sinks).
    for w, ns in ((2048, 0), (4096, 4), (1000, 0)):
        c = info(window=w, n_sink=ns)["cluster_ctas"]
        pmax = (1 if ns else 0) + -(-w // 64) + 1
        longest = -(-pmax // c)
        assert c == 1 or -(-pmax // (c - 1)) > longest, (w, ns, c)


def test_cluster_long_window_sampled():
    """The million-token shape's window (4096 + 4 sinks, 66 pages per head)
    on the cluster partition: 8 rows per KV head, sampled against the oracle."""
    L = 100000
    s = Setup(batch=1, n_q=1, num_q_heads=64, num_kv_heads=8, head_dim=128, dtype="bf16",
              ctx=[L], mode="window", window=4096, n_sink=4, rope_theta=1e6, seed=3)
    assert s.da.info()["cluster_ctas"] >= 1
    out = s.run()
    compare(out, s.oracle(groups=[(0, 0, g) for g in (0, 3, 7)]), "bf16", "1M-shape window")
    assert s.status() == (B.DA_OK, 0)
    s.close()


@pytest.mark.parametrize("n_new", [1, 2, 8, 9])
def test_cluster_step_appends_in_one_launch(n_new):
    """draft_attn_step on the cluster partition appends up to 8 tokens per
    sequence inside the attention kernel (more go through the append kernel):
    either way outputs and caches are bit-identical to draft_attn_append_kv
    followed by draft_attn_run, with the new tokens read in the same call."""
    L0 = [2000, 63, 777]
    s = Setup(batch=3, n_q=1, num_q_heads=64, num_kv_heads=8, head_dim=128, dtype="bf16",
              ctx=L0, mode="window", window=300, n_sink=4, extra_tokens=n_new, seed=37,
              q_pos=[[c + n_new - 1] for c in L0])
    assert s.da.info()["cluster_ctas"] >= 1
    kc, vc = s.k_cache.clone(), s.v_cache.clone()
    lens = torch.tensor([c + n_new for c in L0], dtype=torch.int32, device=s.dev)
    k_new = torch.stack([s.k_raw[b][c:c + n_new] for b, c in enumerate(L0)]).contiguous()
    v_new = torch.stack([s.v[b][c:c + n_new] for b, c in enumerate(L0)]).contiguous()
    pos = torch.tensor([[c + j for j in range(n_new)] for c in L0], dtype=torch.int32,
                       device=s.dev)
    s.da.append_kv(k_new, v_new, pos, s.block_table, s.k_cache, s.v_cache, None)
    want = s.run(ctx_lens=lens).clone()
    got = s.da.step(k_new, v_new, pos, s.q, s.q_pos, lens, s.block_table, kc, vc, None)
    torch.cuda.synchronize()
    assert torch.equal(got, want)
    assert _same(kc, s.k_cache) and _same(vc, s.v_cache)
    compare(got, s.oracle(ctx=[c + n_new for c in L0]), "bf16", f"step {n_new}")
    assert s.status() == (B.DA_OK, 0)
    s.close()


def test_cluster_step_bad_position_sets_status():
    """A new token past the block table: the one-launch step flags it (as the
    append kernel does), writes nothing for it and still attends."""
    L0 = [1000]
    s = Setup(batch=1, n_q=1, num_q_heads=32, num_kv_heads=8, head_dim=128, dtype="bf16",
              ctx=L0, mode="window", window=300, n_sink=4, extra_tokens=1, seed=41,
              q_pos=[[1000]])
    kc, vc = s.k_cache.clone(), s.v_cache.clone()
    far = s.block_table.shape[1] * 64 + 5
    pos = torch.tensor([[far]], dtype=torch.int32, device=s.dev)
    k_new = s.k_raw[0][1000:1001].unsqueeze(0).contiguous()
    v_new = s.v[0][1000:1001].unsqueeze(0).contiguous()
    lens = torch.tensor(L0, dtype=torch.int32, device=s.dev)
    got = s.da.step(k_new, v_new, pos, s.q, s.q_pos, lens, s.block_table, kc, vc, None)
    torch.cuda.synchronize()
    assert s.status() == (B.DA_ERR_DEVICE_FAULT, B.DA_STATUS_BAD_POSITION)
    assert _same(kc, s.k_cache) and _same(vc, s.v_cache)
    compare(got, s.oracle(), "bf16", "step, bad position")
    s.close()
