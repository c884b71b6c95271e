"""GPU parity: the CUDA path through the C ABI against the float64 oracle on
the same seeded inputs.  Small shapes span several pages and a ragged tail;
every engine (rows per KV head 1, 2, 4, 8 on the CUDA cores; 9..32 on the
tensor cores), both dtypes and head dims, and every mode are covered, plus
the selection/gather hook bit-exact, the appended cache contents, split-count
and block-table invariance, and the degenerate cases."""
import numpy as np
import pytest
import torch

import oracle.draft_attn_oracle as orc
from draft_attention_decode_b300 import binding as B
from tests.gpu_cases import Setup, bf16_ulp, compare, equal_up_to_one_rounding

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu(cuda_lib):
    yield


# ---------------------------------------------------------------------------
# KV append + RoPE
# ---------------------------------------------------------------------------

def _fp32_slack(raw, d):
    """Bound on the FP32 rotation's error before the bf16 store, per
    rotate-half pair: the reduced angle rounded to float (half an ulp of pi),
    sincosf's own error and the products' roundings add up to about 5.5
    float32 ulps of |x| + |y|; 8 are allowed."""
    pair = np.abs(raw[..., : d // 2]) + np.abs(raw[..., d // 2:])
    return 8 * 2.0 ** -24 * np.concatenate([pair, pair], axis=-1)


@pytest.mark.parametrize("dtype,d,theta", [("bf16", 128, 1e4), ("bf16", 64, 1e6),
                                           ("fp32", 64, 1e4), ("fp32", 128, 1e6)])
def test_append_cache_contents(dtype, d, theta):
    ctx = [1000, 77]
    s = Setup(batch=2, n_q=1, num_q_heads=8, num_kv_heads=4, head_dim=d, dtype=dtype, ctx=ctx,
              mode="fold", window=64, alpha=2.0, far_mix=0.5, rope_theta=theta)
    # one far-out position too: 1M-scale angles
    bt = s.block_table.cpu().numpy()
    kc = s.k_cache.float().cpu().numpy().astype(np.float64)
    vc = s.v_cache.float().cpu().numpy()
    ks = s.k_side.float().cpu().numpy()
    for b, L in enumerate(ctx):
        pos = np.arange(L)
        phys, slot, _ = orc.page_slot(pos, bt[b], 64)
        raw = s.k_raw[b][:L].float().cpu().numpy().astype(np.float64)
        want = orc.append_rotated_keys(raw, pos, theta)            # [L, H_kv, d]
        got = kc[phys, :, slot, :]
        if dtype == "bf16":
            # the store rounds an FP32 rotation to nearest even: within one
            # bf16 ulp of the exact rotation, plus the FP32 rotation's own
            # error where x cos - y sin cancels to a tiny result
            assert (np.abs(got - want) <= bf16_ulp(want) + _fp32_slack(raw, d)).all()
            assert np.mean(got == orc.round_to_bf16(want)) > 0.97
        else:
            assert np.max(np.abs(got - want)) <= 2e-6 * max(1.0, np.abs(want).max())
        np.testing.assert_array_equal(ks[phys, :, slot, :], s.k_raw[b][:L].float().cpu().numpy())
        np.testing.assert_array_equal(vc[phys, :, slot, :], s.v[b][:L].float().cpu().numpy())
    assert s.status() == (B.DA_OK, 0)
    s.close()


def test_append_large_positions():
    """Angles at positions near 2^20 (1M context, theta 1e6) stay within one
    bf16 ulp: the angle is formed in double precision."""
    d = 128
    s = Setup(batch=1, n_q=1, num_q_heads=8, num_kv_heads=8, head_dim=d, dtype="bf16",
              ctx=[1048576 + 70], mode="full", rope_theta=1e6, fill=False)
    lo, hi = 1048576 - 64, 1048576 + 70
    s.append(0, lo, hi)
    torch.cuda.synchronize()
    bt = s.block_table.cpu().numpy()
    pos = np.arange(lo, hi)
    phys, slot, _ = orc.page_slot(pos, bt[0], 64)
    got = s.k_cache[torch.as_tensor(phys, device=s.dev), :, torch.as_tensor(slot, device=s.dev)]
    got = got.float().cpu().numpy().astype(np.float64)
    raw = s.k_raw[0][lo:hi].float().cpu().numpy().astype(np.float64)
    want = orc.append_rotated_keys(raw, pos, 1e6)
    assert (np.abs(got - want) <= bf16_ulp(want) + _fp32_slack(raw, d)).all()
    assert np.mean(got == orc.round_to_bf16(want)) > 0.97
    s.close()


def test_append_padding_positions_skipped():
    s = Setup(batch=1, n_q=1, num_q_heads=8, num_kv_heads=8, head_dim=64, dtype="bf16",
              ctx=[128], fill=False)
    k = s.k_raw[0][:4].unsqueeze(0).contiguous()
    v = s.v[0][:4].unsqueeze(0).contiguous()
    pos = torch.tensor([[5, -1, 7, -1]], dtype=torch.int32, device=s.dev)
    s.da.append_kv(k, v, pos, s.block_table, s.k_cache, s.v_cache)
    torch.cuda.synchronize()
    pg = int(s.block_table[0, 0])
    written = ~torch.isnan(s.v_cache[pg].float()).any(-1)      # [H_kv, 64]
    assert written[:, 5].all() and written[:, 7].all()
    assert int(written.sum()) == 2 * 8
    assert s.status() == (B.DA_OK, 0)
    s.close()


# ---------------------------------------------------------------------------
# Selection / page gather / RoPE positions, bit-exact
# ---------------------------------------------------------------------------

GATHER_CASES = [
    ("full", 0, 0), ("full", 1, 0), ("full", 4097, 0),
    ("window", 4096, 512, 4), ("window", 600, 512, 4), ("window", 516, 512, 4),
    ("window", 100, 512, 4), ("window", 130, 64, 0), ("window", 3, 1, 10), ("window", 200, 1, 0),
    ("fold", 5000, 2048), ("fold", 2049, 2048), ("fold", 2048, 2048), ("fold", 70, 2048),
    ("fold", 1, 1),
    # FOLD with sinks: sinks, far memory and window apart; sinks touching the
    # window (no far memory); sinks past a page; a sink page shared with the window
    ("fold", 5000, 2048, 4), ("fold", 2052, 2048, 4), ("fold", 2050, 2048, 4),
    ("fold", 700, 300, 100), ("fold", 60, 40, 4), ("fold", 1, 1, 4),
    ("sharp", 777, 0),
]


@pytest.mark.parametrize("case", GATHER_CASES, ids=str)
def test_debug_gather_bit_exact(case):
    mode, L, W = case[:3]
    ns = case[3] if len(case) > 3 else 0
    s = Setup(batch=2, n_q=3, num_q_heads=8, num_kv_heads=2, head_dim=64, dtype="bf16",
              ctx=[L, 64], mode=mode, window=max(W, 1), n_sink=ns, alpha=2.0, far_mix=0.5,
              fill=False)
    qp = s.q_pos.cpu().numpy()
    bt = s.block_table.cpu().numpy()
    for t in range(3):
        g = B.draft_attn_debug_gather(s.da.plan, s.q_pos, s.ctx_lens, s.block_table, 0, t,
                                      capacity=L + 8)
        want = orc.selection_list(mode, L, int(qp[0, t]), s.prm, bt[0], 64)
        assert g["count"] == want["position"].size
        for k in ("position", "phys_slot", "key_rope_pos", "q_rope_pos", "segment"):
            np.testing.assert_array_equal(g[k].cpu().numpy().astype(np.int64),
                                          want[k].astype(np.int64), err_msg=k)
    assert s.status() == (B.DA_OK, 0)
    s.close()


# ---------------------------------------------------------------------------
# Attention outputs vs the oracle (small, every engine and mode)
# ---------------------------------------------------------------------------

# (num_q_heads, num_kv_heads, n_q): rows per KV head 1, 2, 3->4, 4, 8, 12->32, 32
SHAPES = [(8, 8, 1), (16, 8, 1), (6, 2, 1), (8, 2, 1), (64, 8, 1), (8, 2, 2), (12, 4, 4),
          (32, 8, 8)]
MODES = [
    dict(mode="full"),
    dict(mode="window", window=300, n_sink=4),
    dict(mode="window", window=129, n_sink=0),
    dict(mode="fold", window=200, alpha=2.0, far_mix=0.5),
    dict(mode="fold", window=200, n_sink=70, alpha=2.0, far_mix=0.5),
    dict(mode="sharp", scale_slope=0.05, scale_ref=256),
]


def _rows(h, hk, nq):
    return (h // hk) * nq


def _mid(m):
    return m["mode"] + str(m.get("window", "")) + ("s%d" % m["n_sink"] if m.get("n_sink") else "")


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "h%d_%d_q%d" % s)
@pytest.mark.parametrize("mp", MODES, ids=_mid)
@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("bf16", 64), ("fp32", 64), ("fp32", 128)])
def test_parity_small(shape, mp, dtype, d):
    h, hk, nq = shape
    if dtype == "fp32" and _rows(h, hk, nq) > 8:
        pytest.skip("more than 8 rows per KV head is bf16-only (tensor cores)")
    ctx = [1000, 64, 3001, 5] if nq > 1 else [1000, 3001, 129]
    s = Setup(batch=len(ctx), n_q=nq, num_q_heads=h, num_kv_heads=hk, head_dim=d, dtype=dtype,
              ctx=ctx, seed=7, **mp)
    out = s.run()
    compare(out, s.oracle(), dtype, f"{mp} {shape} {dtype} d{d}")
    assert s.status() == (B.DA_OK, 0)
    s.close()


@pytest.mark.parametrize("shape,engine", [((64, 8, 1), "cuda_core"), ((32, 8, 2), "cuda_core"),
                                          ((32, 8, 1), "mma"), ((8, 8, 1), "mma"),
                                          ((16, 8, 1), "mma")],
                         ids=lambda x: str(x))
@pytest.mark.parametrize("mode", ["full", "fold", "window", "sharp", "fold_sinks"])
def test_engine_forced(shape, engine, mode):
    """Either engine, forced, computes the same attention for 1..8 rows."""
    h, hk, nq = shape
    ns = 4 if mode in ("window", "fold_sinks") else 0
    mode = "fold" if mode == "fold_sinks" else mode
    s = Setup(batch=2, n_q=nq, num_q_heads=h, num_kv_heads=hk, head_dim=128, dtype="bf16",
              ctx=[2500, 700], mode=mode, window=600, n_sink=ns,
              alpha=2.0, far_mix=0.5, scale_slope=0.05, scale_ref=256, seed=12, engine=engine)
    assert s.da.info()["engine_name"] == engine
    compare(s.run(), s.oracle(), "bf16", f"{mode} {shape} {engine}")
    s.close()


@pytest.mark.parametrize("num_ctas", [1, 2, 7, 148, 600])
@pytest.mark.parametrize("mode", ["full", "fold", "window", "fold_sinks"])
def test_split_count(num_ctas, mode):
    """Any number of persistent CTAs (hence of split pieces per sequence)
    gives the oracle's result."""
    ns = 4 if mode in ("window", "fold_sinks") else 0
    mode = "fold" if mode == "fold_sinks" else mode
    s = Setup(batch=3, n_q=1, num_q_heads=32, num_kv_heads=8, head_dim=128, dtype="bf16",
              ctx=[5000, 130, 2047], mode=mode, window=1000, n_sink=ns,
              alpha=2.0, far_mix=0.5, num_ctas=num_ctas, seed=3)
    compare(s.run(), s.oracle(), "bf16", f"{mode} ctas={num_ctas}")
    s.close()


def test_block_table_permutation_invariance():
    """The same keys behind another page permutation give a bit-identical
    output: the physical page never enters the arithmetic."""
    outs = []
    for perm_seed in (0, 1):
        s = Setup(batch=2, n_q=1, num_q_heads=32, num_kv_heads=8, head_dim=128, dtype="bf16",
                  ctx=[3000, 777], mode="fold", window=512, alpha=2.0, far_mix=0.5, seed=4,
                  fill=False)
        g = torch.Generator().manual_seed(100 + perm_seed)
        perm = torch.randperm(s.num_pages, generator=g).to(torch.int32).to(s.dev)
        bt = s.block_table.clone()
        valid = bt >= 0
        bt[valid] = perm[bt[valid].long()]
        s.block_table = bt.contiguous()
        for b, c in enumerate(s.ctx):
            s.append(b, 0, c)
        outs.append(s.run().clone())
        s.close()
    assert torch.equal(outs[0], outs[1])


# ---------------------------------------------------------------------------
# Degenerate cases and mode equivalences on the GPU
# ---------------------------------------------------------------------------

def test_empty_context_gives_zero():
    for mode in ("full", "window", "fold", "sharp"):
        s = Setup(batch=2, n_q=1, num_q_heads=8, num_kv_heads=2, head_dim=64, dtype="bf16",
                  ctx=[0, 70], mode=mode, window=16, alpha=2.0, far_mix=0.5, scale_slope=0.05)
        out = s.run()
        assert torch.count_nonzero(out[0]) == 0
        compare(out, s.oracle(), "bf16", mode)
        s.close()


def test_all_contexts_empty():
    s = Setup(batch=3, n_q=2, num_q_heads=8, num_kv_heads=2, head_dim=128, dtype="bf16",
              ctx=[0, 0, 0], mode="full")
    out = s.run()
    assert torch.count_nonzero(out) == 0
    s.close()


def test_single_key_returns_its_value():
    s = Setup(batch=1, n_q=1, num_q_heads=8, num_kv_heads=2, head_dim=128, dtype="fp32",
              ctx=[1], mode="full")
    out = s.run().cpu()
    v0 = s.v[0][0].cpu()
    for h in range(8):
        torch.testing.assert_close(out[0, 0, h], v0[h // 4], atol=1e-6, rtol=0)
    s.close()


def test_window_covering_context_equals_full():
    kw = dict(batch=2, n_q=1, num_q_heads=32, num_kv_heads=8, head_dim=128, dtype="bf16",
              ctx=[900, 1500], seed=5)
    full = Setup(mode="full", **kw)
    win = Setup(mode="window", window=1500, n_sink=4, **kw)
    a, b = full.run(), win.run()
    assert equal_up_to_one_rounding(a, b)   # window and full run different engine variants
    full.close()
    win.close()


def test_fold_without_far_memory_equals_window():
    kw = dict(batch=2, n_q=1, num_q_heads=32, num_kv_heads=8, head_dim=128, dtype="bf16",
              ctx=[300, 512], seed=6)
    fold = Setup(mode="fold", window=512, alpha=2.0, far_mix=0.5, **kw)
    win = Setup(mode="window", window=512, n_sink=0, **kw)
    assert equal_up_to_one_rounding(fold.run(), win.run())
    fold.close()
    win.close()


def test_fold_sinks_reduce_to_window_with_sinks():
    """FOLD with sinks is window attention with the same sinks when lambda = 0,
    and when the sinks reach the window (no far memory) at any lambda."""
    kw = dict(batch=2, n_q=1, num_q_heads=32, num_kv_heads=8, head_dim=128, dtype="bf16",
              ctx=[3000, 700], seed=16)
    for W, ns, lam in ((512, 4, 0.0), (512, 100, 0.0), (600, 2400, 0.7)):
        fold = Setup(mode="fold", window=W, n_sink=ns, alpha=2.0, far_mix=lam, **kw)
        win = Setup(mode="window", window=W, n_sink=ns, **kw)
        fo, wo = fold.run(), win.run()
        diff = (fo.float() - wo.float()).abs().max().item()
        assert equal_up_to_one_rounding(fo, wo), (W, ns, lam, diff)
        compare(fo, fold.oracle(), "bf16", f"fold W={W} sinks={ns} lambda={lam}")
        fold.close()
        win.close()


def test_fold_sinks_differ_from_fold():
    """The sinks move keys from the far memory into the local softmax: the
    output changes, and each one matches its own oracle."""
    kw = dict(batch=1, n_q=1, num_q_heads=32, num_kv_heads=8, head_dim=128, dtype="bf16",
              ctx=[4000], seed=17, mode="fold", window=256, alpha=2.0, far_mix=0.5)
    a = Setup(n_sink=0, **kw)
    b = Setup(n_sink=16, **kw)
    oa, ob = a.run(), b.run()
    compare(oa, a.oracle(), "bf16", "fold")
    compare(ob, b.oracle(), "bf16", "fold sinks")
    assert (oa.float() - ob.float()).abs().max().item() > 1e-3
    a.close()
    b.close()


def test_sharp_slope_zero_equals_full():
    kw = dict(batch=2, n_q=1, num_q_heads=32, num_kv_heads=8, head_dim=128, dtype="bf16",
              ctx=[9000, 100], seed=8)
    sh = Setup(mode="sharp", scale_slope=0.0, scale_ref=16, **kw)
    full = Setup(mode="full", **kw)
    assert torch.equal(sh.run(), full.run())
    sh.close()
    full.close()


# ---------------------------------------------------------------------------
# Faults found on the device are reported, never trapped
# ---------------------------------------------------------------------------

def test_bad_block_table_entry_sets_status():
    s = Setup(batch=1, n_q=1, num_q_heads=8, num_kv_heads=2, head_dim=64, dtype="bf16",
              ctx=[640], mode="full")
    s.block_table[0, 3] = s.num_pages + 5
    out = s.run()
    code, bits = s.status()
    assert code == B.DA_ERR_DEVICE_FAULT and bits & B.DA_STATUS_BAD_PAGE
    assert torch.isfinite(out.float()).all()
    assert s.status() == (B.DA_OK, 0)          # read-and-clear
    s.block_table[0, 3] = -1
    s.run()
    code, bits = s.status()
    assert code == B.DA_ERR_DEVICE_FAULT and bits & B.DA_STATUS_BAD_PAGE
    s.close()


def test_context_beyond_block_table_sets_status():
    s = Setup(batch=1, n_q=1, num_q_heads=8, num_kv_heads=2, head_dim=64, dtype="bf16",
              ctx=[640], mode="full")
    lens = torch.tensor([640 + 64 * 50], dtype=torch.int32, device=s.dev)
    out = s.run(ctx_lens=lens)
    code, bits = s.status()
    assert code == B.DA_ERR_DEVICE_FAULT and bits & B.DA_STATUS_BAD_CTX_LEN
    assert torch.isfinite(out.float()).all()
    s.close()


def test_bounded_wait_gives_up_and_reports():
    """A wait that nothing completes gives up after about a second, sets the
    timeout bit in the status word, and leaves the context usable: a normal
    call after it matches the oracle and reports nothing."""
    s = Setup(batch=1, n_q=1, num_q_heads=8, num_kv_heads=2, head_dim=64, dtype="bf16",
              ctx=[640], mode="full")
    assert s.status() == (B.DA_OK, 0)
    B.draft_attn_debug_wait_timeout(s.da.plan)
    code, bits = s.status()
    assert code == B.DA_ERR_DEVICE_FAULT and bits == B.DA_STATUS_WAIT_TIMEOUT
    assert s.status() == (B.DA_OK, 0)          # read-and-clear
    out = s.run()
    compare(out, s.oracle(), "bf16", "after a wait gave up")
    assert s.status() == (B.DA_OK, 0)
    s.close()


def test_workspace_too_small_rejected():
    s = Setup(batch=1, n_q=1, num_q_heads=8, num_kv_heads=2, head_dim=64, dtype="bf16",
              ctx=[64], mode="full")
    ws = torch.empty(16, dtype=torch.uint8, device=s.dev)
    with pytest.raises(B.DraftAttnError) as e:
        B.draft_attn_run(s.da.plan, s.q, s.q_pos, s.ctx_lens, s.block_table, s.k_cache,
                         s.v_cache, None, torch.empty_like(s.q), ws)
    assert e.value.code == B.DA_ERR_WORKSPACE_TOO_SMALL
    s.close()
