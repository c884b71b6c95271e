"""FOLD with the side cache as FP8 E4M3 codes (da_params.side_fp8): the append
kernel's bytes equal the oracle's codes bit for bit, and the attention over
the quantised far memory matches the float64 oracle, which quantises the same
way, at every row count and engine, split, with sinks, draft trees and the
rotated-K ring; keys outside the saturation limit clamp the same way on both
sides."""
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


def _side_bytes(s, b, L):
    """Side-cache bytes of positions 0..L-1 of sequence b, [L, H_kv, d]."""
    bt = s.block_table[b].cpu().numpy()
    pos = np.arange(L)
    pages = bt[pos // 64]
    side = s.k_side.cpu().numpy()
    return side[pages, :, pos % 64, :]


@pytest.mark.parametrize("scale", [1 / 64, 1.0, 1 / 512], ids=["s64", "s1", "s512-saturating"])
def test_append_writes_e4m3_codes(scale):
    s = Setup(batch=2, n_q=1, num_q_heads=32, num_kv_heads=8, head_dim=128, dtype="bf16",
              ctx=[700, 130], mode="fold", window=100, alpha=2.0, far_mix=0.5, seed=31,
              side_fp8_scale=scale)
    torch.cuda.synchronize()
    for b, L in enumerate(s.ctx):
        got = _side_bytes(s, b, L)
        want = orc.side_fp8_codes(s.k_raw[b][:L].float().cpu().numpy(), scale)
        np.testing.assert_array_equal(got, want)
    if scale == 1 / 512:   # |k| > 448 / 512 saturates: make sure the case occurs
        assert (np.abs(s.k_raw[0][:700].float().cpu().numpy()) > 448 * scale).any()
    assert s.status() == (B.DA_OK, 0)
    s.close()


# rows per KV head 1, 2, 4 (CUDA cores), 8, 16, 32 (tensor cores)
SHAPES = [(8, 8, 1), (16, 8, 1), (32, 8, 1), (64, 8, 1), (32, 8, 4), (32, 8, 8)]


@pytest.mark.parametrize("engine", ["auto", "cuda_core"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda x: "h%d_%d_q%d" % x)
@pytest.mark.parametrize("kw", [dict(), dict(n_sink=70), dict(num_ctas=7), dict(num_ctas=1)],
                         ids=["plain", "sinks", "ctas7", "ctas1"])
def test_fold_fp8_parity(shape, kw, engine):
    h, hk, nq = shape
    rows = (h // hk) * nq
    if engine == "cuda_core" and rows > 4:
        pytest.skip("the CUDA-core engine reads an FP8 side cache at up to 4 rows")
    s = Setup(batch=3, n_q=nq, num_q_heads=h, num_kv_heads=hk, head_dim=128, dtype="bf16",
              ctx=[3000, 129, 1000], mode="fold", window=200, alpha=2.0, far_mix=0.5, seed=33,
              side_fp8_scale=1 / 64, engine=engine, **kw)
    assert s.da.info()["engine_name"] == ("cuda_core" if engine == "cuda_core" else "mma")
    compare(s.run(), s.oracle(), "bf16", f"fold fp8 {shape} {kw}")
    assert s.status() == (B.DA_OK, 0)
    s.close()


@pytest.mark.parametrize("shape,engine", [((8, 8, 1), "cuda_core"), ((32, 8, 1), "cuda_core"),
                                          ((32, 8, 1), "auto"), ((64, 8, 1), "auto"),
                                          ((32, 8, 8), "auto")],
                         ids=["r1-core", "r4-core", "r4-mma", "r8-mma", "r32-mma"])
def test_fold_fp8_head_dim_64(shape, engine):
    """64-byte E4M3 key rows (unswizzled): the append's bytes and the attention
    against the oracle on both engines."""
    h, hk, nq = shape
    s = Setup(batch=2, n_q=nq, num_q_heads=h, num_kv_heads=hk, head_dim=64, dtype="bf16",
              ctx=[2600, 300], mode="fold", window=200, n_sink=4, alpha=2.0, far_mix=0.5,
              seed=39, side_fp8_scale=1 / 32, engine=engine)
    torch.cuda.synchronize()
    for b, L in enumerate(s.ctx):
        np.testing.assert_array_equal(
            _side_bytes(s, b, L), orc.side_fp8_codes(s.k_raw[b][:L].float().cpu().numpy(), 1 / 32))
    compare(s.run(), s.oracle(), "bf16", f"fold fp8 d64 {shape} {engine}")
    assert s.status() == (B.DA_OK, 0)
    s.close()


@pytest.mark.parametrize("h,engine", [(32, "cuda_core"), (64, "auto"), (32, "auto")],
                         ids=["r4-core", "r8-mma", "r4-mma"])
def test_fold_fp8_saturating_scale(h, engine):
    """A scale that saturates part of the keys: both sides clamp to 448."""
    s = Setup(batch=1, n_q=1, num_q_heads=h, num_kv_heads=8, head_dim=128, dtype="bf16",
              ctx=[2500], mode="fold", window=256, alpha=2.0, far_mix=0.7, seed=34,
              side_fp8_scale=1 / 256, engine=engine)
    compare(s.run(), s.oracle(), "bf16", f"fold fp8 saturating {h} {engine}")
    s.close()


def test_fold_fp8_tiny_scale_tensor_cores():
    """A tiny scale (codes far from 1): the tensor-core engine applies it to the
    scores, not to its f16 queries."""
    s = Setup(batch=1, n_q=1, num_q_heads=64, num_kv_heads=8, head_dim=128, dtype="bf16",
              ctx=[3000], mode="fold", window=256, alpha=2.0, far_mix=0.7, seed=38,
              side_fp8_scale=1e-3)
    compare(s.run(), s.oracle(), "bf16", "fold fp8 scale 1e-3")
    s.close()


def test_fold_fp8_differs_from_bf16_side_only_by_quantisation():
    """Same inputs with a bf16 and an FP8 side cache: outputs differ (the far
    keys changed), the local-only case (lambda = 0) is bit-identical."""
    kw = dict(batch=1, n_q=1, num_q_heads=32, num_kv_heads=8, head_dim=128, dtype="bf16",
              ctx=[5000], mode="fold", window=300, alpha=2.0, seed=35)
    for engine in ("mma", "cuda_core"):       # the same engine on both sides
        for lam in (0.0, 0.5):
            a = Setup(far_mix=lam, engine=engine, **kw)
            b = Setup(far_mix=lam, side_fp8_scale=1 / 64, engine=engine, **kw)
            oa, ob = a.run(), b.run()
            if lam == 0.0:
                assert torch.equal(oa, ob), engine
            else:
                assert not torch.equal(oa, ob)
                compare(ob, b.oracle(), "bf16", f"fold fp8 lambda 0.5 {engine}")
            a.close()
            b.close()


def test_fold_fp8_tree():
    """Four tree tokens (4 rows per KV head with 8/8 heads) over an FP8 side cache."""
    L0 = [2000, 300]
    nq = 4
    s = Setup(batch=2, n_q=nq, num_q_heads=8, num_kv_heads=8, head_dim=128, dtype="bf16",
              ctx=[c + nq for c in L0], q_pos=[[c + t for t in range(nq)] for c in L0],
              mode="fold", window=150, alpha=2.0, far_mix=0.5, tree_size=nq, seed=36,
              side_fp8_scale=1 / 32)
    masks = np.array([[1, 3, 5, 9], [1, 3, 7, 15]], dtype=np.uint64)
    tm = torch.tensor(masks.view(np.int64), device=s.dev)
    compare(s.run(tree_mask=tm), s.oracle(tree_masks=masks), "bf16", "fold fp8 tree")
    s.close()


@pytest.mark.parametrize("ns,engine", [(0, "auto"), (70, "auto"), (70, "cuda_core")],
                         ids=["plain", "sinks70", "sinks70-core"])
def test_fold_fp8_with_k_ring(ns, engine):
    """The rotated K in a ring (sink pages in their own slots) and the side cache
    in FP8: the side cache is the one full-length copy of K, at one byte per
    element; outputs equal the paged run's bit for bit."""
    dev = torch.device("cuda", 0)
    W, L, H_kv, d = 300, 4000, 8, 128
    ref = Setup(batch=1, n_q=1, num_q_heads=32, num_kv_heads=H_kv, head_dim=d, dtype="bf16",
                ctx=[L], mode="fold", window=W, n_sink=ns, alpha=2.0, far_mix=0.5, seed=37,
                side_fp8_scale=1 / 64, engine=engine)
    want = ref.run()
    compare(want, ref.oracle(), "bf16", f"fold fp8 sinks={ns} {engine}")
    SP = (ns + 63) // 64
    R = SP + (W + 63) // 64 + 1
    da = B.DraftAttention(device=0, batch=1, n_q=1, num_q_heads=32, num_kv_heads=H_kv,
                          head_dim=d, num_pages=ref.num_pages,
                          max_pages_per_seq=ref.block_table.shape[1], dtype="bf16", mode="fold",
                          window=W, n_sink=ns, alpha=2.0, far_mix=0.5, k_ring_pages=R,
                          side_fp8=1, side_scale=1 / 64, engine=engine)
    kc = torch.full((R, H_kv, 64, d), float("nan"), dtype=torch.bfloat16, device=dev)
    vc = torch.full_like(ref.v_cache, float("nan"))
    ks = torch.full_like(ref.k_side, 0x7F)
    chunk = 64 * (R - SP)                 # page-aligned: no two positions share a slot
    for s0 in range(0, L, chunk):
        n = min(chunk, L - s0)
        pos = torch.arange(s0, s0 + n, dtype=torch.int32, device=dev).unsqueeze(0)
        da.append_kv(ref.k_raw[0][s0:s0 + n].unsqueeze(0).contiguous(),
                     ref.v[0][s0:s0 + n].unsqueeze(0).contiguous(), pos, ref.block_table,
                     kc, vc, ks)
    out = da.run(ref.q, ref.q_pos, ref.ctx_lens, ref.block_table, kc, vc, ks)
    torch.cuda.synchronize()
    assert torch.equal(out, want)
    assert torch.equal(ks, ref.k_side)
    assert da.status() == (B.DA_OK, 0)
    da.close()
    ref.close()


def test_fp8_side_refused_on_the_wide_cuda_core_engine():
    p = B.make_params(batch=1, n_q=1, num_q_heads=64, num_kv_heads=8, head_dim=128,
                      num_pages=10, max_pages_per_seq=10, mode="fold", window=64, alpha=2.0,
                      far_mix=0.5, side_fp8=1, side_scale=1.0, engine="cuda_core")
    with pytest.raises(B.DraftAttnError) as e:
        B.draft_attn_plan(p, 0)
    assert e.value.code == B.DA_ERR_UNSUPPORTED
