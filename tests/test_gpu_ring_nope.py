"""Window-mode draft KV in a ring of pages, and NoPE (rope_theta = 0), on the
GPU against the float64 oracle.  The ring run must also equal, bit for bit,
the same draft steps on a cache that keeps every page: the physical page ids
never enter the arithmetic."""
import numpy as np
import pytest
import torch

import oracle.draft_attn_oracle as orc
from draft_attention_decode_b300 import binding as B
from draft_attention_decode_b300 import workloads as WL
from tests.gpu_cases import Setup, compare

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu(cuda_lib):
    yield


@pytest.mark.parametrize("mode,kw", [("full", {}), ("window", dict(window=300, n_sink=4)),
                                     ("fold", dict(window=200, alpha=2.0, far_mix=0.5)),
                                     ("sharp", dict(scale_slope=0.05, scale_ref=256))])
@pytest.mark.parametrize("shape", [(32, 8, 1), (64, 8, 1), (32, 8, 8)], ids=["r4", "r8", "r32"])
def test_nope_parity(mode, kw, shape):
    h, hk, nq = shape
    s = Setup(batch=2, n_q=nq, num_q_heads=h, num_kv_heads=hk, head_dim=128, dtype="bf16",
              ctx=[3000, 700], mode=mode, rope_theta=0.0, seed=13, **kw)
    compare(s.run(), s.oracle(), "bf16", f"nope {mode} {shape}")
    # the append stored the keys unrotated
    torch.cuda.synchronize()
    pg = int(s.block_table[0, 0])
    assert torch.equal(s.k_cache[pg, :, :64].float().cpu(),
                       s.k_raw[0][:64].permute(1, 0, 2).float().cpu())
    s.close()


def _ring_run(W, ns, L0, steps, H_q, H_kv, d, ring, seed):
    """Draft steps in window mode; returns the outputs and the oracle's."""
    dev = torch.device("cuda", 0)
    B_ = len(L0)
    cap = [c + steps for c in L0]
    max_pages = max((c + 63) // 64 for c in cap)
    k_raw = [WL.randn((c, H_kv, d), torch.bfloat16, dev, seed * 16 + 2 + 1000 * b)
             for b, c in enumerate(cap)]
    v = [WL.randn((c, H_kv, d), torch.bfloat16, dev, seed * 16 + 3 + 1000 * b)
         for b, c in enumerate(cap)]
    if ring:
        n_ring, n_sp = B.draft_attn_ring_size(W, ns)
        rows = [B.draft_attn_ring_block_table(max_pages, np.arange(b * n_ring, (b + 1) * n_ring),
                                              n_sp) for b in range(B_)]
        num_pages = B_ * n_ring
        chunk = 64 * (n_ring - n_sp)        # no two tokens of one append share a slot
    else:
        rows = [np.arange(b * max_pages, (b + 1) * max_pages) for b in range(B_)]
        num_pages = B_ * max_pages
        chunk = 1 << 20
    bt = torch.tensor(np.stack(rows), dtype=torch.int32, device=dev)
    da = B.DraftAttention(device=0, batch=B_, n_q=1, num_q_heads=H_q, num_kv_heads=H_kv,
                          head_dim=d, num_pages=num_pages, max_pages_per_seq=max_pages,
                          dtype="bf16", mode="window", window=W, n_sink=ns, rope_theta=1e4)
    kc = torch.full((num_pages, H_kv, 64, d), float("nan"), dtype=torch.bfloat16, device=dev)
    vc = torch.full_like(kc, float("nan"))
    for b, c in enumerate(L0):
        for s0 in range(0, c, chunk):
            s1 = min(c, s0 + chunk)
            pos = torch.arange(s0, s1, dtype=torch.int32, device=dev)[None]
            da.append_kv(k_raw[b][None, s0:s1].contiguous(), v[b][None, s0:s1].contiguous(), pos,
                         bt[b:b + 1], kc, vc)
    outs, wants = [], []
    prm = orc.Params("window", window=W, n_sink=ns, rope_theta=1e4)
    G = H_q // H_kv
    for st in range(steps):
        for b, c in enumerate(L0):
            pos = torch.tensor([[c + st]], dtype=torch.int32, device=dev)
            da.append_kv(k_raw[b][None, c + st:c + st + 1].contiguous(),
                         v[b][None, c + st:c + st + 1].contiguous(), pos, bt[b:b + 1], kc, vc)
        q = WL.randn((B_, 1, H_q, d), torch.bfloat16, dev, seed * 16 + 1 + 7919 * st)
        q_pos = torch.tensor([[c + st] for c in L0], dtype=torch.int32, device=dev)
        lens = torch.tensor([c + st + 1 for c in L0], dtype=torch.int32, device=dev)
        out = da.run(q, q_pos, lens, bt, kc, vc)
        torch.cuda.synchronize()
        outs.append(out.clone())
        want = np.full(tuple(q.shape), np.nan)
        qh = q.float().cpu().numpy()
        for b, c in enumerate(L0):
            L = c + st + 1
            for g in range(H_kv):
                want[b, 0, g * G:(g + 1) * G] = orc.attend_group(
                    qh[b, 0, g * G:(g + 1) * G], c + st, k_raw[b][:L, g].float().cpu().numpy(),
                    v[b][:L, g].float().cpu().numpy(), L, prm)
        wants.append(want)
    assert da.status() == (B.DA_OK, 0)
    da.close()
    return outs, wants


@pytest.mark.parametrize("W,ns", [(2048, 4), (200, 0), (64, 70)])
def test_ring_draft_loop(W, ns):
    """Window-mode draft steps crossing page boundaries, with the draft KV
    in a ring of ceil(W/64) + 1 (+ sink) pages per sequence."""
    L0 = [64 * 160 - 3, 64 * 41 + 10]
    steps = 6
    ring_out, wants = _ring_run(W, ns, L0, steps, 32, 8, 128, True, 31)
    full_out, _ = _ring_run(W, ns, L0, steps, 32, 8, 128, False, 31)
    for st in range(steps):
        compare(ring_out[st], wants[st], "bf16", f"ring W={W} ns={ns} step {st}")
        assert torch.equal(ring_out[st], full_out[st])
