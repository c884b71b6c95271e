"""FOLD with the rotated keys in a ring (da_params.k_ring_pages): the rotated K
cache keeps only the local window, R pages per sequence, while the far memory
reads the unrotated side cache, which is then the only full-length copy of K.
The outputs of a draft loop that wraps the ring must equal, bit for bit, the
same loop on a fully paged rotated cache (the slots never enter the
arithmetic), and match the float64 oracle."""
import numpy as np
import pytest
import torch

import oracle.draft_attn_oracle as orc
from draft_attention_decode_b300 import binding as B
from draft_attention_decode_b300 import workloads as WL
from tests.gpu_cases import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu(cuda_lib):
    yield


def _fold_run(W, L0, steps, H_q, H_kv, ring, seed, d=128, alpha=2.0, lam=0.5, fused=False,
              n_sink=0):
    """FOLD draft steps; returns the outputs, the oracle's and the K cache."""
    dev = torch.device("cuda", 0)
    B_ = len(L0)
    cap = [c + steps for c in L0]
    max_pages = max((c + 63) // 64 for c in cap)
    k_raw = [WL.randn((c, H_kv, d), torch.bfloat16, dev, seed * 16 + 2 + 1000 * b)
             for b, c in enumerate(cap)]
    v = [WL.randn((c, H_kv, d), torch.bfloat16, dev, seed * 16 + 3 + 1000 * b)
         for b, c in enumerate(cap)]
    rows = [np.random.default_rng(seed + b).permutation(max_pages) + b * max_pages
            for b in range(B_)]
    bt = torch.tensor(np.stack(rows), dtype=torch.int32, device=dev)
    num_pages = B_ * max_pages
    SP = (n_sink + 63) // 64                 # the sinks' pages keep their own slots
    R = SP + (W + 63) // 64 + 1 if ring else 0
    da = B.DraftAttention(device=0, batch=B_, n_q=1, num_q_heads=H_q, num_kv_heads=H_kv,
                          head_dim=d, num_pages=num_pages, max_pages_per_seq=max_pages,
                          dtype="bf16", mode="fold", window=W, alpha=alpha, far_mix=lam,
                          rope_theta=1e4, k_ring_pages=R, n_sink=n_sink)
    k_pages = B_ * R if ring else num_pages
    kc = torch.full((k_pages, H_kv, 64, d), float("nan"), dtype=torch.bfloat16, device=dev)
    vc = torch.full((num_pages, H_kv, 64, d), float("nan"), dtype=torch.bfloat16, device=dev)
    ks = torch.full_like(vc, float("nan"))
    # every sequence in each append (ring rows are sequence indices); no two
    # positions of one append share a ring slot (page-aligned chunks of R - SP
    # pages); padding positions are -1
    chunk = 64 * (R - SP) if ring else 1 << 20
    for s0 in range(0, max(L0), chunk):
        n = min(chunk, max(L0) - s0)
        kk = torch.zeros((B_, n, H_kv, d), dtype=torch.bfloat16, device=dev)
        vv = torch.zeros_like(kk)
        pos = torch.full((B_, n), -1, dtype=torch.int32, device=dev)
        for b, c in enumerate(L0):
            m = max(0, min(n, c - s0))
            kk[b, :m] = k_raw[b][s0:s0 + m]
            vv[b, :m] = v[b][s0:s0 + m]
            pos[b, :m] = torch.arange(s0, s0 + m, dtype=torch.int32, device=dev)
        da.append_kv(kk, vv, pos, bt, kc, vc, ks)
    outs, wants = [], []
    prm = orc.Params("fold", window=W, n_sink=n_sink, alpha=alpha, far_mix=lam, rope_theta=1e4)
    G = H_q // H_kv
    for st in range(steps):
        k_new = torch.stack([k_raw[b][c + st:c + st + 1] for b, c in enumerate(L0)]).contiguous()
        v_new = torch.stack([v[b][c + st:c + st + 1] for b, c in enumerate(L0)]).contiguous()
        pos = torch.tensor([[c + st] for c in L0], dtype=torch.int32, device=dev)
        q = WL.randn((B_, 1, H_q, d), torch.bfloat16, dev, seed * 16 + 1 + 7919 * st)
        lens = torch.tensor([c + st + 1 for c in L0], dtype=torch.int32, device=dev)
        if fused:
            out = da.step(k_new, v_new, pos, q, pos, lens, bt, kc, vc, ks)
        else:
            da.append_kv(k_new, v_new, pos, bt, kc, vc, ks)
            out = da.run(q, pos, lens, bt, kc, vc, ks)
        torch.cuda.synchronize()
        outs.append(out.clone())
        want = np.full(tuple(q.shape), np.nan)
        if st % 3 == 0:   # the oracle on every third step
            qh = q.float().cpu().numpy()
            for b, c in enumerate(L0):
                L = c + st + 1
                for g in range(H_kv):
                    want[b, 0, g * G:(g + 1) * G] = orc.attend_group(
                        qh[b, 0, g * G:(g + 1) * G], c + st,
                        k_raw[b][:L, g].float().cpu().numpy(),
                        v[b][:L, g].float().cpu().numpy(), L, prm)
        wants.append(want)
    assert da.status() == (B.DA_OK, 0)
    da.close()
    return outs, wants, kc, bt


@pytest.mark.parametrize("W,shape,fused,ns", [(200, (32, 8), False, 0), (2048, (32, 8), True, 0),
                                              (64, (64, 8), False, 0), (130, (16, 2), True, 0),
                                              (200, (32, 8), False, 4), (130, (64, 8), True, 70)],
                         ids=["w200-r4", "w2048-r4-step", "w64-r8", "w130-r8-step",
                              "w200-r4-sinks4", "w130-r8-step-sinks70"])
def test_fold_ring_draft_loop(W, shape, fused, ns):
    """Draft steps crossing page boundaries; the initial fill wraps the ring
    many times; the sinks' pages keep their own slots."""
    H_q, H_kv = shape
    L0 = [64 * 70 - 3, 64 * 21 + 10]
    steps = 9
    ring_out, wants, _, _ = _fold_run(W, L0, steps, H_q, H_kv, True, 37, fused=fused, n_sink=ns)
    paged_out, _, _, _ = _fold_run(W, L0, steps, H_q, H_kv, False, 37, fused=fused, n_sink=ns)
    for st in range(steps):
        assert torch.equal(ring_out[st], paged_out[st]), f"step {st}"
        if st % 3 == 0:
            compare(ring_out[st], wants[st], "bf16", f"fold ring W={W} step {st}")


def test_fold_ring_slots_hold_the_window():
    """After the loop, ring slot b*R + (P mod R) holds the rotated keys of
    page P for every page of the local window, equal to the paged cache's."""
    W, L0, steps = 200, [64 * 30 + 5], 4
    _, _, kr, bt = _fold_run(W, L0, steps, 32, 8, True, 41)
    _, _, kp, _ = _fold_run(W, L0, steps, 32, 8, False, 41)
    R = (W + 63) // 64 + 1
    L = L0[0] + steps
    for P in range((L - W) // 64, (L - 1) // 64 + 1):
        lo = max(L - W, P * 64) - P * 64
        hi = min(L, P * 64 + 64) - P * 64
        got = kr[P % R, :, lo:hi]
        want = kp[int(bt[0, P]), :, lo:hi]
        assert torch.equal(got, want), f"page {P}"



def test_fold_ring_append_needs_every_sequence():
    dev = torch.device("cuda", 0)
    da = B.DraftAttention(device=0, batch=2, n_q=1, num_q_heads=8, num_kv_heads=8, head_dim=128,
                          num_pages=8, max_pages_per_seq=4, dtype="bf16", mode="fold", window=100,
                          alpha=2.0, far_mix=0.5, k_ring_pages=3)
    kc = torch.zeros((6, 8, 64, 128), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros((8, 8, 64, 128), dtype=torch.bfloat16, device=dev)
    k = torch.zeros((1, 1, 8, 128), dtype=torch.bfloat16, device=dev)
    pos = torch.zeros((1, 1), dtype=torch.int32, device=dev)
    bt = torch.arange(8, dtype=torch.int32, device=dev).view(2, 4)
    with pytest.raises(B.DraftAttnError) as e:
        da.append_kv(k, k, pos, bt[1:], kc, vc, vc.clone())
    assert e.value.code == B.DA_ERR_INVALID_ARG
    da.close()
