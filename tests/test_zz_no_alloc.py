"""draft_attn_run_static: the entry point for callers that cannot allocate
device memory when they run the draft step (code inside another framework's
allocator or memory pool, or a runtime that only hands out its own buffers).
It runs on a fixed workspace inside the library's device image.  Checked
through the C ABI against the float64 oracle and against draft_attn_run, on
two calls in a row (the array keeps the previous call's contents); that it
allocates nothing; that it clears page counters a previous call left in the
array; and its size limit.

Collected last on purpose: a run that stops at the first failure has run
every other test before this one."""
import numpy as np
import pytest
import torch

from draft_attention_decode_b300 import binding as B
from tests.gpu_cases import Setup, compare

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu(cuda_lib):
    yield


def _static(s, out):
    B.draft_attn_run_static(s.da.plan, s.q, s.q_pos, s.ctx_lens, s.block_table, s.k_cache,
                            s.v_cache, s.k_side, out)


@pytest.mark.parametrize("mode,kw", [
    ("fold", dict(window=512, alpha=2.0, far_mix=0.5)),
    ("window", dict(window=300, n_sink=4)),
    ("sharp", dict(scale_slope=0.05, scale_ref=256)),
])
@pytest.mark.parametrize("shape", [(32, 8, 1), (32, 8, 8)], ids=["rows4", "rows32"])
def test_static_matches_run_twice(mode, kw, shape):
    h, hk, nq = shape
    s = Setup(batch=3, n_q=nq, num_q_heads=h, num_kv_heads=hk, head_dim=128, dtype="bf16",
              ctx=[5000, 130, 2047], mode=mode, seed=21, **kw)
    want = s.run()
    ref = s.oracle()
    outs = [torch.full_like(want, float("nan")) for _ in range(2)]
    for got in outs:
        _static(s, got)
        torch.cuda.synchronize()
        compare(got, want.float().cpu().double().numpy(), "bf16", f"static vs run {mode} {shape}")
        compare(got, ref, "bf16", f"static vs oracle {mode} {shape}")
    assert s.status() == (B.DA_OK, 0)
    s.close()


def test_static_allocates_nothing():
    """After a first call (which loads the module and looks the array's
    address up), further calls change neither the device's free memory nor
    what PyTorch's allocator holds."""
    s = Setup(batch=2, n_q=1, num_q_heads=32, num_kv_heads=8, head_dim=128, dtype="bf16",
              ctx=[3000, 700], mode="window", window=256, n_sink=4, seed=5)
    outs = [torch.full((2, 1, 32, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
            for _ in range(3)]
    _static(s, outs[0])
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    held0 = torch.cuda.memory_allocated()
    for got in outs[1:]:
        _static(s, got)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == held0
    assert free1 == free0, f"device free memory moved by {free0 - free1} bytes"
    ref = s.oracle()
    for got in outs:
        compare(got, ref, "bf16", "static window")
    s.close()


def test_static_clears_counters_left_in_the_array():
    """The array keeps whatever the previous call left.  A plan over one
    sequence (8 page counters, then its partial results from byte 256 on)
    leaves non-zero floats where a plan over twelve sequences keeps page
    counters 64..95; the second call must clear them before its kernel
    runs, or those heads never merge."""
    small = Setup(batch=1, n_q=1, num_q_heads=32, num_kv_heads=8, head_dim=128, dtype="bf16",
                  ctx=[4000], mode="full", seed=7)
    large = Setup(batch=12, n_q=1, num_q_heads=32, num_kv_heads=8, head_dim=128,
                  dtype="bf16", ctx=[300 + 157 * b for b in range(12)], mode="full", seed=8)
    out_small = torch.full((1, 1, 32, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    _static(small, out_small)
    torch.cuda.synchronize()
    compare(out_small, small.oracle(), "bf16", "static, one sequence")
    got = torch.full((12, 1, 32, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    _static(large, got)
    torch.cuda.synchronize()
    assert np.isfinite(got.float().cpu().numpy()).all()
    compare(got, large.oracle(), "bf16", "static, twelve sequences after one")
    want = large.run()
    compare(got, want.float().cpu().double().numpy(), "bf16", "static vs run")
    assert small.status() == (B.DA_OK, 0)
    small.close()
    large.close()


def test_static_rejects_plans_beyond_its_size():
    params = B.make_params(batch=1024, n_q=8, num_q_heads=32, num_kv_heads=8, head_dim=128,
                           num_pages=64, max_pages_per_seq=1, mode="full")
    plan, ws = B.draft_attn_plan(params, 0)
    try:
        assert ws > B.DA_STATIC_WORKSPACE_BYTES
        t = torch.zeros(1, dtype=torch.int32, device="cuda")
        with pytest.raises(B.DraftAttnError) as e:
            B.draft_attn_run_static(plan, t, t, t, t, t, t, None, t)
        assert e.value.code == B.DA_ERR_WORKSPACE_TOO_SMALL
    finally:
        B.draft_attn_plan_destroy(plan)
