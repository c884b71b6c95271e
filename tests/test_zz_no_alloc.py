"""draft_attn_run_static: the entry point for callers that cannot allocate
device memory when they run the draft step (code inside another framework's
allocator or memory pool, or a runtime that only hands out its own buffers).
It runs on a fixed workspace inside the library's device image.  Checked
through the C ABI against draft_attn_run, on two calls in a row (the array
keeps the previous call's contents), and for its size limit.

Collected last on purpose: a run that stops at the first failure has run
every other test before this one."""
import pytest
import torch

from draft_attention_decode_b300 import binding as B
from tests.gpu_cases import Setup, compare

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu(cuda_lib):
    yield


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
    for _ in range(2):
        got = torch.full_like(want, float("nan"))
        B.draft_attn_run_static(s.da.plan, s.q, s.q_pos, s.ctx_lens, s.block_table, s.k_cache,
                                s.v_cache, s.k_side, got)
        torch.cuda.synchronize()
        compare(got, want.float().cpu().double().numpy(), "bf16", f"static {mode} {shape}")
    assert s.status() == (B.DA_OK, 0)
    s.close()


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
