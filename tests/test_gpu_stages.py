"""Pipeline depth (da_params.stages) on the GPU: every depth that fits gives
bit-identical outputs (the depth changes when pages load, never the order of
the arithmetic), the automatic depth is the one the plan reports, and a depth
that does not fit in shared memory is refused at plan time."""
import pytest
import torch

from draft_attention_decode_b300 import binding as B
from tests.gpu_cases import Setup, compare

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu(cuda_lib):
    yield


# window mode pins its cluster size: the automatic one may shrink when a deep
# pipeline leaves rank 0 less room for its partials, and another split of the
# keys is another summation order
MODES = [("full", {}, 6), ("window", dict(window=700, n_sink=4, cluster_ctas=4), 4),
         ("fold", dict(window=600, alpha=2.0, far_mix=0.5), 6)]


@pytest.mark.parametrize("mode,kw,auto", MODES, ids=[m for m, _, _ in MODES])
def test_every_depth_gives_the_same_output(mode, kw, auto):
    base = dict(batch=2, n_q=1, num_q_heads=32, num_kv_heads=8, head_dim=128, dtype="bf16",
                ctx=[6000, 2500], mode=mode, seed=44, **kw)
    s = Setup(**base)
    assert s.da.info()["stages"] == auto
    want = s.run().clone()
    compare(want, s.oracle(groups=[(0, 0, 3), (1, 0, 6)]), "bf16", f"stages auto {mode}")
    for st in (2, 3, 5, 6):
        p = B.make_params(batch=2, n_q=1, num_q_heads=32, num_kv_heads=8, head_dim=128,
                          num_pages=s.num_pages, max_pages_per_seq=s.block_table.shape[1],
                          mode=mode, stages=st, **{k: v for k, v in kw.items()})
        plan, ws_bytes = B.draft_attn_plan(p, 0)
        ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=s.dev)
        out = torch.empty_like(s.q)
        B.draft_attn_run(plan, s.q, s.q_pos, s.ctx_lens, s.block_table, s.k_cache, s.v_cache,
                         s.k_side, out, ws)
        torch.cuda.synchronize()
        info = B.draft_attn_plan_info(plan)
        B.draft_attn_plan_destroy(plan)
        assert info["stages"] == st
        assert torch.equal(out, want), f"{mode} stages={st}"
    s.close()


def test_too_deep_a_pipeline_is_refused():
    p = B.make_params(batch=1, n_q=1, num_q_heads=32, num_kv_heads=8, head_dim=128,
                      num_pages=10, max_pages_per_seq=10, stages=8)
    with pytest.raises(B.DraftAttnError) as e:
        B.draft_attn_plan(p, 0)
    assert e.value.code == B.DA_ERR_UNSUPPORTED
