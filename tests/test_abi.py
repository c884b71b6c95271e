"""The C-ABI library on the CPU: it loads, exports every function the header
declares, validates parameters on the host and reports errors by code.  No
call here launches anything."""
import ctypes
import os
import shutil
import subprocess

import pytest

from draft_attention_decode_b300 import binding as B

pytestmark = pytest.mark.skipif(not os.path.exists(B.LIB_PATH), reason="library not built")


def test_exports_every_header_symbol():
    lib = B.load_library()
    names = B.header_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    assert B.draft_attn_version() == 101


def test_error_strings():
    for code in (0, -1, -2, -3, -4, -5):
        s = B.draft_attn_error_string(code)
        assert s and s != "unknown error"
    assert B.draft_attn_error_string(-99) == "unknown error"


def _ok_params(**kw):
    base = dict(batch=1, n_q=1, num_q_heads=32, num_kv_heads=8, head_dim=128, num_pages=100,
                max_pages_per_seq=100)
    base.update(kw)
    return B.make_params(**base)


@pytest.mark.parametrize("kw,code", [
    ({}, 0),
    (dict(mode="window", window=2048), 0),
    (dict(mode="window", window=2048, n_sink=4), 0),
    (dict(mode="fold", window=2048, alpha=2.0, far_mix=0.5), 0),
    (dict(mode="sharp", scale_slope=0.05, scale_ref=4096), 0),
    (dict(n_q=8), 0),                                  # 32 rows: tensor-core engine
    (dict(head_dim=64, dtype="fp32", num_q_heads=8, num_kv_heads=2), 0),
    (dict(head_dim=96), -1),
    (dict(num_q_heads=30), -1),                        # not a multiple of H_kv
    (dict(batch=0), -1),
    (dict(batch=1025), -1),
    (dict(page_size=32), -1),
    (dict(mode="window", window=0), -1),
    (dict(mode="window", window=16, n_sink=-1), -1),
    (dict(mode="fold", window=16, alpha=0.0), -1),
    (dict(mode="fold", window=16, alpha=2.0, far_mix=1.5), -1),
    (dict(mode="fold", window=16, alpha=2.0, n_sink=4), 0),       # sinks join the local softmax
    (dict(mode="fold", window=16, alpha=2.0, n_sink=-1), -1),
    (dict(mode="fold", window=200, alpha=2.0, far_mix=0.5, n_sink=4, k_ring_pages=5), -1),
    (dict(mode="fold", window=200, alpha=2.0, far_mix=0.5, n_sink=4, k_ring_pages=6), 0),
    (dict(mode="fold", window=200, alpha=2.0, far_mix=0.5, n_sink=70, k_ring_pages=6), -1),
    (dict(mode="fold", window=200, alpha=2.0, far_mix=0.5, n_sink=70, k_ring_pages=7), 0),
    # FOLD side cache as FP8 E4M3 codes
    (dict(mode="fold", window=200, alpha=2.0, far_mix=0.5, side_fp8=1, side_scale=0.05), 0),
    (dict(mode="fold", window=200, alpha=2.0, far_mix=0.5, side_fp8=1, side_scale=0.05,
          k_ring_pages=5, n_sink=0), 0),
    (dict(mode="fold", window=200, alpha=2.0, far_mix=0.5, side_fp8=1, side_scale=0.0), -1),
    (dict(mode="fold", window=200, alpha=2.0, far_mix=0.5, side_fp8=1,
          side_scale=float("inf")), -1),
    (dict(mode="fold", window=200, alpha=2.0, far_mix=0.5, side_fp8=2, side_scale=1.0), -1),
    (dict(mode="fold", window=200, alpha=2.0, far_mix=0.5, side_scale=1.0), -1),
    (dict(mode="window", window=200, side_fp8=1, side_scale=1.0), -1),
    (dict(mode="fold", window=200, alpha=2.0, far_mix=0.5, side_fp8=1, side_scale=1.0,
          head_dim=64), 0),
    (dict(mode="fold", window=200, alpha=2.0, far_mix=0.5, side_fp8=1, side_scale=1.0,
          dtype="fp32"), -2),
    (dict(mode="fold", window=200, alpha=2.0, far_mix=0.5, side_fp8=1, side_scale=1.0,
          num_q_heads=64), 0),                       # 8 rows per KV head: tensor cores
    (dict(mode="fold", window=200, alpha=2.0, far_mix=0.5, side_fp8=1, side_scale=1.0,
          num_q_heads=64, engine="cuda_core"), -2),
    (dict(mode="fold", window=200, alpha=2.0, far_mix=0.5, side_fp8=1, side_scale=1.0,
          engine="mma"), 0),
    (dict(mode="sharp", scale_slope=-1.0), -1),
    (dict(mode="sharp", scale_ref=0), -1),
    (dict(rope_theta=0.0), 0),                         # NoPE
    (dict(rope_theta=-1.0), -1),
    (dict(rope_theta=float("inf")), -1),
    (dict(mode=7), -1),
    (dict(num_ctas=-3), -1),
    (dict(num_pages=40_000_000), -1),                  # 32-bit TMA row index would overflow
    (dict(n_q=16), -2),                                # 64 rows per KV head
    (dict(n_q=4, dtype="fp32"), -2),                   # >8 rows needs bf16 tensor cores
    (dict(n_q=4, engine="cuda_core"), -2),             # 16 rows: CUDA cores stop at 8
    (dict(engine="mma"), 0),                           # 4 rows forced onto tensor cores
    (dict(engine="cuda_core", num_q_heads=64), 0),     # 8 rows forced onto CUDA cores
    (dict(engine="mma", dtype="fp32"), -2),            # tensor-core path is bf16 only
    (dict(engine=3), 0),                               # tcgen05 engine
    (dict(engine=4), -1),
    (dict(engine=3, head_dim=64), -2),
    (dict(engine=3, dtype="fp32", num_q_heads=8), -2),
    (dict(tree_size=8), 0),
    (dict(tree_size=65), -1),
    (dict(tree_size=-1), -1),
    (dict(mode="window", window=16, tree_size=32), -1),   # tree must fit in the window
    (dict(mode="fold", window=64, alpha=2.0, far_mix=0.5, tree_size=64), 0),
    # FOLD's rotated keys in a ring of R >= ceil(W / 64) + 1 pages per sequence
    (dict(mode="fold", window=200, alpha=2.0, far_mix=0.5, k_ring_pages=5), 0),
    (dict(mode="fold", window=200, alpha=2.0, far_mix=0.5, k_ring_pages=4), -1),
    (dict(mode="fold", window=128, alpha=2.0, far_mix=0.5, k_ring_pages=3), 0),
    (dict(mode="full", k_ring_pages=5), -1),
    (dict(mode="window", window=200, k_ring_pages=5), -1),
    # the cluster partition: window mode, 1..16 CTAs per cluster (-1 = flat)
    (dict(mode="window", window=2048, cluster_ctas=16), 0),
    (dict(mode="window", window=2048, cluster_ctas=1), 0),
    (dict(mode="window", window=2048, cluster_ctas=-1), 0),
    (dict(mode="window", window=2048, cluster_ctas=17), -1),
    (dict(mode="window", window=2048, cluster_ctas=-2), -1),
    (dict(mode="full", cluster_ctas=-1), 0),
    (dict(mode="full", cluster_ctas=4), -1),
    (dict(mode="fold", window=64, alpha=2.0, far_mix=0.5, cluster_ctas=2), -1),
    (dict(mode="window", window=2048, cluster_ctas=4, num_ctas=20), -1),
])
def test_check_params(kw, code):
    assert B.draft_attn_check_params(_ok_params(**kw)) == code


@pytest.mark.parametrize("v,code", [(0, 0), (1, 0), (2, -1), (-1, -1)])
def test_tables_ready_is_a_flag(v, code):
    p = _ok_params()
    p.tables_ready = v
    assert B.draft_attn_check_params(p) == code


def test_null_params_and_plan_rejected():
    lib = B.load_library()
    assert lib.draft_attn_check_params(None) == -1
    assert lib.draft_attn_plan(None, 0, None, None) == -1
    assert lib.draft_attn_plan_info(None, None) == -1
    assert lib.draft_attn_get_status(None, None, None) == -1
    assert lib.draft_attn_run(*([None] * 10), 0, None) == -1
    assert lib.draft_attn_append_kv(None, None, None, None, 1, 1, None, None, None, None, None) == -1


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no gcc")
def test_struct_layout_matches_header(tmp_path):
    src = tmp_path / "layout.c"
    src.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "draft_attn.h"\n'
        "int main(void){printf(\"%zu %zu %zu %zu %zu\\n\", sizeof(da_params),"
        " offsetof(da_params, side_scale), offsetof(da_params, tables_ready),"
        " sizeof(da_plan_info), offsetof(da_plan_info, workspace_bytes));return 0;}\n")
    exe = tmp_path / "layout"
    inc = os.path.join(os.path.dirname(B.HEADER))
    subprocess.run(["gcc", f"-I{inc}", str(src), "-o", str(exe)], check=True)
    got = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()
    want = [ctypes.sizeof(B.da_params), B.da_params.side_scale.offset,
            B.da_params.tables_ready.offset, ctypes.sizeof(B.da_plan_info),
            B.da_plan_info.workspace_bytes.offset]
    assert [int(x) for x in got] == want


@pytest.mark.parametrize("W,ns", [(2048, 0), (200, 4), (200, 70), (130, 0), (64, 64)])
def test_ring_size_is_the_smallest_fold_k_ring(W, ns):
    """draft_attn_ring_size gives the smallest k_ring_pages FOLD accepts."""
    n_ring, _ = B.draft_attn_ring_size(W, ns)
    p = _ok_params(mode="fold", window=W, n_sink=ns, alpha=2.0, far_mix=0.5, k_ring_pages=n_ring)
    assert B.draft_attn_check_params(p) == 0
    p.k_ring_pages = n_ring - 1
    assert B.draft_attn_check_params(p) == -1


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    """No CPU or PyTorch fallback: without the built library, loading raises."""
    monkeypatch.setattr(B, "_lib", None)
    with pytest.raises(ImportError, match="no CPU or PyTorch fallback"):
        B.load_library(str(tmp_path / "libdraft_attn.so"))
