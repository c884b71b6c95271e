"""The decode kernel's shared-memory layouts, checked on the host: every
region a kernel addresses is aligned as its accesses need (1024-byte stage
ring for the 128-byte-swizzled TMA copies, 8-byte mbarriers, 16-byte vector
accesses), large enough and disjoint from the next, for every engine
variant, element size, head_dim, row count, pipeline depth and batch a plan
can pick.  Built from the library's own header with nvcc and run on the CPU
(no GPU needed)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _nvcc():
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    return None


def test_every_layout_is_aligned(tmp_path):
    nvcc = _nvcc()
    if nvcc is None:
        pytest.skip("nvcc not found")
    exe = tmp_path / "layout_check"
    src = os.path.join(ROOT, "tests", "native", "layout_check.cu")
    cmd = [nvcc, "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a",
           "-I" + os.path.join(ROOT, "include"),
           "-I" + os.path.join(ROOT, "draft_attention_decode_b300", "csrc"), src, "-o", str(exe)]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.startswith("ok"), r.stdout[-3000:]
