"""The benchmark's multi-process framing on the CPU (gloo, world size 2): the
timing is the max over ranks, the barrier joins every rank, and the
reference arm prints from rank 0 only."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r"""
import os, sys, json
sys.path.insert(0, {root!r})
import bench
d = bench.Dist()
d.init("gloo")
m = d.max(float(d.rank + 1) * 1.5)
d.barrier()
print(json.dumps({{"rank": d.rank, "max": m, "world": d.world}}))
d.close()
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _launch(code, world=2, extra_env=None):
    port = _free_port()
    procs = []
    for r in range(world):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE=str(world),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        env.update(extra_env or {})
        procs.append(subprocess.Popen([sys.executable, "-c", code], env=env, cwd=ROOT,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        o, e = p.communicate(timeout=120)
        assert p.returncode == 0, e[-2000:]
        outs.append(o)
    return outs


def test_max_over_ranks_and_barrier():
    outs = _launch(WORKER.format(root=ROOT))
    rows = [json.loads(o.strip().splitlines()[-1]) for o in outs]
    assert sorted(r["rank"] for r in rows) == [0, 1]
    assert all(r["max"] == 3.0 and r["world"] == 2 for r in rows)


def test_reference_arm_prints_on_rank0_only(tmp_path):
    code = ("import sys; sys.path.insert(0, %r); import bench, types;"
            "bench.HEADLINE = 'tiny_window_fp32';"
            "a = types.SimpleNamespace(steps=1, warmup=3, gpus=2);"
            "bench.run_reference(a, bench.Dist())" % ROOT)
    outs = _launch(code)
    assert outs[1].strip() == ""
    line = json.loads(outs[0].strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_traffic_record_follows_the_kernel_sources(monkeypatch):
    """roofline.traffic comes from the committed ncu record only while the
    headline kernel's sources hash to the value the record was taken on; the
    record's bytes are those of one 128K full-mode call (K and V of 131,075
    keys over 8 KV heads, plus the partials and the output written)."""
    sys.path.insert(0, ROOT)
    import bench
    for f in bench.DECODE_KERNEL_SOURCES:
        assert os.path.exists(os.path.join(ROOT, f)), f
    assert bench.sources_sha() == bench.sources_sha()
    t = bench.profiled_traffic()
    algorithmic = 131075 * 8 * 2 * 128 * 2
    assert t is None or algorithmic <= t <= 1.02 * algorithmic
    monkeypatch.setattr(bench, "sources_sha", lambda: "0" * 16)
    assert bench.profiled_traffic() is None
