"""Draft-step attention benchmark: µs per draft step and achieved KV-read GB/s
(fraction of measured HBM bandwidth), full context versus window.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--no-sweep] [--no-cpu-baseline] [--all OUT.json]

Workload of the headline line: the MTP draft head decode at 128K context --
batch 1, 32 query / 8 KV heads, head_dim 128, bf16 N(0,1) keys and values in a
paged cache (64-token pages, shuffled block table), 4 sequential draft steps
that each append one token (KV append + RoPE) and then attend with the query
at that token, each step one draft_attn_step launch.  One timed step is that
4-step draft loop, replayed from a CUDA graph; full and window (W = 2048) modes are timed separately, and `value` is
the full-mode KV GB/s (the KV bytes the mode must read, divided by the loop
time).  The L2 cache is flushed between timed steps (a 256 MiB write, then a
256 MiB read so no dirty lines are left for the timed step to write back).

A context sweep on the million-token shape (64/8 heads, theta 1e6, W = 4096 +
4 sinks) at 128K, 256K, 512K and 1M shows whether the window latency stays
flat.  `--all` also times the FOLD (4 x 256K) and ragged draft-tree workloads
and writes the table to a file.

Multi-GPU (torchrun): every rank runs an independent replica of the workload
(weak scaling, no collective on the data path); the barrier and the max over
ranks only frame the timing.

`--impl reference` times the float64 CPU oracle on the host cores on the same
workload, metric and unit, each step a bounded sample (two KV-head groups of
one draft step).
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from draft_attention_decode_b300 import workloads as WL  # noqa: E402

METRIC = "draft-step attention µs and KV GB/s (% of HBM peak) vs context, full vs window"
HEADLINE = "mtp_draft_128k"
FLUSH_BYTES = 256 << 20
NOMINAL_HBM_GBS = 8000.0   # the ~8 TB/s HBM3e figure the fractions are also quoted against
MIN_REPLAYS = 50           # tables report the median of at least this many replays
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class L2Flush:
    """Writes a 256 MiB buffer (evicting everything the step touched), then
    reads a second one, so that L2 holds only clean lines and the timed
    step does not pay for writing the flush's dirty lines back."""

    def __init__(self, dev):
        self.w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.sink = torch.empty((), dtype=torch.float32, device=dev)

    def fill_(self, v):
        self.w.fill_(v)
        torch.amax(self.r, dim=0, out=self.sink)


# ---------------------------------------------------------------------------
# Distributed framing
# ---------------------------------------------------------------------------

class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None

    def init(self, backend):
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            if self.pg.get_backend() == "nccl":
                self.pg.barrier(device_ids=[torch.cuda.current_device()])
            else:
                self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        dev = "cuda" if self.pg.get_backend() == "nccl" else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6400.0, "fallback"


# ---------------------------------------------------------------------------
# Clock sampling during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    def __init__(self, device_index: int):
        self.samples = []
        self.proc = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            sel = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            sel = str(device_index)
        self.cmd = ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                    "-lms", "200", "-i", sel]

    def start(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.samples.append(parts)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for s in self.samples:
            try:
                sm.append(float(s[1]))
                mx.append(float(s[2]))
            except ValueError:
                continue
            for n, v in zip(names, s[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# The CUDA path
# ---------------------------------------------------------------------------

class DraftLoop:
    """Caches of one workload shape plus, per mode, a plan and a CUDA graph of
    the draft loop (append one token, attend) x steps."""

    def __init__(self, wl: WL.Workload, dev, modes, cache_ctx=None, engine=0, tables_ready=0,
                 cluster_ctas=0):
        from draft_attention_decode_b300 import binding as B
        self.B = B
        self.tables_ready = tables_ready
        self.cluster_ctas = cluster_ctas
        self.wl = wl
        self.dev = dev
        dt = wl.torch_dtype
        steps = max(wl.draft_steps, 1)
        self.steps = steps
        cap = [c + wl.draft_steps for c in (cache_ctx or wl.ctx)]
        self.cap = cap
        self.bt, self.npg = WL.block_table(cap, wl.seed, device=dev)
        H, d = wl.num_kv_heads, wl.head_dim
        shape = (self.npg, H, WL.PAGE, d)
        need_side = "fold" in modes
        self.k_cache = torch.empty(shape, dtype=dt, device=dev)
        self.v_cache = torch.empty(shape, dtype=dt, device=dev)
        self.k_side = torch.empty(shape, dtype=dt, device=dev) if need_side else None
        # fill the caches through the library's append, sequence by sequence
        filler = self._plan("fold" if need_side else "full")
        for b, c in enumerate(cap):
            for s0 in range(0, c, 1 << 18):
                s1 = min(c, s0 + (1 << 18))
                k = WL.randn((1, s1 - s0, H, d), dt, dev, wl.seed * 16 + 2 + 1000 * b + 7 * s0)
                v = WL.randn((1, s1 - s0, H, d), dt, dev, wl.seed * 16 + 3 + 1000 * b + 7 * s0)
                pos = torch.arange(s0, s1, dtype=torch.int32, device=dev)[None]
                filler.append_kv(k, v, pos, self.bt[b:b + 1], self.k_cache, self.v_cache,
                                 self.k_side)
        torch.cuda.synchronize()
        filler.close()
        # per draft step: the new token, its query, positions and lengths
        self.q, self.k_new, self.v_new, self.pos, self.lens = [], [], [], [], []
        for s in range(steps):
            self.q.append(WL.randn((wl.batch, wl.n_q, wl.num_q_heads, d), dt, dev,
                                   wl.seed * 16 + 1 + 7919 * s))
            if wl.draft_steps:
                self.k_new.append(WL.randn((wl.batch, 1, H, d), dt, dev, 50000 + s))
                self.v_new.append(WL.randn((wl.batch, 1, H, d), dt, dev, 60000 + s))
                self.pos.append(torch.tensor([[c + s] for c in wl.ctx], dtype=torch.int32,
                                             device=dev))
                self.lens.append(torch.tensor([c + s + 1 for c in wl.ctx], dtype=torch.int32,
                                              device=dev))
            else:
                self.pos.append(torch.tensor([[c + t for t in range(wl.n_q)] for c in wl.ctx],
                                             dtype=torch.int32, device=dev))
                self.lens.append(torch.tensor(list(wl.ctx), dtype=torch.int32, device=dev))
        self.qpos = [p.expand(wl.batch, wl.n_q).contiguous() if wl.draft_steps else p
                     for p in self.pos]
        self.out = torch.empty_like(self.q[0])
        self.plans = {m: self._plan(m, engine) for m in modes}

    def _plan(self, mode, engine=0):
        wl = self.wl
        return self.B.DraftAttention(
            device=self.dev.index or 0, batch=wl.batch, n_q=wl.n_q,
            num_q_heads=wl.num_q_heads, num_kv_heads=wl.num_kv_heads, head_dim=wl.head_dim,
            num_pages=self.npg, max_pages_per_seq=self.bt.shape[1], dtype=wl.dtype, mode=mode,
            window=wl.window_for(mode), n_sink=wl.sinks_for(mode), alpha=wl.alpha,
            far_mix=wl.far_mix, scale_slope=wl.scale_slope, scale_ref=wl.scale_ref,
            rope_theta=wl.rope_theta, engine=engine, tables_ready=self.tables_ready,
            cluster_ctas=self.cluster_ctas if mode == "window" else 0)

    # -- one draft loop through the C ABI --------------------------------
    def loop(self, mode, lens=None, fused=True, reps=1):
        """fused: each draft step is one draft_attn_step launch (append +
        attend); otherwise draft_attn_append_kv then draft_attn_run.  reps > 1
        runs the steps again (the same tokens at the same positions: the same
        work per step), to time the steps after the first."""
        da = self.plans[mode]
        for s in [s for _ in range(reps) for s in range(self.steps)]:
            L = self.lens[s] if lens is None else lens
            if self.wl.draft_steps and fused:
                da.step(self.k_new[s], self.v_new[s], self.pos[s], self.q[s], self.qpos[s], L,
                        self.bt, self.k_cache, self.v_cache, self.k_side, out=self.out)
                continue
            if self.wl.draft_steps:
                da.append_kv(self.k_new[s], self.v_new[s], self.pos[s], self.bt, self.k_cache,
                             self.v_cache, self.k_side)
            da.run(self.q[s], self.qpos[s], L, self.bt, self.k_cache, self.v_cache, self.k_side,
                   out=self.out)

    def launches_per_loop(self, fused=True):
        per = 1 + (1 if self.wl.draft_steps and not fused else 0)   # decode (+ append)
        return per * self.steps

    def kv_bytes(self, mode, lens=None):
        """Algorithmic bytes of one draft loop: K and V (and, for FOLD far
        keys, side-cache K) of every selected key, once per KV head."""
        wl = self.wl
        es = 2 if wl.dtype == "bf16" else 4
        per_tok = 2 * wl.num_kv_heads * wl.head_dim * es
        tot = 0
        for s in range(self.steps):
            L = lens if lens is not None else self.lens[s].cpu().tolist()
            for Lb in L:
                tot += selected_keys(mode, Lb, wl.window_for(mode), wl.sinks_for(mode)) * per_tok
        return tot

    def capture(self, mode, lens=None, fused=True, reps=1):
        g = torch.cuda.CUDAGraph()
        st = torch.cuda.Stream()
        st.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(st):
            self.loop(mode, lens, fused)     # warm (plans, lazy module loads)
        torch.cuda.current_stream().wait_stream(st)
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            self.loop(mode, lens, fused, reps)
        torch.cuda.synchronize()
        return g

    def close(self):
        for p in self.plans.values():
            p.close()


def selected_keys(mode, L, W, ns):
    """Number of keys a mode reads for context L (all of them for full, sharp
    and fold; last W plus sinks for window)."""
    if mode in ("full", "sharp", "fold"):
        return L
    return min(L, min(ns, L) + min(W, L) if W + ns < L else L)


def time_graph(g, steps, warmup, flush, dist, stream=None):
    """Replays g warmup times, then times exactly `steps` replays with CUDA
    events, flushing L2 between them.  Returns per-replay ms (max over
    ranks of the mean)."""
    st = stream or torch.cuda.current_stream()
    for _ in range(warmup):
        flush.fill_(1)
        g.replay()
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for i in range(steps):
        flush.fill_(i & 0xff)
        ev[i][0].record(st)
        g.replay()
        ev[i][1].record(st)
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    ms = [a.elapsed_time(b) for a, b in ev]
    return dist.max(sum(ms) / len(ms)), ms


def median_replay(g, steps, warmup, flush, dist):
    """Median ms of at least MIN_REPLAYS timed replays (max over ranks)."""
    _, ms = time_graph(g, max(steps, MIN_REPLAYS), warmup, flush, dist)
    return dist.max(statistics.median(ms))


def rates(nbytes, ms, peak):
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"kv_gbs": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4),
            "frac_of_nominal": round(gbs / NOMINAL_HBM_GBS, 4)}


def time_calls(fn, steps, warmup, flush, dist):
    """Like time_graph for an un-captured callable (the per-launch roofline
    timing of the attention call)."""
    for _ in range(warmup):
        flush.fill_(1)
        fn()
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for i in range(steps):
        flush.fill_(i & 0xff)
        ev[i][0].record(st)
        fn()
        ev[i][1].record(st)
    torch.cuda.synchronize()
    ms = [a.elapsed_time(b) for a, b in ev]
    return dist.max(sum(ms) / len(ms)), dist.max(statistics.median(ms))


# ---------------------------------------------------------------------------
# CPU oracle baseline
# ---------------------------------------------------------------------------

# (workload, modes) the CPU baseline covers: every workload and mode the
# benchmark times on the GPU.
CPU_PLAN = (("mtp_draft_128k", ("full", "window")), ("mtp_draft_1m", ("full", "window")),
            ("fold_4x256k", ("fold", "full", "window")),
            ("ragged_tree_16x8", ("full", "window", "sharp")),
            ("tiny_window_fp32", ("full", "window")))


def host_workers():
    """Host cores this process may run on (its CPU affinity)."""
    return len(os.sched_getaffinity(0))


def oracle_params(wl, mode):
    import oracle.draft_attn_oracle as orc
    return orc.Params(mode=mode, window=wl.window_for(mode), n_sink=wl.sinks_for(mode),
                      alpha=wl.alpha, far_mix=wl.far_mix, scale_slope=wl.scale_slope,
                      scale_ref=wl.scale_ref, rope_theta=wl.rope_theta)


def step_units(wl):
    """The work units of the workload's first draft step: one (sequence b,
    query token t, KV head g) each, with its context length L and query
    position p (draft loops: the first appended token, L = ctx + 1, p = ctx;
    otherwise p = ctx + t)."""
    units = []
    for b, c in enumerate(wl.ctx):
        if wl.draft_steps:
            L, ps = c + 1, [c]
        else:
            L, ps = c, [c + t for t in range(wl.n_q)]
        for t, p in enumerate(ps):
            for g in range(wl.num_kv_heads):
                units.append((b, t, g, L, p))
    return units


def host_kv(wl, L, seed):
    """Host float32 keys and values [L, d] of one KV head (seeded draws of the
    workload's distribution, rounded to its dtype).  Every unit of a
    workload reads this one pair (a sequence shorter than L its prefix): the
    oracle's cost depends on the shapes only."""
    dt = wl.torch_dtype
    k = WL.randn((L, wl.head_dim), dt, "cpu", seed * 16 + 2).float().numpy()
    v = WL.randn((L, wl.head_dim), dt, "cpu", seed * 16 + 3).float().numpy()
    return k, v


def oracle_unit_bytes(wl, mode, L):
    es = 2 if wl.dtype == "bf16" else 4
    return selected_keys(mode, L, wl.window_for(mode), wl.sinks_for(mode)) * 2 * wl.head_dim * es


def run_units(wl, mode, units, kv, workers, budget_s, rng):
    """Runs the float64 oracle over `units` on `workers` host threads (BLAS
    held to one thread each, so the threads are the cores used), submitting
    units until `budget_s` has passed; the ones in flight then finish.
    Returns (KV bytes of the units done, seconds, units done)."""
    from concurrent.futures import FIRST_COMPLETED, ThreadPoolExecutor, wait
    import oracle.draft_attn_oracle as orc
    prm = oracle_params(wl, mode)
    G = wl.num_q_heads // wl.num_kv_heads
    k, v = kv
    qs = [rng.standard_normal((G, wl.head_dim)) for _ in range(len(units))]

    def one(i):
        b, t, g, L, p = units[i]
        orc.attend_group(qs[i], p, k[:max(L, 1)], v[:max(L, 1)], L, prm)
        return oracle_unit_bytes(wl, mode, L)

    try:
        from threadpoolctl import threadpool_limits
        limit = threadpool_limits(limits=1, user_api="blas")
    except Exception:
        limit = None
    nbytes, n_done, nxt = 0, 0, 0
    try:
        with ThreadPoolExecutor(workers) as ex:
            t0 = time.perf_counter()
            running = set()
            while True:
                while (len(running) < workers and nxt < len(units)
                       and time.perf_counter() - t0 < budget_s):
                    running.add(ex.submit(one, nxt))
                    nxt += 1
                if not running:
                    break
                done, running = wait(running, return_when=FIRST_COMPLETED)
                for f in done:
                    nbytes += f.result()
                    n_done += 1
            dt = time.perf_counter() - t0
    finally:
        if limit is not None:
            limit.unregister()
    return nbytes, dt, n_done


def cpu_baseline(budget_s=2.0):
    """The oracle as it stands, timed on the host cores, on a bounded sample of
    every workload and mode the benchmark times: the units (sequence, query
    token, KV head) of each workload's first draft step, in a seeded order,
    on one thread per host core, until `budget_s` per workload and mode (the
    units in flight then finish).  The headline entry is the 128K workload's
    full mode (the line's own metric and workload)."""
    workers = host_workers()
    rng = np.random.default_rng(0)
    rows = []
    for name, modes in CPU_PLAN:
        wl = WL.WORKLOADS[name]
        units = step_units(wl)
        kv = host_kv(wl, max(u[3] for u in units), wl.seed)
        order = rng.permutation(len(units))
        units = [units[i] for i in order]
        for mode in modes:
            nbytes, dt, n_done = run_units(wl, mode, units, kv, workers, budget_s, rng)
            step_bytes = sum(oracle_unit_bytes(wl, mode, u[3]) for u in units)
            rate = nbytes / dt
            rows.append({"workload": name, "mode": mode, "gbs": round(rate / 1e9, 4),
                         "s_per_draft_step": round(step_bytes / rate, 3),
                         "units_timed": n_done, "units_per_step": len(units),
                         "seconds": round(dt, 2)})
        del kv
    head = next(r for r in rows if r["workload"] == HEADLINE and r["mode"] == "full")
    return {"value": head["gbs"], "unit": "GB/s", "cores": workers, "kind": "oracle",
            "sample": (f"float64 numpy oracle, one thread per host core ({workers}, BLAS at one "
                       f"thread each); per workload and mode, units (sequence, query token, KV "
                       f"head) of its first draft step in a seeded order until {budget_s:g} s "
                       f"had passed (units in flight then finished); headline = "
                       f"{HEADLINE} full mode: {head['units_timed']} of "
                       f"{head['units_per_step']} units"),
            "per_workload": rows, "cpu_model": cpu_model()}


def cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return None


def run_reference(args, dist):
    """--impl reference: the oracle on the host cores, same metric/config.
    Each step is one whole full-mode draft step of the 128K workload (its
    eight KV-head groups, one per host thread)."""
    if dist.rank != 0:
        return
    wl = WL.WORKLOADS[HEADLINE]
    units = step_units(wl)
    kv = host_kv(wl, units[0][3], wl.seed)
    workers = host_workers()
    rng = np.random.default_rng(0)
    for _ in range(args.warmup):
        run_units(wl, "full", units, kv, workers, 1e9, rng)
    nbytes, dt = 0, 0.0
    for _ in range(args.steps):
        b, t, _ = run_units(wl, "full", units, kv, workers, 1e9, rng)
        nbytes += b
        dt += t
    val = nbytes / dt / 1e9
    sample = (f"each step: one whole full-mode draft step at L={units[0][3]} (all "
              f"{len(units)} KV-head groups), float64 numpy oracle, one thread per host "
              f"core ({workers}, BLAS at one thread each)")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(val, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(wl, "full"),
        "cpu_baseline": {"value": round(val, 4), "unit": "GB/s", "cores": workers,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(val, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(wl, mode_note):
    return {"workload": f"{wl.name}: batch {wl.batch}, {wl.num_q_heads}/{wl.num_kv_heads} heads, "
                        f"head_dim {wl.head_dim}, {wl.dtype} paged KV (64-token pages, shuffled "
                        f"block table), context {wl.ctx[0]}, {wl.draft_steps} draft steps "
                        f"(append + attend), full vs window W={wl.window}",
            "batch": wl.batch, "context": wl.ctx[0], "draft_steps": wl.draft_steps,
            "value_mode": mode_note, "l2": "flushed between timed steps (256 MiB write, then 256 MiB read)",
            "parallelism": "replicas (one independent workload per GPU)"}


# ---------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------

def e2e_full(dl: DraftLoop, steps, warmup, dist):
    """The headline metric through the public API with host buffers.  One step
    is one draft loop: the inputs of all its draft steps (queries, new K/V
    tokens, positions, lengths) go to the device in one copy from pinned host
    memory, each draft step is one draft_attn_step call, and the outputs of all
    draft steps come back in one copy, read by the host before the next loop."""
    da = dl.plans["full"]
    parts = [dl.q, dl.k_new, dl.v_new, dl.pos, dl.qpos, dl.lens]
    offs, nb = [], 0
    for s in range(dl.steps):            # 256-byte aligned slots of one staging buffer
        row = []
        for p in parts:
            row.append(nb)
            nb += (p[s].numel() * p[s].element_size() + 255) // 256 * 256
        offs.append(row)
    host = torch.empty(nb, dtype=torch.uint8).pin_memory()
    dbuf = torch.empty(nb, dtype=torch.uint8, device=dl.dev)
    views = []
    for s in range(dl.steps):
        vs = []
        for p, o in zip(parts, offs[s]):
            x = p[s].contiguous()
            n = x.numel() * x.element_size()
            host[o:o + n].copy_(x.view(-1).view(torch.uint8).cpu())
            vs.append(dbuf[o:o + n].view(x.dtype).view(x.shape))
        views.append(vs)
    outs = torch.empty((dl.steps,) + tuple(dl.out.shape), dtype=dl.out.dtype, device=dl.dev)
    hout = torch.empty(tuple(outs.shape), dtype=outs.dtype).pin_memory()
    h2d = nb
    d2h = hout.numel() * hout.element_size()

    def one():
        dbuf.copy_(host, non_blocking=True)
        for s in range(dl.steps):
            dq, dk, dv, dp, dqp, dln = views[s]
            da.step(dk, dv, dp, dq, dqp, dln, dl.bt, dl.k_cache, dl.v_cache, dl.k_side,
                    out=outs[s])
        hout.copy_(outs, non_blocking=True)
        torch.cuda.current_stream().synchronize()   # the host reads the loop's outputs
    for _ in range(warmup):
        one()
    torch.cuda.synchronize(); dist.barrier(); torch.cuda.synchronize()
    # each loop ends in a host read of its outputs, so loops are timed one by
    # one on the host clock; the median of them (host jitter between loops is
    # not the path's)
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        one()
        times.append(time.perf_counter() - t0)
    torch.cuda.synchronize(); dist.barrier(); torch.cuda.synchronize()
    dt = dist.max(statistics.median(times))
    return dt, h2d, d2h


def run_ours(args, dist):
    from draft_attention_decode_b300 import binding as B
    B.load_library()
    dev = torch.device("cuda", dist.local)
    torch.cuda.set_device(dev)
    peak, peak_kind = measured_peaks()
    flush = L2Flush(dev)

    wl = WL.WORKLOADS[HEADLINE]
    dl = DraftLoop(wl, dev, ("full", "window"))
    graphs = {m: dl.capture(m) for m in ("full", "window")}
    clocks = ClockSampler(dev.index or 0)
    clocks.start()
    # about a second of the same work before the timed region, so the clock
    # sampler sees the GPU under load
    t_end = time.perf_counter() + 1.0
    while time.perf_counter() < t_end:
        graphs["full"].replay()
        torch.cuda.synchronize()
    res = {}
    torch.cuda.profiler.start()   # profilers started with capture off see only this region
    for m in ("full", "window"):
        ms, all_ms = time_graph(graphs[m], args.steps, args.warmup, flush, dist)
        med = dist.max(statistics.median(all_ms))
        nbytes = dl.kv_bytes(m)
        res[m] = {"ms_per_loop": ms, "us_per_draft_step": ms * 1e3 / dl.steps,
                  "us_per_draft_step_median": med * 1e3 / dl.steps,
                  "kv_bytes_per_loop": nbytes, "kv_gbs": nbytes / (ms * 1e-3) / 1e9,
                  "frac_of_peak": nbytes / (ms * 1e-3) / 1e9 / peak,
                  "frac_of_nominal": nbytes / (ms * 1e-3) / 1e9 / NOMINAL_HBM_GBS}
    torch.cuda.profiler.stop()
    clk = clocks.stop()
    # the same loops with a separate append launch per draft step
    two = {}
    for m in ("full", "window"):
        g2 = dl.capture(m, fused=False)
        ms = median_replay(g2, args.steps, args.warmup, flush, dist)
        two[m] = {"us_per_draft_step": round(ms * 1e3 / dl.steps, 3),
                  **rates(dl.kv_bytes(m), ms, peak)}
        del g2
    # The steps after a loop's first (L2 flushed before each replay, so the
    # first step reads its window from DRAM and starts behind the flush): the
    # loop twice in one graph minus the loop once, per step; also with
    # tables_ready = 1 (lengths, positions and block table read before the
    # wait for the previous step), which this loop satisfies.
    further = {}
    for tr in (0, 1):
        saved = dl.plans
        if tr:
            dl.tables_ready = 1
            dl.plans = {m: dl._plan(m) for m in ("full", "window")}
        for m in ("full", "window"):
            t1 = median_replay(dl.capture(m), args.steps, args.warmup, flush, dist)
            t2 = median_replay(dl.capture(m, reps=2), args.steps, args.warmup, flush, dist)
            further[m + ("_tables_ready" if tr else "")] = {
                "us_per_draft_step": round(t1 * 1e3 / dl.steps, 3),
                "us_per_further_step": round((t2 - t1) * 1e3 / dl.steps, 3)}
        if tr:
            for p in dl.plans.values():
                p.close()
            dl.plans = saved
            dl.tables_ready = 0

    # roofline of the dominant kernel: the full-mode attention call of the
    # last draft step, timed on its own launch stream
    Lr = dl.lens[-1]
    ms_call, ms_call_med = time_calls(
        lambda: dl.plans["full"].run(dl.q[-1], dl.qpos[-1], Lr, dl.bt, dl.k_cache, dl.v_cache,
                                     None, out=dl.out),
        max(args.steps, MIN_REPLAYS), args.warmup, flush, dist)
    call_bytes = wl.batch * int(Lr[0]) * 2 * wl.num_kv_heads * wl.head_dim * 2
    achieved = call_bytes / (ms_call * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": profiled_traffic(),
                "kernel": f"decode_kernel (one draft_attn_run, full mode, L={int(Lr[0])})",
                "bytes_per_launch": call_bytes, "us_per_launch": round(ms_call * 1e3, 2),
                "us_per_launch_median": round(ms_call_med * 1e3, 2),
                "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                "peak_kind": f"{peak_kind} (MEASURED_PEAKS hbm_gbs copy bandwidth)"}

    # the 4-row shape on the tensor cores (an n8 tile half padding), for comparison
    mma = dl._plan("full", engine="mma")
    ms_mma, _ = time_calls(lambda: mma.run(dl.q[-1], dl.qpos[-1], Lr, dl.bt, dl.k_cache,
                                           dl.v_cache, None, out=dl.out),
                           max(args.steps, MIN_REPLAYS), args.warmup, flush, dist)
    mma.close()
    engines = {"cuda_core_us": round(ms_call * 1e3, 2), "tensor_core_padded_us":
               round(ms_mma * 1e3, 2), "note": "attention call alone, full mode; the default "
               "keeps <= 4 rows per KV head on the CUDA cores"}

    e2e_s, h2d, d2h = e2e_full(dl, max(args.steps, MIN_REPLAYS), args.warmup, dist)
    e2e_val = res["full"]["kv_bytes_per_loop"] / e2e_s / 1e9
    launches = dl.launches_per_loop(fused=True) * args.steps * 2
    dl.close()
    del dl, graphs
    torch.cuda.empty_cache()

    sweep = None if args.no_sweep else context_sweep(dev, args, flush, dist, peak)
    others = None if args.no_workloads else all_workloads(
        dev, args, flush, dist, peak, ("fold_4x256k", "ragged_tree_16x8"))
    if others is not None:
        if args.tc_rows:
            others += all_workloads(dev, args, flush, dist, peak, ("ragged_tree_16x8",),
                                    engine="tc05")
        others.append(fold_ring_row(dev, args, flush, dist, peak))
        others.append(fold_fp8_row(dev, args, flush, dist, peak))
        others.append(fold_fp8_row(dev, args, flush, dist, peak, engine="cuda_core"))
    cpu = None
    if dist.rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline()
    line = {
        "metric": METRIC, "value": round(res["full"]["kv_gbs"], 2), "unit": "GB/s",
        "n_gpus": dist.world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(res["full"]["ms_per_loop"], 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(wl, "full (window reported under modes)"),
        "modes": {m: {k: (round(v, 4) if isinstance(v, float) else v) for k, v in r.items()}
                  for m, r in res.items()},
        "window_speedup_vs_full": round(res["full"]["ms_per_loop"] / res["window"]["ms_per_loop"], 2),
        "modes_separate_append": two,
        "loop_steps": further,
        "engines": engines,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_val, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "note": "full mode, pinned host buffers; per step (one 4-draft-step loop) one "
                        "H2D copy of all its inputs, four draft_attn_step calls, one D2H copy "
                        "of the four outputs and a host sync, inside the timed region; each "
                        "loop timed on the host clock, the median of at least 50 loops"},
        "gpu_launches": launches,
        "clocks": clk,
        "sweep": sweep,
        "workloads": others,
    }
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    if args.all and dist.rank == 0:
        table = all_workloads(dev, args, flush, dist, peak,
                              ("fold_4x256k", "ragged_tree_16x8", "tiny_window_fp32"))
        with open(args.all, "w") as f:
            json.dump({"headline": line, "workloads": table}, f, indent=1)


def profiled_traffic():
    """DRAM bytes per launch of the decode kernel from the committed ncu
    summary, when it was taken from the current kernel sources."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.txt")
    try:
        kv = dict(l.strip().split("=", 1) for l in open(path)
                  if "=" in l and not l.lstrip().startswith("#"))
    except OSError:
        return None
    if kv.get("sources_sha") != sources_sha():
        return None
    try:
        return float(kv["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# The files decode_kernel (the CUDA-core, mma.sync and cluster engines) and its
# launch are built from; the tcgen05 kernel, the append kernel and the static
# entry point live elsewhere and do not change its code.
DECODE_KERNEL_SOURCES = ("draft_attention_decode_b300/csrc/common.cuh",
                         "draft_attention_decode_b300/csrc/pipeline.cuh",
                         "draft_attention_decode_b300/csrc/decode.cuh",
                         "draft_attention_decode_b300/csrc/decode.cu",
                         "draft_attention_decode_b300/csrc/api.cu",
                         "draft_attention_decode_b300/csrc/internal.h",
                         "include/draft_attn.h")


def sources_sha():
    """Hash of the sources the headline decode_kernel is compiled from."""
    import hashlib
    h = hashlib.sha256()
    for f in DECODE_KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def context_sweep(dev, args, flush, dist, peak):
    """Million-token shape (64/8 heads, theta 1e6, W 4096 + 4 sinks): one
    1M-token cache, attended at 128K..1M context, full vs window, one draft
    step each (the attention call alone, CUDA-graph replay)."""
    base = WL.WORKLOADS["mtp_draft_1m"]
    wl = dataclasses.replace(base, draft_steps=0)
    dl = DraftLoop(wl, dev, ("full", "window"))
    contexts = (131072, 262144, 524288, 1048576)
    # One graph per mode reads the context length and query position from
    # device tensors that are rewritten between contexts: every context is
    # timed through the same graph instance (separately captured instances of
    # the same call were seen to settle about 1.5 us apart), and the contexts
    # take turns in rounds, so that a drift of the GPU's state reaches every
    # context alike.  The median per context.
    lens = torch.zeros(1, dtype=torch.int32, device=dev)
    qpos = torch.zeros((1, 1), dtype=torch.int32, device=dev)
    graphs = {}
    for m in ("full", "window"):
        da = dl.plans[m]

        def call(da=da):
            da.run(dl.q[0], qpos, lens, dl.bt, dl.k_cache, dl.v_cache, None, out=dl.out)
        lens.fill_(contexts[-1])
        qpos.fill_(contexts[-1])
        call()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            call()
        graphs[m] = g
    times = {(L, m): [] for L in contexts for m in graphs}
    rounds = 5
    per_round = (max(args.steps, MIN_REPLAYS) + rounds - 1) // rounds
    for _ in range(rounds):
        for L in contexts:
            lens.fill_(L)
            qpos.fill_(L)
            for m, g in graphs.items():
                times[(L, m)] += time_graph(g, per_round, args.warmup, flush, dist)[1]
    rows = []
    for L in contexts:
        row = {"context": L}
        for m in ("full", "window"):
            ms = dist.max(statistics.median(times[(L, m)]))
            nb = selected_keys(m, L, wl.window_for(m), wl.sinks_for(m)) * 2 * 8 * 128 * 2
            row[m] = {"us": round(ms * 1e3, 2), **rates(nb, ms, peak)}
        rows.append(row)
    del graphs
    dl.close()
    del dl
    torch.cuda.empty_cache()
    # the configuration's own draft loop: 6 steps (append + attend) at 1M context
    dl = DraftLoop(base, dev, ("full", "window"))
    loop = {"context": base.ctx[0], "draft_steps": dl.steps}
    for m in ("full", "window"):
        g = dl.capture(m)
        ms = median_replay(g, args.steps, args.warmup, flush, dist)
        nb = dl.kv_bytes(m)
        ms2 = median_replay(dl.capture(m, reps=2), args.steps, args.warmup, flush, dist)
        loop[m] = {"us_per_draft_step": round(ms * 1e3 / dl.steps, 2),
                   "us_per_further_step": round((ms2 - ms) * 1e3 / dl.steps, 2), **rates(nb, ms, peak)}
    dl.close()
    del dl
    torch.cuda.empty_cache()
    w = [r["window"]["us"] for r in rows]
    return {"shape": "64/8 heads, d128, bf16, theta 1e6, W=4096 + 4 sinks, 1 query",
            "rows": rows, "window_max_over_min": round(max(w) / min(w), 3),
            "draft_loop_1m": loop}


def all_workloads(dev, args, flush, dist, peak, names, engine=0):
    """The other workloads, each mode's attention call replayed from a CUDA
    graph (inputs resident, L2 flushed between replays); `engine` forces one
    (e.g. "tc05") instead of the automatic choice."""
    table = []
    for name in names:
        wl = WL.WORKLOADS[name]
        dl = DraftLoop(wl, dev, wl.modes, engine=engine)
        for m in wl.modes:
            g = dl.capture(m)
            ms = median_replay(g, args.steps, args.warmup, flush, dist)
            nb = dl.kv_bytes(m)
            info = dl.plans[m].info()
            table.append({"workload": name, "mode": m, "us": round(ms * 1e3, 2),
                          "kv_bytes": nb, **rates(nb, ms, peak),
                          "engine": info["engine_name"], "cluster_ctas": info["cluster_ctas"]})
        dl.close()
        del dl
        torch.cuda.empty_cache()
    return table


def fold_ring_row(dev, args, flush, dist, peak):
    """FOLD 4 x 256K with the rotated keys kept in a ring of ceil(W/64) + 1
    pages per sequence (da_params.k_ring_pages): the attention call timed as in
    all_workloads, with the rotated K cache's bytes beside the paged one's."""
    wl = WL.WORKLOADS["fold_4x256k"]
    dl = DraftLoop(wl, dev, ("fold",))
    R = (wl.window + WL.PAGE - 1) // WL.PAGE + 1
    ring = dl.B.DraftAttention(
        device=dev.index or 0, batch=wl.batch, n_q=wl.n_q, num_q_heads=wl.num_q_heads,
        num_kv_heads=wl.num_kv_heads, head_dim=wl.head_dim, num_pages=dl.npg,
        max_pages_per_seq=dl.bt.shape[1], dtype=wl.dtype, mode="fold", window=wl.window,
        alpha=wl.alpha, far_mix=wl.far_mix, rope_theta=wl.rope_theta, k_ring_pages=R)
    kr = torch.empty((wl.batch * R,) + tuple(dl.k_cache.shape[1:]), dtype=dl.k_cache.dtype,
                     device=dev)
    for b in range(wl.batch):           # set-up: the window's rotated pages into the ring
        L = int(dl.lens[0][b])
        for P in range(max(L - wl.window, 0) // WL.PAGE, (L - 1) // WL.PAGE + 1):
            kr[b * R + P % R] = dl.k_cache[int(dl.bt[b, P])]
    torch.cuda.synchronize()

    def call():
        ring.run(dl.q[0], dl.qpos[0], dl.lens[0], dl.bt, kr, dl.v_cache, dl.k_side, out=dl.out)
    call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    ms = median_replay(g, args.steps, args.warmup, flush, dist)
    nb = dl.kv_bytes("fold")
    row = {"workload": "fold_4x256k", "mode": "fold, rotated K in a ring", "us": round(ms * 1e3, 2),
           "kv_bytes": nb, **rates(nb, ms, peak),
           "k_cache_bytes": kr.numel() * kr.element_size(),
           "k_cache_bytes_paged": dl.k_cache.numel() * dl.k_cache.element_size()}
    assert ring.status() == (dl.B.DA_OK, 0)
    ring.close()
    dl.close()
    del dl
    torch.cuda.empty_cache()
    return row


def fold_fp8_row(dev, args, flush, dist, peak, engine="auto"):
    """FOLD 4 x 256K with the side cache as E4M3 codes (da_params.side_fp8):
    the attention call timed as in all_workloads, on the automatic engine (the
    tensor cores) or forced onto the CUDA cores.  kv_bytes counts what the call must read:
    bf16 K and V of every local key, one-byte K and bf16 V of every far key."""
    wl = WL.WORKLOADS["fold_4x256k"]
    dl = DraftLoop(wl, dev, ("fold",))
    scale = 1.0 / 64            # N(0, 1) keys: |k| / scale stays well below 448
    f8 = dl.B.DraftAttention(
        device=dev.index or 0, batch=wl.batch, n_q=wl.n_q, num_q_heads=wl.num_q_heads,
        num_kv_heads=wl.num_kv_heads, head_dim=wl.head_dim, num_pages=dl.npg,
        max_pages_per_seq=dl.bt.shape[1], dtype=wl.dtype, mode="fold", window=wl.window,
        alpha=wl.alpha, far_mix=wl.far_mix, rope_theta=wl.rope_theta, side_fp8=1,
        side_scale=scale, engine=engine)
    # set-up, outside the timed region: the codes of the float32 quotient,
    # rounded to nearest even (what the append kernel writes for these keys)
    ks8 = torch.empty(dl.k_side.shape, dtype=torch.uint8, device=dev)
    for i in range(0, dl.k_side.shape[0], 1024):
        ks8[i:i + 1024] = (dl.k_side[i:i + 1024].float() / scale).to(
            torch.float8_e4m3fn).view(torch.uint8)
    torch.cuda.synchronize()

    def call():
        f8.run(dl.q[0], dl.qpos[0], dl.lens[0], dl.bt, dl.k_cache, dl.v_cache, ks8, out=dl.out)
    call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    ms = median_replay(g, args.steps, args.warmup, flush, dist)
    nb = 0
    for L in dl.lens[0].cpu().tolist():
        loc = min(wl.window, L)
        nb += wl.num_kv_heads * wl.head_dim * (4 * loc + 3 * (L - loc))
    label = "fold, FP8 E4M3 side cache" + (", CUDA-core engine forced" if engine == "cuda_core" else "")
    row = {"workload": "fold_4x256k", "mode": label, "us": round(ms * 1e3, 2),
           "kv_bytes": nb, **rates(nb, ms, peak),
           "side_cache_bytes": ks8.numel(),
           "side_cache_bytes_bf16": dl.k_side.numel() * dl.k_side.element_size()}
    assert f8.status() == (dl.B.DA_OK, 0)
    f8.close()
    dl.close()
    del dl, ks8
    torch.cuda.empty_cache()
    return row


def profile_loop(args):
    """Runs the draft loop of one workload and mode eagerly `reps` times (no
    timing): the command the ncu launch lists and captures are taken on."""
    from draft_attention_decode_b300 import binding as B
    dev = torch.device("cuda", 0)
    wl = WL.WORKLOADS[args.workload]
    if args.ctx:
        wl = WL.resized(wl, args.ctx)
    if args.ctx_cap:
        wl = WL.resized(wl, [min(c, args.ctx_cap) for c in wl.ctx])
    dl = DraftLoop(wl, dev, (args.profile_loop,), engine=args.engine,
                   cluster_ctas=args.cluster_ctas)
    torch.cuda.synchronize()
    if args.side_fp8:
        # FOLD with the side cache as E4M3 codes: the attention call on the first
        # draft step's inputs, `reps` times (set-up converts the side cache)
        if args.profile_loop != "fold":
            raise SystemExit("--side-fp8 needs --profile-loop fold")
        scale = 1.0 / 64
        da = B.DraftAttention(
            device=0, batch=wl.batch, n_q=wl.n_q, num_q_heads=wl.num_q_heads,
            num_kv_heads=wl.num_kv_heads, head_dim=wl.head_dim, num_pages=dl.npg,
            max_pages_per_seq=dl.bt.shape[1], dtype=wl.dtype, mode="fold", window=wl.window,
            alpha=wl.alpha, far_mix=wl.far_mix, rope_theta=wl.rope_theta, side_fp8=1,
            side_scale=scale, engine=args.engine)
        ks8 = torch.empty(dl.k_side.shape, dtype=torch.uint8, device=dev)
        for i in range(0, dl.k_side.shape[0], 1024):
            ks8[i:i + 1024] = (dl.k_side[i:i + 1024].float() / scale).to(
                torch.float8_e4m3fn).view(torch.uint8)
        torch.cuda.synchronize()
        torch.cuda.profiler.start()
        for _ in range(args.reps):
            da.run(dl.q[0], dl.qpos[0], dl.lens[0], dl.bt, dl.k_cache, dl.v_cache, ks8, out=dl.out)
        torch.cuda.synchronize()
        torch.cuda.profiler.stop()
        code, bits = da.status()
        da.close()
    else:
        torch.cuda.profiler.start()   # with ncu --profile-from-start off: the loop only
        for _ in range(args.reps):
            dl.loop(args.profile_loop)
        torch.cuda.synchronize()
        torch.cuda.profiler.stop()
        code, bits = dl.plans[args.profile_loop].status()
    dl.close()
    if code != B.DA_OK:
        raise SystemExit(f"device status {bits:#x}")
    print(f"profile loop ok: {wl.name} ctx={wl.ctx[0]} mode={args.profile_loop} reps={args.reps}"
          + (" side_fp8" if args.side_fp8 else ""))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the FOLD 4x256K and ragged draft-tree timings")
    ap.add_argument("--tc-rows", action="store_true",
                    help="also time the ragged draft tree on the tcgen05 engine")
    ap.add_argument("--all", default=None, help="also time every workload; write JSON here")
    ap.add_argument("--profile-loop", default=None, metavar="MODE",
                    help="run the draft loop of --workload in MODE --reps times, untimed")
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(WL.WORKLOADS))
    ap.add_argument("--ctx", type=int, default=0, help="override the workload's context")
    ap.add_argument("--ctx-cap", type=int, default=0,
                    help="cap every context of the workload at this length (ragged batches)")
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--engine", default="auto", choices=("auto", "cuda_core", "mma", "tc05"),
                    help="with --profile-loop: force this engine")
    ap.add_argument("--cluster-ctas", type=int, default=0,
                    help="with --profile-loop window: CTAs per cluster (-1: the flat partition)")
    ap.add_argument("--side-fp8", action="store_true",
                    help="with --profile-loop fold: the attention call over an E4M3 side cache")
    args = ap.parse_args()
    if args.profile_loop:
        profile_loop(args)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    dist = Dist()
    if args.impl == "reference":
        run_reference(args, dist)         # rank 0 only; no process group needed
        return
    if dist.world > 1:
        torch.cuda.set_device(dist.local)
    dist.init("nccl")
    run_ours(args, dist)
    dist.close()


if __name__ == "__main__":
    main()
