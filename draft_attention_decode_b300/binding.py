"""Python binding of the C ABI in ``include/draft_attn.h`` (ctypes).

Argument marshalling only: every step of the computation runs in the CUDA
library.  Functions carry the C names.  Tensors are torch tensors on the plan's
device; the stream defaults to torch's current stream.  Loading fails loudly if
the library has not been built: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libdraft_attn.so")
HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "draft_attn.h")

DA_OK = 0
DA_ERR_INVALID_ARG = -1
DA_ERR_UNSUPPORTED = -2
DA_ERR_WORKSPACE_TOO_SMALL = -3
DA_ERR_CUDA = -4
DA_ERR_DEVICE_FAULT = -5

DA_STATUS_BAD_PAGE = 1
DA_STATUS_BAD_CTX_LEN = 2
DA_STATUS_BAD_POSITION = 4
DA_STATUS_WAIT_TIMEOUT = 8
DA_STATIC_WORKSPACE_BYTES = 8 << 20

MODES = {"full": 0, "window": 1, "fold": 2, "sharp": 3}
DTYPES = {"bf16": 0, "fp32": 1}
TORCH_DTYPES = {0: torch.bfloat16, 1: torch.float32}
ENGINES = {0: "cuda_core", 1: "mma", 2: "tc05"}
ENGINE_HINTS = {"auto": 0, "cuda_core": 1, "mma": 2, "tc05": 3}


class DraftAttnError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {draft_attn_error_string(code)} ({code})")
        self.code = code


class da_params(ctypes.Structure):
    _fields_ = [
        ("rope_theta", ctypes.c_double),
        ("batch", ctypes.c_int32),
        ("n_q", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("num_pages", ctypes.c_int32),
        ("max_pages_per_seq", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("mode", ctypes.c_int32),
        ("window", ctypes.c_int32),
        ("n_sink", ctypes.c_int32),
        ("alpha", ctypes.c_float),
        ("far_mix", ctypes.c_float),
        ("scale_slope", ctypes.c_float),
        ("scale_ref", ctypes.c_int32),
        ("softmax_scale", ctypes.c_float),
        ("num_ctas", ctypes.c_int32),
        ("engine", ctypes.c_int32),
        ("min_pages_per_cta", ctypes.c_int32),
        ("stages", ctypes.c_int32),
        ("tree_size", ctypes.c_int32),
        ("k_ring_pages", ctypes.c_int32),
        ("side_fp8", ctypes.c_int32),
        ("side_scale", ctypes.c_float),
        ("cluster_ctas", ctypes.c_int32),
        ("tables_ready", ctypes.c_int32),
    ]


class da_plan_info(ctypes.Structure):
    _fields_ = [
        ("num_ctas", ctypes.c_int32),
        ("num_sms", ctypes.c_int32),
        ("rows_per_kv_head", ctypes.c_int32),
        ("kernel_rows", ctypes.c_int32),
        ("engine", ctypes.c_int32),
        ("stages", ctypes.c_int32),
        ("smem_bytes", ctypes.c_int32),
        ("cluster_ctas", ctypes.c_int32),
        ("workspace_bytes", ctypes.c_size_t),
    ]


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads the library (once) and declares the signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it with `python -m draft_attention_decode_b300.build` "
            "(there is no CPU or PyTorch fallback)")
    lib = ctypes.CDLL(path)
    P, I32, I64, SZ, VP = (ctypes.POINTER, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t,
                           ctypes.c_void_p)
    sig = {
        "draft_attn_check_params": (ctypes.c_int, [P(da_params)]),
        "draft_attn_plan": (ctypes.c_int, [P(da_params), ctypes.c_int, P(VP), P(SZ)]),
        "draft_attn_plan_info": (ctypes.c_int, [VP, P(da_plan_info)]),
        "draft_attn_plan_destroy": (None, [VP]),
        "draft_attn_append_kv": (ctypes.c_int, [VP, VP, VP, VP, I32, I32, VP, VP, VP, VP, VP]),
        "draft_attn_run": (ctypes.c_int, [VP, VP, VP, VP, VP, VP, VP, VP, VP, VP, SZ, VP]),
        "draft_attn_run_tree": (ctypes.c_int, [VP, VP, VP, VP, VP, VP, VP, VP, VP, VP, VP, SZ,
                                               VP]),
        "draft_attn_step": (ctypes.c_int, [VP, VP, VP, VP, I32, VP, VP, VP, VP, VP, VP, VP, VP, VP,
                                           VP, SZ, VP]),
        "draft_attn_run_static": (ctypes.c_int, [VP, VP, VP, VP, VP, VP, VP, VP, VP, VP]),
        "draft_attn_debug_gather": (ctypes.c_int, [VP, VP, VP, VP, VP, I32, I32, VP, VP, VP, VP, VP,
                                                   I64, VP, VP]),
        "draft_attn_get_status": (ctypes.c_int, [VP, VP, P(ctypes.c_uint32)]),
        "draft_attn_debug_wait_timeout": (ctypes.c_int, [VP, VP]),
        "draft_attn_ring_size": (ctypes.c_int, [I32, I32, P(I32), P(I32)]),
        "draft_attn_ring_block_table": (ctypes.c_int, [P(I32), I64, P(I32), I32, I32]),
        "draft_attn_error_string": (ctypes.c_char_p, [ctypes.c_int]),
        "draft_attn_version": (ctypes.c_int, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def header_functions(path: str = HEADER) -> list:
    """Names of the functions include/draft_attn.h declares."""
    text = open(path).read()
    return sorted(set(re.findall(r"\b(draft_attn_\w+)\s*\(", text)))


# ---------------------------------------------------------------------------
# Marshalling helpers
# ---------------------------------------------------------------------------

def make_params(*, batch, n_q, num_q_heads, num_kv_heads, head_dim, num_pages, max_pages_per_seq,
                dtype="bf16", mode="full", window=0, n_sink=0, alpha=1.0, far_mix=0.0,
                scale_slope=0.0, scale_ref=4096, rope_theta=1e4, softmax_scale=0.0, num_ctas=0,
                page_size=64, engine=0, min_pages_per_cta=0, stages=0, tree_size=0,
                k_ring_pages=0, side_fp8=0, side_scale=0.0, cluster_ctas=0,
                tables_ready=0) -> da_params:
    p = da_params()
    p.rope_theta = float(rope_theta)
    p.batch, p.n_q = int(batch), int(n_q)
    p.num_q_heads, p.num_kv_heads, p.head_dim = int(num_q_heads), int(num_kv_heads), int(head_dim)
    p.page_size, p.num_pages, p.max_pages_per_seq = int(page_size), int(num_pages), int(max_pages_per_seq)
    p.dtype = DTYPES[dtype] if isinstance(dtype, str) else int(dtype)
    p.mode = MODES[mode] if isinstance(mode, str) else int(mode)
    p.window, p.n_sink = int(window), int(n_sink)
    p.alpha, p.far_mix, p.scale_slope = float(alpha), float(far_mix), float(scale_slope)
    p.scale_ref, p.softmax_scale, p.num_ctas = int(scale_ref), float(softmax_scale), int(num_ctas)
    p.engine = ENGINE_HINTS[engine] if isinstance(engine, str) else int(engine)
    p.min_pages_per_cta = int(min_pages_per_cta)
    p.stages = int(stages)
    p.tree_size = int(tree_size)
    p.k_ring_pages = int(k_ring_pages)
    p.side_fp8, p.side_scale = int(side_fp8), float(side_scale)
    p.cluster_ctas = int(cluster_ctas)
    p.tables_ready = int(tables_ready)
    return p


def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError("tensor must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(code, what):
    if code != DA_OK:
        raise DraftAttnError(code, what)


# ---------------------------------------------------------------------------
# The C entry points
# ---------------------------------------------------------------------------

def draft_attn_version() -> int:
    return load_library().draft_attn_version()


def draft_attn_error_string(code: int) -> str:
    return load_library().draft_attn_error_string(int(code)).decode()


def draft_attn_check_params(params: da_params) -> int:
    return load_library().draft_attn_check_params(ctypes.byref(params))


def draft_attn_plan(params: da_params, device: int = 0):
    """Returns (plan handle, workspace bytes)."""
    lib = load_library()
    plan = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    _check(lib.draft_attn_plan(ctypes.byref(params), int(device), ctypes.byref(plan), ctypes.byref(ws)),
           "draft_attn_plan")
    return plan, ws.value


def draft_attn_plan_info(plan) -> dict:
    info = da_plan_info()
    _check(load_library().draft_attn_plan_info(plan, ctypes.byref(info)), "draft_attn_plan_info")
    d = {f: getattr(info, f) for f, _ in info._fields_}
    d["engine_name"] = ENGINES.get(d["engine"], "?")
    return d


def draft_attn_plan_destroy(plan) -> None:
    if plan:
        load_library().draft_attn_plan_destroy(plan)


def draft_attn_append_kv(plan, k_new, v_new, pos, block_table, k_cache, v_cache, k_side=None,
                         stream=None) -> None:
    """k_new, v_new: [batch, n_new, H_kv, d]; pos: int32 [batch, n_new]."""
    batch, n_new = int(k_new.shape[0]), int(k_new.shape[1])
    if tuple(v_new.shape) != tuple(k_new.shape) or tuple(pos.shape) != (batch, n_new):
        raise ValueError("k_new, v_new and pos shapes disagree")
    if pos.dtype != torch.int32 or block_table.dtype != torch.int32:
        raise ValueError("pos and block_table must be int32")
    _check(load_library().draft_attn_append_kv(
        plan, _ptr(k_new), _ptr(v_new), _ptr(pos), batch, n_new, _ptr(block_table),
        _ptr(k_cache), _ptr(v_cache), _ptr(k_side), _stream(stream)), "draft_attn_append_kv")


def draft_attn_run(plan, q, q_pos, ctx_lens, block_table, k_cache, v_cache, k_side, out,
                   workspace, stream=None) -> None:
    for name, t in (("q_pos", q_pos), ("ctx_lens", ctx_lens), ("block_table", block_table)):
        if t.dtype != torch.int32:
            raise ValueError(f"{name} must be int32")
    if workspace.dtype != torch.uint8:
        raise ValueError("workspace must be a uint8 tensor")
    _check(load_library().draft_attn_run(
        plan, _ptr(q), _ptr(q_pos), _ptr(ctx_lens), _ptr(block_table), _ptr(k_cache),
        _ptr(v_cache), _ptr(k_side), _ptr(out), _ptr(workspace), workspace.numel(),
        _stream(stream)), "draft_attn_run")


def draft_attn_run_tree(plan, q, q_pos, ctx_lens, block_table, k_cache, v_cache, k_side, tree_mask,
                        out, workspace, stream=None) -> None:
    """tree_mask: int64 tensor [batch, n_q] holding each query's uint64 mask
    of visible draft-tree keys (bit i: tree token i), or None (all visible)."""
    for name, t in (("q_pos", q_pos), ("ctx_lens", ctx_lens), ("block_table", block_table)):
        if t.dtype != torch.int32:
            raise ValueError(f"{name} must be int32")
    if tree_mask is not None and tree_mask.dtype not in (torch.int64, torch.uint64):
        raise ValueError("tree_mask must be a 64-bit integer tensor")
    if workspace.dtype != torch.uint8:
        raise ValueError("workspace must be a uint8 tensor")
    _check(load_library().draft_attn_run_tree(
        plan, _ptr(q), _ptr(q_pos), _ptr(ctx_lens), _ptr(block_table), _ptr(k_cache),
        _ptr(v_cache), _ptr(k_side), _ptr(tree_mask), _ptr(out), _ptr(workspace),
        workspace.numel(), _stream(stream)), "draft_attn_run_tree")


def draft_attn_step(plan, k_new, v_new, pos, q, q_pos, ctx_lens, block_table, k_cache, v_cache,
                    k_side, out, workspace, tree_mask=None, stream=None) -> None:
    """Append k_new / v_new [batch, n_new, H_kv, d] at pos [batch, n_new] and
    attend, in one call (append kernel, then the attention kernel behind it)."""
    n_new = int(k_new.shape[1]) if k_new is not None else 0
    for name, t in (("q_pos", q_pos), ("ctx_lens", ctx_lens), ("block_table", block_table)):
        if t.dtype != torch.int32:
            raise ValueError(f"{name} must be int32")
    if n_new and (pos.dtype != torch.int32 or tuple(pos.shape) != tuple(k_new.shape[:2])):
        raise ValueError("pos must be int32 [batch, n_new]")
    if workspace.dtype != torch.uint8:
        raise ValueError("workspace must be a uint8 tensor")
    _check(load_library().draft_attn_step(
        plan, _ptr(k_new), _ptr(v_new), _ptr(pos), n_new, _ptr(q), _ptr(q_pos), _ptr(ctx_lens),
        _ptr(block_table), _ptr(k_cache), _ptr(v_cache), _ptr(k_side), _ptr(tree_mask), _ptr(out),
        _ptr(workspace), workspace.numel(), _stream(stream)), "draft_attn_step")


def draft_attn_run_static(plan, q, q_pos, ctx_lens, block_table, k_cache, v_cache, k_side, out,
                          stream=None) -> None:
    """draft_attn_run with the library's own fixed device workspace: for
    callers that cannot allocate device memory when they run the step."""
    for name, t in (("q_pos", q_pos), ("ctx_lens", ctx_lens), ("block_table", block_table)):
        if t.dtype != torch.int32:
            raise ValueError(f"{name} must be int32")
    _check(load_library().draft_attn_run_static(
        plan, _ptr(q), _ptr(q_pos), _ptr(ctx_lens), _ptr(block_table), _ptr(k_cache),
        _ptr(v_cache), _ptr(k_side), _ptr(out), _stream(stream)), "draft_attn_run_static")


def draft_attn_debug_gather(plan, q_pos, ctx_lens, block_table, b, t, capacity, stream=None,
                            tree_mask=None) -> dict:
    dev = q_pos.device
    cap = int(capacity)
    out = {
        "position": torch.empty(max(cap, 1), dtype=torch.int32, device=dev),
        "phys_slot": torch.empty(max(cap, 1), dtype=torch.int64, device=dev),
        "key_rope_pos": torch.empty(max(cap, 1), dtype=torch.int32, device=dev),
        "q_rope_pos": torch.empty(max(cap, 1), dtype=torch.int32, device=dev),
        "segment": torch.empty(max(cap, 1), dtype=torch.int8, device=dev),
    }
    count = torch.zeros(1, dtype=torch.int64, device=dev)
    _check(load_library().draft_attn_debug_gather(
        plan, _ptr(q_pos), _ptr(ctx_lens), _ptr(block_table), _ptr(tree_mask), int(b), int(t),
        _ptr(out["position"]), _ptr(out["phys_slot"]), _ptr(out["key_rope_pos"]),
        _ptr(out["q_rope_pos"]), _ptr(out["segment"]), cap, _ptr(count), _stream(stream)),
        "draft_attn_debug_gather")
    n = int(count.item())
    res = {k: v[: min(n, cap)] for k, v in out.items()}
    res["count"] = n
    return res


def draft_attn_ring_size(window, n_sink):
    """Returns (n_ring, n_sink_pages): the smallest ring of pages that holds a
    window-mode draft KV with this window and sink count."""
    n_ring, n_sink_pages = ctypes.c_int32(), ctypes.c_int32()
    _check(load_library().draft_attn_ring_size(int(window), int(n_sink), ctypes.byref(n_ring),
                                               ctypes.byref(n_sink_pages)), "draft_attn_ring_size")
    return n_ring.value, n_sink_pages.value


def draft_attn_ring_block_table(max_pages, ring_pages, n_sink_pages):
    """One block-table row (int32 numpy array of max_pages entries) mapping
    logical pages onto the ring of physical pages `ring_pages`."""
    import numpy as np
    ring = np.ascontiguousarray(np.asarray(ring_pages, dtype=np.int32))
    table = np.empty(int(max_pages), dtype=np.int32)
    I32p = ctypes.POINTER(ctypes.c_int32)
    _check(load_library().draft_attn_ring_block_table(
        table.ctypes.data_as(I32p), int(max_pages), ring.ctypes.data_as(I32p), int(ring.size),
        int(n_sink_pages)), "draft_attn_ring_block_table")
    return table


def draft_attn_debug_wait_timeout(plan, stream=None):
    """Launches the bounded-wait give-up hook (about a second on the device)."""
    _check(load_library().draft_attn_debug_wait_timeout(plan, _stream(stream)),
           "draft_attn_debug_wait_timeout")


def draft_attn_get_status(plan, stream=None):
    """Returns (code, bits); code is DA_OK or DA_ERR_DEVICE_FAULT."""
    bits = ctypes.c_uint32()
    code = load_library().draft_attn_get_status(plan, _stream(stream), ctypes.byref(bits))
    if code not in (DA_OK, DA_ERR_DEVICE_FAULT):
        raise DraftAttnError(code, "draft_attn_get_status")
    return code, bits.value


# ---------------------------------------------------------------------------
# Convenience owner of a plan and its workspace
# ---------------------------------------------------------------------------

class DraftAttention:
    """A plan plus a workspace tensor; methods forward to the C entry points."""

    def __init__(self, device=0, **kw):
        self.params = make_params(**kw)
        self.device = torch.device("cuda", device) if isinstance(device, int) else torch.device(device)
        self.plan, self.workspace_bytes = draft_attn_plan(self.params, self.device.index or 0)
        # zero-filled once: the run keeps its page counters at zero between calls
        self.workspace = torch.zeros(self.workspace_bytes, dtype=torch.uint8, device=self.device)
        self.dtype = TORCH_DTYPES[self.params.dtype]

    def info(self) -> dict:
        return draft_attn_plan_info(self.plan)

    def append_kv(self, k_new, v_new, pos, block_table, k_cache, v_cache, k_side=None, stream=None):
        draft_attn_append_kv(self.plan, k_new, v_new, pos, block_table, k_cache, v_cache, k_side,
                             stream)

    def run(self, q, q_pos, ctx_lens, block_table, k_cache, v_cache, k_side=None, out=None,
            stream=None, tree_mask=None):
        if out is None:
            out = torch.empty_like(q)
        if tree_mask is None:
            draft_attn_run(self.plan, q, q_pos, ctx_lens, block_table, k_cache, v_cache, k_side,
                           out, self.workspace, stream)
        else:
            draft_attn_run_tree(self.plan, q, q_pos, ctx_lens, block_table, k_cache, v_cache,
                                k_side, tree_mask, out, self.workspace, stream)
        return out

    def step(self, k_new, v_new, pos, q, q_pos, ctx_lens, block_table, k_cache, v_cache,
             k_side=None, out=None, stream=None, tree_mask=None):
        if out is None:
            out = torch.empty_like(q)
        draft_attn_step(self.plan, k_new, v_new, pos, q, q_pos, ctx_lens, block_table, k_cache,
                        v_cache, k_side, out, self.workspace, tree_mask, stream)
        return out

    def status(self, stream=None):
        return draft_attn_get_status(self.plan, stream)

    def close(self):
        if self.plan:
            draft_attn_plan_destroy(self.plan)
            self.plan = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
