"""ctypes binding of libpagedkv.so -- argument marshalling only.

Every function here checks the tensors it is given (device, dtype, shape,
contiguity), turns them into raw pointers and calls the C ABI declared in
``include/pagedkv.h``.  All computation runs in the library's CUDA kernels;
there is no fallback of any kind: if the library is missing, calls raise.
PyTorch supplies device memory and streams, nothing else.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libpagedkv.so")

PKV_OK = 0
PKV_ERR_INVALID = -1
PKV_ERR_UNSUPPORTED = -2
PKV_ERR_WORKSPACE = -3
PKV_ERR_CUDA = -4
PKV_ERR_DEVICE_BOUNDS = -5
PKV_ERR_TIMEOUT = -6

EXPORTED = ("pkv_append", "pkv_attention", "pkv_attention_workspace_size",
            "pkv_workspace_init", "pkv_last_error", "pkv_get_device_error",
            "pkv_attention_noalloc", "pkv_copy_blocks", "pkv_append_fp8",
            "pkv_attention_fp8kv", "pkv_cascade_workspace_size", "pkv_attention_cascade",
            "pkv_append_attention", "pkv_append_attention_fp8", "pkv_get_options",
            "pkv_set_options")

# Fields of pkv_options, in declaration order (int32 each).
OPTION_FIELDS = ("pdl", "early_plan", "early_kv", "early_trigger", "plan_cache", "decode_tc",
                 "decode_tc_fp8", "prefill_min_q", "align", "align_slack", "min_chunk",
                 "decode_grid", "wait_limit_us", "debug_withhold_q",
                 "rowgroup_cost")


class PagedKVError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"libpagedkv error {code}: {message}")
        self.code = code


class Dims(ctypes.Structure):
    _fields_ = [("num_reqs", ctypes.c_int32), ("num_q_tokens", ctypes.c_int32),
                ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_blocks", ctypes.c_int32), ("max_blocks_per_req", ctypes.c_int32)]


class Options(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int32) for name in OPTION_FIELDS]


_lock = threading.Lock()
_lib = None


def load_library(path: str = LIB_PATH):
    """Load libpagedkv.so and declare its signatures (raises if absent)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is not built: run paged_kv_cache_195_gb300.build.build() "
                "(the CUDA library is required; there is no fallback)")
        lib = ctypes.CDLL(path)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        dp = ctypes.POINTER(Dims)
        lib.pkv_append.argtypes = [vp, vp, vp, vp, vp, i32, dp, vp]
        lib.pkv_append.restype = ctypes.c_int
        lib.pkv_attention.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_float, vp, dp, vp, sz, vp]
        lib.pkv_attention.restype = ctypes.c_int
        lib.pkv_attention_workspace_size.argtypes = [dp]
        lib.pkv_attention_workspace_size.restype = sz
        lib.pkv_workspace_init.argtypes = [vp, sz, dp, vp]
        lib.pkv_workspace_init.restype = ctypes.c_int
        lib.pkv_last_error.argtypes = []
        lib.pkv_last_error.restype = ctypes.c_char_p
        lib.pkv_get_device_error.argtypes = [vp]
        lib.pkv_get_device_error.restype = ctypes.c_int
        lib.pkv_attention_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_float, vp, dp, vp]
        lib.pkv_attention_noalloc.restype = ctypes.c_int
        lib.pkv_copy_blocks.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, dp, vp]
        lib.pkv_copy_blocks.restype = ctypes.c_int
        lib.pkv_append_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, dp, vp]
        lib.pkv_append_fp8.restype = ctypes.c_int
        lib.pkv_attention_fp8kv.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_float, vp, dp,
                                            vp, sz, vp]
        lib.pkv_attention_fp8kv.restype = ctypes.c_int
        lib.pkv_cascade_workspace_size.argtypes = [dp]
        lib.pkv_cascade_workspace_size.restype = sz
        lib.pkv_attention_cascade.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32,
                                              ctypes.c_float, vp, dp, vp, sz, vp]
        lib.pkv_attention_cascade.restype = ctypes.c_int
        lib.pkv_append_attention.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_float,
                                             vp, dp, vp, sz, vp]
        lib.pkv_append_attention.restype = ctypes.c_int
        lib.pkv_append_attention_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                                 ctypes.c_float, vp, dp, vp, sz, vp]
        lib.pkv_append_attention_fp8.restype = ctypes.c_int
        lib.pkv_get_options.argtypes = [ctypes.POINTER(Options)]
        lib.pkv_get_options.restype = None
        lib.pkv_set_options.argtypes = [ctypes.POINTER(Options)]
        lib.pkv_set_options.restype = ctypes.c_int
        _lib = lib
        return lib


def get_options() -> dict:
    """The library's current launch and routing options (pkv_options)."""
    o = Options()
    load_library().pkv_get_options(ctypes.byref(o))
    return {name: int(getattr(o, name)) for name in OPTION_FIELDS}


def set_options(**changes) -> dict:
    """Change some options (the rest keep their values); returns the old ones."""
    old = get_options()
    unknown = set(changes) - set(OPTION_FIELDS)
    if unknown:
        raise KeyError(f"unknown options: {sorted(unknown)}")
    new = dict(old, **{k: int(v) for k, v in changes.items()})
    o = Options(*(new[name] for name in OPTION_FIELDS))
    _check(load_library().pkv_set_options(ctypes.byref(o)))
    return old


@contextlib.contextmanager
def options(**changes):
    """Run a block with some options changed, then put the old ones back."""
    old = set_options(**changes)
    try:
        yield
    finally:
        set_options(**old)


def pkv_last_error() -> str:
    return load_library().pkv_last_error().decode()


def _check(rc: int):
    if rc != PKV_OK:
        raise PagedKVError(rc, pkv_last_error())


def _stream(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _need(t: torch.Tensor, name: str, dtype, ndim: int):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def check_attention_shapes(q, k_pool, v_pool, block_tables, seq_lens, query_start_loc,
                           out=None):
    """Shape agreement of an attention call's tensors (any device): the
    pools equal in shape with q's head_dim, one table row and length per
    request, query_start_loc one longer, out shaped like q.  Raises
    ValueError before anything reaches the library, whose kernels size every
    pool access from k_pool's shape alone."""
    R = seq_lens.shape[0]
    if query_start_loc.shape[0] != R + 1 or block_tables.shape[0] != R:
        raise ValueError("seq_lens, query_start_loc and block_tables disagree on num_reqs")
    if tuple(v_pool.shape) != tuple(k_pool.shape) or k_pool.shape[3] != q.shape[2]:
        raise ValueError("pool / q shape mismatch: v_pool must have k_pool's shape and "
                         "head_dim must match q's")
    if out is not None and tuple(out.shape) != tuple(q.shape):
        raise ValueError("out must have q's shape")
    return R


def make_dims(q_shape, pool_shape, num_reqs: int, max_blocks_per_req: int) -> Dims:
    Tq, Hq, D = q_shape
    nb, Hkv, bs, D2 = pool_shape
    return Dims(num_reqs, Tq, Hq, Hkv, D, bs, nb, max_blocks_per_req)


def pkv_attention_workspace_size(dims: Dims) -> int:
    return int(load_library().pkv_attention_workspace_size(ctypes.byref(dims)))


class Workspace:
    """A zero-initialised device workspace for pkv_attention (reusable).

    It remembers the (num_q_tokens, num_kv_heads) its counters were zeroed
    for; pkv_attention re-initialises it when a call's dims differ."""

    def __init__(self, dims: Dims, device="cuda"):
        self.nbytes = pkv_attention_workspace_size(dims)
        if self.nbytes == 0:
            raise PagedKVError(PKV_ERR_INVALID, pkv_last_error() or "bad dims")
        self.buf = torch.zeros(self.nbytes + 256, dtype=torch.uint8, device=device)
        off = (-self.buf.data_ptr()) % 256
        self.ptr = self.buf.data_ptr() + off
        self.counter_dims = (dims.num_q_tokens, dims.num_kv_heads)


def pkv_workspace_init(ws: Workspace, dims: Dims, stream=None):
    _check(load_library().pkv_workspace_init(ctypes.c_void_p(ws.ptr), ws.nbytes,
                                             ctypes.byref(dims),
                                             ctypes.c_void_p(_stream(stream, ws.buf.device))))
    ws.counter_dims = (dims.num_q_tokens, dims.num_kv_heads)


def pkv_append(k_new, v_new, slot_mapping, k_pool, v_pool, stream=None):
    """Write k_new/v_new [T, Hkv, D] bf16 into the pools at slot_mapping [T] int64."""
    _need(k_new, "k_new", torch.bfloat16, 3)
    _need(v_new, "v_new", torch.bfloat16, 3)
    _need(slot_mapping, "slot_mapping", torch.int64, 1)
    _need(k_pool, "k_pool", torch.bfloat16, 4)
    _need(v_pool, "v_pool", torch.bfloat16, 4)
    T = k_new.shape[0]
    if v_new.shape != k_new.shape or slot_mapping.shape[0] != T:
        raise ValueError("k_new, v_new and slot_mapping disagree on the token count")
    if v_pool.shape != k_pool.shape or k_pool.shape[1] != k_new.shape[1] or \
            k_pool.shape[3] != k_new.shape[2]:
        raise ValueError("pool shape does not match the new rows")
    nb, Hkv, bs, D = k_pool.shape
    dims = Dims(0, 0, Hkv, Hkv, D, bs, nb, 0)
    _check(load_library().pkv_append(
        ctypes.c_void_p(k_new.data_ptr()), ctypes.c_void_p(v_new.data_ptr()),
        ctypes.c_void_p(slot_mapping.data_ptr()), ctypes.c_void_p(k_pool.data_ptr()),
        ctypes.c_void_p(v_pool.data_ptr()), T, ctypes.byref(dims),
        ctypes.c_void_p(_stream(stream, k_pool.device))))


def pkv_attention(q, k_pool, v_pool, block_tables, seq_lens, query_start_loc, scale,
                  out=None, workspace: Workspace | None = None, stream=None):
    """One step of paged attention; returns out [Tq, Hq, D] bf16."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k_pool, "k_pool", torch.bfloat16, 4)
    _need(v_pool, "v_pool", torch.bfloat16, 4)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    _need(query_start_loc, "query_start_loc", torch.int32, 1)
    R = check_attention_shapes(q, k_pool, v_pool, block_tables, seq_lens, query_start_loc)
    if out is None:
        out = torch.empty_like(q)
    else:
        _need(out, "out", torch.bfloat16, 3)
        if out.shape != q.shape:
            raise ValueError("out must have q's shape")
    dims = make_dims(tuple(q.shape), tuple(k_pool.shape), R, block_tables.shape[1])
    if workspace is not None and workspace.counter_dims != (dims.num_q_tokens, dims.num_kv_heads):
        pkv_workspace_init(workspace, dims, stream)
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (workspace.ptr, workspace.nbytes)
    _check(load_library().pkv_attention(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k_pool.data_ptr()),
        ctypes.c_void_p(v_pool.data_ptr()), ctypes.c_void_p(block_tables.data_ptr()),
        ctypes.c_void_p(seq_lens.data_ptr()), ctypes.c_void_p(query_start_loc.data_ptr()),
        ctypes.c_float(scale), ctypes.c_void_p(out.data_ptr()), ctypes.byref(dims),
        ctypes.c_void_p(ws_ptr), ws_bytes, ctypes.c_void_p(_stream(stream, q.device))))
    return out


def pkv_append_attention(k_new, v_new, slot_mapping, k_pool, v_pool, q, block_tables, seq_lens,
                         query_start_loc, scale, out=None, workspace: Workspace | None = None,
                         stream=None):
    """One layer of an engine step: append the step's new K/V rows (one per
    query token, slot_mapping [Tq] int64 holding each token's own position),
    then attend; returns out [Tq, Hq, D] bf16."""
    _need(k_new, "k_new", torch.bfloat16, 3)
    _need(v_new, "v_new", torch.bfloat16, 3)
    _need(slot_mapping, "slot_mapping", torch.int64, 1)
    _need(q, "q", torch.bfloat16, 3)
    _need(k_pool, "k_pool", torch.bfloat16, 4)
    _need(v_pool, "v_pool", torch.bfloat16, 4)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    _need(query_start_loc, "query_start_loc", torch.int32, 1)
    T = q.shape[0]
    if k_new.shape[0] != T or v_new.shape != k_new.shape or slot_mapping.shape[0] != T:
        raise ValueError("k_new, v_new and slot_mapping need one row per query token")
    if v_pool.shape != k_pool.shape or k_pool.shape[1] != k_new.shape[1] or \
            k_pool.shape[3] != k_new.shape[2] or k_pool.shape[3] != q.shape[2]:
        raise ValueError("pool / new rows / q shape mismatch")
    R = check_attention_shapes(q, k_pool, v_pool, block_tables, seq_lens, query_start_loc)
    if out is None:
        out = torch.empty_like(q)
    else:
        _need(out, "out", torch.bfloat16, 3)
        if out.shape != q.shape:
            raise ValueError("out must have q's shape")
    dims = make_dims(tuple(q.shape), tuple(k_pool.shape), R, block_tables.shape[1])
    if workspace is not None and workspace.counter_dims != (dims.num_q_tokens, dims.num_kv_heads):
        pkv_workspace_init(workspace, dims, stream)
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (workspace.ptr, workspace.nbytes)
    _check(load_library().pkv_append_attention(
        ctypes.c_void_p(k_new.data_ptr()), ctypes.c_void_p(v_new.data_ptr()),
        ctypes.c_void_p(slot_mapping.data_ptr()), ctypes.c_void_p(k_pool.data_ptr()),
        ctypes.c_void_p(v_pool.data_ptr()), ctypes.c_void_p(q.data_ptr()),
        ctypes.c_void_p(block_tables.data_ptr()), ctypes.c_void_p(seq_lens.data_ptr()),
        ctypes.c_void_p(query_start_loc.data_ptr()), ctypes.c_float(scale),
        ctypes.c_void_p(out.data_ptr()), ctypes.byref(dims), ctypes.c_void_p(ws_ptr), ws_bytes,
        ctypes.c_void_p(_stream(stream, q.device))))
    return out


def _need_scales(k_scale, v_scale, Hkv: int):
    for t, name in ((k_scale, "k_scale"), (v_scale, "v_scale")):
        _need(t, name, torch.float32, 1)
        if t.shape[0] != Hkv:
            raise ValueError(f"{name} must have num_kv_heads = {Hkv} entries")


def pkv_append_fp8(k_new, v_new, slot_mapping, k_pool, v_pool, k_scale, v_scale, stream=None):
    """Quantise k_new/v_new [T, Hkv, D] bf16 into e4m3 pools (uint8
    [blocks, Hkv, 16, D]) at slot_mapping [T] int64, with the per-KV-head
    scales k_scale / v_scale [Hkv] fp32: code = e4m3(x / scale)."""
    _need(k_new, "k_new", torch.bfloat16, 3)
    _need(v_new, "v_new", torch.bfloat16, 3)
    _need(slot_mapping, "slot_mapping", torch.int64, 1)
    _need(k_pool, "k_pool", torch.uint8, 4)
    _need(v_pool, "v_pool", torch.uint8, 4)
    T = k_new.shape[0]
    if v_new.shape != k_new.shape or slot_mapping.shape[0] != T:
        raise ValueError("k_new, v_new and slot_mapping disagree on the token count")
    if v_pool.shape != k_pool.shape or k_pool.shape[1] != k_new.shape[1] or \
            k_pool.shape[3] != k_new.shape[2]:
        raise ValueError("pool shape does not match the new rows")
    nb, Hkv, bs, D = k_pool.shape
    _need_scales(k_scale, v_scale, Hkv)
    dims = Dims(0, 0, Hkv, Hkv, D, bs, nb, 0)
    _check(load_library().pkv_append_fp8(
        ctypes.c_void_p(k_new.data_ptr()), ctypes.c_void_p(v_new.data_ptr()),
        ctypes.c_void_p(slot_mapping.data_ptr()), ctypes.c_void_p(k_pool.data_ptr()),
        ctypes.c_void_p(v_pool.data_ptr()), ctypes.c_void_p(k_scale.data_ptr()),
        ctypes.c_void_p(v_scale.data_ptr()), T, ctypes.byref(dims),
        ctypes.c_void_p(_stream(stream, k_pool.device))))


def pkv_attention_fp8kv(q, k_pool, v_pool, k_scale, v_scale, block_tables, seq_lens,
                        query_start_loc, scale, out=None, workspace: Workspace | None = None,
                        stream=None):
    """pkv_attention over e4m3 pools (uint8) dequantised by the per-KV-head
    scales k_scale / v_scale [Hkv] fp32; returns out [Tq, Hq, D] bf16."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k_pool, "k_pool", torch.uint8, 4)
    _need(v_pool, "v_pool", torch.uint8, 4)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    _need(query_start_loc, "query_start_loc", torch.int32, 1)
    R = check_attention_shapes(q, k_pool, v_pool, block_tables, seq_lens, query_start_loc)
    _need_scales(k_scale, v_scale, k_pool.shape[1])
    if out is None:
        out = torch.empty_like(q)
    else:
        _need(out, "out", torch.bfloat16, 3)
        if out.shape != q.shape:
            raise ValueError("out must have q's shape")
    dims = make_dims(tuple(q.shape), tuple(k_pool.shape), R, block_tables.shape[1])
    if workspace is not None and workspace.counter_dims != (dims.num_q_tokens, dims.num_kv_heads):
        pkv_workspace_init(workspace, dims, stream)
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (workspace.ptr, workspace.nbytes)
    _check(load_library().pkv_attention_fp8kv(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k_pool.data_ptr()),
        ctypes.c_void_p(v_pool.data_ptr()), ctypes.c_void_p(k_scale.data_ptr()),
        ctypes.c_void_p(v_scale.data_ptr()), ctypes.c_void_p(block_tables.data_ptr()),
        ctypes.c_void_p(seq_lens.data_ptr()), ctypes.c_void_p(query_start_loc.data_ptr()),
        ctypes.c_float(scale), ctypes.c_void_p(out.data_ptr()), ctypes.byref(dims),
        ctypes.c_void_p(ws_ptr), ws_bytes, ctypes.c_void_p(_stream(stream, q.device))))
    return out


def pkv_append_attention_fp8(k_new, v_new, slot_mapping, k_pool, v_pool, k_scale, v_scale, q,
                             block_tables, seq_lens, query_start_loc, scale, out=None,
                             workspace: Workspace | None = None, stream=None):
    """One layer of an engine step over e4m3 pools: quantise and append the
    step's new K/V rows (one per query token), then attend; returns out
    [Tq, Hq, D] bf16."""
    _need(k_new, "k_new", torch.bfloat16, 3)
    _need(v_new, "v_new", torch.bfloat16, 3)
    _need(slot_mapping, "slot_mapping", torch.int64, 1)
    _need(q, "q", torch.bfloat16, 3)
    _need(k_pool, "k_pool", torch.uint8, 4)
    _need(v_pool, "v_pool", torch.uint8, 4)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    _need(query_start_loc, "query_start_loc", torch.int32, 1)
    T = q.shape[0]
    if k_new.shape[0] != T or v_new.shape != k_new.shape or slot_mapping.shape[0] != T:
        raise ValueError("k_new, v_new and slot_mapping need one row per query token")
    if k_pool.shape[1] != k_new.shape[1] or k_pool.shape[3] != k_new.shape[2]:
        raise ValueError("pool / new rows shape mismatch")
    R = check_attention_shapes(q, k_pool, v_pool, block_tables, seq_lens, query_start_loc)
    _need_scales(k_scale, v_scale, k_pool.shape[1])
    if out is None:
        out = torch.empty_like(q)
    else:
        _need(out, "out", torch.bfloat16, 3)
        if out.shape != q.shape:
            raise ValueError("out must have q's shape")
    dims = make_dims(tuple(q.shape), tuple(k_pool.shape), R, block_tables.shape[1])
    if workspace is not None and workspace.counter_dims != (dims.num_q_tokens, dims.num_kv_heads):
        pkv_workspace_init(workspace, dims, stream)
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (workspace.ptr, workspace.nbytes)
    _check(load_library().pkv_append_attention_fp8(
        ctypes.c_void_p(k_new.data_ptr()), ctypes.c_void_p(v_new.data_ptr()),
        ctypes.c_void_p(slot_mapping.data_ptr()), ctypes.c_void_p(k_pool.data_ptr()),
        ctypes.c_void_p(v_pool.data_ptr()), ctypes.c_void_p(k_scale.data_ptr()),
        ctypes.c_void_p(v_scale.data_ptr()), ctypes.c_void_p(q.data_ptr()),
        ctypes.c_void_p(block_tables.data_ptr()), ctypes.c_void_p(seq_lens.data_ptr()),
        ctypes.c_void_p(query_start_loc.data_ptr()), ctypes.c_float(scale),
        ctypes.c_void_p(out.data_ptr()), ctypes.byref(dims), ctypes.c_void_p(ws_ptr), ws_bytes,
        ctypes.c_void_p(_stream(stream, q.device))))
    return out


class CascadeWorkspace(Workspace):
    """A zero-initialised device workspace for pkv_attention_cascade."""

    def __init__(self, dims: Dims, device="cuda"):
        self.nbytes = int(load_library().pkv_cascade_workspace_size(ctypes.byref(dims)))
        if self.nbytes == 0:
            raise PagedKVError(PKV_ERR_INVALID, pkv_last_error() or "bad dims")
        self.buf = torch.zeros(self.nbytes + 256, dtype=torch.uint8, device=device)
        off = (-self.buf.data_ptr()) % 256
        self.ptr = self.buf.data_ptr() + off
        self.counter_dims = (dims.num_q_tokens, dims.num_kv_heads)


def pkv_attention_cascade(q, k_pool, v_pool, block_tables, seq_lens, query_start_loc,
                          group_first_req, group_num_reqs, group_prefix_blocks, scale,
                          out=None, workspace: CascadeWorkspace | None = None, stream=None):
    """pkv_attention for requests that share prompts: group g is the requests
    group_first_req[g] .. + group_num_reqs[g] - 1, whose first
    group_prefix_blocks[g] table entries are the same physical blocks (int32
    CUDA tensors).  The shared blocks are read once per batch."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k_pool, "k_pool", torch.bfloat16, 4)
    _need(v_pool, "v_pool", torch.bfloat16, 4)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    _need(query_start_loc, "query_start_loc", torch.int32, 1)
    for t, name in ((group_first_req, "group_first_req"), (group_num_reqs, "group_num_reqs"),
                    (group_prefix_blocks, "group_prefix_blocks")):
        _need(t, name, torch.int32, 1)
    G = group_first_req.shape[0]
    if group_num_reqs.shape[0] != G or group_prefix_blocks.shape[0] != G:
        raise ValueError("group arrays disagree on the group count")
    R = check_attention_shapes(q, k_pool, v_pool, block_tables, seq_lens, query_start_loc)
    if out is None:
        out = torch.empty_like(q)
    else:
        _need(out, "out", torch.bfloat16, 3)
        if out.shape != q.shape:
            raise ValueError("out must have q's shape")
    dims = make_dims(tuple(q.shape), tuple(k_pool.shape), R, block_tables.shape[1])
    if workspace is None:
        workspace = CascadeWorkspace(dims, device=q.device)
    if workspace.counter_dims != (dims.num_q_tokens, dims.num_kv_heads):
        pkv_workspace_init(workspace, dims, stream)
    _check(load_library().pkv_attention_cascade(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k_pool.data_ptr()),
        ctypes.c_void_p(v_pool.data_ptr()), ctypes.c_void_p(block_tables.data_ptr()),
        ctypes.c_void_p(seq_lens.data_ptr()), ctypes.c_void_p(query_start_loc.data_ptr()),
        ctypes.c_void_p(group_first_req.data_ptr()), ctypes.c_void_p(group_num_reqs.data_ptr()),
        ctypes.c_void_p(group_prefix_blocks.data_ptr()), G, ctypes.c_float(scale),
        ctypes.c_void_p(out.data_ptr()), ctypes.byref(dims), ctypes.c_void_p(workspace.ptr),
        workspace.nbytes, ctypes.c_void_p(_stream(stream, q.device))))
    return out


def pkv_attention_noalloc(q, k_pool, v_pool, block_tables, seq_lens, query_start_loc, scale,
                          out, stream=None):
    """pkv_attention for callers that cannot allocate: the library's static
    scratch array replaces the workspace and `out` must be given (nothing is
    allocated here either).  Calls sharing the scratch must not overlap."""
    for t, name, dt, nd in ((q, "q", torch.bfloat16, 3), (k_pool, "k_pool", torch.bfloat16, 4),
                            (v_pool, "v_pool", torch.bfloat16, 4),
                            (block_tables, "block_tables", torch.int32, 2),
                            (seq_lens, "seq_lens", torch.int32, 1),
                            (query_start_loc, "query_start_loc", torch.int32, 1),
                            (out, "out", torch.bfloat16, 3)):
        _need(t, name, dt, nd)
    R = check_attention_shapes(q, k_pool, v_pool, block_tables, seq_lens, query_start_loc, out)
    dims = make_dims(tuple(q.shape), tuple(k_pool.shape), R, block_tables.shape[1])
    _check(load_library().pkv_attention_noalloc(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k_pool.data_ptr()),
        ctypes.c_void_p(v_pool.data_ptr()), ctypes.c_void_p(block_tables.data_ptr()),
        ctypes.c_void_p(seq_lens.data_ptr()), ctypes.c_void_p(query_start_loc.data_ptr()),
        ctypes.c_float(scale), ctypes.c_void_p(out.data_ptr()), ctypes.byref(dims),
        ctypes.c_void_p(_stream(stream, q.device))))
    return out


def pkv_copy_blocks(k_src, v_src, k_dst, v_dst, pairs, stream=None):
    """Copy whole blocks (all KV heads, K and V): block pairs[i, 0] of the
    source pools to block pairs[i, 1] of the destination pools.  The pools may
    be CUDA tensors or pinned host tensors (swap out / in); pairs is an int64
    CUDA tensor [n, 2]."""
    for t, name in ((k_src, "k_src"), (v_src, "v_src"), (k_dst, "k_dst"), (v_dst, "v_dst")):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or t.dim() != 4 \
                or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 [blocks, Hkv, 16, 128] tensor")
        if not (t.is_cuda or t.is_pinned()):
            raise ValueError(f"{name} must be a CUDA tensor or pinned host memory")
    _need(pairs, "pairs", torch.int64, 2)
    if k_src.shape[1:] != k_dst.shape[1:] or v_src.shape != k_src.shape or v_dst.shape != k_dst.shape:
        raise ValueError("pool shapes disagree")
    nb, Hkv, bs, D = k_src.shape
    dims = Dims(0, 0, Hkv, Hkv, D, bs, nb, 0)
    dev = pairs.device
    _check(load_library().pkv_copy_blocks(
        ctypes.c_void_p(k_src.data_ptr()), ctypes.c_void_p(v_src.data_ptr()),
        ctypes.c_void_p(k_dst.data_ptr()), ctypes.c_void_p(v_dst.data_ptr()),
        ctypes.c_void_p(pairs.data_ptr()), pairs.shape[0], k_src.shape[0], k_dst.shape[0],
        ctypes.byref(dims), ctypes.c_void_p(_stream(stream, dev))))


def pkv_get_device_error(stream=None) -> int:
    """Synchronise the stream; return (and clear) the device error code."""
    dev = torch.cuda.current_device()
    return int(load_library().pkv_get_device_error(ctypes.c_void_p(_stream(stream, dev))))


# The names the step's calls go by in the serving literature.
paged_kv_append = pkv_append
paged_attention = pkv_attention
