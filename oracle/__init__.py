"""fp64 CPU oracle for the paged-attention step -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The CUDA
library never links, loads or calls it, and nothing here imports the CUDA
library or its Python binding: the two sides share only the seeded input
generator.

The arithmetic lives in ``pkv_oracle.c`` (plain loops, fp64, OpenMP across
independent (query token, query head) rows); this module compiles it with gcc
and marshals numpy arrays into it.  bf16 tensors travel as their uint16 bit
patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``pkv_oracle.c`` into ``oracle/_build/liboracle.so``."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC",
                               "-std=c11", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            p = ctypes.c_void_p
            i32, i64 = ctypes.c_int32, ctypes.c_int64
            lib.oracle_append.argtypes = [p, p, p, i64, i64, i64, i64, i64, p, p]
            lib.oracle_append.restype = ctypes.c_int
            lib.oracle_paged_attention.argtypes = [
                p, p, p, p, p, p, i32, i32, i32, i32, i32, i32, i32,
                ctypes.c_double, p]
            lib.oracle_paged_attention.restype = ctypes.c_int
            u8 = ctypes.c_uint8
            lib.oracle_e4m3_decode.argtypes = [u8]
            lib.oracle_e4m3_decode.restype = ctypes.c_double
            lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
            lib.oracle_e4m3_encode.restype = u8
            lib.oracle_append_fp8.argtypes = [p, p, p, i64, i64, i64, i64, i64, p, p, p, p]
            lib.oracle_append_fp8.restype = ctypes.c_int
            lib.oracle_paged_attention_fp8.argtypes = [
                p, p, p, p, p, p, p, p, i32, i32, i32, i32, i32, i32, i32, ctypes.c_double, p]
            lib.oracle_paged_attention_fp8.restype = ctypes.c_int
            lib.oracle_copy_blocks.argtypes = [p, p, p, p, p, i64, i64, i64, i64, i64, i64]
            lib.oracle_copy_blocks.restype = ctypes.c_int
            lib.oracle_set_threads.argtypes = [ctypes.c_int]
            lib.oracle_set_threads.restype = None
            lib.oracle_max_threads.argtypes = []
            lib.oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def append(k_new, v_new, slot_mapping, k_pool, v_pool):
    """Scatter new K/V rows (bf16 bit patterns) into copies of the pools.

    k_new, v_new: uint16 [T, Hkv, D]; slot_mapping: int64 [T], negative = skip;
    k_pool, v_pool: uint16 [num_blocks, Hkv, bs, D].  Returns the new pools.
    """
    k_new, v_new = _c(k_new, np.uint16), _c(v_new, np.uint16)
    slots = _c(slot_mapping, np.int64)
    kp, vp = _c(k_pool, np.uint16).copy(), _c(v_pool, np.uint16).copy()
    T, Hkv, D = k_new.shape
    nb, hkv2, bs, d2 = kp.shape
    assert (hkv2, d2) == (Hkv, D) and v_new.shape == k_new.shape
    assert slots.shape == (T,) and vp.shape == kp.shape
    rc = _load().oracle_append(_ptr(k_new), _ptr(v_new), _ptr(slots), T, Hkv,
                               D, bs, nb, _ptr(kp), _ptr(vp))
    if rc != 0:
        raise ValueError(f"oracle_append: slot outside the pool (rc={rc})")
    return kp, vp


def paged_attention(q, k_pool, v_pool, block_tables, seq_lens,
                    query_start_loc, scale, num_threads: int | None = None):
    """softmax(scale q K^T) V per request, causal, gathered through the table.

    q: uint16 [Tq, Hq, D]; pools uint16 [num_blocks, Hkv, bs, D];
    block_tables int32 [R, max_blocks]; seq_lens int32 [R];
    query_start_loc int32 [R+1].  Returns float64 [Tq, Hq, D].
    """
    q = _c(q, np.uint16)
    kp, vp = _c(k_pool, np.uint16), _c(v_pool, np.uint16)
    bt = _c(block_tables, np.int32)
    sl = _c(seq_lens, np.int32)
    qsl = _c(query_start_loc, np.int32)
    Tq, Hq, D = q.shape
    nb, Hkv, bs, d2 = kp.shape
    R = sl.shape[0]
    assert d2 == D and vp.shape == kp.shape and qsl.shape == (R + 1,)
    assert bt.ndim == 2 and bt.shape[0] == R and int(qsl[-1]) == Tq
    out = np.zeros((Tq, Hq, D), dtype=np.float64)
    if num_threads is not None:
        set_threads(num_threads)
    rc = _load().oracle_paged_attention(
        _ptr(q), _ptr(kp), _ptr(vp), _ptr(bt), _ptr(sl), _ptr(qsl), R, Hq, Hkv,
        D, bs, nb, bt.shape[1], float(scale), _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle_paged_attention: inconsistent inputs (rc={rc})")
    return out


def e4m3_decode(code: int) -> float:
    """Value of an e4m3 code (NaN for the NaN patterns)."""
    return float(_load().oracle_e4m3_decode(int(code) & 0xFF))


def e4m3_encode(x: float) -> int:
    """Nearest e4m3 code to the fp32 value x (ties to even, saturating)."""
    return int(_load().oracle_e4m3_encode(float(np.float32(x))))


def append_fp8(k_new, v_new, slot_mapping, k_pool, v_pool, k_scale, v_scale):
    """Quantise new rows (bf16 bits) into copies of uint8 e4m3 pools:
    code = encode(fp32(x) / fp32(scale[h]))."""
    k_new, v_new = _c(k_new, np.uint16), _c(v_new, np.uint16)
    slots = _c(slot_mapping, np.int64)
    kp, vp = _c(k_pool, np.uint8).copy(), _c(v_pool, np.uint8).copy()
    ks, vs = _c(k_scale, np.float32), _c(v_scale, np.float32)
    T, Hkv, D = k_new.shape
    nb, _, bs, _ = kp.shape
    rc = _load().oracle_append_fp8(_ptr(k_new), _ptr(v_new), _ptr(slots), T, Hkv, D, bs, nb,
                                   _ptr(ks), _ptr(vs), _ptr(kp), _ptr(vp))
    if rc != 0:
        raise ValueError("oracle_append_fp8: slot outside the pool")
    return kp, vp


def paged_attention_fp8(q, k_pool, v_pool, k_scale, v_scale, block_tables, seq_lens,
                        query_start_loc, scale):
    """paged_attention over uint8 e4m3 pools dequantised by per-KV-head scales."""
    q = _c(q, np.uint16)
    kp, vp = _c(k_pool, np.uint8), _c(v_pool, np.uint8)
    ks, vs = _c(k_scale, np.float32), _c(v_scale, np.float32)
    bt = _c(block_tables, np.int32)
    sl = _c(seq_lens, np.int32)
    qsl = _c(query_start_loc, np.int32)
    Tq, Hq, D = q.shape
    nb, Hkv, bs, _ = kp.shape
    R = sl.shape[0]
    out = np.zeros((Tq, Hq, D), dtype=np.float64)
    rc = _load().oracle_paged_attention_fp8(
        _ptr(q), _ptr(kp), _ptr(vp), _ptr(ks), _ptr(vs), _ptr(bt), _ptr(sl), _ptr(qsl), R, Hq,
        Hkv, D, bs, nb, bt.shape[1], float(scale), _ptr(out))
    if rc != 0:
        raise ValueError("oracle_paged_attention_fp8: inconsistent inputs")
    return out


def copy_blocks(k_src, v_src, k_dst, v_dst, pairs):
    """Copies of the destination pools after moving whole blocks: block
    pairs[i, 0] of the source pools to block pairs[i, 1] of the destination."""
    ks, vs = _c(k_src, np.uint16), _c(v_src, np.uint16)
    kd, vd = _c(k_dst, np.uint16).copy(), _c(v_dst, np.uint16).copy()
    pr = _c(pairs, np.int64).reshape(-1, 2)
    nb_s, Hkv, bs, D = ks.shape
    assert kd.shape[1:] == (Hkv, bs, D) and vs.shape == ks.shape and vd.shape == kd.shape
    rc = _load().oracle_copy_blocks(_ptr(ks), _ptr(vs), _ptr(kd), _ptr(vd), _ptr(pr), pr.shape[0],
                                    nb_s, kd.shape[0], Hkv, bs, D)
    if rc != 0:
        raise ValueError("oracle_copy_blocks: block outside its pool")
    return kd, vd


def set_threads(n: int) -> None:
    """Number of OpenMP threads later oracle calls use."""
    _load().oracle_set_threads(int(n))


def max_threads() -> int:
    """Threads an oracle call will use."""
    return int(_load().oracle_max_threads())


def kv_cache_bytes(layers, kv_heads, head_dim, dtype_bytes, seq_len, batch):
    """Bytes of K and V cached: 2 tensors x layers x KV heads x head dim x
    bytes per element x tokens x sequences (What Actually Runs the Model,
    "The KV cache")."""
    return 2 * layers * kv_heads * head_dim * dtype_bytes * seq_len * batch
