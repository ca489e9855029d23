"""pkv_attention_noalloc: attention for callers that cannot allocate.

Callers that may not call cudaMalloc (plugins whose host framework owns all
device memory, serving loops that forbid allocation after start-up) use this
entry point; its scratch is a fixed array inside the library.  Its output
must match the regular entry point's and the fp64 oracle's, call after call,
even when the dims (and so the scratch layout) change between calls.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_195_gb300 as pkv
from paged_kv_cache_195_gb300 import build as pkv_build
from paged_kv_cache_195_gb300 import workloads as wl

from pkv_testutil import (MAX_ABS, MEAN_ABS, assert_close, host_copy, oracle_full,
                          oracle_pools_after_append, to_f64)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv_build.build()
    pkv.load_library()


def _both(shape):
    inp = wl.make_step(shape, device="cuda", poison=True)
    h = host_copy(inp)
    kp, vp = oracle_pools_after_append(h)
    pkv.pkv_append(inp.k_new, inp.v_new, inp.slot_mapping, inp.k_pool, inp.v_pool)
    ref = pkv.pkv_attention(inp.q, inp.k_pool, inp.v_pool, inp.block_tables, inp.seq_lens,
                            inp.query_start_loc, inp.scale)
    out = torch.full_like(inp.q, float("nan"))
    pkv.pkv_attention_noalloc(inp.q, inp.k_pool, inp.v_pool, inp.block_tables, inp.seq_lens,
                              inp.query_start_loc, inp.scale, out)
    torch.cuda.synchronize()
    assert pkv.pkv_get_device_error() == 0, pkv.pkv_last_error()
    got, want = out.double().cpu().numpy(), ref.double().cpu().numpy()
    assert np.isfinite(got).all()
    err = np.abs(got - want)
    assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, (err.max(), err.mean())
    # and against the fp64 oracle on the same inputs (its own append)
    assert_close(to_f64(out), oracle_full(h, kp, vp), shape.name)


def test_noalloc_matches_pkv_attention_on_consecutive_calls():
    # first call: long contexts split across CTAs (the scratch carries the
    # partial results); second call: different dims, so the counter region
    # the first call left behind is laid out differently
    _both(wl.StepShape("noalloc_a", [3000, 1200, 17, 513], [1, 3, 1, 1], 32, 8, seed=61))
    _both(wl.StepShape("noalloc_b", [700, 2048, 40, 90, 5], [1, 1, 40, 2, 1], 12, 2, seed=62))


def test_noalloc_rejects_dims_beyond_the_array():
    big = pkv.Dims(1, 600_000, 8, 8, 128, 16, 64, 4)  # counters alone exceed the array
    fake = torch.zeros(16, dtype=torch.uint8, device="cuda")
    p = fake.data_ptr()
    import ctypes
    rc = pkv.load_library().pkv_attention_noalloc(
        ctypes.c_void_p(p), ctypes.c_void_p(p), ctypes.c_void_p(p), ctypes.c_void_p(p),
        ctypes.c_void_p(p), ctypes.c_void_p(p), ctypes.c_float(0.1), ctypes.c_void_p(p),
        ctypes.byref(big), None)
    assert rc == pkv._binding.PKV_ERR_WORKSPACE
    assert "static array" in pkv.pkv_last_error()
