"""Host-side checks of the C ABI that need no GPU: the library builds, loads,
exports every symbol include/pagedkv.h declares, and rejects bad arguments
with the documented codes before touching the device."""
import ctypes
import os
import re

import pytest

import paged_kv_cache_195_gb300 as pkv
from paged_kv_cache_195_gb300 import _binding as b
from paged_kv_cache_195_gb300 import build as pkv_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    pkv_build.build()
    return pkv.load_library()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "pagedkv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared_functions()
    assert "pkv_append" in names and "pkv_attention" in names
    assert set(b.EXPORTED) <= set(names)


def test_every_declared_symbol_is_exported(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_constants_match_header():
    text = open(os.path.join(ROOT, "include", "pagedkv.h")).read()
    for name in ("PKV_OK", "PKV_ERR_INVALID", "PKV_ERR_UNSUPPORTED", "PKV_ERR_WORKSPACE",
                 "PKV_ERR_CUDA", "PKV_ERR_DEVICE_BOUNDS", "PKV_ERR_TIMEOUT"):
        m = re.search(rf"#define {name} \(?(-?\d+)\)?", text)
        assert m and int(m.group(1)) == getattr(b, name), name


def _dims(**kw):
    d = dict(num_reqs=2, num_q_tokens=2, num_q_heads=12, num_kv_heads=2, head_dim=128,
             block_size=16, num_blocks=8, max_blocks_per_req=4)
    d.update(kw)
    return b.Dims(*[d[f] for f, _ in b.Dims._fields_])


def _attn(lib, dims, null_q=False):
    fake = ctypes.c_void_p(0x1000)   # never dereferenced: validation fails first
    q = ctypes.c_void_p(0) if null_q else fake
    return lib.pkv_attention(q, fake, fake, fake, fake, fake, ctypes.c_float(0.1), fake,
                             ctypes.byref(dims), None, 0, None)


@pytest.mark.parametrize("kw,code", [
    (dict(head_dim=64), b.PKV_ERR_UNSUPPORTED),
    (dict(block_size=32), b.PKV_ERR_UNSUPPORTED),
    (dict(num_q_heads=13), b.PKV_ERR_INVALID),
    (dict(num_q_heads=18), b.PKV_ERR_UNSUPPORTED),      # group of 9
    (dict(num_reqs=70000), b.PKV_ERR_UNSUPPORTED),
    (dict(num_kv_heads=0), b.PKV_ERR_INVALID),
    (dict(num_q_tokens=-1), b.PKV_ERR_INVALID),
])
def test_attention_rejects_bad_dims(lib, kw, code):
    assert _attn(lib, _dims(**kw)) == code
    assert lib.pkv_last_error().decode()


def test_attention_rejects_null_pointer(lib):
    assert _attn(lib, _dims(), null_q=True) == b.PKV_ERR_INVALID


def test_empty_step_is_a_no_op(lib):
    assert _attn(lib, _dims(num_reqs=0, num_q_tokens=0)) == b.PKV_OK


def test_append_rejects_bad_arguments(lib):
    fake = ctypes.c_void_p(0x1000)
    d = _dims(head_dim=256)
    assert lib.pkv_append(fake, fake, fake, fake, fake, 3, ctypes.byref(d), None) == \
        b.PKV_ERR_UNSUPPORTED
    d = _dims()
    assert lib.pkv_append(fake, fake, fake, fake, fake, -1, ctypes.byref(d), None) == \
        b.PKV_ERR_INVALID
    assert lib.pkv_append(None, fake, fake, fake, fake, 3, ctypes.byref(d), None) == \
        b.PKV_ERR_INVALID
    misaligned = ctypes.c_void_p(0x1008)
    assert lib.pkv_append(misaligned, fake, fake, fake, fake, 3, ctypes.byref(d), None) == \
        b.PKV_ERR_INVALID
    assert lib.pkv_append(fake, fake, fake, fake, fake, 0, ctypes.byref(d), None) == b.PKV_OK


def test_binding_refuses_cpu_tensors():
    import torch
    x = torch.zeros(1, 2, 128, dtype=torch.bfloat16)
    pool = torch.zeros(4, 2, 16, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        pkv.pkv_append(x, x, torch.zeros(1, dtype=torch.int64), pool, pool)


def test_one_layer_call_validates_like_its_parts(lib):
    fake = ctypes.c_void_p(0x1000)
    args = lambda d, k_new=fake: (k_new, fake, fake, fake, fake, fake, fake, fake, fake,
                                  ctypes.c_float(0.1), fake, ctypes.byref(d), None, 0, None)
    assert lib.pkv_append_attention(*args(_dims(head_dim=64))) == b.PKV_ERR_UNSUPPORTED
    assert lib.pkv_append_attention(*args(_dims(num_q_heads=13))) == b.PKV_ERR_INVALID
    assert lib.pkv_append_attention(*args(_dims(), k_new=None)) == b.PKV_ERR_INVALID
    assert lib.pkv_append_attention(*args(_dims(num_reqs=0, num_q_tokens=0))) == b.PKV_OK


def test_cascade_call_rejects_bad_groups_before_the_device(lib):
    fake = ctypes.c_void_p(0x1000)
    d = _dims()

    def call(first, count, blocks, n):
        return lib.pkv_attention_cascade(fake, fake, fake, fake, fake, fake, first, count, blocks,
                                         n, ctypes.c_float(0.1), fake, ctypes.byref(d), fake,
                                         1 << 20, None)
    assert call(fake, fake, fake, -1) == b.PKV_ERR_INVALID
    assert call(None, fake, fake, 2) == b.PKV_ERR_INVALID
    assert call(fake, fake, None, 1) == b.PKV_ERR_INVALID


def test_fp8_calls_reject_bad_arguments(lib):
    fake = ctypes.c_void_p(0x1000)
    d = _dims()
    # attention over e4m3 pools needs both scale arrays
    assert lib.pkv_attention_fp8kv(fake, fake, fake, None, fake, fake, fake, fake,
                                   ctypes.c_float(0.1), fake, ctypes.byref(d), None, 0,
                                   None) == b.PKV_ERR_INVALID
    assert lib.pkv_append_fp8(fake, fake, fake, fake, fake, fake, None, 3, ctypes.byref(d),
                              None) == b.PKV_ERR_INVALID
    assert lib.pkv_append_fp8(fake, fake, fake, fake, fake, fake, fake, -2, ctypes.byref(d),
                              None) == b.PKV_ERR_INVALID
    assert lib.pkv_append_fp8(fake, fake, fake, fake, fake, fake, fake, 0, ctypes.byref(d),
                              None) == b.PKV_OK


def test_copy_blocks_rejects_bad_arguments(lib):
    fake = ctypes.c_void_p(0x1000)
    d = _dims()
    assert lib.pkv_copy_blocks(fake, fake, fake, fake, fake, -1, 8, 8, ctypes.byref(d),
                               None) == b.PKV_ERR_INVALID
    assert lib.pkv_copy_blocks(fake, fake, fake, fake, None, 2, 8, 8, ctypes.byref(d),
                               None) == b.PKV_ERR_INVALID
    assert lib.pkv_copy_blocks(fake, fake, fake, fake, fake, 0, 8, 8, ctypes.byref(d),
                               None) == b.PKV_OK
