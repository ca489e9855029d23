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


# ---------------------------------------------------------------------------
# launch and routing options (pkv_options)
# ---------------------------------------------------------------------------

def test_options_struct_matches_header():
    text = open(os.path.join(ROOT, "include", "pagedkv.h")).read()
    body = re.search(r"typedef struct pkv_options \{(.*?)\} pkv_options;", text, re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    fields = re.findall(r"int32_t\s+(\w+);", body)
    assert tuple(fields) == b.OPTION_FIELDS


def test_options_defaults_and_round_trip(lib):
    o = pkv.get_options()
    assert o["pdl"] in (0, 1) and o["min_chunk"] >= 1 and o["wait_limit_us"] >= 1
    assert o["debug_withhold_q"] == 0 and 0 <= o["rowgroup_cost"] <= 1024
    with pkv.options(prefill_min_q=3, decode_tc=0):
        now = pkv.get_options()
        assert now["prefill_min_q"] == 3 and now["decode_tc"] == 0
        assert {k: v for k, v in now.items() if k not in ("prefill_min_q", "decode_tc")} == \
            {k: v for k, v in o.items() if k not in ("prefill_min_q", "decode_tc")}
    assert pkv.get_options() == o


@pytest.mark.parametrize("bad", [{"min_chunk": 0}, {"wait_limit_us": 0}, {"prefill_min_q": -1},
                                 {"align_slack": -5}, {"decode_grid": -1},
                                 {"rowgroup_cost": -1}, {"rowgroup_cost": 1025}])
def test_out_of_range_options_are_rejected(lib, bad):
    o = pkv.get_options()
    with pytest.raises(pkv.PagedKVError) as e:
        pkv.set_options(**bad)
    assert e.value.code == b.PKV_ERR_INVALID
    assert pkv.get_options() == o


def test_options_come_from_the_environment_once(tmp_path):
    code = ("import paged_kv_cache_195_gb300 as pkv, os, json\n"
            "a = pkv.get_options()\n"
            "os.environ['PKV_PREFILL_MIN_Q'] = '9'\n"
            "b = pkv.get_options()\n"
            "print(json.dumps([a['prefill_min_q'], a['decode_tc'], a['wait_limit_us'],"
            " b['prefill_min_q']]))\n")
    env = dict(os.environ, PKV_PREFILL_MIN_Q="7", PKV_DECODE_TC="0", PKV_WAIT_LIMIT_US="1000")
    import json
    import subprocess
    import sys
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                       cwd=ROOT, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    # read at first use; a later change of the environment is not seen
    assert json.loads(r.stdout.strip().splitlines()[-1]) == [7, 0, 1000, 7]


# ---------------------------------------------------------------------------
# shape checks of the Python binding (before any launch)
# ---------------------------------------------------------------------------

def _attention_tensors(v_pool_shape=None, out_shape=None, R=3):
    import torch
    q = torch.zeros(4, 12, 128, dtype=torch.bfloat16)
    kp = torch.zeros(10, 2, 16, 128, dtype=torch.bfloat16)
    vp = torch.zeros(*(v_pool_shape or kp.shape), dtype=torch.bfloat16)
    bt = torch.zeros(R, 5, dtype=torch.int32)
    sl = torch.zeros(R, dtype=torch.int32)
    qsl = torch.zeros(R + 1, dtype=torch.int32)
    out = torch.zeros(*(out_shape or q.shape), dtype=torch.bfloat16)
    return q, kp, vp, bt, sl, qsl, out


def test_shape_check_accepts_consistent_tensors():
    assert b.check_attention_shapes(*_attention_tensors()) == 3


@pytest.mark.parametrize("vshape", [(8, 2, 16, 128), (10, 1, 16, 128), (10, 2, 16, 64)])
def test_mismatched_v_pool_is_rejected_before_any_launch(vshape):
    with pytest.raises(ValueError, match="v_pool"):
        b.check_attention_shapes(*_attention_tensors(v_pool_shape=vshape))


def test_head_dim_and_out_mismatch_are_rejected():
    q, kp, vp, bt, sl, qsl, out = _attention_tensors()
    import torch
    with pytest.raises(ValueError):
        b.check_attention_shapes(q[:, :, :64].contiguous(), kp, vp, bt, sl, qsl)
    with pytest.raises(ValueError, match="out"):
        b.check_attention_shapes(q, kp, vp, bt, sl, qsl, torch.zeros(3, 12, 128))
    with pytest.raises(ValueError, match="num_reqs"):
        b.check_attention_shapes(q, kp, vp, bt[:2], sl, qsl)
