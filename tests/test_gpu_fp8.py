"""e4m3 KV cache on the GPU against the oracle.

The quantising append must produce the oracle's codes bit for bit (both
round the fp32 quotient x / scale to the nearest e4m3 code, ties to even,
saturating at 448).  Attention over e4m3 pools must match the oracle's fp64
attention over the dequantised pools within the bf16-output tolerance.
Pool codes are seeded inputs (uniform over the non-NaN codes); slots no
request owns hold the NaN code, which must never reach an output.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_195_gb300 as pkv
from paged_kv_cache_195_gb300 import build as pkv_build
from paged_kv_cache_195_gb300 import workloads as wl

from pkv_testutil import assert_close, pool_host, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv_build.build()
    pkv.load_library()
    yield
    assert pkv.pkv_get_device_error() == 0, pkv.pkv_last_error()


def _host(inp):
    return dict(q=wl.bf16_bits(inp.q), k_new=wl.bf16_bits(inp.k_new),
                v_new=wl.bf16_bits(inp.v_new), slots=inp.slot_mapping.cpu().numpy(),
                k_pool=pool_host(inp.k_pool), v_pool=pool_host(inp.v_pool),
                k_scale=inp.k_scale.cpu().numpy(), v_scale=inp.v_scale.cpu().numpy(),
                bt=inp.block_tables.cpu().numpy(), sl=inp.seq_lens.cpu().numpy(),
                qsl=inp.query_start_loc.cpu().numpy(), scale=inp.scale)


def _step(inp, append=True, workspace=None):
    if append:
        pkv.pkv_append_fp8(inp.k_new, inp.v_new, inp.slot_mapping, inp.k_pool, inp.v_pool,
                           inp.k_scale, inp.v_scale)
    return pkv.pkv_attention_fp8kv(inp.q, inp.k_pool, inp.v_pool, inp.k_scale, inp.v_scale,
                                   inp.block_tables, inp.seq_lens, inp.query_start_loc,
                                   inp.scale, workspace=workspace)


def _full_parity(shape, poison=True):
    inp = wl.make_fp8_step(shape, device="cuda", poison=poison)
    h = _host(inp)
    kp, vp = oracle.append_fp8(h["k_new"], h["v_new"], h["slots"], h["k_pool"], h["v_pool"],
                               h["k_scale"], h["v_scale"])
    out = _step(inp)
    torch.cuda.synchronize()
    assert pkv.pkv_get_device_error() == 0, pkv.pkv_last_error()
    assert np.array_equal(pool_host(inp.k_pool), kp), "K codes differ from the oracle's"
    assert np.array_equal(pool_host(inp.v_pool), vp), "V codes differ from the oracle's"
    want = oracle.paged_attention_fp8(h["q"], kp, vp, h["k_scale"], h["v_scale"], h["bt"],
                                      h["sl"], h["qsl"], h["scale"])
    return assert_close(to_f64(out), want, shape.name), inp, out


def test_fp8_append_codes_bit_exact():
    # Values spanning every binade of e4m3 (and beyond 448: saturation),
    # including exact ties, quantised by one scale per head.
    shape = wl.StepShape("fp8_append", [40, 17, 33], [40, 17, 33], 8, 4, seed=81)
    inp = wl.make_fp8_step(shape, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(82)
    mag = torch.exp2(torch.empty(inp.k_new.shape, device="cuda").uniform_(-20, 11, generator=g))
    sign = torch.where(torch.rand(inp.k_new.shape, device="cuda", generator=g) < 0.5, -1.0, 1.0)
    inp.k_new = (mag * sign).to(torch.bfloat16)
    inp.v_new = (-mag * sign).to(torch.bfloat16)
    h = _host(inp)
    kp, vp = oracle.append_fp8(h["k_new"], h["v_new"], h["slots"], h["k_pool"], h["v_pool"],
                               h["k_scale"], h["v_scale"])
    pkv.pkv_append_fp8(inp.k_new, inp.v_new, inp.slot_mapping, inp.k_pool, inp.v_pool,
                       inp.k_scale, inp.v_scale)
    torch.cuda.synchronize()
    assert np.array_equal(pool_host(inp.k_pool), kp)
    assert np.array_equal(pool_host(inp.v_pool), vp)


def test_fp8_append_exact_scale_one():
    # With scale 1 every bf16 value that is an e4m3 value must keep its code,
    # and halfway values must round to the even code.
    shape = wl.StepShape("fp8_scale1", [16], [16], 2, 1, seed=83)
    inp = wl.make_fp8_step(shape, device="cuda")
    vals = torch.tensor([oracle.e4m3_decode(c) for c in range(256) if c not in (0x7F, 0xFF)],
                        dtype=torch.float32)
    grid = vals.repeat(16 * 128 // vals.numel() + 1)[:16 * 128].view(16, 1, 128)
    inp.k_new = grid.to(torch.bfloat16).cuda()
    mids = (grid[..., :-1] + grid[..., 1:]) / 2  # ties where bf16 holds them exactly
    inp.v_new = torch.cat([mids, grid[..., :1]], -1).to(torch.bfloat16).cuda()
    inp.k_scale = torch.ones(1, device="cuda")
    inp.v_scale = torch.ones(1, device="cuda")
    h = _host(inp)
    kp, vp = oracle.append_fp8(h["k_new"], h["v_new"], h["slots"], h["k_pool"], h["v_pool"],
                               h["k_scale"], h["v_scale"])
    pkv.pkv_append_fp8(inp.k_new, inp.v_new, inp.slot_mapping, inp.k_pool, inp.v_pool,
                       inp.k_scale, inp.v_scale)
    torch.cuda.synchronize()
    assert np.array_equal(pool_host(inp.k_pool), kp)
    assert np.array_equal(pool_host(inp.v_pool), vp)


@pytest.mark.parametrize("g", [1, 2, 3, 4, 5, 6, 7, 8])
def test_fp8_every_group_size(g):
    shape = wl.StepShape(f"fp8_g{g}", [1, 31, 300, 129, 2000], [1, 1, 1, 3, 1], 2 * g, 2,
                         seed=90 + g)
    _full_parity(shape)


@pytest.mark.parametrize("g", [4, 6, 8])
def test_fp8_simt_decode_large_groups(g, pkv_opts):
    # groups of 4 or more run on the tensor cores by default (tiles widened
    # to f16); the SIMT decode serves them too when asked
    pkv_opts(decode_tc_fp8=0)
    shape = wl.StepShape(f"fp8_simt_g{g}", [1, 31, 300, 129, 2000], [1, 1, 1, 3, 1], 2 * g, 2,
                         seed=190 + g)
    _full_parity(shape)


def test_fp8_simt_decode_split_and_chunks(pkv_opts):
    pkv_opts(decode_tc_fp8=0)
    _full_parity(wl.StepShape("fp8_simt_long", [20000, 3000, 17], [1, 2, 1], 32, 8, seed=198),
                 poison=False)
    _full_parity(wl.StepShape("fp8_simt_chunks", [700, 64, 230, 5], [64, 64, 200, 1], 32, 8,
                              seed=197))


@pytest.mark.parametrize("seed", range(6))
def test_fp8_random_ragged(seed):
    rng = np.random.default_rng(700 + seed)
    _full_parity(wl.random_small_shape(rng, f"fp8_rand{seed}", max_reqs=6, max_len=300))


def test_fp8_prefill_chunks_in_decode_kernel():
    # q_r of 64 and 200: rows the bf16 path would give to the tensor-core
    # prefill kernel; with e4m3 pools the decode kernel serves them.
    shape = wl.StepShape("fp8_chunks", [700, 64, 230, 5], [64, 64, 200, 1], 32, 8, seed=97)
    _full_parity(shape)


def test_fp8_long_context_split():
    # Long rows cut across many CTAs and merged by log-sum-exp.
    shape = wl.StepShape("fp8_long", [20000, 3000, 17], [1, 2, 1], 32, 8, seed=98)
    _full_parity(shape, poison=False)


def test_fp8_relabelling_bit_identical():
    shape = wl.StepShape("fp8_relabel", [513, 77, 1200], [1, 1, 2], 12, 2, seed=99)
    (_, _), inp, out = _full_parity(shape)
    perm = torch.randperm(shape.num_blocks, generator=torch.Generator().manual_seed(5)).cuda()
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(perm.numel(), device="cuda")
    k2, v2 = inp.k_pool[inv], inp.v_pool[inv]  # block b moves to perm[b]
    bt2 = torch.where(inp.block_tables >= 0, perm[inp.block_tables.clamp(min=0).long()].int(),
                      inp.block_tables)
    out2 = pkv.pkv_attention_fp8kv(inp.q, k2, v2, inp.k_scale, inp.v_scale, bt2, inp.seq_lens,
                                   inp.query_start_loc, inp.scale)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


@pytest.mark.parametrize("factory,layer", [(wl.qwen_decode, 3), (wl.qwen_long_batch, 0)],
                         ids=["qwen_decode", "qwen_long"])
def test_fp8_full_size_every_element(factory, layer):
    shape = factory()
    inp = wl.make_fp8_step(shape, device="cuda", layer=layer)
    h = _host(inp)
    out = _step(inp)
    torch.cuda.synchronize()
    assert pkv.pkv_get_device_error() == 0, pkv.pkv_last_error()
    got = to_f64(out)
    del inp, out
    kp, vp = oracle.append_fp8(h["k_new"], h["v_new"], h["slots"], h["k_pool"], h["v_pool"],
                               h["k_scale"], h["v_scale"])
    want = oracle.paged_attention_fp8(h["q"], kp, vp, h["k_scale"], h["v_scale"], h["bt"],
                                      h["sl"], h["qsl"], h["scale"])
    assert_close(got, want, f"fp8 {shape.name}")


def test_fp8_bad_block_reported():
    shape = wl.StepShape("fp8_bad", [40, 40], [1, 1], 4, 2, seed=101)
    inp = wl.make_fp8_step(shape, device="cuda")
    inp.block_tables[1, 1] = shape.num_blocks + 7
    _step(inp, append=False)
    assert pkv.pkv_get_device_error() == pkv._binding.PKV_ERR_DEVICE_BOUNDS


def test_fp8_null_scales_rejected():
    shape = wl.tiny_decode()
    inp = wl.make_fp8_step(shape, device="cuda")
    import ctypes
    d = pkv.make_dims(tuple(inp.q.shape), tuple(inp.k_pool.shape), shape.num_reqs,
                      inp.block_tables.shape[1])
    rc = pkv.load_library().pkv_attention_fp8kv(
        ctypes.c_void_p(inp.q.data_ptr()), ctypes.c_void_p(inp.k_pool.data_ptr()),
        ctypes.c_void_p(inp.v_pool.data_ptr()), None, None,
        ctypes.c_void_p(inp.block_tables.data_ptr()), ctypes.c_void_p(inp.seq_lens.data_ptr()),
        ctypes.c_void_p(inp.query_start_loc.data_ptr()), ctypes.c_float(inp.scale),
        ctypes.c_void_p(inp.q.data_ptr()), ctypes.byref(d), None, 0, None)
    assert rc == pkv._binding.PKV_ERR_INVALID


# ---------------------------------------------------------------------------
# One layer in one call over e4m3 pools: pkv_append_attention_fp8
# ---------------------------------------------------------------------------

FUSED_MODES = {"early_kv": {}, "early_trigger": {"early_trigger": 1}, "ordered": {"early_kv": 0}}

FUSED_SHAPES = [
    wl.StepShape("fp8_fused_g6", [17, 64, 100, 128, 513, 1000, 33, 16], [1] * 8, 12, 2, seed=411),
    wl.StepShape("fp8_fused_g4", [300, 47, 2049, 160, 161, 5], [1] * 6, 32, 8, seed=412),
    wl.StepShape("fp8_fused_g2", [90, 700, 66, 1025], [1] * 4, 4, 2, seed=413),
    wl.StepShape("fp8_fused_mq", [200, 18, 47, 129], [3, 5, 15, 2], 12, 2, seed=414),
]


def _nan_codes_at_new_slots(inp):
    """The NaN code at the slots this step's append writes (their old contents)."""
    s = inp.slot_mapping[inp.slot_mapping >= 0]
    nb, hkv, bs, d = inp.k_pool.shape
    for pool in (inp.k_pool, inp.v_pool):
        flat = pool.view(nb, hkv, bs, d).permute(0, 2, 1, 3).reshape(nb * bs, hkv, d)
        flat[s] = wl.E4M3_NAN
        pool.copy_(flat.reshape(nb, bs, hkv, d).permute(0, 2, 1, 3))


def _fused_fp8(inp, out=None, workspace=None):
    return pkv.pkv_append_attention_fp8(inp.k_new, inp.v_new, inp.slot_mapping, inp.k_pool,
                                        inp.v_pool, inp.k_scale, inp.v_scale, inp.q,
                                        inp.block_tables, inp.seq_lens, inp.query_start_loc,
                                        inp.scale, out=out, workspace=workspace)


@pytest.mark.parametrize("mode", list(FUSED_MODES))
@pytest.mark.parametrize("shape", FUSED_SHAPES, ids=lambda s: s.name)
def test_fp8_fused_matches_oracle(shape, mode, pkv_opts):
    pkv_opts(**FUSED_MODES[mode])
    inp = wl.make_fp8_step(shape, device="cuda", poison=True)
    h = _host(inp)
    kp, vp = oracle.append_fp8(h["k_new"], h["v_new"], h["slots"], h["k_pool"], h["v_pool"],
                               h["k_scale"], h["v_scale"])
    _nan_codes_at_new_slots(inp)
    out = _fused_fp8(inp)
    torch.cuda.synchronize()
    assert pkv.pkv_get_device_error() == 0, pkv.pkv_last_error()
    assert np.array_equal(pool_host(inp.k_pool), kp), "K codes differ from the oracle's"
    assert np.array_equal(pool_host(inp.v_pool), vp), "V codes differ from the oracle's"
    want = oracle.paged_attention_fp8(h["q"], kp, vp, h["k_scale"], h["v_scale"], h["bt"],
                                      h["sl"], h["qsl"], h["scale"])
    assert_close(to_f64(out), want, shape.name)


@pytest.mark.parametrize("shape", FUSED_SHAPES, ids=lambda s: s.name)
def test_fp8_fused_equals_separate_calls(shape):
    a = wl.make_fp8_step(shape, device="cuda")
    b = wl.make_fp8_step(shape, device="cuda")
    ref = _step(a)
    _nan_codes_at_new_slots(b)
    got = _fused_fp8(b)
    torch.cuda.synchronize()
    assert torch.equal(got, ref)
    assert torch.equal(a.k_pool, b.k_pool) and torch.equal(a.v_pool, b.v_pool)
