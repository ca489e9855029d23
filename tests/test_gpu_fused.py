"""pkv_append_attention (append, then attention, as one call) on the GPU.

The attention kernel streams every K/V tile without one of the step's new
tokens before the append has finished and waits only for the tiles that hold
them.  The tests put NaN in the new tokens' slots before the call, so a tile
read before the append completes shows up as a non-finite output, and compare
with the oracle and with the two separate calls (the same kernels and
arithmetic: bit-identical outputs).
"""
import pytest
import torch

import paged_kv_cache_195_gb300 as pkv
from paged_kv_cache_195_gb300 import build as pkv_build
from paged_kv_cache_195_gb300 import workloads as wl

from pkv_testutil import (assert_close, host_copy, oracle_full, oracle_pools_after_append, to_f64)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv_build.build()
    pkv.load_library()
    yield
    assert pkv.pkv_get_device_error() == 0, pkv.pkv_last_error()


def _nan_new_slots(inp):
    """NaN at the slots this step's append writes (their old contents)."""
    s = inp.slot_mapping[inp.slot_mapping >= 0]
    nb, hkv, bs, d = inp.k_pool.shape
    for pool in (inp.k_pool, inp.v_pool):
        flat = pool.view(nb, hkv, bs, d).permute(0, 2, 1, 3).reshape(nb * bs, hkv, d)
        flat[s] = float("nan")
        pool.copy_(flat.reshape(nb, bs, hkv, d).permute(0, 2, 1, 3))


def _fused(inp, out=None, workspace=None):
    return pkv.pkv_append_attention(inp.k_new, inp.v_new, inp.slot_mapping, inp.k_pool,
                                    inp.v_pool, inp.q, inp.block_tables, inp.seq_lens,
                                    inp.query_start_loc, inp.scale, out=out,
                                    workspace=workspace)


SHAPES = [
    # tensor-core decode (g = 6, 4, 8), ragged lengths, some a block boundary
    wl.StepShape("fused_g6", [17, 64, 100, 128, 513, 1000, 33, 16], [1] * 8, 12, 2, seed=401),
    wl.StepShape("fused_g4", [300, 47, 2049, 160, 161, 5], [1] * 6, 32, 8, seed=402),
    wl.StepShape("fused_g8", [700, 1, 222], [1, 1, 1], 16, 2, seed=403),
    # SIMT decode (g = 2, 1)
    wl.StepShape("fused_g2", [90, 700, 66, 1025], [1] * 4, 4, 2, seed=404),
    wl.StepShape("fused_g1", [31, 250, 4000], [1] * 3, 4, 4, seed=405),
    # multi-query decode rows whose new tokens span two blocks
    wl.StepShape("fused_mq", [200, 18, 47, 129], [3, 5, 15, 2], 12, 2, seed=406),
    # prefill chunks next to decode rows (tensor-core prefill after the decode)
    wl.StepShape("fused_mixed", [600, 80, 333, 1200], [1, 64, 1, 200], 32, 8, seed=407),
]


# launch modes of the fused call: tiles without new tokens read before the
# append finishes (default); also launched as soon as the append starts; and
# the plain order (the attention waits for the whole append)
MODES = {"early_kv": {}, "early_trigger": {"early_trigger": 1}, "ordered": {"early_kv": 0}}


@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
def test_fused_matches_oracle(shape, mode, pkv_opts):
    pkv_opts(**MODES[mode])
    inp = wl.make_step(shape, device="cuda", poison=True)
    h = host_copy(inp)
    kp, vp = oracle_pools_after_append(h)
    _nan_new_slots(inp)
    out = _fused(inp)
    torch.cuda.synchronize()
    assert pkv.pkv_get_device_error() == 0, pkv.pkv_last_error()
    assert_close(to_f64(out), oracle_full(h, kp, vp), shape.name)


@pytest.mark.parametrize("shape", SHAPES[:2] + SHAPES[3:4] + SHAPES[5:], ids=lambda s: s.name)
def test_fused_equals_separate_calls(shape):
    a = wl.make_step(shape, device="cuda")
    b = wl.make_step(shape, device="cuda")
    pkv.pkv_append(a.k_new, a.v_new, a.slot_mapping, a.k_pool, a.v_pool)
    ref = pkv.pkv_attention(a.q, a.k_pool, a.v_pool, a.block_tables, a.seq_lens,
                            a.query_start_loc, a.scale)
    _nan_new_slots(b)
    got = _fused(b)
    torch.cuda.synchronize()
    assert torch.equal(got, ref)
    assert torch.equal(a.k_pool, b.k_pool) and torch.equal(a.v_pool, b.v_pool)


@pytest.mark.parametrize("mode", list(MODES))
def test_fused_layers_in_a_graph(mode, pkv_opts):
    pkv_opts(**MODES[mode])
    # consecutive layers, each its own pools, captured and replayed: every
    # layer's attention follows its own append
    shape = wl.StepShape("fused_graph", [512] * 24 + [1000] * 8, [1] * 32, 12, 2, seed=408)
    layers = [wl.make_step(shape, device="cuda", layer=i) for i in range(6)]
    hosts = [host_copy(x) for x in layers]
    d = pkv.make_dims(tuple(layers[0].q.shape), tuple(layers[0].k_pool.shape), shape.num_reqs,
                      shape.max_blocks_per_req)
    ws = pkv.Workspace(d)
    pkv.pkv_workspace_init(ws, d)
    outs = [torch.empty_like(x.q) for x in layers]
    for x in layers:
        _nan_new_slots(x)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for x, o in zip(layers, outs):
            _fused(x, out=o, workspace=ws)
    g.replay()
    torch.cuda.synchronize()
    assert pkv.pkv_get_device_error() == 0, pkv.pkv_last_error()
    for x, h, o in zip(layers, hosts, outs):
        kp, vp = oracle_pools_after_append(h)
        assert_close(to_f64(o), oracle_full(h, kp, vp), "fused_graph")


def test_fused_qwen_decode_full_size_every_element():
    shape = wl.qwen_decode(layers=1)
    inp = wl.make_step(shape, device="cuda")
    h = host_copy(inp)
    _nan_new_slots(inp)
    out = _fused(inp)
    torch.cuda.synchronize()
    assert pkv.pkv_get_device_error() == 0, pkv.pkv_last_error()
    kp, vp = oracle_pools_after_append(h)
    assert_close(to_f64(out), oracle_full(h, kp, vp), "qwen_decode fused")


def test_fused_padding_tokens_skip_append():
    # a padding token (slot -1) writes nothing; its row's output is whatever
    # the pool held at that position, the same as with the separate calls
    shape = wl.StepShape("fused_pad", [40, 70], [1, 1], 12, 2, seed=409)
    a = wl.make_step(shape, device="cuda")
    b = wl.make_step(shape, device="cuda")
    for x in (a, b):
        x.slot_mapping[1] = -1
    pkv.pkv_append(a.k_new, a.v_new, a.slot_mapping, a.k_pool, a.v_pool)
    ref = pkv.pkv_attention(a.q, a.k_pool, a.v_pool, a.block_tables, a.seq_lens,
                            a.query_start_loc, a.scale)
    got = _fused(b)
    torch.cuda.synchronize()
    assert torch.equal(got, ref)


def _bucket_step(live, pad_rows):
    """A step of `live` plus `pad_rows` trailing token rows past
    query_start_loc[R] (a padded bucket), with the padding tokens' slots
    pointing at free pool slots (not read by any request)."""
    inp = wl.make_step(live, device="cuda", poison=True)
    T = live.num_q_tokens + pad_rows
    nb = inp.k_pool.shape[0]
    used = set(inp.block_tables[inp.block_tables >= 0].tolist())
    free = [b for b in range(nb) if b not in used][:pad_rows]
    assert len(free) == pad_rows

    def grow(x, fill):
        y = torch.full((T,) + tuple(x.shape[1:]), fill, dtype=x.dtype, device=x.device)
        y[:x.shape[0]] = x
        return y

    g = torch.Generator(device="cpu").manual_seed(77)
    inp.q = grow(inp.q, float("nan"))
    inp.k_new = grow(inp.k_new, 0.0)
    inp.v_new = grow(inp.v_new, 0.0)
    inp.k_new[live.num_q_tokens:] = torch.randn(inp.k_new[live.num_q_tokens:].shape,
                                                generator=g).to(inp.k_new)
    inp.v_new[live.num_q_tokens:] = torch.randn(inp.v_new[live.num_q_tokens:].shape,
                                                generator=g).to(inp.v_new)
    inp.slot_mapping = grow(inp.slot_mapping, -1)
    inp.slot_mapping[live.num_q_tokens:] = torch.tensor([b * 16 + 3 for b in free],
                                                        dtype=torch.int64)
    return inp


@pytest.mark.parametrize("mode", list(MODES))
def test_fused_writes_trailing_tokens(mode, pkv_opts):
    # token rows past query_start_loc[R] with a slot: appended like the others
    # (their attention rows are padding: never written)
    pkv_opts(**MODES[mode])
    live = wl.StepShape("fused_trailing", [300, 47, 129, 16], [1] * 4, 12, 2, seed=410)
    a, b = _bucket_step(live, 5), _bucket_step(live, 5)
    pkv.pkv_append(a.k_new, a.v_new, a.slot_mapping, a.k_pool, a.v_pool)
    ref = torch.full_like(a.q, 7.0)
    pkv.pkv_attention(a.q, a.k_pool, a.v_pool, a.block_tables, a.seq_lens, a.query_start_loc,
                      a.scale, out=ref)
    got = torch.full_like(b.q, 7.0)
    pkv.pkv_append_attention(b.k_new, b.v_new, b.slot_mapping, b.k_pool, b.v_pool, b.q,
                             b.block_tables, b.seq_lens, b.query_start_loc, b.scale, out=got)
    torch.cuda.synchronize()
    assert pkv.pkv_get_device_error() == 0, pkv.pkv_last_error()
    # bit patterns: the free slots hold NaN
    assert torch.equal(a.k_pool.view(torch.int16), b.k_pool.view(torch.int16))
    assert torch.equal(a.v_pool.view(torch.int16), b.v_pool.view(torch.int16))
    assert torch.equal(got, ref)
    assert bool((got[live.num_q_tokens:].float() == 7.0).all())

