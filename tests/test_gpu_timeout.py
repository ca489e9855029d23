"""Bounded device waits: a wait that can never complete gives up, reports
PKV_ERR_TIMEOUT, and leaves the device usable.

Every mbarrier wait in the kernels gives up after pkv_options.wait_limit_us,
records the timeout in the device error word and sets the CTA's abort flag,
after which every other wait of the CTA returns at once; the CTA then drains
its copies and MMAs in flight, frees its TMEM and exits.  The test makes one
wait impossible on purpose -- the testing option debug_withhold_q keeps the
tensor-core decode from ever loading the first piece's q -- with a 1 ms limit,
then checks that the call comes back, that the error is reported, that no
output row was written, and that the next ordinary call (on a re-initialised
workspace) matches the oracle.  Nothing here faults or traps the GPU: the
kernel itself stops waiting and returns.
"""
import time

import pytest
import torch

import oracle
import paged_kv_cache_195_gb300 as pkv
from paged_kv_cache_195_gb300 import build as pkv_build
from paged_kv_cache_195_gb300 import workloads as wl

from pkv_testutil import assert_close, host_copy, oracle_full, oracle_pools_after_append, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv_build.build()
    pkv.load_library()
    yield
    assert pkv.pkv_get_device_error() == 0, pkv.pkv_last_error()


def _dims(inp, shape):
    return pkv.make_dims(tuple(inp.q.shape), tuple(inp.k_pool.shape), shape.num_reqs,
                         shape.max_blocks_per_req)


def test_withheld_q_times_out_and_the_next_call_is_correct(pkv_opts):
    # g = 4 query heads per KV head: the tensor-core decode serves every row
    shape = wl.StepShape("timeout_bf16", [300, 40, 129, 700, 2048], [1, 1, 1, 1, 1], 8, 2,
                         seed=901)
    inp = wl.make_step(shape, device="cuda")
    h = host_copy(inp)
    kp, vp = oracle_pools_after_append(h)
    pkv.pkv_append(inp.k_new, inp.v_new, inp.slot_mapping, inp.k_pool, inp.v_pool)
    d = _dims(inp, shape)
    ws = pkv.Workspace(d)
    pkv.pkv_workspace_init(ws, d)
    torch.cuda.synchronize()
    assert pkv.pkv_get_device_error() == 0

    # the withheld q is a feature of the tensor-core decode
    pkv_opts(wait_limit_us=1000, debug_withhold_q=1, decode_tc=1)
    out = torch.full_like(inp.q, float("nan"))
    t0 = time.perf_counter()
    pkv.pkv_attention(inp.q, inp.k_pool, inp.v_pool, inp.block_tables, inp.seq_lens,
                      inp.query_start_loc, inp.scale, out=out, workspace=ws)
    rc = pkv.pkv_get_device_error()  # synchronises the stream
    elapsed = time.perf_counter() - t0
    assert rc == pkv._binding.PKV_ERR_TIMEOUT, (rc, pkv.pkv_last_error())
    assert elapsed < 10.0
    assert torch.isnan(out.float()).all(), "an aborted call wrote output"

    pkv_opts(wait_limit_us=2_000_000, debug_withhold_q=0)
    pkv.pkv_workspace_init(ws, d)
    for _ in range(2):  # TMEM and the aborted CTAs' state are gone: calls run normally
        got = pkv.pkv_attention(inp.q, inp.k_pool, inp.v_pool, inp.block_tables, inp.seq_lens,
                                inp.query_start_loc, inp.scale, workspace=ws)
        torch.cuda.synchronize()
        assert pkv.pkv_get_device_error() == 0, pkv.pkv_last_error()
        assert_close(to_f64(got), oracle_full(h, kp, vp), "after a timeout")


def test_withheld_q_times_out_on_e4m3_pools(pkv_opts):
    shape = wl.StepShape("timeout_fp8", [300, 40, 129, 700, 2048], [1, 1, 1, 1, 1], 8, 2,
                         seed=902)
    inp = wl.make_fp8_step(shape, device="cuda")
    q, bt, sl, qsl = (wl.bf16_bits(inp.q), inp.block_tables.cpu().numpy(),
                      inp.seq_lens.cpu().numpy(), inp.query_start_loc.cpu().numpy())
    ks, vs = inp.k_scale.cpu().numpy(), inp.v_scale.cpu().numpy()
    d = _dims(inp, shape)
    ws = pkv.Workspace(d)
    pkv.pkv_workspace_init(ws, d)

    pkv_opts(wait_limit_us=1000, debug_withhold_q=1, decode_tc=1, decode_tc_fp8=1)
    out = torch.full_like(inp.q, float("nan"))
    pkv.pkv_attention_fp8kv(inp.q, inp.k_pool, inp.v_pool, inp.k_scale, inp.v_scale,
                            inp.block_tables, inp.seq_lens, inp.query_start_loc, inp.scale,
                            out=out, workspace=ws)
    rc = pkv.pkv_get_device_error()
    assert rc == pkv._binding.PKV_ERR_TIMEOUT, (rc, pkv.pkv_last_error())
    assert torch.isnan(out.float()).all(), "an aborted call wrote output"

    pkv_opts(wait_limit_us=2_000_000, debug_withhold_q=0)
    pkv.pkv_workspace_init(ws, d)
    got = pkv.pkv_attention_fp8kv(inp.q, inp.k_pool, inp.v_pool, inp.k_scale, inp.v_scale,
                                  inp.block_tables, inp.seq_lens, inp.query_start_loc,
                                  inp.scale, workspace=ws)
    torch.cuda.synchronize()
    assert pkv.pkv_get_device_error() == 0, pkv.pkv_last_error()
    want = oracle.paged_attention_fp8(q, inp.k_pool.cpu().numpy(), inp.v_pool.cpu().numpy(), ks,
                                      vs, bt, sl, qsl, inp.scale)
    assert_close(to_f64(got), want, "e4m3 after a timeout")
