"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Small cases are compared element by element on every output; the full-size
workloads (in the launch configuration the benchmark times) on sampled rows
the oracle computes one by one, plus properties that hold at any size.
"""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_195_gb300 as pkv
from paged_kv_cache_195_gb300 import build as pkv_build
from paged_kv_cache_195_gb300 import workloads as wl

from pkv_testutil import (assert_close, gpu_step, host_copy, oracle_full,
                          oracle_pools_after_append, snapshot_oracle, snapshot_rows, to_f64)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv_build.build()
    pkv.load_library()
    yield
    assert pkv.pkv_get_device_error() == 0, pkv.pkv_last_error()


def _full_parity(shape, poison=False, append=True):
    inp = wl.make_step(shape, device="cuda", poison=poison)
    h = host_copy(inp)
    kp, vp = oracle_pools_after_append(h) if append else (h["k_pool"], h["v_pool"])
    out = gpu_step(inp, append=append)
    torch.cuda.synchronize()
    if append:
        assert np.array_equal(wl.bf16_bits(inp.k_pool), kp)
        assert np.array_equal(wl.bf16_bits(inp.v_pool), vp)
    want = oracle_full(h, kp, vp)
    return assert_close(to_f64(out), want, shape.name), inp, out


# ---------------------------------------------------------------------------
# KV append: bit-exact
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("factory", [wl.tiny_decode, lambda: wl.qwen_decode(layers=1),
                                     lambda: wl.llama_mixed(num_decode=40, num_prefill=3)])
def test_append_bit_exact(factory):
    inp = wl.make_step(factory(), device="cuda")
    h = host_copy(inp)
    slots = inp.slot_mapping.clone()
    slots[::7] = -1                                   # padding tokens are skipped
    h["slot_mapping"] = slots.cpu().numpy()
    kp, vp = oracle_pools_after_append(h)
    pkv.pkv_append(inp.k_new, inp.v_new, slots, inp.k_pool, inp.v_pool)
    torch.cuda.synchronize()
    assert np.array_equal(wl.bf16_bits(inp.k_pool), kp)
    assert np.array_equal(wl.bf16_bits(inp.v_pool), vp)


def test_append_out_of_range_slot_is_reported_not_written():
    inp = wl.make_step(wl.tiny_decode(), device="cuda")
    before = wl.bf16_bits(inp.k_pool).copy()
    bad = torch.full_like(inp.slot_mapping, 64 * 16 + 5)
    pkv.pkv_append(inp.k_new, inp.v_new, bad, inp.k_pool, inp.v_pool)
    assert pkv.pkv_get_device_error() == pkv._binding.PKV_ERR_DEVICE_BOUNDS
    assert np.array_equal(wl.bf16_bits(inp.k_pool), before)
    assert pkv.pkv_get_device_error() == 0        # the read cleared it


# ---------------------------------------------------------------------------
# Attention: every element on small cases
# ---------------------------------------------------------------------------

def test_tiny_decode_step():
    _full_parity(wl.tiny_decode())


def test_tiny_decode_step_poisoned_free_slots():
    (mx, mean), inp, out = _full_parity(wl.tiny_decode(), poison=True)
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("seed", range(12))
def test_random_ragged_steps(seed):
    rng = np.random.default_rng(500 + seed)
    Hkv = int(rng.choice([1, 2, 4, 8]))
    g = int(rng.integers(1, 9))
    shape = wl.random_small_shape(rng, max_reqs=9, max_len=300, Hq=Hkv * g, Hkv=Hkv,
                                  max_q=int(rng.choice([1, 4, 40])))
    _full_parity(shape, poison=bool(seed % 2))


@pytest.mark.parametrize("g", [6, 2])
@pytest.mark.parametrize("cost", [0, 8, 64, 1024])
def test_rowgroup_cost_does_not_change_the_answer(cost, g, pkv_opts):
    """The plan cuts the CTAs' ranges over weighted row-group lengths (blocks
    plus rowgroup_cost); ranges that meet only a row-group's weight hold no
    piece of it.  Every weight gives the oracle's answer, on the tensor-core
    (g = 6) and SIMT (g = 2) decodes, with short, long and multi-query rows."""
    pkv_opts(rowgroup_cost=cost)
    rng = np.random.default_rng(600 + g)
    lens = rng.integers(1, 900, size=40)
    ql = np.where(rng.random(40) < 0.2, rng.integers(2, 12, size=40), 1)
    lens = np.maximum(lens, ql)
    shape = wl.StepShape(f"cost{cost}_g{g}", lens, ql, 2 * g, 2, seed=610 + g)
    _full_parity(shape, poison=True)


@pytest.mark.parametrize("g", [1, 2, 3, 4, 5, 6, 7, 8])
def test_every_group_size(g):
    shape = wl.StepShape(f"g{g}", [1, 15, 16, 17, 200, 777], [1, 1, 2, 17, 1, 5], 2 * g, 2,
                         seed=90 + g)
    _full_parity(shape, poison=True)


def test_edge_lengths():
    """L = 1, exact block multiples, a fresh prefill (q = L), q_r = 0 rows."""
    shape = wl.StepShape("edges", [1, 16, 32, 48, 33, 20, 5], [1, 1, 16, 0, 33, 0, 1], 12, 2,
                         seed=77)
    _full_parity(shape, poison=True)


def test_empty_step():
    shape = wl.StepShape("empty", [5, 9], [0, 0], 4, 2, seed=1)
    inp = wl.make_step(shape, device="cuda")
    out = gpu_step(inp, append=False)
    assert out.shape == (0, 4, 128)


def test_block_relabelling_is_bit_identical():
    shape = wl.random_small_shape(np.random.default_rng(8), max_reqs=6, max_len=400, Hq=12, Hkv=2)
    inp = wl.make_step(shape, device="cuda")
    out1 = gpu_step(inp, append=False).clone()
    perm = torch.randperm(shape.num_blocks, generator=torch.Generator().manual_seed(3)).cuda()
    kp2 = torch.empty_like(inp.k_pool)
    vp2 = torch.empty_like(inp.v_pool)
    kp2[perm] = inp.k_pool
    vp2[perm] = inp.v_pool
    bt2 = torch.where(inp.block_tables >= 0, perm[inp.block_tables.clamp(min=0).long()].int(),
                      inp.block_tables)
    out2 = pkv.pkv_attention(inp.q, kp2, vp2, bt2.contiguous(), inp.seq_lens,
                             inp.query_start_loc, inp.scale)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))


def test_split_count_does_not_change_the_answer(pkv_opts):
    """Online-softmax merging is exact: any split count gives the same result
    up to fp32 rounding (at most one bf16 ulp of the output).  This holds for
    the SIMT decode, whose probabilities stay in fp32."""
    pkv_opts(decode_tc=0)
    shape = wl.StepShape("splits", [3000, 1200, 17], [1, 3, 1], 32, 8, seed=5)
    inp = wl.make_step(shape, device="cuda")
    outs = []
    for chunk in (1, 3, 4096):
        pkv_opts(min_chunk=chunk)
        outs.append(gpu_step(inp, append=False).float().clone())
    ref = oracle_full(host_copy(inp))
    for o in outs:
        assert_close(to_f64(o.bfloat16()), ref, "split")
        ulp = torch.finfo(torch.bfloat16).eps * outs[-1].abs().clamp(min=2.0**-8)
        assert ((o - outs[-1]).abs() <= ulp + 1e-6).all()


def test_split_count_tensor_core_decode(pkv_opts):
    """The tensor-core decode feeds P to the MMA in bf16 (relative error at
    most 2^-9 per weight), and where a piece starts decides which 128-key
    tiles form; the merge itself is exact.  A softmax-weighted mean with every
    weight perturbed by at most 2^-9 moves by at most 2 * 2^-9 * max_j |v_j - o|,
    so two splits differ by at most twice that plus the output rounding."""
    pkv_opts(decode_tc=1)
    shape = wl.StepShape("splits_tc", [3000, 1200, 17], [1, 3, 1], 32, 8, seed=5)
    inp = wl.make_step(shape, device="cuda")
    outs = []
    for chunk in (1, 3, 4096):
        pkv_opts(min_chunk=chunk)
        outs.append(gpu_step(inp, append=False).float().clone())
    h = host_copy(inp)
    ref = oracle_full(h)
    vmax = float(inp.v_pool.float().abs().max())
    bound = 4 * 2.0 ** -9 * 2 * vmax
    for o in outs:
        assert_close(to_f64(o.bfloat16()), ref, "split")
        ulp = torch.finfo(torch.bfloat16).eps * outs[-1].abs().clamp(min=2.0**-8)
        assert ((o - outs[-1]).abs() <= 2 * ulp + bound).all()


def test_two_chunks_equal_one_chunk():
    """A prefill chunk in one call equals two calls with the cache appended in
    between (chunk k attends to what chunks 0..k-1 wrote)."""
    prefix, q1, q2 = 37, 20, 45
    one = wl.StepShape("c", [prefix + q1 + q2], [q1 + q2], 16, 4, seed=21)
    inp = wl.make_step(one, device="cuda")
    h = host_copy(inp)
    kp, vp = oracle_pools_after_append(h)
    full = gpu_step(inp).clone()
    outs = []
    for lo, hi, L in ((0, q1, prefix + q1), (q1, q1 + q2, prefix + q1 + q2)):
        o = pkv.pkv_attention(inp.q[lo:hi].contiguous(), inp.k_pool, inp.v_pool,
                              inp.block_tables, torch.tensor([L], dtype=torch.int32, device="cuda"),
                              torch.tensor([0, hi - lo], dtype=torch.int32, device="cuda"),
                              inp.scale)
        outs.append(o)
    two = torch.cat(outs)
    want = oracle_full(h, kp, vp)
    assert_close(to_f64(two), want, "two chunks")
    assert_close(to_f64(full), want, "one chunk")


def test_constant_v_returns_the_constant():
    shape = wl.random_small_shape(np.random.default_rng(31), max_reqs=5, max_len=500, Hq=32, Hkv=8)
    inp = wl.make_step(shape, device="cuda")
    inp.v_pool.fill_(0.71875)                              # exact in bf16
    inp.v_new.fill_(0.71875)
    out = gpu_step(inp)
    assert torch.equal(out, torch.full_like(out, 0.71875))


def test_explicit_workspace_reused_across_calls():
    shape = wl.StepShape("ws", [2000, 700, 64], [1, 1, 1], 12, 2, seed=4)
    inp = wl.make_step(shape, device="cuda")
    dims = pkv.make_dims(tuple(inp.q.shape), tuple(inp.k_pool.shape), shape.num_reqs,
                         shape.max_blocks_per_req)
    ws = pkv.Workspace(dims)
    pkv.pkv_workspace_init(ws, dims)
    h = host_copy(inp)
    kp, vp = oracle_pools_after_append(h)
    a = gpu_step(inp, workspace=ws).clone()
    b = gpu_step(inp, append=False, workspace=ws).clone()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert_close(to_f64(a), oracle_full(h, kp, vp), "workspace")


def test_bad_block_id_is_reported():
    shape = wl.StepShape("bad", [40, 40], [1, 1], 4, 2, seed=2)
    inp = wl.make_step(shape, device="cuda")
    inp.block_tables[1, 1] = shape.num_blocks + 3
    gpu_step(inp, append=False)
    assert pkv.pkv_get_device_error() == pkv._binding.PKV_ERR_DEVICE_BOUNDS


def test_inconsistent_lengths_are_reported():
    shape = wl.StepShape("badlen", [40, 40], [1, 1], 4, 2, seed=2)
    inp = wl.make_step(shape, device="cuda")
    inp.seq_lens[0] = 10_000                       # beyond the block table
    gpu_step(inp, append=False)
    assert pkv.pkv_get_device_error() == pkv._binding.PKV_ERR_DEVICE_BOUNDS


# ---------------------------------------------------------------------------
# Full-size workloads: every output element against the oracle (plus
# determinism); the two stress shapes beyond them compare sampled rows
# ---------------------------------------------------------------------------

def _sample_rows(shape, n_rows, seed):
    rng = np.random.default_rng(seed)
    rows = []
    for r in rng.choice(shape.num_reqs, size=min(n_rows, shape.num_reqs), replace=False):
        qr = int(shape.q_lens[r])
        if qr:
            rows.append((int(r), int(rng.integers(0, qr))))
    # always include the longest request's last query row
    rl = int(np.argmax(shape.seq_lens))
    rows.append((rl, int(shape.q_lens[rl]) - 1))
    return rows


def _sampled(shape, n_rows, seed, layer=0, extra_rows=()):
    inp = wl.make_step(shape, device="cuda", layer=layer)
    rows = _sample_rows(shape, n_rows, seed) + list(extra_rows)
    snap = snapshot_rows(inp, rows)
    out = gpu_step(inp)
    again = gpu_step(inp, append=False)
    assert torch.equal(out.view(torch.int16), again.view(torch.int16)), "non-deterministic"
    assert torch.isfinite(out.float()).all()
    want = snapshot_oracle(snap)
    got = to_f64(out[torch.tensor(snap["qrows"], device="cuda")])
    return assert_close(got, want, shape.name)


def _full_size(shape, layer=0):
    """The whole step at full size: append + attention on the GPU, the
    oracle's own append + attention on host copies taken before, compared on
    every element (max and mean over the whole output); a second attention
    call must give the same bits."""
    inp = wl.make_step(shape, device="cuda", layer=layer)
    h = host_copy(inp)
    out = gpu_step(inp)
    again = gpu_step(inp, append=False)
    torch.cuda.synchronize()
    assert pkv.pkv_get_device_error() == 0, pkv.pkv_last_error()
    assert torch.equal(out.view(torch.int16), again.view(torch.int16)), "non-deterministic"
    got = to_f64(out)
    del inp, out, again
    kp, vp = oracle_pools_after_append(h)
    return assert_close(got, oracle_full(h, kp, vp), f"{shape.name} layer {layer}")


@pytest.mark.parametrize("layer", [0, 27])
def test_qwen_decode_full_size_layers(layer):
    _full_size(wl.qwen_decode(), layer=layer)


def test_qwen_long_batch_full_size():
    _full_size(wl.qwen_long_batch())


def test_llama_mixed_full_size():
    _full_size(wl.llama_mixed())


def test_llama_long_context_full_size():
    _full_size(wl.llama_long_context())


def test_maximum_request_count():
    R = 4096
    rng = np.random.default_rng(14)
    shape = wl.StepShape("r4096", rng.integers(1, 200, size=R), np.ones(R, np.int32), 8, 2, seed=14)
    _sampled(shape, 30, 15)


def test_very_long_context():
    shape = wl.StepShape("L131072", [131072, 5], [1, 1], 8, 1, seed=16)
    _sampled(shape, 2, 17)


# ---------------------------------------------------------------------------
# Path routing: requests with q_r >= PKV_PREFILL_MIN_Q (default 16) run on the
# tcgen05 prefill kernel, the rest on the decode kernel; both must agree with
# the oracle whichever way a request is routed.
# ---------------------------------------------------------------------------

def _prefill_shape(g, seed, Hkv=2):
    rng = np.random.default_rng(seed)
    R = int(rng.integers(1, 5))
    q = rng.integers(16, 300, size=R)
    prefix = rng.integers(0, 400, size=R)
    q[0] = 16 + int(rng.integers(0, 3))         # a short chunk
    prefix[-1] = 0                               # a fresh prompt
    seq = (q + prefix).astype(np.int32)
    return wl.StepShape(f"prefill_g{g}_{seed}", seq, q.astype(np.int32), g * Hkv, Hkv, seed=seed)


@pytest.mark.parametrize("g", [1, 2, 3, 4, 5, 6, 7, 8])
def test_prefill_tensor_core_path(g, pkv_opts):
    pkv_opts(prefill_min_q=16)
    _full_parity(_prefill_shape(g, 700 + g), poison=True)


@pytest.mark.parametrize("route", ["decode_only", "prefill_from_2"])
def test_both_routes_agree_with_oracle(route, pkv_opts):
    pkv_opts(prefill_min_q=0 if route == "decode_only" else 2)
    shape = wl.StepShape("mix", [300, 40, 517, 129, 16], [1, 40, 200, 3, 16], 32, 8, seed=41)
    _full_parity(shape, poison=True)


@pytest.mark.parametrize("g", [4, 2])
def test_prefill_chunks_across_request_batches(g, pkv_opts):
    """Prefill chunks in three batches of 32 requests, mixed with decodes and
    empty rows: the work queue numbers items batch by batch, longest request
    first within a batch, and every item must still land once."""
    pkv_opts(prefill_min_q=16)
    rng = np.random.default_rng(900 + g)
    R = 80
    q = rng.integers(16, 70, size=R)
    q[rng.random(R) < 0.3] = 1                    # decode rows between the chunks
    q[5] = 0                                      # a row with nothing this step
    prefix = rng.integers(0, 350, size=R)
    seq = np.maximum(q + prefix, 1).astype(np.int32)
    shape = wl.StepShape(f"prefill_batches_g{g}", seq, q.astype(np.int32), g * 2, 2, seed=901 + g)
    _full_parity(shape, poison=True)


def test_prefill_long_prefix_many_key_tiles(pkv_opts):
    pkv_opts(prefill_min_q=16)
    shape = wl.StepShape("longprefix", [4096 + 512, 1000 + 64], [512, 64], 32, 8, seed=42)
    rows = [(0, i) for i in (0, 1, 31, 32, 255, 511)] + [(1, i) for i in (0, 63)]
    inp = wl.make_step(shape, device="cuda", poison=True)
    snap = snapshot_rows(inp, rows)
    out = gpu_step(inp)
    want = snapshot_oracle(snap)
    assert_close(to_f64(out[torch.tensor(snap["qrows"], device="cuda")]), want, "long prefix")


def test_captured_graph_follows_new_lengths():
    """One captured step serves later steps whose lengths differ: the plan is
    made on the device from seq_lens / query_start_loc (The Serving Playbook,
    "CUDA graphs and the CPU you forgot about": step buffers are fixed, their
    contents change)."""
    R, max_blocks, Hq, Hkv = 16, 40, 12, 2
    shape_a = wl.StepShape("ga", np.full(R, 300), np.ones(R), Hq, Hkv, num_blocks=R * max_blocks,
                           seed=51)
    inp = wl.make_step(shape_a, device="cuda")
    bt = torch.full((R, max_blocks), -1, dtype=torch.int32, device="cuda")
    perm = torch.randperm(R * max_blocks, generator=torch.Generator().manual_seed(9)).int().cuda()
    bt[:] = perm.view(R, max_blocks)
    seq = torch.full((R,), 300, dtype=torch.int32, device="cuda")
    qsl = torch.arange(R + 1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(inp.q)
    dims = pkv.make_dims(tuple(inp.q.shape), tuple(inp.k_pool.shape), R, max_blocks)
    ws = pkv.Workspace(dims)
    pkv.pkv_workspace_init(ws, dims)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        pkv.pkv_attention(inp.q, inp.k_pool, inp.v_pool, bt, seq, qsl, inp.scale, out=out, workspace=ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pkv.pkv_attention(inp.q, inp.k_pool, inp.v_pool, bt, seq, qsl, inp.scale, out=out, workspace=ws)
    rng = np.random.default_rng(52)
    h = host_copy(inp)
    for trial in range(3):
        lens = rng.integers(1, max_blocks * 16 + 1, size=R).astype(np.int32)
        seq.copy_(torch.from_numpy(lens))
        g.replay()
        torch.cuda.synchronize()
        want = oracle.paged_attention(h["q"], h["k_pool"], h["v_pool"], bt.cpu().numpy(), lens,
                                      np.arange(R + 1, dtype=np.int32), inp.scale)
        assert_close(to_f64(out), want, f"graph replay {trial}")


# ---------------------------------------------------------------------------
# Block copies: copy-on-write and swap to / from pinned host memory
# ---------------------------------------------------------------------------

def test_copy_blocks_copy_on_write_bit_exact():
    shape = wl.StepShape("cow", [200, 90], [1, 1], 32, 8, num_blocks=40, seed=33)
    inp = wl.make_step(shape, device="cuda")
    kp0, vp0 = wl.bf16_bits(inp.k_pool), wl.bf16_bits(inp.v_pool)
    pairs = torch.tensor([[3, 30], [17, 31], [0, 39]], dtype=torch.int64, device="cuda")
    pkv.pkv_copy_blocks(inp.k_pool, inp.v_pool, inp.k_pool, inp.v_pool, pairs)
    torch.cuda.synchronize()
    ek, ev = oracle.copy_blocks(kp0, vp0, kp0, vp0, pairs.cpu().numpy())
    assert np.array_equal(wl.bf16_bits(inp.k_pool), ek)
    assert np.array_equal(wl.bf16_bits(inp.v_pool), ev)


def test_swap_out_and_back_through_pinned_host_memory():
    shape = wl.StepShape("swap", [500, 33], [1, 1], 12, 2, num_blocks=60, seed=34)
    inp = wl.make_step(shape, device="cuda")
    host_k = torch.zeros((8,) + tuple(inp.k_pool.shape[1:]), dtype=torch.bfloat16).pin_memory()
    host_v = torch.zeros_like(host_k).pin_memory()
    out_pairs = torch.tensor([[i * 5, i] for i in range(8)], dtype=torch.int64, device="cuda")
    kp0, vp0 = wl.bf16_bits(inp.k_pool), wl.bf16_bits(inp.v_pool)
    pkv.pkv_copy_blocks(inp.k_pool, inp.v_pool, host_k, host_v, out_pairs)   # swap out
    torch.cuda.synchronize()
    ek, ev = oracle.copy_blocks(kp0, vp0, np.zeros_like(wl.bf16_bits(host_k)),
                                np.zeros_like(wl.bf16_bits(host_v)), out_pairs.cpu().numpy())
    assert np.array_equal(wl.bf16_bits(host_k), ek) and np.array_equal(wl.bf16_bits(host_v), ev)
    in_pairs = torch.tensor([[i, 52 + i] for i in range(8)], dtype=torch.int64, device="cuda")
    pkv.pkv_copy_blocks(host_k, host_v, inp.k_pool, inp.v_pool, in_pairs)    # swap back in
    torch.cuda.synchronize()
    ek2, ev2 = oracle.copy_blocks(ek, ev, kp0, vp0, in_pairs.cpu().numpy())
    assert np.array_equal(wl.bf16_bits(inp.k_pool), ek2)
    assert np.array_equal(wl.bf16_bits(inp.v_pool), ev2)


def test_copy_blocks_out_of_range_is_reported():
    shape = wl.StepShape("cowbad", [40], [1], 4, 2, num_blocks=8, seed=35)
    inp = wl.make_step(shape, device="cuda")
    before = wl.bf16_bits(inp.k_pool).copy()
    pairs = torch.tensor([[2, 8]], dtype=torch.int64, device="cuda")
    pkv.pkv_copy_blocks(inp.k_pool, inp.v_pool, inp.k_pool, inp.v_pool, pairs)
    assert pkv.pkv_get_device_error() == pkv._binding.PKV_ERR_DEVICE_BOUNDS
    assert np.array_equal(wl.bf16_bits(inp.k_pool), before)


@pytest.mark.parametrize("R", [31, 32, 33, 100, 255, 256, 257, 600])
@pytest.mark.parametrize("g", [2, 6])
def test_plan_request_counts(R, g):
    # the decode plan batches the request records of small steps (up to 256
    # requests) and walks larger steps in rounds; both must cut the step the
    # same way the oracle reads it
    rng = np.random.default_rng(700 + R + g)
    lens = rng.integers(1, 90, size=R)
    shape = wl.StepShape(f"plan_r{R}_g{g}", lens, np.ones(R, np.int32), 2 * g, 2, seed=700 + R)
    _full_parity(shape)


def test_plan_cache_follows_lengths(pkv_opts):
    # One workspace across calls whose lengths change and come back: the
    # cached per-CTA plans are reused only for identical lengths, so every
    # call matches the oracle, and equals a call with caching switched off.
    R = 40
    rng = np.random.default_rng(720)
    shapes = []
    for seed in (721, 722, 721):
        lens = np.random.default_rng(seed).integers(5, 400, size=R)
        shapes.append(wl.StepShape(f"plan_cache_{seed}", lens, np.ones(R, np.int32), 12, 2,
                                   seed=seed))
    d = None
    ws = None
    for shape in shapes:
        inp = wl.make_step(shape, device="cuda")
        h = host_copy(inp)
        kp, vp = oracle_pools_after_append(h)
        if ws is None:
            d = pkv.make_dims(tuple(inp.q.shape), tuple(inp.k_pool.shape), R,
                              max(s.max_blocks_per_req for s in shapes))
            ws = pkv.Workspace(d)
            pkv.pkv_workspace_init(ws, d)
        bt = torch.full((R, d.max_blocks_per_req), -1, dtype=torch.int32, device="cuda")
        bt[:, :inp.block_tables.shape[1]] = inp.block_tables
        pkv.pkv_append(inp.k_new, inp.v_new, inp.slot_mapping, inp.k_pool, inp.v_pool)
        outs = []
        for _ in range(2):  # the second call reuses the plans of the first
            outs.append(pkv.pkv_attention(inp.q, inp.k_pool, inp.v_pool, bt, inp.seq_lens,
                                          inp.query_start_loc, inp.scale, workspace=ws))
        pkv_opts(plan_cache=0)
        outs.append(pkv.pkv_attention(inp.q, inp.k_pool, inp.v_pool, bt, inp.seq_lens,
                                      inp.query_start_loc, inp.scale, workspace=ws))
        pkv_opts(plan_cache=1)
        torch.cuda.synchronize()
        assert pkv.pkv_get_device_error() == 0, pkv.pkv_last_error()
        assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
        bt_h = bt.cpu().numpy()
        h["block_tables"] = bt_h
        assert_close(to_f64(outs[0]), oracle_full(h, kp, vp), shape.name)


@pytest.mark.parametrize("width", [600, 5000])
def test_wide_table_small_step_matches_narrow_table(width):
    # A table far wider than the lengths need makes the host launch the
    # tensor-core decode on two CTAs per SM; the plan then finds the work
    # small and gives it to the first half of the grid only (the rest exit
    # at once).  The split is the same as with the narrow table: same bits.
    shape = wl.StepShape("wide_table", np.full(64, 512), np.ones(64), 12, 2, seed=81)
    inp = wl.make_step(shape, device="cuda", poison=True)
    h = host_copy(inp)
    kp, vp = oracle_pools_after_append(h)
    narrow = gpu_step(inp)
    wide_bt = torch.full((shape.num_reqs, width), -1, dtype=torch.int32, device="cuda")
    wide_bt[:, :inp.block_tables.shape[1]] = inp.block_tables
    wide = pkv.pkv_attention(inp.q, inp.k_pool, inp.v_pool, wide_bt, inp.seq_lens,
                             inp.query_start_loc, inp.scale)
    torch.cuda.synchronize()
    assert pkv.pkv_get_device_error() == 0, pkv.pkv_last_error()
    assert torch.equal(narrow.view(torch.int16), wide.view(torch.int16))
    assert_close(to_f64(wide), oracle_full(h, kp, vp), "wide table")
