"""Bucketed batch sizes: one CUDA graph per bucket serves every step that fits.

A serving engine captures one graph per batch-size bucket and keeps the step
buffers fixed while their contents change (The Serving Playbook, "CUDA
graphs and the CPU you forgot about").  The library's contract for a step
smaller than its bucket: the unused requests have q_r = 0 (their
query_start_loc entries repeat the last live one) and L_r = 0, their table
rows are not read, padding query rows take slot -1 in the slot mapping, and
rows query_start_loc[R] .. num_q_tokens - 1 of out are never written.

Each test captures one graph (append + attention of one layer) at a bucket
and replays it for several live steps written into the same buffers,
comparing the live rows with the fp64 oracle (its own append on host copies
of the pre-append pools) and checking that the padding rows still hold the
sentinel they were filled with.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_195_gb300 as pkv
from paged_kv_cache_195_gb300 import build as pkv_build
from paged_kv_cache_195_gb300 import workloads as wl

from pkv_testutil import assert_close, host_copy, oracle_full, oracle_pools_after_append, to_f64

pytestmark = pytest.mark.gpu

SENTINEL = 7.0  # a bf16 value no attention output of N(0,1) values reaches


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv_build.build()
    pkv.load_library()
    yield
    assert pkv.pkv_get_device_error() == 0, pkv.pkv_last_error()


class Bucket:
    """The fixed step buffers of one bucket: R requests, T query rows, a
    pool of NB blocks and tables of MB columns."""

    def __init__(self, R, T, Hq, Hkv, NB, MB, fused):
        dev = "cuda"
        self.R, self.T, self.fused = R, T, fused
        self.q = torch.zeros(T, Hq, 128, dtype=torch.bfloat16, device=dev)
        self.k_new = torch.zeros(T, Hkv, 128, dtype=torch.bfloat16, device=dev)
        self.v_new = torch.zeros_like(self.k_new)
        self.slots = torch.full((T,), -1, dtype=torch.int64, device=dev)
        self.k_pool = torch.zeros(NB, Hkv, 16, 128, dtype=torch.bfloat16, device=dev)
        self.v_pool = torch.zeros_like(self.k_pool)
        self.bt = torch.full((R, MB), -1, dtype=torch.int32, device=dev)
        self.seq = torch.zeros(R, dtype=torch.int32, device=dev)
        self.qsl = torch.zeros(R + 1, dtype=torch.int32, device=dev)
        self.out = torch.zeros(T, Hq, 128, dtype=torch.bfloat16, device=dev)
        dims = pkv.make_dims((T, Hq, 128), (NB, Hkv, 16, 128), R, MB)
        self.ws = pkv.Workspace(dims)
        pkv.pkv_workspace_init(self.ws, dims)
        self.scale = 128 ** -0.5

    def layer(self):
        if self.fused:
            pkv.pkv_append_attention(self.k_new, self.v_new, self.slots, self.k_pool, self.v_pool,
                                     self.q, self.bt, self.seq, self.qsl, self.scale,
                                     out=self.out, workspace=self.ws)
        else:
            pkv.pkv_append(self.k_new, self.v_new, self.slots, self.k_pool, self.v_pool)
            pkv.pkv_attention(self.q, self.k_pool, self.v_pool, self.bt, self.seq, self.qsl,
                              self.scale, out=self.out, workspace=self.ws)

    def capture(self):
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            self.layer()  # eager warm-up with the all-padding contents
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            self.layer()
        return g

    def load(self, inp):
        """Write one live step into the buffers; everything past it is padding."""
        n, t = inp.shape.num_reqs, inp.shape.num_q_tokens
        assert n <= self.R and t <= self.T
        self.q.fill_(float("nan"))      # padding rows of q are never read
        self.q[:t] = inp.q
        self.k_new.fill_(float("nan"))
        self.k_new[:t] = inp.k_new
        self.v_new.fill_(float("nan"))
        self.v_new[:t] = inp.v_new
        self.slots.fill_(-1)
        self.slots[:t] = inp.slot_mapping
        self.k_pool.copy_(inp.k_pool)
        self.v_pool.copy_(inp.v_pool)
        self.bt.fill_(-1)
        self.bt[:n, :inp.block_tables.shape[1]] = inp.block_tables
        self.bt[n:] = 1 << 30           # padding rows' tables are not read
        self.seq.zero_()
        self.seq[:n] = inp.seq_lens
        self.qsl.fill_(t)
        self.qsl[:n + 1] = inp.query_start_loc
        self.out.fill_(SENTINEL)


def _replay_and_check(bucket, graph, shape, layer):
    inp = wl.make_step(shape, device="cuda", layer=layer, poison=True)
    h = host_copy(inp)
    bucket.load(inp)
    graph.replay()
    torch.cuda.synchronize()
    assert pkv.pkv_get_device_error() == 0, pkv.pkv_last_error()
    t = shape.num_q_tokens
    assert bool((bucket.out[t:].float() == SENTINEL).all()), "a padding row of out was written"
    kp, vp = oracle_pools_after_append(h)
    assert_close(to_f64(bucket.out[:t]), oracle_full(h, kp, vp), shape.name)


@pytest.mark.parametrize("fused", [False, True], ids=["append_then_attention", "append_attention"])
def test_decode_bucket_of_64_serves_64_50_and_7_requests(fused):
    R, NB, MB = 64, 2600, 40
    bucket = Bucket(R, R, 12, 2, NB, MB, fused)
    graph = bucket.capture()
    rng = np.random.default_rng(830)
    for n in (64, 50, 7):
        lens = rng.integers(1, MB * 16 + 1, size=n)
        shape = wl.StepShape(f"bucket64_live{n}", lens, np.ones(n, np.int32), 12, 2,
                             num_blocks=NB, seed=831 + n)
        _replay_and_check(bucket, graph, shape, layer=n)


def test_mixed_bucket_with_prefill_chunks():
    # a token bucket larger than the live tokens: decode rows and prefill
    # chunks (tensor-core prefill kernel) in front, padding rows behind
    R, T, NB, MB = 16, 640, 1200, 48
    bucket = Bucket(R, T, 32, 8, NB, MB, fused=False)
    graph = bucket.capture()
    steps = [
        ([300, 40, 517, 129, 16, 700], [1, 40, 200, 3, 16, 1]),
        ([90] * 16, [1] * 16),
        ([612, 33], [500, 1]),
    ]
    for i, (lens, ql) in enumerate(steps):
        shape = wl.StepShape(f"bucket_mixed_{i}", lens, ql, 32, 8, num_blocks=NB, seed=840 + i)
        _replay_and_check(bucket, graph, shape, layer=i)
