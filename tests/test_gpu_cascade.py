"""Shared-prefix (cascade) attention on the GPU against the oracle.

Requests in a sharing group point their first table entries at the same
physical blocks.  pkv_attention_cascade reads those blocks once for the whole
group (the prefix pass), reads each member's remaining blocks in the decode,
and merges the two partial softmax states.  Its output must match the
oracle's plain attention over the same tables within the usual tolerance.
"""
import numpy as np
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


def _groups(shape, device="cuda"):
    g = np.array(shape.prefix_groups, dtype=np.int32).reshape(-1, 3)
    return tuple(torch.from_numpy(np.ascontiguousarray(g[:, i])).to(device) for i in range(3))


def _cascade(inp, groups=None, append=True):
    if append:
        pkv.pkv_append(inp.k_new, inp.v_new, inp.slot_mapping, inp.k_pool, inp.v_pool)
    first, count, blocks = groups if groups is not None else _groups(inp.shape)
    return pkv.pkv_attention_cascade(inp.q, inp.k_pool, inp.v_pool, inp.block_tables,
                                     inp.seq_lens, inp.query_start_loc, first, count, blocks,
                                     inp.scale)


def _parity(shape, poison=True):
    inp = wl.make_step(shape, device="cuda", poison=poison)
    h = host_copy(inp)
    kp, vp = oracle_pools_after_append(h)
    out = _cascade(inp)
    torch.cuda.synchronize()
    assert pkv.pkv_get_device_error() == 0, pkv.pkv_last_error()
    return assert_close(to_f64(out), oracle_full(h, kp, vp), shape.name), inp, out


@pytest.mark.parametrize("g", [4, 6, 8])
def test_cascade_group_sizes(g):
    # two groups plus requests outside any group; prefixes of 5 and 12 blocks
    shape = wl.StepShape(f"cascade_g{g}", [100, 95, 130, 300, 210, 222, 17, 400],
                         [1, 1, 1, 1, 1, 1, 1, 1], 2 * g, 2, seed=300 + g,
                         prefix_groups=((0, 3, 5), (3, 3, 12)))
    _parity(shape)


def test_cascade_multi_query_members():
    # members with several query rows (short chunks) behind the prefix
    shape = wl.StepShape("cascade_mq", [200, 180, 190, 64], [3, 1, 5, 2], 24, 4, seed=311,
                         prefix_groups=((0, 3, 9),))
    _parity(shape)


def test_cascade_long_prefix_split_suffix():
    # 50 members share a 1024-token prompt; long private suffixes are split
    # across CTAs, so the merge sees both pieces and the prefix partial
    lens = [1024 + 16 * (i % 7) + 5 + 40 * i for i in range(50)]
    shape = wl.StepShape("cascade_long", lens, [1] * 50, 32, 8, seed=312,
                         prefix_groups=((0, 50, 64),))
    _parity(shape, poison=False)


def test_cascade_groups_across_batches():
    """40 sharing groups of two (the prefix pass takes its groups in batches of
    32, longest shared prefix first within a batch), against plain attention
    in the oracle."""
    rng = np.random.default_rng(320)
    shared = rng.integers(1, 12, size=40)
    lens, groups = [], []
    for i, sb in enumerate(shared):
        lens += [int(sb) * 16 + int(rng.integers(1, 60)) for _ in range(2)]
        groups.append((2 * i, 2, int(sb)))
    shape = wl.StepShape("cascade_batches", lens, [1] * len(lens), 16, 2, seed=321,
                         prefix_groups=tuple(groups))
    _parity(shape)


def test_cascade_member_without_room_falls_back():
    # Requests 0-2 share 5 blocks (80 tokens); request 2's query sits at
    # position 80, right after them.
    shape = wl.StepShape("cascade_fallback", [160, 150, 81, 140], [1, 1, 1, 1], 12, 2, seed=313,
                         prefix_groups=((0, 3, 5),))
    inp = wl.make_step(shape, device="cuda", poison=True)
    h = host_copy(inp)
    kp, vp = oracle_pools_after_append(h)
    out = _cascade(inp)
    torch.cuda.synchronize()
    assert_close(to_f64(out), oracle_full(h, kp, vp), "cascade")
    # A one-member group claiming 6 blocks for request 2 covers its own query
    # position: request 2 reads its whole context itself and the result is
    # unchanged.
    bad = tuple(torch.tensor(v, dtype=torch.int32, device="cuda")
                for v in ([0, 2], [2, 1], [5, 6]))
    out2 = _cascade(inp, bad, append=False)
    torch.cuda.synchronize()
    assert_close(to_f64(out2), oracle_full(h, kp, vp), "cascade_fallback")
    assert pkv.pkv_get_device_error() == 0


def test_cascade_small_group_uses_plain_path():
    # g = 2 runs the SIMT decode: no sharing, same result
    shape = wl.StepShape("cascade_g2", [90, 70, 66], [1, 1, 1], 4, 2, seed=314,
                         prefix_groups=((0, 3, 4),))
    _parity(shape)


def test_cascade_matches_plain_attention():
    shape = wl.StepShape("cascade_vs_plain", [512] * 16, [1] * 16, 12, 2, seed=315,
                         prefix_groups=((0, 8, 20), (8, 8, 24)))
    (mx, mean), inp, out = _parity(shape, poison=False)
    plain = pkv.pkv_attention(inp.q, inp.k_pool, inp.v_pool, inp.block_tables, inp.seq_lens,
                              inp.query_start_loc, inp.scale)
    diff = (out.float() - plain.float()).abs()
    # both within the oracle tolerance; P's bf16 rounding differs between a
    # 128-key prefix tile and the decode's tiles, nothing else
    assert float(diff.max()) <= 2e-2 and float(diff.mean()) <= 1e-3


def test_cascade_qwen_shared_full_size_every_element():
    shape = wl.qwen_shared_prefix(layers=1)
    inp = wl.make_step(shape, device="cuda")
    h = host_copy(inp)
    out = _cascade(inp)
    torch.cuda.synchronize()
    assert pkv.pkv_get_device_error() == 0, pkv.pkv_last_error()
    kp, vp = oracle_pools_after_append(h)
    assert_close(to_f64(out), oracle_full(h, kp, vp), "qwen_shared")


def test_cascade_bad_group_reported(pkv_opts):
    # the groups are checked by the set-up kernel of the tensor-core route
    pkv_opts(decode_tc=1)
    shape = wl.StepShape("cascade_bad", [64, 64], [1, 1], 8, 2, seed=316,
                         prefix_groups=((0, 2, 2),))
    inp = wl.make_step(shape, device="cuda")
    groups = tuple(torch.tensor(v, dtype=torch.int32, device="cuda") for v in ([1], [5], [2]))
    _cascade(inp, groups)
    assert pkv.pkv_get_device_error() == pkv._binding.PKV_ERR_DEVICE_BOUNDS
