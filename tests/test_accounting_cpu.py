"""The benchmark's accounting and its workloads, on the CPU.

Algorithmic bytes and flops (roofline.py) are checked against brute-force
counts over the rows and keys each query row sees, and against the KV-size
formula (What Actually Runs the Model, "The KV cache": 2 x Hkv x D x bytes
per token and layer); the workloads are checked against the recipes they
state (shapes, length ranges, seeded determinism, block placement).
"""
import numpy as np
import pytest

from paged_kv_cache_195_gb300 import roofline as rl
from paged_kv_cache_195_gb300 import workloads as wl


def _brute_keys(seq_lens, q_lens):
    # visible keys summed over every query row (row i of a chunk of q at the
    # end of L sees L - q + i + 1 keys)
    return sum(L - q + i + 1 for L, q in zip(seq_lens, q_lens) for i in range(q))


@pytest.mark.parametrize("seed", range(5))
def test_flops_match_a_row_by_row_count(seed):
    rng = np.random.default_rng(seed)
    q = rng.integers(0, 40, size=12)
    L = q + rng.integers(0, 300, size=12)
    Hq = int(rng.choice([8, 12, 32]))
    assert rl.attention_flops(L, q, Hq) == 4 * _brute_keys(L, q) * Hq * 128


def test_bytes_follow_the_kv_size_formula():
    # Qwen-shaped (Hkv=2): 1 KiB of K+V per token and layer; Llama (Hkv=8): 4 KiB
    assert rl.kv_bytes_per_token(2) == 1024 and rl.kv_bytes_per_token(8) == 4096
    assert rl.kv_bytes_per_token(2, dtype_bytes=1) == 512
    shape = wl.qwen_decode(layers=1)
    b = rl.attention_bytes(shape.seq_lens, shape.q_lens, 12, 2)
    assert b["kv"] == 64 * 512 * 1024
    assert b["q_out"] == 64 * 12 * 128 * 2 * 2
    assert b["total"] == 33947648  # the per-launch figure the profiles quote
    # a request without queries reads nothing
    b2 = rl.attention_bytes([100, 50], [0, 1], 12, 2)
    assert b2["kv"] == 50 * 1024
    # prefill chunks read each key once per (request, KV head)
    b3 = rl.attention_bytes([600], [200], 32, 8)
    assert b3["kv"] == 600 * 4096


def test_shared_prefix_bytes_count_each_prompt_once():
    shape = wl.qwen_shared_prefix(layers=1)
    u = rl.unique_kv_bytes(shape.seq_lens, shape.q_lens, 2, shape.prefix_groups)
    saved = 4 * 15 * 24 * 16  # 4 groups, 15 extra members, 24 blocks of 16 tokens
    assert u == (64 * 512 - saved) * 1024
    assert rl.unique_kv_bytes(shape.seq_lens, shape.q_lens, 2, ()) == 64 * 512 * 1024


def test_append_bytes():
    assert rl.append_bytes(64, 2) == 2 * 64 * 2 * 128 * (2 + 2)
    assert rl.append_bytes(64, 2, kv_dtype_bytes=1) == 2 * 64 * 2 * 128 * (2 + 1)


def test_mixed_workload_follows_its_recipe():
    s = wl.llama_mixed()
    assert s.num_reqs == 256 and s.num_q_heads == 32 and s.num_kv_heads == 8
    dec, pre = slice(0, 248), slice(248, 256)
    assert (s.q_lens[dec] == 1).all() and (s.q_lens[pre] == 512).all()
    assert s.seq_lens[dec].min() >= 16 and s.seq_lens[dec].max() <= 8192
    prefix = s.seq_lens[pre] - 512
    assert prefix.min() >= 0 and prefix.max() <= 4096
    # lognormal around 1000: the median of the decode lengths is near it
    assert 600 <= np.median(s.seq_lens[dec]) <= 1600
    t = wl.llama_mixed()
    assert np.array_equal(s.seq_lens, t.seq_lens) and np.array_equal(s.q_lens, t.q_lens)


@pytest.mark.parametrize("name", sorted(wl.CONFIGS))
def test_every_workload_places_blocks_validly(name):
    s = wl.CONFIGS[name]()
    bt = wl.block_placement(s, s.seed)
    assert s.num_blocks >= s.live_blocks
    shared = set()
    for first, members, blocks in s.prefix_groups:
        for r in range(first + 1, first + members):
            assert (bt[r, :blocks] == bt[first, :blocks]).all()
        shared.update(range(first + 1, first + members))
    used = []
    for r in range(s.num_reqs):
        nb = -(-int(s.seq_lens[r]) // 16)
        row = bt[r, :nb]
        assert (row >= 0).all() and (row < s.num_blocks).all()
        skip = 0
        for first, members, blocks in s.prefix_groups:
            if first < r < first + members:
                skip = blocks
        used.extend(row[skip:].tolist())
    # apart from the shared prompts, no two table entries name the same block
    assert len(used) == len(set(used))
