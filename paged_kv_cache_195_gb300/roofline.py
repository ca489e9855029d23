"""Algorithmic byte and flop accounting of one paged-attention step.

The step reads every cached K and V row a query row may see exactly once per
(request, KV head), whatever the group size g and however the work is split;
it reads q and writes out once.  KV bytes per token and layer are
2 (K and V) x Hkv x D x 2 bytes -- the per-token, per-layer term of the
KV-cache size formula (What Actually Runs the Model, "The KV cache").  Block
tables and lengths are not counted (4 bytes per 16 tokens).  An e4m3 pool
stores one byte per element (The Serving Playbook, "Quantized serving"); q,
out and the appended rows stay bf16.
"""
from __future__ import annotations

import numpy as np

BF16 = 2


def kv_bytes_per_token(num_kv_heads: int, head_dim: int = 128, dtype_bytes: int = BF16) -> int:
    return 2 * num_kv_heads * head_dim * dtype_bytes


def kv_cache_bytes(layers, kv_heads, head_dim, dtype_bytes, seq_len, batch) -> int:
    return 2 * layers * kv_heads * head_dim * dtype_bytes * seq_len * batch


def attention_bytes(seq_lens, q_lens, num_q_heads, num_kv_heads, head_dim=128,
                    kv_dtype_bytes: int = BF16) -> dict:
    """Algorithmic HBM bytes of one attention call.

    Decode rows (q_r = 1) read their L_r keys; a prefill chunk reads its L_r
    keys once per (request, KV head) -- its query tile reuses them on chip.
    """
    seq_lens = np.asarray(seq_lens, np.int64)
    q_lens = np.asarray(q_lens, np.int64)
    active = q_lens > 0
    kv = int(seq_lens[active].sum()) * kv_bytes_per_token(num_kv_heads, head_dim, kv_dtype_bytes)
    qo = int(q_lens.sum()) * num_q_heads * head_dim * BF16 * 2
    return {"kv": kv, "q_out": qo, "total": kv + qo}


def unique_kv_bytes(seq_lens, q_lens, num_kv_heads, prefix_groups, block_size=16,
                    head_dim=128, kv_dtype_bytes: int = BF16) -> int:
    """KV bytes a step must read when each shared prefix (first request,
    members, blocks) is read once for its group instead of once per member."""
    seq_lens = np.asarray(seq_lens, np.int64)
    q_lens = np.asarray(q_lens, np.int64)
    tokens = int(seq_lens[q_lens > 0].sum())
    for first, members, blocks in prefix_groups:
        active = int((q_lens[first:first + members] > 0).sum())
        tokens -= max(0, active - 1) * blocks * block_size
    return tokens * kv_bytes_per_token(num_kv_heads, head_dim, kv_dtype_bytes)


def append_bytes(num_tokens, num_kv_heads, head_dim=128, kv_dtype_bytes: int = BF16) -> int:
    """Read k_new/v_new (bf16) and write them into the pool (bf16 or e4m3)."""
    return 2 * num_tokens * num_kv_heads * head_dim * (BF16 + kv_dtype_bytes)


def attention_flops(seq_lens, q_lens, num_q_heads, head_dim=128) -> int:
    """2 x (QK^T + PV) multiply-adds over the causal keys of every row."""
    total = 0
    for L, q in zip(np.asarray(seq_lens, np.int64), np.asarray(q_lens, np.int64)):
        if q <= 0:
            continue
        keys = q * (L - q) + q * (q + 1) // 2  # sum over rows of visible keys
        total += 4 * int(keys) * num_q_heads * head_dim
    return total


def attended_tokens(seq_lens, q_lens) -> int:
    """Sum of L_r over requests that have queries (tokens attended per call)."""
    seq_lens = np.asarray(seq_lens, np.int64)
    return int(seq_lens[np.asarray(q_lens) > 0].sum())
