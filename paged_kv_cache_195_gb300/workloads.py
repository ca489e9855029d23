"""Seeded synthetic inputs for one paged-attention engine step.

This module is shared by the CUDA path's tests and benchmark and by the fp64
oracle's tests.  It holds none of the attention arithmetic: it only draws
lengths, block placements and N(0,1) values, and lays them out in the shapes
the step consumes.

A step's inputs (one layer):

* ``q``            [Tq, Hq, D] bf16: this step's query rows, requests in order.
* ``k_new/v_new``  [Tq, Hkv, D] bf16: the K/V rows of the same tokens.
* ``slot_mapping`` [Tq] int64: pool slot (block * bs + offset) of each token.
* ``k_pool/v_pool`` [num_blocks, Hkv, bs, D] bf16: the paged cache.  Every
  slot holds N(0,1) values (or NaN for ``poison=True`` at slots no request
  owns, i.e. free blocks and the tails of partly filled last blocks).
* ``block_tables`` [R, max_blocks] int32: physical block of each logical block;
  entries past a request's last block are -1.
* ``seq_lens``     [R] int32: L_r, the request's length including this step's
  tokens.  ``query_start_loc`` [R+1] int32: cumulative query counts.

Physical blocks are handed out from a seeded random permutation of the pool,
in request order, so logical order never matches physical order (the property
the paged cache exists for: The Serving Playbook, "Paged KV cache").
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

BLOCK_SIZE = 16
HEAD_DIM = 128


@dataclasses.dataclass
class StepShape:
    """Lengths and head counts of one step; no tensors."""
    name: str
    seq_lens: np.ndarray          # int32 [R]
    q_lens: np.ndarray            # int32 [R]
    num_q_heads: int
    num_kv_heads: int
    head_dim: int = HEAD_DIM
    block_size: int = BLOCK_SIZE
    num_blocks: int | None = None  # default: 1.25 x live blocks
    layers: int = 1
    seed: int = 195
    # Shared prefixes: (first request, members, blocks).  Requests first ..
    # first + members - 1 point their first `blocks` table entries at the
    # same physical blocks (one copy of a common prompt in the pool).
    prefix_groups: tuple = ()

    def __post_init__(self):
        self.seq_lens = np.asarray(self.seq_lens, dtype=np.int32)
        self.q_lens = np.asarray(self.q_lens, dtype=np.int32)
        assert self.seq_lens.shape == self.q_lens.shape
        assert (self.q_lens >= 0).all() and (self.q_lens <= self.seq_lens).all()
        for first, members, blocks in self.prefix_groups:
            for r in range(first, first + members):
                # every member's new tokens come after the shared prefix
                assert self.seq_lens[r] - self.q_lens[r] >= blocks * self.block_size
        if self.num_blocks is None:
            self.num_blocks = max(1, int(math.ceil(1.25 * self.live_blocks)))
        assert self.num_blocks >= self.live_blocks

    @property
    def num_reqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def blocks_per_req(self) -> np.ndarray:
        return (self.seq_lens + self.block_size - 1) // self.block_size

    @property
    def live_blocks(self) -> int:
        shared = sum((members - 1) * blocks for _, members, blocks in self.prefix_groups)
        return int(self.blocks_per_req.sum()) - shared

    @property
    def max_blocks_per_req(self) -> int:
        return max(1, int(self.blocks_per_req.max(initial=0)))

    @property
    def num_q_tokens(self) -> int:
        return int(self.q_lens.sum())

    @property
    def query_start_loc(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.q_lens)]).astype(np.int32)


# --------------------------------------------------------------------------
# The five workloads (shapes of a Qwen2.5-1.5B and a Llama-3-8B attention
# layer; no weights, no dataset: lengths and values are drawn here).
# --------------------------------------------------------------------------

def tiny_decode() -> StepShape:
    """4 decode requests, L = 17/64/100/128, Hq=12, Hkv=2, 64-block pool."""
    return StepShape("tiny_decode_r4", [17, 64, 100, 128], [1, 1, 1, 1], 12, 2,
                     num_blocks=64, seed=195)


def qwen_decode(layers: int = 28) -> StepShape:
    """64 decode requests of length 512, Qwen2.5-1.5B heads, one pool/layer."""
    return StepShape("qwen2.5-1.5b_decode_r64_L512", [512] * 64, [1] * 64, 12, 2,
                     layers=layers, seed=195)


def qwen_long_batch() -> StepShape:
    """128 decode requests of length 2048, Qwen2.5-1.5B heads."""
    return StepShape("qwen2.5-1.5b_decode_r128_L2048", [2048] * 128, [1] * 128,
                     12, 2, seed=195)


def llama_mixed(num_decode: int = 248, num_prefill: int = 8,
                chunk: int = 512) -> StepShape:
    """Continuous-batching step: lognormal decodes plus chunked prefills.

    Decode lengths: round(exp(N(ln 1000, 1.0))) clamped to 16..8192 (seed 195).
    Prefill chunks: 512 query tokens after a cached prefix uniform on the
    integers 0..4096 (seed 196), so L = prefix + 512.  Decodes come first.
    """
    rng = np.random.default_rng(195)
    dec = np.clip(np.rint(np.exp(rng.normal(math.log(1000.0), 1.0, num_decode))),
                  16, 8192).astype(np.int32)
    rng2 = np.random.default_rng(196)
    prefix = rng2.integers(0, 4096, size=num_prefill, endpoint=True).astype(np.int32)
    seq = np.concatenate([dec, prefix + chunk]).astype(np.int32)
    ql = np.concatenate([np.ones(num_decode, np.int32),
                         np.full(num_prefill, chunk, np.int32)])
    return StepShape(f"llama3-8b_mixed_d{num_decode}_p{num_prefill}x{chunk}", seq, ql, 32, 8,
                     seed=195)


def llama_long_context() -> StepShape:
    """8 decode requests of length 32768, Llama-3-8B heads."""
    return StepShape("llama3-8b_decode_r8_L32768", [32768] * 8, [1] * 8, 32, 8,
                     seed=195)


def qwen_shared_prefix(layers: int = 28) -> StepShape:
    """The Qwen decode step (64 x 512) with a shared prompt: four groups of 16
    requests share their first 384 tokens (24 blocks)."""
    groups = tuple((16 * i, 16, 24) for i in range(4))
    return StepShape("qwen2.5-1.5b_decode_r64_L512_shared4x384", [512] * 64, [1] * 64, 12, 2,
                     layers=layers, seed=195, prefix_groups=groups)


def qwen_shared_long() -> StepShape:
    """The Qwen long batch (128 x 2048) with shared prompts: eight groups of
    16 requests share their first 1536 tokens (96 blocks)."""
    groups = tuple((16 * i, 16, 96) for i in range(8))
    return StepShape("qwen2.5-1.5b_decode_r128_L2048_shared8x1536", [2048] * 128, [1] * 128,
                     12, 2, seed=195, prefix_groups=groups)


CONFIGS = {
    "tiny": tiny_decode,
    "qwen_decode": qwen_decode,
    "qwen_long": qwen_long_batch,
    "llama_mixed": llama_mixed,
    "llama_long": llama_long_context,
    "llama_prefill": lambda: llama_mixed(num_decode=0),
    "llama_decode": lambda: llama_mixed(num_prefill=0),
    "qwen_shared": qwen_shared_prefix,
    "qwen_shared_long": qwen_shared_long,
}


# --------------------------------------------------------------------------
# Tensor generation
# --------------------------------------------------------------------------

@dataclasses.dataclass
class StepInputs:
    shape: StepShape
    q: torch.Tensor
    k_new: torch.Tensor
    v_new: torch.Tensor
    slot_mapping: torch.Tensor
    k_pool: torch.Tensor
    v_pool: torch.Tensor
    block_tables: torch.Tensor
    seq_lens: torch.Tensor
    query_start_loc: torch.Tensor
    scale: float


def block_placement(shape: StepShape, seed: int) -> np.ndarray:
    """[R, max_blocks] int32 physical block ids from a seeded permutation.
    Members of a shared-prefix group after the first reuse the first
    member's leading blocks."""
    perm = np.random.default_rng(seed).permutation(shape.num_blocks).astype(np.int32)
    bt = np.full((shape.num_reqs, shape.max_blocks_per_req), -1, dtype=np.int32)
    share = {}
    for first, members, blocks in shape.prefix_groups:
        for r in range(first + 1, first + members):
            share[r] = (first, blocks)
    nxt = 0
    for r, nb in enumerate(shape.blocks_per_req):
        start = 0
        if r in share:
            first, start = share[r]
            bt[r, :start] = bt[first, :start]
        bt[r, start:nb] = perm[nxt:nxt + nb - start]
        nxt += int(nb) - start
    return bt


def new_token_slots(shape: StepShape, block_tables: np.ndarray) -> np.ndarray:
    """Pool slot of each of this step's tokens: positions L_r - q_r .. L_r - 1."""
    bs = shape.block_size
    slots = np.empty(shape.num_q_tokens, dtype=np.int64)
    t = 0
    for r in range(shape.num_reqs):
        L, ql = int(shape.seq_lens[r]), int(shape.q_lens[r])
        for pos in range(L - ql, L):
            slots[t] = int(block_tables[r, pos // bs]) * bs + pos % bs
            t += 1
    return slots


def owned_slot_mask(shape: StepShape, block_tables: np.ndarray) -> np.ndarray:
    """bool [num_blocks, bs]: True where some request's token lives."""
    bs = shape.block_size
    mask = np.zeros((shape.num_blocks, bs), dtype=bool)
    for r in range(shape.num_reqs):
        L = int(shape.seq_lens[r])
        for b in range((L + bs - 1) // bs):
            n = min(bs, L - b * bs)
            mask[block_tables[r, b], :n] = True
    return mask


def _randn_bf16(shape, gen, device):
    return torch.randn(shape, generator=gen, device=device,
                       dtype=torch.float32).to(torch.bfloat16)


def make_step(shape: StepShape, device="cpu", layer: int = 0,
              poison: bool = False) -> StepInputs:
    """Seeded inputs of one layer of one step (seed = shape.seed + layer)."""
    device = torch.device(device)
    seed = shape.seed + layer
    bt = block_placement(shape, seed)
    slots = new_token_slots(shape, bt)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    Hq, Hkv, D, bs = shape.num_q_heads, shape.num_kv_heads, shape.head_dim, shape.block_size
    T = shape.num_q_tokens
    pool_shape = (shape.num_blocks, Hkv, bs, D)
    k_pool = _randn_bf16(pool_shape, gen, device)
    v_pool = _randn_bf16(pool_shape, gen, device)
    q = _randn_bf16((T, Hq, D), gen, device)
    k_new = _randn_bf16((T, Hkv, D), gen, device)
    v_new = _randn_bf16((T, Hkv, D), gen, device)
    if poison:
        owned = torch.from_numpy(owned_slot_mask(shape, bt)).to(device)
        free = (~owned)[:, None, :, None].expand(pool_shape)
        k_pool = k_pool.masked_fill(free, float("nan"))
        v_pool = v_pool.masked_fill(free, float("nan"))
    return StepInputs(
        shape=shape, q=q, k_new=k_new, v_new=v_new,
        slot_mapping=torch.from_numpy(slots).to(device),
        k_pool=k_pool, v_pool=v_pool,
        block_tables=torch.from_numpy(bt).to(device),
        seq_lens=torch.from_numpy(shape.seq_lens.copy()).to(device),
        query_start_loc=torch.from_numpy(shape.query_start_loc).to(device),
        scale=1.0 / math.sqrt(D))


@dataclasses.dataclass
class Fp8StepInputs:
    """A step over e4m3 pools: the bf16 fields of ``StepInputs`` except the
    pools, which hold uint8 codes, plus the per-KV-head scales."""
    shape: StepShape
    q: torch.Tensor
    k_new: torch.Tensor
    v_new: torch.Tensor
    slot_mapping: torch.Tensor
    k_pool: torch.Tensor   # uint8 [num_blocks, Hkv, bs, D]
    v_pool: torch.Tensor
    k_scale: torch.Tensor  # float32 [Hkv]
    v_scale: torch.Tensor
    block_tables: torch.Tensor
    seq_lens: torch.Tensor
    query_start_loc: torch.Tensor
    scale: float


E4M3_NAN = 0x7F  # the positive NaN code (exponent and mantissa all ones)


def make_fp8_step(shape: StepShape, device="cpu", layer: int = 0,
                  poison: bool = False) -> Fp8StepInputs:
    """Seeded inputs of one layer of one step with e4m3 pools.

    Pool codes are drawn uniformly from the 254 non-NaN codes (they are
    inputs: nothing here encodes a value); per-KV-head scales are drawn from
    [0.003, 0.0045], so a stored value is at most 448 * 0.0045 ~ 2 in
    magnitude.  ``poison`` puts the NaN code at slots no request owns."""
    device = torch.device(device)
    seed = shape.seed + layer
    bt = block_placement(shape, seed)
    slots = new_token_slots(shape, bt)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    Hq, Hkv, D, bs = shape.num_q_heads, shape.num_kv_heads, shape.head_dim, shape.block_size
    T = shape.num_q_tokens
    pool_shape = (shape.num_blocks, Hkv, bs, D)

    def codes():
        r = torch.randint(0, 254, pool_shape, generator=gen, device=device, dtype=torch.int32)
        return (r + (r >= E4M3_NAN).to(torch.int32)).to(torch.uint8)  # skip 0x7F and 0xFF

    k_pool, v_pool = codes(), codes()
    q = _randn_bf16((T, Hq, D), gen, device)
    k_new = _randn_bf16((T, Hkv, D), gen, device)
    v_new = _randn_bf16((T, Hkv, D), gen, device)
    sc = torch.rand((2, Hkv), generator=gen, device=device, dtype=torch.float32)
    k_scale = (0.003 + 0.0015 * sc[0]).contiguous()
    v_scale = (0.003 + 0.0015 * sc[1]).contiguous()
    if poison:
        owned = torch.from_numpy(owned_slot_mask(shape, bt)).to(device)
        free = (~owned)[:, None, :, None].expand(pool_shape)
        k_pool = k_pool.masked_fill(free, E4M3_NAN)
        v_pool = v_pool.masked_fill(free, E4M3_NAN)
    return Fp8StepInputs(
        shape=shape, q=q, k_new=k_new, v_new=v_new,
        slot_mapping=torch.from_numpy(slots).to(device),
        k_pool=k_pool, v_pool=v_pool, k_scale=k_scale, v_scale=v_scale,
        block_tables=torch.from_numpy(bt).to(device),
        seq_lens=torch.from_numpy(shape.seq_lens.copy()).to(device),
        query_start_loc=torch.from_numpy(shape.query_start_loc).to(device),
        scale=1.0 / math.sqrt(D))


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """uint16 bit patterns of a bf16 tensor, on the host."""
    assert t.dtype == torch.bfloat16
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def random_small_shape(rng: np.random.Generator, name="random", max_reqs=5,
                       max_len=70, Hq=None, Hkv=None, block_size=BLOCK_SIZE,
                       head_dim=HEAD_DIM, max_q=None) -> StepShape:
    """A small ragged step: random lengths, random query counts (some 0)."""
    R = int(rng.integers(1, max_reqs + 1))
    seq = rng.integers(1, max_len + 1, size=R).astype(np.int32)
    qmax = seq if max_q is None else np.minimum(seq, max_q)
    ql = np.array([int(rng.integers(0, m + 1)) for m in qmax], dtype=np.int32)
    if ql.sum() == 0:
        ql[0] = 1
    if Hkv is None:
        Hkv = int(rng.choice([1, 2, 4]))
    if Hq is None:
        Hq = Hkv * int(rng.choice([1, 2, 3, 4, 6, 8]))
    return StepShape(name, seq, ql, Hq, Hkv, head_dim=head_dim,
                     block_size=block_size, seed=int(rng.integers(0, 2**31)))
