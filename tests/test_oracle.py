"""Pins for the fp64 oracle: checks against things other than the oracle.

Each test fixes a property that the pages or plain mathematics determine --
hand-derived worked values, a dense (unpaged) computation written here
independently, invariance under relabelling physical blocks, closed forms,
and a brute-force sum on tiny integer inputs -- so that a dropped scale, a
wrong causal offset, a wrong grouped-query mapping or a block-table indexing
slip in the oracle fails at least one of them.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_195_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bits(a: np.ndarray) -> np.ndarray:
    """float array -> bf16 bit patterns (values here are exact in bf16)."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _vals(bits: np.ndarray) -> np.ndarray:
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


def _scatter(logical_k, logical_v, bt, nb, bs, fill):
    """Place per-request logical K/V [L, Hkv, D] into a pool by block table."""
    Hkv, D = logical_k[0].shape[1:]
    kp = np.full((nb, Hkv, bs, D), fill, dtype=np.float32)
    vp = np.full((nb, Hkv, bs, D), fill, dtype=np.float32)
    for r, (K, V) in enumerate(zip(logical_k, logical_v)):
        for j in range(K.shape[0]):
            kp[bt[r, j // bs], :, j % bs, :] = K[j]
            vp[bt[r, j // bs], :, j % bs, :] = V[j]
    return kp, vp


def _dense_reference(q, logical_k, logical_v, seq_lens, qsl, scale, Hq):
    """Unpaged causal GQA attention with numpy einsum on contiguous K/V."""
    out = np.zeros(q.shape, dtype=np.float64)
    for r in range(len(seq_lens)):
        K, V = logical_k[r].astype(np.float64), logical_v[r].astype(np.float64)
        L, Hkv, _ = K.shape
        g = Hq // Hkv
        Kh, Vh = np.repeat(K, g, axis=1), np.repeat(V, g, axis=1)  # [L, Hq, D]
        a, b = qsl[r], qsl[r + 1]
        if b == a:
            continue
        Q = q[a:b].astype(np.float64)                               # [q, Hq, D]
        s = scale * np.einsum("ihd,jhd->hij", Q, Kh)                 # [Hq, q, L]
        qn = b - a
        pos = L - qn + np.arange(qn)
        mask = np.arange(L)[None, :] <= pos[:, None]                 # [q, L]
        s = np.where(mask[None], s, -np.inf)
        s = s - s.max(axis=-1, keepdims=True)
        w = np.exp(s)
        w /= w.sum(axis=-1, keepdims=True)
        out[a:b] = np.einsum("hij,jhd->ihd", w, Vh)
    return out


def _random_problem(rng, shape, fill=np.nan, int_values=False):
    """Logical per-request K/V, q, and a pool placed by a random permutation."""
    Hq, Hkv, D, bs = shape.num_q_heads, shape.num_kv_heads, shape.head_dim, shape.block_size
    draw = (lambda *s: rng.integers(-3, 4, size=s).astype(np.float32)) if int_values \
        else (lambda *s: rng.standard_normal(s).astype(np.float32))
    lk = [_vals(_bits(draw(int(L), Hkv, D))).astype(np.float32) for L in shape.seq_lens]
    lv = [_vals(_bits(draw(int(L), Hkv, D))).astype(np.float32) for L in shape.seq_lens]
    q = _vals(_bits(draw(shape.num_q_tokens, Hq, D))).astype(np.float32)
    bt = wl.block_placement(shape, int(rng.integers(0, 2**31)))
    kp, vp = _scatter(lk, lv, bt, shape.num_blocks, bs, fill)
    return q, lk, lv, bt, kp, vp


def _run_oracle(q, kp, vp, bt, shape, scale):
    return oracle.paged_attention(_bits(q), _bits(kp), _bits(vp), bt,
                                  shape.seq_lens, shape.query_start_loc, scale)


# ---------------------------------------------------------------------------
# Worked values
# ---------------------------------------------------------------------------

def test_golden_pow2_weights():
    g = json.load(open(os.path.join(GOLDEN, "attention_pow2.json")))
    D, bs, Hq, Hkv, nb = g["head_dim"], g["block_size"], g["num_q_heads"], g["num_kv_heads"], g["num_blocks"]
    seq, qsl, bt = g["seq_lens"], g["query_start_loc"], np.array(g["block_tables"], np.int32)
    lk, lv = [], []
    for L in seq:
        K = np.zeros((L, Hkv, D), np.float32)
        V = np.zeros((L, Hkv, D), np.float32)
        for j in range(L):
            K[j, 0] = (j, 0, 0, 0)
            K[j, 1] = (0, 3 - j, 0, 0)
            V[j, 0] = (j, 1, -j, 2)
            V[j, 1] = (2 - j, 0, j * j, 1)
        lk.append(K)
        lv.append(V)
    kp, vp = _scatter(lk, lv, bt, nb, bs, g["unowned_fill"])
    Tq = qsl[-1]
    q = np.tile(np.array(g["q_heads"], np.float32)[None], (Tq, 1, 1))
    scale = float(np.float32(math.log(2.0)))
    out = oracle.paged_attention(_bits(q), _bits(kp), _bits(vp), bt,
                                 np.array(seq, np.int32), np.array(qsl, np.int32), scale)
    want = np.array([[[float(Fraction(x)) for x in row] for row in tok] for tok in g["expected"]])
    np.testing.assert_allclose(out, want, rtol=0, atol=g["tolerance"])


def test_golden_kv_bytes():
    g = json.load(open(os.path.join(GOLDEN, "kv_bytes.json")))
    for c in g["cases"]:
        got = oracle.kv_cache_bytes(c["layers"], c["kv_heads"], c["head_dim"],
                                    c["dtype_bytes"], c["seq_len"], c["batch"])
        assert got == c["bytes"], c["cite"]


# ---------------------------------------------------------------------------
# Dense check and relabelling invariance
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("bs,D", [(16, 128), (4, 8), (3, 5)])
def test_matches_dense_unpaged(seed, bs, D):
    rng = np.random.default_rng(1000 + seed)
    shape = wl.random_small_shape(rng, max_reqs=4, max_len=50, block_size=bs, head_dim=D)
    q, lk, lv, bt, kp, vp = _random_problem(rng, shape)
    scale = 1.0 / math.sqrt(D)
    got = _run_oracle(q, kp, vp, bt, shape, scale)
    want = _dense_reference(q, lk, lv, shape.seq_lens, shape.query_start_loc, scale,
                            shape.num_q_heads)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def test_tiny_decode_matches_dense():
    shape = wl.tiny_decode()
    rng = np.random.default_rng(7)
    q, lk, lv, bt, kp, vp = _random_problem(rng, shape)
    got = _run_oracle(q, kp, vp, bt, shape, 1 / math.sqrt(128))
    want = _dense_reference(q, lk, lv, shape.seq_lens, shape.query_start_loc,
                            1 / math.sqrt(128), shape.num_q_heads)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


@pytest.mark.parametrize("seed", range(4))
def test_block_relabelling_invariance(seed):
    rng = np.random.default_rng(2000 + seed)
    shape = wl.random_small_shape(rng, max_reqs=5, max_len=90)
    q, lk, lv, bt, kp, vp = _random_problem(rng, shape, fill=0.0)
    a = _run_oracle(q, kp, vp, bt, shape, 0.088)
    perm = rng.permutation(shape.num_blocks)            # new home of block b
    kp2, vp2 = np.empty_like(kp), np.empty_like(vp)
    kp2[perm], vp2[perm] = kp, vp
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
    b = _run_oracle(q, kp2, vp2, bt2, shape, 0.088)
    assert np.array_equal(a, b)


def test_unowned_slots_never_read():
    """NaN in free blocks and in the tails of last blocks must not leak."""
    rng = np.random.default_rng(5)
    shape = wl.StepShape("tails", [1, 15, 16, 17, 33], [1, 3, 1, 17, 2], 8, 2, num_blocks=12)
    q, lk, lv, bt, kp, vp = _random_problem(rng, shape, fill=np.nan)
    out = _run_oracle(q, kp, vp, bt, shape, 0.1)
    assert np.isfinite(out).all()
    unused = np.where(bt < 0, 10**6, bt)   # entries past the last block: garbage
    out2 = _run_oracle(q, kp, vp, unused.astype(np.int32), shape, 0.1)
    assert np.array_equal(out, out2)


# ---------------------------------------------------------------------------
# Closed forms and special cases
# ---------------------------------------------------------------------------

def test_constant_v_gives_that_constant():
    rng = np.random.default_rng(11)
    shape = wl.random_small_shape(rng, max_reqs=5, max_len=80)
    q, lk, lv, bt, kp, vp = _random_problem(rng, shape)
    const = np.array([0.5, -1.25, 3.0, 0.0] * (shape.head_dim // 4), np.float32)
    lv = [np.broadcast_to(const, V.shape).copy() for V in lv]
    kp, vp = _scatter(lk, lv, bt, shape.num_blocks, shape.block_size, np.nan)
    out = _run_oracle(q, kp, vp, bt, shape, 1 / math.sqrt(128))
    np.testing.assert_allclose(out, np.broadcast_to(const, out.shape), rtol=0, atol=1e-12)


def test_single_key_returns_v0():
    shape = wl.StepShape("one", [1, 1], [1, 1], 4, 2, num_blocks=4)
    rng = np.random.default_rng(3)
    q, lk, lv, bt, kp, vp = _random_problem(rng, shape)
    out = _run_oracle(q, kp, vp, bt, shape, 0.3)
    for r in range(2):
        np.testing.assert_array_equal(out[r], np.repeat(lv[r][0], 2, axis=0))


def test_first_prefill_query_returns_v0():
    """A chunk with no cached prefix: its first query sees only key 0."""
    shape = wl.StepShape("fresh", [40], [40], 6, 3)
    rng = np.random.default_rng(4)
    q, lk, lv, bt, kp, vp = _random_problem(rng, shape)
    out = _run_oracle(q, kp, vp, bt, shape, 0.3)
    np.testing.assert_array_equal(out[0], np.repeat(lv[0][0], 2, axis=0))


def test_equal_keys_give_mean_of_v():
    rng = np.random.default_rng(6)
    shape = wl.StepShape("eq", [37, 5], [1, 2], 4, 1)
    q, lk, lv, bt, kp, vp = _random_problem(rng, shape)
    lk = [np.broadcast_to(K[:1], K.shape).copy() for K in lk]
    kp, vp = _scatter(lk, lv, bt, shape.num_blocks, shape.block_size, np.nan)
    out = _run_oracle(q, kp, vp, bt, shape, 0.2)
    np.testing.assert_allclose(out[0], np.repeat(lv[0].astype(np.float64).mean(0), 4, 0),
                               rtol=0, atol=1e-12)
    # request 1: queries at positions 3 and 4 average keys 0..3 and 0..4
    np.testing.assert_allclose(out[1], np.repeat(lv[1][:4].astype(np.float64).mean(0), 4, 0),
                               rtol=0, atol=1e-12)
    np.testing.assert_allclose(out[2], np.repeat(lv[1].astype(np.float64).mean(0), 4, 0),
                               rtol=0, atol=1e-12)


def test_dominant_logit_selects_its_value_row():
    shape = wl.StepShape("dom", [50], [1], 2, 1)
    rng = np.random.default_rng(8)
    q, lk, lv, bt, kp, vp = _random_problem(rng, shape)
    D = shape.head_dim
    q[:] = 0
    q[0, :, 0] = 1.0
    K = np.zeros_like(lk[0])
    K[17, 0, 0] = 1.0                       # only key 17 scores above zero
    kp, vp = _scatter([K], lv, bt, shape.num_blocks, shape.block_size, np.nan)
    out = _run_oracle(q, kp, vp, bt, shape, 1000.0)
    np.testing.assert_allclose(out[0], np.repeat(lv[0][17].astype(np.float64), 2, 0),
                               rtol=0, atol=1e-300)
    assert D == 128


# ---------------------------------------------------------------------------
# Brute force on tiny integer inputs
# ---------------------------------------------------------------------------

def _brute_force(q, lk, lv, seq, qsl, scale, Hq):
    """Direct sums with math.fsum and math.exp: no max subtraction, no blocks."""
    out = np.zeros(q.shape, dtype=np.float64)
    for r in range(len(seq)):
        L = int(seq[r])
        Hkv = lk[r].shape[1]
        g = Hq // Hkv
        qn = int(qsl[r + 1] - qsl[r])
        for i in range(qn):
            t = int(qsl[r]) + i
            p = L - qn + i
            for h in range(Hq):
                kh = h // g
                w = [math.exp(scale * math.fsum(float(a) * float(b) for a, b in zip(q[t, h], lk[r][j, kh])))
                     for j in range(p + 1)]
                z = math.fsum(w)
                for d in range(q.shape[2]):
                    out[t, h, d] = math.fsum(wj * float(lv[r][j, kh, d]) for j, wj in enumerate(w)) / z
    return out


@pytest.mark.parametrize("seed", range(5))
def test_brute_force_small_integers(seed):
    rng = np.random.default_rng(3000 + seed)
    shape = wl.random_small_shape(rng, max_reqs=3, max_len=40, block_size=4,
                                  head_dim=int(rng.integers(4, 9)))
    q, lk, lv, bt, kp, vp = _random_problem(rng, shape, int_values=True)
    scale = 0.25
    got = _run_oracle(q, kp, vp, bt, shape, scale)
    want = _brute_force(q, lk, lv, shape.seq_lens, shape.query_start_loc, scale,
                        shape.num_q_heads)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# Chunked prefill equivalence and append
# ---------------------------------------------------------------------------

def test_two_chunks_equal_one_chunk():
    """A q-token chunk in one step equals q1 then q2 tokens in two steps with
    the cache appended in between (The Serving Playbook, "Chunked prefill")."""
    rng = np.random.default_rng(9)
    prefix, q1, q2 = 21, 13, 30
    L = prefix + q1 + q2
    one = wl.StepShape("one", [L], [q1 + q2], 8, 2, num_blocks=10)
    q, lk, lv, bt, kp, vp = _random_problem(rng, one)
    full = _run_oracle(q, kp, vp, bt, one, 0.09)
    # step A: only prefix + q1 tokens exist; the rest of the pool is junk
    Ka, Va = [lk[0][:prefix + q1]], [lv[0][:prefix + q1]]
    kpa, vpa = _scatter(Ka, Va, bt, one.num_blocks, one.block_size, np.nan)
    sa = wl.StepShape("a", [prefix + q1], [q1], 8, 2, num_blocks=10)
    outa = _run_oracle(q[:q1], kpa, vpa, bt, sa, 0.09)
    # step B: append the q2 new tokens through slots, then attend
    slots = np.array([bt[0, p // 16] * 16 + p % 16 for p in range(prefix + q1, L)], np.int64)
    kpb, vpb = oracle.append(_bits(lk[0][prefix + q1:]), _bits(lv[0][prefix + q1:]), slots,
                             _bits(kpa), _bits(vpa))
    sb = wl.StepShape("b", [L], [q2], 8, 2, num_blocks=10)
    outb = oracle.paged_attention(_bits(q[q1:]), kpb, vpb, bt, sb.seq_lens,
                                  sb.query_start_loc, 0.09)
    np.testing.assert_array_equal(np.concatenate([outa, outb]), full)


def test_append_matches_numpy_scatter_and_touches_nothing_else():
    rng = np.random.default_rng(12)
    nb, Hkv, bs, D, T = 9, 3, 16, 128, 40
    kp = rng.integers(0, 2**16, size=(nb, Hkv, bs, D), dtype=np.uint16)
    vp = rng.integers(0, 2**16, size=(nb, Hkv, bs, D), dtype=np.uint16)
    kn = rng.integers(0, 2**16, size=(T, Hkv, D), dtype=np.uint16)
    vn = rng.integers(0, 2**16, size=(T, Hkv, D), dtype=np.uint16)
    slots = rng.permutation(nb * bs)[:T].astype(np.int64)
    slots[[3, 17, 29]] = -1                              # padding tokens
    k2, v2 = oracle.append(kn, vn, slots, kp, vp)
    ek, ev = kp.copy(), vp.copy()
    for t, s in enumerate(slots):
        if s >= 0:
            ek[s // bs, :, s % bs, :] = kn[t]
            ev[s // bs, :, s % bs, :] = vn[t]
    assert np.array_equal(k2, ek) and np.array_equal(v2, ev)
    assert k2.tobytes() != kp.tobytes()


def test_append_rejects_slot_outside_pool():
    kn = np.zeros((1, 1, 8), np.uint16)
    pool = np.zeros((2, 1, 4, 8), np.uint16)
    with pytest.raises(ValueError):
        oracle.append(kn, kn, np.array([8], np.int64), pool, pool)


def test_rejects_inconsistent_lengths():
    q = np.zeros((3, 2, 8), np.uint16)
    pool = np.zeros((4, 1, 4, 8), np.uint16)
    bt = np.zeros((1, 4), np.int32)
    with pytest.raises(ValueError):   # q_r = 3 > L_r = 2
        oracle.paged_attention(q, pool, pool, bt, np.array([2], np.int32),
                               np.array([0, 3], np.int32), 1.0)
    with pytest.raises(ValueError):   # block id beyond the pool
        oracle.paged_attention(q, pool, pool, bt + 7, np.array([5], np.int32),
                               np.array([0, 3], np.int32), 1.0)


def test_copy_blocks_matches_numpy_and_touches_nothing_else():
    rng = np.random.default_rng(21)
    src = rng.integers(0, 2**16, size=(10, 3, 16, 8), dtype=np.uint16)
    vsrc = rng.integers(0, 2**16, size=(10, 3, 16, 8), dtype=np.uint16)
    dst = rng.integers(0, 2**16, size=(6, 3, 16, 8), dtype=np.uint16)
    vdst = rng.integers(0, 2**16, size=(6, 3, 16, 8), dtype=np.uint16)
    pairs = np.array([[7, 0], [2, 5], [9, 3]], np.int64)
    kd, vd = oracle.copy_blocks(src, vsrc, dst, vdst, pairs)
    ek, ev = dst.copy(), vdst.copy()
    ek[pairs[:, 1]] = src[pairs[:, 0]]
    ev[pairs[:, 1]] = vsrc[pairs[:, 0]]
    assert np.array_equal(kd, ek) and np.array_equal(vd, ev)
    with pytest.raises(ValueError):
        oracle.copy_blocks(src, vsrc, dst, vdst, np.array([[10, 0]], np.int64))


# ---------------------------------------------------------------------------
# FP8 (e4m3) KV: the codec against the format's definition, and fp8 attention
# against bf16-free dequantised attention
# ---------------------------------------------------------------------------

def test_e4m3_known_codes():
    assert oracle.e4m3_decode(0x38) == 1.0          # exponent 7 = bias, mantissa 0
    assert oracle.e4m3_decode(0xB8) == -1.0
    assert oracle.e4m3_decode(0x7E) == 448.0        # largest finite
    assert oracle.e4m3_decode(0x08) == 2.0 ** -6    # smallest normal
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9    # smallest subnormal
    assert oracle.e4m3_decode(0x07) == 7 * 2.0 ** -9
    assert oracle.e4m3_decode(0x3C) == 1.5
    assert math.isnan(oracle.e4m3_decode(0x7F)) and math.isnan(oracle.e4m3_decode(0xFF))


def test_e4m3_encode_inverts_decode_and_rounds_to_even():
    for c in range(256):
        v = oracle.e4m3_decode(c)
        if math.isnan(v):
            continue
        assert oracle.e4m3_encode(v) == c, hex(c)
    # midpoints go to the even code: 1.0 (0x38) .. 1.125 (0x39) -> 0x38;
    # 1.125 .. 1.25 (0x3A) -> 0x3A
    assert oracle.e4m3_encode(1.0625) == 0x38
    assert oracle.e4m3_encode(1.1875) == 0x3A
    assert oracle.e4m3_encode(1.07) == 0x39
    assert oracle.e4m3_encode(1000.0) == 0x7E and oracle.e4m3_encode(-1e30) == 0xFE  # saturate
    assert oracle.e4m3_encode(2.0 ** -11) == 0x00                                    # tie to 0
    assert oracle.e4m3_encode(-0.0) == 0x80


def test_fp8_attention_equals_attention_on_dequantised_values():
    """Dequantised fp8 pools, fed to the (pinned) fp64 attention as exact
    values, give the same answer as the fp8 path."""
    rng = np.random.default_rng(77)
    shape = wl.random_small_shape(rng, max_reqs=4, max_len=60, Hq=8, Hkv=2)
    nb, Hkv, bs, D = shape.num_blocks, 2, shape.block_size, shape.head_dim
    k8 = rng.integers(0, 256, size=(nb, Hkv, bs, D), dtype=np.uint8)
    v8 = rng.integers(0, 256, size=(nb, Hkv, bs, D), dtype=np.uint8)
    k8[(k8 & 0x7F) == 0x7F] = 0x30                        # no NaN codes
    v8[(v8 & 0x7F) == 0x7F] = 0x30
    ks = np.array([0.05, 0.02], np.float32)
    vs = np.array([0.01, 0.04], np.float32)
    q = _bits(rng.standard_normal((shape.num_q_tokens, 8, D)).astype(np.float32))
    bt = wl.block_placement(shape, 5)
    got = oracle.paged_attention_fp8(q, k8, v8, ks, vs, bt, shape.seq_lens,
                                     shape.query_start_loc, 0.09)
    lut = np.array([oracle.e4m3_decode(c) for c in range(256)])
    kd = lut[k8] * ks.astype(np.float64)[None, :, None, None]
    vd = lut[v8] * vs.astype(np.float64)[None, :, None, None]
    lk = [np.stack([kd[bt[r, j // bs], :, j % bs] for j in range(L)]) for r, L in enumerate(shape.seq_lens)]
    lv = [np.stack([vd[bt[r, j // bs], :, j % bs] for j in range(L)]) for r, L in enumerate(shape.seq_lens)]
    want = _dense_reference(_vals(q), lk, lv, shape.seq_lens, shape.query_start_loc, 0.09, 8)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def test_fp8_append_codes():
    rng = np.random.default_rng(78)
    kn = _bits(rng.standard_normal((5, 2, 8)).astype(np.float32) * 3)
    vn = _bits(rng.standard_normal((5, 2, 8)).astype(np.float32))
    ks, vs = np.array([0.5, 0.01], np.float32), np.array([2.0, 0.125], np.float32)
    pool = np.zeros((4, 2, 4, 8), np.uint8)
    slots = np.array([0, 5, -1, 14, 9], np.int64)
    kp, vp = oracle.append_fp8(kn, vn, slots, pool, pool, ks, vs)
    kv, vv = _vals(kn).astype(np.float32), _vals(vn).astype(np.float32)
    for t, s in enumerate(slots):
        if s < 0:
            continue
        for h in range(2):
            for d in range(8):
                assert kp[s // 4, h, s % 4, d] == oracle.e4m3_encode(np.float32(kv[t, h, d]) / ks[h])
                assert vp[s // 4, h, s % 4, d] == oracle.e4m3_encode(np.float32(vv[t, h, d]) / vs[h])
    assert kp[0, :, 2].sum() == 0    # untouched slots stay zero


def test_e4m3_encode_matches_torch_in_range():
    """Within +-448 the encoder agrees with torch's float8_e4m3fn cast (an
    independent round-to-nearest-even implementation)."""
    rng = np.random.default_rng(79)
    x = np.concatenate([rng.standard_normal(4000).astype(np.float32) * 50,
                        np.linspace(-448, 448, 2001, dtype=np.float32),
                        (np.arange(256) * 2.0 ** -12).astype(np.float32)])
    t = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    o = np.array([oracle.e4m3_encode(v) for v in x], np.uint8)
    assert np.array_equal(t, o)


def test_shared_prefix_tables_equal_private_copies():
    """Requests whose tables share physical prefix blocks (one copy of a
    common prompt) get exactly the attention of tables pointing at private
    copies of those blocks: the oracle follows each table, so a shared-prefix
    (cascade) call has the plain definition as its reference."""
    shape = wl.StepShape("shared_pin", [40, 37, 52, 20], [1, 2, 1, 1], 8, 2, head_dim=16,
                         seed=31, prefix_groups=((0, 3, 2),))
    inp = wl.make_step(shape)
    bt = inp.block_tables.numpy().copy()
    k, v = wl.bf16_bits(inp.k_pool), wl.bf16_bits(inp.v_pool)
    assert (bt[1, :2] == bt[0, :2]).all() and (bt[2, :2] == bt[0, :2]).all()
    q = wl.bf16_bits(inp.q)
    sl, qsl = inp.seq_lens.numpy(), inp.query_start_loc.numpy()
    shared = oracle.paged_attention(q, k, v, bt, sl, qsl, inp.scale)
    # give requests 1 and 2 private copies of the two prefix blocks
    nb = k.shape[0]
    extra = [bt[0, 0], bt[0, 1], bt[0, 0], bt[0, 1]]
    k2 = np.concatenate([k, k[extra]])
    v2 = np.concatenate([v, v[extra]])
    bt2 = bt.copy()
    bt2[1, :2] = [nb, nb + 1]
    bt2[2, :2] = [nb + 2, nb + 3]
    private = oracle.paged_attention(q, k2, v2, bt2, sl, qsl, inp.scale)
    assert np.array_equal(shared, private)
