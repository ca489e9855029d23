"""Helpers shared by the GPU parity tests: run the CUDA path, run the oracle
on the same inputs (or on a relabelled sub-problem for sampled rows), compare.

Tolerances for attention outputs (bf16 inputs, fp32 accumulation, bf16
output): max |gpu - oracle| <= 1e-2 and mean |gpu - oracle| <= 1e-3, both in
fp64.  Append is compared bit for bit.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import paged_kv_cache_195_gb300 as pkv
from paged_kv_cache_195_gb300 import workloads as wl

MAX_ABS = 1e-2
MEAN_ABS = 1e-3


def gpu_step(inp: wl.StepInputs, append: bool = True, workspace=None):
    """Append (optional) then attention on the GPU; returns out (bf16, device)."""
    if append:
        pkv.pkv_append(inp.k_new, inp.v_new, inp.slot_mapping, inp.k_pool, inp.v_pool)
    out = pkv.pkv_attention(inp.q, inp.k_pool, inp.v_pool, inp.block_tables, inp.seq_lens,
                            inp.query_start_loc, inp.scale, workspace=workspace)
    return out


def oracle_pools_after_append(inp_host: dict):
    """Oracle append applied to the pre-append host pools."""
    return oracle.append(inp_host["k_new"], inp_host["v_new"], inp_host["slot_mapping"],
                         inp_host["k_pool"], inp_host["v_pool"])


def host_copy(inp: wl.StepInputs) -> dict:
    """Host (numpy) copies of every input, bf16 as uint16 bit patterns."""
    return dict(
        q=wl.bf16_bits(inp.q), k_new=wl.bf16_bits(inp.k_new), v_new=wl.bf16_bits(inp.v_new),
        slot_mapping=inp.slot_mapping.cpu().numpy(), k_pool=wl.bf16_bits(inp.k_pool),
        v_pool=wl.bf16_bits(inp.v_pool), block_tables=inp.block_tables.cpu().numpy(),
        seq_lens=inp.seq_lens.cpu().numpy(), qsl=inp.query_start_loc.cpu().numpy(),
        scale=inp.scale)


def oracle_full(h: dict, k_pool=None, v_pool=None) -> np.ndarray:
    kp = h["k_pool"] if k_pool is None else k_pool
    vp = h["v_pool"] if v_pool is None else v_pool
    return oracle.paged_attention(h["q"], kp, vp, h["block_tables"], h["seq_lens"], h["qsl"],
                                  h["scale"])


def to_f64(out: torch.Tensor) -> np.ndarray:
    return out.detach().float().cpu().numpy().astype(np.float64)


def assert_close(got: np.ndarray, want: np.ndarray, what: str = ""):
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite GPU output"
    err = np.abs(got - want)
    mx, mean = float(err.max(initial=0.0)), float(err.mean()) if err.size else 0.0
    assert mx <= MAX_ABS and mean <= MEAN_ABS, f"{what}: max abs {mx:.3e}, mean abs {mean:.3e}"
    return mx, mean


def pool_host(t: torch.Tensor) -> np.ndarray:
    """Host copy of a pool: bf16 bit patterns (uint16) or e4m3 codes (uint8)."""
    return wl.bf16_bits(t) if t.dtype == torch.bfloat16 else t.detach().contiguous().cpu().numpy()


def snapshot_rows(inp, rows: list[tuple[int, int]]) -> dict:
    """Host copy of everything the oracle needs for sampled (request, query
    index) rows, taken BEFORE the GPU step runs: the rows' q, the pool blocks
    they read (pre-append contents) and this step's new K/V with their slots.

    Row i of request r (q_r queries, length L) is the single query of a
    request of length L - q_r + i + 1 with the same table; only the blocks
    those rows read are copied, gathered into a compact pool (physical
    placement does not change the result)."""
    bs = inp.shape.block_size
    qsl = inp.query_start_loc.cpu().numpy()
    sl = inp.seq_lens.cpu().numpy()
    bt = inp.block_tables.cpu().numpy()
    lens, phys_lists, qrows = [], [], []
    for r, i in rows:
        qr = int(qsl[r + 1] - qsl[r])
        Lp = int(sl[r]) - qr + i + 1
        lens.append(Lp)
        phys_lists.append(bt[r, :(Lp + bs - 1) // bs])
        qrows.append(int(qsl[r]) + i)
    uniq = np.unique(np.concatenate(phys_lists)).astype(np.int64)
    remap = {int(b): n for n, b in enumerate(uniq)}
    idx = torch.from_numpy(uniq).to(inp.k_pool.device)
    maxb = max(len(p) for p in phys_lists)
    sub_bt = np.full((len(rows), maxb), -1, np.int32)
    for n, pl in enumerate(phys_lists):
        sub_bt[n, :len(pl)] = [remap[int(b)] for b in pl]
    slots = inp.slot_mapping.cpu().numpy()
    sub_slots = np.array([remap[int(s) // bs] * bs + int(s) % bs
                          if s >= 0 and int(s) // bs in remap else -1 for s in slots], np.int64)
    snap = dict(qrows=qrows, lens=np.array(lens, np.int32), bt=sub_bt,
                q=wl.bf16_bits(inp.q[torch.tensor(qrows, device=inp.q.device)]),
                k_pool=pool_host(inp.k_pool.index_select(0, idx)),
                v_pool=pool_host(inp.v_pool.index_select(0, idx)),
                k_new=wl.bf16_bits(inp.k_new), v_new=wl.bf16_bits(inp.v_new),
                slots=sub_slots, scale=inp.scale)
    if hasattr(inp, "k_scale"):  # e4m3 pools
        snap["k_scale"] = inp.k_scale.cpu().numpy()
        snap["v_scale"] = inp.v_scale.cpu().numpy()
    return snap


def snapshot_oracle(snap: dict, appended: bool = True):
    """Oracle outputs (fp64) of the snapshotted rows, after the oracle's own
    append of this step's new K/V when the GPU step appended too."""
    kp, vp = snap["k_pool"], snap["v_pool"]
    n = len(snap["qrows"])
    qsl = np.arange(n + 1, dtype=np.int32)
    if "k_scale" in snap:
        ks, vs = snap["k_scale"], snap["v_scale"]
        if appended:
            kp, vp = oracle.append_fp8(snap["k_new"], snap["v_new"], snap["slots"], kp, vp, ks, vs)
        return oracle.paged_attention_fp8(snap["q"], kp, vp, ks, vs, snap["bt"], snap["lens"],
                                          qsl, snap["scale"])
    if appended:
        kp, vp = oracle.append(snap["k_new"], snap["v_new"], snap["slots"], kp, vp)
    return oracle.paged_attention(snap["q"], kp, vp, snap["bt"], snap["lens"], qsl,
                                  snap["scale"])
