#!/usr/bin/env python3
"""Benchmark of the paged-attention engine step on GB300.

A step is one pass of the whole hot path over one batch: for each of the 28
layers of a Qwen2.5-1.5B-shaped decode step (64 requests, context 512, Hq=12,
Hkv=2, D=128, 16-token blocks, each layer its own 1.25x pool with shuffled
blocks), append this step's K/V through the slot mapping, then run paged
attention.  The 56 launches are captured once in a CUDA graph and replayed.

Prints one JSON line (rank 0).  ``value`` is algorithmic HBM bytes (KV read +
q read + out write + append traffic) per second over all ranks; the pools of
one step (1.2 GB) exceed L2, so every step streams from HBM.  ``roofline``
times the step's attention launches back to back for about a second
(``--roofline-s``).  ``configs`` adds the same measurements for the other
single-layer workloads (the long batch, the mixed continuous-batching step,
the long-context step, and e4m3 caches), unless ``--no-extra``.

``--impl reference`` times the fp64 CPU oracle on bounded samples of the same
workload on the host cores instead (the reference arm).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from paged_kv_cache_195_gb300 import roofline as rl  # noqa: E402
from paged_kv_cache_195_gb300 import workloads as wl  # noqa: E402

METRIC = "paged-attention step: KV GB/s and % of GB300 HBM peak; attended tokens/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
DECODE_SRCS = [os.path.join(ROOT, "paged_kv_cache_195_gb300", "csrc", f)
               for f in ("pkv_decode_kernel.cuh", "pkv_decode.cu", "pkv_decode_tc.cu",
                         "pkv_plan.cuh")]


def decode_kernel_name(group: int, fp8: bool, opts: dict) -> str:
    """The decode kernel the library routes this step to under the options
    `opts` (4 or more query heads per KV head run on the tensor cores, e4m3
    pools widened to f16 there)."""
    tc = group >= 4 and opts["decode_tc"] != 0 and (not fp8 or opts["decode_tc_fp8"] != 0)
    if tc:
        return f"pkv::decode_tc_kernel<{group}, {'true' if fp8 else 'false'}>"
    return f"pkv::decode_kernel<{group}, {'KvE4m3' if fp8 else 'KvBf16'}>"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def measured_tensor_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def decode_source_sha(paths=None) -> str:
    """Hash of the kernels' code (the decode sources unless `paths` names
    others): the sources with // comments and blank lines removed, so that
    edits to comments keep a profile valid."""
    h = hashlib.sha256()
    for path in (DECODE_SRCS if paths is None else paths):
        with open(path, encoding="utf-8") as f:
            for line in f:
                code = re.sub(r"//.*", "", line).rstrip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def committed_traffic(config: str, kv: str):
    """Per-launch DRAM bytes of the attention call from the committed ncu
    summary of this workload (decode_<config>_<kv>.md for a call that runs
    the decode kernel alone, attention_<config>_<kv>.md for one that also
    runs the prefill kernel), if it was taken on the current sources of the
    kernels it names (its kernel_sources line; the decode sources if it has
    none), else None."""
    text = None
    for stem in ("decode", "attention"):
        try:
            text = open(os.path.join(ROOT, "profiles", f"{stem}_{config}_{kv}.md")).read()
            break
        except OSError:
            continue
    if text is None:
        return None
    m_src = re.search(r"kernel_sources:[ \t]*(\S.*)", text)
    paths = None
    if m_src:
        csrc = os.path.join(ROOT, "paged_kv_cache_195_gb300", "csrc")
        paths = [os.path.join(csrc, f) for f in m_src.group(1).split()]
    try:
        src_sha = decode_source_sha(paths)
    except OSError:
        return None
    m_sha = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    m_tr = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", text)
    if m_sha and m_tr and m_sha.group(1) == src_sha:
        return int(m_tr.group(1))
    return None


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------

def nvsmi_id(local_rank: int) -> str:
    """nvidia-smi --id for this process's GPU (honours CUDA_VISIBLE_DEVICES)."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "").strip()
    if vis:
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if local_rank < len(ids):
            return ids[local_rank]
    return str(local_rank)


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r.split(",") for r in self.file.read().strip().splitlines() if r.strip()]
        os.unlink(self.file.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
                for name, v in zip(names, r[5:9]):
                    if v.strip().lower() == "active":
                        reasons.add(name)
            except (ValueError, IndexError):
                continue
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# raw CUDA events recorded as graph nodes (cudaEventRecordExternal)
# ---------------------------------------------------------------------------

class GraphEvents:
    def __init__(self, n):
        self.rt = ctypes.CDLL("libcudart.so.13")
        self.rt.cudaEventCreate.argtypes = [ctypes.POINTER(ctypes.c_void_p)]
        self.rt.cudaEventRecordWithFlags.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint]
        self.rt.cudaEventElapsedTime.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.c_void_p,
                                                 ctypes.c_void_p]
        self.ev = []
        for _ in range(n):
            e = ctypes.c_void_p()
            assert self.rt.cudaEventCreate(ctypes.byref(e)) == 0
            self.ev.append(e)

    def record(self, i, stream):
        assert self.rt.cudaEventRecordWithFlags(self.ev[i], ctypes.c_void_p(stream.cuda_stream), 1) == 0

    def elapsed_ms(self, a, b):
        ms = ctypes.c_float()
        assert self.rt.cudaEventElapsedTime(ctypes.byref(ms), self.ev[a], self.ev[b]) == 0
        return ms.value


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

# Workloads timed after the headline one, each a single-layer call (attention
# over shuffled pools, plus the append that feeds it): the long batch, the
# mixed continuous-batching step, the long-context step, and the e4m3 cache on
# the two Qwen-shaped decodes.
EXTRA_CONFIGS = (("qwen_long", "bf16"), ("llama_mixed", "bf16"), ("llama_decode", "bf16"),
                 ("llama_long", "bf16"),
                 ("qwen_decode", "fp8"), ("qwen_long", "fp8"))


def lengths_summary(values) -> dict | int:
    """One number for uniform lengths, else their spread."""
    v = np.asarray(values, np.int64)
    if v.size and (v == v[0]).all():
        return int(v[0])
    return {"min": int(v.min()), "median": float(np.median(v)), "max": int(v.max()),
            "sum": int(v.sum())}


def workload_config(shape, ws_n, kv="bf16"):
    """The `config` object of the JSON line (both arms)."""
    kvb = 1 if kv == "fp8" else 2
    return {
        "workload": f"{shape.name} x{shape.layers} layers",
        "num_reqs": shape.num_reqs, "context": lengths_summary(shape.seq_lens),
        "q_tokens_per_req": lengths_summary(shape.q_lens), "layers": shape.layers,
        "num_q_heads": shape.num_q_heads, "num_kv_heads": shape.num_kv_heads,
        "head_dim": shape.head_dim, "block_size": shape.block_size,
        "pool_blocks_per_layer": shape.num_blocks, "parallelism": f"replicas x{ws_n}",
        "kv_cache_dtype": "e4m3 (per-KV-head scales)" if kv == "fp8" else "bf16",
        "l2": f"inputs exceed L2: {shape.layers} distinct pools, "
              f"{2 * shape.layers * shape.num_blocks * shape.num_kv_heads * 2048 * kvb / 1e9:.2f}"
              " GB per step",
        "launch": f"CUDA graph of {shape.layers} x (append + attention)"
                  + ("" if shape.prefix_groups else
                     f", {'pkv_append_attention_fp8' if kv == 'fp8' else 'pkv_append_attention'}"
                     " with early_trigger"),
        **({"shared_prefix": [{"first_request": int(f), "members": int(m), "blocks": int(b)}
                              for f, m, b in shape.prefix_groups],
            "attention_call": "pkv_attention_cascade"} if shape.prefix_groups else {}),
    }


def aggregate_over_ranks(ms_local: float, units_local: float, device=None):
    """Max of the timed region and sum of the work over all ranks (identity
    without an initialised process group)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms_local, units_local
    t = torch.tensor([ms_local], dtype=torch.float64, device=device)
    u = torch.tensor([units_local], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def build_layers(shape, device, rank, kv="bf16", count=None):
    make = wl.make_fp8_step if kv == "fp8" else wl.make_step
    n = shape.layers if count is None else count
    return [make(shape, device=device, layer=layer + 1000 * rank) for layer in range(n)]


def percentile(xs, q):
    return float(np.percentile(np.asarray(xs, np.float64), q))


class ConfigRun:
    """One workload on this GPU: its layers' inputs, a workspace, and three
    CUDA graphs -- the step (every layer's append + attention), the roofline
    pass (attention launches back to back between two event nodes) and, for
    the headline, the end-to-end step through pinned host buffers."""

    def __init__(self, pkv, shape, kv, device, rank, with_e2e):
        self.pkv, self.shape, self.kv, self.device = pkv, shape, kv, device
        # The step's pkv_append_attention calls let the attention launch as
        # soon as the append starts (its documented precondition holds: the
        # kernel before each call is the previous layer's attention, which
        # writes neither the tables, the lengths nor this layer's pool).
        pkv.set_options(early_trigger=1)
        self.fp8 = kv == "fp8"
        self.kvb = 1 if self.fp8 else 2
        # single-layer workloads: two copies of the layer alternate in the
        # roofline pass, so consecutive launches never share data in L2
        n_pools = shape.layers if shape.layers > 1 else 2
        self.layers = build_layers(shape, device, rank, kv, count=n_pools)
        self.step_layers = self.layers[:shape.layers]
        self.roof_seq = list(range(shape.layers)) if shape.layers > 1 else [0, 1] * 4
        L0 = self.layers[0]
        dims = pkv.make_dims(tuple(L0.q.shape), tuple(L0.k_pool.shape), shape.num_reqs,
                             shape.max_blocks_per_req)
        self.cascade = bool(shape.prefix_groups) and not self.fp8
        self.ws = (pkv.CascadeWorkspace if self.cascade else pkv.Workspace)(dims, device=device)
        pkv.pkv_workspace_init(self.ws, dims)
        if self.cascade:
            grp = np.array(shape.prefix_groups, dtype=np.int32).reshape(-1, 3)
            self.grp_t = [torch.from_numpy(np.ascontiguousarray(grp[:, i])).to(device)
                          for i in range(3)]
        self.outs = [torch.empty_like(x.q) for x in self.layers]
        if with_e2e:
            self._stage()
        self.stream = torch.cuda.Stream(device)
        self.gev = GraphEvents(2)
        with torch.cuda.stream(self.stream):
            self.step()  # eager warm-up (module load, attribute set-up)
        torch.cuda.synchronize(device)
        assert pkv.pkv_get_device_error() == 0, pkv.pkv_last_error()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=self.stream):
            self.step()
        self.graph_roof = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph_roof, stream=self.stream):
            self.attention_only()
        self.graph_e2e = None
        if with_e2e:
            self._capture_e2e()

    def attention(self, li):
        pkv, x, out, ws = self.pkv, self.layers[li], self.outs[li], self.ws
        if self.fp8:
            pkv.pkv_attention_fp8kv(x.q, x.k_pool, x.v_pool, x.k_scale, x.v_scale,
                                    x.block_tables, x.seq_lens, x.query_start_loc, x.scale,
                                    out=out, workspace=ws)
        elif self.cascade:
            pkv.pkv_attention_cascade(x.q, x.k_pool, x.v_pool, x.block_tables, x.seq_lens,
                                      x.query_start_loc, *self.grp_t, x.scale, out=out,
                                      workspace=ws)
        else:
            pkv.pkv_attention(x.q, x.k_pool, x.v_pool, x.block_tables, x.seq_lens,
                              x.query_start_loc, x.scale, out=out, workspace=ws)

    def step(self):
        for li in range(len(self.step_layers)):
            self.layer_step(li)

    def layer_step(self, li):
        pkv, x = self.pkv, self.step_layers[li]
        if self.fp8:
            pkv.pkv_append_attention_fp8(x.k_new, x.v_new, x.slot_mapping, x.k_pool,
                                         x.v_pool, x.k_scale, x.v_scale, x.q,
                                         x.block_tables, x.seq_lens, x.query_start_loc,
                                         x.scale, out=self.outs[li], workspace=self.ws)
        elif self.cascade:
            pkv.pkv_append(x.k_new, x.v_new, x.slot_mapping, x.k_pool, x.v_pool)
            self.attention(li)
        else:
            # one layer: the append, then the attention, which streams the
            # tiles without this step's tokens while the append runs
            pkv.pkv_append_attention(x.k_new, x.v_new, x.slot_mapping, x.k_pool, x.v_pool,
                                     x.q, x.block_tables, x.seq_lens, x.query_start_loc,
                                     x.scale, out=self.outs[li], workspace=self.ws)

    def attention_only(self):
        # the attention launches back to back (the pools already hold the
        # step's tokens), bracketed by two event nodes; nothing between the
        # launches, so they overlap as in the step
        s = torch.cuda.current_stream(self.device)
        self.gev.record(0, s)
        for li in self.roof_seq:
            self.attention(li)
        self.gev.record(1, s)

    STEP_INPUTS = ("q", "k_new", "v_new", "slot_mapping", "block_tables", "seq_lens",
                   "query_start_loc")

    def _stage(self):
        """The step's buffers as an engine keeps them: every layer's step
        inputs are views into one device buffer and every layer's output into
        another (each view 256-byte aligned), with pinned host twins, so that
        the end-to-end step moves its inputs in with a few large copies and
        each layer's output out with one."""
        def aligned(n):
            return (n + 255) & ~255

        def restage(tensors):
            total = sum(aligned(t.numel() * t.element_size()) for t in tensors)
            buf = torch.empty(total, dtype=torch.uint8, device=self.device)
            views, ends, off = [], [], 0
            for t in tensors:
                nb = t.numel() * t.element_size()
                v = buf[off:off + nb].view(t.dtype).view(t.shape)
                v.copy_(t)
                views.append(v)
                off += aligned(nb)
                ends.append(off)
            return buf, views, ends

        pairs = [(x, k) for x in self.step_layers for k in self.STEP_INPUTS]
        self.dev_in, views, ends = restage([getattr(x, k) for x, k in pairs])
        m = len(self.STEP_INPUTS)
        self.in_ends = [ends[(i + 1) * m - 1] for i in range(len(self.step_layers))]
        for (x, k), v in zip(pairs, views):
            setattr(x, k, v)
        n = len(self.step_layers)
        # byte range of each layer's output in the output buffer
        self.dev_out, self.outs[:n], oends = restage(self.outs[:n])
        self.out_regions = [(oends[i - 1] if i else 0, oends[i]) for i in range(n)]
        self.host_in = torch.empty(self.dev_in.numel(), dtype=torch.uint8, pin_memory=True)
        self.host_in.copy_(self.dev_in)
        self.host_out = torch.empty(self.dev_out.numel(), dtype=torch.uint8, pin_memory=True)

    def _capture_e2e(self):
        # Pinned host inputs -> device in a few growing chunks of layers on a
        # copy stream (the step waits for a chunk only before its first
        # layer, so the later chunks' copies overlap the earlier layers);
        # outputs -> pinned host on a second copy stream, in four chunks of
        # layers, each copied as soon as its last layer has written it.  The
        # byte counts are the copies'.
        self.h2d = self.host_in.numel()
        self.d2h = self.host_out.numel()
        s_in, s_out = torch.cuda.Stream(self.device), torch.cuda.Stream(self.device)
        n = len(self.step_layers)
        firsts = sorted({0} | {f for f in (1, 4, 11) if f < n})  # input chunk starts
        chunks = [(a, (firsts + [n])[c + 1]) for c, a in enumerate(firsts)]
        lasts = sorted({n - 1} | {f for f in (6, 13, 20) if f < n - 1})  # output chunk ends
        ev_in = {a: torch.cuda.Event() for a, _ in chunks}
        ev_out = {li: torch.cuda.Event() for li in lasts}
        self.graph_e2e = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph_e2e, stream=self.stream):
            s_in.wait_stream(self.stream)
            s_out.wait_stream(self.stream)
            with torch.cuda.stream(s_in):
                for a, b in chunks:
                    lo = self.in_ends[a - 1] if a else 0
                    hi = self.in_ends[b - 1]
                    self.dev_in[lo:hi].copy_(self.host_in[lo:hi], non_blocking=True)
                    ev_in[a].record(s_in)
            first_out = 0
            for li in range(n):
                if li in ev_in:
                    self.stream.wait_event(ev_in[li])
                self.layer_step(li)
                if li in ev_out:
                    ev_out[li].record(self.stream)
                    s_out.wait_event(ev_out[li])
                    a, b = self.out_regions[first_out][0], self.out_regions[li][1]
                    with torch.cuda.stream(s_out):
                        self.host_out[a:b].copy_(self.dev_out[a:b], non_blocking=True)
                    first_out = li + 1
            self.stream.wait_stream(s_in)
            self.stream.wait_stream(s_out)

    def timed(self, g, k, warmup, barrier=lambda: None):
        for _ in range(warmup):
            g.replay()
        torch.cuda.synchronize(self.device)
        barrier()
        torch.cuda.synchronize(self.device)
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(self.stream)
        with torch.cuda.stream(self.stream):
            for _ in range(k):
                g.replay()
        t1.record(self.stream)
        torch.cuda.synchronize(self.device)
        barrier()
        return t0.elapsed_time(t1)

    def roofline_pass(self, warmup, min_s, clocks=None):
        """Replays the back-to-back attention graph for at least min_s
        seconds; per replay, the bracketed time over its launches."""
        durs = []
        with torch.cuda.stream(self.stream):
            for _ in range(warmup):
                self.graph_roof.replay()
            torch.cuda.synchronize(self.device)
            if clocks:
                clocks.start()
            t_end = time.perf_counter() + min_s
            while len(durs) < 3 or (time.perf_counter() < t_end and len(durs) < 20000):
                self.graph_roof.replay()
                self.stream.synchronize()
                durs.append(self.gev.elapsed_ms(0, 1) / len(self.roof_seq))
        clock_info = clocks.stop() if clocks else None
        return durs, clock_info

    def unique_bytes(self):
        shape = self.shape
        att = rl.attention_bytes(shape.seq_lens, shape.q_lens, shape.num_q_heads,
                                 shape.num_kv_heads, kv_dtype_bytes=self.kvb)
        # The roofline counts the bytes the kernels must read: with shared
        # prefixes, each group's prefix once.
        if shape.prefix_groups and self.cascade:
            return rl.unique_kv_bytes(shape.seq_lens, shape.q_lens, shape.num_kv_heads,
                                      shape.prefix_groups, kv_dtype_bytes=self.kvb) + att["q_out"]
        return att["total"]

    def has_prefill(self):
        """Whether the library's routing sends part of this step to the
        tensor-core prefill kernel (bf16 pools, a request with at least
        prefill_min_q query tokens possible)."""
        shape = self.shape
        min_q = self.pkv.get_options()["prefill_min_q"]
        return (not self.fp8 and not self.cascade and min_q >= 1 and
                shape.num_q_tokens - shape.num_reqs + 1 >= min_q)

    def kernels_per_layer(self):
        return 2 + (1 if self.has_prefill() else 0) + (2 if self.cascade else 0)

    def kernel_label(self):
        """The kernels one attention call runs on this step."""
        group = self.shape.num_q_heads // self.shape.num_kv_heads
        name = decode_kernel_name(group, self.fp8, self.pkv.get_options())
        if self.has_prefill():
            name += f" + pkv::prefill_kernel<{group}>"
        return name

    def roofline(self, durs_ms, config_name, clock_info):
        peak, peak_src = measured_peak()
        unique = self.unique_bytes()
        mean_ms = statistics.mean(durs_ms)
        achieved = unique / (mean_ms * 1e-3) / 1e9
        shape = self.shape
        return {
            "bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "traffic": committed_traffic(config_name, self.kv),
            "kernel": self.kernel_label(),
            "timing": (f"{len(self.roof_seq)} attention launches back to back "
                       f"({'distinct layers' if shape.layers > 1 else 'two copies alternating'})"
                       f", one event pair per replay, {len(durs_ms)} replays"),
            "algorithmic_bytes_per_launch": unique,
            "avg_launch_us": round(mean_ms * 1e3, 3),
            "p10_us": round(percentile(durs_ms, 10) * 1e3, 3),
            "p50_us": round(percentile(durs_ms, 50) * 1e3, 3),
            "p90_us": round(percentile(durs_ms, 90) * 1e3, 3),
            "peak_source": peak_src,
            "frac_of_nominal_8tbs": round(achieved / NOMINAL_HBM_GBS, 4),
            "clocks": clock_info,
        }


def measure_extra(pkv, config, kv, device, rank, args, local):
    """A single-layer workload: the per-layer step time and the roofline of
    its attention launches."""
    shape = wl.CONFIGS[config]()
    run = ConfigRun(pkv, shape, kv, device, rank, with_e2e=False)
    ms = run.timed(run.graph, max(3, args.steps), args.warmup) / max(3, args.steps)
    durs, clk = run.roofline_pass(args.warmup, args.roofline_s, ClockSampler(nvsmi_id(local)))
    assert pkv.pkv_get_device_error() == 0, pkv.pkv_last_error()
    att = rl.attention_bytes(shape.seq_lens, shape.q_lens, shape.num_q_heads,
                             shape.num_kv_heads, kv_dtype_bytes=run.kvb)
    app = rl.append_bytes(shape.num_q_tokens, shape.num_kv_heads, kv_dtype_bytes=run.kvb)
    rec = {
        "workload": f"{shape.name}", "kv_cache_dtype": workload_config(shape, 1, kv)["kv_cache_dtype"],
        "num_reqs": shape.num_reqs, "context": lengths_summary(shape.seq_lens),
        "q_tokens_per_req": lengths_summary(shape.q_lens),
        "us_per_layer": round(ms * 1e3 / shape.layers, 3),
        "step_gb_per_s": round((att["total"] + app) * shape.layers / (ms * 1e-3) / 1e9, 1),
        "attended_tokens_per_s": round(rl.attended_tokens(shape.seq_lens, shape.q_lens)
                                       * shape.layers / (ms * 1e-3), 1),
        "roofline": run.roofline(durs, config, clk),
    }
    flops = rl.attention_flops(shape.seq_lens, shape.q_lens, shape.num_q_heads)
    if shape.num_q_tokens > shape.num_reqs:
        rec["attention_tflops_per_layer_call"] = round(flops / 1e12, 4)
    troof = tensor_roofline(shape, durs)
    if troof is not None:
        rec["tensor_roofline"] = troof
    del run
    torch.cuda.empty_cache()
    return rec


def tensor_roofline(shape, durs):
    """The tensor-core roofline of a step whose every request is a prefill
    chunk (a contraction timed alone takes the burst bf16 peak); None for a
    step with decode requests, which HBM bounds."""
    if int((shape.q_lens > 1).sum()) != shape.num_reqs:
        return None
    flops = rl.attention_flops(shape.seq_lens, shape.q_lens, shape.num_q_heads)
    tpk, tsrc = measured_tensor_peak()
    ach = flops / (statistics.mean(durs) * 1e-3) / 1e12
    return {"bound": "tensor", "achieved": round(ach, 1), "peak": tpk, "unit": "TFLOP/s",
            "frac": round(ach / tpk, 4), "peak_source": tsrc, "flops_per_launch": flops}


def run_ours(args):
    import paged_kv_cache_195_gb300 as pkv
    from paged_kv_cache_195_gb300 import build as pkv_build

    ws_n, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if ws_n > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    if rank == 0 or ws_n == 1:
        pkv_build.build()
    if ws_n > 1:
        torch.distributed.barrier()
        pkv_build.build()
    pkv.load_library()

    def barrier():
        if ws_n > 1:
            torch.distributed.barrier()

    shape = wl.CONFIGS[args.config]()
    run = ConfigRun(pkv, shape, args.kv, device, rank, with_e2e=True)
    fp8 = run.fp8
    att = rl.attention_bytes(shape.seq_lens, shape.q_lens, shape.num_q_heads, shape.num_kv_heads,
                             kv_dtype_bytes=run.kvb)
    app = rl.append_bytes(shape.num_q_tokens, shape.num_kv_heads, kv_dtype_bytes=run.kvb)
    bytes_per_step = (att["total"] + app) * shape.layers
    tokens_per_step = rl.attended_tokens(shape.seq_lens, shape.q_lens) * shape.layers

    # the timed steps, with clocks sampled from their start to the end of the
    # roofline pass that follows (the steps alone can be shorter than one
    # sampling period)
    clocks = ClockSampler(nvsmi_id(local))
    clocks.start()
    ms_local = run.timed(run.graph, args.steps, args.warmup, barrier)
    ms_total, _ = aggregate_over_ranks(ms_local, 0.0, device)
    ms_step = ms_total / args.steps
    durs, _ = run.roofline_pass(args.warmup, args.roofline_s)
    clock_info = clocks.stop()

    n_e2e = max(1, args.steps // 4)
    e2e_ms = run.timed(run.graph_e2e, n_e2e, args.warmup, barrier) / n_e2e
    e2e_ms, _ = aggregate_over_ranks(e2e_ms, 0.0, device)
    assert pkv.pkv_get_device_error() == 0, pkv.pkv_last_error()
    kernels_per_layer = run.kernels_per_layer()
    value = bytes_per_step * ws_n / (ms_step * 1e-3) / 1e9
    roof = run.roofline(durs, args.config, None)
    troof = tensor_roofline(shape, durs)
    h2d, d2h = run.h2d, run.d2h
    layers_cpu = run.layers[:2]
    del run
    torch.cuda.empty_cache()

    extras = {}
    if not args.no_extra and rank == 0 and ws_n == 1:
        for config, kv in EXTRA_CONFIGS:
            if (config, kv) == (args.config, args.kv):
                continue
            extras[f"{config}/{kv}"] = measure_extra(pkv, config, kv, device, rank, args, local)

    cpu = (cpu_baseline(shape, layers_cpu, args.kv)
           if (rank == 0 and ws_n == 1 and not args.no_cpu) else None)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws_n,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 KV, bf16 q/out, f32 math" if fp8 else "bf16",
        "data": ("synthetic (seeded uniform e4m3 codes, N(0,1) bf16 q/new K/V, shuffled block "
                 "placement; no weights)" if fp8 else
                 "synthetic (seeded N(0,1) bf16 K/V/q, shuffled block placement; no weights)"),
        "config": workload_config(shape, ws_n, args.kv),
        "attended_tokens_per_s": round(tokens_per_step * ws_n / (ms_step * 1e-3), 1),
        "us_per_layer": round(ms_step * 1e3 / shape.layers, 3),
        "frac_of_nominal_8tbs": round(value / ws_n / NOMINAL_HBM_GBS, 4),
        "roofline": roof,
        "e2e": {"value": round(bytes_per_step * ws_n / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 5), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "copies": "every step: all layers' q, new K/V, slot mappings, tables and "
                          "lengths copied from pinned host memory (one 256-byte aligned "
                          "buffer, in chunks of layers 0, 1-3, 4-10, 11-27 on a copy stream; "
                          "each chunk awaited before its first layer's pkv_append_attention); "
                          "the outputs copied back to pinned host memory on a second copy "
                          "stream in chunks of layers 0-6, 7-13, 14-20, 21-27, each as soon as "
                          "its last layer has written it"},
        "gpu_launches": kernels_per_layer * shape.layers * args.steps,
        "clocks": clock_info,
        "cpu_baseline": cpu,
        "configs": extras,
    }
    if troof is not None:
        line["tensor_roofline"] = troof
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws_n > 1:
        torch.distributed.destroy_process_group()


# ---------------------------------------------------------------------------
# CPU baseline / reference arm: the fp64 oracle on bounded samples
# ---------------------------------------------------------------------------

def _oracle_sample(shape, inp_host, n_reqs):
    """Oracle attention for the first n_reqs requests of one layer."""
    import oracle
    qsl = inp_host["qsl"]
    sub_qsl = qsl[:n_reqs + 1]
    t = int(sub_qsl[-1])
    h = inp_host
    if "k_scale" in h:
        return oracle.paged_attention_fp8(h["q"][:t], h["k_pool"], h["v_pool"], h["k_scale"],
                                          h["v_scale"], h["block_tables"][:n_reqs],
                                          h["seq_lens"][:n_reqs], sub_qsl, h["scale"])
    return oracle.paged_attention(h["q"][:t], h["k_pool"], h["v_pool"],
                                  h["block_tables"][:n_reqs], h["seq_lens"][:n_reqs],
                                  sub_qsl, h["scale"])


def _host_layer(inp):
    fp8 = inp.k_pool.dtype == torch.uint8
    pool = (lambda t: t.cpu().numpy()) if fp8 else wl.bf16_bits
    h = dict(q=wl.bf16_bits(inp.q), k_pool=pool(inp.k_pool), v_pool=pool(inp.v_pool),
             block_tables=inp.block_tables.cpu().numpy(), seq_lens=inp.seq_lens.cpu().numpy(),
             qsl=inp.query_start_loc.cpu().numpy(), scale=inp.scale)
    if fp8:
        h["k_scale"] = inp.k_scale.cpu().numpy()
        h["v_scale"] = inp.v_scale.cpu().numpy()
    return h


def sample_bytes(shape, n_reqs, kv):
    """Algorithmic bytes of the attention of the first n_reqs requests."""
    return rl.attention_bytes(shape.seq_lens[:n_reqs], shape.q_lens[:n_reqs], shape.num_q_heads,
                              shape.num_kv_heads,
                              kv_dtype_bytes=1 if kv == "fp8" else 2)["total"]


def cpu_model() -> str:
    """The host CPU's model name (x86 'model name', else lscpu's)."""
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


def _time_oracle(shape, host, n_reqs, budget_s):
    """Calls on the first n_reqs requests, cycling over the host layers,
    until budget_s of oracle time; returns (calls, seconds)."""
    n_calls, t_total = 0, 0.0
    while t_total < budget_s or n_calls == 0:
        h = host[n_calls % len(host)]
        t1 = time.perf_counter()
        _oracle_sample(shape, h, n_reqs)
        t_total += time.perf_counter() - t1
        n_calls += 1
    return n_calls, t_total


def cpu_baseline(shape, layers, kv, budget_s=10.0, budget_1t_s=4.0):
    """The fp64 oracle on the host cores: whole layers with every thread,
    then a sample of requests on one thread."""
    import oracle
    oracle.build()
    host = [_host_layer(x) for x in layers]
    t0 = time.perf_counter()
    threads = oracle.max_threads()
    n_calls, t_all = _time_oracle(shape, host, shape.num_reqs, budget_s)
    value = sample_bytes(shape, shape.num_reqs, kv) * n_calls / t_all / 1e9
    # one thread: as many requests as fit about a tenth of the budget per call
    oracle.set_threads(1)
    try:
        t1 = time.perf_counter()
        _oracle_sample(shape, host[0], 1)
        one = max(1e-4, time.perf_counter() - t1)
        n1 = int(max(1, min(shape.num_reqs, 0.1 * budget_1t_s / one)))
        c1, t_1 = _time_oracle(shape, host, n1, budget_1t_s)
    finally:
        oracle.set_threads(threads)
    value_1t = sample_bytes(shape, n1, kv) * c1 / t_1 / 1e9
    return {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{n_calls} full layers ({shape.num_reqs} requests each) of {shape.name}, "
                      f"fp64 C oracle, OpenMP, {t_all:.1f} s",
            "one_thread": {"value": round(value_1t, 4), "unit": "GB/s", "cores": 1,
                           "sample": f"{c1} calls on the first {n1} requests, {t_1:.1f} s"},
            "nproc": os.cpu_count(), "cpu_model": cpu_model(),
            "wall_s": round(time.perf_counter() - t0, 2)}


def run_reference(args):
    ws_n, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    shape = wl.CONFIGS[args.config]()
    # inputs generated on the host (same seeded recipe as the GPU arm)
    n_layers = min(shape.layers, 2)
    make = wl.make_fp8_step if args.kv == "fp8" else wl.make_step
    host = [_host_layer(make(shape, device="cpu", layer=li)) for li in range(n_layers)]
    # size each step so that warm-up + timed steps fit in about a minute
    t1 = time.perf_counter()
    _oracle_sample(shape, host[0], 1)
    one = max(1e-4, time.perf_counter() - t1)
    budget = 60.0 / max(1, args.steps + args.warmup)
    n_reqs = int(max(1, min(shape.num_reqs, budget / one)))
    for i in range(args.warmup):
        _oracle_sample(shape, host[i % n_layers], n_reqs)
    t0 = time.perf_counter()
    for i in range(args.steps):
        _oracle_sample(shape, host[i % n_layers], n_reqs)
    dt = time.perf_counter() - t0
    value = sample_bytes(shape, n_reqs, args.kv) * args.steps / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": ws_n, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3 / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(shape, ws_n, args.kv),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": oracle.max_threads(),
                         "kind": "oracle",
                         "sample": f"each step: attention of the first {n_reqs} of "
                                   f"{shape.num_reqs} requests of one layer, fp64 C oracle",
                         "nproc": os.cpu_count(), "cpu_model": cpu_model()},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="qwen_decode", choices=sorted(wl.CONFIGS))
    ap.add_argument("--kv", choices=["bf16", "fp8"], default="bf16",
                    help="KV-cache element type (fp8: e4m3 with per-KV-head scales)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-baseline leg")
    ap.add_argument("--no-extra", action="store_true",
                    help="time only the chosen workload (not the other single-layer ones)")
    ap.add_argument("--roofline-s", type=float, default=1.0,
                    help="seconds of back-to-back attention replays per roofline pass")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
