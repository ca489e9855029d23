"""bench.py's host-side helpers and its reference arm, on the CPU.

The reference arm times the fp64 oracle on the host cores and must print the
benchmark's JSON line; the ours arm reports `roofline.traffic` from a
committed ncu summary only while the decode kernels' code still hashes to
the value recorded there (comments may change freely).
"""
import importlib.util
import json
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_source_hash_ignores_comments_but_not_code(bench, tmp_path, monkeypatch):
    srcs = []
    for path in bench.DECODE_SRCS:
        dst = tmp_path / os.path.basename(path)
        shutil.copy(path, dst)
        srcs.append(str(dst))
    monkeypatch.setattr(bench, "DECODE_SRCS", srcs)
    h0 = bench.decode_source_sha()
    with open(srcs[1], "a") as f:
        f.write("\n// a note about the code\n\n")
    assert bench.decode_source_sha() == h0
    with open(srcs[1], "a") as f:
        f.write("static int an_extra_symbol = 1;\n")
    assert bench.decode_source_sha() != h0


def test_committed_traffic_is_read_while_the_hash_matches(bench, tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "decode_qwen_decode_bf16.md").write_text(
        "# summary\n\nkernel_source_sha256_16: %s\ndram_bytes_per_launch: 123456\n"
        % bench.decode_source_sha())
    (prof / "decode_qwen_decode_fp8.md").write_text(
        "kernel_source_sha256_16: 0000000000000000\ndram_bytes_per_launch: 777\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.committed_traffic("qwen_decode", "bf16") == 123456
    assert bench.committed_traffic("qwen_decode", "fp8") is None   # other code
    assert bench.committed_traffic("no_such_config", "bf16") is None


def test_committed_traffic_is_dropped_when_code_changes(bench, tmp_path, monkeypatch):
    srcs = []
    for path in bench.DECODE_SRCS:
        dst = tmp_path / os.path.basename(path)
        shutil.copy(path, dst)
        srcs.append(str(dst))
    with open(srcs[0], "a") as f:
        f.write("static int changed = 2;\n")
    monkeypatch.setattr(bench, "DECODE_SRCS", srcs)
    assert bench.committed_traffic("qwen_decode", "bf16") is None


def test_decode_kernel_names_follow_the_routing(bench):
    on = {"decode_tc": 1, "decode_tc_fp8": 1}
    assert bench.decode_kernel_name(6, False, on) == "pkv::decode_tc_kernel<6, false>"
    assert bench.decode_kernel_name(4, True, on) == "pkv::decode_tc_kernel<4, true>"
    assert bench.decode_kernel_name(2, False, on) == "pkv::decode_kernel<2, KvBf16>"
    assert bench.decode_kernel_name(3, True, on) == "pkv::decode_kernel<3, KvE4m3>"
    simt_fp8 = {"decode_tc": 1, "decode_tc_fp8": 0}
    assert bench.decode_kernel_name(6, True, simt_fp8) == "pkv::decode_kernel<6, KvE4m3>"
    assert bench.decode_kernel_name(6, False, simt_fp8) == "pkv::decode_tc_kernel<6, false>"
    simt = {"decode_tc": 0, "decode_tc_fp8": 1}
    assert bench.decode_kernel_name(6, False, simt) == "pkv::decode_kernel<6, KvBf16>"


def test_reference_arm_prints_the_benchmark_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "tiny", "--steps", "3", "--warmup", "3"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["value"] > 0 and line["unit"] == "GB/s" and line["higher_is_better"] is True
    assert line["steps"] == 3 and line["warmup"] == 3
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["config"]["workload"]


def test_cpu_sample_bytes_follow_the_requests_run(bench):
    # ragged lengths: the bytes of the first n requests, not n x request 0's
    from paged_kv_cache_195_gb300 import roofline as rl
    from paged_kv_cache_195_gb300 import workloads as wl
    shape = wl.llama_mixed()
    for n in (1, 7, 100, shape.num_reqs):
        want = rl.attention_bytes(shape.seq_lens[:n], shape.q_lens[:n], 32, 8)["total"]
        assert bench.sample_bytes(shape, n, "bf16") == want
    per_req0 = rl.attention_bytes(shape.seq_lens[:1], shape.q_lens[:1], 32, 8)["total"]
    assert bench.sample_bytes(shape, 100, "bf16") != 100 * per_req0
    e4m3 = bench.sample_bytes(shape, 10, "fp8")
    assert e4m3 == rl.attention_bytes(shape.seq_lens[:10], shape.q_lens[:10], 32, 8,
                                      kv_dtype_bytes=1)["total"]


def test_lengths_summary(bench):
    assert bench.lengths_summary([512] * 64) == 512
    s = bench.lengths_summary([16, 1000, 8192, 40])
    assert s == {"min": 16, "median": 520.0, "max": 8192, "sum": 9248}


def test_cpu_model_is_named(bench):
    name = bench.cpu_model()
    assert isinstance(name, str) and name


def test_committed_traffic_of_a_two_kernel_call_hashes_its_listed_sources(bench, tmp_path,
                                                                           monkeypatch):
    csrc = tmp_path / "paged_kv_cache_195_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name in ("a.cu", "b.cuh"):
        (csrc / name).write_text("int %s_symbol = 1;\n" % name[0])
    sha = bench.decode_source_sha([str(csrc / "a.cu"), str(csrc / "b.cuh")])
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "attention_mixed_bf16.md").write_text(
        "kernel_sources: a.cu b.cuh\nkernel_source_sha256_16: %s\n"
        "dram_bytes_per_launch: 4242\n" % sha)
    (prof / "attention_gone_bf16.md").write_text(
        "kernel_sources: a.cu missing.cu\nkernel_source_sha256_16: %s\n"
        "dram_bytes_per_launch: 1\n" % sha)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.committed_traffic("mixed", "bf16") == 4242
    assert bench.committed_traffic("gone", "bf16") is None     # a listed source is missing
    with open(csrc / "b.cuh", "a") as f:
        f.write("int another = 2;\n")
    assert bench.committed_traffic("mixed", "bf16") is None    # the code changed



def test_tensor_roofline_only_for_prefill_only_steps(bench):
    import paged_kv_cache_195_gb300.roofline as rl
    from paged_kv_cache_195_gb300 import workloads as wl
    # a step with decode rows is bounded by HBM: no tensor-core line
    assert bench.tensor_roofline(wl.llama_mixed(), [0.4]) is None
    # the eight prefill chunks alone: flops over the mean launch time
    shape = wl.llama_mixed(num_decode=0)
    t = bench.tensor_roofline(shape, [0.15, 0.17])
    flops = rl.attention_flops(shape.seq_lens, shape.q_lens, shape.num_q_heads)
    assert t["bound"] == "tensor" and t["unit"] == "TFLOP/s"
    assert t["flops_per_launch"] == flops
    assert abs(t["achieved"] - flops / 0.16e-3 / 1e12) < 0.1
    assert abs(t["frac"] - t["achieved"] / t["peak"]) < 1e-3
