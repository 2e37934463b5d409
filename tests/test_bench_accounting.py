"""The bench's accounting on the CPU: the algorithmic bytes and flops it divides by, the
committed ncu summaries it takes `traffic` from (each must still describe the current kernel
sources, else the bench would report a stale figure), and the reference arm's JSON line."""
import glob
import os
import re

import pytest

import bench
from stream_gated_residual_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bytes_per_token_of_the_workloads():
    # bf16 prefill: R in and out (4·D·2 each), y in and x out (D·2 each), s in and out (4·4 each)
    assert bench.bytes_per_token(wl.WORKLOADS["prefill"]) == 2 * 4 * 4096 * 2 + 2 * 4096 * 2 + 32
    # FP8 state: codes and block exponents in and out, y and x bf16
    D = 4096
    assert bench.bytes_per_token(wl.WORKLOADS["prefill_fp8"]) == \
        2 * (4 * D + 4 * D // 32) + 2 * D * 2 + 32
    assert bench.bytes_per_token(wl.WORKLOADS["tiny_fp32"]) == 2 * 4 * 256 * 4 + 2 * 256 * 4 + 32


def test_flops_of_the_large_rank_and_backward_legs():
    w = wl.WORKLOADS["paper_rank"]
    K = 4 * w.d_model
    assert bench.tc_flops_per_token(w) == 2 * (w.rank + 4) * K + 2 * K * w.rank
    p = wl.WORKLOADS["prefill"]
    Kp, r = 4 * p.d_model, p.rank
    assert bench.backward_flops_per_token(p) == 2 * Kp * (6 * r + 13) + 16 * Kp


def test_decomposition_bytes_count_every_pair():
    w = wl.WORKLOADS["deep_stack"]
    two = bench.decompose_bytes(w, 2)   # one reader with one writer
    es, D, N, r = 2, w.d_model, w.n_tokens, w.rank
    assert two == N * (2 * 4 * D * es + (D * es + 16) + 4 * 6 + 4) + \
        4 * (4 * D + 2 * r * 4 * D + 4 * 4 * D)
    assert bench.decompose_bytes(w, 40) > 39 * two   # the writers' share grows with the reader


@pytest.mark.parametrize("path", sorted(glob.glob(os.path.join(ROOT, "profiles", "*__*.md"))))
def test_committed_profiles_match_the_sources(path):
    """A summary that carries a source hash and a DRAM figure is the one the bench reads for its
    kernel path and workload; the hash must be that of the current sources."""
    text = open(path).read()
    m_s = re.search(r"^source_sha256:\s*([0-9a-f]{64})", text, re.M)
    m_b = re.search(r"^dram_bytes_per_launch:\s*(\d+)", text, re.M)
    if not (m_s and m_b):
        pytest.skip("launch list only (no traffic figure)")
    kernel_path, workload = os.path.basename(path)[:-3].split("__")
    assert workload in wl.WORKLOADS
    assert m_s.group(1) == bench.kernel_source_sha(kernel_path), \
        f"{os.path.basename(path)} describes sources that have changed since"
    assert bench.profiled_traffic(kernel_path, workload) == int(m_b.group(1))


@pytest.mark.parametrize("workload,extra", [("tiny_fp32", []), ("prefill", ["--n-tokens", "48"])])
def test_reference_arm_prints_one_json_line(workload, extra):
    """`bench.py --impl reference` times the fp64 oracle on the host cores (no GPU) and prints
    one JSON line with the arm's keys: the same metric and unit as the CUDA arm, the oracle's
    core count and sample, and an end-to-end figure that moves no bytes to or from a device."""
    import json
    import subprocess
    import sys
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", workload, "--steps", "2", "--warmup", "1", *extra],
                         cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["metric"] == bench.METRIC
    assert rec["unit"] == bench.UNIT and rec["value"] > 0 and rec["higher_is_better"] is True
    assert rec["steps"] == 2 and rec["warmup"] == 1 and rec["dtype"] == "f64"
    cb = rec["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == rec["value"]
    e2e = rec["e2e"]
    assert e2e["value"] == rec["value"] and e2e["unit"] == rec["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    # the same config object as the CUDA arm's line for this workload at one GPU
    w = wl.WORKLOADS[workload]
    if extra:
        w = w.scaled(n_tokens=int(extra[1]))
    assert rec["config"] == bench.bench_config(w, 1, bench.l2_policy(w, bench.L2_BYTES_DEFAULT)[1])


def test_l2_policy_flushes_only_inputs_below_twice_the_l2():
    l2 = bench.L2_BYTES_DEFAULT
    for name, flush in [("decode", True), ("tiny_fp32", True), ("prefill", False),
                        ("large_skewed", False), ("prefill_fp8", False)]:
        f, note = bench.l2_policy(wl.WORKLOADS[name], l2)
        assert f is flush, name
        assert note.startswith("L2 flushed" if flush else "inputs larger than L2"), name
    # the deep-stack sublayer: 8192 tokens of a [4, 2048] bf16 state (128 MiB) plus y, x, s
    f, _ = bench.l2_policy(wl.WORKLOADS["deep_stack"], l2)
    assert f is True


def test_cpu_baseline_reports_all_cores_and_one_core():
    """The CUDA arm's `cpu_baseline`: the oracle on all host cores, repeated until its sample
    covers the target time, and on one core; the thread count is restored afterwards."""
    import oracle
    oracle.build()
    before = oracle.num_threads()
    cb = bench.cpu_baseline(wl.WORKLOADS["tiny_fp32"], target_s=0.5)
    assert oracle.num_threads() == before
    assert cb["kind"] == "oracle" and cb["unit"] == bench.UNIT and cb["value"] > 0
    assert cb["cores"] == before and "time(s)" in cb["sample"]
    sc = cb["single_core"]
    assert sc["cores"] == 1 and sc["value"] > 0 and sc["unit"] == bench.UNIT
