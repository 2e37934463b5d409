#!/usr/bin/env python
"""Throughput of the fused Gated Residual write→read on GB300.

One step = one fused gr_write_then_read over the whole workload (default: prefill, N=16384
tokens, D=4096, 4 branches, r=16, bf16 states), with the write strengths ping-ponged from step
to step like a chain of sublayers. The state (512 MiB) is larger than L2, so no flush is
needed between steps. Prints one JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gr|reference] [--workload NAME]

For N > 1 (torchrun, one process per GPU) every rank processes its own token shard of the
same size (weak scaling); there is no data-path collective, only the timing barrier and a
max over ranks. `--impl reference` times the fp64 CPU oracle on this host's cores on a bounded
sample of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import platform
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

METRIC = "GR fused read/write tokens/s & HBM GB/s vs GB300 peak (4 branches, D=4096)"
UNIT = "tokens/s"
BAD_REASONS = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[1])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["gr", "reference"], default="gr")
    ap.add_argument("--workload", default=None,
                    help="workload name (default: prefill; deep_stack with --decompose)")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch every timed step from the host instead of replaying a CUDA graph "
                         "of them")
    ap.add_argument("--backward", action="store_true",
                    help="time one sublayer's GR backward (gr_read_backward, then "
                         "gr_write_backward in place) instead of the fused forward step")
    ap.add_argument("--decompose", action="store_true",
                    help="time the contribution decomposition of a stack of --blocks GR blocks "
                         "(every reader against all its writers) instead of the fused step")
    ap.add_argument("--blocks", type=int, default=40,
                    help="blocks of the decomposed stack (40: the pages' 780 block pairs)")
    ap.add_argument("--n-tokens", type=int, default=None,
                    help="run the workload's shape with this many tokens instead (small cases "
                         "for profiling; the line then reports no ncu traffic)")
    return ap.parse_args(argv)


# ---------------------------------------------------------------------------------------------
# accounting

def bytes_per_token(w) -> int:
    """Algorithmic HBM bytes of one token in the fused step: R read and written (4·D each),
    y read, x written (D each), s_prev read and s_next written (4 fp32 each). On the FP8 state
    R is 4·D one-byte codes plus 4·D/32 one-byte block exponents, and y and x are bf16."""
    D = w.d_model
    if w.dtype == "fp8":
        return 2 * (4 * D + 4 * D // 32) + 2 * D * 2 + 2 * 4 * 4
    b = w.state_bytes_per_elem()
    return 2 * 4 * D * b + 2 * D * b + 2 * 4 * 4


def weight_bytes(w) -> int:
    """Parameter bytes a fused launch reads once: W_d, W_w, W_u (fp32 on the fp32 path, bf16
    otherwise), gamma fp32."""
    b = 4 if w.dtype == "f32" else 2
    K = 4 * w.d_model
    return (2 * w.rank + 4) * K * b + K * 4


def workload_desc(w) -> str:
    return (f"{w.name}: fused GR write->read, N={w.n_tokens} tokens, D={w.d_model}, 4 branches, "
            f"r={w.rank}, {w.dtype} states, fp32 accumulation")


def l2_policy(w, l2_bytes: int) -> tuple[bool, str]:
    """Whether the timed steps flush L2, and the sentence that says so. Inputs at least twice
    the L2 stream from HBM by themselves; smaller ones (decode) get the L2 flushed before every
    step, outside that step's timed window."""
    n, D = w.n_tokens, w.d_model
    if w.dtype == "fp8":
        state = n * 4 * (D + D // 32)
    else:
        state = n * 4 * D * w.state_bytes_per_elem()
    io = 2 * n * D * (4 if w.dtype == "f32" else 2) + 2 * n * 16
    in_bytes = state + io
    if in_bytes < 2 * l2_bytes:
        return True, (f"L2 flushed before every step ({2 * l2_bytes >> 20} MiB written; inputs "
                      f"{in_bytes >> 20} MiB), per-step event windows")
    return False, f"inputs larger than L2 (state {state >> 20} MiB), no flush"


def bench_config(w, world: int, l2_note: str) -> dict:
    """The `config` object of a bench line: the same keys and values in both arms for one
    workload and world size, so that the two lines describe one workload."""
    return {"workload": workload_desc(w), "n_tokens_per_gpu": w.n_tokens,
            "d_model": w.d_model, "rank": w.rank, "n_branch": 4, "state_dtype": w.dtype,
            "accumulate": "fp32", "parallelism": f"dp{world}", "l2": l2_note}


L2_BYTES_DEFAULT = 126 << 20   # a GB300's L2, for a process that has no device to ask


def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained") or 0) or None,
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def tc_flops_per_token(w) -> int:
    """Tensor-core arithmetic of one token on the large-rank path (FMA = 2 FLOP): the down
    projection [W_d; W_w] (r + 4 outputs over 4·D inputs) and the up projection W_u (4·D outputs
    over r inputs)."""
    K = 4 * w.d_model
    return 2 * (w.rank + 4) * K + 2 * K * w.rank


def kernel_source_sha(kernel_path: str) -> str:
    """Hash of the sources that decide a kernel path's device traffic: the kernels' .cu files and
    the PTX wrappers they share; a split path ("fused_bf16+tiled_bf16") adds the split dispatch
    (gr_split.cu), which decides how many tokens each kernel gets."""
    from stream_gated_residual_gb300 import build as gbuild
    files = {"fused_bf16": "gr_fused_bf16.cu", "tiled_bf16": "gr_tiled_bf16.cu",
             "tiled_fp8": "gr_tiled_bf16.cu", "generic": "gr_generic.cu",
             "tc_bf16": "gr_rank_tc.cu", "decompose": "gr_decompose.cu"}
    names = [files[k] for k in kernel_path.split("+")]
    if kernel_path == "tc_bf16":
        names.append("gr_tc.cuh")
    if len(names) > 1:
        names.append("gr_split.cu")
    h = hashlib.sha256()
    for p in [os.path.join(gbuild.CSRC, n) for n in names + ["gr_ptx.cuh"]]:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profiled_traffic(kernel_path: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary of this kernel and workload, if the
    kernel source has not changed since it was captured; else None."""
    path = os.path.join(ROOT, "profiles", f"{kernel_path}__{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_b = re.search(r"^dram_bytes_per_launch:\s*(\d+)", text, re.M)
    m_s = re.search(r"^source_sha256:\s*([0-9a-f]{64})", text, re.M)
    if not (m_b and m_s) or m_s.group(1) != kernel_source_sha(kernel_path):
        return None
    return int(m_b.group(1))


# ---------------------------------------------------------------------------------------------
# clocks

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while the timed region runs."""

    QUERY = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = (uuid or "").lower()
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="gr_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-f", self.path], stdout=subprocess.DEVNULL,
                stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        rows = []
        if self.path and os.path.exists(self.path):
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                if self.uuid and self.uuid not in parts[1].lower():
                    continue
                rows.append(parts)
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(s):
            try:
                return float(s)
            except ValueError:
                return None
        sm = [num(r[2]) for r in rows if num(r[2]) is not None]
        mx = [num(r[3]) for r in rows if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[6 + k] == "Active"})
        loaded = [v for v in sm if mx and v >= 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------------------------
# CPU oracle (baseline and reference arm)

class OracleInputs:
    """The workload's inputs in fp64 for the first n tokens (generated once)."""

    def __init__(self, w, n_tokens: int):
        import oracle
        from stream_gated_residual_gb300 import workloads as wl
        self.w = w
        self.n = n_tokens
        self.R = wl.to_f64(wl.make_state(w, n_tokens))
        if w.dtype == "fp8":   # the FP8 state of the same values (the oracle's own encoding)
            self.codes, self.scales = oracle.fp8_encode(self.R)
        self.y = wl.to_f64(wl.make_y(w, 0, n_tokens))
        self.sp = wl.make_s_prev(w, n_tokens)
        self.p = wl.make_params(w, 1)

    def run(self, a: int, b: int) -> float:
        """Seconds of one fused oracle step on tokens a..b-1."""
        import oracle
        t0 = time.perf_counter()
        if self.w.dtype == "fp8":
            oracle.write_then_read_fp8(self.codes[a:b], self.scales[a:b], self.y[a:b],
                                       self.sp[a:b], self.p, self.w.eps)
        else:
            oracle.write_then_read(self.R[a:b], self.y[a:b], self.sp[a:b], self.p, self.w.eps)
        return time.perf_counter() - t0


def cpu_baseline(w, target_s: float = 12.0) -> dict:
    import oracle
    oracle.build()
    probe = 64
    t = OracleInputs(w, probe).run(0, probe)
    n = int(max(probe, min(w.n_tokens, target_s * probe / max(t, 1e-9))))
    inp = OracleInputs(w, n)
    t = inp.run(0, n)
    # a workload the oracle finishes well inside the target is repeated, for a stable figure
    reps = 1
    while t < 0.8 * target_s and reps < 1000:
        t += inp.run(0, n)
        reps += 1
    cores = oracle.num_threads()
    # the same oracle on one core, on a sample sized for about 3 s
    oracle.set_num_threads(1)
    try:
        t1 = OracleInputs(w, probe).run(0, probe)
        n1 = int(max(1, min(n, 3.0 * probe / max(t1, 1e-9))))
        t1, reps1 = inp.run(0, n1), 1
        while t1 < 2.0 and reps1 < 1000:
            t1 += inp.run(0, n1)
            reps1 += 1
    finally:
        oracle.set_num_threads(cores)
    return {"value": reps * n / t, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"first {n} of {w.n_tokens} tokens of the {w.name} workload, one fused "
                      f"write->read in fp64, {reps} time(s) ({t:.1f} s)",
            "host": f"{os.cpu_count()} logical CPUs, {platform.machine()}",
            "single_core": {"value": reps1 * n1 / t1, "unit": UNIT, "cores": 1,
                            "sample": f"first {n1} tokens, {reps1} time(s) ({t1:.1f} s)"}}


def reference_l2_bytes() -> int:
    """The L2 size the GPU arm's timing policy is decided with (asked of the device when one is
    visible; the reference arm itself runs on the host cores)."""
    try:
        import torch
        if torch.cuda.is_available():
            return int(torch.cuda.get_device_properties(0).L2_cache_size) or L2_BYTES_DEFAULT
    except Exception:   # noqa: BLE001 - no device: the default
        pass
    return L2_BYTES_DEFAULT


def run_reference(args, w) -> None:
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    steps, warmup = max(1, args.steps), max(0, args.warmup)
    probe = OracleInputs(w, 32)
    probe_t = probe.run(0, 32)
    budget_s = 150.0
    per_step = int(max(1, min(w.n_tokens, budget_s * 32 / probe_t / (steps + warmup))))
    pool = min(w.n_tokens, max(per_step, 2048))
    inp = OracleInputs(w, pool)

    def window(i):
        a = (i * per_step) % max(1, pool - per_step + 1)
        return a, a + per_step

    for i in range(warmup):
        inp.run(*window(i))
    total = 0.0
    for i in range(steps):
        total += inp.run(*window(i))
    value = steps * per_step / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": steps, "warmup": warmup, "ms_per_step": 1e3 * total / steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": bench_config(w, args.gpus, l2_policy(w, reference_l2_bytes())[1]),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(),
                         "kind": "oracle",
                         "sample": f"{per_step} of the first {pool} tokens of the {w.name} "
                                   f"workload per step (fused write->read, fp64)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------------------------
# multi-rank host logic (weak scaling: one token shard per rank, no data-path collective)

def shard(w, rank: int):
    """The workload rank `rank` processes: the same shape on every rank, its own seed."""
    return w.scaled(seed=w.seed + rank)


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest of the ranks' values (the slowest rank sets a job's time)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def any_over_ranks(flag: bool, world: int, device=None) -> bool:
    """True on every rank if any rank's flag is set: one decision that all ranks act on, so
    that they all run the same collectives afterwards (a re-measurement is taken by every rank
    or by none)."""
    if world <= 1:
        return bool(flag)
    return max_over_ranks(1.0 if flag else 0.0, world, device) > 0.5


def job_tokens_per_s(world: int, n_tokens_per_rank: int, steps: int, seconds: float) -> float:
    """Whole-job throughput: the tokens every rank processed over the slowest rank's time."""
    return world * n_tokens_per_rank * steps / seconds


# ---------------------------------------------------------------------------------------------
# GPU arm

def run_gr(args, w) -> None:
    import numpy as np
    import torch
    import torch.distributed as dist

    from stream_gated_residual_gb300 import gr
    from stream_gated_residual_gb300 import workloads as wl

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    gr.load()
    fp8 = w.dtype == "fp8"
    tdt = torch.float32 if w.dtype == "f32" else torch.bfloat16   # y and x
    sdt = gr.FP8 if fp8 else tdt                                  # the state, for shapes

    # each rank owns its own shard of tokens (a different seed), same size on every rank
    wr = shard(w, rank)

    def dev_tensor(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(a).to(dev)

    R_h, y_h, sp_h = wl.make_state(wr), wl.make_y(wr), wl.make_s_prev(wr)
    p = wl.make_params(wr, 1)
    y = dev_tensor(y_h)
    if fp8:   # the FP8 state, encoded by the library from the workload's fp32 values
        src = dev_tensor(R_h)
        codes, scales = gr.fp8_encode(src)
        del src
        state = (codes, scales)
    else:
        R = dev_tensor(R_h)
        state = (R,)
    s_a = torch.from_numpy(sp_h).to(dev)
    s_b = torch.empty_like(s_a)
    x = torch.empty((w.n_tokens, w.d_model), dtype=tdt, device=dev)
    pt = {k: torch.from_numpy(v).to(dev) for k, v in p.items()}
    P = gr.pack_params(pt["gamma"], pt["w_down"], pt["w_up"], pt["w_write"], sdt, w.eps)
    path = gr.kernel_path(w.n_tokens, w.d_model, w.rank, sdt)
    stream = torch.cuda.current_stream(dev)
    # "fused_bf16+tiled_bf16": two kernels a step; the large-rank path: three
    launches_per_step = 3 if path == "tc_bf16" else len(path.split("+"))
    ws_need = 0 if fp8 else gr.step_workspace_size(w.n_tokens, w.d_model, w.rank, sdt)
    ws = None
    if ws_need:
        wsb = torch.empty(ws_need + 256, dtype=torch.uint8, device=dev)
        ws = wsb[(-wsb.data_ptr()) % 256:][:ws_need]

    def fused(sp, sn, st):
        if fp8:
            gr.write_then_read_fp8(codes, scales, y, sp, P, x=x, s_next=sn, stream=st)
        else:
            gr.write_then_read(R, y, sp, P, x=x, s_next=sn, stream=st, workspace=ws)

    def step(i):
        sp, sn = (s_a, s_b) if i % 2 == 0 else (s_b, s_a)
        fused(sp, sn, stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)

    props = torch.cuda.get_device_properties(dev)
    uuid = str(getattr(props, "uuid", "") or "")
    # Inputs at least twice the L2 stream from HBM by themselves; smaller ones (decode) get the
    # L2 flushed before every step, outside that step's timed window.
    l2_bytes = int(getattr(props, "L2_cache_size", 0) or L2_BYTES_DEFAULT)
    flush, l2_note = l2_policy(w, l2_bytes)
    fbuf = torch.empty(2 * l2_bytes, dtype=torch.uint8, device=dev) if flush else None

    # The timed steps replay CUDA graphs of the same launches (no host work per step: the small
    # workloads are otherwise bound by the host's launch path). With the flush, one graph per
    # parity of the step (the s buffers alternate); without it, one graph of all timed steps.
    graphs = None
    if not args.no_graph:
        graphs = []
        for rng_ in ([(0,), (1,)] if flush else [tuple(range(args.steps))]):
            g_ = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_, capture_error_mode="relaxed"):
                cs = torch.cuda.current_stream(dev)
                for i in rng_:
                    sp, sn = (s_a, s_b) if i % 2 == 0 else (s_b, s_a)
                    fused(sp, sn, cs)
            g_.replay()   # one untimed replay
            graphs.append(g_)
        torch.cuda.synchronize(dev)

    def run_step(i):
        if graphs is None:
            step(i)
        else:
            graphs[i % 2].replay()

    def timed():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        sampler = ClockSampler(uuid)
        sampler.start()
        # The GPU idled while the sampler started. Untimed steps (as many as the warm-up) are
        # queued right before the first timed event, so that the window opens on a busy GPU.
        for i in range(max(1, args.warmup)):
            step(i)
        if flush:
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(args.steps)]
            for i in range(args.steps):
                fbuf.fill_(i & 0xff)
                ev[i][0].record(stream)
                run_step(i)
                ev[i][1].record(stream)
        else:
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            if graphs is not None:
                graphs[0].replay()
            else:
                for i in range(args.steps):
                    step(i)
            e1.record(stream)
        torch.cuda.synchronize(dev)
        clocks = sampler.stop()
        if world > 1:
            dist.barrier()
        local = sum(a.elapsed_time(b) for a, b in ev) if flush else e0.elapsed_time(e1)
        ms = max_over_ranks(local, world, dev)
        return ms, clocks

    ms, clocks = timed()
    # one re-measurement, on every rank, if any rank saw a thermal or hardware slowdown
    if any_over_ranks(bool(BAD_REASONS & set(clocks["reasons"])), world, dev):
        ms, clocks = timed()
        clocks["remeasured"] = True
    ms_step = ms / args.steps
    tokens_per_s = job_tokens_per_s(world, w.n_tokens, args.steps, ms / 1e3)

    # roofline of the one kernel of the step
    peaks = load_peaks()
    alg_bytes = w.n_tokens * bytes_per_token(w) + weight_bytes(w)
    achieved = alg_bytes / (ms_step / 1e3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "peak_source": peaks["source"],
                "kernel": path, "algorithmic_bytes_per_launch": alg_bytes,
                "traffic": None if args.n_tokens is not None else profiled_traffic(path, w.name)}
    if path == "tc_bf16":
        # the pages' rank makes the read a dense contraction: against the bf16 tensor peak
        # (sustained: the step is timed over a long loop), the HBM figures beside it
        flops = w.n_tokens * tc_flops_per_token(w)
        tflops = flops / (ms_step / 1e3) / 1e12
        tpeak = peaks.get("bf16_tflops_sustained") or 1700.0
        roofline = {"bound": "tensor", "achieved": tflops, "peak": tpeak, "unit": "TFLOP/s",
                    "frac": tflops / tpeak, "peak_source": peaks["source"] + " (bf16 sustained)",
                    "kernel": path, "algorithmic_flops_per_step": flops,
                    "hbm": {"achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                            "frac": achieved / peaks["hbm_gbs"],
                            "algorithmic_bytes_per_step": alg_bytes},
                    "traffic": None if args.n_tokens is not None
                    else profiled_traffic(path, w.name)}

    # bandwidth reference: single-stream x += y on [N, D]
    xr = torch.zeros((w.n_tokens, w.d_model), dtype=tdt, device=dev)
    yr = y.clone()
    for _ in range(5):
        gr.residual_add_ref(xr, yr, stream=stream)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    nref = 50
    e0.record(stream)
    for _ in range(nref):
        gr.residual_add_ref(xr, yr, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ref_gbs = 3 * xr.numel() * xr.element_size() / (e0.elapsed_time(e1) / nref / 1e3) / 1e9
    del xr, yr

    if fp8:
        e2e = e2e_device_copies(args, w, world, dev, stream, (codes, scales, y, s_a),
                                (codes, scales, x, s_b), s_a, s_b, fused,
                                "gr_write_then_read_fp8 with pinned-host torch copies on the "
                                "same stream")
    elif path == "tc_bf16":
        e2e = e2e_device_copies(args, w, world, dev, stream, (R, y, s_a), (R, x, s_b), s_a, s_b,
                                fused, "gr_write_then_read_ws with pinned-host torch copies on "
                                       "the same stream")
    else:
        e2e = e2e_host_entry(args, w, world, dev, stream, tdt, R_h, y_h, sp_h, P)
        del R
    del state, y, x, s_a, s_b
    torch.cuda.empty_cache()

    base = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        base = cpu_baseline(w)

    if rank == 0:
        line = {
            "metric": METRIC, "value": tokens_per_s, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
            "data": "synthetic (seeded numpy PCG64; no dataset)",
            "config": bench_config(w, world, l2_note),
            "launch": "host launches" if graphs is None else "CUDA graphs of the timed steps",
            "hbm_gbs": achieved,
            "roofline": roofline,
            "bandwidth_reference": {"kernel": "gr_residual_add_ref (x += y, single stream)",
                                    "gbs": ref_gbs, "frac": ref_gbs / peaks["hbm_gbs"]},
            "cpu_baseline": base,
            "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def backward_flops_per_token(w) -> int:
    """Arithmetic of one token's GR backward (FMA = 2 FLOP), per element of vec R̂ (4·D): the
    forward projections recomputed (z, u: r+4; g: r), W_uᵀ dg (r), W_dᵀ dz + W_wᵀ du (r+4), the
    parameter-gradient products (dW_u: r, dW_d and dW_w: r+4, dγ: 1), and about 12 more for the
    element-wise chain (σ, dG, dR̂, the RMSNorm backward); then the write's backward (4 per
    element)."""
    r, K = w.rank, 4 * w.d_model
    return 2 * K * ((r + 4) + r + r + (r + 4) + r + (r + 4) + 1) + 12 * K + 4 * K


def run_backward(args, w) -> None:
    """gr_read_backward then gr_write_backward (in place on the same dR) on the workload, K
    timed steps after W warm-up steps, one GPU (a replica per rank under torchrun)."""
    import numpy as np
    import torch
    import torch.distributed as dist

    from stream_gated_residual_gb300 import gr
    from stream_gated_residual_gb300 import workloads as wl
    if w.dtype == "fp8":
        raise SystemExit("the backward takes bf16 or fp32 states")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    gr.load()
    wr = shard(w, rank)
    tdt = torch.float32 if w.dtype == "f32" else torch.bfloat16

    def dev_tensor(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(a).to(dev)

    R, y = dev_tensor(wl.make_state(wr)), dev_tensor(wl.make_y(wr))
    s = torch.from_numpy(wl.make_s_prev(wr)).to(dev)
    p = {k: torch.from_numpy(v).to(dev) for k, v in wl.make_params(wr, 1).items()}
    rng = np.random.default_rng(wr.seed + 1000)
    dx = torch.from_numpy(rng.standard_normal((w.n_tokens, w.d_model), dtype=np.float32)).to(dev)
    ds = torch.from_numpy(rng.standard_normal((w.n_tokens, 4), dtype=np.float32)).to(dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        dR, _ = gr.read_backward(R, p["gamma"], p["w_down"], p["w_up"], p["w_write"], dx, ds,
                                 w.eps, workspace=ws, stream=stream)
        gr.write_backward(dR, y, s, stream=stream)

    import ctypes
    need = ctypes.c_size_t(0)
    shape = gr.make_shape(w.n_tokens, w.d_model, w.rank, tdt, w.eps)
    gr.load().gr_read_backward_workspace_size(ctypes.byref(shape), ctypes.byref(need))
    wsb = torch.empty(need.value + 256, dtype=torch.uint8, device=dev)
    ws = wsb[(-wsb.data_ptr()) % 256:][:need.value]
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    props = torch.cuda.get_device_properties(dev)
    if world > 1:
        dist.barrier()
    sampler = ClockSampler(str(getattr(props, "uuid", "") or ""))
    sampler.start()
    step()   # untimed, queued right before the window: it opens on a busy GPU
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    ms_step = ms / args.steps
    # fp32 CUDA-core peak: SMs × 128 fp32 lanes × 2 FLOP × the SM clock seen under load
    mhz = clocks.get("sm_mhz") or 2070.0
    peak = props.multi_processor_count * 128 * 2 * mhz * 1e6 / 1e12
    flops = w.n_tokens * backward_flops_per_token(w)
    achieved = flops / (ms_step / 1e3) / 1e12
    if rank == 0:
        line = {
            "metric": "GR read+write backward tokens/s (one sublayer)",
            "value": job_tokens_per_s(world, w.n_tokens, args.steps, ms / 1e3), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded numpy PCG64; no dataset)",
            "config": {"workload": workload_desc(w), "n_tokens_per_gpu": w.n_tokens,
                       "d_model": w.d_model, "rank": w.rank, "state_dtype": w.dtype,
                       "pass": "backward (gr_read_backward + gr_write_backward)"},
            "roofline": {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak, "traffic": None,
                         "peak_source": "SMs x 128 fp32 lanes x 2 x sampled SM clock"},
            "gpu_launches": 6 * args.steps,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def decompose_bytes(w, blocks: int) -> int:
    """Algorithmic HBM bytes of one decomposition of a stack of ``blocks`` GR blocks: for every
    reader v = 1..blocks-1, its state and the initial state (4·D each, state dtype), its v
    writers' outputs (D, state dtype) and write strengths (4 fp32), and its outputs per token
    (v writer norms, 4v branch norms, v fractions and the initial state's share, fp32), plus
    its parameters (fp32) once."""
    es = w.state_bytes_per_elem()
    D, r, N = w.d_model, w.rank, w.n_tokens
    total = 0
    for v in range(1, blocks):
        total += N * (2 * 4 * D * es + v * (D * es + 16) + v * 4 * 6 + 4)
        total += 4 * (4 * D + 2 * r * 4 * D + 4 * 4 * D)
    return total


def run_decompose(args, w) -> None:
    """The contribution decomposition (eq auv and π) of a stack of --blocks GR blocks on the
    workload's shape: the stack's states, write strengths and block outputs are made once by
    the library's own forward chain (seeded y, fresh weights per block); one step decomposes
    every reader v = 1..blocks-1 against its v writers and the initial state (all
    blocks·(blocks-1)/2 ordered pairs), one gr_decompose launch per reader."""
    import ctypes

    import numpy as np
    import torch
    import torch.distributed as dist

    from stream_gated_residual_gb300 import gr
    from stream_gated_residual_gb300 import workloads as wl
    if w.dtype not in ("bf16", "f32"):
        raise SystemExit("the decomposition takes bf16 or fp32 states")
    L = args.blocks
    if L < 2:
        raise SystemExit("--blocks must be >= 2")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    gr.load()
    wr = shard(w, rank)
    tdt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    N, D, r = w.n_tokens, w.d_model, w.rank

    def dev_tensor(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(a).to(dev)

    # the stack: states before every read, write strengths and outputs of every block
    states = torch.empty((L, N, 4, D), dtype=tdt, device=dev)
    Y = torch.empty((L, N, D), dtype=tdt, device=dev)
    S = torch.empty((L, N, 4), dtype=torch.float32, device=dev)
    params = []
    R = dev_tensor(wl.make_state(wr))
    R0 = R.clone()
    x = torch.empty((N, D), dtype=tdt, device=dev)
    for v in range(L):
        p = {k: torch.from_numpy(a).to(dev) for k, a in wl.make_params(wr, v + 1).items()}
        params.append(p)
        P = gr.pack_params(p["gamma"], p["w_down"], p["w_up"], p["w_write"], tdt, w.eps)
        if v == 0:
            _, s = gr.read(R, P)
        else:   # the write of block v-1, in place, then block v's read
            _, s = gr.write_then_read(R, Y[v - 1], S[v - 1], P)
        states[v].copy_(R)   # the state block v read
        S[v].copy_(s)
        Y[v].copy_(dev_tensor(wl.make_y(wr, v)))
    torch.cuda.synchronize(dev)
    outs = []
    for v in range(1, L):
        outs.append((torch.empty((N, v), dtype=torch.float32, device=dev),
                     torch.empty((N, v, 4), dtype=torch.float32, device=dev),
                     torch.empty((N, v), dtype=torch.float32, device=dev),
                     torch.empty((N,), dtype=torch.float32, device=dev)))
    lib = gr.load()
    stream = torch.cuda.current_stream(dev)
    shape = gr.make_shape(N, D, r, tdt, w.eps)
    P_ = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731

    def step():
        for v in range(1, L):
            p = params[v]
            o = outs[v - 1]
            st = lib.gr_decompose(ctypes.byref(shape), P_(states[v]), P_(p["gamma"]),
                                  P_(p["w_down"]), P_(p["w_up"]), P_(p["w_write"]), v, P_(Y),
                                  P_(S), P_(R0), P_(o[0]), P_(o[1]), P_(o[2]), P_(o[3]),
                                  ctypes.c_void_p(stream.cuda_stream))
            if st != 0:
                raise RuntimeError(f"gr_decompose: {gr.status_string(st)}")

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    props = torch.cuda.get_device_properties(dev)
    if world > 1:
        dist.barrier()
    sampler = ClockSampler(str(getattr(props, "uuid", "") or ""))
    sampler.start()
    step()   # untimed, queued right before the window: it opens on a busy GPU
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    if gr.device_status(clear=True) != 0:
        raise RuntimeError("device status set during the decomposition")
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    ms_step = ms / args.steps
    alg = decompose_bytes(w, L)
    peaks = load_peaks()
    peak = peaks["hbm_gbs"]
    achieved = alg / (ms_step / 1e3) / 1e9
    if rank == 0:
        line = {
            "metric": f"GR contribution decomposition tokens/s ({L * (L - 1) // 2} block pairs "
                      f"of a {L}-block stack)",
            "value": job_tokens_per_s(world, N, args.steps, ms / 1e3), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic (seeded numpy PCG64; states from the library's "
                                    "own forward chain; no dataset)",
            "config": {"workload": f"{w.name} shape: N={N} tokens, D={D}, r={r}, "
                                   f"{w.dtype} states; {L} blocks, readers 1..{L - 1} each "
                                   f"against all earlier writers and the initial state",
                       "n_tokens_per_gpu": N, "d_model": D, "rank": r, "state_dtype": w.dtype,
                       "blocks": L, "l2": "inputs larger than L2 (writers' outputs "
                                         f"{L * N * D * (2 if w.dtype == 'bf16' else 4) >> 20} "
                                         "MiB), no flush",
                       "pass": "decomposition (gr_decompose per reader)"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak,
                         "traffic": None if args.n_tokens is not None or L != 40
                         else profiled_traffic("decompose", w.name),
                         "peak_source": peaks["source"], "algorithmic_bytes_per_step": alg},
            "gpu_launches": (L - 1) * args.steps,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def e2e_host_entry(args, w, world, dev, stream, tdt, R_h, y_h, sp_h, P) -> dict:
    """End to end through the host-buffer C entry: H2D of R, y, s_prev; D2H of R', x, s_next."""
    import numpy as np
    import torch
    import torch.distributed as dist

    from stream_gated_residual_gb300 import gr
    Rh = torch.from_numpy(R_h.view(np.int16) if R_h.dtype == np.uint16 else R_h)
    yh = torch.from_numpy(y_h.view(np.int16) if y_h.dtype == np.uint16 else y_h)
    if tdt == torch.bfloat16:
        Rh, yh = Rh.view(torch.bfloat16), yh.view(torch.bfloat16)
    Rh, yh = Rh.pin_memory(), yh.pin_memory()
    sph = torch.from_numpy(sp_h).pin_memory()
    xh = torch.empty((w.n_tokens, w.d_model), dtype=tdt).pin_memory()
    snh = torch.empty((w.n_tokens, 4), dtype=torch.float32).pin_memory()
    nws = gr.host_workspace_size(w.n_tokens, w.d_model, tdt)
    wsb = torch.empty(nws + 256, dtype=torch.uint8, device=dev)
    ws = wsb[(-wsb.data_ptr()) % 256:][:nws]
    for _ in range(3):  # warm-up (the first transfers from freshly pinned pages are slow)
        gr.write_then_read_host(Rh, yh, sph, P, xh, snh, ws, stream=stream)
    if world > 1:
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(args.e2e_steps):
        gr.write_then_read_host(Rh, yh, sph, P, xh, snh, ws, stream=stream)
    e2e_s = max_over_ranks(time.perf_counter() - t0, world, dev)
    es = w.state_bytes_per_elem()
    h2d = w.n_tokens * (4 * w.d_model * es + w.d_model * es + 16)
    d2h = h2d
    return {"value": job_tokens_per_s(world, w.n_tokens, args.e2e_steps, e2e_s), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "api": "gr_write_then_read_host (pinned host buffers)"}


def e2e_device_copies(args, w, world, dev, stream, ins, outs, s_prev, s_next, fused,
                      api) -> dict:
    """End to end through the device entry with host buffers: per step, pinned host copies of
    the inputs `ins` go to the device, the step runs, and `outs` come back (torch copies on the
    same stream, not pipelined). For the paths the host-buffer C entry does not take: the FP8
    state and the large-rank path."""
    import torch
    import torch.distributed as dist
    host = [t.cpu().pin_memory() for t in ins]
    hout = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outs]

    def one():
        for h, d in zip(host, ins):
            d.copy_(h, non_blocking=True)
        fused(s_prev, s_next, stream)
        for h, d in zip(hout, outs):
            h.copy_(d, non_blocking=True)
        stream.synchronize()

    for _ in range(3):
        one()
    if world > 1:
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(args.e2e_steps):
        one()
    e2e_s = max_over_ranks(time.perf_counter() - t0, world, dev)
    h2d = sum(t.numel() * t.element_size() for t in ins)
    d2h = sum(t.numel() * t.element_size() for t in outs)
    return {"value": job_tokens_per_s(world, w.n_tokens, args.e2e_steps, e2e_s), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "api": api}


def main(argv=None):
    args = parse_args(argv)
    from stream_gated_residual_gb300 import workloads as wl
    if args.workload is None:
        args.workload = "deep_stack" if args.decompose else "prefill"
    if args.workload not in wl.WORKLOADS:
        raise SystemExit(f"unknown workload {args.workload}; one of {sorted(wl.WORKLOADS)}")
    w = wl.WORKLOADS[args.workload]
    if args.n_tokens is not None:
        if args.n_tokens < 1:
            raise SystemExit("--n-tokens must be >= 1")
        w = w.scaled(n_tokens=args.n_tokens)
    if args.impl == "reference":
        run_reference(args, w)
    elif args.backward:
        run_backward(args, w)
    elif args.decompose:
        run_decompose(args, w)
    else:
        run_gr(args, w)


if __name__ == "__main__":
    main()
