#!/usr/bin/env python
"""Benchmark of the stabilized parallel mLSTM forward on GB300.

One step = the whole parallel hot path over one batch: gate preprocessing
(log-sigmoid prefix sums, prefix-max stabilizer) and the fused causal kernel
(Q K^T, gating, signed row sum, C'V, normalization).  Workload at N=1: the
125M-scale layer, B=8, H=4, T=2048, d_qk=d_v=384, bf16 q/k/v, fp32 gates,
synthetic seeded inputs.  The recurrent generation step (B=256, H=4, d=512,
fp32 state, in place) is timed in the same run and reported beside it.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line on rank 0.  Under torchrun (N > 1) every rank runs the
same per-GPU workload on its own GPU (heads are independent: weak scaling, no
collective on the data path); value = work of all ranks / max time over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mlstm_matrix_memory_gb300 import workloads as W  # noqa: E402

METRIC = "mLSTM parallel fwd causal TFLOP/s + tokens/s at T=2048 (1×GB300, % of peak)"
L2_FLUSH_BYTES = 512 << 20          # > 129 MB L2
# nominal GB300 figures, beside the measured denominators
NOMINAL_BF16_TFLOPS = 2250.0        # dense bf16
NOMINAL_HBM_GBS = 8000.0            # HBM3e


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--workload", default=W.L125M.name, choices=sorted(W.PARALLEL_WORKLOADS))
    p.add_argument("--algo", default="auto", choices=("auto", "tc", "simt"))
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-step", action="store_true", help="skip the recurrent-step measurement")
    p.add_argument("--no-other-configs", action="store_true",
                   help="skip the forward on the other bf16 layer shapes (350M-scale, T=16384)")
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--profile-kernel", choices=("fwd", "fwd_call", "fs", "step", "step_full", "step_seq", "rbwd", "bwd",
                                                "bwd_saved"),
                   default=None,
                   help="no timing: one warm-up and one launch of the fused forward kernel (on --workload), "
                        "of the parallel-to-recurrent hand-off (on --workload), of the recurrent step (B=64, H=4, d=512: 256 MB of state), of the 64-token prefill "
                        "(same heads), of the recurrent backward (B=4, H=8, T=256, d=384) or of the parallel "
                        "backward (on --workload), for ncu captures")
    return p.parse_args()


def dist_setup(n):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, ws: int) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return d["bf16_tflops"], d["hbm_gbs"], "measured"
    except Exception:
        return 1900.0, 6800.0, "fallback"


class Clocks:
    """nvidia-smi sampler of SM clocks and throttle reasons while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.proc = None
        # raw samples: the system temp folder, or MLSTM_CLOCKS_DIR to keep them
        self.path = os.path.join(os.environ.get("MLSTM_CLOCKS_DIR", tempfile.gettempdir()),
                                 f"clocks_bench_{os.getpid()}.csv")
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def kernel_traffic(name: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the kernel source that is built now (else null)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)[name]
        srcs = d["source"] if isinstance(d["source"], list) else [d["source"]]
        h = hashlib.sha256()
        for name_ in srcs:
            h.update(open(os.path.join(ROOT, "mlstm_matrix_memory_gb300", "csrc", name_), "rb").read())
        return d["bytes_per_launch"] if h.hexdigest()[:16] == d["source_sha256_16"] else None
    except Exception:
        return None


def oracle_rows(w, heads: int, stride: int = 8):
    """A bounded sample of the workload for the CPU oracle: every `stride`-th
    query row of `heads` (b,h) sequences.  Returns (inputs, rows, causal
    flops of those rows: 2 (i+1) (d_qk + d_v) per row i)."""
    x = W.parallel_inputs(w, 0, B=1, H=heads)
    rows, flops = [], 0.0
    for bh in range(heads):
        for i in range(stride - 1, w.T, stride):
            rows.append(bh * w.T + i)
            flops += 2.0 * (i + 1) * (w.d_qk + w.d_v)
    return x, rows, flops


def host_cores() -> int:
    """The host cores this process may run on: the oracle's OpenMP team, set
    explicitly (a launcher such as torch.distributed.run exports
    OMP_NUM_THREADS=1 to every rank, while only rank 0 times the oracle)."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_time(x, rows, reps_or_seconds, by_time, threads):
    import oracle
    a = (x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"])
    f = [oracle.f64(t) for t in a]            # widen once, outside the timed region
    n, t0 = 0, time.perf_counter()
    while True:
        oracle.parallel_rows(*f, rows, nthreads=threads)
        n += 1
        el = time.perf_counter() - t0
        if (by_time and el >= reps_or_seconds) or (not by_time and n >= reps_or_seconds):
            return n, el


def cpu_baseline(w, seconds):
    cores = host_cores()
    x, rows, flops = oracle_rows(w, heads=max(1, cores))
    n, el = oracle_time(x, rows, seconds, by_time=True, threads=cores)
    return {"value": n * flops / el / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"every 8th query row of {max(1, cores)} heads of {w.name} (fp64, OpenMP over rows), "
                      f"{n} passes in {el:.1f} s"}


def run_reference(args, ws, rank):
    """The oracle, as it stands, timed on the host cores on a bounded sample of
    the workload per step (rank 0 only)."""
    w = W.PARALLEL_WORKLOADS[args.workload]
    if rank != 0:
        return
    cores = host_cores()
    x, rows, flops = oracle_rows(w, heads=max(1, cores))
    oracle_time(x, rows[: max(1, len(rows) // 16)], args.warmup, by_time=False, threads=cores)
    n, el = oracle_time(x, rows, args.steps, by_time=False, threads=cores)
    ms = el * 1e3 / n
    tflops = flops / (ms * 1e-3) / 1e12
    sample = f"every 8th query row of {max(1, cores)} heads of {w.name} per step (fp64, OpenMP over rows)"
    line = {"impl": "reference", "metric": METRIC, "value": tflops, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "sample": sample, "l2": "n/a (CPU)"},
            "cpu_baseline": {"value": tflops, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": tflops, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def time_parallel(M, w, xd, algo, steps, warmup, flush):
    """The step (gate pass + fused kernel through the public call) timed with
    CUDA events on the launching stream, L2 flushed before every step; then
    the fused kernel alone (gate terms already in the workspace), same way,
    for its roofline."""
    stream = torch.cuda.current_stream()
    B, H, T = w.B, w.H, w.T
    ws = torch.empty(M.parallel_fwd_workspace_bytes(B, H, T), dtype=torch.uint8, device="cuda")
    h = torch.empty((B, H, T, w.d_v), dtype=w.dtype, device="cuda")

    def step():
        M.parallel_fwd(xd["q"], xd["k"], xd["v"], xd["igate_pre"], xd["fgate_pre"], h=h, workspace=ws, algo=algo)

    def timed(fn):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        torch.cuda.synchronize()
        for i in range(steps):
            flush.zero_()
            ev[i][0].record(stream)
            fn()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in ev]

    for _ in range(warmup):
        step()
    step_ms = timed(step)
    fwd_ms = timed(lambda: M.parallel_fwd_gated(xd["q"], xd["k"], xd["v"], ws, h, algo=algo))
    gate_ms = timed(lambda: M.gate_prep(xd["igate_pre"], xd["fgate_pre"], ws))
    if M.last_device_status() != 0:
        raise RuntimeError("device status word set during the timed region")
    return step_ms, fwd_ms, gate_ms


def time_other_parallel(M, w, steps, warmup, flush):
    """The forward (public call) and the fused kernel alone on another bf16
    layer shape, timed as the main workload is."""
    xd = {k: v.cuda() for k, v in W.parallel_inputs(w, 0).items()}
    algo = "tc" if M.tc_supported(w.d_qk, w.d_v, w.dtype) else "simt"
    step_ms, fwd_ms, gate_ms = time_parallel(M, w, xd, algo, steps, warmup, flush)
    del xd
    return statistics.mean(step_ms), statistics.mean(fwd_ms), statistics.mean(gate_ms), algo


def launches_per_step(w, algo):
    """Kernel launches of one forward call: the gate pass and the fused kernel."""
    return 2


def time_e2e(M, w, xh, algo, steps, warmup):
    """Through the public host-buffer call (``mlstm_parallel_fwd_host``): the
    step's inputs in pinned host memory, h returned to pinned host memory,
    uploads, compute and downloads overlapped by chunks of heads inside the
    call, all inside the timed region."""
    stream = torch.cuda.current_stream()
    xp = {k: v.pin_memory() for k, v in xh.items()}
    h_host = torch.empty((w.B, w.H, w.T, w.d_v), dtype=w.dtype).pin_memory()
    ws = torch.empty(M.parallel_fwd_host_workspace_bytes(w.B, w.H, w.T, w.d_qk, w.d_v, w.dtype),
                     dtype=torch.uint8, device="cuda")

    def one():
        M.parallel_fwd_host(xp["q"], xp["k"], xp["v"], xp["igate_pre"], xp["fgate_pre"], h=h_host, workspace=ws)

    for _ in range(warmup):
        one()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        one()
    e1.record(stream)
    torch.cuda.synchronize()
    h2d = sum(v.numel() * v.element_size() for v in xh.values())
    return e0.elapsed_time(e1) / steps, h2d, h_host.numel() * h_host.element_size()


def time_step(M, steps, warmup):
    """The recurrent generation step, B=256, H=4, d=512, state updated in place
    (1 GiB of C read and written per step: larger than L2)."""
    w = W.STEP
    x = W.step_inputs(w, 0)
    xd = {k: v.cuda() for k, v in x.items()}
    stream = torch.cuda.current_stream()
    h = torch.empty((w.B, w.H, w.d_v), dtype=w.dtype, device="cuda")

    def one():
        M.step(xd["C"], xd["n"], xd["m"], xd["q"], xd["k"], xd["v"], xd["igate_pre"], xd["fgate_pre"], xd["o"],
               h=h)

    for _ in range(warmup):
        one()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize()
    for i in range(steps):
        ev[i][0].record(stream)
        one()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    BH = w.B * w.H
    nbytes = (2 * BH * w.d_v * w.d_qk * 4 + 2 * BH * w.d_qk * 4 + 2 * BH * 4   # C, n, m read+write
              + BH * (2 * w.d_qk + 3 * w.d_v) * 2 + 2 * BH * 4)                # q,k,v,o,h (bf16), gates
    return ms, nbytes, w


def time_step_seq(M, reps, L=64):
    """L recurrent steps per head in one call (recurrent prefill), B=256, H=4,
    d=512: the state is read and written once per call."""
    w = W.STEP
    xd = {k: v.cuda() for k, v in W.step_seq_inputs(w, L, 0).items()}
    h = torch.empty((w.B, w.H, L, w.d_v), dtype=w.dtype, device="cuda")
    stream = torch.cuda.current_stream()

    def one():
        M.step_seq(xd["C"], xd["n"], xd["m"], xd["q"], xd["k"], xd["v"], xd["igate_pre"], xd["fgate_pre"],
                   xd["o"], h=h)

    for _ in range(2):
        one()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    torch.cuda.synchronize()
    for i in range(reps):
        ev[i][0].record(stream)
        one()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    flops = 4.0 * w.B * w.H * L * w.d_v * w.d_qk          # rank-one update + C q per token
    return ms, flops, w, L


def time_final_state(M, w, xd, reps, flush):
    """The parallel-to-recurrent hand-off on the parallel workload: (C, n, m)
    after the last token from the gate terms; 2 T d_qk d_v flops per head.
    Device time per call: `reps` calls, each after an L2 flush, queued behind a
    spin kernel long enough for the host to enqueue all of them (a single call
    is shorter than its host-side preparation), less the flushes timed the
    same way."""
    ws_buf = torch.empty(M.parallel_fwd_workspace_bytes(w.B, w.H, w.T), dtype=torch.uint8, device="cuda")
    M.gate_prep(xd["igate_pre"], xd["fgate_pre"], ws_buf)
    stream = torch.cuda.current_stream()
    for _ in range(2):
        M.parallel_final_state(xd["k"], xd["v"], ws_buf)

    def queued(fn):
        torch.cuda.synchronize()
        torch.cuda._sleep(8_000_000)            # a few ms of GPU time ahead of the host
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            flush.zero_()
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    t_flush = min(queued(lambda: None) for _ in range(2))
    ms = min(queued(lambda: M.parallel_final_state(xd["k"], xd["v"], ws_buf)) for _ in range(2)) - t_flush
    # algorithmic bytes: k and v read once, C and n written (fp32), the gate terms read
    nbytes = (w.B * w.H * w.T * (w.d_qk + w.d_v) * w.dtype.itemsize + 4.0 * w.B * w.H * w.d_v * w.d_qk
              + 4.0 * w.B * w.H * w.d_qk + 4.0 * w.B * w.H * w.T)
    return ms, 2.0 * w.B * w.H * w.T * w.d_qk * w.d_v, nbytes


def time_backward(M, w, xd, reps, flush):
    """The parallel backward on the parallel workload for a seeded output
    gradient: algorithmic work T^2 (3 d_qk + 2 d_v) flops per head (the five
    causal products S, dC, dQ, dK, dV).  Also timed given the forward's saved
    outputs (no forward pass inside)."""
    lib = M.library()
    dh = torch.randn((w.B, w.H, w.T, w.d_v), generator=torch.Generator().manual_seed(1)).to(w.dtype).cuda()
    ws_buf = torch.empty(int(lib.mlstm_parallel_bwd_workspace(w.B, w.H, w.T, 1 if w.dtype == torch.bfloat16 else 0)),
                         dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def one():
        M.parallel_bwd(xd["q"], xd["k"], xd["v"], xd["igate_pre"], xd["fgate_pre"], dh, workspace=ws_buf)

    # the same with the forward's saved H~, n and signed b (a training step's backward)
    saved = M.parallel_fwd(xd["q"], xd["k"], xd["v"], xd["igate_pre"], xd["fgate_pre"], return_stats=True)
    saved = (saved[0], saved[2], saved[3])

    def one_saved():
        M.parallel_bwd(xd["q"], xd["k"], xd["v"], xd["igate_pre"], xd["fgate_pre"], dh, workspace=ws_buf,
                       saved=saved)

    def timed(fn):
        for _ in range(2):
            fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        torch.cuda.synchronize()
        for i in range(reps):
            flush.zero_()
            ev[i][0].record(stream)
            fn()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in ev)

    ms = timed(one)
    ms_saved = timed(one_saved)
    return ms, float(w.B * w.H * w.T * w.T * (3 * w.d_qk + 2 * w.d_v)), ws_buf.numel(), ms_saved


def time_recurrent_backward(M, w, xd, reps):
    """The recurrent backward (backpropagation through time) on the parallel
    workload: algorithmic work 12 d_qk d_v flops per token and head (each of
    the two sweeps makes three fused multiply-adds per state entry: the
    state update, the row product and the column product)."""
    lib = M.library()
    dh = torch.randn((w.B, w.H, w.T, w.d_v), generator=torch.Generator().manual_seed(1)).to(w.dtype).cuda()
    ws_buf = torch.empty(int(lib.mlstm_recurrent_bwd_workspace(w.B, w.H, w.T, w.d_qk, w.d_v)), dtype=torch.uint8,
                         device="cuda")
    stream = torch.cuda.current_stream()

    def one():
        M.recurrent_bwd(xd["q"], xd["k"], xd["v"], xd["igate_pre"], xd["fgate_pre"], dh, workspace=ws_buf)

    for _ in range(2):
        one()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    torch.cuda.synchronize()
    for i in range(reps):
        ev[i][0].record(stream)
        one()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    return ms, float(12 * w.B * w.H * w.T * w.d_qk * w.d_v), ws_buf.numel()


def fp32_alu_peak_tflops():
    """FP32 FMA peak of the CUDA cores: SMs x 128 lanes x 2 flops x the
    maximum SM clock from MEASURED_PEAKS.json (else 2070 MHz)."""
    mhz = 2070.0
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            mhz = float(json.load(f).get("sm_max_mhz", mhz))
    except Exception:
        pass
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    return sms * 128 * 2 * mhz * 1e6 / 1e12, sms, mhz


def profile_once(args):
    """One warm-up and one profiled launch of a single kernel (small, L2-exceeding case)."""
    import mlstm_matrix_memory_gb300 as M
    if args.profile_kernel == "fwd":
        w = W.PARALLEL_WORKLOADS[args.workload]
        xd = {k: v.cuda() for k, v in W.parallel_inputs(w, 0).items()}
        ws = torch.empty(M.parallel_fwd_workspace_bytes(w.B, w.H, w.T), dtype=torch.uint8, device="cuda")
        h = torch.empty((w.B, w.H, w.T, w.d_v), dtype=w.dtype, device="cuda")
        M.gate_prep(xd["igate_pre"], xd["fgate_pre"], ws)
        for _ in range(2):
            M.parallel_fwd_gated(xd["q"], xd["k"], xd["v"], ws, h, algo=args.algo)
    elif args.profile_kernel == "fwd_call":
        # the public forward call as the benchmark's step makes it
        w = W.PARALLEL_WORKLOADS[args.workload]
        xd = {k: v.cuda() for k, v in W.parallel_inputs(w, 0).items()}
        ws = torch.empty(M.parallel_fwd_workspace_bytes(w.B, w.H, w.T), dtype=torch.uint8, device="cuda")
        h = torch.empty((w.B, w.H, w.T, w.d_v), dtype=w.dtype, device="cuda")
        for _ in range(2):
            M.parallel_fwd(xd["q"], xd["k"], xd["v"], xd["igate_pre"], xd["fgate_pre"], h=h, workspace=ws,
                           algo=args.algo)
    elif args.profile_kernel == "fs":
        # the parallel-to-recurrent hand-off (final C, n, m) on the parallel workload
        w = W.PARALLEL_WORKLOADS[args.workload]
        xd = {k: v.cuda() for k, v in W.parallel_inputs(w, 0).items()}
        ws = torch.empty(M.parallel_fwd_workspace_bytes(w.B, w.H, w.T), dtype=torch.uint8, device="cuda")
        M.gate_prep(xd["igate_pre"], xd["fgate_pre"], ws)
        for _ in range(2):
            M.parallel_final_state(xd["k"], xd["v"], ws)
    elif args.profile_kernel == "bwd":
        w = W.PARALLEL_WORKLOADS[args.workload]
        xd = {k: v.cuda() for k, v in W.parallel_inputs(w, 0).items()}
        dh = torch.randn((w.B, w.H, w.T, w.d_v), generator=torch.Generator().manual_seed(1)).to(w.dtype).cuda()
        for _ in range(2):
            M.parallel_bwd(xd["q"], xd["k"], xd["v"], xd["igate_pre"], xd["fgate_pre"], dh)
    elif args.profile_kernel == "bwd_saved":
        # the training-step backward: one forward (its launches first), then two
        # backward calls given its saved outputs
        w = W.PARALLEL_WORKLOADS[args.workload]
        xd = {k: v.cuda() for k, v in W.parallel_inputs(w, 0).items()}
        dh = torch.randn((w.B, w.H, w.T, w.d_v), generator=torch.Generator().manual_seed(1)).to(w.dtype).cuda()
        sv = M.parallel_fwd(xd["q"], xd["k"], xd["v"], xd["igate_pre"], xd["fgate_pre"], return_stats=True)
        for _ in range(2):
            M.parallel_bwd(xd["q"], xd["k"], xd["v"], xd["igate_pre"], xd["fgate_pre"], dh, saved=(sv[0], sv[2], sv[3]))
    elif args.profile_kernel == "rbwd":
        # the recurrent backward on 32 heads of the 125M-scale layer's shape, T=256
        x = {k: v.cuda() for k, v in W.sequence_inputs(4, 8, 256, 384, 384, torch.bfloat16, seed=1).items()}
        dh = torch.randn((4, 8, 256, 384), generator=torch.Generator().manual_seed(1)).to(torch.bfloat16).cuda()
        for _ in range(2):
            M.recurrent_bwd(x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"], dh)
    elif args.profile_kernel == "step_seq":
        xd = {k: v.cuda() for k, v in W.step_seq_inputs(W.STEP, 64, 0, B=64).items()}
        for _ in range(2):
            M.step_seq(xd["C"], xd["n"], xd["m"], xd["q"], xd["k"], xd["v"], xd["igate_pre"], xd["fgate_pre"],
                       xd["o"])
    elif args.profile_kernel == "step_full":
        # the benchmark's recurrent step at full size: B=256, H=4, d=512 (1 GiB of state)
        xd = {k: v.cuda() for k, v in W.step_inputs(W.STEP, 0).items()}
        for _ in range(2):
            M.step(xd["C"], xd["n"], xd["m"], xd["q"], xd["k"], xd["v"], xd["igate_pre"], xd["fgate_pre"], xd["o"])
    else:
        xd = {k: v.cuda() for k, v in W.step_inputs(W.STEP, 0, B=64).items()}
        for _ in range(2):
            M.step(xd["C"], xd["n"], xd["m"], xd["q"], xd["k"], xd["v"], xd["igate_pre"], xd["fgate_pre"], xd["o"])
    torch.cuda.synchronize()
    if M.last_device_status() != 0:
        raise RuntimeError("device status word set")
    print("profile run done")


def main():
    args = parse()
    ws, rank, local = dist_setup(args.gpus)
    if args.profile_kernel:
        profile_once(args)
        return
    if args.impl == "reference":
        run_reference(args, ws, rank)
        return
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    from mlstm_matrix_memory_gb300 import build
    if rank == 0:
        build.build()
    barrier(ws)
    import mlstm_matrix_memory_gb300 as M

    w = W.PARALLEL_WORKLOADS[args.workload]
    algo = args.algo
    if algo == "auto":
        algo = "tc" if M.tc_supported(w.d_qk, w.d_v, w.dtype) else "simt"
    xh = W.parallel_inputs(w, seed=rank)
    xh = {k: v.pin_memory() for k, v in xh.items()}
    xd = {k: v.cuda() for k, v in xh.items()}
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    clocks = Clocks(torch.cuda.current_device()) if rank == 0 else None

    barrier(ws)
    torch.cuda.synchronize()
    step_ms, fwd_ms, gate_ms = time_parallel(M, w, xd, algo, args.steps, args.warmup, flush)
    torch.cuda.synchronize()
    barrier(ws)
    t_step = max_over_ranks(statistics.mean(step_ms), ws)
    t_fwd = max_over_ranks(statistics.mean(fwd_ms), ws)
    e2e_ms, h2d, d2h = time_e2e(M, w, xh, algo, max(5, args.steps // 5), 2)
    e2e_ms = max_over_ranks(e2e_ms, ws)
    rec = seq = fs = None
    if not args.no_step:
        rec = time_step(M, max(10, args.steps // 2), 3)
        seq = time_step_seq(M, 5)
    others = {}
    if not args.no_other_configs and w.name == W.L125M.name:
        for key, ow in (("parallel_350m", W.L350M), ("parallel_long", W.LONG)):
            others[key] = (ow, time_other_parallel(M, ow, max(10, args.steps // 2) if ow.T <= 2048 else 10, 3,
                                                   flush))
    bwd = rbwd = None
    if algo == "tc":
        fs = time_final_state(M, w, xd, 10, flush)
        bwd = time_backward(M, w, xd, 5, flush)
        rbwd = time_recurrent_backward(M, w, xd, 3)
    clk = clocks.stop() if clocks else None

    flops = w.causal_flops
    value = ws * flops / (t_step * 1e-3) / 1e12
    peak_tf, peak_bw, src = peaks()
    nlaunch = launches_per_step(w, algo)
    # the dominant kernel: with one launch per step it is the step itself
    # (gate terms computed inside); else the fused kernel timed alone
    t_kern = t_step if nlaunch == 1 else t_fwd
    achieved = flops / (t_kern * 1e-3) / 1e12
    traffic = kernel_traffic("fwd_tc_" + w.name) if algo == "tc" else None
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w.dtype == torch.bfloat16 else "f32",
        "data": "synthetic (seeded N(0,1) q/k/v, N(0,1) input and N(3,1) forget pre-activations)",
        "tokens_per_s": ws * w.tokens / (t_step * 1e-3),
        "frac_of_peak": value / ws / peak_tf,
        "frac_of_nominal_peak": value / ws / NOMINAL_BF16_TFLOPS,
        "config": {"workload": w.name, "B": w.B, "H": w.H, "T": w.T, "d_qk": w.d_qk, "d_v": w.d_v,
                   "kernel": algo, "l2": "flushed before every timed step (512 MB memset)",
                   "parallelism": f"{ws} independent replica(s), heads independent, no collective"},
        "gate_prep_ms_alone": statistics.mean(gate_ms),
        "fused_kernel_ms_alone": statistics.mean(fwd_ms),
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": achieved / peak_tf, "peak_source": f"{src} bf16 dense (burst)",
                     "frac_of_nominal": achieved / NOMINAL_BF16_TFLOPS,
                     "nominal_peak": NOMINAL_BF16_TFLOPS,
                     "traffic": traffic, "kernel": f"mlstm fwd_{algo}",
                     "work": "causal flops T^2 (d_qk+d_v) per head per launch",
                     "timing": ("the step's single launch (gate terms computed in the kernel)" if nlaunch == 1
                                else "fused kernel alone") + ", CUDA events per launch, L2 flushed before each"},
        "e2e": {"value": ws * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": nlaunch * args.steps,
        "launches_per_step": nlaunch,
    }
    if rec is not None:
        ms, nbytes, sw = rec
        gbs = nbytes / (ms * 1e-3) / 1e9
        line["recurrent_step"] = {"workload": sw.name, "ms": ms, "GB_per_s": gbs, "bytes": nbytes,
                                  "tokens_per_s": sw.B / (ms * 1e-3),
                                  "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak_bw,
                                               "unit": "GB/s", "frac": gbs / peak_bw,
                                               "peak_source": f"{src} copy bandwidth",
                                               "frac_of_nominal": gbs / NOMINAL_HBM_GBS,
                                               "nominal_peak": NOMINAL_HBM_GBS,
                                               "traffic": kernel_traffic("step_" + sw.name)}}
    if seq is not None:
        ms, fl, sw, L = seq
        tf = fl / (ms * 1e-3) / 1e12
        alu_peak, sms, mhz = fp32_alu_peak_tflops()
        line["recurrent_prefill"] = {"workload": f"{sw.name}_L{L}", "tokens_per_call": L, "ms": ms,
                                     "tokens_per_s": sw.B * L / (ms * 1e-3),
                                     "roofline": {"bound": "alu", "achieved": tf, "peak": alu_peak,
                                                  "unit": "TFLOP/s", "frac": tf / alu_peak,
                                                  "peak_source": f"FP32 FMA: {sms} SMs x 128 lanes x 2 x {mhz:.0f} MHz",
                                                  "traffic": kernel_traffic(f"step_seq_{sw.name}_L{L}")}}
    for key, (ow, (oms, ofwd, ogate, oalgo)) in others.items():
        fl = ow.causal_flops
        onl = launches_per_step(ow, oalgo)
        tf_step, tf_kern = fl / (oms * 1e-3) / 1e12, fl / ((oms if onl == 1 else ofwd) * 1e-3) / 1e12
        line[key] = {"workload": ow.name, "B": ow.B, "H": ow.H, "T": ow.T, "d_qk": ow.d_qk, "d_v": ow.d_v,
                     "kernel": oalgo, "ms": oms, "TFLOP_per_s": tf_step, "tokens_per_s": ow.tokens / (oms * 1e-3),
                     "frac_of_peak": tf_step / peak_tf, "frac_of_nominal_peak": tf_step / NOMINAL_BF16_TFLOPS,
                     "gate_prep_ms_alone": ogate, "fused_kernel_ms_alone": ofwd, "launches_per_step": onl,
                     "roofline": {"bound": "tensor", "achieved": tf_kern, "peak": peak_tf, "unit": "TFLOP/s",
                                  "frac": tf_kern / peak_tf, "peak_source": f"{src} bf16 dense (burst)",
                                  "frac_of_nominal": tf_kern / NOMINAL_BF16_TFLOPS,
                                  "traffic": kernel_traffic("fwd_tc_" + ow.name) if oalgo == "tc" else None,
                                  "work": "causal flops T^2 (d_qk+d_v) per head per launch"}}
    if fs is not None:
        # The hand-off's arithmetic intensity (flops per algorithmic byte) is
        # below the ridge point of the measured peaks, so its roofline is HBM
        # bandwidth; the tensor fraction is reported beside it.
        ms, fl, nb = fs
        tf = fl / (ms * 1e-3) / 1e12
        gbs = nb / (ms * 1e-3) / 1e9
        ai, ridge = fl / nb, peak_tf * 1e12 / (peak_bw * 1e9)
        if ai < ridge:
            roof = {"bound": "hbm", "achieved": gbs, "peak": peak_bw, "unit": "GB/s", "frac": gbs / peak_bw,
                    "peak_source": f"{src} HBM copy", "frac_of_nominal": gbs / NOMINAL_HBM_GBS}
        else:
            roof = {"bound": "tensor", "achieved": tf, "peak": peak_tf, "unit": "TFLOP/s", "frac": tf / peak_tf,
                    "peak_source": f"{src} bf16 dense (burst)", "frac_of_nominal": tf / NOMINAL_BF16_TFLOPS}
        roof["traffic"] = kernel_traffic("final_state_" + w.name)
        line["final_state"] = {"workload": w.name, "ms": ms, "timing": "device time per call, L2 flushed, calls queued",
                               "flop_per_byte": ai, "ridge_flop_per_byte": ridge, "roofline": roof,
                               "tensor": {"achieved_tflops": tf, "frac": tf / peak_tf,
                                          "frac_of_nominal": tf / NOMINAL_BF16_TFLOPS}}
    if bwd is not None:
        # The backward of a training step: the forward's H~, n and b are saved
        # (mlstm_parallel_bwd_saved) and the call computes the five causal
        # products and the gate gradients.  The call that recomputes the
        # forward first is timed beside it.
        ms_recompute, fl, wsb, ms = bwd
        tf = fl / (ms * 1e-3) / 1e12
        line["backward"] = {"workload": w.name, "ms": ms, "call": "with the forward's saved outputs",
                            "workspace_bytes": wsb, "ms_with_forward_recompute": ms_recompute,
                            "tflops_with_forward_recompute": fl / (ms_recompute * 1e-3) / 1e12,
                            "roofline": {"bound": "tensor", "achieved": tf, "peak": peak_tf, "unit": "TFLOP/s",
                                         "frac": tf / peak_tf, "peak_source": f"{src} bf16 dense (burst)",
                                         "frac_of_nominal": tf / NOMINAL_BF16_TFLOPS,
                                         "work": "causal T^2 (3 d_qk + 2 d_v) per head",
                                         "traffic": kernel_traffic("backward_saved_" + w.name),
                                         "traffic_scope": "all kernels of one call"}}
    if rbwd is not None:
        ms, fl, wsb = rbwd
        tf = fl / (ms * 1e-3) / 1e12
        alu_peak, sms, mhz = fp32_alu_peak_tflops()
        line["recurrent_backward"] = {
            "workload": w.name, "ms": ms, "workspace_bytes": wsb,
            "roofline": {"bound": "alu", "achieved": tf, "peak": alu_peak, "unit": "TFLOP/s", "frac": tf / alu_peak,
                         "peak_source": f"FP32 FMA: {sms} SMs x 128 lanes x 2 x {mhz:.0f} MHz",
                         "work": "12 d_qk d_v per token and head (two sweeps)", "traffic": None}}
    if clk:
        line["clocks"] = clk
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
