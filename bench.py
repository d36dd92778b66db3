#!/usr/bin/env python3
"""Benchmark of the dual-weight GLU GEMV on GB300.

Default workload: glu_gemv at M=1, K=2560, N=9728 (Qwen3.5-4B MLP gate/up),
HF-boundary rounding, 32 independent weight pairs (3.19 GB) cycled so every
call streams its ~100 MB of weights from HBM (inputs larger than L2).

A step is one pass over the cycled layers (one call per layer), captured
once as a CUDA graph and replayed, as a decode step replays its graph.
Metric: achieved HBM GB/s of algorithmic bytes (both weights once, h, out),
plus us/call.  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mine|reference]
                  [--workload NAME] [--M M] [--mode fused|hf] [--layers L]
Under torchrun every rank runs its own replica (weak scaling, no collective
on the data path); the timing is max over ranks.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import glu_inputs as gi  # noqa: E402

NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
# mbglu_last_variant() -> the kernel that streams the weights
ROW_BLOCKS = 7   # mbglu_last_variant() of a batch above one pass's rows, run as row blocks
TCGEN05 = 9      # mbglu_last_variant() of a batch above 16 rows in one pass on the tcgen05 kernel
BLOCK_M = 16     # batch rows per pass over the weights (MBGLU_BLOCK_M in include/mbglu.h)


def row_blocks(w, M):
    """Row blocks (passes over the weights) of one call of workload w at M
    rows: glu_gemv takes a batch above 16 rows in one pass (the tcgen05
    kernel, on the aligned operands the bench uses); add_rmsnorm_glu runs it
    as row blocks of 16."""
    return -(-M // BLOCK_M) if w.op == "add_rmsnorm_glu" and M > BLOCK_M else 1
KERNEL_NAMES = {1: "glu_stream_kernel", 2: "glu_generic_kernel", 4: "glu_mma_kernel", 5: "silu_mul_kernel",
                9: "glu_tc_kernel (tcgen05)", 10: "glu_slice_kernel",
                6: "gdn_gates_kernel",
                8: "glu_backward (the forward kernel with the dG/dU epilogue, then glu_bwd_mma_kernel at "
                   "M = 3-8 or glu_bwd_hw_kernel at M <= 2, and glu_bwd_h_reduce8_kernel)"}
KERNEL_SOURCES = ["memory_bound_glu_gb300/csrc/glu_kernels.cuh", "memory_bound_glu_gb300/csrc/ptx.cuh",
                  "memory_bound_glu_gb300/csrc/mbglu_api.cu", "memory_bound_glu_gb300/csrc/glu_backward.cuh",
                  "memory_bound_glu_gb300/csrc/glu_tc.cuh", "memory_bound_glu_gb300/csrc/tcgen05.cuh",
                  "memory_bound_glu_gb300/csrc/glu_slice.cuh"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["mine", "reference"], default="mine")
    ap.add_argument("--workload", default=gi.HEADLINE, choices=sorted(gi.WORKLOADS))
    ap.add_argument("--M", type=int, default=None)
    ap.add_argument("--mode", default=None, choices=["fused", "hf"])
    ap.add_argument("--layers", type=int, default=None)
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--norm-kernels", type=int, default=1, choices=[1, 2],
                    help="add_rmsnorm_glu as one kernel (workspace entry point) or as two")
    ap.add_argument("--split", action="store_true",
                    help="under torchrun: split each layer column-parallel over N (rank p streams rows "
                         "column_shard(N, P, p) of both weights and writes its columns of out; strong scaling, "
                         "no collective); default: one whole replica per rank (weak scaling)")
    ap.add_argument("--policy", type=int, default=None, choices=[0, 1, 2],
                    help="launch policy (default: the library's, 2 = PDL + weight prefetch)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _code_only(text: str) -> str:
    """C/C++ source without comments and with whitespace collapsed: what the
    compiler sees, so that editing a comment does not mark a profile stale."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == '"':                                   # string literal, kept verbatim
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash():
    """Hash of the kernel sources' code (comments and whitespace ignored)."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload, M, mode):
    """(current, last): DRAM bytes per launch from the committed ncu summary.
    current is the figure if the kernel sources still hash to what was
    profiled, else None; last describes the newest capture either way (None
    if the workload was never captured)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
    except Exception:
        return None, None
    rec = d.get(f"{workload}/M{M}/{mode}")
    if not rec:
        return None, None
    same = rec.get("source_hash") == kernel_source_hash()
    last = {"dram_bytes_per_launch": rec.get("dram_bytes_per_launch"), "kernel": rec.get("kernel"),
            "source_hash": rec.get("source_hash"), "sources_changed_since": not same}
    return (rec.get("dram_bytes_per_launch") if same else None), last


def smi_id(local):
    """The nvidia-smi id of this process's CUDA device `local`: its entry in
    CUDA_VISIBLE_DEVICES when that variable remaps the devices (an index or a
    UUID, both of which nvidia-smi --id takes), else `local` itself."""
    ids = [x.strip() for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x.strip()]
    return ids[local] if 0 <= local < len(ids) else str(local)


class ClockSampler:
    """nvidia-smi samples during the timed region (200 ms period)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, t0, t1):
        if not self.proc:
            return None
        time.sleep(0.3)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in self.lines:
            if not (t0 <= ts <= t1 + 0.25):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power) if power else None}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def sum_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# CPU baseline: the oracle as it stands, on a bounded sample
# ---------------------------------------------------------------------------

def oracle_sample_rate(w, M, mode, seconds, max_rows=None):
    """Times oracle calls on row slices of layer 0 until `seconds` pass.
    Returns (GB/s of algorithmic bytes, description, threads)."""
    import oracle
    threads = oracle.default_threads()
    if w.op == "silu_mul":
        return _oracle_silu_mul_rate(w, M, mode, seconds)
    if w.op == "gdn_gates":
        return _oracle_gdn_rate(w, M, seconds)
    g, u = gi.layer_weights(w, 0)
    gb, ub = gi.bits(g), gi.bits(u)
    rows = w.N if max_rows is None else min(w.N, max_rows)
    gb, ub = np.ascontiguousarray(gb[:rows]), np.ascontiguousarray(ub[:rows])
    if w.op == "glu_gemv":
        hb = gi.bits(gi.hidden(w, M))
        call = lambda: oracle.glu_gemv(hb, gb, ub, mode, nthreads=threads)  # noqa: E731
        per_call = 2 * rows * w.K * 2 + M * w.K * 2 + M * rows * 2
    elif w.op == "glu_backward":
        hb = gi.bits(gi.hidden(w, M))
        db = np.ascontiguousarray(gi.bits(gi.upstream(w, M))[:, :rows])
        call = lambda: oracle.glu_backward(hb, gb, ub, db, nthreads=threads)  # noqa: E731
        per_call = 4 * rows * w.K * 2 + 2 * M * w.K * 2 + M * rows * 2
    else:
        x, r, nw = (gi.bits(t) for t in gi.norm_inputs(w, M))
        call = lambda: oracle.add_rmsnorm_glu(x, r, nw, w.eps, gb, ub, mode, nthreads=threads)  # noqa: E731
        per_call = 2 * rows * w.K * 2 + 3 * M * w.K * 2 + w.K * 2 + M * rows * 2
    call()  # warm
    n, t0 = 0, time.perf_counter()
    while True:
        call()
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    desc = (f"{n} oracle calls of {w.op} M={M} K={w.K} N={rows} ({mode}) on layer 0 "
            f"(rows 0..{rows - 1} of {w.N}), {threads} threads, {el:.1f} s")
    return per_call * n / el / 1e9, desc, threads, el / n, per_call


def _oracle_silu_mul_rate(w, M, mode, seconds, rows=64):
    """silu_mul: the oracle (single-threaded C) on the first `rows` tokens of
    input 0, repeated until `seconds` pass."""
    import oracle
    xb = gi.bits(gi.projections(w, min(M, rows), 0))
    per_call = xb.shape[0] * 3 * w.N * 2
    oracle.silu_mul(xb, mode)
    n, t0 = 0, time.perf_counter()
    while True:
        oracle.silu_mul(xb, mode)
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    desc = (f"{n} oracle calls of silu_mul on tokens 0..{xb.shape[0] - 1} of input 0 (of M={M}), N={w.N}, "
            f"{mode} mode, 1 thread, {el:.1f} s")
    return per_call * n / el / 1e9, desc, 1, el / n, per_call


def _oracle_gdn_rate(w, T, seconds, tokens=4096):
    """gdn_gates: the oracle (single-threaded C) on the first `tokens` tokens of
    input 0, repeated until `seconds` pass."""
    import oracle
    a, b, A_log, dt = gi.gdn_inputs(w, min(T, tokens), 0)
    ab, bb, An, dn = gi.bits(a), gi.bits(b), A_log.numpy(), dt.numpy()
    per_call = w.algorithmic_bytes(ab.shape[0])
    oracle.gdn_gates(ab, bb, An, dn)
    n, t0 = 0, time.perf_counter()
    while True:
        oracle.gdn_gates(ab, bb, An, dn)
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    desc = (f"{n} oracle calls of gdn_gates on tokens 0..{ab.shape[0] - 1} of input 0 (of T={T}), H={w.N}, "
            f"1 thread, {el:.1f} s")
    return per_call * n / el / 1e9, desc, 1, el / n, per_call


def run_reference(args, w, M, mode, world, rank):
    """Reference arm: the fp64 oracle on the host cores, bounded steps."""
    if rank != 0:
        return
    steps, warm = max(1, args.steps), max(0, args.warmup)
    import oracle
    if w.op == "silu_mul":
        return _reference_silu_mul(args, w, M, mode, world, steps, warm)
    if w.op == "gdn_gates":
        v, desc, thr, el, _ = _oracle_gdn_rate(w, M, max(1.0, 60.0 / (steps + warm)))
        line = {
            "impl": "reference", "metric": "GLU GEMV achieved HBM GB/s (cold L2), us/call at M=1",
            "value": round(v, 4), "unit": "GB/s", "higher_is_better": True, "n_gpus": world,
            "steps": steps, "warmup": warm, "ms_per_step": round(el * 1e3, 4),
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(w, M, mode, w.layers, blocks=row_blocks(w, M)),
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": thr, "kind": "oracle", "sample": desc},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }
        print(json.dumps(line), flush=True)
        return
    g, u = gi.layer_weights(w, 0)
    threads = oracle.default_threads()
    # size the per-step row sample so the whole run stays within ~2 minutes
    hb = gi.bits(gi.hidden(w, M)) if w.op in ("glu_gemv", "glu_backward") else None
    db = gi.bits(gi.upstream(w, M)) if w.op == "glu_backward" else None
    probe_rows = min(w.N, 256)
    t0 = time.perf_counter()
    if w.op == "glu_backward":
        oracle.glu_backward(hb, gi.bits(g[:probe_rows]), gi.bits(u[:probe_rows]),
                            np.ascontiguousarray(db[:, :probe_rows]), nthreads=threads)
    else:
        oracle.glu_gemv(hb if hb is not None else gi.bits(gi.norm_inputs(w, M)[0]),
                        gi.bits(g[:probe_rows]), gi.bits(u[:probe_rows]), mode, nthreads=threads)
    per_row = (time.perf_counter() - t0) / probe_rows
    budget = 120.0 / (steps + warm)
    rows = int(max(8, min(w.N, budget / max(per_row, 1e-9))))
    gb, ub = np.ascontiguousarray(gi.bits(g)[:rows]), np.ascontiguousarray(gi.bits(u)[:rows])
    if w.op == "glu_gemv":
        call = lambda: oracle.glu_gemv(hb, gb, ub, mode, nthreads=threads)  # noqa: E731
        per_step = 2 * rows * w.K * 2 + M * w.K * 2 + M * rows * 2
    elif w.op == "glu_backward":
        dr = np.ascontiguousarray(db[:, :rows])
        call = lambda: oracle.glu_backward(hb, gb, ub, dr, nthreads=threads)  # noqa: E731
        per_step = 4 * rows * w.K * 2 + 2 * M * w.K * 2 + M * rows * 2
    else:
        x, r, nw = (gi.bits(t) for t in gi.norm_inputs(w, M))
        call = lambda: oracle.add_rmsnorm_glu(x, r, nw, w.eps, gb, ub, mode, nthreads=threads)  # noqa: E731
        per_step = 2 * rows * w.K * 2 + 3 * M * w.K * 2 + w.K * 2 + M * rows * 2
    for _ in range(warm):
        call()
    t0 = time.perf_counter()
    for _ in range(steps):
        call()
    el = time.perf_counter() - t0
    value = per_step * steps / el / 1e9
    sample = (f"each step: one oracle call of {w.op} M={M} K={w.K} on rows 0..{rows - 1} of layer 0 "
              f"(of N={w.N}), {mode} mode")
    line = {
        "impl": "reference", "metric": "GLU GEMV achieved HBM GB/s (cold L2), us/call at M=1",
        "value": round(value, 4), "unit": "GB/s", "higher_is_better": True, "n_gpus": world,
        "steps": steps, "warmup": warm, "ms_per_step": round(el / steps * 1e3, 4),
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(w, M, mode, w.layers, blocks=row_blocks(w, M)),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _reference_silu_mul(args, w, M, mode, world, steps, warm):
    import oracle
    rows = min(M, 64)
    xb = gi.bits(gi.projections(w, rows, 0))
    for _ in range(warm):
        oracle.silu_mul(xb, mode)
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle.silu_mul(xb, mode)
    el = time.perf_counter() - t0
    value = rows * 3 * w.N * 2 * steps / el / 1e9
    line = {
        "impl": "reference", "metric": "GLU GEMV achieved HBM GB/s (cold L2), us/call at M=1",
        "value": round(value, 4), "unit": "GB/s", "higher_is_better": True, "n_gpus": world,
        "steps": steps, "warmup": warm, "ms_per_step": round(el / steps * 1e3, 4),
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(w, M, mode, w.layers, blocks=row_blocks(w, M)),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"each step: one oracle call of silu_mul on tokens 0..{rows - 1} (of M={M}), "
                                   f"N={w.N}, {mode} mode"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_dict(w, M, mode, layers, norm_kernels=None, blocks=1, policy=None):
    """The workload description; `policy` is the library's launch policy name
    (the GPU arm only: the reference arm never loads the library)."""
    wb = w.input_bytes(M) * layers
    extra = {} if w.op == "glu_gemv" or norm_kernels is None else {"norm_kernels": norm_kernels}
    if blocks > 1:
        extra["row_blocks"] = blocks
    return {"workload": w.name, "op": w.op, "M": M, "K": w.K, "N": w.N,
            "mode": None if w.op == "gdn_gates" else mode, "layers": layers, **extra,
            "l2": f"inputs larger than L2: {layers} cycled {'inputs' if w.op in ('silu_mul', 'gdn_gates') else 'weight pairs'}, "
                  f"{wb / 1e9:.2f} GB",
            "launch": f"one CUDA graph of {layers} calls per step",
            **({"launch_policy": policy} if policy else {})}


POLICY_NAMES = {0: "serial", 1: "pdl", 2: "pdl+weight-prefetch"}


# ---------------------------------------------------------------------------
# my arm
# ---------------------------------------------------------------------------

def main():
    args = parse()
    w = gi.WORKLOADS[args.workload]
    M = args.M if args.M is not None else w.Ms[0]
    mode = args.mode or w.modes[0]
    L = args.layers or w.layers
    world, rank, local = dist_setup()

    if args.impl == "reference":
        run_reference(args, w, M, mode, world, rank)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    import memory_bound_glu_gb300 as mb
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    mb.lib()
    if args.policy is not None:
        mb.set_launch_policy(args.policy)

    # the column split: this rank's rows of both weights, its columns of out
    split = args.split and w.op in ("glu_gemv", "add_rmsnorm_glu")
    lo, hi = mb.column_shard(w.N, world, rank) if split else (0, w.N)

    # inputs: resident in HBM before the timed region
    gates, ups = [], []
    for layer in range(L if w.op in ("glu_gemv", "add_rmsnorm_glu", "glu_backward") else 0):
        g, u = gi.layer_weights(w, layer)
        gates.append(g[lo:hi].contiguous().to(dev))
        ups.append(u[lo:hi].contiguous().to(dev))
        del g, u
    if w.op == "silu_mul":
        xs_cpu = [gi.projections(w, M, layer) for layer in range(L)]
        xs = [t.to(dev) for t in xs_cpu]
    elif w.op == "gdn_gates":
        gdn_cpu = [gi.gdn_inputs(w, M, layer) for layer in range(L)]
        gdn = [tuple(t.to(dev) for t in four) for four in gdn_cpu]
        gs = [torch.empty((M, w.N), dtype=torch.float32, device=dev) for _ in range(L)]
    elif w.op == "glu_gemv":
        h_cpu = gi.hidden(w, M)
        h = h_cpu.to(dev)
    elif w.op == "glu_backward":
        h_cpu, d_cpu = gi.hidden(w, M), gi.upstream(w, M)
        h, dout = h_cpu.to(dev), d_cpu.to(dev)
        grad_gates = [torch.empty((w.N, w.K), dtype=torch.bfloat16, device=dev) for _ in range(L)]
        grad_ups = [torch.empty((w.N, w.K), dtype=torch.bfloat16, device=dev) for _ in range(L)]
        grad_hs = torch.empty((L, M, w.K), dtype=torch.bfloat16, device=dev)
        bws = torch.empty(mb.lib().glu_backward_workspace_bytes(M, w.N, w.K), dtype=torch.uint8, device=dev)
    else:
        x_cpu, r_cpu, nw_cpu = gi.norm_inputs(w, M)
        x, nw = x_cpu.to(dev), nw_cpu.to(dev)
        residuals = [r_cpu.to(dev) for _ in range(L)]
    outs = torch.empty((L, M, w.N), dtype=torch.bfloat16, device=dev)
    single = w.op == "add_rmsnorm_glu" and args.norm_kernels == 1
    ws = mb.new_workspace(dev) if single else None
    # a batch above one pass's rows runs as row blocks, one GEMV launch each
    blocks = row_blocks(w, M)
    block_rows = [min(BLOCK_M, M - m0) for m0 in range(0, M, BLOCK_M)] if blocks > 1 else [M]
    launches_per_call = blocks * (2 if (w.op == "add_rmsnorm_glu" and not single) else 1)
    if w.op == "glu_backward":   # dG/dU per 16-row block, grad_h and its reduce per 8-row pass, the weight gradients
        launches_per_call = -(-M // 16) + 2 * (-(-M // 8)) + 1

    def one_step():
        for i in range(L):
            if w.op == "silu_mul":
                mb.silu_mul(xs[i], out=outs[i], mode=mode)
            elif w.op == "gdn_gates":
                mb.gdn_gates(gdn[i][0], gdn[i][1], gdn[i][2], gdn[i][3], g=gs[i], beta=outs[i])
            elif w.op == "glu_gemv":
                mb.glu_gemv(h, gates[i], ups[i], out=outs[i][:, lo:hi], mode=mode)
            elif w.op == "glu_backward":
                mb.glu_backward(h, gates[i], ups[i], dout, grad_h=grad_hs[i], grad_gate=grad_gates[i],
                                grad_up=grad_ups[i], workspace=bws)
            else:
                mb.add_rmsnorm_glu(x, residuals[i], nw, w.eps, gates[i], ups[i], out=outs[i][:, lo:hi], mode=mode,
                                   workspace=ws)

    stream = torch.cuda.Stream(dev)
    stream.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(stream):
        one_step()  # first calls initialise the library's per-device table before capture
        torch.cuda.synchronize(dev)
        variant = mb.last_variant()
        if variant == TCGEN05:      # the whole batch in one pass: one launch per call
            blocks, block_rows, launches_per_call = 1, [M], 1
        if variant == ROW_BLOCKS:   # the kernel of a full block: one call on the first block's rows
            blocks = -(-M // BLOCK_M)
            block_rows = [min(BLOCK_M, M - m0) for m0 in range(0, M, BLOCK_M)]
            launches_per_call = blocks * (2 if (w.op == "add_rmsnorm_glu" and not single) else 1)
            if w.op == "glu_gemv":
                mb.glu_gemv(h[:block_rows[0]], gates[0], ups[0], out=outs[0, :block_rows[0], lo:hi], mode=mode)
            else:
                r_probe = residuals[0][:block_rows[0]].clone()
                mb.add_rmsnorm_glu(x[:block_rows[0]], r_probe, nw, w.eps, gates[0], ups[0],
                                   out=outs[0, :block_rows[0], lo:hi], mode=mode, workspace=ws)
            torch.cuda.synchronize(dev)
            variant = mb.last_variant()
        kernel_name = KERNEL_NAMES.get(variant, f"variant {variant}")
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            one_step()
    torch.cuda.synchronize(dev)

    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            graph.replay()
    torch.cuda.synchronize(dev)

    sampler = ClockSampler(smi_id(local))
    t_load0 = None
    if not args.no_clocks:
        sampler.start()
        time.sleep(0.5)
        # a load window of >= 1.5 s of the same replays right before the timed
        # region, so that the 200 ms clock samples see the GPU under this load
        # even when the timed region itself is a few milliseconds
        t_load0 = time.time()
        with torch.cuda.stream(stream):
            while time.time() - t_load0 < 1.5:
                for _ in range(20):
                    graph.replay()
                torch.cuda.synchronize(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    start.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(args.steps):
            graph.replay()
    end.record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    barrier(world)
    ms = start.elapsed_time(end)
    clocks = None if args.no_clocks else sampler.stop(t_load0, t_wall1)
    if clocks is not None:
        clocks["window"] = (f"nvidia-smi every 200 ms over a {t_wall1 - t_load0:.2f} s load window: "
                            f"{t_wall0 - t_load0:.2f} s of the same graph replays, then the timed region")
    ms_max = max_over_ranks(ms, world, dev)
    err = mb.read_device_error()
    if err:
        raise RuntimeError(f"device error word {err} after the timed region")

    # isolated launches: one call at a time (eager, the stream synchronised on
    # both sides), each on the next cycled layer so that its inputs are cold;
    # the chained figure above lets each call's ramp overlap the previous
    # call's tail (programmatic dependent launch), this one does not
    iso = []
    with torch.cuda.stream(stream):
        for rep in range(max(2, min(L, 16)) * 2):
            i = rep % L
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(dev)
            # a short device-side sleep first, so that the host has enqueued the
            # call (descriptors encoded, launched) before the start event is
            # reached: the two events then bracket the call's device time only
            torch.cuda._sleep(200000)
            e0.record(stream)
            if w.op == "glu_gemv":
                mb.glu_gemv(h, gates[i], ups[i], out=outs[i][:, lo:hi], mode=mode)
            elif w.op == "add_rmsnorm_glu":
                mb.add_rmsnorm_glu(x, residuals[i], nw, w.eps, gates[i], ups[i], out=outs[i][:, lo:hi], mode=mode,
                                   workspace=ws)
            else:
                break
            e1.record(stream)
            torch.cuda.synchronize(dev)
            if rep >= 2:   # the first two warm the launch path
                iso.append(e0.elapsed_time(e1) * 1e3)
    iso_us = statistics.median(iso) if iso else None

    def call_bytes(m):
        """Algorithmic bytes of this rank's call on m rows (its shard of N
        under the column split)."""
        if not split:
            return w.algorithmic_bytes(m)
        n = hi - lo
        if w.op == "glu_gemv":
            return 2 * n * w.K * 2 + m * w.K * 2 + m * n * 2
        return 2 * n * w.K * 2 + 3 * m * w.K * 2 + w.K * 2 + m * n * 2

    bytes_per_call = call_bytes(M)
    calls = args.steps * L
    us_per_call = ms_max * 1e3 / calls
    gbs = bytes_per_call / (us_per_call * 1e-6) / 1e9
    # the dominant kernel's roofline: per launch, the algorithmic bytes of the
    # rows it takes (each block streams both weights) over the mean launch
    # time; with one launch per call this is the call's own figure
    gemv_launch_bytes = sum(call_bytes(m) for m in block_rows)
    launch_gbs = gemv_launch_bytes / (us_per_call * 1e-6) / 1e9
    # the whole job's bytes per call: every rank's shard of the layer under
    # the column split, every replica otherwise
    job_bytes_per_call = sum_over_ranks(bytes_per_call, world, dev) if split else bytes_per_call * world
    value = job_bytes_per_call / (us_per_call * 1e-6) / 1e9
    peak, peak_kind = measured_peaks()

    # e2e: the public Python API, pinned host input -> device, results -> host
    e2e = None
    e2e_steps = min(args.e2e_steps, 10) if w.op in ("silu_mul", "gdn_gates") else args.e2e_steps   # 100s of MB
    if e2e_steps > 0:
        if w.op == "gdn_gates":
            ab_host = [(t[0].pin_memory(), t[1].pin_memory()) for t in gdn_cpu]
            in_bytes = sum(x.numel() + y.numel() for x, y in ab_host) * 2
        elif w.op == "silu_mul":
            xs_host = [t.pin_memory() for t in xs_cpu]
            in_bytes = sum(t.numel() for t in xs_host) * 2
        elif w.op == "glu_gemv":
            h_host = h_cpu.pin_memory()
            in_bytes = h_host.numel() * 2
        elif w.op == "glu_backward":
            h_host, d_host = h_cpu.pin_memory(), d_cpu.pin_memory()
            in_bytes = (h_host.numel() + d_host.numel()) * 2
        else:
            x_host = x_cpu.pin_memory()
            r_host = r_cpu.pin_memory()
            in_bytes = (x_host.numel() + r_host.numel() * L) * 2
        # the step's result read back: out, or for the backward grad_h (the
        # weight gradients stay on the device, where an optimizer uses them)
        result = grad_hs if w.op == "glu_backward" else outs
        out_host = torch.empty(tuple(result.shape), dtype=torch.bfloat16).pin_memory()

        def e2e_step():
            if w.op == "gdn_gates":
                for i in range(L):
                    gdn[i][0].copy_(ab_host[i][0], non_blocking=True)
                    gdn[i][1].copy_(ab_host[i][1], non_blocking=True)
            elif w.op == "silu_mul":
                for i in range(L):
                    xs[i].copy_(xs_host[i], non_blocking=True)
            elif w.op == "glu_gemv":
                h.copy_(h_host, non_blocking=True)
            elif w.op == "glu_backward":
                h.copy_(h_host, non_blocking=True)
                dout.copy_(d_host, non_blocking=True)
            else:
                x.copy_(x_host, non_blocking=True)
                for i in range(L):
                    residuals[i].copy_(r_host, non_blocking=True)
            one_step()
            out_host.copy_(result, non_blocking=True)

        with torch.cuda.stream(stream):
            for _ in range(5):
                e2e_step()
            torch.cuda.synchronize(dev)
            barrier(world)
            t0 = time.perf_counter()
            for _ in range(e2e_steps):
                e2e_step()
            torch.cuda.synchronize(dev)
            el = max_over_ranks(time.perf_counter() - t0, world, dev)
            barrier(world)
        e2e = {"value": round(job_bytes_per_call * L * e2e_steps / el / 1e9, 2), "unit": "GB/s",
               "h2d_bytes_per_step": in_bytes, "d2h_bytes_per_step": out_host.numel() * 2,
               "ms_per_step": round(el / e2e_steps * 1e3, 4),
               "how": "eager public-API calls (no graph), host copies inside the timed region"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, desc, thr, _, _ = oracle_sample_rate(w, M, mode, args.cpu_seconds)
        cpu = {"value": round(v, 4), "unit": "GB/s", "cores": thr, "kind": "oracle", "sample": desc}

    if rank == 0:
        traffic, traffic_last = recorded_traffic(w.name, M, mode)
        line = {
            "metric": "GLU GEMV achieved HBM GB/s (cold L2), us/call at M=1",
            "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": round(ms_max / args.steps, 5),
            "higher_is_better": True, "scaling": "strong" if split else "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded torch.randn, bf16)",
            "config": {**config_dict(w, M, mode, L, args.norm_kernels, blocks, POLICY_NAMES[mb.get_launch_policy()]),
                       "parallelism": (f"column split over N: {world} ranks, rows {lo}..{hi - 1} on rank 0"
                                       if split else f"{world} independent replica(s)")},
            "us_per_call": round(us_per_call, 3), "bytes_per_call": bytes_per_call,
            "frac_of_nominal_8tbs": round(gbs / NOMINAL_HBM_GBS, 4),
            "roofline": {"bound": "hbm", "achieved": round(launch_gbs, 2), "peak": peak, "unit": "GB/s",
                         "frac": round(launch_gbs / peak, 4), "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                         if peak_kind == "measured" else "fallback 6.8 TB/s",
                         "traffic": traffic, "traffic_last_capture": traffic_last, "kernel": kernel_name,
                         "isolated": ({"us_per_launch": round(iso_us, 3),
                                       "achieved": round(gemv_launch_bytes / (iso_us * 1e-6) / 1e9, 2),
                                       "frac": round(gemv_launch_bytes / (iso_us * 1e-6) / 1e9 / peak, 4),
                                       "how": "median CUDA-event time of single calls, stream synchronised on both "
                                              "sides and the call enqueued behind a device sleep before the start "
                                              "event, cycled (cold) layers"} if iso_us else None),
                         "achieved_how": "algorithmic bytes per launch / (CUDA-event time of the timed "
                                         "graph replays / launches): calls chained in one graph with "
                                         "programmatic dependent launch"
                                         + (f"; {blocks} row blocks per call, each streaming both weights"
                                            if blocks > 1 else "")},
            "gpu_launches": calls * launches_per_call,
            "clocks": clocks, "e2e": e2e, "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
