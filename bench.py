"""Benchmark of the fused causal attention forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one forward (attn_fwd through the C ABI) over the long-context
causal workload B=1, H=32, S=16384, D=128 (bf16 in, fp32 accumulate, bf16 out
+ fp32 lse), inputs resident in HBM.  The inputs (403 MB) exceed the 129 MB L2,
so no flush is needed between steps.  Prints one JSON line (rank 0).

Under torchrun (N > 1) the job is one global problem of N times the
workload's batch, split by (batch, head) slices over the ranks with
attn_shard_range (one process per GPU, no exchange step: every slice is
independent); rank r holds batch block r, drawn with seed r, so rank 0's
inputs are the N = 1 workload's.  Timing is bracketed by a barrier +
synchronize on both sides and the max over ranks is taken ("scaling":
"weak": the work per GPU is fixed).

--impl reference times the fp64 CPU oracle on the host cores instead (each
step a bounded sample of query rows of the same workload), rank 0 only.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import threading
import time

import numpy as np
import torch

from exact_attention_68_gb300.workloads import (WORKLOADS, Workload, algorithmic_bytes,
                                                counted_flops, default_scale, make_qkv)

ROOT = os.path.dirname(os.path.abspath(__file__))
METRIC = "causal bf16 attention fwd TFLOP/s on 1 GB300 and % of dense-BF16 peak"
WORKLOAD = "c5"
# The forward kernels' device code (the one-Q-tile kernel runs the causal
# D=128 workload, the two-tile kernel the non-causal and D=64 side workloads)
# and the two-tile kernel's grid schedule (schedule.h).
KERNEL_SOURCES = ["exact_attention_68_gb300/csrc/attn_fwd_1qp_sm103.cu",
                  "exact_attention_68_gb300/csrc/attn_fwd_1q_sm103.cu",
                  "exact_attention_68_gb300/csrc/ptx.cuh", "exact_attention_68_gb300/csrc/umma.cuh",
                  "exact_attention_68_gb300/csrc/attn_fwd.h", "exact_attention_68_gb300/csrc/schedule.h"]
# DRAM bytes (read + write) per launch of the forward kernel on the default
# workload, from ncu captures, keyed by the hash of the kernel sources they
# were taken on (a changed kernel reports null until captured again).
NCU_TRAFFIC_BYTES = {
    # B=1 H=32 S=16384 D=128 causal (attn_fwd_1qp_kernel<128,true,bf16>):
    # 441,948,928 read + 113,420,544 written
    "5323868f1f83d203": 555369472,
}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def kernel_hash() -> str:
    """Hash of the kernel sources with // comments and blank lines left out."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), encoding="utf-8") as fh:
            for line in fh:
                code = line.split("//", 1)[0].rstrip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi every 20 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.samples = []  # (t, sm_mhz, max_mhz, power, {reason: active})
        self.proc = None
        self.thread = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "20"]
        if gpu_id:
            cmd += ["-i", gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm, mx = float(parts[1]), float(parts[2])
                pw = float(parts[3]) if parts[3] not in ("[N/A]", "N/A") else None
            except ValueError:
                continue
            reasons = {n: v.strip().lower() in ("active", "1") for n, v in zip(names, parts[5:9])}
            self.samples.append((time.time(), sm, mx, pw, reasons))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        used = inside if inside else [s for s in self.samples if s[0] >= t0 - 1.0]
        if not used:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = sorted({n for s in used for n, a in s[4].items() if a})
        pw = [s[3] for s in used if s[3] is not None]
        return {"sm_mhz": statistics.median(s[1] for s in used), "sm_max_mhz": max(s[2] for s in used),
                "reasons": reasons, "samples": len(used), "in_timed_region": bool(inside),
                "power_w_max": max(pw) if pw else None}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def reduce_max(x: float, world: int, device) -> float:
    """Max over ranks of a host float (the timing reduction; no data-path collective)."""
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def parity_of_outputs(checked, out, lse):
    """The benchmark's outputs (those of its last end-to-end step, which the
    tests show equal the device path's bit for bit) on the rows the CPU
    baseline computed, against the oracle's values, with the parity tests' bars."""
    idx = np.concatenate([c[0] for c in checked])
    ro = np.concatenate([c[1] for c in checked])
    rl = np.concatenate([c[2] for c in checked])
    b, h, r = (torch.from_numpy(idx[:, n]) for n in range(3))
    og = out.cpu()[b, h, r].double().numpy()
    lg = lse.cpu()[b, h, r].double().numpy()
    err, lerr = np.abs(og - ro), np.abs(lg - rl)
    res = {"rows": int(idx.shape[0]), "out_max_err": float(err.max()),
           "out_mean_err": float(err.mean()), "lse_max_err": float(lerr.max()),
           "bars": {"out_max": 2e-2, "out_mean": 2e-3, "lse_max": 1e-3}}
    res["pass"] = bool(res["out_max_err"] <= 2e-2 and res["out_mean_err"] <= 2e-3
                       and res["lse_max_err"] <= 1e-3 and np.isfinite(og).all())
    return res


def as_numpy(q, k, v):
    """bf16 tensors -> float32 numpy arrays (exact), converted once per run."""
    return tuple(x.float().numpy() for x in (q, k, v))


def oracle_rows_sample(qn, kn, vn, scale, causal, rows_per_head, heads, budget_s, results=None):
    """Time the fp64 oracle (row form) on evenly spaced rows; return (tflops, rows, secs).
    If `results` is a list, each head's (index, out rows, lse rows) is appended to it."""
    from oracle import attention_rows  # CPU baseline leg only
    B, H, S, D = qn.shape
    rows = np.linspace(0, S - 1, rows_per_head).round().astype(np.int64)
    done, flops, t0 = 0, 0, time.perf_counter()
    for h in heads:
        idx = np.stack([np.zeros_like(rows), np.full_like(rows, h), rows], 1)
        ro, rl = attention_rows(qn, kn, vn, scale, causal, idx)
        if results is not None:
            results.append((idx, ro, rl))
        done += len(rows)
        n_keys = (rows + 1) if causal else np.full_like(rows, S)
        flops += int(4 * D * n_keys.sum())
        if time.perf_counter() - t0 > budget_s:
            break
    secs = time.perf_counter() - t0
    return flops / secs / 1e12, done, secs


def bench_config(w, world, scale):
    """The `config` of the JSON line (the same for both arms)."""
    return {"workload": w.about, "B": w.B, "H": w.H, "S": w.S, "D": w.D, "causal": w.causal,
            "global_batch": w.B * world, "scale": scale,
            "seed": "rank r holds batch block r, drawn with seed r (rank 0: seed 0)",
            "l2": (f"inputs {3 * w.B * w.H * w.S * w.D * 2 / 1e6:.0f} MB "
                   f"{'>' if 3 * w.B * w.H * w.S * w.D * 2 > 129e6 else '<='} 129 MB L2: "
                   "no flush between steps"),
            "parallelism": f"head-sharded x{world}: the global problem's (b, h) slices split "
                           "contiguously over the ranks (attn_shard_range), no collective"}


def run_reference(args, world, rank):
    """The oracle on the host cores: `steps` timed samples after `warmup` untimed ones."""
    if rank != 0:
        return
    w = WORKLOADS[args.workload]
    qn, kn, vn = as_numpy(*make_qkv(w, seed=0))
    scale = default_scale(w.D)
    rows_per_step = 256  # the same per-head sample as the cpu_baseline leg of the other arm
    for i in range(args.warmup):
        oracle_rows_sample(qn, kn, vn, scale, w.causal, rows_per_step, [i % w.H], 1e9)
    flops, t0 = 0, time.perf_counter()
    for i in range(args.steps):
        _, n, _ = oracle_rows_sample(qn, kn, vn, scale, w.causal, rows_per_step, [i % w.H], 1e9)
        rows = np.linspace(0, w.S - 1, rows_per_step).round()
        flops += int(4 * w.D * (rows + 1).sum())
    secs = time.perf_counter() - t0
    val = flops / secs / 1e12
    cores = len(os.sched_getaffinity(0))
    sample = (f"{rows_per_step} evenly spaced query rows of one head per step (head = step mod {w.H}) "
              f"of the {w.about} workload; oracle row form, fp64 numpy")
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": secs / max(args.steps, 1) * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": bench_config(w, world, scale),
            "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def time_steps(fn, steps, stream, per_step=False):
    """Total ms of `steps` calls between two events on `stream`; with per_step,
    also an event after every call and the per-call durations (ms)."""
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1 if per_step else 2)]
    torch.cuda.synchronize()
    ev[0].record(stream)
    for i in range(steps):
        fn()
        if per_step:
            ev[i + 1].record(stream)
    if not per_step:
        ev[1].record(stream)
    ev[-1].synchronize()
    total = ev[0].elapsed_time(ev[-1])
    if not per_step:
        return total
    return total, [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]


def executed_flops(B, H, S, D, causal):
    """FLOPs of the 128x128 tiles the kernel actually runs (diagonal tiles whole)."""
    n = (S + 127) // 128
    tiles = n * (n + 1) // 2 if causal else n * n
    return 4 * B * H * tiles * 128 * 128 * D


def blas_threads():
    """(threads, how it was found) of the BLAS numpy calls."""
    try:
        from threadpoolctl import threadpool_info
        n = max((i.get("num_threads", 0) for i in threadpool_info()), default=0)
        if n:
            return n, "threadpoolctl"
    except Exception:
        pass
    # no threadpoolctl: ask the OpenBLAS numpy loaded (its library is mapped
    # into this process) through its exported thread-count query
    import ctypes
    np.dot(np.ones((2, 2)), np.ones((2, 2)))  # make sure BLAS is loaded
    try:
        with open("/proc/self/maps") as f:
            libs = sorted({ln.split()[-1] for ln in f if "openblas" in ln.lower() and ".so" in ln})
    except OSError:
        libs = []
    for path in libs:
        try:
            lib = ctypes.CDLL(path)
        except OSError:
            continue
        for sym in ("scipy_openblas_get_num_threads64_", "openblas_get_num_threads64_",
                    "scipy_openblas_get_num_threads", "openblas_get_num_threads"):
            fn = getattr(lib, sym, None)
            if fn is not None:
                fn.restype = ctypes.c_int
                return int(fn()), f"{sym} ({os.path.basename(path)})"
    v = os.environ.get("OMP_NUM_THREADS")
    if v and v.isdigit():
        return int(v), "OMP_NUM_THREADS"
    return os.cpu_count(), "os.cpu_count (no BLAS thread query available)"


def full_parity(ref_out, ref_lse, out, lse):
    """Every element of a GPU output against the oracle's, with the parity bars."""
    og, lg = out.double().numpy(), lse.double().numpy()
    err, lerr = np.abs(og - ref_out), np.abs(lg - ref_lse)
    res = {"rows": int(lg.size), "out_max_err": float(err.max()),
           "out_mean_err": float(err.mean()), "lse_max_err": float(lerr.max())}
    res["pass"] = bool(res["out_max_err"] <= 2e-2 and res["out_mean_err"] <= 2e-3
                       and res["lse_max_err"] <= 1e-3 and np.isfinite(og).all())
    return res


def oracle_per_config(budget_s, full_cap_s=30.0, kept=None):
    """Wall time of the fp64 oracle on c1-c4.  c1 runs whole.  c2-c4 are first
    timed on evenly spaced rows of every head for about `budget_s` seconds;
    c2 and c4 then run whole if that rate puts the whole problem under
    `full_cap_s`, and c3 (like c5, the cpu_baseline) keeps the time
    extrapolated from the rate in counted FLOPs, flagged as such.  With
    `kept` (the GPU outputs of the side timings), each entry also carries the
    GPU output's errors against the oracle on the rows it computed."""
    from oracle import attention_fwd
    res = {}
    for name in ("c1", "c2", "c3", "c4"):
        w = WORKLOADS[name]
        qn, kn, vn = as_numpy(*make_qkv(w, seed=0))
        scale = default_scale(w.D)
        total = counted_flops(w.B, w.H, w.S, w.D, w.causal)
        rows = w.B * w.H * w.S
        est = None
        if name != "c1":
            checked = []
            tf, n_rows, secs = oracle_rows_sample(qn, kn, vn, scale, w.causal, min(w.S, 256),
                                                  list(range(w.H)), budget_s, checked)
            est = total / (tf * 1e12)
            if name == "c3" or est > full_cap_s:
                res[name] = {"rows": n_rows, "s": secs, "tflops": tf, "full_s": est,
                             "extrapolated": True}
                if kept is not None and name in kept:
                    res[name]["parity"] = parity_of_outputs(checked, *kept[name])
                continue
        t0 = time.perf_counter()
        ref_out, ref_lse = attention_fwd(qn, kn, vn, scale, w.causal)
        secs = time.perf_counter() - t0
        res[name] = {"rows": rows, "s": secs, "tflops": total / secs / 1e12, "full_s": secs,
                     "extrapolated": False, "sample_estimate_s": est}
        if kept is not None and name in kept:
            res[name]["parity"] = full_parity(ref_out, ref_lse, *kept[name])
    return res


def side_workloads(device, stream, kept=None):
    """TFLOP/s of the other workloads (context; L2 flushed between launches).
    If `kept` is a dict, c1-c4's last outputs are copied into it (host tensors)
    for the per-workload parity check of the CPU leg."""
    from exact_attention_68_gb300 import binding
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=device)
    res = {}
    for name in ("c1", "c2", "c3", "c4"):
        w = WORKLOADS[name]
        q, k, v = (x.to(device) for x in make_qkv(w, seed=0))
        out, lse = torch.empty_like(q), torch.empty(w.B, w.H, w.S, device=device)
        scale = default_scale(w.D)
        for _ in range(3):
            binding.attn_fwd(q, k, v, scale, w.causal, out, lse)
        times = []
        for _ in range(20):
            flush.zero_()
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            binding.attn_fwd(q, k, v, scale, w.causal, out, lse)
            e.record(stream)
            e.synchronize()
            times.append(s.elapsed_time(e))
        ms = statistics.median(times)
        if kept is not None:
            kept[name] = (out.cpu(), lse.cpu())
        res[name] = {"about": w.about, "ms": ms,
                     "tflops": counted_flops(w.B, w.H, w.S, w.D, w.causal) / (ms * 1e-3) / 1e12}
    # the default workload with fp16 inputs (attn_fwd_ex), 20 back-to-back launches
    w = WORKLOADS[WORKLOAD]
    q, k, v = (x.to(device) for x in make_qkv(w, seed=0, dtype=torch.float16))
    out, lse = torch.empty_like(q), torch.empty(w.B, w.H, w.S, device=device)
    scale = default_scale(w.D)
    for _ in range(3):
        binding.attn_fwd(q, k, v, scale, w.causal, out, lse)
    ms = time_steps(lambda: binding.attn_fwd(q, k, v, scale, w.causal, out, lse), 20, stream) / 20
    res[WORKLOAD + "_fp16"] = {"about": w.about + ", fp16 inputs", "ms": ms,
                               "tflops": counted_flops(w.B, w.H, w.S, w.D, w.causal) / (ms * 1e-3) / 1e12}
    # other head dimensions at the long-context shape (the same 16384-key rows):
    # 256 and 192 have their own forward kernel widths, 96 runs on the next
    # width up
    for D, H in ((256, 16), (96, 32), (192, 16)):
        gen = torch.Generator(device=device).manual_seed(D)
        q, k, v = (torch.randn((1, H, 16384, D), generator=gen, device=device).to(torch.bfloat16)
                   for _ in range(3))
        out, lse = torch.empty_like(q), torch.empty(1, H, 16384, device=device)
        scale = default_scale(D)
        for _ in range(3):
            binding.attn_fwd(q, k, v, scale, True, out, lse)
        ms = time_steps(lambda: binding.attn_fwd(q, k, v, scale, True, out, lse), 10, stream) / 10
        res[f"d{D}"] = {"about": f"causal B=1 H={H} S=16384 D={D}, N(0,1)", "ms": ms,
                        "tflops": counted_flops(1, H, 16384, D, True) / (ms * 1e-3) / 1e12}
        del q, k, v, out, lse
    return res


def backward_leg(w, q, k, v, out, lse, scale, stream, steps):
    """The gradient of the same workload (attn_bwd: dq+delta kernel, then dk/dv
    kernel), timed over `steps` calls with CUDA events after 3 warm-up calls."""
    from exact_attention_68_gb300 import binding
    g = torch.Generator().manual_seed(1)
    dout = torch.randn(w.shape, generator=g, dtype=torch.float32).to(torch.bfloat16).to(q.device)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    delta = torch.empty_like(lse)

    def call():
        binding.attn_bwd(q, k, v, out, lse, dout, scale, w.causal, dq, dk, dv, delta)

    for _ in range(3):
        call()
    ms = time_steps(call, steps, stream) / steps
    counted = 2.5 * counted_flops(w.B, w.H, w.S, w.D, w.causal)
    executed = 3.5 * executed_flops(w.B, w.H, w.S, w.D, w.causal)
    return {"metric": "attention backward TFLOP/s (counted: 2.5x the forward's FLOPs)",
            "value": counted / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": ms,
            "steps": steps, "executed_tflops": executed / (ms * 1e-3) / 1e12,
            "executed_over_counted_flops": executed / counted,
            "kernels": ["attn_bwd_dq_kernel<128,true>", "attn_bwd_dkdv_kernel<128,true>"],
            "gpu_launches": 2 * steps}


def backward_side(device, stream):
    """TFLOP/s of the backward at head dimension 256 (its own kernels) on the
    long-context shape: counted 2.5x the forward's causal FLOPs."""
    from exact_attention_68_gb300 import binding
    B, H, S, D = 1, 16, 16384, 256
    gen = torch.Generator(device=device).manual_seed(D)
    q, k, v, dout = (torch.randn((B, H, S, D), generator=gen, device=device).to(torch.bfloat16)
                     for _ in range(4))
    scale = default_scale(D)
    out, lse = binding.attn_fwd(q, k, v, scale, True)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    delta = torch.empty_like(lse)

    def call():
        binding.attn_bwd(q, k, v, out, lse, dout, scale, True, dq, dk, dv, delta)

    for _ in range(3):
        call()
    ms = time_steps(call, 5, stream) / 5
    counted = 2.5 * counted_flops(B, H, S, D, True)
    return {"d256": {"about": f"causal B={B} H={H} S={S} D={D}, N(0,1)", "ms": ms,
                     "tflops": counted / (ms * 1e-3) / 1e12,
                     "kernels": ["attn_bwd_dq256_kernel<true>", "attn_bwd_dkdv_q64_kernel<256,true>"]}}


def run_ours(args, world, rank, local):
    from exact_attention_68_gb300 import binding
    from exact_attention_68_gb300.build import build_library

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    build_library()
    binding.load_library()
    w = WORKLOADS[args.workload]
    if args.shape:
        B, H, S, D = (int(x) for x in args.shape.split(","))
        w = Workload("shape", B, H, S, D, True, about=f"causal B={B} H={H} S={S} D={D}, N(0,1)")
    scale = default_scale(w.D)
    flops = counted_flops(w.B, w.H, w.S, w.D, w.causal)  # per rank
    # this rank's share of the global problem (world batch blocks of w.B
    # elements): world divides the slices evenly, so it is batch block `rank`
    units = w.B * w.H * world
    first, count = binding.shard_range(units, world, rank)
    assert (first, count) == (rank * w.B * w.H, w.B * w.H), (first, count)
    q_h, k_h, v_h = (x.pin_memory() for x in make_qkv(w, seed=rank))
    q, k, v = (x.to(device) for x in (q_h, k_h, v_h))
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)

    def step():
        binding.attn_fwd(q, k, v, scale, w.causal, out, lse)

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
    except Exception:
        pass
    clocks = ClockSampler(uuid)
    time.sleep(0.5)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    ms, per_launch = time_steps(step, args.steps, stream, per_step=True)
    t1 = time.time()
    torch.cuda.synchronize()
    barrier(world)
    status = binding.device_status(device)
    ms_max = reduce_max(ms, world, device)
    clk = clocks.summary(t0, t1)
    # clock check: the same step back to back for about a second (not part of
    # the value), long enough for several clock samples; its per-launch time
    # times the median SM clock gives the cycles a launch takes
    clock_check = None
    if args.clock_check_s > 0:
        n_chk = max(10, int(args.clock_check_s * 1000.0 / max(ms / args.steps, 1e-3)))
        c0 = time.time()
        chk_ms = time_steps(step, n_chk, stream) / n_chk
        c1 = time.time()
        chk = clocks.summary(c0, c1)
        clock_check = {"launches": n_chk, "ms_per_launch": chk_ms, "sm_mhz_median": chk["sm_mhz"],
                       "reasons": chk["reasons"], "samples": chk["samples"],
                       "mcycles_per_launch": (chk_ms * 1e-3 * chk["sm_mhz"]
                                              if chk["sm_mhz"] else None)}

    # end to end: host inputs (pinned) -> device -> kernel -> host outputs, per step
    out_h = torch.empty_like(q_h).pin_memory()
    lse_h = torch.empty((w.B, w.H, w.S), dtype=torch.float32).pin_memory()
    e2e_steps = max(3, min(args.steps, 20))

    def e2e_step():
        binding.attn_fwd_staged(q_h, k_h, v_h, out_h, lse_h, q, k, v, out, lse, scale, w.causal)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = reduce_max(time_steps(e2e_step, e2e_steps, stream), world, device)
    clocks.stop()

    peaks, peak_src = load_peaks()
    per_launch_s = ms_max / args.steps * 1e-3
    achieved = flops / per_launch_s / 1e12
    peak = float(peaks["bf16_tflops"])
    traffic = NCU_TRAFFIC_BYTES.get(kernel_hash())
    value = flops * world * args.steps / (ms_max * 1e-3) / 1e12
    extra = {}
    kept_outputs = {}
    if rank == 0 and world == 1 and not args.no_side:
        extra["other_workloads"] = side_workloads(device, stream, kept_outputs)
    if not args.no_bwd:
        bwd = backward_leg(w, q, k, v, out, lse, scale, stream, max(3, min(args.steps, 50)))
        bwd["roofline"] = {"bound": "tensor", "achieved": bwd["value"],
                           "peak": float(peaks["bf16_tflops"]), "unit": "TFLOP/s",
                           "frac": bwd["value"] / float(peaks["bf16_tflops"])}
        extra["backward"] = bwd
        if rank == 0 and world == 1 and not args.no_side:
            extra["backward_other"] = backward_side(device, stream)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        checked = []
        tf, n_rows, secs = oracle_rows_sample(*as_numpy(q_h, k_h, v_h), scale, w.causal, 256,
                                              list(range(w.H)), args.cpu_budget, checked)
        nthr, how = blas_threads()
        cpu = {"value": tf, "unit": "TFLOP/s", "cores": len(os.sched_getaffinity(0)),
               "kind": "oracle", "blas_threads": nthr, "blas_threads_source": how,
               "full_problem_s_extrapolated": flops / (tf * 1e12),
               "sample": f"{n_rows} query rows (256 evenly spaced per head, heads in order) of the "
                         f"{w.about} workload, oracle row form in fp64 numpy, {secs:.1f} s"}
        extra["parity"] = parity_of_outputs(checked, out_h, lse_h)
        if not args.no_side:
            extra["oracle_per_config"] = oracle_per_config(args.cpu_budget / 4, kept=kept_outputs)
    if rank != 0:
        return
    nb = w.B * w.H * w.S * w.D * 2
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": bench_config(w, world, scale),
        "shard": {"rank": rank, "world": world, "first": first, "count": count, "units": units},
        "pct_of_peak": 100.0 * achieved / peak,
        "ms_per_launch": {"mean": ms_max / args.steps, "median": statistics.median(per_launch),
                          "min": min(per_launch), "max": max(per_launch),
                          "all": [round(x, 4) for x in per_launch]},
        "executed_over_counted_flops": executed_flops(w.B, w.H, w.S, w.D, w.causal) / flops,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": f"{peak_src} bf16_tflops (burst, cuBLAS 8192^3)",
                     # context: the timed loop runs long enough to meet the power cap,
                     # the regime of the sustained cuBLAS figure
                     "peak_sustained": float(peaks.get("bf16_tflops_sustained", peak)),
                     "frac_of_sustained": achieved / float(peaks.get("bf16_tflops_sustained", peak)),
                     "kernel": "attn_fwd_1qp_kernel<128,true,bf16>",
                     "algorithmic_flops_per_launch": flops,
                     "algorithmic_bytes_per_launch": algorithmic_bytes(w.B, w.H, w.S, w.D)},
        "e2e": {"value": flops * e2e_steps / (e2e_ms * 1e-3) / 1e12 * world, "unit": "TFLOP/s",
                "h2d_bytes_per_step": 3 * nb, "d2h_bytes_per_step": nb + w.B * w.H * w.S * 4,
                "ms_per_step": e2e_ms / e2e_steps, "steps": e2e_steps},
        "gpu_launches": args.steps,
        "clocks": clk,
        "clock_check": clock_check,
        "device_status": status,
        "cpu_baseline": cpu,
        "kernel_hash": kernel_hash(),
    }
    line.update(extra)
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-side", action="store_true", help="skip the other-workload timings")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU baseline")
    ap.add_argument("--no-bwd", action="store_true", help="skip the backward timing")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle time")
    ap.add_argument("--shape", default=None,
                    help="B,H,S,D of a causal workload to time instead (profiling runs)")
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(WORKLOADS),
                    help="which workload the timed steps run (profiling runs; default c5)")
    ap.add_argument("--clock-check-s", type=float, default=1.0,
                    help="seconds of back-to-back steps after the timed region whose clocks "
                         "are sampled (0: none)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
