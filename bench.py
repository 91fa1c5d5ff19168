#!/usr/bin/env python3
"""Benchmark of the exact tiled attention hot path on GB300.

One step = one forward (fa_fwd) and one backward (fa_bwd: preprocess, main
kernel, dQ cast) over the whole workload, inputs resident in device memory.
The default workload is the largest single-GPU one, causal attention over
32768 tokens (B=1, H=8, d=128).  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the fp64 CPU oracle, timed on the host cores

FLOPs are counted as 4 N^2 d per (batch, head) for the forward, halved when
causal, and 2.5x that for the backward (five N x N x d products).
Between timed steps the L2 cache is flushed by writing a 256 MiB buffer
(outside the per-step CUDA events).  N > 1 (torchrun) runs one independent
copy of the workload per GPU (weak scaling, no collective on the data path).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from exact_tiled_attention_08_gb300.workloads import (  # noqa: E402
    WORKLOADS, make_inputs, rotation_signs, to_f32_numpy)

METRIC = "attention fwd/bwd TFLOP/s at d=128 BF16 and % of GB300 dense BF16 peak"
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = "causal_long_b1_h8_n32768_d128"
# nominal dense (no 2:4 sparsity) bf16 tensor throughput of one GPU of this
# generation, for context beside the measured peaks
NOMINAL_DENSE_BF16_TFLOPS = 2250.0
L2_FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
# the sources each kernel's DRAM traffic depends on (its own header, the PTX
# building blocks and the host code that configures its launch)
KERNEL_SOURCES = {
    "fa_fwd_kernel": ["fa_fwd.cuh", "sm103_ptx.cuh", "fa_lib.cu"],
    "fa_fwd_kernel/fp8": ["fa_fwd.cuh", "fa_fp8.cuh", "sm103_ptx.cuh", "fa_lib.cu"],
    "fa_bwd_kernel": ["fa_bwd.cuh", "sm103_ptx.cuh", "fa_lib.cu"],
    "fa_bwd_kernel/deterministic": ["fa_bwd.cuh", "sm103_ptx.cuh", "fa_lib.cu"],
    "fa_bwd_dq_kernel": ["fa_bwd_dq.cuh", "sm103_ptx.cuh", "fa_lib.cu"],
}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--e2e-chunks", type=int, default=1,
                    help="head chunks per step in the end-to-end leg (steps are pipelined over copy-in / compute / "
                         "copy-out streams either way; more chunks also overlap copies within a step, but each "
                         "launch then covers fewer heads)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="budget of the oracle CPU baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--deterministic", action="store_true",
                    help="backward by fa_bwd_deterministic (dQ by the separate query-major pass, no atomics)")
    ap.add_argument("--sustained-seconds", type=float, default=2.0,
                    help="length of the back-to-back leg whose steps give the sustained figure (0: skip)")
    ap.add_argument("--no-fp8", action="store_true", help="skip the FP8 forward leg")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------
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
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist

    dev = torch.device("cuda", torch.cuda.current_device()) if torch.cuda.is_available() else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def _code_only(text: str) -> str:
    """C++ source without comments and with whitespace runs collapsed, so that
    editing a comment does not count as changing a kernel."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash(kernel: str = "fa_bwd_kernel") -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "exact_tiled_attention_08_gb300", "csrc", name), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_profile(kernel: str, workload: str) -> dict:
    """The committed ncu figures of `kernel` on `workload` (DRAM bytes per
    launch, tensor-pipe activity), or {} when there are none or the kernel's
    sources changed since they were taken."""
    if not os.path.exists(TRAFFIC_FILE):
        return {}
    with open(TRAFFIC_FILE) as f:
        d = json.load(f)
    e = d.get(kernel, {}).get(workload)
    if not e or kernel not in KERNEL_SOURCES or e.get("source_hash") != kernel_source_hash(kernel):
        return {}
    return e


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, or None
    when there is none for this workload or the kernel sources changed since."""
    return recorded_profile(kernel, workload).get("dram_bytes_per_launch")


def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info

        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return os.cpu_count() or 1


def sample_flops(w, rows: int) -> float:
    """Algorithmic fwd+bwd FLOPs of the first `rows` query rows of one head."""
    pairs = rows * (rows + 1) / 2 if w.causal else rows * w.N
    if w.causal and rows == w.N:
        pairs = w.N * w.N / 2
    return 4.0 * w.d * pairs * 3.5


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.device = device_index

    def start(self):
        try:
            uuid = str(torch.cuda.get_device_properties(self.device).uuid)
            sel = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            sel = str(self.device)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", sel], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "note": "nvidia-smi unavailable"}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(self.REASONS, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU oracle timings (the reference arm and the cpu_baseline leg)
# ---------------------------------------------------------------------------
def oracle_step(inp_np, w, b, h, rows):
    from oracle import attention_bwd_ref, attention_fwd_ref

    q, k, v, do = (inp_np[x][b, h] for x in ("q", "k", "v", "do"))
    attention_fwd_ref(q[:rows], k, v, w.scale, w.causal)
    attention_bwd_ref(q[:rows], k, v, do[:rows], w.scale, w.causal)


def oracle_rows_for_budget(inp_np, w, seconds_per_step: float) -> int:
    """Largest number of leading query rows of one head whose fwd+bwd oracle
    fits the per-step budget (measured on a probe of 128 rows)."""
    probe = min(128, w.N)
    t0 = time.perf_counter()
    oracle_step(inp_np, w, 0, 0, probe)
    dt = max(time.perf_counter() - t0, 1e-4)
    per_row = dt / probe
    rows = int(seconds_per_step / per_row)
    return max(1, min(w.N, rows))


def cpu_inputs(w, seed_offset=0):
    inp = make_inputs(w.B, w.H, w.N, w.d, w.seed + seed_offset, w.key_outliers)
    return inp, {x: to_f32_numpy(t) for x, t in inp.items()}


def run_reference(args, rank, world):
    if rank != 0:
        return
    w = WORKLOADS[args.workload]
    _, inp_np = cpu_inputs(w)
    total = args.steps + args.warmup
    rows = oracle_rows_for_budget(inp_np, w, seconds_per_step=min(2.0, 150.0 / max(total, 1)))
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    for i in range(args.warmup):
        oracle_step(inp_np, w, *heads[i % len(heads)], rows)
    times = []
    for i in range(args.steps):
        t0 = time.perf_counter()
        oracle_step(inp_np, w, *heads[i % len(heads)], rows)
        times.append(time.perf_counter() - t0)
    ms = 1e3 * statistics.mean(times)
    value = sample_flops(w, rows) / (ms / 1e3) / 1e12
    sample = f"per step: fwd+bwd of the first {rows} of {w.N} query rows of one (batch, head), cycling over heads"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
                   "sample_rows_per_step": rows},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": blas_threads(), "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def cpu_baseline(w, inp_np, budget_s: float):
    rows = oracle_rows_for_budget(inp_np, w, seconds_per_step=min(budget_s / 3, 4.0))
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    done, flops = 0, 0.0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < budget_s and done < len(heads):
        oracle_step(inp_np, w, *heads[done], rows)
        flops += sample_flops(w, rows)
        done += 1
    dt = time.perf_counter() - t0
    rate = flops / dt
    return {"value": rate / 1e12, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
            "sample": f"fwd+bwd of the first {rows} of {w.N} query rows of {done} of {len(heads)} heads "
                      f"({dt:.1f} s, fp64 numpy)",
            "extrapolated": rows < w.N or done < len(heads),
            "extrapolated_step_s": (w.fwd_flops() + w.bwd_flops()) / rate,
            "note": "rate measured on the sample, extrapolated to the whole workload as step FLOPs / rate"}


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------
def run_ours(args, rank, world, local):
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device; the GPU arm has no CPU fallback")
    from exact_tiled_attention_08_gb300 import fa
    from exact_tiled_attention_08_gb300.build import build_library

    build_library()
    fa.load_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = WORKLOADS[args.workload]
    scale = w.scale
    inp_cpu, inp_np = cpu_inputs(w, seed_offset=7919 * rank)
    q, k, v, do = (inp_cpu[x].to(dev) for x in ("q", "k", "v", "do"))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.fa_bwd_workspace_bytes(w.B, w.H, w.N, w.d), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)
    fwd_flops, bwd_flops = w.fwd_flops(), w.bwd_flops()
    step_flops = fwd_flops + bwd_flops
    bwd_entry = fa.fa_bwd_deterministic if args.deterministic else fa.fa_bwd
    # the main backward kernel does all five products, or four of them when dQ
    # is left to the deterministic pass (whose time is then in "other_ms")
    bwd_main_flops = bwd_flops * (0.8 if args.deterministic else 1.0)

    def step():
        fa.fa_fwd(q, k, v, o, lse, scale, w.causal, stream)
        bwd_entry(q, k, v, o, do, lse, dq, dk, dv, ws, scale, w.causal, stream)

    K, W = args.steps, args.warmup
    with torch.cuda.stream(stream):
        for _ in range(W):
            flush.zero_()
            step()
        st = fa.fa_check_device_status(stream)
        if st != fa.FA_OK:
            raise SystemExit(f"bench.py: device status {fa.fa_status_string(st)} after warm-up")
        if not (torch.isfinite(o.float()).all() and torch.isfinite(dq.float()).all()):
            raise SystemExit("bench.py: non-finite outputs after warm-up")
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(K)]
        for e in ev:
            for x in e:
                x.record(stream)  # creates the event so its handle can be passed to the library
        torch.cuda.synchronize(dev)
        clocks = ClockSampler(local)
        clocks.start()
        barrier(world)
        torch.cuda.synchronize(dev)
        for i in range(K):
            flush.zero_()
            e = ev[i]
            fa.fa_set_timing_events(e[2], e[3], e[4], e[5])
            e[0].record(stream)
            step()
            e[1].record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        clock_info = clocks.stop()
        fa.fa_set_timing_events()
        st = fa.fa_check_device_status(stream)
        if st != fa.FA_OK:
            raise SystemExit(f"bench.py: device status {fa.fa_status_string(st)} in the timed region")
    # ---- the FP8 forward (fa_fwd_fp8) on the same inputs, d = 128 only: the
    # whole call (operand preparation + E4M3 attention kernel) and the kernel
    fp8 = None
    if w.d == 128 and not args.no_fp8:
        signs = rotation_signs(w.d, w.seed).to(dev)
        ws8 = torch.empty(fa.fa_fwd_fp8_workspace_bytes(w.B, w.H, w.N, w.d), dtype=torch.uint8, device=dev)
        o8 = torch.empty_like(o)
        lse8 = torch.empty_like(lse)
        with torch.cuda.stream(stream):
            for _ in range(3):
                fa.fa_fwd_fp8(q, k, v, signs, o8, lse8, ws8, scale, w.causal, stream)
            calls, kers = [], []
            for _ in range(20):
                flush.zero_()
                e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
                for x in e:
                    x.record(stream)
                fa.fa_set_timing_events(e[2], e[3], None, None)
                e[0].record(stream)
                fa.fa_fwd_fp8(q, k, v, signs, o8, lse8, ws8, scale, w.causal, stream)
                e[1].record(stream)
                calls.append(e)
            torch.cuda.synchronize(dev)
            fa.fa_set_timing_events()
            if fa.fa_check_device_status(stream) != fa.FA_OK:
                raise SystemExit("bench.py: device status error in the FP8 forward")
        call_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in calls)
        ker_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in calls)
        fp8 = {"call_ms": call_ms, "call_tflops": fwd_flops / (call_ms / 1e3) / 1e12, "kernel_ms": ker_ms,
               "kernel_tflops": fwd_flops / (ker_ms / 1e3) / 1e12,
               "note": "fa_fwd_fp8: Q, K rotated and quantised per 128-row block, V per channel, E4M3 products; "
                       "the call includes the operand preparation"}

    # ---- sustained: the same step back to back for a few seconds (L2 still
    # flushed before every step), the clocks sampled meanwhile; this is the
    # figure to set against the measured sustained (power-capped) peak
    sustained = None
    if args.sustained_seconds > 0:
        n_sus = max(3, int(math.ceil(args.sustained_seconds * 1e3 / statistics.mean(
            e[0].elapsed_time(e[1]) for e in ev))))
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        sus_clocks = ClockSampler(local)
        sus_clocks.start()
        with torch.cuda.stream(stream):
            s0.record(stream)
            for _ in range(n_sus):
                flush.zero_()
                step()
            s1.record(stream)
        torch.cuda.synchronize(dev)
        sus_clock_info = sus_clocks.stop()
        if fa.fa_check_device_status(stream) != fa.FA_OK:
            raise SystemExit("bench.py: device status error in the sustained leg")
        sus_ms = s0.elapsed_time(s1) / n_sus  # includes the L2 flush between steps
        sustained = {"steps": n_sus, "seconds": s0.elapsed_time(s1) / 1e3, "ms_per_step_incl_flush": sus_ms,
                     "tflops_incl_flush": step_flops / (sus_ms / 1e3) / 1e12, "clocks": sus_clock_info}

    step_times = [e[0].elapsed_time(e[1]) for e in ev]
    step_ms = statistics.mean(step_times)
    fwd_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in ev)
    bwd_ms = statistics.mean(e[4].elapsed_time(e[5]) for e in ev)
    step_ms_max = max_over_ranks(step_ms, world)
    value = world * step_flops / (step_ms_max / 1e3) / 1e12

    # ---- end to end through the C ABI with pinned host buffers.  Every step
    # copies its inputs (Q, K, V, dO) from pinned host memory to the device and
    # its results (O, LSE, dQ, dK, dV) back, inside the timed region.  The
    # heads are split into chunks (every tensor is laid out head-major, so a
    # range of heads is a contiguous slice) and the work is pipelined over
    # three streams, within a step and across steps: the device tensors are
    # double-buffered by step parity, so while step i is computed, step i+1's
    # inputs come in and step i-1's results go out.  Each chunk is one
    # fa_fwd + fa_bwd call on its heads.
    o_ref = o.clone()
    h_in = {x: inp_cpu[x].pin_memory() for x in ("q", "k", "v", "do")}
    h_out = {"o": torch.empty_like(o, device="cpu").pin_memory(), "lse": torch.empty_like(lse, device="cpu").pin_memory(),
             "dq": torch.empty_like(dq, device="cpu").pin_memory(), "dk": torch.empty_like(dk, device="cpu").pin_memory(),
             "dv": torch.empty_like(dv, device="cpu").pin_memory()}
    h2d = sum(t.numel() * t.element_size() for t in h_in.values())
    d2h = sum(t.numel() * t.element_size() for t in h_out.values())
    sets = [({"q": q, "k": k, "v": v, "do": do}, {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv})]
    sets.append(({x: torch.empty_like(t) for x, t in sets[0][0].items()},
                 {x: torch.empty_like(t) for x, t in sets[0][1].items()}))
    BH = w.B * w.H
    chunks = max(1, min(args.e2e_chunks, BH))
    bounds = [(c * BH // chunks, (c + 1) * BH // chunks) for c in range(chunks)]

    def heads(t, lo, hi):
        # [B, H, ...] -> [1, hi - lo, ...] view of heads lo..hi-1 (contiguous)
        return t.view(1, BH, *t.shape[2:])[:, lo:hi]

    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    # per (buffer set, chunk): inputs consumed by the compute, results copied out
    consumed = [[None] * chunks for _ in range(2)]
    copied_out = [[None] * chunks for _ in range(2)]

    def e2e_step(i):
        d_in, d_out = sets[i % 2]
        for c, (lo, hi) in enumerate(bounds):
            with torch.cuda.stream(s_in):
                if consumed[i % 2][c] is not None:
                    s_in.wait_event(consumed[i % 2][c])
                for name, t in d_in.items():
                    heads(t, lo, hi).copy_(heads(h_in[name], lo, hi), non_blocking=True)
                got_in = torch.cuda.Event()
                got_in.record(s_in)
            stream.wait_event(got_in)
            if copied_out[i % 2][c] is not None:
                stream.wait_event(copied_out[i % 2][c])
            with torch.cuda.stream(stream):
                qc, kc, vc, doc = (heads(d_in[x], lo, hi) for x in ("q", "k", "v", "do"))
                oc, lc = heads(d_out["o"], lo, hi), heads(d_out["lse"], lo, hi)
                fa.fa_fwd(qc, kc, vc, oc, lc, scale, w.causal, stream)
                bwd_entry(qc, kc, vc, oc, doc, lc, heads(d_out["dq"], lo, hi), heads(d_out["dk"], lo, hi),
                          heads(d_out["dv"], lo, hi), ws, scale, w.causal, stream)
                done = torch.cuda.Event()
                done.record(stream)
            consumed[i % 2][c] = done
            s_out.wait_event(done)
            with torch.cuda.stream(s_out):
                for name, t in h_out.items():
                    heads(t, lo, hi).copy_(heads(d_out[name], lo, hi), non_blocking=True)
                out_ev = torch.cuda.Event()
                out_ev.record(s_out)
            copied_out[i % 2][c] = out_ev

    E = max(1, args.e2e_steps)
    for i in range(3):  # warm-up
        e2e_step(i)
    torch.cuda.synchronize(dev)
    barrier(world)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_start.record(s_in)
    for i in range(3, 3 + E):
        e2e_step(i)
    s_out.wait_stream(stream)
    s_out.wait_stream(s_in)
    t_end.record(s_out)
    torch.cuda.synchronize(dev)
    barrier(world)
    assert fa.fa_check_device_status(stream) == fa.FA_OK
    # the pipelined run computed exactly what the device-resident one did
    if not torch.equal(h_out["o"], o_ref.cpu()):
        raise SystemExit("bench.py: end-to-end outputs differ from the device-resident run")
    e2e_ms = max_over_ranks(t_start.elapsed_time(t_end) / E, world)
    e2e_value = world * step_flops / (e2e_ms / 1e3) / 1e12

    if rank != 0:
        return
    peaks, peak_source = load_peaks()
    fwd_tf = fwd_flops / (fwd_ms / 1e3) / 1e12
    # exponentials: one per score in the forward (N^2 per head, half with the
    # mask), against the MUFU's 32 ex2 per clock per SM (probe) x SMs x the
    # median SM clock sampled under load
    fwd_exps = w.fwd_flops() / (4.0 * w.d)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    ex2_peak = 32.0 * sms * clock_info["sm_mhz"] * 1e6 if clock_info.get("sm_mhz") else None
    exp_rate = {"fwd_exps_per_s": fwd_exps / (fwd_ms / 1e3), "ex2_peak_per_s": ex2_peak,
                "frac": (fwd_exps / (fwd_ms / 1e3) / ex2_peak) if ex2_peak else None,
                "note": "N^2 exponentials per head (half with the mask) over the forward kernel's time; "
                        "peak = 32 ex2 per clock per SM x SMs x median SM clock"}
    bwd_tf = bwd_main_flops / (bwd_ms / 1e3) / 1e12
    # dominant kernel: the one with the larger share of the step
    if bwd_ms >= fwd_ms:
        dom, dom_tf, dom_name = "bwd", bwd_tf, "fa_bwd_kernel"
    else:
        dom, dom_tf, dom_name = "fwd", fwd_tf, "fa_fwd_kernel"
    # The timed region is K steps of milliseconds, not a seconds-long run at
    # the power cap, so the kernel is set against the burst peak; the
    # sustained peak belongs to the sustained leg.
    peak = peaks["bf16_tflops"]
    dom_key = dom_name + ("/deterministic" if args.deterministic and dom == "bwd" else "")
    prof = recorded_profile(dom_key, w.name)
    roofline = {"bound": "tensor", "achieved": dom_tf, "peak": peak, "unit": "TFLOP/s", "frac": dom_tf / peak,
                "traffic": prof.get("dram_bytes_per_launch"), "kernel": dom_name,
                "peak_source": f"{peak_source} bf16 burst (cuBLAS 8192^3, best of 10; of {peak_source})",
                "frac_of_sustained_peak": dom_tf / peaks["bf16_tflops_sustained"],
                "frac_of_nominal_dense_peak": dom_tf / NOMINAL_DENSE_BF16_TFLOPS,
                "tensor_pipe_active_pct_ncu": prof.get("tensor_pipe_pct"),
                "algorithmic_flops_per_launch": bwd_main_flops if dom == "bwd" else fwd_flops}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": step_ms_max, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
                   "l2": "flushed before every timed step (256 MiB write, outside the step's events)",
                   "step": ("fa_fwd + fa_bwd_deterministic (preprocess, dK/dV kernel, dQ pass)" if args.deterministic
                            else "fa_fwd + fa_bwd (preprocess, main kernel, dQ cast)"),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": roofline,
        "breakdown": {"fwd_kernel_ms": fwd_ms, "fwd_tflops": fwd_tf, "bwd_kernel_ms": bwd_ms, "bwd_tflops": bwd_tf,
                      "other_ms": step_ms - fwd_ms - bwd_ms,
                      "step_ms_median": statistics.median(step_times), "step_ms_best": min(step_times),
                      "fwd_exp_rate": exp_rate,
                      "fwd_frac_of_burst_peak": fwd_tf / peak, "bwd_frac_of_burst_peak": bwd_tf / peak,
                      "fwd_frac_of_nominal_dense_peak": fwd_tf / NOMINAL_DENSE_BF16_TFLOPS,
                      "bwd_frac_of_nominal_dense_peak": bwd_tf / NOMINAL_DENSE_BF16_TFLOPS,
                      "fwd_tensor_pipe_active_pct_ncu": recorded_profile("fa_fwd_kernel", w.name).get("tensor_pipe_pct"),
                      "bwd_tensor_pipe_active_pct_ncu": recorded_profile(
                          "fa_bwd_kernel" + ("/deterministic" if args.deterministic else ""), w.name).get(
                          "tensor_pipe_pct"),
                      "fp8_forward": fp8},
        "sustained": (dict(sustained, frac_of_sustained_peak=sustained["tflops_incl_flush"]
                           / peaks["bf16_tflops_sustained"]) if sustained else None),
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms, "chunks": chunks, "steps": E,
                "pipelining": "head chunks over copy-in/compute/copy-out streams; device buffers double-buffered "
                              "by step parity, so step i+1's inputs and step i-1's results move during step i"},
        "gpu_launches": 4 * K,
        "clocks": clock_info,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, inp_np, args.cpu_seconds)
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    rank, world, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
