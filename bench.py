#!/usr/bin/env python3
"""Benchmark of the per-linear-layer DP-SGD clipping path on GB300.

Workload: the MLP up_proj shape of a Llama-3.2-1B layer, B=4 sequences of
T=4096 tokens, d=2048 inputs, p=8192 outputs, bf16 activations/gradients with
fp32 accumulation, k=32 probes, C=0.5, sigma=0.8 (synthetic inputs from the
seeded generator).  One step runs every row of the hot path once:
  Hutch norms (probe generation, sketch G P, projection A^T(GP), reduction),
  Hutch++ norms (3 sweeps + QR), exact direct norms, exact ghost norms,
  clip scales + clipped noisy gradient (with the Hutch norms).
Metric: tokens per second of that step (B*T tokens per step), whole job.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl dpclip|reference]

Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the path has no exchange step), timing is the max over ranks and `value` sums
the tokens of all ranks.  `--impl reference` times the fp64 CPU oracle on a
bounded sample of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD_ID = 4
METRIC = "clip+noise tokens/s per linear layer (Hutch/Hutch++/exact); % bf16 tensor peak"
ROWS = ("hutch", "hutchpp", "exact_direct", "exact_ghost", "clipped_noisy_grad")
# measured after the step, not part of it: the Rademacher-probe variants
EXTRA_ROWS = ("hutch_rademacher", "hutchpp_rademacher", "exact_direct_stored",
              "stored_clipped_noisy_grad", "bias_grads", "clipped_noisy_grad_sgd",
              "fiber_step", "clipped_noisy_grad_fiber")
# kernels each ABI call launches for bf16 inputs (memsets of the control block excluded)
# kernels per call: the exact and gradient calls start with one that clears their control words
LAUNCHES = {"hutch": 3, "hutchpp": 8, "exact_direct": 2, "exact_ghost": 2, "clipped_noisy_grad": 2}


# the other standard workloads, timed after the step with the rows each names
OTHER_WORKLOADS = (1, 2, 3, 5)
WORKLOAD_ROWS = {1: ("exact_direct", "hutch", "hutchpp", "clipped_noisy_grad"),
                 2: ("exact_ghost", "exact_direct", "clipped_noisy_grad"),
                 3: ("hutch", "clipped_noisy_grad"),
                 5: ("hutch", "hutchpp", "exact_direct", "clipped_noisy_grad")}


L2_BYTES = 129e6


def time_workload(api, L, W, wid, dev, reps, peaks):
    """Latency of each row a standard workload names.  Workloads whose inputs
    are larger than L2 are timed as the step's rows are: `reps` calls of the
    row back to back between one event pair, the median of three such
    blocks.  The others (whose inputs would
    stay in L2) one call at a time with a CUDA event pair around it and L2
    flushed before it (a 256 MB write outside the events), median of `reps`.
    Three warm-up calls first.  Returns {workload name: {"rows": ...,
    "layer_totals": ...}}; the fp32 workload is latency-bound and gets no
    roofline fraction."""
    import torch
    wl = W.get(wid)
    inp = W.make_inputs(wl)
    if wl.dtype == "bf16":
        A = torch.from_numpy(inp.A_dev.view(np.int16)).view(torch.bfloat16).to(dev)
        G = torch.from_numpy(inp.G_dev.view(np.int16)).view(torch.bfloat16).to(dev)
        dt = L.BF16
    else:
        A = torch.from_numpy(inp.A_dev).to(dev)
        G = torch.from_numpy(inp.G_dev).to(dev)
        dt = L.F32
    B, T, d, p, k = wl.B, wl.T, wl.d, wl.p, wl.k
    f32 = dict(dtype=torch.float32, device=dev)
    q = {r: torch.empty(B, **f32) for r in ("hutch", "hutchpp", "exact_direct", "exact_ghost")}
    grad, scales = torch.empty(d, p, **f32), torch.empty(B, **f32)
    clipped = torch.empty(B, dtype=torch.uint8, device=dev)

    def ws_for(op, param):
        n = api.workspace_bytes(op, B, T, d, p, dt, param)
        return torch.empty(max(n, 256), dtype=torch.uint8, device=dev)

    ws = {"hutch": ws_for(L.OP_NORMS_HUTCH, k), "hutchpp": ws_for(L.OP_NORMS_HUTCHPP, k),
          "exact_direct": ws_for(L.OP_NORMS_EXACT, L.EXACT_DIRECT),
          "exact_ghost": ws_for(L.OP_NORMS_EXACT, L.EXACT_GHOST),
          "clipped_noisy_grad": ws_for(L.OP_CLIPPED_NOISY_GRAD, 0)}
    rows = WORKLOAD_ROWS[wid]
    # the gradient is clipped with the norms of the workload's first estimator
    qsrc = q["hutch"] if "hutch" in rows else q["exact_direct"]

    def call(r, step):
        if r == "hutch":
            api.norms_hutch(A, G, k, wl.seed, step, out=q[r], ws=ws[r])
        elif r == "hutchpp":
            api.norms_hutchpp(A, G, k, wl.seed, step, out=q[r], ws=ws[r])
        elif r == "exact_direct":
            api.norms_exact(A, G, L.EXACT_DIRECT, out=q[r], ws=ws[r])
        elif r == "exact_ghost":
            api.norms_exact(A, G, L.EXACT_GHOST, out=q[r], ws=ws[r])
        else:
            api.clipped_noisy_grad(A, G, qsrc, wl.C, wl.sigma, wl.seed, step, grad=grad,
                                   scales=scales, clipped=clipped, ws=ws[r])

    stream = torch.cuda.current_stream(dev)
    times = {r: [] for r in rows}
    large = A.numel() * A.element_size() + G.numel() * G.element_size() > L2_BYTES
    if large:
        timing = f"{reps} calls back to back per row (inputs larger than L2), median of 3 such blocks"
        for r in rows:
            for step in range(3):
                call(r, step)
            for blk in range(3):
                torch.cuda.synchronize(dev)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for step in range(reps):
                    call(r, 3 + step)
                e1.record(stream)
                torch.cuda.synchronize(dev)
                times[r].append(e0.elapsed_time(e1) / reps)
    else:
        timing = f"median of {reps} calls, L2 flushed before each"
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        for step in range(3 + reps):
            for r in rows:
                flush.fill_(step & 0xFF)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                call(r, step)
                e1.record(stream)
                torch.cuda.synchronize(dev)
                if step >= 3:
                    times[r].append(e0.elapsed_time(e1))
    for r in rows:
        if r in ws and api.workspace_status(ws[r]) != 0:
            raise SystemExit(f"{wl.name} {r}: device reported a status")
    work = algorithmic_work(wl)
    out = {}
    for r in rows:
        ms = statistics.median(times[r])
        if wl.dtype == "bf16":
            out[r] = row_entry(work[r], ms, B * T, peaks)
        else:
            out[r] = {"ms": round(ms, 4), "tokens_per_s": B * T / (ms * 1e-3), "bound": "latency"}
    totals = {}
    for r in rows:
        if r != "clipped_noisy_grad":
            ms = out[r]["ms"] + out["clipped_noisy_grad"]["ms"]
            totals[r + "+grad"] = {"ms": round(ms, 4), "tokens_per_s": B * T / (ms * 1e-3)}
    return {wl.name: {"B": B, "T": T, "d": d, "p": p, "k": k, "C": wl.C, "sigma": wl.sigma,
                      "timing": timing,
                      "rows": out, "layer_totals": totals}}


def algorithmic_work(wl):
    """Per-call algorithmic work of each row: (amount, unit, bound).
    Bytes are the compulsory HBM reads of A and G (bf16) plus outputs;
    flops are 2 per multiply-add of the defining products."""
    B, T, d, p, k = wl.B, wl.T, wl.d, wl.p, wl.k
    ag = 2.0 * B * T * (d + p)
    return {
        "hutch": (ag + 2.0 * k * p, "bytes", "hbm"),
        "hutchpp": (3.0 * ag, "bytes", "hbm"),
        "hutch_rademacher": (ag + 2.0 * k * p, "bytes", "hbm"),
        "hutchpp_rademacher": (3.0 * ag, "bytes", "hbm"),
        # exact direct norms that keep every A_i^T G_i, then the clipped sum
        # as one elementwise pass over them (read B d p fp32, write d p fp32)
        "exact_direct_stored": (2.0 * B * T * d * p, "flops", "tensor"),
        "stored_clipped_noisy_grad": (4.0 * (B + 1) * d * p, "bytes", "hbm"),
        # per-sample bias gradients and their squared norms: one read of G
        "bias_grads": (2.0 * B * T * p, "bytes", "hbm"),
        # the clipped noisy gradient applied to fp32 weights in its epilogue
        "clipped_noisy_grad_sgd": (2.0 * B * T * d * p, "flops", "tensor"),
        # FIBER step on d x p parameters: read g, read and write the parameter
        # and its four states (fp32)
        "fiber_step": (44.0 * d * p, "bytes", "hbm"),
        "clipped_noisy_grad_fiber": (2.0 * B * T * d * p, "flops", "tensor"),
        "exact_direct": (2.0 * B * T * d * p, "flops", "tensor"),
        "exact_ghost": (1.0 * B * T * (T + 1) * (d + p), "flops", "tensor"),
        "clipped_noisy_grad": (2.0 * B * T * d * p, "flops", "tensor"),
    }


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return {"hbm_gbs": pk["hbm_gbs"], "bf16_tflops": pk["bf16_tflops"],
                "bf16_tflops_sustained": pk.get("bf16_tflops_sustained", pk["bf16_tflops"]),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


def row_entry(work, ms, tokens, peaks):
    """Latency, tokens/s and roofline fraction of one row.  Tensor-bound rows
    run for well under a millisecond at full clock, so they are divided by the
    burst bf16 peak; the sustained (power-capped) peak is kept as a second
    fraction."""
    amount, unit, bound = work
    e = {"ms": round(ms, 4), "tokens_per_s": tokens / (ms * 1e-3), "bound": bound}
    if unit == "bytes":
        ach = amount / (ms * 1e-3) / 1e9
        e.update(achieved=round(ach, 2), peak=peaks["hbm_gbs"], unit="GB/s",
                 frac=round(ach / peaks["hbm_gbs"], 4))
    else:
        ach = amount / (ms * 1e-3) / 1e12
        e.update(achieved=round(ach, 2), peak=peaks["bf16_tflops"], unit="TFLOP/s",
                 frac=round(ach / peaks["bf16_tflops"], 4),
                 frac_sustained=round(ach / peaks["bf16_tflops_sustained"], 4))
    return e


class ClockSampler:
    """nvidia-smi samples (every 100 ms) of SM clocks and throttle reasons."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        """Ends sampling; summary() then reads any window of the samples."""
        self.rows = []
        if self.proc is None:
            return
        time.sleep(0.15)
        self.proc.terminate()
        self.proc.wait()
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    frac = float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                    rows.append((ts + frac, float(parts[2]), float(parts[3]), parts[5:]))
                except (ValueError, IndexError):
                    continue
        os.unlink(self.file.name)
        self.rows = rows

    def summary(self, t0: float, t1: float):
        """Median SM clock and the throttle reasons seen between t0 and t1
        (wall clock), from the samples inside the window, else the two
        nearest to it."""
        rows = getattr(self, "rows", [])
        if not rows:
            return None
        inside = [r for r in rows if t0 - 0.1 <= r[0] <= t1 + 0.1]
        use = inside or sorted(rows, key=lambda r: min(abs(r[0] - t0), abs(r[0] - t1)))[:2]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[j] for r in use for j, v in enumerate(r[3][1:5]) if v == "Active"})
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "reasons": reasons, "samples": len(use), "samples_in_window": len(inside)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def cpu_baseline(wl, reps: int = 1):
    """Times the fp64 oracle (as it stands) on a bounded sample of the
    workload: all of sample 0 (T tokens at full width), running every row.
    Much of the oracle's work (the noise over d x p, the Hutch++ basis over
    p) does not depend on the number of tokens, so a slice of the sample
    would understate its rate.  Returns (tokens/s, seconds, threads,
    sample description)."""
    import oracle as O
    from dp_sgd_clipping_gb300 import workloads as W
    sub = wl.with_(B=1)
    inp = W.make_inputs(sub)
    times = []
    for _ in range(reps):
        t0 = time.perf_counter()
        Ms = list(O.per_sample_grads(inp.A, inp.G))
        O.sqnorms_ghost(inp.A, inp.G)
        q_exact = np.array([np.sum(M * M) for M in Ms])
        P = O.hutch_probe(sub.p, sub.k, sub.seed, 0, "bf16")
        q_h = O.sqnorms_hutch(None, None, P, Ms=Ms)
        S, Gp = O.hutchpp_probes(sub.p, sub.k, sub.seed, 0, "bf16")
        O.sqnorms_hutchpp(None, None, S, Gp, Ms=Ms)
        O.clipped_noisy_grad(None, None, q_h, sub.C, sub.sigma, sub.seed, 0, Ms=Ms)
        times.append(time.perf_counter() - t0)
        del q_exact
    t = statistics.median(times)
    tall = sum(times)
    threads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    desc = (f"sample 0 ({wl.T} tokens, d={wl.d}, p={wl.p}), all rows (exact direct+ghost, "
            f"Hutch, Hutch++, clip, noisy grad); numpy fp64 with its BLAS on all host threads; "
            f"median of {reps} run(s), {tall:.1f} s in all")
    return wl.T / t, t, threads, desc


def run_reference(args, world, rank):
    """The oracle arm: rank 0 times the fp64 CPU oracle; other ranks idle.
    Each step is the measurement cpu_baseline makes: every row over all of
    sample 0 (4096 tokens at full width), so that this arm and the
    cpu_baseline of the GPU arm time the oracle the same way."""
    from dp_sgd_clipping_gb300 import workloads as W
    if rank != 0:
        return
    wl = W.get(WORKLOAD_ID)
    for _ in range(args.warmup):
        cpu_baseline(wl)
    t_total = 0.0
    for _ in range(args.steps):
        v, t, threads, desc = cpu_baseline(wl)
        t_total += t
    value = wl.T * args.steps / t_total
    desc = desc.replace("median of 1 run(s)", f"one run per step, {args.steps} steps")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * t_total / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(wl),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads,
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def config_of(wl):
    return {"workload": wl.name, "B": wl.B, "T": wl.T, "d": wl.d, "p": wl.p, "k": wl.k,
            "C": wl.C, "sigma": wl.sigma, "step": list(ROWS),
            "l2": "inputs larger than L2 (A+G = %.0f MB bf16 > 129 MB), two input sets "
                  "alternating between steps and between calls of a row"
                  % (2 * wl.B * wl.T * (wl.d + wl.p) / 1e6),
            "parallelism": "replicas"}


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="dpclip", choices=("dpclip", "reference"))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the extra (non-step) rows")
    ap.add_argument("--extra-rows", default=",".join(EXTRA_ROWS),
                    help="comma-separated subset of the extra rows (default: all)")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-workload rows of the other standard workloads")
    ap.add_argument("--rows", default=",".join(ROWS),
                    help="comma-separated subset of rows (default: all, the full step)")
    args = ap.parse_args()
    world, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, world, rank)
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    import torch
    import __graft_entry__
    __graft_entry__.build()
    from dp_sgd_clipping_gb300 import api
    from dp_sgd_clipping_gb300 import workloads as W

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    rows = tuple(r for r in args.rows.split(",") if r)
    wl = W.get(WORKLOAD_ID)
    inp = W.make_inputs(wl)
    A_h = torch.from_numpy(inp.A_dev.view(np.int16)).view(torch.bfloat16).pin_memory()
    G_h = torch.from_numpy(inp.G_dev.view(np.int16)).view(torch.bfloat16).pin_memory()
    A = A_h.to(dev)
    G = G_h.to(dev)
    B, T, d, p, k = wl.B, wl.T, wl.d, wl.p, wl.k
    f32 = dict(dtype=torch.float32, device=dev)
    q_h, q_pp, q_d, q_g = (torch.empty(B, **f32) for _ in range(4))
    grad = torch.empty(d, p, **f32)
    scales = torch.empty(B, **f32)
    clipped = torch.empty(B, dtype=torch.uint8, device=dev)
    from dp_sgd_clipping_gb300 import _lib as L

    def ws_for(op, param):
        n = api.workspace_bytes(op, B, T, d, p, L.BF16, param)
        return torch.empty(max(n, 256), dtype=torch.uint8, device=dev)

    ws = {"hutch": ws_for(L.OP_NORMS_HUTCH, k), "hutchpp": ws_for(L.OP_NORMS_HUTCHPP, k),
          "exact_direct": ws_for(L.OP_NORMS_EXACT, L.EXACT_DIRECT),
          "exact_ghost": ws_for(L.OP_NORMS_EXACT, L.EXACT_GHOST),
          "clipped_noisy_grad": ws_for(L.OP_CLIPPED_NOISY_GRAD, 0)}
    stored = {}   # StoredGradients of the stored-direct extra rows

    def ensure_stored_ws():
        if "ws" not in stored:
            stored["ws"] = ws_for(L.OP_STORED_DIRECT, 0)
        return stored["ws"]
    stream = torch.cuda.current_stream(dev)
    # Two layers' worth of inputs (the second: the same samples in reverse
    # order, at other addresses), used by alternate steps and calls, so that
    # no timed call finds its inputs in L2 from the call before it (the
    # inputs, 336 MB, exceed L2, but one of them, A, does not)
    sets = [None, {"A": A.flip(0).contiguous(), "G": G.flip(0).contiguous(),
                   "q_h": torch.empty(B, **f32), "q_pp": torch.empty(B, **f32),
                   "q_d": torch.empty(B, **f32), "q_g": torch.empty(B, **f32),
                   "grad": torch.empty(d, p, **f32), "scales": torch.empty(B, **f32),
                   "clipped": torch.empty(B, dtype=torch.uint8, device=dev)}]

    def row_fn(name, step, bufs=None):
        """The ABI call of one row of the step on a set of buffers."""
        b = bufs or {"A": A, "G": G, "q_h": q_h, "q_pp": q_pp, "q_d": q_d, "q_g": q_g,
                     "grad": grad, "scales": scales, "clipped": clipped}
        if name == "hutch":
            return lambda: api.norms_hutch(b["A"], b["G"], k, wl.seed, step, out=b["q_h"], ws=ws[name])
        if name == "hutchpp":
            return lambda: api.norms_hutchpp(b["A"], b["G"], k, wl.seed, step, out=b["q_pp"],
                                             ws=ws[name])
        if name == "hutch_rademacher":
            return lambda: api.norms_hutch(b["A"], b["G"], k, wl.seed, step, out=b["q_h"],
                                           ws=ws["hutch"], probe="rademacher")
        if name == "hutchpp_rademacher":
            return lambda: api.norms_hutchpp(b["A"], b["G"], k, wl.seed, step, out=b["q_pp"],
                                             ws=ws["hutchpp"], probe="rademacher")
        if name == "exact_direct":
            return lambda: api.norms_exact(b["A"], b["G"], L.EXACT_DIRECT, out=b["q_d"], ws=ws[name])
        if name == "exact_direct_stored":
            def call():
                _, stored["h"] = api.norms_direct_store(b["A"], b["G"], sqnorms=b["q_d"],
                                                        ws=ensure_stored_ws())
            return call
        if name == "bias_grads":
            if "bias_ws" not in stored:
                stored["bias_ws"] = ws_for(L.OP_BIAS, 0)
                stored["bias"] = torch.empty(B, p, **f32)
            return lambda: L.check("dpclip_bias_grads", L.lib.dpclip_bias_grads(
                b["G"].data_ptr(), B, T, p, L.BF16, 1, b["q_d"].data_ptr(),
                stored["bias"].data_ptr(), stored["bias_ws"].data_ptr(),
                stored["bias_ws"].numel(), stream.cuda_stream))
        if name == "clipped_noisy_grad_sgd":
            if "theta" not in stored:
                stored["theta"] = torch.zeros(d, p, **f32)
            upd = api.SGDUpdate(stored["theta"], 1e-3, float(B), store_grad=False)
            return lambda: api.clipped_noisy_grad(b["A"], b["G"], b["q_h"], wl.C, wl.sigma, wl.seed,
                                                  step, scales=b["scales"], clipped=b["clipped"],
                                                  ws=ws["clipped_noisy_grad"], update=upd)
        if name in ("fiber_step", "clipped_noisy_grad_fiber"):
            if "fiber" not in stored:
                nv = (wl.sigma * wl.C / B) ** 2
                stored["fiber"] = api.FiberAdamW(torch.zeros(d, p, **f32), lr=1e-4, denom=float(B),
                                                 noise_var=nv)
            if name == "fiber_step":
                return lambda: api.fiber_step(b["grad"], stored["fiber"])
            return lambda: api.clipped_noisy_grad(b["A"], b["G"], b["q_h"], wl.C, wl.sigma, wl.seed,
                                                  step, grad=b["grad"], scales=b["scales"],
                                                  clipped=b["clipped"], ws=ws["clipped_noisy_grad"],
                                                  fiber=stored["fiber"])
        if name == "stored_clipped_noisy_grad":
            if "h" not in stored:
                row_fn("exact_direct_stored", step, bufs)()
            return lambda: api.stored_clipped_noisy_grad(stored["h"], b["q_d"], wl.C, wl.sigma,
                                                         wl.seed, step, grad=b["grad"],
                                                         scales=b["scales"], clipped=b["clipped"])
        if name == "exact_ghost":
            return lambda: api.norms_exact(b["A"], b["G"], L.EXACT_GHOST, out=b["q_g"], ws=ws[name])
        return lambda: api.clipped_noisy_grad(b["A"], b["G"], b["q_h"], wl.C, wl.sigma, wl.seed, step,
                                              grad=b["grad"], scales=b["scales"],
                                              clipped=b["clipped"], ws=ws[name])

    def barrier():
        torch.cuda.synchronize(dev)
        if pg is not None:
            pg.barrier()
        torch.cuda.synchronize(dev)

    # ---------------------------------------------------------------- device-resident timing
    for s in range(args.warmup):
        for r in rows:
            row_fn(r, s, sets[s % 2])()
    vis = [x for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x.strip()]
    smi_index = int(vis[local]) if local < len(vis) and vis[local].strip().isdigit() else local
    clocks = ClockSampler(smi_index)
    if rank == 0:
        clocks.start()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(rows) + 1)]
          for _ in range(args.steps)]
    barrier()
    wall0 = time.time()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for s in range(args.steps):
        for r in rows:
            row_fn(r, args.warmup + s, sets[s % 2])()
    end.record(stream)
    barrier()
    wall1 = time.time()
    elapsed_ms = start.elapsed_time(end)
    # Per-row durations, two ways.  row_ms: each row alone, calls back to
    # back between one event pair (the steady state of a loop over layers:
    # each call's launch and prologue overlap the previous call's tail; the
    # inputs are larger than L2), see below.  in_step_ms: a second pass of the step
    # with an event pair around every row; an event between two calls keeps
    # the second call's first kernel from launching early, so these rows add
    # up to a little more than the step timed above.
    for s in range(args.steps):
        ev[s][0].record(stream)
        for j, r in enumerate(rows):
            row_fn(r, args.warmup + s, sets[s % 2])()
            ev[s][j + 1].record(stream)
    barrier()
    in_step_ms = {r: statistics.mean(ev[s][j].elapsed_time(ev[s][j + 1])
                                     for s in range(args.steps))
                  for j, r in enumerate(rows)}
    # Three such blocks per row, the median kept, so that a stall of the host
    # or the box during one block does not decide a row's figure.  Long runs
    # of one tensor-bound row can reach the board's power cap (sw_power_cap,
    # SM clock near 1.84 GHz seen in the ghost row), which the mixed step
    # does not: clocks_rows records the clocks of these passes, and the
    # roofline below uses the rows as timed inside the step.
    row_ms = {}
    for r in rows:
        for s_ in range(3):
            row_fn(r, s_, sets[s_ % 2])()
        blocks = []
        for b_ in range(3):
            barrier()
            r0 = torch.cuda.Event(enable_timing=True)
            r1 = torch.cuda.Event(enable_timing=True)
            r0.record(stream)
            for s_ in range(args.steps):
                row_fn(r, args.warmup + s_, sets[s_ % 2])()
            r1.record(stream)
            barrier()
            blocks.append(r0.elapsed_time(r1) / args.steps)
        row_ms[r] = statistics.median(blocks)
    wall2 = time.time()
    if rank == 0:
        clocks.stop()
    # the step's window, and the window of the rows timed alone (long runs of
    # one tensor-bound row draw more power than the mixed step)
    clk = clocks.summary(wall0, wall1) if rank == 0 else None
    clk_rows = clocks.summary(wall1, wall2) if rank == 0 else None
    for name in rows:
        if name not in ws:
            continue
        st = api.workspace_status(ws[name])
        if st != 0:
            raise SystemExit(f"{name}: device reported status {st}")
    elapsed_ms = max_over_ranks(elapsed_ms, pg, dev)

    # ---------------------------------------------------------------- end to end, host buffers
    # Every step copies its inputs from pinned host memory and its results
    # (the four norm vectors, the gradient, scales, flags) back to pinned host
    # memory.  Steps are pipelined the way a training loop would run them:
    # two device buffer sets; step s+1's inputs travel on a copy stream and
    # step s-1's results on another while step s computes.
    e2e = None
    if not args.no_e2e:
        def buffer_set():
            return {"A": torch.empty_like(A), "G": torch.empty_like(G),
                    "q_h": torch.empty(B, **f32), "q_pp": torch.empty(B, **f32),
                    "q_d": torch.empty(B, **f32), "q_g": torch.empty(B, **f32),
                    "grad": torch.empty(d, p, **f32), "scales": torch.empty(B, **f32),
                    "clipped": torch.empty(B, dtype=torch.uint8, device=dev)}

        def host_set():
            return {"q": torch.empty(4, B, dtype=torch.float32).pin_memory(),
                    "grad": torch.empty(d, p, dtype=torch.float32).pin_memory(),
                    "scales": torch.empty(B, dtype=torch.float32).pin_memory(),
                    "clipped": torch.empty(B, dtype=torch.uint8).pin_memory()}

        bufs = [buffer_set(), buffer_set()]
        hosts = [host_set(), host_set()]
        qs = [torch.empty(4, B, **f32), torch.empty(4, B, **f32)]
        s_h2d = torch.cuda.Stream(dev)
        s_d2h = torch.cuda.Stream(dev)
        ev = lambda: torch.cuda.Event()
        h2d_done = [ev(), ev()]
        comp_done = [ev(), ev()]
        d2h_done = [ev(), ev()]
        for e in comp_done + d2h_done:
            e.record(stream)

        def e2e_step(sidx):
            bi = sidx % 2
            bset, hset = bufs[bi], hosts[bi]
            with torch.cuda.stream(s_h2d):
                s_h2d.wait_event(comp_done[bi])        # step sidx-2 no longer reads them
                bset["A"].copy_(A_h, non_blocking=True)
                bset["G"].copy_(G_h, non_blocking=True)
                h2d_done[bi].record(s_h2d)
            stream.wait_event(h2d_done[bi])
            stream.wait_event(d2h_done[bi])            # step sidx-2's results are out
            for r in rows:
                row_fn(r, sidx, bset)()
            for j, key in enumerate(("q_h", "q_pp", "q_d", "q_g")):
                qs[bi][j].copy_(bset[key])
            comp_done[bi].record(stream)
            with torch.cuda.stream(s_d2h):
                s_d2h.wait_event(comp_done[bi])
                hset["q"].copy_(qs[bi], non_blocking=True)
                hset["grad"].copy_(bset["grad"], non_blocking=True)
                hset["scales"].copy_(bset["scales"], non_blocking=True)
                hset["clipped"].copy_(bset["clipped"], non_blocking=True)
                d2h_done[bi].record(s_d2h)

        for sidx in range(args.warmup):
            e2e_step(sidx)
        stream.wait_event(d2h_done[0])
        stream.wait_event(d2h_done[1])
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for e in comp_done + d2h_done:          # the copy streams start after e0
            e.record(stream)
        for sidx in range(args.steps):
            e2e_step(args.warmup + sidx)
        stream.wait_event(d2h_done[0])
        stream.wait_event(d2h_done[1])
        e1.record(stream)
        barrier()
        e2e_ms = e0.elapsed_time(e1)
        e2e_ms = max_over_ranks(e2e_ms, pg, dev)
        h2d = A_h.numel() * 2 + G_h.numel() * 2
        d2h = sum(t.numel() * t.element_size() for t in hosts[0].values())
        e2e = {"value": job_tokens_per_s(world, B * T, args.steps, e2e_ms), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e2e_ms / args.steps,
               "pipelining": "inputs of step s+1 and results of step s-1 copied on two "
                             "copy streams while step s computes"}

    # ---------------------------------------------------------------- extra rows (not in the step)
    extra_ms = {}
    if not args.no_extra:
        for r in (x for x in args.extra_rows.split(",") if x):
            if r not in EXTRA_ROWS:
                raise SystemExit(f"unknown extra row {r}")
            for s_ in range(args.warmup):
                row_fn(r, s_)()
            barrier()
            x0 = torch.cuda.Event(enable_timing=True)
            x1 = torch.cuda.Event(enable_timing=True)
            x0.record(stream)
            for s_ in range(args.steps):
                row_fn(r, args.warmup + s_)()
            x1.record(stream)
            barrier()
            extra_ms[r] = x0.elapsed_time(x1) / args.steps

    # ---------------------------------------------------------------- the other workloads
    peaks = load_peaks()
    per_config = {}
    if not args.no_configs:
        for wid in OTHER_WORKLOADS:
            per_config.update(time_workload(api, L, W, wid, dev, min(args.steps, 20), peaks))

    if rank != 0:
        if pg is not None:
            pg.barrier()
            pg.destroy_process_group()
        return

    # ---------------------------------------------------------------- roofline and report
    work = algorithmic_work(wl)
    breakdown = {}
    for r in rows:
        breakdown[r] = row_entry(work[r], row_ms[r], B * T, peaks)
        breakdown[r]["algorithmic"] = work[r][0]
        breakdown[r]["in_step_ms"] = round(in_step_ms[r], 4)
    extra = {}
    for r, ms in extra_ms.items():
        extra[r] = row_entry(work[r], ms, B * T, peaks)
    if "exact_direct_stored" in extra_ms and "stored_clipped_noisy_grad" in extra_ms:
        # exact norms + clipped noisy gradient of the layer, against the same
        # two results from exact_direct + clipped_noisy_grad (two GEMMs)
        ms = extra_ms["exact_direct_stored"] + extra_ms["stored_clipped_noisy_grad"]
        extra["layer_exact_stored_total"] = {"ms": round(ms, 4),
                                             "tokens_per_s": B * T / (ms * 1e-3)}
    # per-layer totals: one norm method, then clip + clipped noisy gradient
    layer_totals = {}
    if "clipped_noisy_grad" in row_ms:
        for r in ("hutch", "hutchpp", "exact_direct", "exact_ghost"):
            if r in row_ms:
                ms = row_ms[r] + row_ms["clipped_noisy_grad"]
                layer_totals[r + "+grad"] = {"ms": round(ms, 4), "tokens_per_s": B * T / (ms * 1e-3)}
    # The dominant row's roofline as it runs inside the step (the second,
    # event-bracketed pass of the step: same mix and clocks as the timed
    # region, whose clock record shows full clock and no throttle reason).
    dom = max(rows, key=lambda r: in_step_ms[r])
    traffic = _traffic_from_profiles(dom)
    roof = row_entry(work[dom], in_step_ms[dom], B * T, peaks)
    roofline = {"kernel": dom, "bound": roof["bound"], "achieved": roof["achieved"],
                "peak": roof["peak"], "unit": roof["unit"], "frac": roof["frac"],
                "traffic": traffic, "timing": "inside the step (in_step_ms of the row)",
                "peak_source": peaks["source"] + (
                    " (burst bf16: a sub-millisecond kernel at full clock)"
                    if roof["unit"] == "TFLOP/s" else " (HBM copy)")}
    if "frac_sustained" in roof:
        roofline["frac_sustained"] = roof["frac_sustained"]
    ms_step = elapsed_ms / args.steps
    line = {"metric": METRIC, "value": job_tokens_per_s(world, B * T, args.steps, elapsed_ms),
            "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": config_of(wl), "gpu_launches": args.steps * sum(LAUNCHES[r] for r in rows),
            "roofline": roofline, "breakdown": breakdown, "layer_totals": layer_totals,
            "extra_rows": extra, "configs": per_config, "clocks": clk, "clocks_rows": clk_rows,
            "e2e": e2e}
    if world == 1 and not args.no_cpu_baseline:
        # all of sample 0 (its tokens-independent work, the noise and the
        # Hutch++ basis over p, is then shared by 4096 tokens), twice
        v, t, threads, desc = cpu_baseline(wl, reps=2)
        line["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": threads,
                                "kind": "oracle", "sample": desc, "seconds": round(t, 2)}
    print(json.dumps(line), flush=True)
    if pg is not None:
        pg.barrier()
        pg.destroy_process_group()


def _sha256(path):
    """Digest of a source file's code: comments and whitespace are dropped, so
    that a capture stays valid across comment edits but not code edits."""
    import hashlib
    import re
    with open(path, encoding="utf-8") as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    text = re.sub(r"\s+", " ", text).strip()
    return hashlib.sha256(text.encode("utf-8")).hexdigest()


def _traffic_from_profiles(row):
    """DRAM bytes per launch of the row's main kernel from the committed ncu
    summary (profiles/traffic.json), or None when there is no capture or when
    any source file of the kernel changed since the capture (hash mismatch)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            entry = json.load(f).get(row)
    except (OSError, ValueError):
        return None
    if not entry:
        return None
    for src, digest in entry.get("sources", {}).items():
        p = os.path.join(ROOT, src)
        if not os.path.exists(p) or _sha256(p) != digest:
            return None
    return entry.get("dram_bytes_per_launch")


def max_over_ranks(value: float, dist=None, device=None) -> float:
    """Largest `value` over all ranks (the job's time is its slowest rank)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world: int, tokens_per_step: int, steps: int, elapsed_ms: float) -> float:
    """Whole-job throughput: every rank processes its own batch each step."""
    return world * tokens_per_step * steps / (elapsed_ms / 1e3)


if __name__ == "__main__":
    main()
