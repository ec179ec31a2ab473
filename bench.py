#!/usr/bin/env python
"""Benchmark of the GB300 exact solver (Dixon p-adic lifting).

One step = one full exact solve (range check + Hadamard terms, batched
modular inverse over all 53 primes, the m-step lift, digits to host, host
rational reconstruction) of the n=1024, c=1 system with 24-bit entries
(uniform in [-2^23, 2^23), seed 0): the workload the exact-solve card's
§Measured table quotes (24-bit entries, n = 1024, c = 1).  --workload names
another system of inputs.WORKLOADS (the rest of that table's grid, the
planted and scaled-Hilbert systems, the test configurations).

Prints ONE JSON line (rank 0).  `value` = ms per solve with A and b already
in HBM (CUDA events on the solve's stream; the host reconstruction is inside
the bracket because the call returns only once it is done); L2 is flushed
(256 MiB write) between timed steps.  `e2e` = the same through es_solve with
pinned host buffers (host->device copy of A and b and device->host copy of
the results inside the timed region).  `roofline` = the lift's dominant
kernel (at c = 1 the fused lift, all m steps in one launch), its algorithmic
bytes per launch over its CUDA-event launch time; the fused lift reads B_j
from L2 after the first step, so its bound is labelled "l2/latency" and its
DRAM traffic is given beside the algorithmic bytes.  `configs` carries the
n = 4096, c = 64 system (16-bit entries) measured in the same run: ms per
solve, phases, lift time per step, and the tcgen05 product's roofline with
its tensor-pipe and HBM fractions and whichever binds.  `cpu_baseline` =
the CPU oracle (Python-int Bareiss) on leading principal subsystems of the
same system, extrapolated to n.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
  torchrun --nproc-per-node N bench.py --gpus N ...   (independent replicas, one per GPU)
"""

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "full exact-solve ms at n=1024,c=1"
WORKLOAD = "n1024_c1_24bit"
# exact-solve card §Measured: median full solves with 24-bit entries on H200 (the
# faster of its two GPUs at n = 1024: 2411 ms RTX PRO 6000 Blackwell / 2235 ms H200).
# Another machine's numbers: context for --workload runs of the same grid point.
PAGES_H200_MS = {"n128_c1_24bit": 33.0, "n256_c1_24bit": 97.0, "n512_c1_24bit": 437.0,
                 "n1024_c1_24bit": 2235.0, "n256_c16_24bit": 448.0, "n512_c16_24bit": 2624.0}
L2_FLUSH_BYTES = 256 << 20
# the card's multi-column regime at full size, measured beside the headline
MANY_COLUMN_WORKLOAD = "n4096_c64_16bit"


def metric_for(workload):
    return METRIC if workload == WORKLOAD else "full exact-solve ms (%s)" % workload


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=5)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    p.add_argument("--workload", default=WORKLOAD)
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--cpu-budget", type=float, default=20.0, help="seconds of oracle work for cpu_baseline")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-many-column", action="store_true",
                   help="skip the n=4096, c=64 figures that the default line carries under `configs`")
    p.add_argument("--c5-steps", type=int, default=3, help="timed solves of the n=4096, c=64 system")
    p.add_argument("--lift-only", type=int, default=0, metavar="K",
                   help="profiling aid: inverse once, then time lifts of K steps only (es_lift_device); "
                        "prints a lift line instead of the solve line")
    p.add_argument("--one-stream", action="store_true",
                   help="inverse on the solve's stream alone (for profilers that do not see the SM partitions)")
    return p.parse_args()


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


def max_over_ranks(x, dist, device):
    """The largest of every rank's x (each replica's time; the job ends with the slowest)."""
    if dist is None:
        return x
    import torch

    t = torch.tensor([x], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ clocks
class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return
        # the sampler's start-up takes host cores for a while: let it reach its
        # first sample before the timed region begins (it keeps sampling there)
        t0 = time.time()
        while time.time() - t0 < 3.0 and self.proc.poll() is None:
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.05)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.3)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if "Active" in r[5 + i] and "Not" not in r[5 + i]})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ oracle baseline
def oracle_sample(A, b, budget_s, sizes=None):
    """Time the CPU oracle (as it stands) on leading principal subsystems of
    the same system, growing k until the budget is spent; fit t = C k^alpha on
    the two largest and extrapolate to n.  Returns (ms at n, description)."""
    from oracle import exact

    n = A.shape[0]
    pts = []
    spent = 0.0
    sizes = sizes or (32, 48, 64, 80, 96, 112, 128, 160, 192, 224, 256)
    if n <= sizes[0]:
        sizes = (n,)  # small systems: the whole solve
    for k in sizes:
        if k > n:
            break
        t0 = time.perf_counter()
        exact.solve(A[:k, :k].tolist(), b[:k].tolist())
        dt = time.perf_counter() - t0
        pts.append((k, dt))
        spent += dt
        if spent > budget_s or dt * 2.5 > budget_s - spent:
            break
    if pts[-1][0] == n:
        return pts[-1][1] * 1e3, f"oracle full solve at n={n}", pts
    (k1, t1), (k2, t2) = pts[-2], pts[-1]
    alpha = math.log(t2 / t1) / math.log(k2 / k1)
    est = t2 * (n / k2) ** alpha
    desc = (f"oracle (Python-int Bareiss + back-substitution) on the leading k x k subsystems of the same "
            f"system, k={[k for k, _ in pts]} ({spent:.1f} s, 1 core); t(k) = C k^{alpha:.2f} fitted on "
            f"k={k1},{k2} and extrapolated to n={n}")
    return est * 1e3, desc, pts


def load_peaks():
    """(HBM GB/s, 16-bit tensor TFLOP/s sustained, "measured" | "fallback")."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"])), "measured"
    except Exception:
        return 6800.0, 1700.0, "fallback"


KERNEL_SOURCE = {"k_lift_fused": "k_lift_fused.cu", "k_lift_gemv": "k_lift.cu", "k_lift_gemm": "k_lift.cu",
                 "k_lift_gemm_tc": "k_lift_tc.cu"}


def traffic_for(kernel, workload):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu
    summaries (profiles/traffic.json, keyed by kernel and workload), if the
    kernel's source has not changed since the capture; else None."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)[kernel][workload]
        src = os.path.join(ROOT, "dixon_adic_lifting_gb300", "csrc", KERNEL_SOURCE[kernel])
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()
        return float(t["dram_bytes_per_launch"]) if t.get("source_sha256") == h else None
    except Exception:
        return None


class SolveFigures:
    """The per-solve figures the bench line reports, without the result."""

    def __init__(self, s):
        for k in ("n", "c", "m", "primes_used", "launches", "phase_ms", "top_kernel", "top_launches", "top_ms",
                  "top_bytes_per_launch"):
            setattr(self, k, getattr(s, k))


# ------------------------------------------------------------------ arms
def run_reference(args, rank, world):
    """The oracle as the reference arm: each step a bounded sample of the same
    workload (leading subsystems), extrapolated to the full solve."""
    import numpy as np  # noqa: F401
    from dixon_adic_lifting_gb300 import inputs

    if rank != 0:
        return
    A, b = inputs.workload(args.workload, seed=args.seed)
    sizes = (48, 64, 96, 128)
    for _ in range(args.warmup):
        oracle_sample(A, b, 1e9, sizes=(32, 48))
    vals, desc = [], ""
    t0 = time.perf_counter()
    for _ in range(args.steps):
        v, desc, _ = oracle_sample(A, b, 1e9, sizes=sizes)
        vals.append(v)
    wall = time.perf_counter() - t0
    v = statistics.median(vals)
    line = {"impl": "reference", "metric": metric_for(args.workload), "value": v, "unit": "ms", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": v, "higher_is_better": False,
            "scaling": "weak",
            "vs_baseline": (v / PAGES_H200_MS[args.workload]) if args.workload in PAGES_H200_MS else None,
            "dtype": "int (Python big integers)",
            "data": "synthetic", "config": {"workload": args.workload, "seed": args.seed},
            "cpu_baseline": {"value": v, "unit": "ms", "cores": 1, "kind": "oracle", "sample": desc},
            "e2e": {"value": v, "unit": "ms", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": round(wall, 1)}
    print(json.dumps(line), flush=True)


def roofline_of(fig, workload, hbm_peak, tensor_peak, peak_kind):
    """Roofline object of the lift's dominant kernel from a list of solve
    figures: algorithmic bytes (and, for the many-column tensor-core product,
    MMA operations) per launch over the mean CUDA-event launch time."""
    s0 = fig[-1]
    launches = sum(s.top_launches for s in fig)
    launch_ms = sum(s.top_ms for s in fig) / max(launches, 1)
    secs = launch_ms * 1e-3
    bytes_launch = s0.top_bytes_per_launch
    gbs = bytes_launch / secs / 1e9 if secs > 0 else 0.0
    traffic = traffic_for(s0.top_kernel, workload)
    r = {"kernel": s0.top_kernel, "launch_us": round(launch_ms * 1e3, 3), "launches_per_solve": s0.top_launches,
         "bytes_per_launch": bytes_launch, "traffic": traffic, "peak_kind": peak_kind}
    if s0.top_kernel == "k_lift_gemm_tc":
        # 2 E' n^2 c multiply-adds of residues per step (f16 MMA, exact)
        ops = 2.0 * s0.primes_used * s0.n * s0.n * s0.c
        tflops = ops / secs / 1e12 if secs > 0 else 0.0
        t_tensor, t_hbm = ops / (tensor_peak * 1e12), bytes_launch / (hbm_peak * 1e9)
        bound = "tensor" if t_tensor >= t_hbm else "hbm"
        r.update({"bound": bound, "unit": "GB/s" if bound == "hbm" else "TFLOP/s",
                  "achieved": round(gbs if bound == "hbm" else tflops, 1),
                  "peak": hbm_peak if bound == "hbm" else tensor_peak,
                  "frac": round(max(t_tensor, t_hbm) / secs, 4) if secs > 0 else 0.0,
                  "ops_per_launch": ops, "tflops": round(tflops, 1),
                  "tensor_frac": round(tflops / tensor_peak, 4), "hbm_gbs": round(gbs, 1),
                  "hbm_frac": round(gbs / hbm_peak, 4),
                  "tensor_peak": tensor_peak, "hbm_peak": hbm_peak,
                  "tensor_peak_note": "16-bit MMA, sustained (kind::f16 operands; the part has no integer MMA kind)"})
    elif s0.top_kernel == "k_lift_fused":
        # all m steps in one launch; B is L2-resident after the first step, so
        # the bound that binds is L2 / shared-memory delivery and the two grid
        # barriers per step, not HBM: frac is against HBM, labelled as such
        r.update({"bound": "l2/latency", "unit": "GB/s", "achieved": round(gbs, 1), "peak": hbm_peak,
                  "frac": round(gbs / hbm_peak, 4), "frac_of": "HBM copy bandwidth (algorithmic bytes; "
                  "served from L2 after the first step)",
                  "dram_frac": round(traffic / bytes_launch, 4) if traffic else None})
    else:
        r.update({"bound": "hbm", "unit": "GB/s", "achieved": round(gbs, 1), "peak": hbm_peak,
                  "frac": round(gbs / hbm_peak, 4)})
    return r


def time_solves(api, torch, At, bt, steps, warmup, one_stream, flush):
    """Warm-up solves, then `steps` solves each bracketed by CUDA events on the
    solve's stream (L2 flushed before each); returns (ms per step, figures)."""
    stream = torch.cuda.current_stream()
    for _ in range(warmup):  # the same call as the timed ones
        s = api.solve_device(At, bt, stream=stream, timing=2, one_stream=one_stream)
    s = None
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    fig = []
    torch.cuda.synchronize()
    for k in range(steps):
        flush.zero_()
        ev[k][0].record(stream)
        s = api.solve_device(At, bt, stream=stream, timing=2, one_stream=one_stream)
        ev[k][1].record(stream)
        # keep the step's figures, not its result: a caller that drops each
        # result lets the next solve reuse its page-locked block
        fig.append(SolveFigures(s))
        s = None
    torch.cuda.synchronize()
    return [e0.elapsed_time(e1) for e0, e1 in ev], fig


PHASES = ["stats_residues", "inverse", "lift", "digits_d2h", "reconstruct_host", "total_wall"]


def many_column_figures(api, torch, args, flush, hbm_peak, tensor_peak, peak_kind):
    """The n = 4096, c = 64 system (16-bit entries): ms per solve, phases, lift
    time per step and the tensor-core product's roofline."""
    from dixon_adic_lifting_gb300 import inputs

    name = MANY_COLUMN_WORKLOAD
    A, b = inputs.workload(name, seed=args.seed)
    n, c = A.shape[0], b.shape[1]
    At = torch.as_tensor(A, device="cuda")
    bt = torch.as_tensor(b, device="cuda")
    step_ms, fig = time_solves(api, torch, At, bt, args.c5_steps, 1, args.one_stream, flush)
    s0 = fig[-1]
    phases = {k: round(statistics.mean(s.phase_ms[i] for s in fig), 3) for i, k in enumerate(PHASES)}
    lift_us = phases["lift"] * 1e3 / s0.m
    E = s0.primes_used
    step_bytes = E * n * n + 2 * n * n  # B_j once, A as 16-bit
    del At, bt
    return {"workload": name, "n": n, "c": c, "entries": inputs.WORKLOADS[name].description, "seed": args.seed,
            "m": s0.m, "primes_used": E, "steps": args.c5_steps, "warmup": 1,
            "ms_per_solve": round(statistics.mean(step_ms), 3), "step_ms": [round(x, 2) for x in step_ms],
            "phases_ms": phases,
            "lift_us_per_step": round(lift_us, 2),
            "lift_step": {"bytes": step_bytes, "gbs": round(step_bytes / (lift_us * 1e-6) / 1e9, 1),
                          "hbm_frac": round(step_bytes / (lift_us * 1e-6) / 1e9 / hbm_peak, 4),
                          "note": "whole step (product, CRT digit, residual update, residues of r_{i+1}) "
                                  "against E' n^2 + 2 n^2 bytes"},
            "roofline": roofline_of(fig, name, hbm_peak, tensor_peak, peak_kind)}


def run_lift_only(args):
    """Inverse once, then `warmup` + `steps` lifts of K steps through
    es_lift_device (little device memory: no digit store for the whole solve,
    no reconstruction); prints the mean lift time per step."""
    import torch

    from dixon_adic_lifting_gb300 import _lib, api, build as _b, inputs

    if not _b.up_to_date():
        _b.build()
    _lib.load()
    A, b = inputs.workload(args.workload, seed=args.seed)
    At = torch.as_tensor(A, device="cuda")
    bt = torch.as_tensor(b, device="cuda")
    B, good = api.inverse_mod_device(At)
    K = args.lift_only
    for _ in range(args.warmup):
        api.lift_device(At, bt, B, good, K)
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(args.steps):
        api.lift_device(At, bt, B, good, K)
    e1.record(stream)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / (args.steps * K)
    print(json.dumps({"lift_only": args.workload, "steps_per_lift": K, "lifts": args.steps,
                      "us_per_step": round(us, 2), "primes_used": int(good.sum().item())}), flush=True)


def run_gb300(args, rank, local_rank, world):
    import numpy as np  # noqa: F401
    import torch

    from dixon_adic_lifting_gb300 import _lib, api, build as _b, inputs

    if not _b.up_to_date():
        _b.build()
    _lib.load()
    assert torch.cuda.is_available(), "bench needs a CUDA device"
    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    A, b = inputs.workload(args.workload, seed=args.seed)
    n, c = A.shape[0], b.shape[1]
    At = torch.as_tensor(A, device="cuda")
    bt = torch.as_tensor(b, device="cuda")
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    hbm_peak, tensor_peak, peak_kind = load_peaks()
    clocks = Clocks(local_rank)
    # the sampler starts before the warm-up, so that the timed solves follow
    # the warm-up ones with no idle gap (after one the host pool's workers and
    # the cores are asleep) and still run with the sampler going
    clocks.start()
    for _ in range(args.warmup):  # the same call as the timed ones
        api.solve_device(At, bt, stream=torch.cuda.current_stream(), timing=2, one_stream=args.one_stream)
    barrier()
    step_ms, sols = time_solves(api, torch, At, bt, args.steps, 0, args.one_stream, flush)
    barrier()
    ms = max_over_ranks(sum(step_ms) / len(step_ms), dist, "cuda")
    s0 = sols[-1]
    phases = {k: round(statistics.mean(s.phase_ms[i] for s in sols), 4) for i, k in enumerate(PHASES)}
    roof = roofline_of(sols, args.workload, hbm_peak, tensor_peak, peak_kind)

    # e2e through the host API, pinned host buffers
    e2e = None
    if not args.no_e2e:
        Ah = torch.empty((n, n), dtype=torch.int64, pin_memory=True)
        bh = torch.empty((n, c), dtype=torch.int64, pin_memory=True)
        Ah.copy_(torch.as_tensor(A))
        bh.copy_(torch.as_tensor(b))
        An, bn = Ah.numpy(), bh.numpy()
        for _ in range(2):
            api.solve_canonical(An, bn)
        times = []
        for _ in range(args.steps):
            flush.zero_()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            s = api.solve_canonical(An, bn)
            times.append((time.perf_counter() - t0) * 1e3)
        e2e_ms = max_over_ranks(sum(times) / len(times), dist, "cuda")
        # device->host: sampled components' digits (4 x m digits: 48 B each as a
        # copy, 96 B each as the fused lift's self-tagged stream for c = 1,
        # n <= 1024), the numerators (n c limbs x 8 B), the acceptance flags
        # (n c B) and the good-prime flags
        per_digit = 96 if (c == 1 and n <= 1024) else 48
        e2e = {"value": round(e2e_ms, 4), "unit": "ms", "h2d_bytes_per_step": int(8 * (n * n + n * c)),
               "d2h_bytes_per_step": int(min(4, n * c) * s.m * per_digit + n * c * s.limbs * 8 + n * c + 53)}
        s = None

    many = None
    if args.workload == WORKLOAD and not args.no_many_column:
        del At, bt
        many = many_column_figures(api, torch, args, flush, hbm_peak, tensor_peak, peak_kind)
    clk = clocks.stop()

    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        v, desc, _ = oracle_sample(A, b, args.cpu_budget)
        cpu = {"value": round(v, 1), "unit": "ms", "cores": 1, "kind": "oracle", "sample": desc}
    base_ms = PAGES_H200_MS.get(args.workload)
    line = {
        "metric": metric_for(args.workload),
        "value": round(ms, 4), "unit": "ms", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": round(ms / base_ms, 6) if base_ms else None,
        "dtype": "int8", "data": "synthetic",
        "config": {"workload": args.workload, "n": n, "c": c,
                   "entries": inputs.WORKLOADS[args.workload].description,
                   "seed": args.seed, "m": s0.m, "primes_used": s0.primes_used,
                   "l2": "flushed between timed steps (256 MiB write)",
                   "parallelism": "replicas" if world > 1 else "single"},
        "phases_ms": phases,
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": int(sum(s.launches for s in sols)),
        "clocks": clk,
        "step_ms": [round(x, 3) for x in step_ms],
    }
    if many is not None:
        line["configs"] = {many["workload"]: many}
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def main():
    args = parse()
    rank, local_rank, world = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
    elif args.lift_only:
        run_lift_only(args)
    else:
        run_gb300(args, rank, local_rank, world)


if __name__ == "__main__":
    main()
