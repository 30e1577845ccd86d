#!/usr/bin/env python
"""Benchmark of the Laplacian-Nystrom attention forward on GB300.

One step = one full forward (pooling, Newton-Schulz, fused L1-distance + exp for the query and
key blocks, whitening statistics, B V, X (B V), output) over one batch of the synthetic
workload, inputs resident in HBM.  Default workload: the stage-1 vision shape (B=8, H=2,
56x56 tokens, d=32, m=49, T=20, fp32, heavy-tailed Q/K), the shape the L1-distance roofline is
quoted on.

Prints one JSON line (rank 0).  Multi-GPU (torchrun): every rank runs its own copy of the
workload (independent (batch, head) slices, no data-path collective): weak scaling.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]
                  [--kernel laplacian|gaussian] [--solver newton_schulz|cg] [--backward]

--kernel gaussian runs the same pipeline with the Gaussian kernel exp(-|x - y|_2^2 / lambda)
in place of the Laplacian one (the softmax-free baseline the method is set against).
--solver cg replaces the Newton-Schulz inverse by T conjugate-gradient iterations on
W M = B V (the solver the method is compared with).
--backward times a training step instead: lapl_attn_forward_train followed by
lapl_attn_backward for a fixed synthetic dLoss/dO (its own metric line; the forward line
above is the headline).
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from lapl_workloads import WORKLOADS, make_inputs  # noqa: E402

METRIC = "Laplacian-Nyström attn fwd tokens/s on 1 GB300; L1-cdist % of FP32 ALU peak"
UNIT = "tokens/s"
L2_BYTES = 129 * 1024 * 1024
FLUSH_BYTES = 512 * 1024 * 1024
CLEAN_BYTES = 256 * 1024 * 1024

# DRAM traffic (read + write bytes) of one launch of the distance kernel, from an ncu capture
# (summaries under profiles/), per (feed, workload, kernel) with the sha256 of the distance kernel's
# source files it was taken on; reported as null when the sources have changed since.
CDIST_TRAFFIC = {
    ("l1", "stage1_f32", "laplacian"): (
        13019136 + 7936, "d1b8b4f63f047ce56f71705050c3178df9733c6e113d90c488903e658c38bf8f"),
    ("gtc", "stage1_f32", "gaussian"): (
        12994816 + 0, "d1b8b4f63f047ce56f71705050c3178df9733c6e113d90c488903e658c38bf8f"),
}
CDIST_SOURCES = ["cdist_kernel.cuh", "cdist_tma.cuh", "cdist_l1.cuh", "cdist.cu", "cdist_d32.cu",
                 "cdist_d64.cu", "cdist_d0.cu", "cdist_tma_f32.cu", "cdist_tma_bf16.cu",
                 "cdist_l1.cu", "cdist_l1_bf16.cu", "cdist_gauss_d32.cu", "cdist_gauss_d64.cu",
                 "cdist_gauss_d0.cu",
                 "cdist_gauss_tc.cu", "common.cuh"]
CDIST_KERNEL = {
    ("l1", "laplacian"): "cdist_l1_kernel (fused L1 distance + exp, query and key blocks; "
                         "TMA-fed, helper warp, element terms split between the FP32 and ALU "
                         "pipes)",
    ("tma", "laplacian"): "cdist_tma_kernel (fused L1 distance + exp, query and key blocks; "
                          "TMA-fed)",
    ("cp.async", "laplacian"): "cdist_exp_kernel (fused L1 distance + exp, query and key "
                               "blocks; cp.async-fed)",
    ("cp.async", "gaussian"): "cdist_exp_kernel (fused squared-l2 distance + exp, query and key "
                              "blocks; cp.async-fed)",
    ("gtc", "gaussian"): "gauss_tc_kernel (squared-l2 distance as |x|^2 + |l|^2 - 2 x.l with x.l "
                         "on the tensor cores (tcgen05, TF32 high/low) + exp, query and key "
                         "blocks)",
}
OPS_CONVENTION = {
    "laplacian": "3 per (token, landmark, channel): subtract, absolute value, add",
    "gaussian": "3 per (token, landmark, channel): subtract, multiply, add (a subtract and an "
                "FMA)",
}
KERNEL_IDS = {"laplacian": 0, "gaussian": 1}
SOLVER_IDS = {"newton_schulz": 0, "cg": 1}


def cdist_sources_sha() -> str:
    hs = hashlib.sha256()
    for f in CDIST_SOURCES:
        hs.update(open(os.path.join(ROOT, "laplacian_nystr_attention_gb300", "csrc", f), "rb").read())
    return hs.hexdigest()


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="stage1_f32", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--kernel", default="laplacian", choices=sorted(KERNEL_IDS))
    ap.add_argument("--solver", default="newton_schulz", choices=sorted(SOLVER_IDS))
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="budget of the oracle CPU-baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--backward", action="store_true",
                    help="time forward (keeping the backward's state) + backward instead")
    ap.add_argument("--inner-loop", action="store_true",
                    help="build and run bench_l1_loop.cu: elements/clock/SM of the L1-distance "
                         "inner loop in its instruction forms (no forward)")
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def workload_desc(w, kernel: str, solver: str = "newton_schulz") -> dict:
    return {
        "workload": (f"{w.name}: B={w.batch} H={w.heads} grid {w.grid_h}x{w.grid_w} "
                     f"(N={w.n}) d={w.head_dim} m={w.num_landmarks} T={w.ns_steps} "
                     f"lambda={w.lam:g} eps={w.eps:g} delta={w.delta:g} {w.dtype} {w.dist}"
                     + ("" if kernel == "laplacian" else f"; {kernel} kernel")
                     + ("" if solver == "newton_schulz" else f"; {solver} solver")),
        "batch": w.batch, "heads": w.heads, "seq_len": w.n, "head_dim": w.head_dim,
        "landmarks": w.num_landmarks, "ns_steps": w.ns_steps, "kernel": kernel,
        "solver": solver,
    }


def oracle_cfg(w, kernel: str, solver: str = "newton_schulz") -> dict:
    cfg = w.config()
    cfg["kernel"] = KERNEL_IDS[kernel]
    cfg["solver"] = SOLVER_IDS[solver]
    return cfg


def cdist_ops_per_launch(w) -> float:
    """Algorithmic FP32 operations of the distance kernel: 3 (subtract, absolute value, add; or
    for the Gaussian kernel subtract, multiply, add) per (token, landmark, channel) element, for
    the query block and the key block."""
    return 3.0 * 2.0 * w.batch * w.heads * w.n * w.num_landmarks * w.head_dim


def cdist_bytes_per_launch(w) -> int:
    """Algorithmic bytes of the distance kernel: Q and K read once, A^T and B^T (fp32) written
    once; the landmarks (m x d per head, L2-resident) are not counted."""
    esz = 2 if w.dtype == "bf16" else 4
    bh = w.batch * w.heads
    return 2 * bh * w.n * w.head_dim * esz + 2 * bh * w.n * w.num_landmarks * 4


def fp32_peak_tflops(num_sms: int, sm_mhz: float) -> float:
    """FP32 CUDA-core peak: SMs x 128 FP32 lanes x 2 (an FMA counts 2) x SM clock."""
    return num_sms * 128 * 2 * sm_mhz * 1e6 / 1e12


def gemm_chain_roofline(w, stage_ms: dict, peaks: dict, plan: dict) -> list:
    """The two contractions of the output chain against the measured HBM bandwidth: algorithmic
    bytes per launch / the stage's in-step CUDA-event time.  B V's stage also holds the column
    statistics of A (they read A^T once); the output stage reads A^T and writes O."""
    bh, n, m, d = w.batch * w.heads, w.n, w.num_landmarks, w.head_dim
    esz = 2 if w.dtype == "bf16" else 4
    hbm = float(peaks.get("hbm_gbs", 6800.0))
    bv_bytes = bh * m * n * 4 + bh * n * d * esz + bh * m * n * 4
    out_bytes = bh * m * n * 4 + bh * n * d * 4
    flops = 2.0 * bh * n * m * d
    tc = bool(plan.get("bv_tensor_core"))
    out_tc = bool(plan.get("out_tensor_core"))
    entries = []
    for name, key, nbytes, kern in (
            ("B V + column statistics", "bv", bv_bytes,
             "col_stats_kernel + bv_tc_kernel (tcgen05, TF32 high/low)" if tc
             else "bv_kernel (statistics CTAs + CUDA-core FMA tiles)"),
            ("O = A^ M (whitening applied on load)", "output", out_bytes,
             "out_tc_kernel (tcgen05, TF32 high/low)" if out_tc
             else "output_kernel (CUDA-core FMA tiles)")):
        ms = stage_ms[key]
        gbs = nbytes / (ms / 1e3) / 1e9
        entries.append({"stage": name, "kernel": kern, "bound": "hbm", "achieved": gbs,
                        "peak": hbm, "unit": "GB/s", "frac": gbs / hbm, "bytes": nbytes,
                        "flops": flops, "tflops": flops / (ms / 1e3) / 1e12, "kernel_ms": ms,
                        "peak_source": "MEASURED_PEAKS.json hbm_gbs (of measured)"})
    return entries


def dominant_kernel_entry(w, stage_ms: dict, peaks: dict, plan: dict, ms: float):
    """The Newton-Schulz solve, the stage-1 step's largest kernel (a launch-list share of about
    47 %): a chain of 2T dependent products, bound by latency.  Its tensor-core work (the TF32
    high/low split as one 128 x 128 x 8 MMA per K step, ceil(m/8) steps per product, 2T
    products per head) against the TF32 peak (the measured bf16 peak / 2), and its time per
    step."""
    if not plan.get("ns_tensor_core"):
        return None
    bh, m, T = w.batch * w.heads, w.num_landmarks, w.ns_steps
    ksteps = (((m + 3) // 4 * 4) + 7) // 8
    flops = 2.0 * bh * 2 * T * ksteps * 128 * 128 * 8
    t = stage_ms["newton_schulz"] / 1e3
    peak = float(peaks.get("bf16_tflops", 1900.0)) / 2.0
    ach = flops / t / 1e12
    return {"kernel": "ns_tc_kernel (W, T Newton-Schulz steps; tcgen05 TF32 high/low)",
            "bound": "latency", "achieved": ach, "peak": peak, "unit": "TFLOP/s",
            "frac": ach / peak, "kernel_ms": stage_ms["newton_schulz"],
            "stage_us_per_step": stage_ms["newton_schulz"] * 1e3 / max(T, 1),
            "share_of_forward": stage_ms["newton_schulz"] / ms,
            "note": "2T dependent products per head; the step waits on MMA issue (about 60 "
                    "cycles per instruction), tensor-memory reads and CTA barriers, not on a "
                    "pipe's throughput; peak = TF32 = measured bf16 / 2"}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "sm_max_mhz": 2070.0}, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle sampling in the background during a timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        time.sleep(0.2)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        rows = []
        if self.path and os.path.exists(self.path):
            for line in open(self.path):
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "samples": len(rows),
                "reasons": reasons}


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def oracle_rate(w, q, k, v, budget_s: float, threads: int, kernel: str = "laplacian",
                solver: str = "newton_schulz"):
    """Whole (b,h) slices of the fp64 oracle, `threads` at a time (the oracle's C call releases
    the GIL), cycling over the workload's slices until the budget is spent (at least one wave).
    Returns (tokens/s, slices done, seconds)."""
    import concurrent.futures as cf
    import oracle
    oracle.build()
    cfg = oracle_cfg(w, kernel, solver)
    q64, k64, v64 = (np.ascontiguousarray(x, dtype=np.float64) for x in (q, k, v))
    slices = w.batch * w.heads
    done, t0 = 0, time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        while done == 0 or time.perf_counter() - t0 < budget_s:
            wave = threads
            list(ex.map(lambda j: oracle.forward(cfg, q64, k64, v64, slices=(j % slices, 1)),
                        range(done, done + wave)))
            done += wave
    dt = time.perf_counter() - t0
    return done * w.n / w.heads / dt, done, dt      # tokens are counted once across heads


def cpu_baseline(w, q, k, v, budget_s: float, kernel: str = "laplacian",
                 solver: str = "newton_schulz") -> dict:
    """The fp64 oracle on a bounded sample: whole (b,h) slices on all host cores until the
    budget is spent, and the same on one core for reference."""
    cores = host_cores()
    one, n1, t1 = oracle_rate(w, q, k, v, budget_s / 4, 1, kernel, solver)
    allc, na, ta = oracle_rate(w, q, k, v, budget_s, cores, kernel, solver)
    return {"value": allc, "unit": UNIT, "cores": cores, "kind": "oracle",
            "value_1_core": one,
            "sample": f"{na} slices ({na / (w.batch * w.heads):.1f} passes over the "
                      f"{w.batch * w.heads} (batch, head) slices of {w.name}) in "
                      f"{ta:.2f} s on {cores} threads (one slice per thread), and {n1} slices in "
                      f"{t1:.2f} s on 1 thread; fp64 C oracle; tokens/s = slices * N / H / "
                      "seconds"}


def max_over_ranks(value: float, world: int, device) -> float:
    """The largest of every rank's `value` (the job's time is its slowest rank's); the value
    itself on one rank.  Works on any process-group backend (NCCL with a CUDA device, gloo on
    the CPU)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as tdist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world: int, tokens_per_rank: int, ms: float) -> float:
    """Whole-job tokens/s: every rank processes its own copy of the workload (independent
    (batch, head) slices), in the max-over-ranks time `ms`."""
    return world * tokens_per_rank / (ms / 1e3)


def run_reference(args, w):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import concurrent.futures as cf
    q, k, v = make_inputs(w)
    import oracle
    oracle.build()
    cfg = oracle_cfg(w, args.kernel, args.solver)
    q64, k64, v64 = (np.ascontiguousarray(x, dtype=np.float64) for x in (q, k, v))
    slices = w.batch * w.heads
    cores = host_cores()
    per_step = max(1, min(slices, cores))
    times = []
    with cf.ThreadPoolExecutor(max_workers=cores) as ex:
        for step in range(args.warmup + args.steps):
            s0 = (step * per_step) % slices
            cnt = min(per_step, slices - s0)
            t0 = time.perf_counter()
            list(ex.map(lambda s: oracle.forward(cfg, q64, k64, v64, slices=(s, 1)),
                        range(s0, s0 + cnt)))
            dt = time.perf_counter() - t0
            if step >= args.warmup:
                times.append((dt, cnt))
    tot_t = sum(t for t, _ in times)
    tot_tok = sum(c for _, c in times) * w.n / w.heads
    value = tot_tok / tot_t
    sample = (f"{per_step} (batch, head) slice(s) of {w.name} per step, one per thread on "
              f"{cores} threads, fp64 C oracle; tokens/s = slices * N / H / seconds")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tot_t / len(times), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_desc(w, args.kernel, args.solver),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, w):
    import torch
    import torch.distributed as tdist

    world, rank, local = dist_env()
    if world > 1:
        tdist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    if not os.path.exists(os.path.join(ROOT, "laplacian_nystr_attention_gb300",
                                       "liblapl_attn.so")):
        import __graft_entry__
        __graft_entry__.build()
    import laplacian_nystr_attention_gb300 as lna
    from laplacian_nystr_attention_gb300 import _lib

    q, k, v = make_inputs(w)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    hq, hk, hv = (torch.from_numpy(x).to(tdt).pin_memory() for x in (q, k, v))
    dq, dk, dv = (x.to(dev) for x in (hq, hk, hv))
    cfg = lna.make_config(**{**w.config(), "in_dtype": w.dtype, "kernel": args.kernel,
                             "solver": args.solver})
    att = lna.LaplacianNystromAttention(cfg)
    out = torch.empty((w.batch, w.heads, w.n, w.head_dim), dtype=torch.float32, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    clean = torch.ones(CLEAN_BYTES // 4, dtype=torch.float32, device=dev)

    def flush_l2():
        # Write a buffer larger than L2 (evicts every input and intermediate), then read another
        # one, so that the written lines are back in memory before the timed forward starts
        # rather than written back during its first kernel.
        flush.zero_()
        clean.sum()

    stream = torch.cuda.current_stream()

    def step():
        att.forward(dq, dk, dv, out=out)

    def barrier():
        if world > 1:
            tdist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        flush_l2()
        step()
    barrier()

    # ---- timed region: K forwards, L2 flushed before each (flush not timed) ----
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(local) as clocks:
        barrier()
        for i in range(args.steps):
            flush_l2()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        barrier()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = max_over_ranks(sum(step_ms) / len(step_ms), world, dev)
    kernels = lna.lapl_attn_kernels_per_forward(att.handle)
    gpu_launches = kernels * args.steps

    # ---- stage times of the same forward, recorded with CUDA events on its streams ----
    lna.lapl_attn_set_timing(att.handle, True)
    stage = {s: [] for s in _lib.STAGES}
    for i in range(args.steps):
        flush_l2()
        step()
        for key, val in lna.lapl_attn_stage_times(att.handle).items():
            stage[key].append(val)
    lna.lapl_attn_set_timing(att.handle, False)
    stage_ms = {key: sum(vals) / len(vals) for key, vals in stage.items()}

    # ---- the same forward captured once in a CUDA graph and replayed ----
    graph = None
    if not args.no_graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        torch.cuda.synchronize()
        for _ in range(args.warmup):
            flush_l2()
            g.replay()
        barrier()
        g0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        g1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        for i in range(args.steps):
            flush_l2()
            g0[i].record(stream)
            g.replay()
            g1[i].record(stream)
        barrier()
        gms = max_over_ranks(sum(a.elapsed_time(b) for a, b in zip(g0, g1)) / args.steps,
                             world, dev)
        graph = {"value": job_rate(world, w.tokens, gms), "unit": UNIT, "ms_per_step": gms,
                 "note": "lapl_attn_forward captured in one CUDA graph (both streams), "
                         "replayed; L2 flushed before each replay"}
        del g

    # ---- end to end through the C ABI with host buffers (pinned) ----
    e2e = None
    if not args.no_e2e:
        h = lna.lapl_attn_create(cfg)
        nbytes = lna.lapl_attn_host_staging_size(h)
        staging = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        hout = torch.empty(out.shape, dtype=torch.float32).pin_memory()
        args_h = (h, hq.data_ptr(), hk.data_ptr(), hv.data_ptr(), None, hout.data_ptr(),
                  staging.data_ptr(), nbytes, stream.cuda_stream)
        for _ in range(args.warmup):
            lna.lapl_attn_forward_host(*args_h)
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            lna.lapl_attn_forward_host(*args_h)
        e1.record(stream)
        barrier()
        e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, dev)
        in_b = hq.numel() * hq.element_size()
        e2e = {"value": job_rate(world, w.tokens, e2e_ms), "unit": UNIT,
               "h2d_bytes_per_step": 3 * in_b,
               "d2h_bytes_per_step": hout.numel() * hout.element_size(),
               "ms_per_step": e2e_ms}
        lna.lapl_attn_destroy(h)

    # No bounded device-side wait may have given up during any of the forwards above.
    flags = lna.lapl_attn_device_errors(att.handle, stream.cuda_stream)
    assert flags == 0, flags

    if rank != 0:
        if world > 1:
            tdist.destroy_process_group()
        return

    peaks, peaks_src = measured_peaks()
    props = torch.cuda.get_device_properties(dev)
    sm_max = float(peaks.get("sm_max_mhz", 2070.0))
    peak = fp32_peak_tflops(props.multi_processor_count, sm_max)
    achieved = cdist_ops_per_launch(w) / (stage_ms["cdist"] / 1e3) / 1e12
    plan = lna.lapl_attn_plan_info_get(att.handle)
    feed = {3: "gtc", 2: "l1", 1: "tma"}.get(plan["cdist_tma"], "cp.async")
    rec = CDIST_TRAFFIC.get((feed, w.name, args.kernel))
    traffic = rec[0] if rec and rec[1] == cdist_sources_sha() else None
    if feed == "gtc":
        # The cross term is a contraction on the tensor cores; what is left is bound by HBM.
        hbm = float(peaks.get("hbm_gbs", 6800.0))
        nbytes = cdist_bytes_per_launch(w)
        gbs = nbytes / (stage_ms["cdist"] / 1e3) / 1e9
        roofline = {
            "kernel": CDIST_KERNEL[(feed, args.kernel)],
            "bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
            "traffic": traffic,
            "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({peaks_src})",
            "bytes_per_launch": nbytes,
            "bytes_convention": "Q and K read once, A^T and B^T written once (fp32)",
            "kernel_ms": stage_ms["cdist"],
        }
    else:
        roofline = {
            "kernel": CDIST_KERNEL[(feed, args.kernel)],
            "bound": "alu", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak, "traffic": traffic,
            "peak_source": (f"derived: {props.multi_processor_count} SMs x 128 FP32 lanes x 2 x "
                            f"{sm_max:g} MHz (max SM clock, MEASURED_PEAKS {peaks_src})"),
            "ops_per_launch": cdist_ops_per_launch(w),
            "ops_convention": OPS_CONVENTION[args.kernel],
            "kernel_ms": stage_ms["cdist"],
        }
    clk = clocks.summary()
    line = {
        "metric": METRIC, "value": job_rate(world, w.tokens, ms), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic",
        "config": {**workload_desc(w, args.kernel, args.solver),
                   "l2": f"flushed before every timed step ({FLUSH_BYTES >> 20} MiB write, "
                         f"then a {CLEAN_BYTES >> 20} MiB read; not timed)",
                   "parallelism": f"replicas x{world} (independent (batch, head) slices)",
                   "plan": plan},
        "roofline": roofline,
        "gemm_chain_roofline": gemm_chain_roofline(w, stage_ms, peaks, plan),
        "dominant_kernel": dominant_kernel_entry(w, stage_ms, peaks, plan, ms),
        "stage_ms": stage_ms,
        "cpu_baseline": None,
        "e2e": e2e,
        "graph": graph,
        "memory": {"workspace_bytes": att.workspace_bytes,
                   "io_bytes": sum(x.numel() * x.element_size() for x in (dq, dk, dv, out)),
                   "note": "device memory of one forward: Q, K, V, O and the workspace"},
        "gpu_launches": gpu_launches,
        "clocks": clk,
        "impl": "ours",
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, q, k, v, args.cpu_seconds, args.kernel,
                                            args.solver)
    print(json.dumps(line), flush=True)
    att.close()
    if world > 1:
        tdist.destroy_process_group()


METRIC_BWD = "Laplacian-Nyström attn fwd+bwd tokens/s on 1 GB300"


def run_backward(args, w):
    """Training step: forward keeping the backward's state, then the backward for a fixed
    synthetic dLoss/dO; L2 flushed before every step; CUDA events on the launching stream."""
    import torch
    import torch.distributed as tdist

    world, rank, local = dist_env()
    if world > 1:
        tdist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if not os.path.exists(os.path.join(ROOT, "laplacian_nystr_attention_gb300",
                                       "liblapl_attn.so")):
        import __graft_entry__
        __graft_entry__.build()
    import laplacian_nystr_attention_gb300 as lna

    q, k, v = make_inputs(w)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    dq_, dk_, dv_ = (torch.from_numpy(x).to(tdt).to(dev) for x in (q, k, v))
    gen = torch.Generator(device=dev).manual_seed(21)
    G = torch.randn(dq_.shape, generator=gen, device=dev, dtype=torch.float32)
    cfg = lna.make_config(**{**w.config(), "in_dtype": w.dtype, "kernel": args.kernel})
    att = lna.LaplacianNystromAttention(cfg)
    out = torch.empty(dq_.shape, dtype=torch.float32, device=dev)
    grads = None
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    clean = torch.ones(CLEAN_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def flush_l2():
        flush.zero_()
        clean.sum()

    def barrier():
        if world > 1:
            tdist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        flush_l2()
        att.forward(dq_, dk_, dv_, out=out, keep_for_backward=True)
        gq, gk, gv, gb = att.backward(dq_, dk_, dv_, G, grads=grads)
        grads = dict(dq=gq, dk=gk, dv=gv, dbias=gb)
    barrier()
    e = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    with ClockSampler(local) as clocks:
        barrier()
        for i in range(args.steps):
            flush_l2()
            e[i][0].record(stream)
            att.forward(dq_, dk_, dv_, out=out, keep_for_backward=True)
            e[i][1].record(stream)
            att.backward(dq_, dk_, dv_, G, grads=grads)
            e[i][2].record(stream)
        barrier()
    fwd = sum(a.elapsed_time(b) for a, b, _ in e) / args.steps
    bwd = sum(b.elapsed_time(c) for _, b, c in e) / args.steps
    ms = max_over_ranks(fwd + bwd, world, dev)
    launches = (lna.lapl_attn_kernels_per_forward(att.handle) +
                lna.lapl_attn_backward_kernels(att.handle)) * args.steps
    flags = lna.lapl_attn_device_errors(att.handle, stream.cuda_stream)
    assert flags == 0, flags
    if rank == 0:
        line = {
            "metric": METRIC_BWD, "value": job_rate(world, w.tokens, ms), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.dtype, "data": "synthetic",
            "config": {**workload_desc(w, args.kernel),
                       "l2": f"flushed before every timed step ({FLUSH_BYTES >> 20} MiB write, "
                             f"then a {CLEAN_BYTES >> 20} MiB read; not timed)",
                       "parallelism": f"replicas x{world} (independent (batch, head) slices)",
                       "step": "lapl_attn_forward_train + lapl_attn_backward (dq, dk, dv, "
                               "dbias for a fixed synthetic dLoss/dO)"},
            "forward_ms": fwd, "backward_ms": bwd,
            "memory": {"workspace_bytes": att.workspace_bytes,
                       "backward_workspace_bytes": att.bwd_workspace_bytes},
            "gpu_launches": launches, "clocks": clocks.summary(), "impl": "ours",
        }
        print(json.dumps(line), flush=True)
    att.close()
    if world > 1:
        tdist.destroy_process_group()


def run_inner_loop(args):
    """The L1-distance inner-loop microbenchmark (bench_l1_loop.cu), one JSON line: per form and
    CTAs per SM, elements / clock / SM (mean over SMs), and the 3-op fraction of FP32 peak."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    build = os.path.join(ROOT, "_build")
    os.makedirs(build, exist_ok=True)
    exe = os.path.join(build, "bench_l1_loop")
    src = os.path.join(ROOT, "bench_l1_loop.cu")
    if not os.path.exists(exe) or os.path.getmtime(exe) < os.path.getmtime(src):
        subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-o", exe,
                        src], check=True)
    outp = subprocess.run([exe], check=True, capture_output=True, text=True).stdout
    forms = []
    for line in outp.splitlines():
        parts = line.split()
        if len(parts) < 5 or "=" not in parts[1]:
            continue
        kv = dict(tok.split("=") for tok in parts[1:] if tok.count("=") == 1)
        mean = float(kv["mean"])
        forms.append({"form": parts[0], "landmarks_per_warp": int(kv["C"]),
                      "ctas_per_sm": int(kv["ctas_per_sm"]), "registers": int(kv["regs"]),
                      "elem_per_clk_per_sm": mean, "min_over_sms": float(kv["min"]),
                      "max_over_sms": float(kv["max"]),
                      "frac_of_fp32_peak_3op": 3.0 * mean / 256.0})
    print(json.dumps({"metric": "L1-distance inner loop elements/clock/SM", "unit": "elem/clk/SM",
                      "forms": forms, "note": "3-op fraction = 3 x elements / (128 lanes x 2)"}),
          flush=True)


def main():
    args = parse()
    w = WORKLOADS[args.workload]
    if args.inner_loop:
        run_inner_loop(args)
        return
    if args.impl == "reference":
        run_reference(args, w)
    elif args.backward:
        run_backward(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
