"""Benchmark of the Mamba-2 SSD chunked-scan forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
                    [--path auto|tc|chain|simt] [--step | --conv | --norm]

One step = one full forward (all five stages) over one batch of the
workload's synthetic inputs, already resident in HBM. Prints one JSON line
(rank 0). Under torchrun every rank runs the whole workload on its own GPU
(independent replicas: the path has no exchange step), so scaling is weak.

The roofline's achieved figure divides the algorithmic bytes by the main
kernel's own mean launch time, which the library records with CUDA events
in a separate pass (ssd_kernel_timing); path_achieved divides by the whole
call. e2e goes through ssd_fwd_host with pinned host buffers. --step,
--conv and --norm time the decode step, the conv1d + SiLU and the gated
RMSNorm instead.

--impl reference times the fp64 CPU oracle (the only reference arm: the
pages ship no runnable implementation) on the host cores, on a bounded
sample of the same workload.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mamba_ssd_chunked_gb300.inputs import HEADLINE, WORKLOADS, Workload, make_inputs  # noqa: E402

METRIC = "SSD fwd tokens/s and % of roofline (Mamba2-2.7B layer shape), 1 GB300"
UNIT = "tokens/s"
FLUSH_BYTES = 256 << 20  # > 129 MB L2
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# the source file of each fused kernel: a committed ncu summary's DRAM traffic is
# reported only while the kernel source it was taken on is unchanged
KERNEL_SOURCES = {"tc": ["mamba_ssd_chunked_gb300/csrc/ssd_tc.cu"],
                  "chain": ["mamba_ssd_chunked_gb300/csrc/ssd_chain.cu"],
                  "step": ["mamba_ssd_chunked_gb300/csrc/ssd_step.cu"],
                  "conv": ["mamba_ssd_chunked_gb300/csrc/ssd_layer.cu"],
                  "norm": ["mamba_ssd_chunked_gb300/csrc/ssd_layer.cu"]}
PROFILE_NAMES = {"tc": "ssd_tc_fused", "chain": "ssd_chain_fused", "step": "ssd_step_rows4",
                 "conv": "conv1d_fwd", "norm": "gated_rmsnorm"}


# ----------------------------------------------------------------------------- roofline arithmetic
def algorithmic_bytes(w: Workload) -> int:
    """Bytes the forward must move through HBM at least: x and y, B and C, dt,
    the per-head parameters, the initial state (when given) and the final
    state. Chunk states and C.B^T are intermediates and are not counted."""
    eb = 4 if w.io_dtype == "f32" else 2
    x = w.batch * w.seqlen * w.nheads * w.headdim * eb
    bc = w.batch * w.seqlen * w.ngroups * w.dstate * eb
    dt = w.batch * w.seqlen * w.nheads * 4
    state = w.batch * w.nheads * w.headdim * w.dstate * 4
    init = state if w.init != "zero" else 0
    return 2 * x + 2 * bc + dt + init + state + 3 * w.nheads * 4


def algorithmic_flops(w: Workload) -> int:
    """Causal (lower-triangular) work of the chunked method at chunk_len Q:
    per token and head 4pn (state in and out) + Qp (causal half of the
    intra-chunk product), plus Q^2 n per (batch, chunk, group) for C.B^T."""
    Q = w.chunk_len
    nchunks = -(-w.seqlen // Q)
    per_token_head = 4 * w.headdim * w.dstate + Q * w.headdim
    return w.batch * w.seqlen * w.nheads * per_token_head + w.batch * nchunks * w.ngroups * Q * Q * w.dstate


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash(path: str = "tc") -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[path]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, kpath: str = "tc"):
    """DRAM bytes per launch of the fused kernel from the committed ncu
    summary, if it was taken on the current kernel source; else None."""
    if kpath not in PROFILE_NAMES:
        return None
    path = os.path.join(ROOT, "profiles", f"{PROFILE_NAMES[kpath]}_{workload}.md")
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if line.startswith("traffic_bytes_per_launch:") or line.startswith("kernel_source_hash:"):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    if vals.get("kernel_source_hash") != kernel_source_hash(kpath):
        return None
    try:
        return int(vals["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def aggregate(step_seconds_per_rank, tokens_per_step, world):
    """Weak-scaling aggregate: every rank processes tokens_per_step per step;
    the job's time per step is the slowest rank's."""
    t = max(step_seconds_per_rank)
    return world * tokens_per_step / t, t


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """Samples nvidia-smi SM clocks and throttle reasons in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.rows = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.rows.append((time.time(), parts))

    def mark(self):
        return time.time()

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        rows = [r for (ts, r) in self.rows if t0 - 0.15 <= ts <= t1 + 0.15]
        window = "timed region"
        if not rows:
            rows = [r for (_, r) in self.rows]
            window = "whole run (timed region shorter than the sampling period)"
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        smmax = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smmax) if smmax else None,
                "reasons": reasons, "samples": len(rows), "window": window,
                "power_w_max": max((num(r[3]) or 0.0) for r in rows)}


# ----------------------------------------------------------------------------- distributed
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        if backend == "nccl":
            import torch
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
        pg = dist
    return world, rank, local, pg


def barrier(pg):
    if pg is not None:
        pg.barrier()


def max_over_ranks(pg, value: float, device=None) -> float:
    if pg is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- CPU oracle timing
def time_oracle(w: Workload, inp, budget_s: float, nthreads: int):
    """Times the fp64 oracle on whole (b, h) chains, batch after batch of
    `nthreads` chains, until `budget_s` has elapsed or every chain ran.
    Returns (layer tokens/s equivalent, chains run, seconds)."""
    import oracle
    chains = [(b, h) for b in range(w.batch) for h in range(w.nheads)]
    rng = np.random.Generator(np.random.PCG64(7))
    rng.shuffle(chains)
    done, elapsed = 0, 0.0
    while done < len(chains) and elapsed < budget_s:
        batch = chains[done:done + nthreads]
        t0 = time.perf_counter()
        oracle.recurrence(inp["x"], inp["dt"], inp["dt_bias"], inp["A"], inp["B"], inp["C"], inp["D"],
                          inp["init_state"], chains=batch, nthreads=nthreads, want_y=True)
        elapsed += time.perf_counter() - t0
        done += len(batch)
    # a layer token carries nheads chain-steps
    return done * w.seqlen / w.nheads / elapsed, done, elapsed


# ----------------------------------------------------------------------------- arms
def run_reference(args, w: Workload, world, rank):
    if rank != 0:
        return None
    inp = make_inputs(w.batch, w.seqlen, w.nheads, w.headdim, w.ngroups, w.dstate, io_dtype=w.io_dtype,
                      init=w.init, seed=w.seed)
    cores = os.cpu_count() or 1
    per_step_budget = max(1.0, min(20.0, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        time_oracle(w, inp, 1e-9, cores)  # one batch of chains
    vals, chains_total, secs_total = [], 0, 0.0
    for _ in range(args.steps):
        v, n, s = time_oracle(w, inp, per_step_budget, cores)
        vals.append(v)
        chains_total += n
        secs_total += s
    value = chains_total * w.seqlen / w.nheads / secs_total
    sample = (f"{chains_total} whole (batch, head) chains of {w.seqlen} tokens over {args.steps} steps "
              f"(~{per_step_budget:.0f} s each) out of {w.batch * w.nheads} chains; "
              f"value = chains x seqlen / nheads / seconds")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * w.batch * w.seqlen / value,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; shapes and distributions of the workload)",
        "config": config_dict(w),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def config_dict(w: Workload):
    return {"workload": w.name, "batch": w.batch, "seqlen": w.seqlen, "nheads": w.nheads, "headdim": w.headdim,
            "ngroups": w.ngroups, "dstate": w.dstate, "chunk_len": w.chunk_len, "io_dtype": w.io_dtype,
            "init_state": w.init, "parallelism": "replicas",
            "l2": "flushed between timed steps (256 MiB write); inputs also exceed L2"}


KERNEL_NAMES = {"tc": "ssd_tc_fused", "chain": "ssd_chain_fused", "simt": "simt (3 kernels)"}


def run_ours(args, w: Workload, world, rank, local, pg):
    import torch

    import mamba_ssd_chunked_gb300 as pkg
    from mamba_ssd_chunked_gb300 import build as pkg_build

    if not os.path.exists(pkg.LIBRARY):
        pkg_build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    inp = make_inputs(w.batch, w.seqlen, w.nheads, w.headdim, w.ngroups, w.dstate, io_dtype=w.io_dtype,
                      init=w.init, seed=w.seed)
    tdt = torch.bfloat16 if w.io_dtype == "bf16" else torch.float32
    host = {}
    for k, v in inp.items():
        if v is None:
            host[k] = None
            continue
        t = torch.from_numpy(v)
        if k in ("x", "B", "C"):
            t = t.to(tdt)
        host[k] = t.contiguous().pin_memory()
    d = {k: (None if v is None else v.to(dev, non_blocking=True)) for k, v in host.items()}
    y = torch.empty_like(d["x"])
    fs = torch.empty((w.batch, w.nheads, w.headdim, w.dstate), dtype=torch.float32, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    ws = None
    if args.path != "auto":
        need = pkg.ssd_fwd_workspace_bytes(w.batch, w.seqlen, w.nheads, w.headdim, w.ngroups, w.dstate, w.io_dtype,
                                           w.chunk_len, args.path)
        if need == 0 and args.path != "simt":
            raise RuntimeError(f"path {args.path} does not support workload {w.name}")
        ws = torch.zeros(max(need, 1), dtype=torch.uint8, device=dev)

    def step():
        if ws is None:
            pkg.ssd_fwd(d["x"], d["dt"], d["dt_bias"], d["A"], d["B"], d["C"], d["D"], d["init_state"],
                        chunk_len=w.chunk_len, y=y, final_state=fs, stream=stream.cuda_stream)
        else:
            pkg.ssd_fwd(d["x"], d["dt"], d["dt_bias"], d["A"], d["B"], d["C"], d["D"], d["init_state"],
                        chunk_len=w.chunk_len, y=y, final_state=fs, stream=stream.cuda_stream, path=args.path,
                        workspace=ws)

    visible = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    ids = [v.strip() for v in visible.split(",") if v.strip()]
    clocks = ClockSampler(ids[local] if local < len(ids) else str(local))
    clocks.start()
    time.sleep(0.3)
    for _ in range(max(3, args.warmup)):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    st = pkg.ssd_device_status(stream.cuda_stream)
    if st != 0:
        raise RuntimeError(f"device status {st} after warm-up")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(pg)
    torch.cuda.synchronize(dev)
    launches0 = pkg.ssd_kernel_launches()
    t_wall0 = clocks.mark()
    for i in range(args.steps):
        flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    barrier(pg)
    t_wall1 = clocks.mark()
    launches = pkg.ssd_kernel_launches() - launches0
    st = pkg.ssd_device_status(stream.cuda_stream)
    if st != 0:
        raise RuntimeError(f"device status {st} in the timed region")
    per_step = [s.elapsed_time(e) / 1e3 for s, e in zip(starts, ends)]
    mean_step = sum(per_step) / len(per_step)
    mean_step_max = max_over_ranks(pg, mean_step, dev)
    tokens = w.batch * w.seqlen
    value, _ = aggregate([mean_step_max], tokens, world)

    # the main kernel's own launch time, in a separate pass (the library records CUDA
    # events on the launching stream around it, which keeps it from overlapping the
    # kernels before it): the roofline's achieved figure
    n_kernel = max(3, min(args.steps, 50))
    pkg.ssd_kernel_timing(True)
    for _ in range(n_kernel):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    pkg.ssd_kernel_timing(False)
    k_ms, k_n = pkg.ssd_kernel_timing_read()
    kernel_s = max_over_ranks(pg, k_ms / max(k_n, 1) / 1e3, dev)

    # end to end through ssd_fwd_host: pinned host inputs in, y and final state out, every step
    e2e = None
    if not args.no_e2e:
        y_h = torch.empty_like(host["x"]).pin_memory()
        fs_h = torch.empty((w.batch, w.nheads, w.headdim, w.dstate), dtype=torch.float32).pin_memory()

        def e2e_step():
            pkg.ssd_fwd_host(host["x"], host["dt"], host["dt_bias"], host["A"], host["B"], host["C"], host["D"],
                             host["init_state"], chunk_len=w.chunk_len, y=y_h, final_state=fs_h,
                             stream=stream.cuda_stream)

        for _ in range(2):
            e2e_step()
        barrier(pg)
        n_e2e = max(3, min(args.steps, 20))
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            e2e_step()
        e2e_s = (time.perf_counter() - t0) / n_e2e
        e2e_s = max_over_ranks(pg, e2e_s, dev)
        h2d = sum(v.numel() * v.element_size() for v in host.values() if v is not None)
        d2h = y_h.numel() * y_h.element_size() + fs_h.numel() * fs_h.element_size()
        e2e = {"value": world * tokens / e2e_s, "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": n_e2e}

    clocks.stop()
    if rank != 0:
        return None

    peaks, peak_src = load_peaks()
    abytes = algorithmic_bytes(w)
    aflops = algorithmic_flops(w)
    t_bytes = abytes / (peaks["hbm_gbs"] * 1e9)
    t_flops = aflops / (peaks["bf16_tflops"] * 1e12)
    bound = "hbm" if t_bytes >= t_flops else "tensor"
    path = args.path if args.path != "auto" else pkg.ssd_select_path(
        w.batch, w.seqlen, w.nheads, w.headdim, w.ngroups, w.dstate, w.io_dtype, w.chunk_len)
    if bound == "hbm":
        achieved, peak, unit = abytes / kernel_s / 1e9, peaks["hbm_gbs"], "GB/s"
        path_achieved = abytes / mean_step / 1e9
    else:
        achieved, peak, unit = aflops / kernel_s / 1e12, peaks["bf16_tflops"], "TFLOP/s"
        path_achieved = aflops / mean_step / 1e12
    traffic = profiled_traffic(w.name, path) if w == WORKLOADS[w.name] else None

    cpu = None
    if not args.no_cpu_baseline:
        cores = os.cpu_count() or 1
        v, n, s = time_oracle(w, inp, args.cpu_budget, cores)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"{n} of {w.batch * w.nheads} whole (batch, head) chains of {w.seqlen} tokens in "
                         f"{s:.1f} s; value = chains x seqlen / nheads / seconds"}

    ck = clocks.summary(t_wall0, t_wall1)
    return {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": mean_step_max * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.io_dtype,
        "data": "synthetic (seeded; shapes and distributions of the workload)",
        "config": config_dict(w),
        "path": path,
        "tflops": aflops / mean_step / 1e12,
        "roofline_time_us": max(t_bytes, t_flops) * 1e6,
        "pct_of_roofline": 100.0 * max(t_bytes, t_flops) / mean_step,
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
                     "traffic": traffic, "peak_source": f"{peak_src} (burst)",
                     "algorithmic_bytes": abytes, "algorithmic_flops": aflops,
                     "kernel": KERNEL_NAMES[path], "kernel_us": kernel_s * 1e6, "kernel_launches": k_n,
                     "timing": "achieved: algorithmic bytes / the main kernel's mean launch time, CUDA events "
                               "recorded by the library on the launching stream right around it, in a separate pass "
                               f"of {n_kernel} calls; path_achieved / path_frac: the same bytes / the whole call "
                               "(all launches of the path), as timed in the steps",
                     "path_achieved": path_achieved, "path_frac": path_achieved / peak},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": ck,
        "step_ms": {"min": min(per_step) * 1e3, "median": statistics.median(per_step) * 1e3,
                    "max": max(per_step) * 1e3},
    }


# ----------------------------------------------------------------------------- decode step (--step)
STEP_WORKLOAD = {"name": "mamba2_2p7b_decode_b64", "batch": 64, "nheads": 80, "headdim": 64, "ngroups": 1,
                 "dstate": 128, "io_dtype": "bf16", "seed": 1240}


def step_algorithmic_bytes(sw) -> int:
    """HBM bytes one decode step must move: the fp32 state read and written,
    x and y, B and C, dt, and the per-head parameters."""
    b, h, p, g, n = sw["batch"], sw["nheads"], sw["headdim"], sw["ngroups"], sw["dstate"]
    e = 2 if sw["io_dtype"] == "bf16" else 4
    return 2 * b * h * p * n * 4 + 2 * b * h * p * e + 2 * b * g * n * e + b * h * 4 + 3 * h * 4


def _time_op(args, dev, stream, op):
    """Warm up, then time args.steps calls of op() on `stream` with CUDA events
    (L2 flushed before each call, clocks sampled during the timed region).
    Returns (seconds per call, library launches in the timed region, clocks)."""
    import torch

    import mamba_ssd_chunked_gb300 as pkg

    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    visible = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    ids = [v.strip() for v in visible.split(",") if v.strip()]
    clocks = ClockSampler(ids[0] if ids else "0")
    clocks.start()
    time.sleep(0.3)
    for _ in range(max(3, args.warmup)):
        flush.zero_()
        op()
    torch.cuda.synchronize(dev)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    launches0 = pkg.ssd_kernel_launches()
    t_wall0 = clocks.mark()
    for i in range(args.steps):
        flush.zero_()
        starts[i].record(stream)
        op()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = clocks.mark()
    launches = pkg.ssd_kernel_launches() - launches0
    time.sleep(0.3)
    clocks.stop()
    per = [s_.elapsed_time(e_) / 1e3 for s_, e_ in zip(starts, ends)]
    return per, launches, clocks.summary(t_wall0, t_wall1)


def _op_line(args, metric, units_per_call, unit, per, launches, ck, cfg, abytes, kpath, kernel, dtype):
    peaks, peak_src = load_peaks()
    mean = sum(per) / len(per)
    achieved = abytes / mean / 1e9
    return {
        "metric": metric, "value": units_per_call / mean, "unit": unit, "n_gpus": 1, "steps": args.steps,
        "warmup": max(3, args.warmup), "us_per_step": mean * 1e6, "higher_is_better": True, "dtype": dtype,
        "data": "synthetic", "config": cfg,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": profiled_traffic(cfg["workload"], kpath),
                     "algorithmic_bytes": abytes, "peak_source": f"{peak_src} (burst)", "kernel": kernel},
        "gpu_launches": launches, "clocks": ck,
        "step_us": {"min": min(per) * 1e6, "median": statistics.median(per) * 1e6, "max": max(per) * 1e6},
    }


def _load_pkg():
    import mamba_ssd_chunked_gb300 as pkg
    from mamba_ssd_chunked_gb300 import build as pkg_build

    if not os.path.exists(pkg.LIBRARY):
        pkg_build.build()
    return pkg


def run_step(args):
    """Time ssd_step (one decode token per sequence, state updated in place)."""
    import torch

    pkg = _load_pkg()
    sw = STEP_WORKLOAD
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    b, h, p, g, n = sw["batch"], sw["nheads"], sw["headdim"], sw["ngroups"], sw["dstate"]
    inp = make_inputs(b, 1, h, p, g, n, io_dtype=sw["io_dtype"], init="normal", seed=sw["seed"])
    tdt = torch.bfloat16 if sw["io_dtype"] == "bf16" else torch.float32
    d = {}
    for k, v in inp.items():
        if v is None:
            d[k] = None
            continue
        t = torch.from_numpy(v).to(dev)
        if k in ("x", "B", "C"):
            t = t.to(tdt)
        if k in ("x", "dt", "B", "C"):
            t = t[:, 0].contiguous()
        d[k] = t
    state = d["init_state"]
    y = torch.empty_like(d["x"])
    stream = torch.cuda.current_stream(dev)

    def op():
        pkg.ssd_step(d["x"], d["dt"], d["dt_bias"], d["A"], d["B"], d["C"], d["D"], state, y=y,
                     stream=stream.cuda_stream)

    per, launches, ck = _time_op(args, dev, stream, op)
    cfg = {"workload": sw["name"], "batch": b, "nheads": h, "headdim": p, "ngroups": g, "dstate": n,
           "l2": "flushed between timed steps (256 MiB write); the 168 MB state also exceeds L2"}
    return _op_line(args, "SSD decode step tokens/s (one token per sequence, Mamba2-2.7B layer heads), 1 GB300",
                    b, "tokens/s", per, launches, ck, cfg, step_algorithmic_bytes(sw), "step", "ssd_step_rows4",
                    sw["io_dtype"])


def conv_algorithmic_bytes(cw) -> int:
    """xBC read once and x/B/C written once (io dtype), plus the taps and bias."""
    es = 2 if cw["io_dtype"] == "bf16" else 4
    cd = cw["d_inner"] + 2 * cw["ngroups"] * cw["dstate"]
    tokens = cw["batch"] * cw["seqlen"]
    return 2 * tokens * cd * es + cd * (cw["kernel_size"] + 1) * 4


def norm_algorithmic_bytes(nw) -> int:
    """y and z read once, out written once (io dtype), plus the weight."""
    es = 2 if nw["io_dtype"] == "bf16" else 4
    tokens = nw["batch"] * nw["seqlen"]
    return 3 * tokens * nw["d_inner"] * es + nw["d_inner"] * 4


def run_layer_op(args, which):
    """Time ssd_conv1d_silu or ssd_gated_rmsnorm on the 2.7B-layer shape, reading
    xBC / the gate in place from a synthetic in_proj output."""
    import torch

    from mamba_ssd_chunked_gb300.inputs import CONV_WORKLOAD, NORM_WORKLOAD, make_layer_inputs

    pkg = _load_pkg()
    cw = CONV_WORKLOAD if which == "conv" else NORM_WORKLOAD
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    b, L, di, g, n, h = cw["batch"], cw["seqlen"], cw["d_inner"], cw["ngroups"], cw["dstate"], cw["nheads"]
    K = cw.get("kernel_size", 4)
    inp = make_layer_inputs(b, L, di, g, n, h, kernel_size=K, io_dtype=cw["io_dtype"], seed=cw["seed"])
    tdt = torch.bfloat16 if cw["io_dtype"] == "bf16" else torch.float32
    zx = torch.from_numpy(inp["zxbcdt"]).to(dev).to(tdt)
    cd = di + 2 * g * n
    stream = torch.cuda.current_stream(dev)
    cfg = {"workload": cw["name"], "batch": b, "seqlen": L, "d_inner": di, "ngroups": g, "dstate": n,
           "in_proj_row": int(zx.shape[-1]),
           "l2": "flushed between timed steps (256 MiB write); the inputs also exceed L2"}
    if which == "conv":
        w = torch.from_numpy(inp["conv_w"]).to(dev)
        bias = torch.from_numpy(inp["conv_b"]).to(dev)
        xbc = zx[..., di:di + cd]
        cfg["kernel_size"] = K

        def op():
            pkg.ssd_conv1d_silu(xbc, w, bias, di, g, n, stream=stream.cuda_stream)

        per, launches, ck = _time_op(args, dev, stream, op)
        return _op_line(args, "causal conv1d + SiLU tokens/s (Mamba2-2.7B layer xBC), 1 GB300", b * L, "tokens/s",
                        per, launches, ck, cfg, conv_algorithmic_bytes(cw), "conv", "conv1d_fwd", cw["io_dtype"])
    y = torch.from_numpy(inp["y"]).to(dev).to(tdt)
    z = zx[..., :di]
    nw = torch.from_numpy(inp["norm_w"]).to(dev)
    out = torch.empty_like(y)
    cfg["eps"] = cw["eps"]

    def op():
        pkg.ssd_gated_rmsnorm(y, z, nw, eps=cw["eps"], out=out, stream=stream.cuda_stream)

    per, launches, ck = _time_op(args, dev, stream, op)
    return _op_line(args, "gated RMSNorm tokens/s (Mamba2-2.7B layer, norm_before_gate=False), 1 GB300", b * L,
                    "tokens/s", per, launches, ck, cfg, norm_algorithmic_bytes(cw), "norm", "gated_rmsnorm",
                    cw["io_dtype"])


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(WORKLOADS))
    ap.add_argument("--seqlen", type=int, default=None,
                    help="a shorter (or longer) case of the workload: its shapes and recipe with this sequence "
                         "length (for profiler captures of a smaller case; the line's config carries the length)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--path", default="auto", choices=["auto", "tc", "chain", "simt"],
                    help="kernel path of the timed step (auto: the library's choice)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle timing for cpu_baseline")
    ap.add_argument("--step", action="store_true",
                    help="time the decode step (ssd_step) on its own workload instead of the forward")
    ap.add_argument("--conv", action="store_true", help="time the causal conv1d + SiLU (ssd_conv1d_silu)")
    ap.add_argument("--norm", action="store_true", help="time the gated RMSNorm (ssd_gated_rmsnorm)")
    args = ap.parse_args(argv)
    if args.steps < 1:
        ap.error("--steps must be >= 1")
    if args.step:
        print(json.dumps(run_step(args)), flush=True)
        return
    if args.conv or args.norm:
        print(json.dumps(run_layer_op(args, "conv" if args.conv else "norm")), flush=True)
        return
    w = WORKLOADS[args.workload]
    if args.seqlen is not None:
        if args.seqlen < 1:
            ap.error("--seqlen must be >= 1")
        w = dataclasses.replace(w, seqlen=args.seqlen)
    world, rank, local, pg = dist_setup(args)
    if args.impl == "reference":
        out = run_reference(args, w, world, rank)
    else:
        out = run_ours(args, w, world, rank, local, pg)
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
