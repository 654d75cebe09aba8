"""Benchmark of the exact tiled attention forward (one JSON line on rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--cpu-sample-s SECONDS]

One step = one forward of the whole path (every query tile of every head) over
the headline workload B=1, H=32, N=8192, d=128, bf16, causal, with inputs
already resident in device memory. Q, K, V and O total 268 MB, more than the
126 MB L2, so no flush is done between steps (stated in ``config``).

``value`` is attention TFLOP/s (4*B*H*N^2*d, halved for causal) summed over all
ranks; each rank runs its own copy of the workload (independent problems, no
collective on the data path; weak scaling). ``e2e`` is the same metric through
the C ABI with pinned host buffers: each step copies Q, K, V host->device and
O, lse device->host inside the timed region, through ``fa_fwd_host`` (the copies
of one head chunk overlap the forward of another). ``roofline`` compares the kernel's
algorithmic flops per launch / its CUDA-event duration with the measured dense
bf16 tensor peak. ``cpu_baseline`` times the fp64 oracle on a bounded sample of
query rows of the same workload on the host cores (rank 0, N=1 only).

``--impl reference`` times that fp64 oracle as the reference arm (the method's
pages ship no code to run); its value is a deliberately slow program's rate.
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from io_aware_exact_13_gb300.shard import head_range  # noqa: E402
from io_aware_exact_13_gb300.inputs import (BWD_WORKLOADS, DECODE_WORKLOADS, GQA_WORKLOADS, HEADLINE,  # noqa: E402
                                            VARLEN_WORKLOADS, WORKLOADS, make_bwd, make_decode, make_gqa,
                                            make_varlen, make_workload, sample_rows)

METRIC = "attention fwd TFLOP/s and % of GB300 dense BF16 peak (B=1,H=32,N=8192,d=128 causal)"
UNIT = "TFLOP/s"
KERNEL_SOURCES = ["io_aware_exact_13_gb300/csrc/fa_fwd_bk128.cuh", "io_aware_exact_13_gb300/csrc/fa_fwd_kernel.cuh",
                  "io_aware_exact_13_gb300/csrc/ptx.cuh",
                  "io_aware_exact_13_gb300/csrc/fa_launch.cuh"]
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_BF16_TFLOPS = 1900.0
E2E_CHUNKS = 4  # head chunks of the pipelined host-memory forward (1.24 ms vs 1.76 ms serial on the headline)


L2_BYTES = 126 * 1024 * 1024  # GB300 L2 as reported by the driver


def workload_bytes(w) -> int:
    """Bytes of Q, K, V, O, lse (and the mask) of one forward of a dense workload."""
    eb = {"bf16": 2, "fp16": 2, "fp32": 4}[w.dtype]
    n = 4 * w.B * w.H * w.N * w.d * eb + 4 * w.B * w.H * w.N
    return n + (4 * w.B * w.N * w.N if w.has_mask else 0)


def fits_in_l2(w) -> bool:
    """Inputs and outputs that L2 could hold (with room to spare): timed on rotating copies (l2_copies)."""
    return workload_bytes(w) < 2 * L2_BYTES


def l2_copies(w) -> int:
    """Copies of a workload that fits in L2, used in turn step by step: a copy comes back only after
    more than twice the L2 has been touched by the others."""
    return int(math.ceil(2 * L2_BYTES / workload_bytes(w))) + 1


def bench_config(w, world: int, split: bool = False) -> dict:
    """The ``config`` object of both arms' JSON lines (the same workload, the same keys)."""
    mb = workload_bytes(w) / 1e6
    l2 = (f"inputs and outputs ({mb:.0f} MB) exceed the 126 MB L2; no flush between steps" if not fits_in_l2(w)
          else f"inputs and outputs ({mb:.2f} MB) fit in L2: each step uses the next of {l2_copies(w)} copies "
               f"({l2_copies(w) * mb:.0f} MB in all, so none is in L2 when it comes back), and the timed steps "
               f"are replayed from CUDA graphs")
    par = (f"heads split over {world} ranks (one problem, no collective)" if split
           else f"replicas x{world} (independent problems, no collective)")
    return dict(w.describe(), l2=l2, parallelism=par)


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_hbm_peak():
    try:
        with open(PEAKS_FILE) as f:
            return float(json.load(f)["hbm_gbs"]), "measured copy bandwidth (MEASURED_PEAKS.json)"
    except Exception:
        return 6800.0, "fallback 6.8 TB/s (no measured peak file)"


def load_peak():
    try:
        with open(PEAKS_FILE) as f:
            pk = json.load(f)
        return float(pk["bf16_tflops"]), "measured bf16 burst (MEASURED_PEAKS.json)"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback 1.9 PFLOP/s bf16 (no measured peak file)"


def load_traffic(workload: str, kernel: str = "fa_fwd_bk128_kernel"):
    """DRAM bytes per launch from the committed ncu summary of this kernel and
    workload, if it was taken on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    try:
        txt = open(path).read()
    except OSError:
        return None
    m = re.search(r"kernel_source_hash:\s*([0-9a-f]+)", txt)
    t = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    if not m or not t or m.group(1) != kernel_source_hash():
        return None
    return float(t.group(1))


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples taken while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return world, rank, local


def barrier(world, dev=None):
    if world > 1:
        import torch.distributed as dist

        dist.barrier(device_ids=[dev.index] if dev is not None and dev.type == "cuda" else None)


def max_over_ranks(world, x: float, dev) -> float:
    if world == 1:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, units_per_rank: float, max_ms: float) -> float:
    """Units per second of the whole job: every rank processes its own copy of the
    workload, and the slowest rank's time (max over ranks) is the job's time."""
    return world * units_per_rank / (max_ms * 1e-3)


def oracle_sample(w, q, k, v, mask, n_rows: int, seed: int):
    """Time the fp64 oracle on n_rows sampled query rows; return (seconds, flops, threads)."""
    import oracle

    rows = sample_rows(w.B * w.H * w.N, n_rows, seed).numpy()
    i = rows % w.N
    keys = (i + 1) if w.causal else w.N
    flops = float((4.0 * w.d * keys).sum() if w.causal else 4.0 * w.d * w.N * len(rows))
    q64, k64, v64 = (t.double().numpy() for t in (q, k, v))
    m64 = None if mask is None else mask.double().numpy()
    t0 = time.perf_counter()
    oracle.attention_rows(q64, k64, v64, rows, mask=m64, scale=w.scale, causal=w.causal)
    return time.perf_counter() - t0, flops, oracle.num_threads()


def calibrate_rows(w, q, k, v, mask, target_s: float):
    """Number of sampled rows whose oracle run takes about target_s seconds."""
    n = 256
    while True:
        dt, _, _ = oracle_sample(w, q, k, v, mask, n, seed=99)
        if dt > 0.5 or n >= w.B * w.H * w.N:
            return max(1, min(w.B * w.H * w.N, int(n * target_s / max(dt, 1e-6))))
        n *= 4


def run_reference(args, w):
    world, rank, _ = dist_setup()
    if rank != 0:
        return 0
    q, k, v, mask = make_workload(w)
    # keep the whole reference run to about two minutes of oracle work
    per_step = min(args.ref_step_s, max(0.2, 120.0 / max(1, args.steps + args.warmup)))
    n_rows = calibrate_rows(w, q, k, v, mask, per_step)
    for s in range(args.warmup):
        oracle_sample(w, q, k, v, mask, n_rows, seed=s)
    tot_t, tot_f, threads = 0.0, 0.0, 1
    for s in range(args.steps):
        dt, fl, threads = oracle_sample(w, q, k, v, mask, n_rows, seed=1000 + s)
        tot_t += dt
        tot_f += fl
    value = tot_f / tot_t / 1e12
    sample = f"{n_rows} uniformly sampled query rows of {w.name} per step (fp64 materialised rows)"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * tot_t / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": bench_config(w, world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, w):
    world, rank, local = dist_setup()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from io_aware_exact_13_gb300 import fa

    entry = {"bf16": fa.fa_fwd, "fp16": fa.fa_fwd_fp16, "fp32": fa.fa_fwd_fp32}[w.dtype]
    q, k, v, mask = make_workload(w)
    if mask is not None and w.dtype in ("bf16", "fp16") and not args.fp32_mask:
        # the masked entry point with its workspace: the mask is packed to one bit per entry in every call
        masked_fn = fa.fa_fwd_masked if w.dtype == "bf16" else fa.fa_fwd_masked_fp16
        mask_ws = torch.empty(fa.fa_fwd_masked_workspace_bytes(w.B, w.N), dtype=torch.uint8, device=dev)

        def entry(q_, k_, v_, m_, o_, l_, s_, c_, st_):
            masked_fn(q_, k_, v_, m_, o_, l_, s_, c_, mask_ws, st_)
    # --partition heads: this rank computes heads [h0, h1) of every batch index of the one problem
    # (strong scaling, no collective); otherwise every rank computes the whole problem (replicas)
    split = args.partition == "heads" and world > 1
    h0, h1 = head_range(w.H, world, rank) if split else (0, w.H)
    if split:
        q, k, v = (t[:, h0:h1].contiguous() for t in (q, k, v))
    units_rank = w.flops * (h1 - h0) / w.H
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    md = None if mask is None else mask.to(dev)
    od = torch.empty_like(qd)
    lsed = torch.empty((w.B, h1 - h0, w.N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        entry(qd, kd, vd, md, od, lsed, w.scale, w.causal, stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    if fa.fa_get_device_status(stream) != 0:
        raise SystemExit("device status word set during warm-up")

    # ---------------------------------------------------------------- device-resident timing
    # The K-step region is timed `repeats` times (each bracketed by a barrier and a synchronize) so
    # that the clock sampler sees the kernel for about a second; the median repeat is reported.
    # A workload that fits in L2 runs each step on the next of several copies of its tensors (so every
    # step starts from DRAM) and replays the K steps from CUDA graphs, one per group of K copies: host
    # launch overhead and an L2 flush between steps would otherwise be what the events measure.
    rotate = fits_in_l2(w)
    graphs = []
    if rotate:
        n_copies = l2_copies(w)
        copies = [(qd.clone(), kd.clone(), vd.clone(), None if md is None else md.clone(), torch.empty_like(od),
                   torch.empty_like(lsed)) for _ in range(n_copies)]
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        for g0 in range(0, n_copies, args.steps):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(cap):
                for i in range(args.steps):  # every copy once before the capture (warm-up)
                    c = copies[(g0 + i) % n_copies]
                    entry(c[0], c[1], c[2], c[3], c[4], c[5], w.scale, w.causal, cap)
            cap.synchronize()
            with torch.cuda.graph(g, stream=cap):
                for i in range(args.steps):
                    c = copies[(g0 + i) % n_copies]
                    entry(c[0], c[1], c[2], c[3], c[4], c[5], w.scale, w.causal, cap)
            graphs.append(g)
        torch.cuda.synchronize(dev)
        for g in graphs:  # warm replays
            g.replay()
        torch.cuda.synchronize(dev)
    sampler = ClockSampler(dev.index) if rank == 0 else None
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    step()
    torch.cuda.synchronize(dev)
    est_ms = max(1e-3, (time.perf_counter() - t0) * 1e3)
    repeats = max(1, min(args.max_repeats, int(math.ceil(args.timed_s * 1e3 / (est_ms * args.steps)))))
    if sampler:
        sampler.start()
        time.sleep(0.3)
    launch_ms, rep_ms = [], []
    for rep in range(repeats):
        barrier(world, dev)
        torch.cuda.synchronize(dev)
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        if rotate:
            g = graphs[rep % len(graphs)]
            t_start.record(stream)
            g.replay()
            t_end.record(stream)
            torch.cuda.synchronize(dev)
            region = t_start.elapsed_time(t_end)
            launch_ms += [region / args.steps] * args.steps
        else:
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(args.steps)]
            t_start.record(stream)
            for i in range(args.steps):
                ev[i][0].record(stream)
                step()
                ev[i][1].record(stream)
            t_end.record(stream)
            torch.cuda.synchronize(dev)
            launch_ms += [a.elapsed_time(b) for a, b in ev]
            region = t_start.elapsed_time(t_end)
        barrier(world, dev)
        rep_ms.append(max_over_ranks(world, region, dev))
    clocks = sampler.stop() if sampler else None
    total_ms = statistics.median(rep_ms)
    status = fa.fa_get_device_status(stream)
    if status != 0:
        raise SystemExit(f"device status word {status} after the timed region")
    ms_per_step = total_ms / args.steps
    # the whole job: every rank's units (a replica each, or a share of one problem) over the slowest rank's time
    job_units = (w.flops if split else world * w.flops) * args.steps
    value = job_units / (total_ms * 1e-3) / 1e12

    # ---------------------------------------------------------------- end to end through host buffers
    qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
    mh = None if mask is None else mask.pin_memory()
    oh = torch.empty(od.shape, dtype=od.dtype).pin_memory()
    lh = torch.empty(lsed.shape, dtype=torch.float32).pin_memory()

    # Through the host-memory entry point (copies pipelined with the forward over 4 head chunks) where it
    # applies (bf16 / fp16, no mask); otherwise copy in, forward, copy out in sequence.
    host_entry = {"bf16": fa.fa_fwd_host, "fp16": fa.fa_fwd_host}.get(w.dtype) if mh is None else None

    def e2e_step():
        if host_entry is not None:
            host_entry(qh, kh, vh, oh, lh, qd, kd, vd, od, lsed, w.scale, w.causal, E2E_CHUNKS, stream)
            return
        qd.copy_(qh, non_blocking=True)
        kd.copy_(kh, non_blocking=True)
        vd.copy_(vh, non_blocking=True)
        if mh is not None:
            md.copy_(mh, non_blocking=True)
        step()
        oh.copy_(od, non_blocking=True)
        lh.copy_(lsed, non_blocking=True)

    e2e_steps = max(1, min(args.steps, 20))
    e2e_step()
    torch.cuda.synchronize(dev)
    barrier(world, dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world, dev)
    e2e_ms = max_over_ranks(world, e0.elapsed_time(e1), dev) / e2e_steps
    job_flops = w.flops if split else world * w.flops
    h2d = sum(t.numel() * t.element_size() for t in (qh, kh, vh) + ((mh,) if mh is not None else ()))
    d2h = oh.numel() * oh.element_size() + lh.numel() * 4

    if rank != 0:
        return 0
    peak, peak_src = load_peak()
    mean_launch_s = statistics.mean(launch_ms) * 1e-3
    achieved = units_rank / mean_launch_s / 1e12
    if w.dtype == "fp32":
        # CUDA-core FFMA path: 128 fp32 FMA lanes per SM (2 flop each) at the maximum SM clock
        peak, peak_src = 2 * 128 * fa.fa_num_sms() * 2.07e9 / 1e12, "fp32 FFMA rate at 2070 MHz (unit counts)"
    roofline = {"bound": "alu" if w.dtype == "fp32" else "tensor", "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": (None if w.dtype == "fp32" else
                            load_traffic(w.name, "fa_fwd_kernel" if args.fp32_mask else "fa_fwd_bk128_kernel")),
                "peak_source": peak_src,
                "kernel": ("fa_fwd_fp32_kernel" if w.dtype == "fp32" else
                           "fa_fwd_kernel (64-key blocks, fp32 mask)" if (w.has_mask and args.fp32_mask) else
                           "fa_fwd_bk128_kernel (mask packed to one bit per entry; the timed call includes the "
                           "packing pass)" if w.has_mask else "fa_fwd_bk128_kernel"),
                "launch_ms_mean": 1e3 * mean_launch_s,
                "launch_ms_median": statistics.median(launch_ms),
                "launch_ms_min": min(launch_ms), "launch_ms_max": max(launch_ms)}
    # second denominator: the tensor core's own rate (8192 flop/clk/SM for dense 16-bit MMAs, measured at
    # 8190 in isolation) at the median SM clock sampled during the timed region
    mhz = clocks.get("sm_mhz") if clocks else None
    if mhz and w.dtype in ("bf16", "fp16"):
        at_clock = 8192.0 * fa.fa_num_sms() * mhz * 1e6 / 1e12
        roofline["peak_at_sampled_clock"] = at_clock
        roofline["frac_at_sampled_clock"] = achieved / at_clock
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "strong" if split else "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": bench_config(w, world, split),
        "timing": {"repeats": len(rep_ms), "ms_per_step_median": ms_per_step,
                   "ms_per_step_min": min(rep_ms) / args.steps, "ms_per_step_max": max(rep_ms) / args.steps,
                   "timed_s": sum(rep_ms) * 1e-3,
                   "ms_x_mhz": (ms_per_step * clocks["sm_mhz"]) if clocks and clocks.get("sm_mhz") else None},
        "pct_of_peak": 100.0 * value / (world * peak),
        "e2e": {"value": job_flops / (e2e_ms * 1e-3) / 1e12, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "path": (f"fa_fwd_host, {E2E_CHUNKS} head chunks, copies pipelined with the forward"
                         if host_entry is not None else
                         "copy in (mask included), fa_fwd_masked with its workspace, copy out"
                         if (w.has_mask and w.dtype != "fp32" and not args.fp32_mask) else
                         "copy in, fa_fwd, copy out")},
        # kernels per call: the forward; with a mask also the packing pass and the fp32-mask kernel (which
        # returns at once for a 0/-inf mask)
        "gpu_launches": args.steps * len(rep_ms) * (3 if (w.has_mask and w.dtype != "fp32" and not args.fp32_mask)
                                                    else 1),
        "roofline": roofline,
        "clocks": clocks,
    }
    if world == 1 and not args.no_cpu_baseline:
        n_rows = calibrate_rows(w, q, k, v, mask, args.cpu_sample_s)
        dt, fl, threads = oracle_sample(w, q, k, v, mask, n_rows, seed=12345)
        line["cpu_baseline"] = {"value": fl / dt / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
                                "sample": f"{n_rows} uniformly sampled query rows of {w.name} "
                                          f"(fp64 materialised rows, {dt:.1f} s)"}
    print(json.dumps(line), flush=True)
    return 0


def run_decode(args, w):
    """Split-KV decoding forward: HBM-bound (every K and V byte read once per call)."""
    world, rank, local = dist_setup()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from io_aware_exact_13_gb300 import fa

    q, k, v = make_decode(w)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    n_splits = fa.fa_splitkv_num_splits(w.B, w.H, w.Nq, w.Nk, w.d)
    ws = torch.empty(fa.fa_splitkv_workspace_bytes(w.B, w.H, w.Nq, w.d, n_splits), dtype=torch.uint8, device=dev)
    od = torch.empty_like(qd)
    lsed = torch.empty((w.B, w.H, w.Nq), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    entry = fa.fa_fwd_splitkv if w.dtype == "bf16" else fa.fa_fwd_splitkv_fp16

    def step():
        entry(qd, kd, vd, od, lsed, w.scale, w.causal, n_splits, ws, stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(dev.index) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    barrier(world, dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):
        step()
    b.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop() if sampler else None
    ms = max_over_ranks(world, a.elapsed_time(b), dev) / args.steps
    if rank != 0:
        return 0
    peak, src = load_hbm_peak()
    bytes_alg = w.kv_bytes + 2 * qd.numel() * qd.element_size() + lsed.numel() * 4
    gbs = bytes_alg / (ms * 1e-3) / 1e9
    line = {"metric": "split-KV decode effective HBM GB/s", "value": world * gbs, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": dict(w.describe(), n_splits=n_splits,
                           l2="K/V (%.0f MB) exceed the 126 MB L2; no flush" % (w.kv_bytes / 1e6)),
            "gpu_launches": 2 * args.steps,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                         "traffic": None, "peak_source": src, "kernel": "fa_splitkv_partial + fa_splitkv_combine",
                         "tflops": w.flops / (ms * 1e-3) / 1e12},
            "clocks": clocks}
    print(json.dumps(line), flush=True)
    return 0


def run_varlen(args, w):
    """Packed variable-length batch through the persistent forward kernel."""
    world, rank, local = dist_setup()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from io_aware_exact_13_gb300 import fa

    L = w.lengths()
    q, k, v, cu = make_varlen(L, w.H, w.H, w.d, w.dtype, seed=w.seed)
    qd, kd, vd, cud = q.to(dev), k.to(dev), v.to(dev), cu.to(dev)
    od = torch.empty_like(qd)
    lsed = torch.empty((w.H, w.total), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    entry = fa.fa_fwd_varlen if w.dtype == "bf16" else fa.fa_fwd_varlen_fp16

    def step():
        entry(qd, kd, vd, od, lsed, cud, max(L), w.scale, w.causal, stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    if fa.fa_get_device_status(stream) != 0:
        raise SystemExit("device status word set during warm-up")
    sampler = ClockSampler(dev.index) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    barrier(world, dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):
        step()
    b.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world, dev)
    clocks = sampler.stop() if sampler else None
    ms = max_over_ranks(world, a.elapsed_time(b), dev) / args.steps
    if rank != 0:
        return 0
    peak, src = load_peak()
    tflops = w.flops() / (ms * 1e-3) / 1e12
    line = {"metric": "attention fwd TFLOP/s, packed variable-length batch", "value": world * tflops,
            "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": dict(w.describe(), workload=args.workload, l2="no flush between steps"),
            "gpu_launches": args.steps,
            "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s",
                         "frac": tflops / peak, "traffic": None, "peak_source": src,
                         "kernel": "fa_fwd_kernel (packed batch)"},
            "clocks": clocks}
    print(json.dumps(line), flush=True)
    return 0


def run_gqa(args, w):
    """Grouped-query forward: H query heads over Hkv key/value heads, the persistent forward kernel."""
    world, rank, local = dist_setup()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from io_aware_exact_13_gb300 import fa

    q, k, v = make_gqa(w)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    od = torch.empty_like(qd)
    lsed = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    entry = fa.fa_fwd_gqa if w.dtype == "bf16" else fa.fa_fwd_gqa_fp16

    def step():
        entry(qd, kd, vd, None, od, lsed, w.scale, w.causal, stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    if fa.fa_get_device_status(stream) != 0:
        raise SystemExit("device status word set during warm-up")
    sampler = ClockSampler(dev.index) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    barrier(world, dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):
        step()
    b.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world, dev)
    clocks = sampler.stop() if sampler else None
    ms = max_over_ranks(world, a.elapsed_time(b), dev) / args.steps
    if rank != 0:
        return 0
    peak, src = load_peak()
    tflops = w.flops() / (ms * 1e-3) / 1e12
    line = {"metric": "attention fwd TFLOP/s, grouped-query attention", "value": world * tflops, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": dict(w.describe(), workload=args.workload, l2="no flush between steps"),
            "gpu_launches": args.steps,
            "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s",
                         "frac": tflops / peak, "traffic": None, "peak_source": src,
                         "kernel": "fa_fwd_kernel (grouped-query)"},
            "clocks": clocks}
    print(json.dumps(line), flush=True)
    return 0


def materialised_backward(q, k, v, dout, scale, causal):
    """The stored-state comparison path of the backward measurement, in plain
    torch ops: S and P are materialised ([B,H,N,N]) by the forward and P is
    kept for the backward, as a conventional autograd graph does. Returns a
    callable that runs one backward from the saved P."""
    N = q.shape[2]
    s = torch.matmul(q, k.transpose(-1, -2)).float() * scale
    if causal:
        s.masked_fill_(torch.ones(N, N, dtype=torch.bool, device=q.device).triu_(1), float("-inf"))
    p = torch.softmax(s, dim=-1).to(q.dtype)
    del s

    def backward():
        dv = torch.matmul(p.transpose(-1, -2), dout)
        dp = torch.matmul(dout, v.transpose(-1, -2)).float()
        ds = (p.float() * (dp - (dp * p.float()).sum(-1, keepdim=True))).to(q.dtype)
        del dp
        dq = torch.matmul(ds, k) * scale
        dk = torch.matmul(ds.transpose(-1, -2), q) * scale
        return dq, dk, dv

    return p, backward


def run_bwd(args, w):
    """Backward by recomputation (three launches per call: row statistics, the
    tiled tcgen05 backward, dQ conversion) against the materialised path."""
    world, rank, local = dist_setup()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from io_aware_exact_13_gb300 import fa

    q, k, v, do = make_bwd(w.B, w.H, w.N, w.d, w.dtype, seed=w.seed)
    qd, kd, vd, dod = q.to(dev), k.to(dev), v.to(dev), do.to(dev)
    stream = torch.cuda.current_stream(dev)
    od, lsed = fa.attention(qd, kd, vd, scale=w.scale, causal=w.causal)
    ws = torch.empty(fa.fa_bwd_workspace_bytes(w.B, w.H, w.N, w.d), dtype=torch.uint8, device=dev)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    entry = fa.fa_bwd if w.dtype == "bf16" else fa.fa_bwd_fp16

    def step():
        entry(qd, kd, vd, od, dod, lsed, dq, dk, dv, w.scale, w.causal, ws, stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    if fa.fa_get_device_status(stream) != 0:
        raise SystemExit("device status word set during warm-up")
    sampler = ClockSampler(dev.index) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    barrier(world, dev)
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):
        step()
    b.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world, dev)
    clocks = sampler.stop() if sampler else None
    ms = max_over_ranks(world, a.elapsed_time(b), dev) / args.steps
    if fa.fa_get_device_status(stream) != 0:
        raise SystemExit("device status word set in the timed region")

    # peak device memory of one forward + backward, each path on its own
    def peak_of(fn):
        torch.cuda.synchronize(dev)
        torch.cuda.empty_cache()
        base = torch.cuda.memory_allocated(dev)
        torch.cuda.reset_peak_memory_stats(dev)
        fn()
        torch.cuda.synchronize(dev)
        return torch.cuda.max_memory_allocated(dev) - base

    def ours_fwd_bwd():
        o, l = fa.attention(qd, kd, vd, scale=w.scale, causal=w.causal)
        fa.attention_backward(qd, kd, vd, o, dod, l, scale=w.scale, causal=w.causal)

    def mat_fwd_bwd():
        p, bwd = materialised_backward(qd, kd, vd, dod, w.scale, w.causal)
        torch.matmul(p, vd)
        bwd()

    peak_ours = peak_of(ours_fwd_bwd)
    peak_mat = mat_ms = None
    if not args.no_materialised:
        peak_mat = peak_of(mat_fwd_bwd)
        p, bwd = materialised_backward(qd, kd, vd, dod, w.scale, w.causal)
        for _ in range(3):
            bwd()
        torch.cuda.synchronize(dev)
        m_steps = max(1, min(args.steps, 50))
        a.record(stream)
        for _ in range(m_steps):
            bwd()
        b.record(stream)
        torch.cuda.synchronize(dev)
        mat_ms = a.elapsed_time(b) / m_steps
        del p, bwd
    if rank != 0:
        return 0
    peak, src = load_peak()
    tflops = w.flops() / (ms * 1e-3) / 1e12
    n2 = w.B * w.H * w.N * w.N
    line = {"metric": "attention bwd TFLOP/s (recomputation)", "value": world * tflops, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
            "data": "synthetic", "config": dict(w.describe(), workload=args.workload, l2="no flush between steps"),
            "gpu_launches": 3 * args.steps,
            "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s",
                         "frac": tflops / peak, "traffic": None, "peak_source": src,
                         "kernel": "fa_bwd call (fa_bwd_pre + fa_bwd_kernel + fa_bwd_post)"},
            "recompute": {"ms": ms, "peak_bytes_fwd_bwd": peak_ours},
            "materialised": {"ms": mat_ms, "peak_bytes_fwd_bwd": peak_mat,
                             "p_bytes": n2 * qd.element_size(),
                             "path": "torch matmul/softmax with P saved in the input type"},
            "clocks": clocks}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE,
                    choices=sorted(WORKLOADS) + sorted(DECODE_WORKLOADS) + sorted(BWD_WORKLOADS)
                    + sorted(VARLEN_WORKLOADS) + sorted(GQA_WORKLOADS))
    ap.add_argument("--cpu-sample-s", type=float, default=10.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--ref-step-s", type=float, default=5.0, help="seconds of oracle work per reference step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--fp32-mask", action="store_true",
                    help="masked workload through fa_fwd / fa_fwd_fp16 without a workspace (the fp32-mask kernel)")
    ap.add_argument("--timed-s", type=float, default=2.0,
                    help="repeat the K-step timed region until about this many seconds are covered")
    ap.add_argument("--max-repeats", type=int, default=5000)
    ap.add_argument("--partition", choices=["replicas", "heads"], default="replicas",
                    help="N>1: every rank runs the whole workload (replicas, weak scaling) or one share of its "
                         "heads (heads, strong scaling)")
    ap.add_argument("--no-materialised", action="store_true",
                    help="backward workloads: skip the materialised comparison leg")
    args = ap.parse_args()
    if args.workload in DECODE_WORKLOADS:
        return run_decode(args, DECODE_WORKLOADS[args.workload])
    if args.workload in BWD_WORKLOADS:
        return run_bwd(args, BWD_WORKLOADS[args.workload])
    if args.workload in VARLEN_WORKLOADS:
        return run_varlen(args, VARLEN_WORKLOADS[args.workload])
    if args.workload in GQA_WORKLOADS:
        return run_gqa(args, GQA_WORKLOADS[args.workload])
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
