"""Throughput of the SCAPE optimizer step on one GB300 (or N independent replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl scape|reference]
                    [--workload NAME] [--density D]

A step is one pass of the whole hot path (offsets of M_{t-1}, the per-worker
streaming pass, the fixed-order reduction with the AdamS update, the
partitioned top-k) over one batch of W synthetic bf16 gradients already
resident in HBM.  Default workload: the Llama-style 1775.4M-parameter layout,
W=4 emulated workers, density 0.01, chunk 65536.  Prints one JSON line.

--impl reference times the CPU oracle instead (single thread, host cores) on a
bounded sample of whole chunks of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "SCAPE optimizer step params/s and achieved HBM GB/s (% of 8 TB/s) on 1 GB300"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3, help=">= 1; the first warm-up step is step 0")
    ap.add_argument("--impl", default="scape", choices=["scape", "reference"])
    ap.add_argument("--workload", default=synth.BENCH_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--density", type=float, default=None)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-pageable", action="store_true",
                    help="also time the staged-copy path with pageable host gradients")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-dense", action="store_true", help="skip the dense AdamS comparator")
    ap.add_argument("--mask-stats", action="store_true",
                    help="report mask overlap and the fill-in of per-worker global top-k")
    ap.add_argument("--workers", type=int, default=None, help="override W of the workload")
    ap.add_argument("--seed", type=int, default=None,
                    help="override the workload's generator seed (recorded in config)")
    ap.add_argument("--per-tensor", action="store_true", help="chunks restart at every tensor")
    ap.add_argument("--residual-host", action="store_true",
                    help="keep the residuals in page-locked host memory")
    ap.add_argument("--union-mask", action="store_true",
                    help="the non-partitioned variant: the union of every worker's top-k")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the sweep over every layout and density (the 'workloads' rows)")
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


class Ranks:
    """Process-group plumbing of the replica runs: barrier, max over ranks.
    ``backend`` None means a single process (no group)."""

    def __init__(self, backend: str | None, device=None):
        self.dist = None
        self.device = device
        if backend:
            import torch.distributed as dist
            if backend == "nccl":
                dist.init_process_group("nccl", device_id=device)
            else:
                dist.init_process_group(backend)
            self.dist = dist

    def barrier(self):
        if self.dist:
            self.dist.barrier()

    def max(self, x: float) -> float:
        if not self.dist:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64,
                         device=self.device if self.device is not None else "cpu")
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.dist:
            self.dist.destroy_process_group()


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def needs_l2_flush(working_bytes: int, l2_bytes: int) -> bool:
    """A working set under four times the L2 size could be partly served from
    L2 between back-to-back steps: the bench then evicts it before every
    timed step."""
    return working_bytes < 4 * l2_bytes


# The GB300's L2; the flush decision and the config's L2 note use this
# figure on both arms (the GPU arm sizes its flush buffer from the device).
GB300_L2_BYTES = 126 << 20

# Work of the oracle sample both CPU legs time, in coordinate x worker x step
# units: about 12 s on one Grace core (the oracle runs at about 13 M
# coordinate-steps/s at W = 4 and its cost grows with W).
CPU_SAMPLE_WORK = 6.4e8


def baseline_sample_size(N: int, chunk: int, W: int, work: float = CPU_SAMPLE_WORK):
    """(chunks, timed steps) of the oracle sample: 13 timed steps (after the
    untimed step 0) over as many whole chunks as `work` allows, or every chunk
    over more steps when the whole layout fits.  Fixed by the workload alone,
    so the cpu_baseline leg and the reference arm time the same sample."""
    nch = -(-N // chunk)
    n_st = 13
    n_ch = int(work / (n_st * chunk * W))
    if n_ch >= nch:
        n_ch, n_st = nch, max(13, int(work / (N * W)))
    return max(1, n_ch), n_st


def static_K(wl, density: float, per_tensor: bool = False) -> int:
    """Kept coordinates per step of the partitioned rule: the sum over chunks
    of floor(density * chunk length) (flat chunks, or each tensor's own)."""
    import math
    lens = []
    if per_tensor:
        for n in wl.numel:
            lens += [min(wl.chunk, n - x) for x in range(0, n, wl.chunk)]
    else:
        nch = -(-wl.N // wl.chunk)
        lens = [wl.chunk] * (nch - 1) + [wl.N - (nch - 1) * wl.chunk]
    return sum(math.floor(density * ln) for ln in lens)


def working_set_bytes(N: int, W: int, K: int, n_batches: int = 2) -> int:
    """Bytes a step touches on the device: theta, v, u_w, e_w, the two masks,
    the compact buffers and the gradient batches the steps alternate."""
    return N * (8 + 8 * W) + N // 4 + K * (4 * W + 8) + n_batches * W * N * 2


def line_config(wl, density: float, args, world: int) -> dict:
    """The JSON line's `config`, computed from the workload alone (the same on
    the scape and the reference arms)."""
    K = static_K(wl, density, args.per_tensor)
    working = working_set_bytes(wl.N, wl.W, K)
    flush = needs_l2_flush(working, GB300_L2_BYTES)
    return {"workload": wl.name, "N": wl.N, "W": wl.W, "density": density, "chunk": wl.chunk,
            "seed": wl.seed, "K": K, "grad_dtype": "bf16", "grad_batches": 2,
            "chunking": "per-tensor" if args.per_tensor else "flat",
            "residuals": "host (page-locked)" if args.residual_host else "HBM",
            "mask": ("union of every worker's top-k (non-partitioned)" if args.union_mask
                     else "partitioned (SCAPE)"),
            "parallelism": "replicas" if world > 1 else "single GPU, W emulated workers",
            "l2": (f"flushed before every timed step (twice the L2 written, untimed): "
                   f"{working / 1e6:.0f} MB working set" if flush else
                   f"no flush: {working / 1e9:.1f} GB working set, far larger than the L2")}


def alg_bytes(N: int, W: int, K: int) -> dict:
    """Algorithmic (compulsory) HBM bytes of one step, all in the fused step kernel:
    per coordinate W*(2 g + 8 u + 8 e + 1/8 applied mask) + 8 theta + 8 v + 1/8 new mask,
    per kept coordinate W*(4 write + 4 read) of the compact values + 4 bbar + 4 idx.
    (The owner's accumulator is ranked on-chip, so it is not read back.)"""
    step = N * (W * (2 + 8 + 8 + 0.125) + 8 + 8 + 0.125) + K * (8 * W + 8)
    return {"step": step}


# throttle reasons that make a timed run invalid (sw_power_cap is only noted)
THROTTLED = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.p = None
        self.idx = gpu_index

    def start(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}",
                                       "--format=csv,noheader,nounits", "-i", str(self.idx),
                                       "-lms", "100"], stdout=subprocess.PIPE,
                                      stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.p = None

    def stop(self) -> dict | None:
        if self.p is None:
            return None
        self.p.terminate()
        try:
            out, _ = self.p.communicate(timeout=5)
        except Exception:
            self.p.kill()
            out, _ = self.p.communicate()
        return self.parse(out)

    @staticmethod
    def parse(out: str) -> dict | None:
        """Median and maximum SM clock and the throttle reasons seen active in
        nvidia-smi's csv,noheader,nounits lines of FIELDS."""
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                smax.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


def ncu_traffic(kernel: str, N: int, workload: str | None = None):
    """Per-launch DRAM bytes (read + write) of the kernel from the committed ncu
    summary: bytes per coordinate of a one-launch capture, times N.  A capture
    on the workload itself is preferred; otherwise one on a smaller layout of
    the same kernel is scaled (its traffic grows in proportion to the
    coordinates).  None when every capture was taken on another source of the
    kernel."""
    src = {"step_chunks": "k_fused.cu"}.get(kernel)
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not src or not os.path.exists(path):
        return None, None
    h = hashlib.sha256(open(os.path.join(ROOT, "sparse_communication_distributed_gb300", "csrc",
                                         src), "rb").read()).hexdigest()[:16]
    found = None
    for line in open(path):
        f = line.split()
        if len(f) >= 4 and f[0] == kernel and f[3] == h:
            if workload is not None and f[1] == workload:
                return float(f[2]) * N, f"ncu capture on {f[1]} itself (one launch)"
            if found is None:
                found = (float(f[2]) * N, f"scaled from an ncu capture on {f[1]}")
    return found if found else (None, None)


def timed_steps(step_fn, steps: int, stream, scratch=None) -> float:
    """Device milliseconds of `steps` calls of step_fn(i) on `stream`, from CUDA
    events.  With `scratch` (a buffer larger than L2) the L2 is flushed before
    every step by an untimed write and each step is timed on its own."""
    import torch
    if scratch is None:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(steps):
            step_fn(i)
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b)
    evs = []
    for i in range(steps):
        scratch.fill_(i & 0xFF)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        step_fn(i)
        b.record(stream)
        evs.append((a, b))
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in evs)


# Every layout and density the throughput is reported on (the five workloads,
# both densities of the 2^26 and Llama-500M layouts).
SWEEP = [("flat-2^20-w4", 0.10), ("flat-2^26-w8-ties", 0.10), ("flat-2^26-w8-ties", 0.01),
         ("gpt2-medium-w8", 0.01), ("llama-500m-w8", 0.01), ("llama-500m-w8", 0.10),
         ("llama-1.8b-w4", 0.01)]


def sweep_steps(steps: int, probe_ms: float, min_ms: float = 400.0, cap: int = 5000) -> int:
    """Timed steps of a sweep row: at least `steps`, and enough for the timed
    region to last min_ms (so the 100 ms clock sampler sees it under load)."""
    want = int(np.ceil(min_ms / max(probe_ms, 1e-3)))
    return int(min(cap, max(steps, want)))


def time_workload(wl, density: float, steps: int, warmup: int, dev, local: int, ranks,
                  peak: float) -> dict:
    """One sweep row: libscape on the workload's layout, `warmup` untimed steps
    (step 0 first), then the timed steps; L2 flushed before every timed step
    when the working set is under four L2 sizes.  The handle and its
    gradients are freed before returning."""
    import torch
    from sparse_communication_distributed_gb300 import THETA, Scape
    world = ranks.dist.get_world_size() if ranks.dist else 1
    N, W = wl.N, wl.W
    sc = Scape.for_workload(wl, density)
    try:
        th = torch.empty(N, dtype=torch.float32, device=dev)
        synth.gpu().theta_into(wl, th)
        torch.cuda.synchronize()
        sc.load(THETA, th)
        del th
        batches = []
        for b in range(2):
            bufs = [torch.empty(N, dtype=torch.int16, device=dev) for _ in range(W)]
            for w in range(W):
                synth.gpu().grads_into(wl, w, b, bufs[w])
            batches.append(bufs)
        stream = torch.cuda.current_stream(dev)
        for i in range(warmup):
            sc.step(batches[i % 2], stream)
        torch.cuda.synchronize()
        l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
        working = working_set_bytes(N, W, sc.K)
        flush = needs_l2_flush(working, GB300_L2_BYTES)
        scratch = torch.empty(2 * l2_bytes, dtype=torch.uint8, device=dev) if flush else None

        def step_fn(i):
            sc.step(batches[i % 2], stream)

        probe_ms = timed_steps(step_fn, 3, stream, scratch) / 3
        n = int(ranks.max(float(sweep_steps(steps, probe_ms))))  # the same count on every rank

        def measure():
            clocks = ClockSampler(local)
            clocks.start()
            time.sleep(0.3)
            ranks.barrier()
            torch.cuda.synchronize()
            ms = timed_steps(step_fn, n, stream, scratch)
            ranks.barrier()
            return ms, clocks.stop()

        ms, clk = measure()
        if clk and THROTTLED & set(clk["reasons"]):
            first = sorted(THROTTLED & set(clk["reasons"]))
            ms, clk = measure()
            if clk:
                clk["remeasured_after"] = first
        ms_per_step = ranks.max(ms) / n
        info = sc._info()
        K = sc.K
        ab = alg_bytes(N, W, K)["step"]
        gbs = ab / (ms_per_step * 1e-3) / 1e9
        row = {"workload": wl.name, "density": density, "N": N, "W": W, "chunk": wl.chunk,
               "K": K, "steps": n, "ms_per_step": ms_per_step,
               "params_per_s": world * N / (ms_per_step * 1e-3),
               "alg_bytes_per_step": ab, "achieved_gbs": gbs, "frac": gbs / peak,
               "frac_of_8tbs": gbs / NOMINAL_HBM_GBS,
               "select_fallback_chunks": info["select_fallbacks"],
               "steps_run": info["step"],
               "l2": (f"flushed before every timed step ({2 * l2_bytes >> 20} MB written, "
                      f"untimed): {working / 1e6:.0f} MB working set" if flush else
                      f"no flush: {working / 1e9:.1f} GB working set"),
               "clocks": clk}
        del batches, scratch
        return row
    finally:
        sc.close()
        torch.cuda.empty_cache()


def link_copy_gbs(dev, nbytes=1 << 30, reps=3):
    """Copy-engine rates of the host link from page-locked memory, each
    direction alone: (host-to-device GB/s, device-to-host GB/s), best of
    `reps` 1 GiB copies timed with CUDA events."""
    import torch
    h = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    s = torch.cuda.Stream(dev)
    best = [0.0, 0.0]
    for _ in range(reps):
        for j, (dst, src) in enumerate(((d, h), (h, d))):
            torch.cuda.synchronize(dev)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s)
            with torch.cuda.stream(s):
                dst.copy_(src, non_blocking=True)
            b.record(s)
            torch.cuda.synchronize(dev)
            best[j] = max(best[j], nbytes / (a.elapsed_time(b) * 1e-3) / 1e9)
    del h, d
    return best[0], best[1]


def oracle_sample(wl, density, n_chunks: int, steps: int, warm: int = 1, n_batches: int = 2,
                  union_mask: bool = False):
    """Time the oracle (as it stands) on n_chunks whole chunks spread over the
    shards: `warm` untimed steps (step 0 first), then `steps` timed steps,
    over ``n_batches`` gradient batches used in turn (generated before the
    loop).  Returns (params/s, timed seconds, sample params, chunks)."""
    import oracle
    nch = -(-wl.N // wl.chunk)
    ids = np.unique(np.linspace(0, nch - 1, n_chunks).astype(np.int64))
    o = oracle.Oracle.for_workload(wl, density, chunk_ids=ids, union_mask=union_mask)
    o.set(oracle.THETA, synth.cpu().theta0(wl, o.index))
    grads = [np.stack([synth.cpu().grads(wl, w, t, idx=o.index) for w in range(wl.W)])
             for t in range(min(n_batches, warm + steps))]
    for t in range(warm):
        o.step(grads[t % len(grads)])
    t0 = time.perf_counter()
    for t in range(warm, warm + steps):
        o.step(grads[t % len(grads)])
    dt = time.perf_counter() - t0
    return o.n * steps / dt, dt, o.n, ids.size


def cpu_sample_note(wl, density, nc, n, warm, steps, dt) -> str:
    return (f"{nc} whole chunks ({n} params) of {wl.name}, W={wl.W}, density {density}: "
            f"{warm} untimed step(s) (step 0 first), then {steps} timed steps over 2 gradient "
            f"batches, {dt:.1f} s of oracle time; single-threaded C++ oracle on one host core")


def run_reference(args, wl, density):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    n_chunks, _ = baseline_sample_size(wl.N, wl.chunk, wl.W)
    rate, dt, n, nc = oracle_sample(wl, density, n_chunks, args.steps, warm=args.warmup,
                                    union_mask=args.union_mask)
    per_step_ms = dt / args.steps * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": "params/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": per_step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": line_config(wl, density, args, world),
        "cpu_baseline": {"value": rate, "unit": "params/s", "cores": 1, "kind": "oracle",
                         "sample": cpu_sample_note(wl, density, nc, n, args.warmup, args.steps,
                                                   dt)},
        "e2e": {"value": rate, "unit": "params/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def link_duplex_gbs(dev, nbytes=1 << 30, reps=3):
    """Host-link ceiling for state kept in host memory: one page-locked buffer
    copied to the device while another comes back, on two streams at once
    (bytes of both directions / time, best of `reps`)."""
    import torch
    h_in = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    h_out = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d_in = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    d_out = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    best = 0.0
    for _ in range(reps):
        torch.cuda.synchronize(dev)
        a, b, c = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        a.record(s1)
        s2.wait_event(a)
        with torch.cuda.stream(s1):
            d_in.copy_(h_in, non_blocking=True)
        with torch.cuda.stream(s2):
            h_out.copy_(d_out, non_blocking=True)
        c.record(s2)
        s1.wait_event(c)
        b.record(s1)
        torch.cuda.synchronize(dev)
        best = max(best, 2 * nbytes / (a.elapsed_time(b) * 1e-3) / 1e9)
    return best


def run_scape(args, wl, density):
    import torch
    from sparse_communication_distributed_gb300 import THETA, Scape

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ranks = Ranks("nccl" if world > 1 else None, dev)
    barrier = ranks.barrier

    N, W = wl.N, wl.W
    from sparse_communication_distributed_gb300.scape import (CHUNK_PER_TENSOR, RESIDUAL_HOST,
                                                              UNION_MASK)
    flags = ((CHUNK_PER_TENSOR if args.per_tensor else 0) |
             (RESIDUAL_HOST if args.residual_host else 0) | (UNION_MASK if args.union_mask else 0))
    sc = Scape.for_workload(wl, density, flags=flags)
    K = sc.K
    th = torch.empty(N, dtype=torch.float32, device=dev)
    synth.gpu().theta_into(wl, th)
    torch.cuda.synchronize()
    sc.load(THETA, th)
    del th
    n_batches = 2
    batches = []
    for b in range(n_batches):
        bufs = [torch.empty(N, dtype=torch.int16, device=dev) for _ in range(W)]
        for w in range(W):
            synth.gpu().grads_into(wl, w, b, bufs[w])
        batches.append(bufs)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)

    # step 0 (the step-0 mask plus the first step), timed on its own
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    sc.step(batches[0], stream)
    e1.record(stream)
    torch.cuda.synchronize()
    step0_ms = e0.elapsed_time(e1)
    for i in range(1, args.warmup):
        sc.step(batches[i % n_batches], stream)
    torch.cuda.synchronize()

    # A working set that L2 could hold is evicted before every timed step by
    # writing a buffer of twice the L2 size (untimed); larger ones are not.
    l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
    config = line_config(wl, density, args, world)
    flush = needs_l2_flush(working_set_bytes(N, W, config["K"], n_batches), GB300_L2_BYTES)
    scratch = torch.empty(2 * l2_bytes, dtype=torch.uint8, device=dev) if flush else None

    def timed(step_fn, steps):
        return timed_steps(step_fn, steps, stream, scratch)

    def measure():
        clocks = ClockSampler(local)
        clocks.start()
        time.sleep(0.3)
        barrier()
        torch.cuda.synchronize()
        ms = timed(lambda i: sc.step(batches[i % n_batches], stream), args.steps)
        barrier()
        # per-kernel breakdown: the same steps again with events around each phase
        sc.profile(True)
        for i in range(args.steps):
            if flush:
                scratch.fill_(i & 0xFF)
            sc.step(batches[i % n_batches], stream)
        torch.cuda.synchronize()
        phases = sc.profile_read()
        sc.profile(False)
        return ms, phases, clocks.stop()

    ms, phases, clk = measure()
    if clk and THROTTLED & set(clk["reasons"]):
        # a run the GPU throttled (hardware or thermal slowdown) is not a
        # measurement: take it again once and report the second run
        first = sorted(THROTTLED & set(clk["reasons"]))
        ms, phases, clk = measure()
        if clk:
            clk["remeasured_after"] = first
    if args.union_mask:
        K = sc.K  # the compact count of the last step (it varies with the union's fill-in)

    ms_per_step = ranks.max(ms) / args.steps

    # end to end through the public API: host gradients in, mask out
    e2e = None
    if not args.no_e2e:
        # each step's M_t comes back on a side stream into one of two pinned
        # buffers, while the next step streams its gradients in
        outs = [torch.empty(sc.info["mask_words"], dtype=torch.int32).pin_memory()
                for _ in range(2)]
        read_stream = torch.cuda.Stream(dev)
        e2e_steps = min(args.steps, 5)

        def timed_host_steps(host):
            sc.step_host(host, stream)
            sc.mask_into_async(outs[0], read_stream)
            barrier()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            for i in range(e2e_steps):
                sc.step_host(host, stream)
                sc.mask_into_async(outs[i % 2], read_stream)
            torch.cuda.synchronize()
            return ranks.max(time.perf_counter() - t0)

        # W x N bf16 of page-locked host memory per rank; every rank takes the
        # same branch (the collectives inside the timing must match)
        why = ""
        try:
            pinned = [batches[0][w].cpu().pin_memory() for w in range(W)]
        except RuntimeError as ex:
            pinned, why = None, str(ex).splitlines()[0][:160]
        if ranks.max(0.0 if pinned is not None else 1.0) > 0.0:
            e2e = {"unavailable": "page-locked host gradients could not be allocated on every "
                                  f"rank ({why or 'another rank'})",
                   "h2d_bytes_per_step": W * N * 2}
        else:
            dt = timed_host_steps(pinned)
            h2d_bytes = W * N * 2
            link_h2d, link_d2h = link_copy_gbs(dev)
            got_h2d = h2d_bytes / (dt / e2e_steps) / 1e9
            e2e = {"value": world * N * e2e_steps / dt, "unit": "params/s",
                   "h2d_bytes_per_step": h2d_bytes,
                   "d2h_bytes_per_step": sc.info["mask_words"] * 4,
                   "ms_per_step": dt / e2e_steps * 1e3, "steps": e2e_steps,
                   "host_buffers": "pinned, read in place by the step kernel",
                   "result_read": "scape_mask_async on a side stream, overlapping the next step",
                   "link_h2d_gbs": link_h2d, "link_d2h_gbs": link_d2h,
                   "achieved_h2d_gbs": got_h2d, "frac_of_link": got_h2d / link_h2d,
                   "link_bound_ms": h2d_bytes / (link_h2d * 1e9) * 1e3,
                   "link_note": "link_*: copy-engine rate of 1 GiB page-locked copies in each "
                                "direction alone, measured in this run; the step reads its "
                                "gradients over the link while M_t goes back on a side stream"}
        del pinned
        if args.e2e_pageable and "value" in e2e:
            pageable = [batches[0][w].cpu() for w in range(W)]
            dtp = timed_host_steps(pageable)
            e2e["pageable_staged_ms_per_step"] = dtp / e2e_steps * 1e3
            del pageable
        del outs

    mstats = None
    if args.mask_stats:
        st = sc.mask_stats()
        mstats = {"kept": st["kept"], "overlap_prev_frac": st["overlap_prev"] / st["kept"],
                  "union_global_topk": st["union_global_topk"],
                  "fill_in": st["union_global_topk"] / st["kept"],
                  "step": sc.step_count}

    # the pages' comparator on the same layout and gradients: dense AdamS
    dense = None
    if not args.no_dense:
        from sparse_communication_distributed_gb300.scape import dense_adams_step
        th_d = torch.empty(N, dtype=torch.float32, device=dev)
        synth.gpu().theta_into(wl, th_d)
        m_d = torch.zeros(N, dtype=torch.float32, device=dev)
        v_d = torch.zeros(N, dtype=torch.float32, device=dev)
        hyper = dict(beta1=wl.beta1, beta2=wl.beta2, lr=wl.lr, wd=wl.wd, eps=wl.eps)
        for i in range(args.warmup):
            dense_adams_step(th_d, m_d, v_d, batches[i % n_batches], stream=stream, **hyper)
        barrier()
        torch.cuda.synchronize()
        d_ms = ranks.max(timed(lambda i: dense_adams_step(th_d, m_d, v_d, batches[i % n_batches],
                                                          stream=stream, **hyper),
                               args.steps)) / args.steps
        d_bytes = N * (2 * W + 24)
        dense = {"ms_per_step": d_ms, "params_per_s": world * N / (d_ms * 1e-3),
                 "alg_bytes_per_step": d_bytes, "achieved_gbs": d_bytes / (d_ms * 1e-3) / 1e9,
                 "exchange_bytes_per_worker": {
                     "dense_allreduce_fp32": 4 * N,
                     "scape_sparse_fp32_plus_mask":
                         4 * K + (N // 8 if args.union_mask else N // (8 * W))},
                 "note": "one GPU: both steps' exchanges are emulated in HBM, so this compares "
                         "memory work, not network time"}
        del th_d, m_d, v_d

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n_ch, n_st = baseline_sample_size(N, wl.chunk, W)
        rate, dt, n, nc = oracle_sample(wl, density, n_ch, n_st, warm=1,
                                        union_mask=args.union_mask)
        cpu = {"value": rate, "unit": "params/s", "cores": 1, "kind": "oracle",
               "sample": cpu_sample_note(wl, density, nc, n, 1, n_st, dt)}

    link = None
    if args.residual_host:
        duplex = link_duplex_gbs(dev)
        rb = 8.0 * W * N  # every residual read and written once per step
        link = {"residual_bytes_per_step": rb,
                "achieved_gbs": rb / (ms_per_step * 1e-3) / 1e9,
                "duplex_copy_gbs": duplex,
                "frac": rb / (ms_per_step * 1e-3) / 1e9 / duplex,
                "peak_kind": "measured here: concurrent page-locked copies in both directions"}
    peak, peak_kind = measured_peak()
    fallbacks = sc._info()["select_fallbacks"]
    workloads = None
    variant = (args.per_tensor or args.residual_host or args.union_mask or args.workers is not None
               or args.seed is not None or args.density is not None)
    if not args.no_workloads and not variant and wl.name == synth.BENCH_WORKLOAD:
        # every layout and density, one handle at a time (the headline row is
        # the measurement above)
        sc.close()
        del batches
        torch.cuda.empty_cache()
        workloads = []
        for name, d in SWEEP:
            if name == wl.name and d == density:
                gbs = alg_bytes(N, W, K)["step"] / (ms_per_step * 1e-3) / 1e9
                workloads.append({"workload": name, "density": d, "N": N, "W": W,
                                  "chunk": wl.chunk, "K": K, "steps": args.steps,
                                  "ms_per_step": ms_per_step,
                                  "params_per_s": world * N / (ms_per_step * 1e-3),
                                  "alg_bytes_per_step": alg_bytes(N, W, K)["step"],
                                  "achieved_gbs": gbs, "frac": gbs / peak,
                                  "frac_of_8tbs": gbs / NOMINAL_HBM_GBS,
                                  "select_fallback_chunks": fallbacks,
                                  "l2": "no flush (the line's own measurement)", "clocks": clk,
                                  "headline": True})
                continue
            workloads.append(time_workload(synth.WORKLOADS[name], d, args.steps, args.warmup,
                                           dev, local, ranks, peak))
    if rank != 0:
        ranks.close()
        return
    ab = alg_bytes(N, W, K)
    traffic, traffic_src = ncu_traffic("step_chunks", N, wl.name)
    if args.union_mask:  # the counters were captured on the partitioned kernel
        traffic, traffic_src = None, None
    a_ms, a_n = phases["step"]
    a_launch_ms = a_ms / max(a_n, 1)
    achieved = ab["step"] / (a_launch_ms * 1e-3) / 1e9
    step_gbs = ab["step"] / (ms_per_step * 1e-3) / 1e9
    line = {
        "metric": METRIC,
        "value": world * N / (ms_per_step * 1e-3),
        "unit": "params/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": config,
        "step_hbm": {"alg_bytes_per_step": ab["step"], "achieved_gbs": step_gbs,
                     "frac_of_8tbs": step_gbs / NOMINAL_HBM_GBS,
                     "frac_of_peak": step_gbs / peak, "peak_kind": peak_kind},
        "roofline": {"kernel": "step_chunks", "bound": "hbm", "achieved": achieved,
                     "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic, "traffic_source": traffic_src,
                     "alg_bytes_per_launch": ab["step"], "launch_ms": a_launch_ms,
                     "peak_kind": f"{peak_kind} (hbm_gbs)"},
        "kernels_ms_per_step": {k: v[0] / args.steps for k, v in phases.items() if v[1]},
        "gpu_launches": args.steps * 2,
        "step0_ms": step0_ms,
        "select_fallback_chunks": fallbacks,
        "clocks": clk,
        "e2e": e2e,
        "residual_link": link,
        "dense_adams": dense,
        "mask_stats": mstats,
        "cpu_baseline": cpu,
        "workloads": workloads,
    }
    if args.union_mask:
        line["union_K"] = K  # compact values per worker in the last step (the union's fill-in)
    print(json.dumps(line), flush=True)
    ranks.close()


def main():
    args = parse()
    if args.impl == "scape" and args.warmup < 1:
        raise SystemExit("--warmup must be >= 1 (the first warm-up step is step 0)")
    wl = synth.WORKLOADS[args.workload]
    import dataclasses
    if args.workers is not None:
        wl = dataclasses.replace(wl, W=args.workers)
    if args.seed is not None:
        wl = dataclasses.replace(wl, seed=args.seed)
    density = args.density if args.density is not None else wl.densities[0]
    if args.impl == "reference":
        run_reference(args, wl, density)
    else:
        run_scape(args, wl, density)


if __name__ == "__main__":
    main()
