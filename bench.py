"""Benchmark of the fused partitioned mixed-precision ZeRO Adam step on GB300.

Default workload: the 1.5B-parameter flat vector over N_d = 16 simulated
data-parallel ranks (fp16 gradients scaled by 2^12, dynamic loss scale, Adam
without weight decay, +Inf injected every 50th step so those steps are
skipped).  A step is one call of zero_step_fused: the reduce-scatter sum of
the 16 gradient buffers, unscale, overflow check, Adam on the fp32 master
weights and moments, and the fp16 cast into the flat parameter buffer.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--workload NAME]
With --gpus N > 1 (under torchrun) every GPU runs its own replica of the
workload (the simulated group does not span GPUs): weak scaling, no
collective on the data path.  --impl reference times the CPU oracle on the
host cores instead (rank 0 only).

Prints one JSON line.
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
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused ZeRO Adam step: G params updated/s and achieved HBM GB/s vs GB300 peak"
UNIT = "Gparams/s"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129e6  # GB300 L2


def algorithmic_bytes_per_elem(world: int, clip: bool, staged: bool, micro: int = 1) -> int:
    """Bytes an ideal step moves per padded element: read the N_d half
    gradients, read and write fp32 master/m/v, write the half parameter.
    A clipped step needs a second pass: +8 (stage written and read) or
    +2 N_d (gradients read again).  With gradient accumulation over micro > 1
    micro-steps each micro-step reads the N_d gradients and writes the fp32
    accumulator (all but the first also read it), and the step reads the
    accumulator (twice with clipping) instead of the gradients."""
    if micro > 1:
        return micro * (2 * world + 8) - 4 + 4 + 26 + (4 if clip else 0)
    b = 2 * world + 24 + 2
    if clip:
        b += 8 if staged else 2 * world
    return b


STEP_KERNEL_SOURCES = ("step.cu", "kernels.cuh", "internal.h", "staged.cuh")


def _code_only(data: bytes) -> bytes:
    """C/C++ source without its comments and with runs of whitespace collapsed,
    so that an edit to comments alone keeps the hash."""
    import re
    text = data.decode("utf-8")
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split()).encode()


def kernel_source_hash(read=None) -> str:
    """Hash of the code (comments stripped) of the sources the fused step
    kernel is compiled from."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "zero_partitioned_mixed_step_gb300", "csrc")
    for name in STEP_KERNEL_SOURCES:
        if read is None:
            with open(os.path.join(csrc, name), "rb") as f:
                data = f.read()
        else:
            data = read(name)
        h.update(name.encode() + _code_only(data))
    return h.hexdigest()[:16]


def dominant_kernel(wl) -> str:
    """The kernel that carries a step of the workload, by the library's rule:
    every-rank one-pass steps with the reduction in fp32, device-resident
    state and N_d = 16 run the shared-memory staged kernel; everything else
    runs the register kernel."""
    clip = wl.max_grad_norm > 0
    if wl.micro_steps > 1:
        return "step_kernel (accumulate passes, then the step from the accumulator)"
    if wl.per_bucket and clip:
        return "step_kernel (two passes, each one launch per bucket on two streams, then the commit)"
    if wl.per_bucket:
        base = ("staged_fused_kernel" if wl.rank is None and not wl.half_reduce
                and not wl.offload_state and wl.world == 16 else "step_kernel")
        return base + " (one launch per bucket on two streams, then the commit)"
    if clip:
        return "step_kernel (two passes)"
    if (wl.rank is None and not wl.half_reduce and not wl.offload_state
            and wl.world == 16):
        return "staged_fused_kernel (TMA bulk copies into shared memory, one pass)"
    return "step_kernel (registers, one pass)"


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": FALLBACK_HBM_GBS}, "fallback"


def recorded_traffic(workload: str):
    """dram bytes per launch of the fused kernel from the committed ncu
    summary, valid only while the kernel sources are unchanged."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    want = kernel_source_hash()
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 3 and not line.startswith("#") and parts[0] == workload \
                    and parts[1] == want:
                return float(parts[2])
    return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = None

    def __enter__(self):
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.out.seek(0)
        rows = [r.split(", ") for r in self.out.read().strip().splitlines() if r.strip()]
        os.unlink(self.out.name)
        sm, mx, power = [], [], []
        reasons = set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
                power.append(float(r[3]))
            except (ValueError, IndexError):
                continue
            for name, val in zip(names, r[5:9]):
                if val.strip() == "Active":
                    reasons.add(name)
        loaded = [s for s, p in zip(sm, power) if p > 0.5 * max(power)] if power else sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------- inputs

def lib_cfg(wl):
    import zero_partitioned_mixed_step_gb300 as zs
    return zs.adam_cfg(lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2, eps=wl.eps,
                       weight_decay=wl.weight_decay, adamw=wl.adamw,
                       max_grad_norm=wl.max_grad_norm, dynamic_scale=wl.dynamic_scale)


def make_group(wl, device):
    """Device buffers of the workload, filled by the seeded GPU generator:
    master ~ N(0, 0.02) by flat index, m = v = 0, params = RNE(master), and
    every rank's step-1 gradient ~ N(0, 1e-3) x loss scale, zero in padding."""
    import torch
    import synth
    import zero_partitioned_mixed_step_gb300 as zs

    rank = -1 if wl.rank is None else wl.rank
    z = zs.ZeroStep(wl.numels, wl.world, wl.dtype, lib_cfg(wl), loss_scale=wl.loss_scale,
                    rank=rank, bucket_numel=wl.bucket, grads_are_slices=wl.grads_are_slices,
                    device=device, half_reduce=wl.half_reduce, offload_state=wl.offload_state)
    L = z.layout
    gaps = synth.gaps(z.offsets, wl.numels, L.padded_numel)
    segs = [(0, L.padded_numel)] if rank < 0 else z.segments(rank)

    def fill_by_flat(out, fill):
        pos = 0
        for fs, ln in segs:
            fill(out[pos:pos + ln], fs)
            for a, b in gaps:  # zero the padding that falls inside this range
                lo, hi = max(a, fs), min(b, fs + ln)
                if lo < hi:
                    out[pos + lo - fs:pos + hi - fs].zero_()
            pos += ln

    master0 = z.master[0] if z.master[0].is_cuda else torch.empty(
        z.master[0].numel(), dtype=torch.float32, device=device)
    fill_by_flat(master0, lambda o, fs: synth.gpu_fill_f32(wl.master_key(), fs, o,
                                                           wl.master_sigma))
    if rank < 0:
        synth.gpu_round_half(master0, z.params[0], wl.dtype)
    if master0 is not z.master[0]:  # offloaded state: copy the weights to host memory
        z.master[0].copy_(master0)
        del master0
    hdt = zs.torch_dtype(wl.dtype)
    grads = []
    sigma = wl.grad_sigma * wl.loss_scale
    for q in range(wl.world):
        g = torch.empty(z.grad_numel(), dtype=hdt, device=device)
        if wl.grads_are_slices:
            fill_by_flat(g, lambda o, fs, q=q: synth.gpu_fill_half(wl.grad_key(1, q), fs, o,
                                                                   sigma, wl.dtype))
        else:
            synth.gpu_fill_half(wl.grad_key(1, q), 0, g, sigma, wl.dtype)
            for a, b in gaps:
                g[a:b].zero_()
        grads.append(g)
    torch.cuda.synchronize()
    return z, grads


# --------------------------------------------------------------------------- CPU legs

def oracle_sample(wl, sample_elems: int):
    """The CPU oracle's inputs for a bounded sample of the workload: one
    rank's first ``sample_elems`` owned elements with all N_d gradient
    buffers (seeded like the GPU inputs)."""
    import numpy as np
    import oracle
    import synth

    lay = oracle.layout((sample_elems * wl.world,), wl.world)  # a flat sample, same N_d
    grads = [synth.fill_half(wl.grad_key(1, q), 0, lay.padded, wl.grad_sigma * wl.loss_scale,
                             wl.dtype) for q in range(wl.world)]
    cfg = oracle.AdamCfg(lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2, eps=wl.eps,
                         weight_decay=wl.weight_decay, adamw=wl.adamw,
                         max_grad_norm=wl.max_grad_norm, dynamic_scale=wl.dynamic_scale)
    st = oracle.State(loss_scale=wl.loss_scale)
    w = synth.fill_f32(wl.master_key(), 0, lay.owned, wl.master_sigma)
    bufs = (w, np.zeros_like(w), np.zeros_like(w), np.zeros(lay.padded, np.uint16))

    def step():
        oracle.step(grads, wl.dtype, lay, cfg, st, *bufs, rank=0, openmp=True)
    return step


def sample_elems_for(wl) -> int:
    """About 2^28 gradient values per sample step, at most 2^24 elements."""
    return max(1 << 18, min(1 << 24, (1 << 28) // wl.world))


def oracle_sample_rate(wl, target_s: float = 12.0):
    """cpu_baseline: the oracle (OpenMP build, all host cores) on the bounded
    sample, stepped for about target_s seconds.  Returns (params/s, threads,
    description)."""
    n = sample_elems_for(wl) // 4
    step = oracle_sample(wl, n)
    step()  # warm
    steps = 0
    t0 = time.perf_counter()
    while True:
        step()
        steps += 1
        el = time.perf_counter() - t0
        if el >= target_s:
            break
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    desc = (f"{steps} oracle steps of one rank's first {n} elements with all {wl.world} "
            f"gradient buffers ({wl.world * n * 2 / 1e6:.0f} MB of gradients per step)")
    return n * steps / el, threads, desc


def run_reference(args, wl):
    """--impl reference: the CPU oracle on the host cores, same metric: W
    untimed and K timed steps, each on the bounded sample of the workload."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    n = sample_elems_for(wl)
    step = oracle_sample(wl, n)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    rate = n * args.steps / el
    value = rate / 1e9
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    desc = (f"{args.steps} timed oracle steps (after {args.warmup} untimed) of one rank's first "
            f"{n} elements with all {wl.world} gradient buffers "
            f"({wl.world * n * 2 / 1e6:.0f} MB of gradients per step)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": wl.name, "psi": wl.numel, "world": wl.world,
                   "sample_elems": n},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


# --------------------------------------------------------------------------- GPU leg

def max_over_ranks(x: float) -> float:
    """The largest value of x over the ranks of the process group (x itself
    without one).  The benchmark takes the slowest rank's time."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_ours(args, wl):
    import torch
    import torch.distributed as dist
    import zero_partitioned_mixed_step_gb300 as zs

    world_size = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    distributed = world_size > 1
    if distributed:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)

    z, grads = make_group(wl, device)
    L = z.layout
    inf_bits = 0x7C00 if wl.dtype == zs.F16 else 0x7F80
    stream = torch.cuda.current_stream()

    # Overflow injection (every 50th step of the workload): one element of
    # one rank's gradient is set to +Inf before the step and restored after.
    def injections(step):
        return [(q, i) for q, i in wl.injections(step)
                if (not wl.grads_are_slices) or i < z.grad_numel()]

    saved = {}

    def before(step):
        for q, i in injections(step):
            saved[(q, i)] = grads[q][i:i + 1].clone()
            grads[q][i:i + 1].view(torch.int16).fill_(inf_bits - 65536 if inf_bits > 32767 else inf_bits)

    def after(step):
        for q, i in injections(step):
            grads[q][i:i + 1].copy_(saved.pop((q, i)))

    clip = wl.max_grad_norm > 0
    bpe = algorithmic_bytes_per_elem(wl.world, clip, z.g_stage is not None, wl.micro_steps)
    n_elems = L.padded_numel if wl.rank is None else L.owned_numel
    # A step that moves less than a few L2 sizes could be served from L2 on
    # the next step: then a 256 MB write flushes L2 between timed steps, and
    # the time is the sum of the per-step events (the flush is not counted).
    flush = None
    if n_elems * bpe < 4 * L2_BYTES:
        flush = torch.empty(64 << 20, dtype=torch.float32, device=device)

    micro = wl.micro_steps
    side = [torch.cuda.Stream(device), torch.cuda.Stream(device)] if wl.per_bucket else None
    first_bucket_done = []  # per step: event after the first bucket's launch

    def one_step():
        if micro > 1:  # gradient accumulation: the same buffers stand for every micro-step
            for k in range(micro):
                z.accumulate(grads, k > 0, stream)
            z.step_accumulated(stream)
        elif wl.per_bucket:  # one launch per bucket (per pass), alternating streams, then the commit
            def fork():
                go = torch.cuda.Event()
                go.record(stream)
                for st in side:
                    st.wait_event(go)

            def join():
                for st in side:
                    e = torch.cuda.Event()
                    e.record(st)
                    stream.wait_event(e)

            def buckets(launch):
                fork()
                for b in range(L.num_buckets):
                    launch(b, side[b % 2])
                    if b == 0:  # bucket 0's parameters are final here
                        e = torch.cuda.Event(enable_timing=True)
                        e.record(side[0])
                        bucket0.append(e)
                join()

            bucket0 = []
            if clip:  # first pass on every bucket, the norm, the second pass on every bucket
                buckets(lambda b, st: z.pass1_buckets(grads, b, 1, st))
                z.norm_buckets(stream)
                bucket0.clear()
                buckets(lambda b, st: z.pass2_buckets(grads, b, 1, st))
            else:
                buckets(lambda b, st: z.step_buckets(grads, b, 1, st))
            first_bucket_done.extend(bucket0)
            z.commit(stream)
        else:
            z.step(grads, stream)

    for s in range(1, args.warmup + 1):
        one_step()
    torch.cuda.synchronize()
    first_bucket_done.clear()

    nsteps = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(nsteps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    if distributed:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        t_start.record(stream)
        for s in range(1, nsteps + 1):
            before(s)
            if flush is not None:
                flush.fill_(float(s))
            ev[s - 1][0].record(stream)
            one_step()
            ev[s - 1][1].record(stream)
            after(s)
        t_end.record(stream)
        torch.cuda.synchronize()
    if distributed:
        dist.barrier()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    region_ms = sum(step_ms) if flush is not None else t_start.elapsed_time(t_end)
    total_ms = max_over_ranks(region_ms)
    st = z.read_state()

    # A step that fits in L2 cannot reach the copy bandwidth of a large copy:
    # time torch's device copy of the same bytes (half read, half written)
    # the same way (L2 flushed before each, per-copy events) for context.
    size_copy = None
    if flush is not None:
        half = max(1, n_elems * bpe // 2 // 4)
        src = torch.ones(half, dtype=torch.float32, device=device)
        dst = torch.empty_like(src)
        cev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(nsteps)]
        for k in range(-3, nsteps):
            flush.fill_(float(k))
            if k >= 0:
                cev[k][0].record(stream)
            dst.copy_(src)
            if k >= 0:
                cev[k][1].record(stream)
        torch.cuda.synchronize()
        copy_ms = statistics.median(a.elapsed_time(b) for a, b in cev)
        size_copy = {"bytes": 2 * half * 4, "median_ms": copy_ms,
                     "step_median_ms": statistics.median(step_ms),
                     "gbs": 2 * half * 4 / (copy_ms / 1e3) / 1e9,
                     "note": "torch's device copy of the step's bytes (half read, half "
                             "written), L2 flushed before each like the steps: what a copy "
                             "reaches at this size"}
        del src, dst

    # end to end: the same step through the public API from pinned host buffers
    e2e = run_e2e(z, grads, wl, args)

    if rank != 0:
        if distributed:
            dist.destroy_process_group()
        return
    params_per_step = wl.numel if wl.rank is None else min(L.owned_numel, wl.numel)
    value = params_per_step * nsteps * world_size / (total_ms / 1e3) / 1e9
    kernel_ms = statistics.mean(step_ms)
    achieved = n_elems * bpe / (kernel_ms / 1e3) / 1e9
    peaks, kind = measured_peaks()
    peak = peaks["hbm_gbs"]
    traffic = recorded_traffic(wl.name)
    rate, threads, desc = oracle_sample_rate(wl)
    # the step's last kernel also ends the step: one launch per pass (and the
    # norm's tree kernel between the passes of a clipped step), plus one per
    # accumulated micro-step
    launches_per_step = (3 if clip else 1) + (wl.micro_steps if wl.micro_steps > 1 else 0)
    pipeline = {}
    if wl.per_bucket:
        launches_per_step = (2 * L.num_buckets + 2) if clip else (L.num_buckets + 1)
        firsts = [a.elapsed_time(f) for (a, _), f in zip(ev, first_bucket_done)]
        pipeline = {"pipeline": {"buckets": L.num_buckets, "streams": 2,
                                 "passes": 2 if clip else 1,
                                 "first_bucket_ready_ms": statistics.median(firsts),
                                 "note": "time from the step's start until the first bucket's "
                                         "parameters are final (an all-gather could start)"}}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world_size,
        "steps": nsteps, "warmup": args.warmup, "ms_per_step": total_ms / nsteps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": wl.name, "psi": wl.numel, "padded": L.padded_numel,
                   "world": wl.world, "grad_dtype": "f16" if wl.dtype == zs.F16 else "bf16",
                   "rank_view": wl.rank, "bucket": wl.bucket, "clip": clip,
                   "bytes_per_elem": bpe, "replicas": world_size,
                   "micro_steps": wl.micro_steps,
                   "l2": ("no flush: each step streams %.1f GB (> 129 MB L2)" % (n_elems * bpe / 1e9)
                          if flush is None else
                          "L2 flushed (256 MB write) between timed steps; time = sum of steps"),
                   "skipped_steps": st.skipped},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_kind": f"{kind} hbm_gbs",
                     "kernel": dominant_kernel(wl),
                     "kernel_ms": kernel_ms, "bytes_per_launch": n_elems * bpe},
        "cpu_baseline": {"value": rate / 1e9, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": desc},
        "e2e": e2e,
        "gpu_launches": launches_per_step * nsteps,
        **({"host_link": {"bytes_per_step": n_elems * 24,
                          "gbs": n_elems * 24 / (kernel_ms / 1e3) / 1e9,
                          "note": "master/m/v read and written in Grace memory over NVLink-C2C"}}
           if wl.offload_state else {}),
        **pipeline,
        **({"size_matched_copy": size_copy} if size_copy else {}),
        "clocks": clocks.summary(),
    }
    print(json.dumps(line))
    if distributed:
        dist.destroy_process_group()


def run_e2e(z, grads, wl, args, steps: int = 20):
    """End to end through ZeroStep.step_from_host: every rank's gradient sits
    in page-locked host memory (the library's zero_host_alloc blocks) and the
    step's kernels load it over the host link (zero-copy: every step moves
    the gradients host -> device inside the timed region), then the step
    state is read back to the
    host; each of `steps` steps is timed on its own with the host clock (the
    call returns after the state has reached the host).  The value is the
    median step's rate; min and max of the rate and the link rate of the same
    steps are reported beside it (the host link is shared with the rest of
    the machine and its rate moves from run to run)."""
    import torch
    import zero_partitioned_mixed_step_gb300 as zs
    try:
        host = [zs.host_empty(g.numel(), g.dtype) for g in grads]
    except (RuntimeError, zs.ZeroError) as e:  # not enough pinnable host memory
        return {"value": None, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0,
                "unavailable": f"pinned host buffers: {str(e).splitlines()[0]}"}
    for h, g in zip(host, grads):
        h.copy_(g)
    stream = torch.cuda.current_stream()
    dev = None  # the step's kernels load the gradients straight from host memory
    z.step_from_host(host, dev, stream, wl.micro_steps)  # warm-up
    torch.cuda.synchronize()
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        z.step_from_host(host, dev, stream, wl.micro_steps)
        times.append(time.perf_counter() - t0)
    h2d = sum(g.numel() * g.element_size() for g in grads) * wl.micro_steps
    params = wl.numel if wl.rank is None else min(z.layout.owned_numel, wl.numel)
    del host
    med = statistics.median(times)
    return {"value": params / med / 1e9, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": ctypes.sizeof(zs.StepState), "steps": steps, "stat": "median of per-step rates",
            "min": params / max(times) / 1e9, "max": params / min(times) / 1e9,
            "link_gbs": h2d / med / 1e9, "link_gbs_min": h2d / max(times) / 1e9,
            "link_gbs_max": h2d / min(times) / 1e9,
            "h2d": "the step's kernels load the gradients from page-locked host memory"}


def run_host_overhead(calls: int = 2000):
    """--host-overhead: host time per zero_step_fused call (CPU timer around
    `calls` enqueues, the device nearly idle: each step is small) for three
    group shapes: 16 ranks every rank (131,072 parameters), one rank of 64
    (262,144), 2 ranks (1,048,576).  Prints one JSON line."""
    import torch
    import zero_partitioned_mixed_step_gb300 as zs
    torch.cuda.set_device(0)
    out = {}
    for world, n, rank in ((16, 16 * 8192, -1), (64, 64 * 4096, 0), (2, 1 << 20, -1)):
        z = zs.ZeroStep((n,), world, zs.F16, zs.adam_cfg(), rank=rank)
        grads = [torch.zeros(z.grad_numel(), dtype=torch.float16, device="cuda")
                 for _ in range(world)]
        for _ in range(20):
            z.step(grads)
        torch.cuda.synchronize()
        per = []
        for _ in range(5):
            t0 = time.perf_counter()
            for _ in range(calls):
                z.step(grads)
            per.append((time.perf_counter() - t0) / calls * 1e6)
            torch.cuda.synchronize()
        out[f"world{world}_rank{rank}_n{n}"] = {"us_per_call_median": statistics.median(per),
                                                 "us_per_call_min": min(per)}
    print(json.dumps({"host_overhead": out, "calls": calls,
                      "what": "ZeroStep.step -> zero_step_fused enqueue, ctypes included"}))


def main():
    from synth.workloads import BY_NAME, CFG3
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=CFG3.name, choices=sorted(BY_NAME))
    ap.add_argument("--host-overhead", action="store_true",
                    help="print the host time per step call instead of the benchmark")
    args = ap.parse_args()
    if args.host_overhead:
        run_host_overhead()
        return
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    wl = BY_NAME[args.workload]
    if args.impl == "reference":
        run_reference(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()
