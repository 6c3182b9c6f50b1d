"""Benchmark of the fused attention forward pass (tensorized online softmax) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--all] [--sweep]

One step = one pass of the whole hot path (one fat_attn_fwd call) over the
workload; the default workload is the long-sequence causal shape
B2 H16 N8192 d128 (bf16, X = 128).  Prints ONE JSON line (rank 0).

Metric: attention forward TFLOP/s, FLOPs = 4 B H N^2 d (halved when causal),
and the fraction of the measured dense bf16 tensor peak.  Inputs are seeded
synthetic N(0,1) tensors resident in HBM; L2 is flushed (256 MiB write)
before every timed step; each step is timed with CUDA events on the stream
the kernel is launched on.

--impl reference times the CPU oracle (plain double-precision definition) on
the host cores, each step a bounded sample (one head, 1/8 of its rows).
With N > 1 ranks every rank runs its own replica (weak scaling; attention
heads are independent, there is no data-path collective).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "b2h16n8192d128_causal"
METRIC = "attn fwd TFLOPS on 1 GB300 (bf16/fp8, causal+full) and % of dense tensor peak"
L2_FLUSH_BYTES = 256 << 20

# DRAM bytes (read + write) of one launch of the headline kernel from one
# ncu capture (dram__bytes_read.sum + dram__bytes_write.sum).  The hash guards
# it: the number is reported only while the forward kernel's sources
# (FWD_SOURCES below) hash to the value they had when the capture was taken,
# and as null once they change.
MEASURED_TRAFFIC = {
    "workload": "b2h16n8192d128_causal",
    "variant": "tensor",
    "bytes": 253.138176e6 + 102.671872e6,
    "csrc_sha256": "9938c9f15db6b2df3507a99db0e6901bd26fbadb317190ea241a987e2b269ef4",
}


# the sources that make the forward kernel of the bench line and its launch
FWD_SOURCES = ("fat_attn_api.cu", "fat_fwd_kernel.cuh", "fat_inst_bf16_d128_lvec.cu",
               "fat_launch.cuh", "fat_schedule.h", "sm103_ptx.cuh")


def csrc_sha256() -> str:
    """Hash of the forward kernel's sources (file names and contents)."""
    import hashlib
    d = os.path.join(ROOT, "tensorized_online_softmax_gb300", "csrc")
    h = hashlib.sha256()
    for name in FWD_SOURCES:
        h.update(name.encode())
        with open(os.path.join(d, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def measured_traffic(workload: str, variant: str):
    """Per-launch DRAM traffic if it was captured on these exact kernel sources."""
    t = MEASURED_TRAFFIC
    if t["workload"] == workload and t["variant"] == variant and t["csrc_sha256"] == csrc_sha256():
        return t["bytes"]
    return None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return {"bf16_tflops": float(pk["bf16_tflops"]),
                "bf16_tflops_sustained": float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"])),
                "hbm_gbs": float(pk["hbm_gbs"]), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0,
                "source": "fallback"}


class ClockSampler:
    """Samples nvidia-smi clocks / throttle reasons while the timed region runs."""

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
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
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
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def max_over_ranks(value: float, dist=None, device=None) -> float:
    """Largest value over all ranks (the slowest rank's time); identity at N = 1."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    import torch

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world: int, flops_per_step: float, steps: int, max_total_ms: float) -> float:
    """Every rank runs its own replica of the workload (weak scaling): the
    whole job processes world * steps workloads in the slowest rank's time."""
    return world * flops_per_step * steps / (max_total_ms * 1e-3) / 1e12


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def cpu_oracle_sample(w, inp, budget_s: float = 10.0):
    """Time the oracle as it stands on this host's cores over whole heads of
    the workload until about ``budget_s`` seconds of work have run."""
    import oracle
    from tensorized_online_softmax_gb300 import inputs as gen

    q64, k64, v64 = (gen.widened(inp, n) for n in ("q", "k", "v"))
    flops_head = w.flops / (w.B * w.H)
    done, t_total, heads = 0.0, 0.0, 0
    for b in range(w.B):
        for h in range(w.H):
            qs, ks, vs = (t[b:b + 1, h:h + 1].numpy() for t in (q64, k64, v64))
            t0 = time.perf_counter()
            oracle.attn_fwd(qs, ks, vs, w.causal, w.scale)
            t_total += time.perf_counter() - t0
            done += flops_head
            heads += 1
            if t_total >= budget_s:
                break
        if t_total >= budget_s:
            break
    return {"value": done / t_total / 1e12, "unit": "TFLOP/s", "cores": oracle.available_cores(),
            "kind": "oracle",
            "sample": f"{heads} of {w.B * w.H} heads of {w.name}, all rows, float64 "
                      f"({t_total:.1f} s)"}


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), for the record."""
    import subprocess

    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def run_cpu_all(args):
    """The oracle as it stands, timed on this host's cores on every benchmark
    workload (whole heads until about --cpu-budget seconds of work have run),
    and on one thread for the two smallest; one JSON line per measurement.
    Needs no GPU."""
    import oracle
    from tensorized_online_softmax_gb300 import inputs as gen

    model, cores = cpu_model(), oracle.available_cores()
    names = ["tiny", "b4h16n2048d128", "b4h16n2048d128_causal", DEFAULT_WORKLOAD,
             "stress_b1h32n16384d64", "fp8_b4h16n4096d128"]
    for name in names:
        w = gen.WORKLOADS[name]
        inp = gen.make_inputs(w)
        q64, k64, v64 = (gen.widened(inp, n) for n in ("q", "k", "v"))
        flops_head = w.flops / (w.B * w.H)
        for threads in ([0, 1] if name in ("tiny", "b4h16n2048d128") else [0]):
            done, t_total, heads = 0.0, 0.0, 0
            for bh in range(w.B * w.H):
                b, h = divmod(bh, w.H)
                qs, ks, vs = (t[b:b + 1, h:h + 1].numpy() for t in (q64, k64, v64))
                t0 = time.perf_counter()
                oracle.attn_fwd(qs, ks, vs, w.causal, w.scale, nthreads=threads)
                t_total += time.perf_counter() - t0
                done += flops_head
                heads += 1
                if t_total >= args.cpu_budget:
                    break
            print(json.dumps({
                "cpu_oracle": name, "threads": threads if threads else cores, "cores": cores,
                "cpu_model": model, "value": done / t_total / 1e12, "unit": "TFLOP/s",
                "gflops_per_s": done / t_total / 1e9, "heads": heads, "of_heads": w.B * w.H,
                "seconds": t_total, "seconds_per_head": t_total / heads,
                "dtype": "f64", "kind": "oracle"}), flush=True)


def run_reference(args, w):
    """The CPU oracle as the reference arm (rank 0 only)."""
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    import oracle
    from tensorized_online_softmax_gb300 import inputs as gen

    inp = gen.make_inputs(w)
    q64, k64, v64 = (gen.widened(inp, n) for n in ("q", "k", "v"))
    per_step, flops = [], 0.0
    for step in range(args.warmup + args.steps):
        b, h = step % w.B, (step // w.B) % w.H
        r0 = step % 8
        qs, ks, vs = (t[b:b + 1, h:h + 1].numpy() for t in (q64, k64, v64))
        rows = range(r0, w.N, 8)
        step_flops = sum(4.0 * w.d * ((r + 1) if w.causal else w.N) for r in rows)
        t0 = time.perf_counter()
        oracle.attn_fwd(qs, ks, vs, w.causal, w.scale, rows=slice(r0, w.N, 8))
        dt = time.perf_counter() - t0
        if step >= args.warmup:
            per_step.append(dt)
            flops += step_flops
    total = sum(per_step)
    value = flops / total / 1e12
    cores = oracle.available_cores()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / len(per_step), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(w, "oracle", l2="n/a (host cores)"),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step: 1/8 of the rows of one head of {w.name}"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def phase_trace(fat, torch, w, dev, variant, l_mode, stream, sm_mhz, peak_tflops):
    """One traced launch: per-iteration clock stamps of the first thread block.

    Returns the median steady-state iteration period (one K/V tile against
    the block's 128 query rows), the median softmax time per K/V tile (S
    received -> P published, by the set of softmax warps that takes it), and the
    vector-interval ratio: the share of an iteration in which the tensor pipe
    has no work because it waits for the softmax, estimated as
    1 - (ideal tensor cycles of the iteration) / (measured period), with the
    ideal cycles from the measured dense peak at the sampled SM clock.
    """
    import numpy as np

    I = fat.TRACE_ITERS
    tr = torch.zeros(fat.TRACE_WORDS, dtype=torch.int64, device=dev["q"].device)
    with torch.cuda.stream(stream):
        fat.attn_fwd(dev["q"], dev["k"], dev["v"], w.causal, w.scale, w.X, variant=variant,
                     l_mode=l_mode, stream=stream, trace=tr)
    stream.synchronize()
    t = tr.cpu().numpy().astype(np.int64)
    ev = t[:10 * I].reshape(5, 2, I)
    n = int((ev[3, 0] > 0).sum())
    if n < 12:
        return None
    mid = slice(4, n - 3)
    period = float(np.median(np.diff(ev[3, 0])[mid]))
    # the two softmax sets take alternate K/V tiles (set t the tiles j = t mod 2)
    soft = np.concatenate([(ev[2, t] - ev[0, t])[t:n:2][2:-2] for t in (0, 1)])
    softmax = float(np.median(soft))
    out = {"period_cycles": period, "softmax_cycles": softmax, "iterations": n}
    if sm_mhz:
        n_sm = torch.cuda.get_device_properties(dev["q"].device).multi_processor_count
        flop_per_clk = peak_tflops * 1e12 / (n_sm * sm_mhz * 1e6)
        ideal = 4.0 * 128 * 128 * w.d / flop_per_clk  # PV + S of one 128-row tile
        out["ideal_tensor_cycles"] = ideal
        out["vector_interval_ratio"] = max(0.0, 1.0 - ideal / period)
    # the same at the nominal dense bf16 rate of one SM, 8192 flop per cycle
    # (one 128 x 128 x 16 tcgen05 MMA per 64 cycles)
    out["nominal_tensor_cycles"] = 4.0 * 128 * 128 * w.d / 8192
    return out


def config_dict(w, variant, l2="flushed before every timed step (256 MiB write)"):
    return {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
            "X": w.X, "dtype": w.dtype, "variant": variant, "l2": l2}


def time_variant(fat, torch, w, dev, args, variant, flush, stream, l_mode="vector",
                 z_mode="vector"):
    """Device time (ms) of each of args.steps launches, L2 flushed before each."""
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    out = (torch.empty((w.B, w.H, w.N, w.d), dtype=torch.float32, device=dev["q"].device),
           torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev["q"].device))

    def call():
        if w.dtype == "e4m3":
            fat.attn_fwd_fp8(dev["q"], dev["k"], dev["v"], dev["q_descale"], dev["k_descale"],
                             dev["v_descale"], w.causal, w.scale, w.X, out=out, stream=stream)
        else:
            fat.attn_fwd(dev["q"], dev["k"], dev["v"], w.causal, w.scale, w.X, variant=variant,
                         out=out, stream=stream, l_mode=l_mode, z_mode=z_mode)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush.zero_()
            call()
        stream.synchronize()
        yield "start"
        for i in range(args.steps):
            flush.zero_()
            starts[i].record(stream)
            call()
            ends[i].record(stream)
        stream.synchronize()
    yield [s.elapsed_time(e) for s, e in zip(starts, ends)]


def paired_times(fat, torch, w, dev, arms, pairs, flush, stream):
    """Device times (ms) of `pairs` launches of each arm, interleaved launch by
    launch (arm 0, arm 1, ..., then again) so that clock drift and box-to-box
    differences cancel in the ratios; L2 flushed before each launch.  arms:
    list of (variant, l_mode)."""
    out = (torch.empty((w.B, w.H, w.N, w.d), dtype=torch.float32, device=dev["q"].device),
           torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev["q"].device))
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(pairs)] for _ in arms]
    with torch.cuda.stream(stream):
        for i in range(pairs + 3):
            for a, (variant, l_mode) in enumerate(arms):
                flush.zero_()
                if i >= 3:
                    ev[a][i - 3][0].record(stream)
                fat.attn_fwd(dev["q"], dev["k"], dev["v"], w.causal, w.scale, w.X,
                             variant=variant, l_mode=l_mode, out=out, stream=stream)
                if i >= 3:
                    ev[a][i - 3][1].record(stream)
        stream.synchronize()
    return [[s.elapsed_time(e) for s, e in arm] for arm in ev]


def other_configs(fat, torch, device, flush, stream, steps, peaks):
    """The other workloads of the benchmark's config list, tensorized and vec
    launches interleaved (`steps` of each, L2 flushed before each): TFLOP/s,
    fraction of the dense peak (fp8: 2x bf16, the nominal ratio) and the
    tensorized / vec ratio, with the clocks of the whole measurement."""
    from tensorized_online_softmax_gb300 import inputs as gen

    names = ("b4h16n2048d128", "b4h16n2048d128_causal", "stress_b1h32n16384d64",
             "fp8_b4h16n4096d128")
    sampler = ClockSampler(device.index or 0)
    sampler.start()
    out = {}
    for name in names:
        w = gen.WORKLOADS[name]
        inp = gen.make_inputs(w)
        q, k, v = (inp[n].to(device) for n in ("q", "k", "v"))
        o = torch.empty((w.B, w.H, w.N, w.d), dtype=torch.float32, device=device)
        lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=device)
        kw = {}
        if w.dtype == "e4m3":
            kw = dict(dtype="e4m3", descales=(inp["q_descale"], inp["k_descale"], inp["v_descale"]))
        ts = {"tensor": [], "vec": []}
        with torch.cuda.stream(stream):
            for i in range(steps + 3):
                for variant in ("tensor", "vec"):
                    flush.zero_()
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    fat.attn_fwd(q, k, v, w.causal, w.scale, w.X, variant=variant, out=(o, lse),
                                 stream=stream, **kw)
                    e1.record(stream)
                    if i >= 3:
                        ts[variant].append((e0, e1))
            stream.synchronize()
        ms = {a: statistics.median(s_.elapsed_time(e_) for s_, e_ in ts[a]) for a in ts}
        peak = peaks["bf16_tflops"] * (2.0 if w.dtype == "e4m3" else 1.0)
        out[name] = {"dtype": w.dtype, "causal": w.causal, "X": w.X,
                     "tensor_tflops": w.flops / ms["tensor"] / 1e9,
                     "vec_tflops": w.flops / ms["vec"] / 1e9,
                     "tensor_ms": ms["tensor"], "vec_ms": ms["vec"],
                     "frac_tensor": w.flops / ms["tensor"] / 1e9 / peak,
                     "tensor_speedup_vs_vec": ms["vec"] / ms["tensor"]}
    out["clocks"] = sampler.stop()
    out["steps_per_arm"] = steps
    return out


def sustained_run(fat, torch, w, dev, flush, stream, gpu_index, seconds=2.0, est_ms=1.0):
    """The timed step (L2 flush + launch) back to back for about `seconds`, with
    nvidia-smi sampling the clocks throughout (tens of samples, where the
    timed region of a few steps gets one): TFLOP/s over that run, the clock
    record, and device time x median SM clock per step."""
    n = max(20, int(seconds * 1e3 / max(est_ms, 1e-3)))
    out = (torch.empty((w.B, w.H, w.N, w.d), dtype=torch.float32, device=dev["q"].device),
           torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev["q"].device))
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    sampler = ClockSampler(gpu_index)
    sampler.start()
    time.sleep(0.3)  # the sampler's first line
    with torch.cuda.stream(stream):
        for i in range(n):
            flush.zero_()
            starts[i].record(stream)
            fat.attn_fwd(dev["q"], dev["k"], dev["v"], w.causal, w.scale, w.X, out=out,
                         stream=stream)
            ends[i].record(stream)
        stream.synchronize()
    clocks = sampler.stop()
    ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    avg = sum(ms) / n
    res = {"steps": n, "ms_per_step": avg, "value": w.flops / (avg * 1e-3) / 1e12,
           "unit": "TFLOP/s", "clocks": clocks}
    if clocks.get("sm_mhz"):
        res["kcycles_per_step_at_median_mhz"] = avg * 1e-3 * clocks["sm_mhz"] * 1e6 / 1e3
    return res


DECODE_SHAPES = ((8, 32, 1, 16384, 128), (4, 32, 16, 32768, 128))  # B, H, Nq, Nk, d


def decode_lines(fat, torch, device, timeit, peaks, steps):
    """Split-KV decode shapes, one JSON line each, with their HBM roofline (K
    and V read once: 2 * B * H * Nk * d * 2 bytes): per call back to back
    (ms, frac_hbm) and with an L2 flush before each (ms_flushed)."""
    for B, H, Nq, Nk, d in DECODE_SHAPES:
        g = torch.Generator().manual_seed(2000 + Nq)
        q = torch.randn((B, H, Nq, d), generator=g).to(torch.bfloat16).to(device)
        k = torch.randn((B, H, Nk, d), generator=g).to(torch.bfloat16).to(device)
        v = torch.randn((B, H, Nk, d), generator=g).to(torch.bfloat16).to(device)
        splits = fat.load_library().fat_attn_splitkv_default_splits(B, H, Nq, Nk)
        ws = torch.empty(fat.load_library().fat_attn_splitkv_workspace_bytes(B, H, Nq, d, splits),
                         dtype=torch.uint8, device=device)
        out = (torch.empty((B, H, Nq, d), dtype=torch.float32, device=device),
               torch.empty((B, H, Nq), dtype=torch.float32, device=device))

        def call():
            fat.attn_fwd_splitkv(q, k, v, False, None, 128, splits, workspace=ws, out=out)

        # L2 flushed before each call
        ms_flushed = timeit(call, steps)
        # calls back to back as a serving loop issues them (K and V, 2-4 GB,
        # are far larger than L2, so nothing carries over between calls)
        e0, e1 = torch.cuda.Event(True), torch.cuda.Event(True)
        call()
        e0.record()
        for _ in range(steps):
            call()
        e1.record()
        e1.synchronize()
        ms = e0.elapsed_time(e1) / steps
        kv_bytes = 2.0 * B * H * Nk * d * 2
        print(json.dumps({"workload": f"decode_b{B}h{H}q{Nq}k{Nk}d{d}", "splits": splits,
                          "ms": ms, "ms_flushed": ms_flushed,
                          "tflops": 4.0 * B * H * Nq * Nk * d / ms / 1e9,
                          "hbm_gbs": kv_bytes / ms / 1e6, "hbm_peak_gbs": peaks["hbm_gbs"],
                          "frac_hbm": kv_bytes / ms / 1e6 / peaks["hbm_gbs"],
                          "frac_hbm_flushed": kv_bytes / ms_flushed / 1e6 / peaks["hbm_gbs"]}),
              flush=True)


def run_decode(args):
    """Only the split-KV decode lines of --all."""
    import torch

    import tensorized_online_softmax_gb300 as fat

    device = torch.device("cuda", 0)
    decode_lines(fat, torch, device, event_timer(torch, device), load_peaks(),
                 max(1, min(args.steps, 100)))


def run_all(args):
    """One JSON line per workload (results tables): both softmax variants for
    bf16, the tensorized one for e4m3, the split-KV decode shapes
    (decode_lines) and the backward pass."""
    import torch

    import tensorized_online_softmax_gb300 as fat
    from tensorized_online_softmax_gb300 import inputs as gen

    device = torch.device("cuda", 0)
    peaks = load_peaks()
    timeit = event_timer(torch, device)
    steps = max(10, min(args.steps, 100))
    for name, w in gen.WORKLOADS.items():
        if name == "tiny":
            continue
        inp = gen.make_inputs(w)
        q, k, v = (inp[n].to(device) for n in ("q", "k", "v"))
        out = (torch.empty((w.B, w.H, w.N, w.d), dtype=torch.float32, device=device),
               torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=device))
        kw = {}
        if w.dtype == "e4m3":
            kw = dict(dtype="e4m3", descales=(inp["q_descale"], inp["k_descale"], inp["v_descale"]))
        arms = {}
        sampler = ClockSampler(0)
        sampler.start()
        for variant in ("tensor", "vec"):
            ms = timeit(lambda: fat.attn_fwd(q, k, v, w.causal, w.scale, w.X, variant=variant,
                                             out=out, **kw), steps)
            arms[variant] = {"ms": ms, "tflops": w.flops / ms / 1e9}
        clocks = sampler.stop()
        peak = peaks["bf16_tflops"] * (2.0 if w.dtype == "e4m3" else 1.0)
        print(json.dumps({"workload": name, "dtype": w.dtype, "causal": w.causal, "X": w.X,
                          "arms": arms, "peak_tflops": peak,
                          "peak_source": peaks["source"] + (" bf16 x 2 (fp8 nominal ratio)"
                                                            if w.dtype == "e4m3" else " bf16"),
                          "frac_tensor": arms["tensor"]["tflops"] / peak,
                          "tensor_speedup_vs_vec": arms["vec"]["ms"] / arms["tensor"]["ms"],
                          "clocks": clocks}), flush=True)
    decode_lines(fat, torch, device, timeit, peaks, steps)
    run_bwd(args, BWD_WORKLOADS, steps)


def event_timer(torch, device):
    """fn, steps -> median device time (ms) of fn over `steps` calls, each
    preceded by an L2 flush, after 3 untimed calls.  The calls are queued
    without waiting for each other, so the host's time per call overlaps the
    device's work as in the benchmark line."""
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)

    def timeit(fn, steps):
        for _ in range(3):
            flush.zero_()
            fn()
        ev = [(torch.cuda.Event(True), torch.cuda.Event(True)) for _ in range(steps)]
        for s0, s1 in ev:
            flush.zero_()
            s0.record()
            fn()
            s1.record()
        ev[-1][1].synchronize()
        return statistics.median(s0.elapsed_time(s1) for s0, s1 in ev)

    return timeit


BWD_WORKLOADS = ("b4h16n2048d128", "b4h16n2048d128_causal", "b2h16n8192d128_causal",
                 "stress_b1h32n16384d64")


def run_bwd(args, names, steps):
    """Backward pass on the shapes of bf16 workloads (dout ~ N(0, 1)), one
    JSON line each: five GEMMs of 2 N^2 d FLOPs per head (S, dP, dV, dK, dQ;
    halved causal), i.e. 2.5x the forward's; the time includes the D / LSE
    preparation and the clearing of dq."""
    import torch

    import tensorized_online_softmax_gb300 as fat
    from tensorized_online_softmax_gb300 import inputs as gen

    device = torch.device("cuda", 0)
    peaks = load_peaks()
    timeit = event_timer(torch, device)
    for name in names:
        w = gen.WORKLOADS[name]
        inp = gen.make_inputs(w)
        q, k, v = (inp[n].to(device) for n in ("q", "k", "v"))
        g = torch.Generator().manual_seed(77)
        do = torch.randn(q.shape, generator=g).to(torch.bfloat16).to(device)
        o, lse = fat.attn_fwd(q, k, v, w.causal, w.scale, w.X)
        ws = torch.empty(fat.load_library().fat_attn_bwd_workspace_bytes(w.B, w.H, w.N),
                         dtype=torch.uint8, device=device)
        grads = tuple(torch.empty(q.shape, dtype=torch.float32, device=device) for _ in range(3))
        ms = timeit(lambda: fat.attn_bwd(q, k, v, o, lse, do, w.causal, w.scale, workspace=ws,
                                         out=grads), steps)
        if fat.check_device_error() != fat.FAT_OK:
            raise SystemExit("device error word set during the backward run")
        flops = 2.5 * w.flops
        print(json.dumps({"workload": name + "_bwd", "ms": ms, "tflops": flops / ms / 1e9,
                          "peak_tflops": peaks["bf16_tflops"],
                          "frac_tensor": flops / ms / 1e9 / peaks["bf16_tflops"]}),
              flush=True)


def run_sweep(args):
    """The pages' sweep (FA-T summary A4, Fig. 8): 16384 tokens (B * N) and
    hidden size 2048 (H * d), N in 512 .. 8192, d in {64, 128}, causal and
    non-causal, FP16-FP32 and FP8-FP32 (e4m3 with d = 128), both softmax
    variants; one JSON line per shape (a Fig.-8-style table)."""
    import torch

    import tensorized_online_softmax_gb300 as fat
    from tensorized_online_softmax_gb300 import inputs as gen

    device = torch.device("cuda", 0)
    peaks = load_peaks()
    steps = max(5, min(args.steps, 30))
    timer = event_timer(torch, device)

    def timeit(fn):
        return timer(fn, steps)

    for dtype in ("fp16", "e4m3"):
        for d in (64, 128):
            if dtype == "e4m3" and d != 128:
                continue
            for N in (512, 1024, 2048, 4096, 8192):
                for causal in (False, True):
                    B, H = 16384 // N, 2048 // d
                    w = gen.Workload(f"sweep_{dtype}_n{N}_d{d}", B, H, N, d, causal, 128,
                                     dtype=dtype, seed=3000 + N + d)
                    inp = gen.make_inputs(w)
                    q, k, v = (inp[n].to(device) for n in ("q", "k", "v"))
                    kw = {"dtype": dtype}
                    if dtype == "e4m3":
                        kw["descales"] = (inp["q_descale"], inp["k_descale"], inp["v_descale"])
                    arms = {}
                    for variant in ("tensor", "vec"):
                        ms = timeit(lambda: fat.attn_fwd(q, k, v, causal, w.scale, w.X,
                                                         variant=variant, **kw))
                        arms[variant] = {"ms": ms, "tflops": w.flops / ms / 1e9}
                    peak = peaks["bf16_tflops"] * (2.0 if dtype == "e4m3" else 1.0)
                    print(json.dumps({
                        "sweep": "tokens16384_hidden2048", "dtype": dtype, "B": B, "H": H, "N": N,
                        "d": d, "causal": causal, "X": w.X, "arms": arms,
                        "tensor_speedup_vs_vec": arms["vec"]["ms"] / arms["tensor"]["ms"],
                        "peak_tflops": peak, "frac_tensor": arms["tensor"]["tflops"] / peak}),
                        flush=True)
                    del q, k, v, inp


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-ablation", action="store_true", help="skip timing the vec variant")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--pairs", type=int, default=200,
                    help="interleaved tensorized / vec launches of each arm for the ablation ratio")
    ap.add_argument("--sustain-s", type=float, default=2.0,
                    help="seconds of back-to-back steps with the clocks sampled (0: skip)")
    ap.add_argument("--other-steps", type=int, default=20,
                    help="launches per arm of each other workload in the line (0: skip)")
    ap.add_argument("--all", action="store_true",
                    help="one line per workload (results tables) instead of the benchmark line")
    ap.add_argument("--sweep", action="store_true",
                    help="the pages' fp16 / fp8 sweep, one line per shape")
    ap.add_argument("--bwd", action="store_true",
                    help="time the backward pass on --workload (bf16) only, one line")
    ap.add_argument("--decode", action="store_true",
                    help="only the split-KV decode lines of --all")
    ap.add_argument("--cpu-all", action="store_true",
                    help="time the CPU oracle on every workload (no GPU), one line each")
    ap.add_argument("--cpu-budget", type=float, default=5.0,
                    help="seconds of oracle work per --cpu-all line")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.cpu_all:
        run_cpu_all(args)
        return
    if args.bwd:
        run_bwd(args, [args.workload], max(1, args.steps))
        return
    if args.sweep:
        run_sweep(args)
        return
    if args.all:
        run_all(args)
        return
    if args.decode:
        run_decode(args)
        return

    from tensorized_online_softmax_gb300 import inputs as gen

    w = gen.WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
        return

    import torch

    import tensorized_online_softmax_gb300 as fat

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=device)
        pg = dist

    inp = gen.make_inputs(w)
    dev = {k: (v.to(device) if isinstance(v, torch.Tensor) and k in ("q", "k", "v") else v)
           for k, v in inp.items()}
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.Stream(device)
    peaks = load_peaks()

    def timed(variant, sample_clocks, l_mode="vector", z_mode="vector"):
        gen_ = time_variant(fat, torch, w, dev, args, variant, flush, stream, l_mode, z_mode)
        next(gen_)  # warm-up done
        if pg:
            pg.barrier()
        torch.cuda.synchronize(device)
        sampler = ClockSampler(local) if sample_clocks else None
        if sampler:
            sampler.start()
        t0 = time.perf_counter()
        times = next(gen_)
        torch.cuda.synchronize(device)
        wall = time.perf_counter() - t0
        if pg:
            pg.barrier()
        clocks = sampler.stop() if sampler else None
        return times, wall, clocks

    times, wall, clocks = timed("tensor", True)
    if fat.check_device_error(stream) != fat.FAT_OK:
        raise SystemExit("device error word set during the timed run")
    total_ms = max_over_ranks(sum(times), pg, device)
    value = whole_job_tflops(world, w.flops, args.steps, total_ms)
    avg_ms = total_ms / args.steps
    achieved = w.flops / (avg_ms * 1e-3) / 1e12

    ablation = None
    if not args.no_ablation and w.dtype == "bf16":
        # tensorized against the vector softmax: launches interleaved pair by
        # pair, at least 200 of each
        pairs = max(args.pairs, args.steps)
        pt, pv = paired_times(fat, torch, w, dev, [("tensor", "vector"), ("vec", "vector")],
                              pairs, flush, stream)
        t_avg, v_avg = sum(pt) / pairs, sum(pv) / pairs
        ratios = sorted(b / a for a, b in zip(pt, pv))
        lt, _, _ = timed("tensor", False, "tensor")
        l_avg = sum(lt) / len(lt)
        ablation = {"pairs": pairs,
                    "tensor_value_paired": w.flops / (t_avg * 1e-3) / 1e12,
                    "vec_value": w.flops / (v_avg * 1e-3) / 1e12, "vec_ms_per_step": v_avg,
                    "tensor_speedup_vs_vec": v_avg / t_avg,
                    "tensor_speedup_vs_vec_p10_p50_p90": [
                        ratios[len(ratios) // 10], ratios[len(ratios) // 2],
                        ratios[(9 * len(ratios)) // 10]],
                    "tensor_lsum_value": w.flops / (l_avg * 1e-3) / 1e12,
                    "tensor_lsum_ms_per_step": l_avg}
        if w.X == 128:
            # the subtraction of Z on the tensor pipe, alone and together with
            # the tensor row sum (the pages' "AllTensor" arm); FLOPs counted
            # as for the other arms (the extra bias K step is not counted)
            zt, _, _ = timed("tensor", False, "vector", "tensor")
            at, _, _ = timed("tensor", False, "tensor", "tensor")
            z_avg = sum(zt) / len(zt)
            a_avg = sum(at) / len(at)
            ablation.update({"tensor_zmma_value": w.flops / (z_avg * 1e-3) / 1e12,
                             "tensor_zmma_ms_per_step": z_avg,
                             "alltensor_value": w.flops / (a_avg * 1e-3) / 1e12,
                             "alltensor_ms_per_step": a_avg})

    # end to end through the C ABI with host buffers (fat_attn_fwd_host): every
    # step copies q, k, v from page-locked host memory, runs the kernel and
    # copies o and lse back, chunk by chunk with the copies overlapping the
    # kernels; each step starts after the previous one has ended
    e2e = None
    if args.e2e_steps > 0 and w.dtype == "bf16":
        host = {n: inp[n].pin_memory() for n in ("q", "k", "v")}
        o_host = torch.empty((w.B, w.H, w.N, w.d), dtype=torch.float32).pin_memory()
        l_host = torch.empty((w.B, w.H, w.N), dtype=torch.float32).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = o_host.numel() * 4 + l_host.numel() * 4
        ws = torch.empty(fat.load_library().fat_attn_fwd_host_workspace_bytes(
            w.B, w.H, w.N, w.d, 0), dtype=torch.uint8, device=device)
        with torch.cuda.stream(stream):
            e_s = torch.cuda.Event(enable_timing=True)
            e_e = torch.cuda.Event(enable_timing=True)
            for i in range(2 + args.e2e_steps):
                if i == 2:
                    stream.synchronize()
                    e_s.record(stream)
                fat.attn_fwd_host(host["q"], host["k"], host["v"], w.causal, w.scale, w.X,
                                  out=(o_host, l_host), workspace=ws, stream=stream)
            e_e.record(stream)
            stream.synchronize()
        e2e_ms = e_s.elapsed_time(e_e) / args.e2e_steps
        e2e = {"value": w.flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms}

    sustained = None
    if rank == 0 and w.dtype == "bf16" and args.sustain_s > 0:
        sustained = sustained_run(fat, torch, w, dev, flush, stream, local, args.sustain_s,
                                  est_ms=avg_ms + 0.05)

    others = None
    if rank == 0 and args.other_steps > 0 and args.workload == DEFAULT_WORKLOAD:
        others = other_configs(fat, torch, device, flush, stream, args.other_steps, peaks)

    traces = None
    if w.dtype == "bf16" and w.N >= 2048:
        mhz = ((sustained or {}).get("clocks") or {}).get("sm_mhz") or (clocks or {}).get("sm_mhz")
        traces = {"tensor": phase_trace(fat, torch, w, dev, "tensor", "vector", stream, mhz,
                                        peaks["bf16_tflops"]),
                  "vec": phase_trace(fat, torch, w, dev, "vec", "vector", stream, mhz,
                                     peaks["bf16_tflops"])}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_oracle_sample(w, inp)

    if rank == 0:
        peak = peaks["bf16_tflops"]
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": avg_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.dtype, "data": "synthetic", "config": config_dict(w, "tensor"),
            "pct_of_peak": 100.0 * achieved / peak,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak,
                         "unit": "TFLOP/s", "frac": achieved / peak,
                         "traffic": measured_traffic(w.name, "tensor"),
                         "peak_source": f"{peaks['source']} bf16 dense (burst)"},
            "ablation": ablation, "phase_trace": traces, "e2e": e2e, "cpu_baseline": cpu,
            "gpu_launches": args.steps, "clocks": clocks, "sustained": sustained,
            "other_configs": others,
            "wall_s_timed_region": wall,
        }
        print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
