"""Benchmark: bf16 implicit-GEMM conv3d on one GB300 (per layer TFLOP/s and chain ms).

Headline workload (one step = one pass of the whole chain): the 30-call causal
video-VAE encoder tile of the FlyDSL issue's MiniMax-H3 "Shapes" table, N = 1,
17 frames, every call a 3x3x3 convolution with causal temporal zero pad 2 and
reflect spatial pad 1 (conv_in 3->128 at 256^2, 128->128 x4, the strided and
widening calls down to 1024->1024 at 16^2, conv_out 1024->48), NDHWC throughout,
each call reading the previous call's output.  Inputs are seeded synthetic
tensors of those shapes (the real model's activations and weights are not
needed to time the convolutions).

Prints one JSON line.  `value` is chain TFLOP/s (algorithmic FLOP of the 30 calls
/ device time of one chain), the chain's input resident in HBM, L2 flushed
between steps; the step replays the 30 calls recorded once as a CUDA graph
(`ladder_eager` holds the same chain issued call by call).  `e2e` is the same
metric with the chain's input copied in from pinned host memory and its output
copied out inside the timed region.  `layers` holds per-call rows of the ladder
(times inside the eager chain) and of the other workloads (the Wan-like chain, the
fused 160 blocks, the T=1 image-VAE layers, the x2-upsample decoder convolutions,
the ladder's layers with FP8 e4m3 operands), each timed alone after an L2 flush.
`--impl reference` times the CPU oracle on a bounded sample of the ladder.
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
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as wl  # noqa: E402

WORKLOAD_NAME = "ladder"
METRIC = "bf16 conv3d TFLOP/s (chain)"
L2_FLUSH_BYTES = 256 << 20


# DRAM bytes (read + write) of one launch of the dominant kernel, from one ncu
# capture (profiles/), keyed by a hash of the kernel's sources (comments and
# whitespace left out) and the call it was captured on: a changed kernel reports
# null until it is captured again.
KERNEL_SOURCES = ["conv_cm.cu", "conv_cm_kernel.cuh", "conv_cm_halo.cu", "epilogue_cm.cuh",
                  "epilogue.cuh", "kernel_common.cuh",
                  "ptx.cuh", "internal.h"]
NCU_TRAFFIC = {
    # profiles/conv_cm_ladder_L0_halo.md: L0_0 as in the haloed ladder chain
    ("ff151339c2fd4ecf", "L0_0"): 290725376 + 251654144,
}


def source_code_only(text):
    """C++ source text without comments and whitespace (what the compiler sees)."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return "".join(text.split())


def kernel_source_hash(read=None):
    import hashlib
    h = hashlib.sha1()
    d = os.path.join(ROOT, "video_vae_convolution_gb300", "csrc")
    for f in KERNEL_SOURCES:
        if read is None:
            with open(os.path.join(d, f), encoding="utf-8") as fh:
                text = fh.read()
        else:
            text = read(f)
        h.update(source_code_only(text).encode())
    return h.hexdigest()[:16]


def measured_traffic(call_name):
    return NCU_TRAFFIC.get((kernel_source_hash(), call_name))


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


def cpu_info(threads=None):
    """CPU model, logical CPUs (nproc) and the oracle's OpenMP thread count."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if not model:
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    if line.lower().startswith(("model name", "cpu part")):
                        model = line.split(":", 1)[1].strip()
                        break
        except Exception:
            pass
    return {"cpu_model": model or "unknown", "nproc": os.cpu_count(), "omp_threads": threads}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0):
        self.index = index
        self.proc = None
        self.lines = []  # (perf_counter time, csv line)
        self.t0 = self.t1 = None

    def start(self):
        """Starts nvidia-smi and waits (up to 3 s) for its first sample, so that the
        timed region that follows is sampled from its beginning."""
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            deadline = time.perf_counter() + 3.0
            while not self.lines and time.perf_counter() < deadline:
                time.sleep(0.01)
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def begin(self):
        self.t0 = time.perf_counter()

    def end(self):
        self.t1 = time.perf_counter()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        # samples taken inside the timed region (the last one before it when none is)
        lines = [ln for t, ln in self.lines
                 if self.t0 is None or (self.t0 <= t <= (self.t1 or t))]
        if not lines and self.lines:
            before = [ln for t, ln in self.lines if self.t0 is None or t <= self.t0]
            lines = before[-1:] or [self.lines[0][1]]
        for ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_init(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def workload_config(world=1, extra=None):
    cfg = {"workload": "causal VAE encoder ladder, 30 calls chained: conv_in 3->128 "
                       "[1,17,256,256]; 128->128 x4, 128->128 s(1,2,2); 128->256, 256->256 x3 "
                       "@[17,128,128], s(2,2,2); 256->256 x4 @[9,64,64], s(2,2,2); 256->512, "
                       "512->512 x3 @[5,32,32], s(1,2,2); 512->512 x4, 512->1024, "
                       "1024->1024 x3 @[5,16,16]; conv_out 1024->48; 3x3x3, causal T pad "
                       "(2,0) zero + reflect H,W (1,1); NDHWC in and out",
           "calls_per_step": 30, "layout": "NDHWC",
           "intermediates": "each call but the last writes its output inside a tensor with a "
                            "1-pixel reflect border (the next call's spatial padding) and the "
                            "next call applies only the causal T padding; conv_in pads the "
                            "model input itself",
           "l2": "flushed between steps (256 MiB write, untimed); inside a step each call "
                 "reads the previous call's output",
           "inputs": "seeded synthetic: x N(0,1) bf16, weights N(0,1/sqrt(fan_in)) bf16",
           "parallelism": f"replicas x{world}"}
    if extra:
        cfg.update(extra)
    return cfg


def call_class(name):
    """Layer class of a ladder call: its name without the repeat index."""
    base, _, idx = name.rpartition("_")
    return base if idx.isdigit() and base else name


# ---- CPU oracle legs ------------------------------------------------------------------------

def oracle_ladder_rate(target_s=12.0):
    """Times the oracle on sampled output pixels of each layer class of the ladder
    and extrapolates to the whole chain.  Returns (TFLOP/s, extrapolated chain ms,
    threads, sample description)."""
    import oracle
    oracle.build()
    threads = oracle.num_threads(0)
    calls = wl.ladder().calls
    classes = {}
    for c in calls:
        classes.setdefault(call_class(c.name), []).append(c)
    per_class = max(0.2, target_s / len(classes))
    chain_s = 0.0
    pixels = 0
    spent_total = 0.0
    for cls, members in classes.items():
        call = members[0]
        inp = wl.make_inputs("ladder", call, wl.NDHWC)
        xb, wb = wl.bits(inp["x"]), wl.bits(inp["w"])
        Do, Ho, Wo = call.out_dims()
        fpp = 2.0 * call.Cout * call.K  # FLOP per output pixel
        rng = np.random.default_rng(1)
        n = 16
        spent = flops = 0.0
        while spent < per_class:
            pts = np.stack([rng.integers(0, call.N, n), rng.integers(0, Do, n),
                            rng.integers(0, Ho, n), rng.integers(0, Wo, n)], 1)
            t0 = time.perf_counter()
            oracle.conv3d_acc_points(xb, wl.NDHWC, wb, pts, call.stride, call.pads)
            spent += time.perf_counter() - t0
            flops += fpp * n
            pixels += n
            n = min(n * 2, 1 << 16)
        rate = flops / spent  # FLOP/s on this class
        chain_s += sum(c.flops for c in members) / rate
        spent_total += spent
    total = sum(c.flops for c in calls)
    desc = (f"oracle direct conv (fp64 accumulate) on {pixels} sampled output pixels of the "
            f"{len(classes)} ladder layer classes ({spent_total:.1f} s), extrapolated to the "
            f"30-call chain by each class's FLOP")
    return total / chain_s / 1e12, chain_s * 1e3, threads, desc


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    # bounded: the whole run stays within about two minutes of CPU time
    budget = max(1.5, min(10.0, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_ladder_rate(target_s=min(1.5, budget))
    t0 = time.perf_counter()
    rates, chain_ms = [], []
    desc, threads = "", 0
    for _ in range(args.steps):
        r, ms, threads, desc = oracle_ladder_rate(target_s=budget)
        rates.append(r)
        chain_ms.append(ms)
    elapsed = time.perf_counter() - t0
    value = statistics.median(rates)
    info = cpu_info(threads)
    line = {"impl": "reference", "metric": METRIC, "value": value,
            "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": statistics.median(chain_ms),
            "ms_per_step_note": "extrapolated from the oracle's time on sampled output pixels "
                                "(a full chain would take this long)",
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(world),
            "cpu_baseline": dict({"value": value, "unit": "TFLOP/s", "cores": threads,
                                  "kind": "oracle", "sample": desc}, **info),
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "wall_s": elapsed}
    print(json.dumps(line), flush=True)
    return 0


# ---- GPU arm -------------------------------------------------------------------------------

def device_inputs(call, dev, layout, seed):
    """Synthetic inputs of one call drawn on the device (same distributions as the
    workloads module; used for the per-layer rows, where only the timing counts)."""
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    N, C, D, H, W = call.N, call.Cin, call.D, call.H, call.W
    shape = (N, C, D, H, W) if layout == wl.NCDHW else (N, D, H, W, C)
    x = torch.randn(shape, generator=g, device=dev).to(torch.bfloat16)
    kt, kr, ks = call.kernel
    w = (torch.randn((call.Cout, C, kt, kr, ks), generator=g, device=dev) /
         float(np.sqrt(C * kt * kr * ks))).to(torch.bfloat16)
    Do, Ho, Wo = call.out_dims()
    out = {"x": x, "w": w, "bias": None, "residual": None, "residual_bias": None, "gamma": None}
    if call.epi & wl.EPI_BIAS:
        out["bias"] = 0.1 * torch.randn(call.Cout, generator=g, device=dev)
    if call.epi & wl.EPI_RESIDUAL:
        rs = (N, call.Cout, Do, Ho, Wo) if layout == wl.NCDHW else (N, Do, Ho, Wo, call.Cout)
        out["residual"] = torch.randn(rs, generator=g, device=dev).to(torch.bfloat16)
    if call.epi & wl.EPI_RESIDUAL_BIAS:
        out["residual_bias"] = 0.1 * torch.randn(call.Cout, generator=g, device=dev)
    if call.epi & wl.EPI_L2NORM_SILU:
        out["gamma"] = (1 + 0.1 * torch.randn(call.Cout, generator=g, device=dev)).to(
            torch.bfloat16).float()
    return out


# HBM bandwidth the targets are written against (nominal; the measured copy rate is the
# roofline denominator)
HBM_NOMINAL_GBS = 8000.0


def layer_row(call, ms, pk, launches, layout, workload, extra=None):
    tf = call.flops / (ms * 1e-3) / 1e12
    gbs = call.bytes() / (ms * 1e-3) / 1e9
    row = {"workload": workload, "name": call.name,
           "layout": "NCDHW" if layout == wl.NCDHW else "NDHWC",
           "cin": call.Cin, "cout": call.Cout, "kernel": list(call.kernel),
           "stride": list(call.stride), "ms": round(ms, 4), "tflops": round(tf, 1),
           "frac_bf16": round(tf / pk["bf16_tflops"], 3),
           "frac_bf16_sustained": round(tf / pk["bf16_tflops_sustained"], 3),
           "gbs": round(gbs, 1), "frac_hbm": round(gbs / pk["hbm_gbs"], 3),
           "frac_hbm_nominal": round(gbs / HBM_NOMINAL_GBS, 3), "launches": launches}
    if extra:
        row.update(extra)
    return row


def time_alone(c, stream, flush, reps, warm=2):
    """Median device time of one call, L2 flushed before each launch."""
    for _ in range(warm):
        flush.zero_()
        c(stream)
    ts = []
    for _ in range(reps):
        flush.zero_()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        rc = c.run(stream)
        b.record(stream)
        if rc != 0:
            raise RuntimeError(f"conv3d_fwd failed: {rc}")
        ts.append((a, b))
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in ts)


# streaming causal convolution (cuDNN frontend doc, "Causal Conv3D with Cache"): one
# 4-frame NCTHW chunk of the 12-channel (2x2 patchified RGB) input after two history
# frames, 12 -> 160 at the 160-channel blocks' [104, 180] plane
CAUSAL_CHUNK = (1, 12, 4, 104, 180)
CAUSAL_COUT = 160


def causal_cache_row(dev, stream, flush, pk, reps):
    """The packing launch and the convolution of one chunk, timed together."""
    import video_vae_convolution_gb300 as vvc
    N, C, T, H, W = CAUSAL_CHUNK
    Co = CAUSAL_COUT
    g = torch.Generator(device=dev)
    g.manual_seed(20250)
    x = torch.randn(CAUSAL_CHUNK, generator=g, device=dev).to(torch.bfloat16)
    prev = torch.randn((N, 2, H, W, C), generator=g, device=dev).to(torch.bfloat16)
    w = (torch.randn((Co, C, 3, 3, 3), generator=g, device=dev) * (C * 27) ** -0.5).to(
        torch.bfloat16)
    cc = vvc.CausalConv3dWithCache(CAUSAL_CHUNK, vvc.pack_weight(w), Co, history_frames=2,
                                   device=dev)

    class Step:
        def run(self, s):
            cc(x, prev, s)
            return 0

        def __call__(self, s):
            return self.run(s)

    ms = time_alone(Step(), stream, flush, reps)
    flop = 2.0 * N * T * H * W * Co * C * 27
    nbytes = 2 * (x.numel() + prev.numel() + N * T * H * W * Co + N * 2 * H * W * C +
                  w.numel())
    tf = flop / (ms * 1e-3) / 1e12
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"workload": "causal_cache", "name": "causal_12to160_chunk4_hist2",
            "layout": "NCTHW in, NDHWC out", "cin": C, "cout": Co, "kernel": [3, 3, 3],
            "stride": [1, 1, 1], "ms": round(ms, 4), "tflops": round(tf, 1),
            "frac_bf16": round(tf / pk["bf16_tflops"], 3),
            "frac_bf16_sustained": round(tf / pk["bf16_tflops_sustained"], 3),
            "gbs": round(gbs, 1), "frac_hbm": round(gbs / pk["hbm_gbs"], 3),
            "frac_hbm_nominal": round(gbs / HBM_NOMINAL_GBS, 3), "launches": cc.launches,
            "timed": "packing (history, causal and spatial zeros, 12 -> 16 channels, cache) "
                     "and the valid convolution, alone; FLOP of the 12 real channels"}


def other_layers(dev, stream, flush, pk, reps):
    """Per-call rows of the Wan-like chain (both layouts), the fused 160 blocks, the
    T=1 image-VAE layers (both layouts) and the decoder's upsample convolutions (x2
    nearest upsample fused into the convolution), each call timed alone."""
    import video_vae_convolution_gb300 as vvc
    rows = []
    sums = {}
    for name in ("wan", "fused160", "t1", "up2"):
        w = wl.all_workloads()[name]
        for call in w.calls:
            for lay, out_lay in w.layouts:
                inp = device_inputs(call, dev, lay, wl.seed_of(name, call))
                wp = vvc.pack_weight(inp["w"])
                c = vvc.Conv3d(inp["x"], wp, call.Cout, call.kernel, call.stride, call.pads,
                               lay, out_lay, call.epi, bias=inp["bias"],
                               residual=inp["residual"], residual_bias=inp["residual_bias"],
                               gamma=inp["gamma"], input_upsample=call.upsample)
                ms = time_alone(c, stream, flush, reps)
                rows.append(layer_row(call, ms, pk, c.launches, lay, name))
                key = (name, rows[-1]["layout"])
                sums[key] = sums.get(key, 0.0) + ms
                del c, wp, inp
        torch.cuda.empty_cache()
    rows.append(causal_cache_row(dev, stream, flush, pk, reps))
    wan_flop = sum(c.flops for c in wl.wan().calls)
    wan = {"calls": "3 shapes, each NCDHW->NCDHW and NDHWC->NDHWC, timed alone",
           "ms_ndhwc": round(sums[("wan", "NDHWC")], 4),
           "ms_ncdhw": round(sums[("wan", "NCDHW")], 4),
           "tflops": round(2 * wan_flop / ((sums[("wan", "NDHWC")] +
                                            sums[("wan", "NCDHW")]) * 1e-3) / 1e12, 1)}
    return rows, wan


# chained ladder: each intermediate carries the next call's spatial (reflect) padding as
# a 1-pixel halo; the next call applies the causal T padding itself
LADDER_HALO = ((0, 0, wl.ZERO), (1, 1, wl.REFLECT), (1, 1, wl.REFLECT))
CAUSAL_T = ((2, 0, wl.ZERO), (0, 0, wl.ZERO), (0, 0, wl.ZERO))


def build_ladder(dev, halo):
    """The 30 ladder calls on the device, each reading the previous call's output.
    halo: every call but the last writes its output inside a tensor with a 1-pixel
    reflect border (the next call's spatial padding) and every call but the first reads
    it with only the causal T padding of its own; otherwise each call applies its own
    causal + reflect padding.  Returns (calls, pinned host copy of the chain's input)."""
    import video_vae_convolution_gb300 as vvc
    calls = []
    x = None
    host_in = None
    ladder = wl.ladder().calls
    for i, call in enumerate(ladder):
        if x is None:
            inp = wl.make_inputs("ladder", call, wl.NDHWC, wl.NDHWC)
            host_in = inp["x"].pin_memory()
            x = inp["x"].to(dev)
        else:
            inp = {"w": wl.make_inputs("ladder", call, wl.NDHWC, wl.NDHWC, crop=(1, 3, 3))["w"]}
        wp = vvc.pack_weight(inp["w"].to(dev))
        last = i == len(ladder) - 1
        pads = call.pads if (i == 0 or not halo) else CAUSAL_T
        kw = {"out_halo": LADDER_HALO} if (halo and not last) else {}
        c = vvc.Conv3d(x, wp, call.Cout, call.kernel, call.stride, pads, wl.NDHWC, wl.NDHWC,
                       call.epi, **kw)
        calls.append((call, c))
        x = c.y
    return calls, host_in


def time_chain(calls, stream, flush, steps, warmup, world, sampler=None):
    """Times `steps` passes of the chain (L2 flushed before each); returns (mean step
    ms over the steps, per-call median ms, wall seconds)."""
    import video_vae_convolution_gb300 as vvc

    def chain(evs=None):
        for i, (_, c) in enumerate(calls):
            if evs is not None:
                evs[i].record(stream)
            rc = c.run(stream)
            if rc != 0:
                raise RuntimeError(f"conv3d_fwd failed: {rc}")
        if evs is not None:
            evs[-1].record(stream)

    for _ in range(max(3, warmup)):
        flush.zero_()
        chain()
    torch.cuda.synchronize()
    assert vvc.device_status() == 0
    barrier(world)
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    if sampler is not None:
        sampler.begin()
    step_ev = []
    for _ in range(steps):
        flush.zero_()
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)]
        chain(evs)
        step_ev.append(evs)
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - t_wall
    if sampler is not None:
        sampler.end()
    status = vvc.device_status()
    if status != 0:
        raise RuntimeError(f"device status {status}")
    per_call = [[] for _ in calls]
    step_ms = []
    for evs in step_ev:
        step_ms.append(evs[0].elapsed_time(evs[-1]))
        for i in range(len(calls)):
            per_call[i].append(evs[i].elapsed_time(evs[i + 1]))
    return statistics.mean(step_ms), [statistics.median(t) for t in per_call], wall, chain


def time_graph(chain, stream, flush, steps, warmup, world, sampler=None):
    """Times `steps` replays of a recorded chain (vvc.Chain), L2 flushed before each;
    returns (mean step ms, wall seconds)."""
    import video_vae_convolution_gb300 as vvc
    for _ in range(max(3, warmup)):
        flush.zero_()
        chain.run(stream)
    torch.cuda.synchronize()
    assert vvc.device_status() == 0
    barrier(world)
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    if sampler is not None:
        sampler.begin()
    evs = []
    for _ in range(steps):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        chain.run(stream)
        e1.record(stream)
        evs.append((e0, e1))
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - t_wall
    if sampler is not None:
        sampler.end()
    status = vvc.device_status()
    if status != 0:
        raise RuntimeError(f"device status {status}")
    return statistics.mean(a.elapsed_time(b) for a, b in evs), wall


def e4m3_layers(dev, stream, flush, pk, reps):
    """The ladder's layer classes with FP8 e4m3 operands (FlyDSL PR, the FP8 suite), each
    as in the haloed chain (valid convolution of a haloed input, haloed output but for
    conv_out) and timed alone; conv_in (3 input channels) has no e4m3 plan.  Rows carry
    the fraction of the e4m3 tensor peak, taken as 2 x the measured bf16 burst peak (the
    nominal dense fp8 / bf16 ratio, 4.5 / 2.25 PFLOP/s).  Also returns the sum over the
    29 calls (each class time x its repeats)."""
    import video_vae_convolution_gb300 as vvc
    rows = []
    total_ms = total_flop = 0.0
    ladder = wl.ladder().calls
    seen = {}
    for i, call in enumerate(ladder):
        cls = call_class(call.name)
        seen[cls] = seen.get(cls, 0) + 1
    done = set()
    for i, call in enumerate(ladder):
        cls = call_class(call.name)
        if call.Cin % 16 or cls in done:
            continue
        done.add(cls)
        g = torch.Generator(device=dev)
        g.manual_seed(wl.seed_of("ladder", call))
        shape = (call.N, call.D, call.H + 2, call.W + 2, call.Cin)
        x8 = wl.to_e4m3_bytes(torch.randn(shape, generator=g, device=dev) * 16.0)
        w8 = wl.to_e4m3_bytes(torch.randn((call.Cout, call.Cin) + tuple(call.kernel),
                                          generator=g, device=dev) * 4.0)
        wp = vvc.pack_weight_e4m3(w8)
        kw = {} if i == len(ladder) - 1 else {"out_halo": LADDER_HALO}
        c = vvc.Conv3d(x8, wp, call.Cout, call.kernel, call.stride, CAUSAL_T, wl.NDHWC,
                       wl.NDHWC, call.epi, dtype=vvc.DTYPE_E4M3,
                       fp8_scale=wl.E4M3_X_SCALE * wl.e4m3_weight_scale(call), **kw)
        ms = time_alone(c, stream, flush, reps)
        tf = call.flops / (ms * 1e-3) / 1e12
        row = layer_row(call, ms, pk, c.launches, wl.NDHWC, "ladder_e4m3",
                        {"dtype": "e4m3", "frac_e4m3": round(tf / (2 * pk["bf16_tflops"]), 3),
                         "calls_in_ladder": seen[cls],
                         "timed": "alone, haloed input as in the chain"})
        del row["frac_bf16"]  # measured against the e4m3 peak instead
        # one byte per input and weight element
        row["gbs"] = round((call.bytes() - call.N * call.Cin * call.D * call.H * call.W -
                            call.Cout * call.K) / (ms * 1e-3) / 1e9, 1)
        row["frac_hbm"] = round(row["gbs"] / pk["hbm_gbs"], 3)
        rows.append(row)
        total_ms += ms * seen[cls]
        total_flop += call.flops * seen[cls]
        del c, wp, x8, w8
    torch.cuda.empty_cache()
    summary = {"calls": "the 29 ladder calls with Cin % 16 == 0, each layer class timed alone "
                        "once and counted for its repeats",
               "ms_sum": round(total_ms, 4),
               "tflops": round(total_flop / (total_ms * 1e-3) / 1e12, 2) if total_ms else None,
               "peak_tflops": 2 * pk["bf16_tflops"],
               "peak_source": pk["source"] + " bf16 burst x 2 (nominal fp8 / bf16 ratio)"}
    return rows, summary


def run_gpu(args, rank, world):
    import video_vae_convolution_gb300 as vvc
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    pk = peaks()
    calls, host_in = build_ladder(dev, halo=True)
    torch.cuda.synchronize()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    total_flop = sum(call.flops for call, _ in calls)
    launches_per_step = sum(c.launches for _, c in calls)
    # input staging launches (the staged tap gather of a narrow input; NDHWC needs no
    # layout staging)
    staging_launches = sum(1 for _, c in calls if c.plan.im2col == 1)

    # per-call rows: the calls issued one by one, an event between each two
    eager_ms, call_ms, _, _ = time_chain(calls, stream, flush, args.steps, args.warmup, world)
    # the step: the 30 calls recorded once as a CUDA graph and replayed
    graph = vvc.Chain([c for _, c in calls], stream)
    sampler = ClockSampler(dev.index)
    sampler.start()
    ms_step, wall = time_graph(graph, stream, flush, args.steps, args.warmup, world, sampler)
    clocks = sampler.stop()
    ms_step = max_over_ranks(ms_step, world)
    value = world * total_flop / (ms_step * 1e-3) / 1e12

    layers = []
    class_ms = {}
    for (call, c), ms in zip(calls, call_ms):
        layers.append(layer_row(call, ms, pk, c.launches, wl.NDHWC, "ladder",
                                {"timed": "inside the chain, haloed intermediates"}))
        class_ms.setdefault(call_class(call.name), []).append((call, c, ms))
    # dominant kernel: the layer class with the largest share of the chain's time
    dom_cls, members = max(class_ms.items(), key=lambda kv: sum(m[2] for m in kv[1]))
    dom_call, dom_c, _ = members[0]
    dom_ms = statistics.mean(m[2] for m in members)
    achieved = dom_call.flops / (dom_ms * 1e-3) / 1e12
    roofline = {"bound": "tensor", "achieved": round(achieved, 1), "peak": pk["bf16_tflops"],
                "unit": "TFLOP/s", "frac": round(achieved / pk["bf16_tflops"], 4),
                "traffic": measured_traffic(dom_call.name),
                "kernel": f"vvc::conv_cm_kernel ({dom_cls}: {dom_call.Cin}->{dom_call.Cout} "
                          f"[{dom_call.D},{dom_call.H},{dom_call.W}], {len(members)} calls, "
                          f"{dom_c.launches} launch(es) each)",
                "share_of_chain": round(sum(m[2] for m in members) / eager_ms, 3),
                "peak_source": pk["source"] + " burst bf16",
                "algorithmic_flop": dom_call.flops, "algorithmic_bytes": dom_call.bytes()}

    # e2e: the chain's input from pinned host memory and its output back, every step
    out_host = torch.empty(calls[-1][1].y.shape, dtype=torch.bfloat16).pin_memory()
    x0 = calls[0][1].x
    y_last = calls[-1][1].y
    h2d = host_in.numel() * 2
    d2h = out_host.numel() * 2

    def e2e_step():
        x0.copy_(host_in, non_blocking=True)
        graph.run(stream)
        out_host.copy_(y_last, non_blocking=True)

    for _ in range(max(2, min(args.warmup, 3))):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e2e_steps = max(1, args.steps)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    e2e_ms = max_over_ranks(e2e_ms, world)
    e2e_val = world * total_flop / (e2e_ms * 1e-3) / 1e12

    # the same ladder with every call applying its own padding (no haloed tensors)
    plain_calls, _ = build_ladder(dev, halo=False)
    plain_ms, plain_call_ms, _, _ = time_chain(plain_calls, stream, flush, args.steps,
                                               args.warmup, world)
    for (call, c), ms in zip(plain_calls, plain_call_ms):
        layers.append(layer_row(call, ms, pk, c.launches, wl.NDHWC, "ladder_per_call_padding",
                                {"timed": "inside the chain, each call pads its own input"}))
    ladder_plain = {"ms_per_step": round(plain_ms, 4),
                    "tflops": round(total_flop / (plain_ms * 1e-3) / 1e12, 2),
                    "launches_per_step": sum(c.launches for _, c in plain_calls)}
    del plain_calls
    torch.cuda.empty_cache()

    # per-layer rows of the other workloads (each call alone, L2 flushed)
    other, wan = ([], None)
    e4m3_rows, e4m3 = ([], None)
    if not args.ladder_only:
        other, wan = other_layers(dev, stream, flush, pk, reps=max(3, min(args.steps, 10)))
        e4m3_rows, e4m3 = e4m3_layers(dev, stream, flush, pk, reps=max(3, min(args.steps, 10)))
    layers += other + e4m3_rows
    def wide_stats(rows):
        return {"calls": len(rows), "at_or_above_0.60": sum(r["frac_bf16"] >= 0.6 for r in rows),
                "min_frac_bf16": min((r["frac_bf16"] for r in rows), default=None)}

    bf16 = [r for r in layers if r.get("dtype", "bf16") == "bf16"]
    wide = [r for r in bf16 if r["cin"] >= 128 and r["cout"] >= 128 and
            r["kernel"] == [3, 3, 3] and r["layout"] == "NDHWC"]
    narrow = [r for r in bf16 if (min(r["cin"], r["cout"]) <= 16) and r["layout"] == "NDHWC" and
              r["workload"] != "ladder_per_call_padding"]
    targets = {
        "wide_3x3x3_ge128_ndhwc": wide_stats(
            [r for r in wide if r["workload"] != "ladder_per_call_padding"]),
        "wide_3x3x3_ge128_ndhwc_ladder_per_call_padding": wide_stats(
            [r for r in wide if r["workload"] == "ladder_per_call_padding"]),
        "narrow_ndhwc": {"calls": len(narrow),
                         "at_or_above_0.70_hbm": sum(r["frac_hbm"] >= 0.7 for r in narrow),
                         "min_frac_hbm": min((r["frac_hbm"] for r in narrow), default=None)},
        "ladder_staging_launches": staging_launches,
    }

    line = {"metric": METRIC, "value": round(value, 2),
            "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": workload_config(world),
            "roofline": roofline, "clocks": clocks,
            "e2e": {"value": round(e2e_val, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4)},
            "gpu_launches": launches_per_step * args.steps,
            "launch": "the 30 calls recorded once as a CUDA graph (vvc.Chain) and replayed "
                      "each step",
            "targets": targets, "wan_chain": wan, "ladder_per_call_padding": ladder_plain,
            "ladder_eager": {"ms_per_step": round(max_over_ranks(eager_ms, world), 4),
                             "tflops": round(world * total_flop / (eager_ms * 1e-3) / 1e12, 2),
                             "launch": "the 30 calls issued one by one (the per-call rows "
                                       "are timed this way)"},
            "ladder_e4m3": e4m3,
            "layers": layers, "wall_s": round(wall, 3)}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        r, ms, threads, desc = oracle_ladder_rate(target_s=12.0)
        line["cpu_baseline"] = dict({"value": r, "unit": "TFLOP/s", "cores": threads,
                                     "kind": "oracle", "sample": desc,
                                     "ms_per_step_extrapolated": ms}, **cpu_info(threads))
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def run_case(args):
    """One call of a workload, timed alone (for profiling and tuning)."""
    import video_vae_convolution_gb300 as vvc

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    work = wl.all_workloads()[args.workload]
    call = next(c for c in work.calls if c.name == args.case)
    lay = wl.NCDHW if args.layout == "ncdhw" else wl.NDHWC
    f8 = args.e4m3
    if f8:
        # FP8 e4m3 operands (NDHWC), the per-tensor scales of the workloads module
        lay = wl.NDHWC
        inp = wl.make_inputs_e4m3(args.workload, call)
    else:
        inp = wl.make_inputs(args.workload, call, lay, lay)
    g = lambda k: None if inp[k] is None else inp[k].to(dev)
    tun = None
    if args.tune:
        tun = vvc.Tuning(**{k: int(v) for k, v in (kv.split("=") for kv in args.tune.split(","))})
    wp = vvc.pack_weight_e4m3(inp["w8"].to(dev)) if f8 else vvc.pack_weight(inp["w"].to(dev))
    epi, extra = call.epi, {}
    if f8:
        extra = {"dtype": vvc.DTYPE_E4M3, "fp8_scale": inp["scale"]}
    if args.pad_cache >= 0:
        # padded output + two-frame cache after the fused norm, P history frames
        epi |= vvc.EPI_PAD_CACHE
        extra = {"history_frames": args.pad_cache}
    out_lay = wl.NDHWC if call.upsample else lay
    x = inp["x8" if f8 else "x"].to(dev)
    pads = call.pads
    if args.chain_halo and args.workload == "ladder":
        # as in the ladder chain: the input arrives with a 1-pixel spatial border and
        # the call applies the causal T padding; the output goes into a haloed tensor
        # unless this is the chain's last call
        if call.name != "conv_in":
            xp = torch.zeros((call.N, call.D, call.H + 2, call.W + 2, call.Cin),
                             dtype=x.dtype, device=dev)
            xp[:, :, 1:-1, 1:-1] = x
            x, pads = xp, CAUSAL_T
        if call.name != "conv_out":
            extra = dict(extra, out_halo=LADDER_HALO)
    c = vvc.Conv3d(x, wp, call.Cout, call.kernel, call.stride, pads, lay,
                   out_lay, epi, bias=g("bias"), residual=g("residual"),
                   residual_bias=g("residual_bias"), gamma=g("gamma"), tuning=tun,
                   input_upsample=call.upsample, **extra)
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        flush.zero_()
        c(stream)
    torch.cuda.synchronize()
    ts = []
    for _ in range(args.steps):
        flush.zero_()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        c(stream)
        b.record(stream)
        b.synchronize()
        ts.append(a.elapsed_time(b))
    assert vvc.device_status() == 0
    ms = statistics.median(ts)
    line = {"case": call.name, "layout": args.layout, "ms": round(ms, 4),
            "tflops": round(call.flops / (ms * 1e-3) / 1e12, 1),
            "gbs": round(call.bytes() / (ms * 1e-3) / 1e9, 1),
            "launches": c.launches, "tune": args.tune}
    if args.pad_cache >= 0:
        line["pad_cache"] = args.pad_cache
    if args.chain_halo:
        line["chain_halo"] = True
    if f8:
        line["dtype"] = "e4m3"
    print(json.dumps(line), flush=True)
    return 0


def run_norm_pad(args):
    """The standalone post-operations with padded output and cache, timed alone,
    beside the contiguous standalone call on the same input."""
    import video_vae_convolution_gb300 as vvc

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    C, T, H, W, P = (int(v) for v in args.norm_pad.split(","))
    gen = torch.Generator().manual_seed(4000 + C)
    x = torch.randn((1, T, H, W, C), generator=gen).to(torch.bfloat16).to(dev)
    gamma = (1 + 0.1 * torch.randn(C, generator=gen)).to(torch.bfloat16).float().to(dev)
    bias = (0.1 * torch.randn(C, generator=gen)).to(dev)
    prev = torch.randn((1, P, H, W, C), generator=gen).to(torch.bfloat16).to(dev) if P else None
    padded = torch.empty((1, T + 2, H + 2, W + 2, C), dtype=torch.bfloat16, device=dev)
    cache = torch.empty((1, min(2, T + P), H, W, C), dtype=torch.bfloat16, device=dev)
    y = torch.empty_like(x)
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def timed(fn):
        for _ in range(args.warmup):
            flush.zero_()
            fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(args.steps):
            flush.zero_()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            ts.append(a.elapsed_time(b))
        return statistics.median(ts)

    ms_pad = timed(lambda: vvc.l2norm_silu_pad(x, gamma, bias, previous=prev, padded=padded,
                                               cache=cache, stream=stream))
    ms_flat = timed(lambda: vvc.l2norm_silu(x, gamma, bias, y=y, stream=stream))
    assert vvc.device_status() == 0
    # algorithmic bytes: read x (+ history), write the padded tensor and the cache
    nbytes = 2 * (x.numel() + padded.numel() + cache.numel() + (prev.numel() if P else 0))
    print(json.dumps({"case": f"l2norm_silu_pad C{C} [1,{T},{H},{W}] P{P}",
                      "ms": round(ms_pad, 4), "gbs": round(nbytes / (ms_pad * 1e-3) / 1e9, 1),
                      "ms_contiguous": round(ms_flat, 4),
                      "gbs_contiguous": round(4 * x.numel() / (ms_flat * 1e-3) / 1e9, 1),
                      "launches": 2}), flush=True)
    return 0


def run_causal_cache(args):
    """The streaming causal 12 -> 160 call (packing + convolution) timed alone, as the
    bench line's causal_cache row."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    row = causal_cache_row(dev, stream, flush, peaks(), max(3, args.steps))
    print(json.dumps(row), flush=True)
    return 0


def run_group_norm(args):
    """Channels-last GroupNorm + SiLU with time-isolated groups, timed alone."""
    import video_vae_convolution_gb300 as vvc

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    C, D, H, W, G = (int(v) for v in args.group_norm.split(","))
    gen = torch.Generator().manual_seed(5000 + C)
    x = torch.randn((1, D, H, W, C), generator=gen).to(torch.bfloat16).to(dev)
    gamma = (1 + 0.1 * torch.randn(C, generator=gen)).to(dev)
    beta = (0.1 * torch.randn(C, generator=gen)).to(dev)
    y = torch.empty_like(x)
    ws = torch.empty(vvc._lib().group_norm_workspace_bytes(1, D, H, W, C, G, 1),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    run = lambda: vvc.group_norm_silu(x, G, gamma, beta, y=y, workspace=ws, stream=stream)
    for _ in range(args.warmup):
        flush.zero_()
        run()
    torch.cuda.synchronize()
    ts = []
    for _ in range(args.steps):
        flush.zero_()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        run()
        b.record(stream)
        b.synchronize()
        ts.append(a.elapsed_time(b))
    assert vvc.device_status() == 0
    ms = statistics.median(ts)
    nbytes = 4 * x.numel()  # algorithmic: x read once, y written once
    print(json.dumps({"case": f"group_norm_silu C{C} [1,{D},{H},{W}] G{G} time-isolated",
                      "ms": round(ms, 4), "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1),
                      "launches": 2}), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="ladder")
    ap.add_argument("--case", default=None, help="time one call of --workload alone")
    ap.add_argument("--layout", default="ndhwc", choices=["ndhwc", "ncdhw"])
    ap.add_argument("--tune", default="", help="plan overrides, e.g. R=2,kc=32")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--chain-halo", action="store_true",
                    help="with --workload ladder --case: run the call as in the chained ladder "
                         "(haloed input read as a valid convolution, haloed output)")
    ap.add_argument("--e4m3", action="store_true",
                    help="with --case: FP8 e4m3 operands (NDHWC)")
    ap.add_argument("--ladder-only", action="store_true",
                    help="time the ladder chain only (no per-layer rows of the other workloads)")
    ap.add_argument("--pad-cache", type=int, default=-1,
                    help="with --case: padded output + cache, this many history frames")
    ap.add_argument("--norm-pad", default="",
                    help="time the standalone padded post-operations: C,T,H,W,P")
    ap.add_argument("--group-norm", default="",
                    help="time the channels-last GroupNorm + SiLU: C,D,H,W,groups")
    ap.add_argument("--causal-cache", action="store_true",
                    help="time the streaming causal 12 -> 160 call (packing + convolution)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3) if args.impl != "reference" else args.warmup
    if args.group_norm:
        return run_group_norm(args)
    if args.causal_cache:
        return run_causal_cache(args)
    if args.norm_pad:
        return run_norm_pad(args)
    if args.case:
        return run_case(args)
    rank, world = dist_init(args)
    if args.impl == "reference":
        rc = run_reference(args, rank, world)
    else:
        rc = run_gpu(args, rank, world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return rc


if __name__ == "__main__":
    sys.exit(main())
