"""Benchmark: bf16 implicit-GEMM conv3d on one GB300 (per layer TFLOP/s and chain ms).

Workload (one step = one pass of the whole chain): the Wan-like channel-constant
chain of valid convolutions (pad applied outside) — x [1,96,6,354,642] with
w [96,96,3,3,3]; x [1,384,3,46,82] with w [384,384,3,3,3]; rank-4 x [4,96,353,641]
with w [96,96,3,3] — each run once with NCDHW input/output and once with NDHWC
throughout.  Inputs are seeded synthetic tensors of those shapes.

Prints one JSON line.  `value` is chain TFLOP/s (algorithmic FLOP of the six
calls / device time of one chain), inputs resident in HBM, L2 flushed between
steps.  `e2e` is the same metric with pinned host inputs copied in and outputs
copied out inside the timed region.  `--impl reference` times the CPU oracle
on a bounded sample of the same workload.
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

WORKLOAD_NAME = "wan"
L2_FLUSH_BYTES = 256 << 20


# DRAM bytes (read + write) of one launch of the dominant kernel, from one ncu
# capture (profiles/conv_cm_wan96_ndhwc.md), keyed by a hash of the kernel's
# sources (comments and whitespace left out): a changed kernel reports null until
# it is captured again.
KERNEL_SOURCES = ["conv_cm.cu", "epilogue_cm.cuh", "epilogue.cuh", "kernel_common.cuh",
                  "ptx.cuh", "internal.h"]
NCU_TRAFFIC = {"f2e0061935f07fe9": 262620928 + 140352512}


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


def measured_traffic():
    return NCU_TRAFFIC.get(kernel_source_hash())


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


def chain_calls():
    w = wl.wan()
    out = []
    for lay in (wl.NCDHW, wl.NDHWC):
        for call in w.calls:
            out.append((call, lay))
    return out


def workload_config(args, extra=None):
    cfg = {"workload": "wan_chain: valid 3x3x3 96->96 [1,96,6,354,642], 384->384 "
                       "[1,384,3,46,82], 3x3 96->96 [4,96,353,641]; each NCDHW->NCDHW and "
                       "NDHWC->NDHWC",
           "calls_per_step": 6, "l2": "flushed between steps (256 MiB write, untimed)",
           "inputs": "seeded synthetic N(0,1) bf16, weights N(0,1/sqrt(fan_in))"}
    if extra:
        cfg.update(extra)
    return cfg


# ---- CPU oracle legs ------------------------------------------------------------------------

def oracle_rate(target_s=12.0, max_points=None):
    """Times the oracle on sampled output pixels of every chain call; returns
    (TFLOP/s, cores, sample description)."""
    import oracle
    oracle.build()
    cores = oracle.num_threads(0)
    flops = 0.0
    t_total = 0.0
    samples = []
    per_call = target_s / 3.0
    for call in wl.wan().calls:
        inp = wl.make_inputs("wan", call, wl.NDHWC)
        xb, wb = wl.bits(inp["x"]), wl.bits(inp["w"])
        Do, Ho, Wo = call.out_dims()
        fpp = 2.0 * call.Cout * call.K  # FLOP per output pixel
        rng = np.random.default_rng(1)
        n = 64
        spent = 0.0
        while spent < per_call and (max_points is None or n <= max_points):
            pts = np.stack([rng.integers(0, call.N, n), rng.integers(0, Do, n),
                            rng.integers(0, Ho, n), rng.integers(0, Wo, n)], 1)
            t0 = time.perf_counter()
            oracle.conv3d_acc_points(xb, wl.NDHWC, wb, pts, call.stride, call.pads)
            dt = time.perf_counter() - t0
            spent += dt
            t_total += dt
            flops += fpp * n
            samples.append(n)
            n = min(n * 2, 1 << 16)
    rate = flops / t_total / 1e12
    desc = (f"oracle direct conv (fp64 accumulate) on {sum(samples)} sampled output pixels "
            f"across the 3 chain shapes, {t_total:.1f} s")
    return rate, cores, desc


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    # bounded: the whole run stays within about two minutes of CPU time
    budget = max(1.0, min(8.0, 120.0 / max(1, args.steps + args.warmup)))
    rates = []
    for _ in range(args.warmup):
        oracle_rate(target_s=min(1.0, budget))
    t0 = time.perf_counter()
    desc = ""
    cores = 0
    for _ in range(args.steps):
        r, cores, desc = oracle_rate(target_s=budget)
        rates.append(r)
    elapsed = time.perf_counter() - t0
    value = statistics.median(rates)
    total_flop = sum(c.flops for c, _ in chain_calls())
    line = {"impl": "reference", "metric": "bf16 conv3d TFLOP/s (chain)", "value": value,
            "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": total_flop / (value * 1e12) * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(args),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "wall_s": elapsed}
    print(json.dumps(line), flush=True)
    return 0


# ---- GPU arm -------------------------------------------------------------------------------

def run_gpu(args, rank, world):
    import video_vae_convolution_gb300 as vvc

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    pk = peaks()
    calls = []
    host = []
    for call, lay in chain_calls():
        inp = wl.make_inputs("wan", call, lay, lay)
        x = inp["x"].to(dev)
        wp = vvc.pack_weight(inp["w"].to(dev))
        c = vvc.Conv3d(x, wp, call.Cout, call.kernel, call.stride, call.pads, lay, lay, 0)
        calls.append((call, lay, c))
        host.append(inp["x"].pin_memory())
    torch.cuda.synchronize()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    total_flop = sum(call.flops for call, _, _ in calls)
    launches_per_step = sum(c.launches for _, _, c in calls)

    def chain(evs=None):
        for i, (_, _, c) in enumerate(calls):
            if evs is not None:
                evs[i][0].record(stream)
            rc = c.run(stream)
            if rc != 0:
                raise RuntimeError(f"conv3d_fwd failed: {rc}")
            if evs is not None:
                evs[i][1].record(stream)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        chain()
    torch.cuda.synchronize()
    assert vvc.device_status() == 0

    sampler = ClockSampler(dev.index)
    sampler.start()
    per_call = [[] for _ in calls]
    barrier(world)
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    sampler.begin()
    step_ev = []
    for _ in range(args.steps):
        flush.zero_()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in calls]
        chain(evs)
        step_ev.append(evs)
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - t_wall
    sampler.end()
    clocks = sampler.stop()
    status = vvc.device_status()
    if status != 0:
        raise RuntimeError(f"device status {status}")
    step_ms = []
    for evs in step_ev:
        tot = 0.0
        for i, (a, b) in enumerate(evs):
            ms = a.elapsed_time(b)
            per_call[i].append(ms)
            tot += ms
        step_ms.append(tot)
    ms_step = statistics.mean(step_ms)
    ms_step = max_over_ranks(ms_step, world)
    value = world * total_flop / (ms_step * 1e-3) / 1e12

    layers = []
    for (call, lay, c), ts in zip(calls, per_call):
        ms = statistics.median(ts)
        tf = call.flops / (ms * 1e-3) / 1e12
        layers.append({"name": call.name, "layout": "NCDHW" if lay == wl.NCDHW else "NDHWC",
                       "ms": round(ms, 4), "tflops": round(tf, 1),
                       "frac_bf16": round(tf / pk["bf16_tflops"], 3),
                       "gbs": round(call.bytes() / (ms * 1e-3) / 1e9, 1),
                       "launches": c.launches})
    # dominant kernel: the 96->96 3-D call in NDHWC (one conv launch)
    dom_i = next(i for i, (call, lay, c) in enumerate(calls)
                 if call.name == "wan_96_3d" and lay == wl.NDHWC)
    dom_call, _, dom_c = calls[dom_i]
    dom_ms = statistics.mean(per_call[dom_i])
    achieved = dom_call.flops / (dom_ms * 1e-3) / 1e12
    roofline = {"bound": "tensor", "achieved": round(achieved, 1), "peak": pk["bf16_tflops"],
                "unit": "TFLOP/s", "frac": round(achieved / pk["bf16_tflops"], 4),
                "traffic": measured_traffic(), "kernel": "vvc::conv_cm_kernel (wan_96_3d, NDHWC)",
                "peak_source": pk["source"] + " burst bf16",
                "algorithmic_bytes": dom_call.bytes()}

    # e2e: pinned host inputs -> device, the chain through the C ABI, outputs -> pinned
    # host, every step.  The calls are independent, so the copies run on their own
    # streams: call i's input copy overlaps call i-1's convolution and call i-2's
    # output copy (events order each call's copy-in, convolution and copy-out, and a
    # buffer is rewritten only after the previous step is done with it).
    outs_host = [torch.empty(c.y.shape, dtype=torch.bfloat16).pin_memory() for _, _, c in calls]
    h2d = sum(h.numel() * 2 for h in host)
    d2h = sum(o.numel() * 2 for o in outs_host)
    e2e_steps = max(1, min(args.steps, 10))
    # one copy stream per direction (splitting a copy over several streams measured
    # slower: concurrent copies in one direction contend)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    n = len(calls)
    ev_in = [torch.cuda.Event() for _ in range(n)]
    ev_conv = [torch.cuda.Event() for _ in range(n)]
    ev_out = [torch.cuda.Event() for _ in range(n)]
    def e2e_steps_run(count):
        for step in range(count):
            for i, ((call, lay, c), h, o) in enumerate(zip(calls, host, outs_host)):
                if step:
                    s_in.wait_event(ev_conv[i])    # the previous step has read c.x
                with torch.cuda.stream(s_in):
                    c.x.copy_(h, non_blocking=True)
                ev_in[i].record(s_in)
                stream.wait_event(ev_in[i])
                if step:
                    stream.wait_event(ev_out[i])   # the previous step's c.y has been copied out
                rc = c.run(stream)
                if rc != 0:
                    raise RuntimeError(f"conv3d_fwd failed: {rc}")
                ev_conv[i].record(stream)
                s_out.wait_event(ev_conv[i])
                with torch.cuda.stream(s_out):
                    o.copy_(c.y, non_blocking=True)
                ev_out[i].record(s_out)
        for i in range(n):
            stream.wait_event(ev_out[i])

    # untimed warm-up passes (first use of the copy streams and pinned buffers)
    e2e_steps_run(max(1, min(args.warmup, 3)))
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    e2e_steps_run(e2e_steps)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    e2e_ms = max_over_ranks(e2e_ms, world)
    e2e_val = world * total_flop / (e2e_ms * 1e-3) / 1e12

    line = {"metric": "bf16 conv3d TFLOP/s (chain)", "value": round(value, 2),
            "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": workload_config(args, {"parallelism": f"replicas x{world}"}),
            "roofline": roofline, "clocks": clocks,
            "e2e": {"value": round(e2e_val, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 3)},
            "gpu_launches": launches_per_step * args.steps,
            "layers": layers, "wall_s": round(wall, 3)}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        r, cores, desc = oracle_rate(target_s=12.0)
        line["cpu_baseline"] = {"value": r, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                                "sample": desc}
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
    inp = wl.make_inputs(args.workload, call, lay, lay)
    g = lambda k: None if inp[k] is None else inp[k].to(dev)
    tun = None
    if args.tune:
        tun = vvc.Tuning(**{k: int(v) for k, v in (kv.split("=") for kv in args.tune.split(","))})
    wp = vvc.pack_weight(inp["w"].to(dev))
    epi, extra = call.epi, {}
    if args.pad_cache >= 0:
        # padded output + two-frame cache after the fused norm, P history frames
        epi |= vvc.EPI_PAD_CACHE
        extra = {"history_frames": args.pad_cache}
    c = vvc.Conv3d(inp["x"].to(dev), wp, call.Cout, call.kernel, call.stride, call.pads, lay, lay,
                   epi, bias=g("bias"), residual=g("residual"),
                   residual_bias=g("residual_bias"), gamma=g("gamma"), tuning=tun, **extra)
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
    ap.add_argument("--workload", default="wan")
    ap.add_argument("--case", default=None, help="time one call of --workload alone")
    ap.add_argument("--layout", default="ndhwc", choices=["ndhwc", "ncdhw"])
    ap.add_argument("--tune", default="", help="plan overrides, e.g. R=2,kc=32")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--pad-cache", type=int, default=-1,
                    help="with --case: padded output + cache, this many history frames")
    ap.add_argument("--norm-pad", default="",
                    help="time the standalone padded post-operations: C,T,H,W,P")
    ap.add_argument("--group-norm", default="",
                    help="time the channels-last GroupNorm + SiLU: C,D,H,W,groups")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3) if args.impl != "reference" else args.warmup
    if args.group_norm:
        return run_group_norm(args)
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
