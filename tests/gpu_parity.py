"""Helpers for the GPU parity tests: run one call through the C ABI and compare
with the CPU oracle.

Tolerances (stated once, used by every GPU test):
* conv / bias / residual values: |gpu - ref| <= 2^-7 * |ref| + 1e-3 per element,
  where ref = B(oracle fp32 accumulator).  The GPU sums in fp32 in its own
  order, so a 1-ulp difference of B(conv) is allowed; 2^-7 |ref| bounds one
  bf16 ulp.
* epilogue: the oracle's epilogue run on the GPU's own B(conv) must reproduce
  the GPU's value exactly (<= 1 ulp allowed) and the fused L2-norm/SiLU output
  within 3 bf16 ulp.
* end to end (reported, and bounded by the pre-cancellation magnitude):
  |gpu - ref| <= 2^-7 (|conv| + |bias| + |skip|) + 1e-3 for values.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle
import video_vae_convolution_gb300 as vvc
import workloads as wl

ORC_FLAGS = {wl.EPI_BIAS: oracle.BIAS, wl.EPI_RESIDUAL: oracle.RESIDUAL,
             wl.EPI_RESIDUAL_BIAS: oracle.RESIDUAL_BIAS, wl.EPI_L2NORM_SILU: oracle.L2NORM_SILU}


def orc_flags(epi: int) -> int:
    f = 0
    for k, v in ORC_FLAGS.items():
        if epi & k:
            f |= v
    return f


def bits(t: torch.Tensor) -> np.ndarray:
    return wl.bits(t.detach().cpu().contiguous())


def f32(b: np.ndarray) -> np.ndarray:
    return oracle.bf16_to_f32(b)


def ulp_dist(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    def ordinal(u):
        i = u.astype(np.int32)
        mag = i & 0x7FFF
        return np.where((i & 0x8000) != 0, -mag, mag)
    return np.abs(ordinal(a) - ordinal(b))


class GpuCall:
    """Runs one workload call on the GPU; keeps CPU copies of inputs and outputs."""

    def __init__(self, call: wl.ConvCall, inp: dict, layout=wl.NDHWC, out_layout=wl.NDHWC,
                 tuning=None, debug_conv=True, extra_epi=0, extra_kw=None):
        self.call, self.inp, self.layout, self.out_layout = call, inp, layout, out_layout
        dev = torch.device("cuda")
        x = inp["x"].to(dev)
        w = inp["w"].to(dev)
        self.w_packed = vvc.pack_weight(w)
        epi = call.epi | extra_epi | (vvc.EPI_DEBUG_STORE_CONV if debug_conv else 0)
        g = lambda k: None if inp[k] is None else inp[k].to(dev).contiguous()
        self.c = vvc.Conv3d(x, self.w_packed, call.Cout, call.kernel, call.stride, call.pads,
                            layout, out_layout, epi, bias=g("bias"), residual=g("residual"),
                            residual_bias=g("residual_bias"), gamma=g("gamma"), tuning=tuning,
                            **(extra_kw or {}))
        rc = self.c.run()
        assert rc == vvc.OK, vvc._lib().conv3d_status_string(rc)
        torch.cuda.synchronize()
        assert vvc.device_status() == 0
        self.y = bits(self.c.y)
        self.conv = None if self.c.conv_out is None else bits(self.c.conv_out)
        self.value = None if self.c.value_out is None else bits(self.c.value_out)
        self.epi = epi

    def x_bits(self):
        return wl.bits(self.inp["x"])

    def w_bits(self):
        w = self.inp["w"]
        return wl.bits(w)


def check_conv(gpu_conv_bits: np.ndarray, ref_acc: np.ndarray, what="",
               chunk: int = 1 << 24):
    """Stage 1 on every element: |gpu - B(acc)| <= 2^-7 |B(acc)| + 1e-3.  Large
    outputs are compared in flat chunks of `chunk` elements (bounded host memory)."""
    g_all = np.ascontiguousarray(gpu_conv_bits).reshape(-1)
    a_all = np.ascontiguousarray(ref_acc).reshape(-1)
    assert g_all.size == a_all.size, (g_all.size, a_all.size)
    worst, nbad = 0.0, 0
    for i in range(0, a_all.size, chunk):
        ref = f32(oracle.round_bf16(a_all[i:i + chunk])).astype(np.float64)
        g = f32(g_all[i:i + chunk]).astype(np.float64)
        err = np.abs(g - ref)
        nbad += int(np.count_nonzero(err > 2.0 ** -7 * np.abs(ref) + 1e-3))
        if err.size:
            worst = max(worst, float(err.max()))
    assert nbad == 0, (f"{what}: {nbad} of {a_all.size} conv elements out of tolerance; "
                       f"max err {worst:.4g}")
    return worst


def to_ndhwc(t_bits, layout):
    return oracle.from_layout(t_bits, layout)


def check_epilogue(gc: GpuCall, value_ref_cpu=None):
    """Stage 2: oracle epilogue on the GPU's own B(conv) vs the GPU outputs."""
    call, inp = gc.call, gc.inp
    conv = gc.conv  # NDHWC unpadded
    res = None
    if inp["residual"] is not None:
        res = to_ndhwc(wl.bits(inp["residual"]), gc.out_layout)
    np_or_none = lambda t: None if t is None else t.numpy()
    e = oracle.epilogue(conv, orc_flags(call.epi), np_or_none(inp["bias"]), res,
                        np_or_none(inp["residual_bias"]), np_or_none(inp["gamma"]))
    y = to_ndhwc(gc.y, gc.out_layout)
    if call.epi & wl.EPI_OUT_PAD_BR:
        N, D, H, W, C = y.shape
        assert np.all(y[:, :, H - 1] == 0) and np.all(y[:, :, :, W - 1] == 0)
        y = np.ascontiguousarray(y[:, :, :H - 1, :W - 1])
    if call.epi & wl.EPI_L2NORM_SILU:
        d = ulp_dist(y, e["act"])
        assert d.max() <= 3, f"fused L2-norm/SiLU: max {d.max()} ulp"
        if gc.value is not None:
            dv = ulp_dist(to_ndhwc(gc.value, gc.out_layout), e["value"])
            assert dv.max() <= 1, f"value: max {dv.max()} ulp"
        return int(d.max())
    d = ulp_dist(y, e["value"])
    assert d.max() <= 1, f"value: max {d.max()} ulp"
    return int(d.max())


def full_reference(gc: GpuCall, x_bits_ncdhw_or_ndhwc=None):
    """Oracle fp32 accumulator for the whole call, [N, Do, Ho, Wo, Co]."""
    call = gc.call
    xb = gc.x_bits() if x_bits_ncdhw_or_ndhwc is None else x_bits_ncdhw_or_ndhwc
    return oracle.conv3d_acc(xb, gc.layout, gc.w_bits(), call.stride, call.pads)


def sample_points(N, Do, Ho, Wo, k, seed=0, tile_w=128):
    """Border, tile-boundary and random output pixels (n, d, h, w)."""
    rng = np.random.default_rng(seed)
    k = min(k, N * Do * Ho * Wo)
    pts = set()
    ws = sorted({0, 1, Wo - 2, Wo - 1} | {min(Wo - 1, max(0, t + o))
                                          for t in range(0, Wo, tile_w) for o in (-1, 0)})
    hs = sorted({0, 1, Ho - 2, Ho - 1})
    ds = sorted({0, Do - 1})
    for n in {0, N - 1}:
        for d in ds:
            for h in hs:
                for w in ws:
                    if 0 <= h < Ho and 0 <= w < Wo:
                        pts.add((n, d, h, w))
    while len(pts) < k:
        pts.add((int(rng.integers(N)), int(rng.integers(Do)), int(rng.integers(Ho)),
                 int(rng.integers(Wo))))
    return np.array(sorted(pts), dtype=np.int64)


def border_and_random_points(N, Do, Ho, Wo, k_random, seed=0, tile_w=128):
    """Every border pixel of every (n, d) plane (the outer two rows and columns),
    the columns on either side of each tile_w boundary, the first and last output
    frames whole, plus k_random random pixels; all pixels when that is more than
    the output holds.  Returns int64 [P, 4] (n, d, h, w)."""
    M = N * Do * Ho * Wo
    hh, ww = np.meshgrid(np.arange(Ho), np.arange(Wo), indexing="ij")
    cols = {0, 1, Wo - 2, Wo - 1} | {c for t in range(tile_w, Wo, tile_w) for c in (t - 1, t)}
    edge = (hh < 2) | (hh >= Ho - 2) | np.isin(ww, sorted(c for c in cols if 0 <= c < Wo))
    e_h, e_w = hh[edge].ravel(), ww[edge].ravel()
    pts = set()
    for n in range(N):
        for d in range(Do):
            if d in (0, Do - 1):
                pts.update((n, d, h, w) for h in range(Ho) for w in range(Wo))
            else:
                pts.update(zip([n] * e_h.size, [d] * e_h.size, e_h.tolist(), e_w.tolist()))
    if len(pts) + k_random >= M:
        g = np.stack(np.meshgrid(np.arange(N), np.arange(Do), np.arange(Ho), np.arange(Wo),
                                 indexing="ij"), -1)
        return g.reshape(-1, 4).astype(np.int64)
    rng = np.random.default_rng(seed)
    target = len(pts) + k_random
    while len(pts) < target:
        need = target - len(pts)
        r = np.stack([rng.integers(N, size=need), rng.integers(Do, size=need),
                      rng.integers(Ho, size=need), rng.integers(Wo, size=need)], 1)
        pts.update(map(tuple, r.tolist()))
    return np.array(sorted(pts), dtype=np.int64)


def check_points(gc: GpuCall, pts: np.ndarray):
    """Stage 1 at the given output pixels (all channels) and stage 2 on the whole
    output; returns (max conv error, max epilogue ulp)."""
    call = gc.call
    acc = oracle.conv3d_acc_points(gc.x_bits(), gc.layout, gc.w_bits(), pts, call.stride,
                                   call.pads)
    conv = gc.conv[pts[:, 0], pts[:, 1], pts[:, 2], pts[:, 3]]
    err = check_conv(conv, acc, call.name)
    return err, check_epilogue(gc)


def check_sampled(gc: GpuCall, k=1024, seed=0):
    """Full-size check on sampled pixels: conv (stage 1) at each sampled pixel,
    and the epilogue (stage 2) on the whole output."""
    call = gc.call
    Do, Ho, Wo = gc.c.out_dims
    N = gc.c.dims[0]
    pts = sample_points(N, Do, Ho, Wo, k, seed)
    acc = oracle.conv3d_acc_points(gc.x_bits(), gc.layout, gc.w_bits(), pts, call.stride,
                                   call.pads)
    conv = gc.conv[pts[:, 0], pts[:, 1], pts[:, 2], pts[:, 3]]
    err = check_conv(conv, acc, call.name)
    ulp = check_epilogue(gc)
    return err, ulp
