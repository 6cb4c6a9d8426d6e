"""Seeded synthetic inputs and the workload definitions.

This module holds no arithmetic of the method: it only draws random numbers,
rounds them to bf16 storage and describes the shapes of each call.  Both the
CUDA path and the oracle take their inputs from here.

Workloads are shaped like the VAE convolution layers the source pages list:

* "wan": the Wan encoder's dominant shapes, valid convolution with the pad
  applied outside (ROCm/FlyDSL issue "[Feature]: conv3d_implicit — accept and
  emit NDHWC ...", section "Why").
* "ladder": the 30-call causal-VAE encoder tile (same issue, MiniMax-H3 comment,
  "Shapes" table), causal temporal zero pad 2 + reflect spatial pad 1.
* "fused160": the base_dim=160 fused post-op blocks (cuDNN frontend doc
  "Fused Conv3D + Bias + Residual + RMSNorm + SiLU", "Requirements" table).
* "t1": the T=1 image-VAE convolutions (ROCm/FlyDSL PR "[Flydsl] Add
  Qwen-Image VAE classic conv shapes to conv3d tests", "Test shapes").
* "up2": the decoder's 3x3 convolutions after a nearest-exact x2 upsample (same
  PR, "Upsample Conv2d"), with the upsample fused into the convolution's input.
* "tiny": a small correctness case.

Seeds: seed = 1000 * workload_id + call_index, plus 0 for x, 1 for W, 2 for
bias, 3 for residual, 4 for gamma, 5 for residual_bias.  Values are drawn in
fp32 with torch's CPU generator and rounded to bf16 (round to nearest even).
x ~ N(0, 1) (U[-1, 1] for "tiny"); W ~ N(0, std = 1/sqrt(Cin*KT*KR*KS));
bias, residual_bias ~ N(0, 0.1) fp32; residual ~ N(0, 1) bf16;
gamma ~ N(1, 0.1) fp32 holding bf16-representable values.
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Tuple

import numpy as np
import torch

NCDHW = 0
NDHWC = 1
ZERO = 0
REFLECT = 1

# epilogue flags (same meaning as the library's; values are plain bits)
EPI_BIAS = 1
EPI_RESIDUAL = 2
EPI_RESIDUAL_BIAS = 4
EPI_L2NORM_SILU = 8
EPI_SAVE_VALUE = 16
EPI_OUT_PAD_BR = 32

WORKLOAD_IDS = {"tiny": 1, "wan": 2, "ladder": 3, "fused160": 4, "t1": 5, "up2": 6, "test": 9}


@dataclass
class ConvCall:
    name: str
    N: int
    Cin: int
    D: int
    H: int
    W: int
    Cout: int
    kernel: Tuple[int, int, int] = (3, 3, 3)
    stride: Tuple[int, int, int] = (1, 1, 1)
    # (before, after, mode) for T, H, W
    pads: Tuple[Tuple[int, int, int], ...] = ((0, 0, ZERO),) * 3
    epi: int = 0
    x_dist: str = "normal"          # "normal" | "uniform"
    zero_pad_br_input: bool = False  # input made by ZeroPad2d((0,1,0,1))
    rank4: bool = False              # originally a 2-D (NCHW) convolution
    index: int = 0
    upsample: int = 0                # 2: the convolution reads the x2 nearest upsample of x

    @property
    def K(self) -> int:
        kt, kr, ks = self.kernel
        return self.Cin * kt * kr * ks

    def out_dims(self):
        kt, kr, ks = self.kernel
        up = 2 if self.upsample == 2 else 1
        L = (self.D, self.H * up, self.W * up)
        K = (kt, kr, ks)
        return tuple((L[i] + self.pads[i][0] + self.pads[i][1] - K[i]) // self.stride[i] + 1
                     for i in range(3))

    @property
    def M(self) -> int:
        Do, Ho, Wo = self.out_dims()
        return self.N * Do * Ho * Wo

    @property
    def flops(self) -> int:
        """Algorithmic FLOP = 2 * M * Cout * Cin * KT * KR * KS (real channels)."""
        return 2 * self.M * self.Cout * self.K

    def bytes(self) -> int:
        """Algorithmic bytes: input + output (+ residual, + value) + weights, once (the
        input of an upsampling call is the low-resolution tensor)."""
        Do, Ho, Wo = self.out_dims()
        out_elems = self.N * Do * Ho * Wo * self.Cout
        if self.epi & EPI_OUT_PAD_BR:
            out_elems = self.N * Do * (Ho + 1) * (Wo + 1) * self.Cout
        b = 2 * self.N * self.Cin * self.D * self.H * self.W + 2 * out_elems
        b += 2 * self.Cout * self.K
        if self.epi & EPI_RESIDUAL:
            b += 2 * self.N * Do * Ho * Wo * self.Cout
        if self.epi & EPI_SAVE_VALUE:
            b += 2 * self.N * Do * Ho * Wo * self.Cout
        return b


@dataclass
class Workload:
    name: str
    calls: List[ConvCall]
    chained: bool = False
    layouts: List[Tuple[int, int]] = field(default_factory=lambda: [(NDHWC, NDHWC)])


def _causal_reflect():
    return ((2, 0, ZERO), (1, 1, REFLECT), (1, 1, REFLECT))


def _same2d():
    return ((0, 0, ZERO), (1, 1, ZERO), (1, 1, ZERO))


def tiny() -> Workload:
    pads = ((1, 1, ZERO),) * 3
    calls = [
        ConvCall("tiny_conv_bias", 1, 16, 4, 12, 12, 32, pads=pads, epi=EPI_BIAS,
                 x_dist="uniform", index=0),
        ConvCall("tiny_fused", 1, 16, 4, 12, 12, 32, pads=pads,
                 epi=EPI_BIAS | EPI_RESIDUAL | EPI_L2NORM_SILU | EPI_SAVE_VALUE,
                 x_dist="uniform", index=1),
    ]
    return Workload("tiny", calls)


def wan() -> Workload:
    calls = [
        ConvCall("wan_96_3d", 1, 96, 6, 354, 642, 96, index=0),
        ConvCall("wan_384_3d", 1, 384, 3, 46, 82, 384, index=1),
        ConvCall("wan_96_2d", 4, 96, 1, 353, 641, 96, kernel=(1, 3, 3), rank4=True, index=2),
    ]
    return Workload("wan", calls, layouts=[(NCDHW, NCDHW), (NDHWC, NDHWC)])


def ladder() -> Workload:
    p = _causal_reflect()
    spec = [
        # (name, Cin, D, H, W, Cout, stride, repeat)
        ("conv_in", 3, 17, 256, 256, 128, (1, 1, 1), 1),
        ("L0", 128, 17, 256, 256, 128, (1, 1, 1), 4),
        ("L0s", 128, 17, 256, 256, 128, (1, 2, 2), 1),
        ("L1a", 128, 17, 128, 128, 256, (1, 1, 1), 1),
        ("L1", 256, 17, 128, 128, 256, (1, 1, 1), 3),
        ("L1s", 256, 17, 128, 128, 256, (2, 2, 2), 1),
        ("L2", 256, 9, 64, 64, 256, (1, 1, 1), 4),
        ("L2s", 256, 9, 64, 64, 256, (2, 2, 2), 1),
        ("L3a", 256, 5, 32, 32, 512, (1, 1, 1), 1),
        ("L3", 512, 5, 32, 32, 512, (1, 1, 1), 3),
        ("L3s", 512, 5, 32, 32, 512, (1, 2, 2), 1),
        ("L4", 512, 5, 16, 16, 512, (1, 1, 1), 4),
        ("L5a", 512, 5, 16, 16, 1024, (1, 1, 1), 1),
        ("L5", 1024, 5, 16, 16, 1024, (1, 1, 1), 3),
        ("conv_out", 1024, 5, 16, 16, 48, (1, 1, 1), 1),
    ]
    calls = []
    for name, cin, d, h, w, cout, stride, rep in spec:
        for k in range(rep):
            nm = name if rep == 1 else f"{name}_{k}"
            calls.append(ConvCall(nm, 1, cin, d, h, w, cout, stride=stride, pads=p,
                                  index=len(calls)))
    assert len(calls) == 30
    return Workload("ladder", calls, chained=True,
                    layouts=[(NDHWC, NDHWC), (NCDHW, NCDHW)])


def fused160() -> Workload:
    norm = EPI_BIAS | EPI_L2NORM_SILU
    padres = EPI_BIAS | EPI_RESIDUAL | EPI_RESIDUAL_BIAS | EPI_OUT_PAD_BR
    calls = [
        ConvCall("f160_160", 1, 160, 8, 106, 182, 160, epi=norm, index=0),
        ConvCall("f160_320", 1, 160, 8, 106, 182, 320, epi=norm, index=1),
        ConvCall("f320_320", 1, 320, 8, 106, 182, 320, epi=norm, index=2),
        ConvCall("f320_640", 1, 320, 8, 106, 182, 640, epi=padres, index=3),
        ConvCall("f640_640", 1, 640, 8, 106, 182, 640, epi=padres, index=4),
    ]
    return Workload("fused160", calls)


def t1() -> Workload:
    p = _same2d()
    k2 = (1, 3, 3)
    spec = [
        ("96_1024", 96, 1024, 96), ("96_1328", 96, 1328, 96), ("192_512", 192, 512, 192),
        ("384_256", 384, 256, 384), ("384_128", 384, 128, 384), ("384_166", 384, 166, 384),
        ("3to96_1024", 3, 1024, 96), ("96to3_1024", 96, 1024, 3),
        ("16to384_128", 16, 128, 384), ("384to32_128", 384, 128, 32),
    ]
    calls = []
    for name, cin, hw, cout in spec:
        calls.append(ConvCall(f"t1_{name}", 1, cin, 1, hw, hw, cout, kernel=k2, pads=p,
                              rank4=True, index=len(calls)))
    for c, hw in ((96, 1025), (192, 513), (384, 257)):
        calls.append(ConvCall(f"t1_down{c}_{hw}", 1, c, 1, hw, hw, c, kernel=k2,
                              stride=(1, 2, 2), rank4=True, zero_pad_br_input=True,
                              index=len(calls)))
    return Workload("t1", calls, layouts=[(NDHWC, NDHWC), (NCDHW, NCDHW)])


def up2() -> Workload:
    p = _same2d()
    spec = [("dec_d0_384_256", 384, 128, 192), ("dec_d1_384_512", 384, 256, 192),
            ("dec_d2_192_1024", 192, 512, 96)]
    calls = [ConvCall(name, 1, cin, 1, hw, hw, cout, kernel=(1, 3, 3), pads=p, epi=EPI_BIAS,
                      rank4=True, upsample=2, index=i)
             for i, (name, cin, hw, cout) in enumerate(spec)]
    return Workload("up2", calls, layouts=[(NDHWC, NDHWC), (NCDHW, NDHWC)])


def all_workloads():
    return {"tiny": tiny(), "wan": wan(), "ladder": ladder(), "fused160": fused160(),
            "t1": t1(), "up2": up2()}


# ---- generation -------------------------------------------------------------------

def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def normal(shape, seed, mean=0.0, std=1.0) -> torch.Tensor:
    t = torch.randn(tuple(shape), generator=_gen(seed), dtype=torch.float32)
    return t * std + mean


def uniform(shape, seed, lo=-1.0, hi=1.0) -> torch.Tensor:
    t = torch.rand(tuple(shape), generator=_gen(seed), dtype=torch.float32)
    return t * (hi - lo) + lo


def to_bf16(t: torch.Tensor) -> torch.Tensor:
    return t.to(torch.bfloat16)


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 torch tensor (CPU) -> numpy uint16 bit patterns."""
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bits(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


def to_e4m3_bytes(t: torch.Tensor) -> torch.Tensor:
    """Float tensor -> e4m3fn codes as torch.uint8 (values clamped to +-448 first,
    then torch's float8_e4m3fn conversion)."""
    return t.float().clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)


# per-tensor scale of the e4m3 activations: x / 2^-4 spreads N(0, 1) over +-64
E4M3_X_SCALE = 2.0 ** -4


def e4m3_weight_scale(call: "ConvCall") -> float:
    """Power of two near a quarter of the weights' standard deviation, so that the
    e4m3 codes of w / scale spread over about +-16 (normal range, 3 mantissa bits)."""
    kt, kr, ks = call.kernel
    std = 1.0 / np.sqrt(call.Cin * kt * kr * ks)
    return float(2.0 ** np.round(np.log2(std / 4.0)))


def make_inputs_e4m3(workload: str, call: "ConvCall", crop=None) -> dict:
    """The bf16 recipe of make_inputs (NDHWC) quantised to e4m3fn with per-tensor
    power-of-two scales: adds x8 (uint8 NDHWC), w8 (uint8 OITRS) and scale = the
    product of the two scales (the accumulator factor).  bias, residual, gamma as in
    make_inputs."""
    base = make_inputs(workload, call, NDHWC, NDHWC, crop=crop)
    sx, sw = E4M3_X_SCALE, e4m3_weight_scale(call)
    base["x8"] = to_e4m3_bytes(base["x"].float() / sx).contiguous()
    base["w8"] = to_e4m3_bytes(base["w"].float() / sw).contiguous()
    base["scale"] = sx * sw
    return base


def seed_of(workload: str, call: ConvCall) -> int:
    return 1000 * WORKLOAD_IDS[workload] + call.index


def make_inputs(workload: str, call: ConvCall, layout: int = NDHWC, out_layout: int = NDHWC,
                x_override: Optional[torch.Tensor] = None, crop=None):
    """Seeded inputs of one call, as CPU tensors.

    Returns dict: x (bf16, `layout`), w (bf16 OITRS, KT=1 for 2-D kernels),
    bias / residual_bias / gamma (fp32 or None), residual (bf16, out_layout,
    unpadded output shape, or None).  `crop` = (D, H, W) draws a smaller input
    with the same recipe (for CPU-sized checks).
    """
    s = seed_of(workload, call)
    N, C, D, H, W = call.N, call.Cin, call.D, call.H, call.W
    if crop is not None:
        D, H, W = crop
    if x_override is not None:
        x_ncdhw = x_override
    elif call.zero_pad_br_input:
        inner = to_bf16(normal((N, C, D, H - 1, W - 1), s))
        x_ncdhw = torch.zeros((N, C, D, H, W), dtype=torch.bfloat16)
        x_ncdhw[:, :, :, :H - 1, :W - 1] = inner
    elif call.x_dist == "uniform":
        x_ncdhw = to_bf16(uniform((N, C, D, H, W), s))
    else:
        x_ncdhw = to_bf16(normal((N, C, D, H, W), s))
    x = x_ncdhw if layout == NCDHW else x_ncdhw.permute(0, 2, 3, 4, 1).contiguous()
    kt, kr, ks = call.kernel
    fan_in = C * kt * kr * ks
    w = to_bf16(normal((call.Cout, C, kt, kr, ks), s + 1, std=1.0 / np.sqrt(fan_in)))
    out = {"x": x.contiguous(), "w": w.contiguous(), "bias": None, "residual": None,
           "residual_bias": None, "gamma": None}
    if call.epi & EPI_BIAS:
        out["bias"] = normal((call.Cout,), s + 2, std=0.1)
    if call.epi & EPI_RESIDUAL:
        L = (D, H, W)
        K = call.kernel
        Do, Ho, Wo = ((L[i] + call.pads[i][0] + call.pads[i][1] - K[i]) // call.stride[i] + 1
                      for i in range(3))
        r = to_bf16(normal((N, call.Cout, Do, Ho, Wo), s + 3))
        out["residual"] = (r if out_layout == NCDHW else r.permute(0, 2, 3, 4, 1)).contiguous()
    if call.epi & EPI_RESIDUAL_BIAS:
        out["residual_bias"] = normal((call.Cout,), s + 5, std=0.1)
    if call.epi & EPI_L2NORM_SILU:
        out["gamma"] = to_bf16(normal((call.Cout,), s + 4, mean=1.0, std=0.1)).float()
    return out
