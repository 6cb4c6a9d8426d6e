"""GPU cases of the fused and standalone L2-norm / SiLU at its two degenerate
points (cuDNN frontend doc "Fused Conv3D + Bias + Residual + RMSNorm + SiLU",
"Operation Contract"):

* an all-zero value row: den = max(sqrt(0), 1e-12) = 1e-12, every normalised
  value 0, and the activation 0 / (1 + exp(0)) = +0 in every channel;
* a row whose affine value lies far below -88: exp(-affine) overflows to +inf in
  fp32 and the activation affine / (1 + inf) is -0.

Through conv3d_fwd the rows are made exactly: the input is zero over a block of
the volume, so the output pixels whose receptive field lies inside it have
conv = 0 exactly, and there the value is the residual (no bias): zero rows, rows
with a single negative entry (normalised to -1, scaled to -sqrt(C), times
gamma = 20 -> about -113) and ordinary rows.  Every plan that computes the fused
norm runs: the channel-major kernel (both output layouts), the pixel-major
kernel, the pixel-major mode of the persistent kernel and the split reduction.
The oracle epilogue on the GPU's own B(conv) must agree within 3 bf16 ulp
everywhere, and the degenerate rows must be +0 / -0 bit for bit.
"""

import numpy as np
import pytest
import torch

import oracle
import video_vae_convolution_gb300 as vvc
import workloads as wl
from gpu_parity import GpuCall, check_epilogue, ulp_dist

pytestmark = pytest.mark.gpu

Z = wl.ZERO
P1 = ((1, 1, Z),) * 3
POS_ZERO, NEG_ZERO = 0x0000, 0x8000


def _gamma(C, seed):
    g = wl.to_bf16(wl.normal((C,), seed, mean=1.0, std=0.1)).float()
    g[0::2] = 20.0  # even channels: a one-hot -1 row overflows exp there
    return g


def _edge_inputs(call, out_layout, seed):
    """Input zero over d < D, h < 6, w < 20; residual rows of three kinds inside the
    output block h < 5, w < 19 (zero, one-hot negative on an even channel,
    ordinary) and N(0, 1) elsewhere."""
    inp = wl.make_inputs("test", call, wl.NDHWC, wl.NDHWC)
    x = inp["x"].clone()
    x[:, :, :6, :20, :] = 0
    inp["x"] = x
    Do, Ho, Wo = call.out_dims()
    C = call.Cout
    res = wl.to_bf16(wl.normal((call.N, Do, Ho, Wo, C), seed + 3))
    kind = np.zeros((call.N, Do, Ho, Wo), dtype=np.int8)  # 0 ordinary, 1 zero, 2 one-hot
    hot = np.zeros((call.N, Do, Ho, Wo), dtype=np.int64)
    rng = np.random.default_rng(seed)
    for n in range(call.N):
        for d in range(Do):
            for h in range(5):
                for w in range(19):
                    k = (h * 19 + w + d) % 3
                    kind[n, d, h, w] = k
                    if k == 1:
                        res[n, d, h, w, :] = 0
                    elif k == 2:
                        c = 2 * int(rng.integers(C // 2))
                        hot[n, d, h, w] = c
                        res[n, d, h, w, :] = 0
                        res[n, d, h, w, c] = -float(rng.uniform(0.25, 3.0))
    inp["residual"] = res if out_layout == wl.NDHWC else res.permute(0, 4, 1, 2, 3).contiguous()
    inp["gamma"] = _gamma(C, seed + 4)
    return inp, kind, hot


def _check_degenerate(y_ndhwc, kind, hot):
    zero_rows = y_ndhwc[kind == 1]
    assert zero_rows.size and np.all(zero_rows == POS_ZERO), "zero rows must give +0"
    oh = np.nonzero(kind == 2)
    rows = y_ndhwc[oh]
    c = hot[oh]
    assert rows.size
    assert np.all(rows[np.arange(rows.shape[0]), c] == NEG_ZERO), "overflowed exp must give -0"
    rest = rows.copy()
    rest[np.arange(rows.shape[0]), c] = POS_ZERO
    assert np.all(rest == POS_ZERO), "the other channels of a one-hot row are +0"


PLANS = [
    ("channel_major", None, wl.NDHWC),
    ("channel_major_ncdhw", None, wl.NCDHW),
    ("pixel_major_kernel", dict(kernel=1), wl.NDHWC),
    ("pixel_major_mode", dict(kernel=3), wl.NDHWC),
    ("split_reduction", dict(k_splits=3), wl.NDHWC),
]


@pytest.mark.parametrize("plan", PLANS, ids=lambda p: p[0])
@pytest.mark.parametrize("C", [32, 160])
def test_fused_norm_degenerate_rows(plan, C):
    name, tune, out_layout = plan
    if tune and tune.get("kernel") == 3 and C > 128:
        pytest.skip("pixel-major mode covers Cout <= 128")
    call = wl.ConvCall(f"norm_edge_{C}", 1, 16, 3, 10, 40, C, pads=P1,
                       epi=wl.EPI_RESIDUAL | wl.EPI_L2NORM_SILU, index=60 + C)
    inp, kind, hot = _edge_inputs(call, out_layout, 7000 + C)
    gc = GpuCall(call, inp, wl.NDHWC, out_layout,
                 tuning=vvc.Tuning(**tune) if tune else None)
    # conv is exactly zero where the receptive field lies in the zero block
    assert np.all((gc.conv[kind > 0] & 0x7FFF) == 0)
    check_epilogue(gc)
    y = oracle.from_layout(gc.y, out_layout)
    _check_degenerate(y, kind, hot)


@pytest.mark.parametrize("C", [640, 160, 36])
def test_standalone_norm_degenerate_rows(C):
    rows = 999
    rng = np.random.default_rng(C)
    x = rng.standard_normal((rows, C)).astype(np.float32)
    kind = np.arange(rows) % 3
    hot = 2 * rng.integers(C // 2, size=rows)
    x[kind == 1] = 0
    for r in np.nonzero(kind == 2)[0]:
        x[r] = 0
        x[r, hot[r]] = -rng.uniform(0.25, 3.0)
    xb = wl.to_bf16(torch.from_numpy(x))
    g = _gamma(C, 90 + C)
    y = wl.bits(vvc.l2norm_silu(xb.cuda(), g.cuda()).cpu())
    ref, _ = oracle.l2norm_silu(wl.bits(xb), g.numpy())
    assert ulp_dist(y, ref).max() <= 3
    _check_degenerate(y.reshape(1, 1, 1, rows, C), kind.reshape(1, 1, 1, rows),
                      hot.reshape(1, 1, 1, rows))
