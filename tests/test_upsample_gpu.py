"""GPU parity of the convolution that reads the nearest-exact x2 upsampling of its
input (conv3d_params.input_upsample = 2; ROCm/FlyDSL PR "[Flydsl] Add Qwen-Image
VAE classic conv shapes to conv3d tests", "Upsample Conv2d": the decoder's 3x3,
stride-1, pad-1 convolution after nearest-exact x2).  The upsampled tensor is
never written: each of the four output parity classes is a convolution of the
low-resolution input with its own row / column tap offsets.

Stage 1 compares every element of the GPU's B(conv) with the oracle's plain
definition (upsample, then convolve) within the conv tolerance; stage 2 runs the
oracle epilogue on the GPU's own B(conv).  The production run (bulk tensor stores
of each class through a strided map of y) must give the same y bit for bit as the
checked run (per-thread stores beside the debug conv store).
"""

import numpy as np
import pytest
import torch

import oracle
import video_vae_convolution_gb300 as vvc
import workloads as wl
from gpu_parity import GpuCall, check_conv, check_epilogue

pytestmark = pytest.mark.gpu

Z = wl.ZERO
P2D = ((0, 0, Z), (1, 1, Z), (1, 1, Z))


def up_call(name, Cin, D, H, W, Cout, kernel=(1, 3, 3), pads=P2D, epi=wl.EPI_BIAS, index=0):
    return wl.ConvCall(name, 1, Cin, D, H, W, Cout, kernel=kernel, pads=pads, epi=epi,
                       upsample=2, index=index)


CASES = [
    up_call("up_small", 64, 1, 7, 9, 32, index=1),
    up_call("up_strips", 64, 1, 20, 150, 64, index=2),
    up_call("up_two_ctiles", 96, 1, 6, 40, 200, index=3),
    up_call("up_no_bias", 32, 1, 9, 33, 48, epi=0, index=4),
    up_call("up_3d_causal", 32, 4, 6, 10, 64, kernel=(3, 3, 3),
            pads=((2, 0, Z), (1, 1, Z), (1, 1, Z)), index=5),
]


def _reference(gc):
    call = gc.call
    xb = oracle.from_layout(gc.x_bits(), gc.layout)
    return oracle.conv3d_acc(oracle.upsample2x_nearest(xb), oracle.NDHWC, gc.w_bits(),
                             call.stride, call.pads)


def _run(call, inp, layout, debug):
    return GpuCall(call, inp, layout, wl.NDHWC, debug_conv=debug,
                   extra_kw={"input_upsample": 2})


def _check(name, call, layout):
    inp = wl.make_inputs(name, call, layout, wl.NDHWC)
    gc = _run(call, inp, layout, True)
    assert gc.c.out_dims[1:] == (2 * call.H, 2 * call.W)
    assert gc.c.launches == 1 + (layout == wl.NCDHW)
    check_conv(gc.conv, _reference(gc), call.name)
    check_epilogue(gc)
    prod = _run(call, inp, layout, False)
    assert prod.c.plan.bulk_store == 1
    np.testing.assert_array_equal(prod.y, gc.y)
    return gc


@pytest.mark.parametrize("call", CASES, ids=lambda c: c.name)
@pytest.mark.parametrize("layout", [wl.NDHWC, wl.NCDHW], ids=["ndhwc", "ncdhw"])
def test_upsample_conv(call, layout):
    _check("test", call, layout)


@pytest.mark.parametrize("call", wl.up2().calls, ids=lambda c: c.name)
def test_upsample_decoder_shapes_full_output(call):
    """The pages' decoder upsample convolutions at full size, every output element."""
    _check("up2", call, wl.NDHWC)
    torch.cuda.empty_cache()


def test_upsample_rejected_combinations():
    call = up_call("up_bad", 16, 1, 6, 8, 32)
    inp = wl.make_inputs("test", call, wl.NDHWC, wl.NDHWC)
    dev = torch.device("cuda")
    x = inp["x"].to(dev)
    wp = vvc.pack_weight(inp["w"].to(dev))
    bad = [
        dict(pads=((0, 0, Z), (0, 0, Z), (1, 1, Z))),           # pad 1 along H and W only
        dict(pads=((0, 0, Z), (1, 1, wl.REFLECT), (1, 1, Z))),  # zero padding
        dict(out_layout=wl.NCDHW),                              # NDHWC output
        dict(stride=(1, 2, 2)),                                  # stride 1 along H and W
        dict(epi=wl.EPI_RESIDUAL),                               # no residual
    ]
    for kw in bad:
        pads = kw.get("pads", P2D)
        with pytest.raises(vvc.Conv3dError):
            vvc.Conv3d(x, wp, 32, (1, 3, 3), kw.get("stride", (1, 1, 1)), pads, wl.NDHWC,
                       kw.get("out_layout", wl.NDHWC), kw.get("epi", 0),
                       residual=torch.zeros((1, 1, 12, 16, 32), dtype=torch.bfloat16,
                                            device=dev),
                       input_upsample=2)
