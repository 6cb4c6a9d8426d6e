"""Padded output and two-frame cache (cuDNN frontend doc "Fused Conv3D + Bias +
Residual + RMSNorm + SiLU", "Normalization and Padding Variant" and "Standalone
Normalization and Padding Variant") on the GPU.

Convolution variant: the same call is run once with contiguous output (checked
against the oracle like every other call) and once with the padded output and
cache, on buffers prefilled with a sentinel.  The padded call must equal the
oracle's placement rules applied to the contiguous call's activations, bit for
bit: the arithmetic is the same and only the destinations differ.

Standalone variant: checked against the oracle (post-operations within 3 bf16
ulp, value within 1, zeros and history copies exact) and against the GPU's own
contiguous l2norm_silu bit for bit.
"""

import numpy as np
import pytest
import torch

import oracle
import video_vae_convolution_gb300 as vvc
import workloads as wl
from gpu_parity import GpuCall, bits, check_conv, check_epilogue, full_reference, ulp_dist

pytestmark = pytest.mark.gpu

Z = wl.ZERO
VALID = ((0, 0, Z),) * 3
NORM = wl.EPI_BIAS | wl.EPI_L2NORM_SILU
SENTINEL = 0x3F80  # bf16 1.0 in every byte pair a call must leave alone

CONV_CASES = [
    # (call, tuning): fused-norm channel-major kernel, split reduction, pixel-major kernel
    (wl.ConvCall("padc_norm", 1, 32, 5, 7, 9, 40, pads=VALID, epi=NORM, index=61), None),
    (wl.ConvCall("padc_res_value", 2, 16, 4, 6, 10, 64, pads=VALID,
                 epi=NORM | wl.EPI_RESIDUAL | wl.EPI_RESIDUAL_BIAS, index=62),
     vvc.Tuning(k_splits=2)),
    (wl.ConvCall("padc_pixel_major", 1, 24, 3, 8, 8, 48, pads=VALID, epi=NORM, index=63),
     vvc.Tuning(kernel=1)),
]


@pytest.mark.parametrize("case", CONV_CASES, ids=lambda c: c[0].name)
@pytest.mark.parametrize("P", [0, 1, 2])
def test_conv_padded_output_and_cache(case, P):
    call, tuning = case
    inp = wl.make_inputs("test", call)
    save = bool(call.epi & wl.EPI_RESIDUAL)  # residual_output: the saved value
    gc = GpuCall(call, inp, tuning=tuning,  # contiguous, oracle-checked
                 extra_epi=vvc.EPI_SAVE_VALUE if save else 0)
    check_conv(gc.conv, full_reference(gc), call.name)
    check_epilogue(gc)
    dev = torch.device("cuda")
    N, Cout = call.N, call.Cout
    Do, Ho, Wo = gc.c.out_dims
    K = min(2, Do + P)
    y = torch.full((N, Do + 2, Ho + 2, Wo + 2, Cout), 1.0, dtype=torch.bfloat16, device=dev)
    cache = torch.full((N, K, Ho, Wo, Cout), 1.0, dtype=torch.bfloat16, device=dev)
    g = lambda k: None if inp[k] is None else inp[k].to(dev)
    c = vvc.Conv3d(inp["x"].to(dev), vvc.pack_weight(inp["w"].to(dev)), Cout, call.kernel,
                   call.stride, call.pads, wl.NDHWC, wl.NDHWC,
                   call.epi | vvc.EPI_PAD_CACHE | (vvc.EPI_SAVE_VALUE if save else 0),
                   bias=g("bias"), residual=g("residual"), residual_bias=g("residual_bias"),
                   gamma=g("gamma"), y=y, cache_out=cache, history_frames=P, tuning=tuning)
    assert c.launches == gc.c.launches + 1
    c()
    torch.cuda.synchronize()
    act = gc.y  # the contiguous call's activations, NDHWC bits
    ref_padded, ref_cache = oracle.pad_cache_fused(
        act, P, np.full(tuple(y.shape), SENTINEL, np.uint16),
        np.full(tuple(cache.shape), SENTINEL, np.uint16))
    np.testing.assert_array_equal(bits(y.cpu()), ref_padded)
    np.testing.assert_array_equal(bits(cache.cpu()), ref_cache)
    if save:  # residual_output: the pre-normalisation value, unpadded
        np.testing.assert_array_equal(bits(c.value_out.cpu()), gc.value)


@pytest.mark.parametrize("P", [0, 1, 2])
@pytest.mark.parametrize("shape", [(1, 1, 5, 7, 16), (2, 3, 4, 6, 40), (1, 4, 3, 130, 24)])
def test_standalone_padded_output_and_cache(shape, P):
    N, T, H, W, C = shape
    rng = np.random.default_rng(100 * P + T)
    f = lambda a: wl.to_bf16(torch.from_numpy(a.astype(np.float32)))
    x = f(rng.standard_normal(shape))
    res = f(rng.standard_normal(shape))
    b = torch.from_numpy((rng.standard_normal(C) * 0.1).astype(np.float32))
    rb = torch.from_numpy((rng.standard_normal(C) * 0.1).astype(np.float32))
    gamma = f(1 + 0.1 * rng.standard_normal(C)).float()
    prev = f(rng.standard_normal((N, P, H, W, C))) if P else None
    dev = torch.device("cuda")
    cu = lambda t: None if t is None else t.to(dev)
    padded, cache, value = vvc.l2norm_silu_pad(cu(x), cu(gamma), cu(b), cu(res), cu(rb),
                                               previous=cu(prev), save_value=True)
    ref_act, ref_value = oracle.l2norm_silu(wl.bits(x), gamma.numpy(), b.numpy(), wl.bits(res),
                                            rb.numpy())
    ref_padded, ref_cache = oracle.pad_cache_standalone(
        ref_act, None if prev is None else wl.bits(prev))
    got_padded, got_cache = bits(padded.cpu()), bits(cache.cpu())
    assert got_padded.shape == ref_padded.shape and got_cache.shape == ref_cache.shape
    assert ulp_dist(got_padded, ref_padded).max() <= 3
    assert ulp_dist(got_cache, ref_cache).max() <= 3
    assert ulp_dist(bits(value.cpu()), ref_value).max() <= 1
    border = np.ones((H + 2, W + 2), bool)
    border[1:-1, 1:-1] = False
    assert not got_padded[:, :, border].any() and not got_padded[:, :2 - P].any()
    if P:
        np.testing.assert_array_equal(got_padded[:, 2 - P:2, 1:-1, 1:-1], wl.bits(prev))
    # the same post-operations as the contiguous standalone call, bit for bit
    y = vvc.l2norm_silu(cu(x), cu(gamma), cu(b), cu(res), cu(rb))
    np.testing.assert_array_equal(got_padded[:, 2:, 1:-1, 1:-1], bits(y.cpu()))
