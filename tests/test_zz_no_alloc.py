"""GPU test of conv3d_fwd_static_scratch, the allocation-free convolution call.

That entry point serves callers that cannot allocate device memory when they
run a convolution: it takes the scratch that conv3d_fwd would take from the
caller's workspace from a static 16 MiB device array instead.  This file is
named so that pytest collects it last.

Each case runs the regular entry point (conv3d_fwd, torch-allocated workspace)
and then the allocation-free one twice in a row, on two different inputs, and
compares the outputs within the GPU parity tolerance (|a - b| <= 2^-7 |b| + 1e-3;
the plan and the arithmetic are the same, so they are expected to match bit for
bit).  A call that needs more than the static array is rejected without launching.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
import video_vae_convolution_gb300 as vvc
import workloads as wl

pytestmark = pytest.mark.gpu

Z, R = wl.ZERO, wl.REFLECT


def _bits(t):
    return wl.bits(t.detach().cpu().contiguous())


def _within_tolerance(a_bits, b_bits):
    a = oracle.bf16_to_f32(a_bits).astype(np.float64)
    b = oracle.bf16_to_f32(b_bits).astype(np.float64)
    return bool(np.all(np.abs(a - b) <= 2.0 ** -7 * np.abs(b) + 1e-3))


def _prepare(call, layout, seed_shift, extra_epi=0, tuning=None, **kw):
    c = call
    inp = wl.make_inputs("test", wl.ConvCall(c.name, c.N, c.Cin, c.D, c.H, c.W, c.Cout,
                                             kernel=c.kernel, stride=c.stride, pads=c.pads,
                                             epi=c.epi, index=c.index + seed_shift),
                         layout, layout)
    dev = torch.device("cuda")
    g = lambda k: None if inp[k] is None else inp[k].to(dev)
    wp = vvc.pack_weight(inp["w"].to(dev))
    conv = vvc.Conv3d(inp["x"].to(dev), wp, call.Cout, call.kernel, call.stride, call.pads,
                      layout, layout, call.epi | extra_epi, bias=g("bias"),
                      residual=g("residual"), residual_bias=g("residual_bias"),
                      gamma=g("gamma"), tuning=tuning, **kw)
    conv.inputs = inp
    return conv


def _static_call(conv: vvc.Conv3d) -> int:
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return vvc._lib().conv3d_fwd_static_scratch(ctypes.byref(conv.params), stream)


CASES = [
    # NCDHW input: the scratch holds the channels-last staging copy (and partials)
    (wl.ConvCall("noalloc_ncdhw", 1, 40, 3, 10, 70, 64, pads=((2, 0, Z), (1, 1, R), (1, 1, R)),
                 epi=wl.EPI_BIAS, index=40), wl.NCDHW),
    # small layer: the scratch holds split-reduction partial sums
    (wl.ConvCall("noalloc_split", 1, 64, 2, 6, 20, 96, pads=((1, 1, Z),) * 3,
                 epi=wl.EPI_BIAS | wl.EPI_RESIDUAL, index=41), wl.NDHWC),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0].name)
def test_static_scratch_matches_regular_entry_point(case):
    call, layout = case
    # the case must actually use scratch, and fit in the static array
    c0 = _prepare(call, layout, 0)
    assert 0 < c0.workspace_bytes <= (16 << 20)
    results = []
    for shift in (0, 100):  # two calls in a row, different inputs
        c = _prepare(call, layout, shift)
        c()
        torch.cuda.synchronize()
        ref = _bits(c.y)
        c.y.fill_(float("nan"))
        rc = _static_call(c)
        assert rc == vvc.OK, vvc._lib().conv3d_status_string(rc)
        torch.cuda.synchronize()
        assert vvc.device_status() == 0
        got = _bits(c.y)
        assert _within_tolerance(got, ref)
        results.append(np.array_equal(got, ref))
    assert all(results), "same plan and arithmetic: expected identical outputs"


def test_static_scratch_rejects_oversize():
    # NCDHW staging copy of 96 x 3 x 100 x 300 bf16 = 17.3 MB > 16 MiB
    call = wl.ConvCall("noalloc_big", 1, 96, 3, 100, 300, 96, pads=((1, 1, Z),) * 3, index=42)
    c = _prepare(call, wl.NCDHW, 0)
    assert c.workspace_bytes > (16 << 20)
    c.y.fill_(1.0)
    torch.cuda.synchronize()
    rc = _static_call(c)
    assert rc == vvc.ERR_SCRATCH_LIMIT
    assert b"16 MiB" in vvc._lib().conv3d_status_string(rc)
    torch.cuda.synchronize()
    assert bool(torch.all(c.y == 1.0))


def test_static_scratch_norm_falls_back_to_pixel_major():
    """A fused-norm call whose channel-major value rows (152 CTAs x 256 pixels x 256
    channels of bf16 = 19.9 MB) do not fit the 16 MiB array runs on the pixel-major
    kernel, which needs no scratch: same output as conv3d_fwd_ex with kernel = 1,
    bit for bit, and the oracle epilogue on its own B(conv) within 3 bf16 ulp."""
    call = wl.ConvCall("noalloc_norm_fallback", 1, 32, 4, 40, 256, 256, pads=((1, 1, Z),) * 3,
                       epi=wl.EPI_BIAS | wl.EPI_L2NORM_SILU, index=43)
    c0 = _prepare(call, wl.NDHWC, 0)
    assert c0.plan.kernel == 2 and c0.workspace_bytes > (16 << 20)
    pm = _prepare(call, wl.NDHWC, 0, extra_epi=vvc.EPI_DEBUG_STORE_CONV,
                  tuning=vvc.Tuning(kernel=1))
    assert pm.workspace_bytes == 0
    for _ in range(2):  # two calls in a row
        pm()
        torch.cuda.synchronize()
        ref = _bits(pm.y)
        conv_ref = _bits(pm.conv_out)
        pm.y.fill_(float("nan"))
        pm.conv_out.fill_(float("nan"))
        rc = _static_call(pm)
        assert rc == vvc.OK, vvc._lib().conv3d_status_string(rc)
        torch.cuda.synchronize()
        assert vvc.device_status() == 0
        got = _bits(pm.y)
        assert np.array_equal(got, ref)
        assert np.array_equal(_bits(pm.conv_out), conv_ref)
    inp = pm.inputs
    e = oracle.epilogue(_bits(pm.conv_out), oracle.BIAS | oracle.L2NORM_SILU,
                        inp["bias"].numpy(), None, None, inp["gamma"].numpy())
    ordinal = lambda u: np.where(u & 0x8000, -(u.astype(np.int32) & 0x7FFF),
                                 u.astype(np.int32) & 0x7FFF)
    assert np.abs(ordinal(got) - ordinal(e["act"])).max() <= 3


def test_static_scratch_pad_cache():
    """Padded output + cache: the contiguous activations that the last launch places
    live in the static array.  Same padded output and cache as conv3d_fwd."""
    call = wl.ConvCall("noalloc_pad_cache", 1, 16, 4, 8, 16, 32, pads=((1, 1, Z),) * 3,
                       epi=wl.EPI_BIAS | wl.EPI_L2NORM_SILU, index=44)
    for shift in (0, 100):
        c = _prepare(call, wl.NDHWC, shift, extra_epi=vvc.EPI_PAD_CACHE, history_frames=1)
        assert 0 < c.workspace_bytes <= (16 << 20)
        c.y.fill_(3.0)
        c.cache_out.fill_(3.0)
        c()
        torch.cuda.synchronize()
        ref_y, ref_c = _bits(c.y), _bits(c.cache_out)
        c.y.fill_(3.0)
        c.cache_out.fill_(3.0)
        rc = _static_call(c)
        assert rc == vvc.OK, vvc._lib().conv3d_status_string(rc)
        torch.cuda.synchronize()
        assert vvc.device_status() == 0
        assert np.array_equal(_bits(c.y), ref_y)
        assert np.array_equal(_bits(c.cache_out), ref_c)
