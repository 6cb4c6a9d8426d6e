"""GPU parity of the FP8 e4m3fn convolution (conv3d_params.dtype = E4M3) against the
oracle (ROCm/FlyDSL PR "[Flydsl] Add Qwen-Image VAE classic conv shapes to conv3d
tests", "Summary" / "Test shapes": e4m3fn activations and weights, fp32 bias, bf16
output).

The oracle convolves the exact values of the e4m3 codes (fp64 sums), multiplies the
fp32 accumulator by the per-tensor scale and runs the same epilogue as for bf16, so
every check uses the bf16 path's tolerances (tests/gpu_parity.py): B(conv) within
2^-7 |ref| + 1e-3 on every output element, the oracle epilogue on the GPU's own
B(conv) within 1 ulp (3 ulp for the fused L2 norm / SiLU).  Inputs are the seeded
bf16 recipe quantised to e4m3 with power-of-two per-tensor scales
(workloads.make_inputs_e4m3).
"""

import numpy as np
import pytest
import torch

import oracle
import video_vae_convolution_gb300 as vvc
import workloads as wl
from gpu_parity import check_conv, orc_flags, ulp_dist

pytestmark = pytest.mark.gpu

Z, R = wl.ZERO, wl.REFLECT
CR = ((2, 0, Z), (1, 1, R), (1, 1, R))
SAME = ((1, 1, Z),) * 3
HALO = ((2, 0, Z), (1, 1, R), (1, 1, R))


def _bits(t):
    return wl.bits(t.detach().cpu().contiguous())


class F8Call:
    """One e4m3 call through the C ABI, with the debug B(conv) store."""

    def __init__(self, call, inp, out_layout=wl.NDHWC, tuning=None, y=None, out_halo=None,
                 debug_conv=True):
        dev = torch.device("cuda")
        g = lambda k: None if inp[k] is None else inp[k].to(dev).contiguous()
        self.w_packed = vvc.pack_weight_e4m3(inp["w8"].to(dev))
        epi = call.epi | (vvc.EPI_DEBUG_STORE_CONV if debug_conv else 0)
        self.c = vvc.Conv3d(inp["x8"].to(dev), self.w_packed, call.Cout, call.kernel,
                            call.stride, call.pads, wl.NDHWC, out_layout, epi, bias=g("bias"),
                            residual=g("residual"), residual_bias=g("residual_bias"),
                            gamma=g("gamma"), tuning=tuning, y=y, out_halo=out_halo,
                            dtype=vvc.DTYPE_E4M3, fp8_scale=inp["scale"])
        rc = self.c.run()
        assert rc == vvc.OK, vvc._lib().conv3d_status_string(rc)
        torch.cuda.synchronize()
        assert vvc.device_status() == 0
        self.y = _bits(self.c.y)
        self.conv = None if self.c.conv_out is None else _bits(self.c.conv_out)


def _acc(call, inp):
    return oracle.conv3d_acc_e4m3(inp["x8"].numpy(), oracle.NDHWC, inp["w8"].numpy(),
                                  inp["scale"], call.stride, call.pads)


def _check_epilogue(call, inp, conv_bits, y_bits, out_layout):
    np_or_none = lambda t: None if t is None else t.numpy()
    res = None
    if inp["residual"] is not None:
        res = oracle.from_layout(wl.bits(inp["residual"]), out_layout)
    e = oracle.epilogue(conv_bits, orc_flags(call.epi), np_or_none(inp["bias"]), res,
                        np_or_none(inp["residual_bias"]), np_or_none(inp["gamma"]))
    y = oracle.from_layout(y_bits, out_layout)
    if call.epi & wl.EPI_L2NORM_SILU:
        assert ulp_dist(y, e["act"]).max() <= 3
    else:
        assert ulp_dist(y, e["value"]).max() <= 1


CASES = [
    # (call, out_layout, tuning): every e4m3 plan shape on small sizes that still span
    # several tiles and a ragged tail
    (wl.ConvCall("f8_c16_same", 1, 16, 3, 10, 20, 32, pads=SAME, epi=wl.EPI_BIAS, index=0),
     wl.NDHWC, None),
    (wl.ConvCall("f8_c96_causal_reflect", 1, 96, 4, 12, 40, 96, pads=CR, epi=wl.EPI_BIAS,
                 index=1), wl.NDHWC, None),
    (wl.ConvCall("f8_c160_256_split", 1, 160, 1, 20, 30, 256, kernel=(1, 3, 3),
                 pads=((0, 0, Z), (1, 1, Z), (1, 1, Z)), epi=wl.EPI_BIAS, index=2),
     wl.NDHWC, dict(k_splits=3)),
    (wl.ConvCall("f8_c128_flat", 1, 128, 5, 18, 18, 128, pads=((0, 0, Z),) * 3, index=3),
     wl.NDHWC, None),
    (wl.ConvCall("f8_c64_norm", 1, 64, 3, 9, 33, 64, pads=CR,
                 epi=wl.EPI_BIAS | wl.EPI_L2NORM_SILU, index=4), wl.NDHWC, None),
    (wl.ConvCall("f8_c32_stride2", 1, 32, 5, 17, 34, 64, stride=(1, 2, 2), pads=CR,
                 epi=wl.EPI_BIAS, index=5), wl.NDHWC, None),
    (wl.ConvCall("f8_c48_residual_ncdhw_out", 1, 48, 3, 8, 24, 40, pads=SAME,
                 epi=wl.EPI_BIAS | wl.EPI_RESIDUAL | wl.EPI_RESIDUAL_BIAS, index=6),
     wl.NCDHW, None),
    (wl.ConvCall("f8_c256_512_small_m", 1, 256, 3, 8, 8, 512, pads=CR, epi=wl.EPI_BIAS,
                 index=7), wl.NDHWC, None),
    # compact volume tiles (im2col map) with e4m3 operands: a spatially haloed input with
    # the causal T padding in the call, tiles straddling frames
    (wl.ConvCall("f8_c128_compact", 1, 128, 5, 18, 18, 128,
                 pads=((2, 0, Z), (0, 0, Z), (0, 0, Z)), epi=wl.EPI_BIAS, index=13),
     wl.NDHWC, dict(compact=1, k_splits=1)),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0].name)
def test_e4m3_conv_parity(case):
    call, out_layout, tune = case
    inp = wl.make_inputs_e4m3("test", call)
    if out_layout == wl.NCDHW and inp["residual"] is not None:
        inp["residual"] = inp["residual"].permute(0, 4, 1, 2, 3).contiguous()
    gc = F8Call(call, inp, out_layout, vvc.Tuning(**tune) if tune else None)
    if tune and "k_splits" in tune:
        assert gc.c.plan.k_splits == tune["k_splits"]
    if tune and tune.get("compact") == 1:
        assert gc.c.plan.flat == 3
    check_conv(gc.conv, _acc(call, inp), call.name)
    _check_epilogue(call, inp, gc.conv, gc.y, out_layout)


def test_e4m3_pack_weight_bit_exact():
    call = wl.ConvCall("f8_pack", 1, 144, 1, 4, 4, 40, index=8)
    inp = wl.make_inputs_e4m3("test", call)
    got = vvc.pack_weight_e4m3(inp["w8"].cuda()).cpu().numpy()
    np.testing.assert_array_equal(got, oracle.pack_weight_e4m3(inp["w8"].numpy()))


def test_e4m3_output_halo():
    # a valid convolution of a haloed input writing a haloed output (the chained form)
    call = wl.ConvCall("f8_halo", 1, 128, 5, 18, 34, 128, pads=((0, 0, Z),) * 3,
                       epi=wl.EPI_BIAS, index=9)
    inp = wl.make_inputs_e4m3("test", call)
    plain = F8Call(call, inp)
    check_conv(plain.conv, _acc(call, inp), call.name)
    Do, Ho, Wo = plain.c.out_dims
    y = torch.full((1, Do + 2, Ho + 2, Wo + 2, call.Cout), 7.0, dtype=torch.bfloat16,
                   device="cuda")
    F8Call(call, inp, y=y, out_halo=HALO, debug_conv=False)
    got = _bits(y)
    assert np.all(got[:, :2] == 0x40E0)           # T halo frames are left as they were
    t = np.pad(plain.y, ((0, 0), (0, 0), (1, 1), (0, 0), (0, 0)), mode="reflect")
    t = np.pad(t, ((0, 0), (0, 0), (0, 0), (1, 1), (0, 0)), mode="reflect")
    np.testing.assert_array_equal(got[:, 2:], t)


def test_e4m3_scale_enters_once():
    # the same codes with scales s and 2 s: every B(conv) doubles exactly (a power of two
    # scales a bf16 value without rounding), so the scale is applied once, before B()
    call = wl.ConvCall("f8_scale", 1, 64, 2, 6, 20, 64, pads=SAME, index=10)
    inp = wl.make_inputs_e4m3("test", call)
    a = F8Call(call, inp).conv
    inp2 = dict(inp)
    inp2["scale"] = inp["scale"] * 2.0
    b = F8Call(call, inp2).conv
    np.testing.assert_array_equal(oracle.bf16_to_f32(b), 2.0 * oracle.bf16_to_f32(a))


def test_e4m3_full_size_t1_384():
    # the T = 1 image layer 384 -> 384 at 256^2 (FlyDSL PR "Test shapes"), every element
    call = [c for c in wl.t1().calls if c.name == "t1_384_256"][0]
    inp = wl.make_inputs_e4m3("t1", call)
    gc = F8Call(call, inp)
    check_conv(gc.conv, _acc(call, inp), call.name)
    _check_epilogue(call, inp, gc.conv, gc.y, wl.NDHWC)


def test_e4m3_full_size_ladder_l0_sampled():
    # the ladder's 128 -> 128 layer at [17, 256, 256], causal + reflect padding: every
    # border pixel, the first and last frames and 64k random pixels (all channels)
    from gpu_parity import border_and_random_points
    call = wl.ladder().calls[1]
    inp = wl.make_inputs_e4m3("ladder", call)
    gc = F8Call(call, inp)
    Do, Ho, Wo = gc.c.out_dims
    pts = border_and_random_points(1, Do, Ho, Wo, 65536, seed=5)
    acc = oracle.conv3d_acc_points(oracle.e4m3_to_bf16(inp["x8"].numpy()), oracle.NDHWC,
                                   oracle.e4m3_to_bf16(inp["w8"].numpy()), pts, call.stride,
                                   call.pads)
    acc = (acc.astype(np.float64) * float(np.float32(inp["scale"]))).astype(np.float32)
    check_conv(gc.conv[pts[:, 0], pts[:, 1], pts[:, 2], pts[:, 3]], acc, call.name)
    _check_epilogue(call, inp, gc.conv, gc.y, wl.NDHWC)
