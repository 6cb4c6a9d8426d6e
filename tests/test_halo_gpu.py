"""GPU tests of the output halo (conv3d_params.out_halo): the convolution writes
its output inside a larger NDHWC tensor whose one-pixel H / W border holds the
reflection of the output (or zeros), so that the next call of a chain reads it
as an already padded input and runs a valid convolution (ROCm/FlyDSL issue
"[Feature]: conv3d_implicit — ...", MiniMax-H3 comment: causal temporal zero pad
and reflect spatial pad before every encoder convolution).

Each case runs the same call twice, without and with the halo: the output inside
the haloed tensor must equal the plain output bit for bit (same plan, same MMA
order); the halo rows and columns must be what PyTorch 'reflect' (or zero)
padding of that output gives, corners included; the leading and trailing T halo
frames must keep the caller's contents.  The plain output is checked against the
oracle (conv tolerance, and the oracle epilogue on the GPU's own B(conv)).

The encoder ladder is then run as a chain of haloed tensors: every call after the
first reads the previous haloed output as a valid convolution, and is checked
against the oracle (original padding on the unpadded input) at every border
pixel, the first and last frames and 65536 random pixels.
"""

import numpy as np
import pytest
import torch

import oracle
import video_vae_convolution_gb300 as vvc
import workloads as wl
from gpu_parity import (GpuCall, border_and_random_points, check_conv, check_epilogue,
                        check_points, full_reference)

pytestmark = pytest.mark.gpu

Z, R = wl.ZERO, wl.REFLECT
CR = ((2, 0, Z), (1, 1, R), (1, 1, R))
VALID = ((0, 0, Z),) * 3
LADDER_HALO = ((2, 0, Z), (1, 1, R), (1, 1, R))
# the chain form the benchmark runs: a spatial halo only, and every later call applies
# the causal T padding itself (its kernel leaves out the all-padding temporal taps)
HW_HALO = ((0, 0, Z), (1, 1, R), (1, 1, R))
CAUSAL_T = ((2, 0, Z), (0, 0, Z), (0, 0, Z))
CHAIN_FORMS = {"t_halo": (LADDER_HALO, VALID, 2), "t_pad": (HW_HALO, CAUSAL_T, 0)}
SENTINEL = 0x40E0  # bf16 7.0: the caller's contents of the T halo frames


def _bits(t):
    return wl.bits(t.detach().cpu().contiguous())


def _expected_halo(y, halo):
    """numpy: y [N, D, H, W, C] bits -> haloed tensor with the T halo = SENTINEL."""
    (tb, ta, _), (hb, ha, hm), (wb, wa, wm) = halo
    N, D, H, W, C = y.shape
    out = np.full((N, D + tb + ta, H + hb + ha, W + wb + wa, C), SENTINEL, dtype=np.uint16)
    pad_h = (hb, ha)
    pad_w = (wb, wa)
    mode = {R: "reflect", Z: "constant"}
    t = np.pad(y, ((0, 0), (0, 0), pad_h, (0, 0), (0, 0)), mode=mode[hm])
    t = np.pad(t, ((0, 0), (0, 0), (0, 0), pad_w, (0, 0)), mode=mode[wm])
    out[:, tb:tb + D] = t
    return out


CASES = [
    # (call, tuning, halo)
    (wl.ConvCall("halo_strip_reflect", 1, 32, 4, 10, 40, 64, pads=CR, epi=wl.EPI_BIAS, index=70),
     None, LADDER_HALO),
    (wl.ConvCall("halo_strip_bulk", 1, 32, 4, 10, 40, 64, pads=CR, index=88),
     dict(k_splits=1), LADDER_HALO),
    (wl.ConvCall("halo_flat_valid", 1, 64, 5, 12, 34, 96, pads=VALID, index=71), None,
     LADDER_HALO),
    (wl.ConvCall("halo_flat_bulk", 1, 64, 5, 12, 34, 96, pads=VALID, index=89),
     dict(k_splits=1), LADDER_HALO),
    (wl.ConvCall("halo_zero_bulk", 1, 32, 3, 9, 20, 32, pads=((1, 1, Z),) * 3, index=90),
     dict(k_splits=1), ((1, 1, Z), (1, 1, Z), (1, 1, Z))),
    (wl.ConvCall("halo_zero_mode", 1, 32, 3, 9, 20, 32, pads=((1, 1, Z),) * 3, index=72), None,
     ((1, 1, Z), (1, 1, Z), (1, 1, Z))),
    (wl.ConvCall("halo_asym", 1, 16, 3, 7, 19, 48, pads=CR, epi=wl.EPI_BIAS, index=73), None,
     ((0, 2, Z), (1, 0, R), (0, 1, R))),
    (wl.ConvCall("halo_h3", 1, 32, 3, 3, 70, 32, pads=CR, index=74), None, LADDER_HALO),
    (wl.ConvCall("halo_residual", 1, 64, 3, 8, 36, 64, pads=CR,
                 epi=wl.EPI_BIAS | wl.EPI_RESIDUAL | wl.EPI_RESIDUAL_BIAS, index=75),
     dict(k_splits=1), LADDER_HALO),
    (wl.ConvCall("halo_residual_split", 1, 64, 3, 8, 36, 64, pads=CR,
                 epi=wl.EPI_BIAS | wl.EPI_RESIDUAL | wl.EPI_RESIDUAL_BIAS, index=91), None,
     LADDER_HALO),
    (wl.ConvCall("halo_split", 1, 128, 3, 6, 6, 128, pads=CR, epi=wl.EPI_BIAS, index=76),
     dict(k_splits=3), LADDER_HALO),
    (wl.ConvCall("halo_pixel_major", 1, 32, 3, 8, 24, 64, pads=CR, index=77), dict(kernel=1),
     LADDER_HALO),
    (wl.ConvCall("halo_pm_mode", 1, 32, 3, 8, 24, 16, pads=CR, index=78), dict(kernel=3),
     LADDER_HALO),
    (wl.ConvCall("halo_stride2", 1, 32, 5, 12, 40, 64, stride=(2, 2, 2), pads=CR, index=79),
     None, LADDER_HALO),
    (wl.ConvCall("halo_narrow_in", 1, 3, 4, 16, 64, 32, pads=CR, index=80), None, LADDER_HALO),
]


FLAT3_CASES = [
    # valid convolutions over small planes: the tiles run across frames
    (wl.ConvCall("flat3_valid", 1, 64, 6, 10, 10, 64, pads=VALID, epi=wl.EPI_BIAS, index=82),
     dict(k_splits=1)),
    (wl.ConvCall("flat3_valid_split", 1, 64, 6, 10, 10, 64, pads=VALID, epi=wl.EPI_BIAS,
                 index=87), None),
    (wl.ConvCall("flat3_causal_t", 1, 128, 5, 9, 11, 96, pads=((2, 0, Z), (0, 0, Z), (0, 0, Z)),
                 index=83), None),
    (wl.ConvCall("flat3_split", 1, 256, 7, 18, 18, 256, pads=VALID, epi=wl.EPI_BIAS, index=84),
     None),
    (wl.ConvCall("flat3_paired", 1, 96, 6, 12, 12, 64, pads=VALID, index=85), dict(k_splits=1)),
    (wl.ConvCall("flat3_residual", 1, 64, 4, 8, 8, 32, pads=VALID,
                 epi=wl.EPI_BIAS | wl.EPI_RESIDUAL, index=86), None),
]


# Compact volume tiles (conv3d_tuning.compact): the flattened volume without the input
# rows below each frame's last output row, read through a TMA im2col map.  Tiles span
# frames (and, past the last one, the next batch item's rows or the zero fill).
COMPACT_CASES = [
    (wl.ConvCall("compact_two_ctiles", 1, 128, 6, 12, 14, 136, pads=CAUSAL_T, epi=wl.EPI_BIAS,
                 index=92), dict(k_splits=1)),
    (wl.ConvCall("compact_batch2", 2, 64, 4, 10, 10, 64, pads=CAUSAL_T, index=93),
     dict(k_splits=1)),
    (wl.ConvCall("compact_split", 1, 256, 5, 18, 18, 128, pads=CAUSAL_T, epi=wl.EPI_BIAS,
                 index=94), None),
    (wl.ConvCall("compact_kt1", 1, 64, 5, 10, 12, 64, kernel=(1, 3, 3), pads=VALID, index=95),
     dict(k_splits=1)),
    (wl.ConvCall("compact_t_both", 1, 64, 5, 10, 10, 64, pads=((1, 1, Z), (0, 0, Z), (0, 0, Z)),
                 index=96), None),
]


def _compact_form(call):
    """The volume-tile form a compact request plans: the compact one when every
    64-channel chunk is whole (its im2col copies are planned only for those), else the
    tiled one."""
    return 3 if call.Cin % 64 == 0 else 2


def _flat_form(call, inp, tune, compact):
    tuning = vvc.Tuning(**dict(tune or {}, compact=compact))
    gc = GpuCall(call, inp, wl.NDHWC, wl.NDHWC, tuning=tuning)
    if compact == 1:
        assert gc.c.plan.flat == _compact_form(call), call.name
    return gc, tuning


@pytest.mark.parametrize("case", FLAT3_CASES + COMPACT_CASES, ids=lambda c: c[0].name)
def test_flat_volume_tiles(case):
    """Both forms of volume tiles on the same inputs: the tiled map over the whole
    volume (halo rows included) and the compact im2col form; each against the oracle,
    and bit for bit equal to each other where their stage schedules are the same."""
    call, tune = case
    inp = wl.make_inputs("test", call, wl.NDHWC, wl.NDHWC)
    tiled, _ = _flat_form(call, inp, tune, 2)
    if call.name.startswith("flat3"):
        assert tiled.c.plan.flat == 2, call.name
    if call.name == "flat3_paired":
        assert tiled.c.plan.paired == 1
    comp, tuning = _flat_form(call, inp, tune, 1)
    form = _compact_form(call)
    if form == 3:
        assert comp.c.plan.paired == 0
    ref = full_reference(comp)
    check_conv(comp.conv, ref, call.name + " compact")
    check_epilogue(comp)
    if tiled.c.plan.paired or tiled.c.plan.k_splits != comp.c.plan.k_splits:
        check_conv(tiled.conv, ref, call.name + " tiled")
        check_epilogue(tiled)
    else:
        np.testing.assert_array_equal(comp.conv, tiled.conv)
        np.testing.assert_array_equal(comp.y, tiled.y)
    # and into a haloed tensor: the same output inside it
    dev = torch.device("cuda")
    Do, Ho, Wo = comp.c.out_dims
    y = torch.full((call.N, Do + 2, Ho + 2, Wo + 2, call.Cout), 7.0, dtype=torch.bfloat16,
                   device=dev)
    g = lambda k: None if inp[k] is None else inp[k].to(dev)
    c = vvc.Conv3d(inp["x"].to(dev), comp.w_packed, call.Cout, call.kernel, call.stride,
                   call.pads, wl.NDHWC, wl.NDHWC, call.epi, bias=g("bias"),
                   residual=g("residual"), y=y, out_halo=LADDER_HALO, tuning=tuning)
    assert c.plan.flat == form
    c()
    torch.cuda.synchronize()
    assert vvc.device_status() == 0
    np.testing.assert_array_equal(_bits(y), _expected_halo(comp.y, LADDER_HALO))


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0].name)
def test_output_halo(case):
    call, tune, halo = case
    tuning = vvc.Tuning(**tune) if tune else None
    inp = wl.make_inputs("test", call, wl.NDHWC, wl.NDHWC)
    plain = GpuCall(call, inp, wl.NDHWC, wl.NDHWC, tuning=tuning)
    check_conv(plain.conv, full_reference(plain), call.name)
    check_epilogue(plain)
    # the same call writing into a haloed tensor prefilled with the sentinel
    dev = torch.device("cuda")
    Do, Ho, Wo = plain.c.out_dims
    (tb, ta, _), (hb, ha, _), (wb, wa, _) = halo
    y = torch.full((1, Do + tb + ta, Ho + hb + ha, Wo + wb + wa, call.Cout), 7.0,
                   dtype=torch.bfloat16, device=dev)
    g = lambda k: None if inp[k] is None else inp[k].to(dev)
    c = vvc.Conv3d(inp["x"].to(dev), plain.w_packed, call.Cout, call.kernel, call.stride,
                   call.pads, wl.NDHWC, wl.NDHWC, call.epi, bias=g("bias"),
                   residual=g("residual"), residual_bias=g("residual_bias"), y=y,
                   tuning=tuning, out_halo=halo)
    assert c.plan.mma_n == plain.c.plan.mma_n and c.plan.k_splits == plain.c.plan.k_splits
    c()
    torch.cuda.synchronize()
    assert vvc.device_status() == 0
    np.testing.assert_array_equal(_bits(y), _expected_halo(plain.y, halo))


def test_output_halo_rejected_combinations():
    call = wl.ConvCall("halo_bad", 1, 16, 3, 6, 16, 32, pads=CR, index=81)
    inp = wl.make_inputs("test", call, wl.NDHWC, wl.NDHWC)
    dev = torch.device("cuda")
    x = inp["x"].to(dev)
    wp = vvc.pack_weight(inp["w"].to(dev))
    bad = [
        dict(out_halo=LADDER_HALO, out_layout=wl.NCDHW),            # NDHWC only
        dict(out_halo=((1, 0, R), (1, 1, R), (1, 1, R))),           # T halo is not written
        dict(out_halo=((0, 0, Z), (2, 2, R), (1, 1, R))),           # at most one pixel
        dict(out_halo=LADDER_HALO, epi=wl.EPI_L2NORM_SILU),         # not with the norm
    ]
    for kw in bad:
        out_layout = kw.pop("out_layout", wl.NDHWC)
        epi = kw.pop("epi", 0)
        with pytest.raises(vvc.Conv3dError):
            vvc.Conv3d(x, wp, 32, (3, 3, 3), (1, 1, 1), CR, wl.NDHWC, out_layout, epi,
                       gamma=torch.ones(32, device=dev),
                       y=torch.zeros((1, 6, 8, 18, 32), dtype=torch.bfloat16, device=dev), **kw)


@pytest.mark.parametrize("form", sorted(CHAIN_FORMS))
def test_ladder_chained_through_halos(form):
    """The 30-call encoder ladder with haloed intermediates: conv_in reads the model
    input with its causal + reflect padding and writes a haloed output; every
    later call reads the previous haloed tensor, as a valid convolution (t_halo: two
    zero frames lead each intermediate) or with the causal T padding applied by the
    call itself (t_pad: spatial halo only)."""
    halo, later_pads, lead = CHAIN_FORMS[form]
    dev = torch.device("cuda")
    w = wl.ladder()
    prev = None          # previous haloed output (device)
    prev_plain = None    # its output inside the halo (CPU, NCDHW) = the oracle's input
    for i, call in enumerate(w.calls):
        last = i == len(w.calls) - 1
        inp = wl.make_inputs("ladder", call, wl.NDHWC, wl.NDHWC, x_override=prev_plain)
        wp = vvc.pack_weight(inp["w"].to(dev))
        if prev is None:
            x, pads = inp["x"].to(dev), call.pads
        else:
            x, pads = prev, later_pads
        Do, Ho, Wo = call.out_dims()
        if last:
            c = vvc.Conv3d(x, wp, call.Cout, call.kernel, call.stride, pads, wl.NDHWC, wl.NDHWC,
                           vvc.EPI_DEBUG_STORE_CONV)
        else:
            y = torch.full((1, Do + lead, Ho + 2, Wo + 2, call.Cout), 7.0, dtype=torch.bfloat16,
                           device=dev)
            y[:, :lead] = 0
            c = vvc.Conv3d(x, wp, call.Cout, call.kernel, call.stride, pads, wl.NDHWC, wl.NDHWC,
                           vvc.EPI_DEBUG_STORE_CONV, y=y, out_halo=halo)
        if prev is not None:
            assert c.plan.launches == 1 + (1 if c.plan.k_splits > 1 else 0), call.name
        c()
        torch.cuda.synchronize()
        assert vvc.device_status() == 0
        conv = _bits(c.conv_out)
        out = _bits(c.y)
        inner = out if last else out[:, lead:, 1:-1, 1:-1, :]
        # no epilogue ops: the output is B(conv) itself
        np.testing.assert_array_equal(inner, conv)
        if not last:
            exp = _expected_halo(inner, halo)
            exp[:, :lead] = 0
            np.testing.assert_array_equal(out, exp)
        # the oracle on the unpadded input with the call's own padding
        xb = wl.bits(inp["x"])
        pts = border_and_random_points(1, Do, Ho, Wo, 65536, seed=call.index)
        acc = oracle.conv3d_acc_points(xb, wl.NDHWC, wl.bits(inp["w"]), pts, call.stride,
                                       call.pads)
        check_conv(conv[pts[:, 0], pts[:, 1], pts[:, 2], pts[:, 3]], acc, call.name)
        prev = c.y
        prev_plain = torch.from_numpy(inner.view(np.int16)).view(torch.bfloat16).permute(
            0, 4, 1, 2, 3).contiguous()
        del c
    torch.cuda.empty_cache()
