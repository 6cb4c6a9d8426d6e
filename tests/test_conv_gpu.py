"""GPU parity of the convolution library against the CPU oracle, through the C ABI.

Small shapes are checked element by element on the whole output; they span
several M-tiles, ragged W / H tails, every padding mode (zero, causal temporal,
reflect spatial), strides 1 and 2, both layouts on both sides, narrow input and
output channels, split reductions, and each plan variant (halo / direct, K
chunk 16 / 32 / 64, tiles per CTA).  Tolerances are in tests/gpu_parity.py.
"""

import numpy as np
import pytest
import torch

import oracle
import video_vae_convolution_gb300 as vvc
import workloads as wl
from gpu_parity import GpuCall, check_conv, check_epilogue, full_reference, ulp_dist

pytestmark = pytest.mark.gpu

Z = wl.ZERO
R = wl.REFLECT
CR = ((2, 0, Z), (1, 1, R), (1, 1, R))     # causal T + reflect H, W
P1 = ((1, 1, Z),) * 3
P2D = ((0, 0, Z), (1, 1, Z), (1, 1, Z))
VALID = ((0, 0, Z),) * 3


def mk(name, N, Cin, D, H, W, Cout, kernel=(3, 3, 3), stride=(1, 1, 1), pads=P1, epi=0,
       index=0, **kw):
    return wl.ConvCall(name, N, Cin, D, H, W, Cout, kernel=kernel, stride=stride, pads=pads,
                       epi=epi, index=index, **kw)


def run_and_check(call, layout=wl.NDHWC, out_layout=wl.NDHWC, tuning=None, extra_epi=0):
    inp = wl.make_inputs("test", call, layout, out_layout)
    gc = GpuCall(call, inp, layout, out_layout, tuning=tuning, extra_epi=extra_epi)
    acc = full_reference(gc)
    check_conv(gc.conv, acc, call.name)
    check_epilogue(gc)
    return gc, acc


def test_pack_weight_bit_exact():
    for shape in [(32, 16, 3, 3, 3), (96, 3, 3, 3, 3), (3, 96, 1, 3, 3), (40, 130, 1, 1, 1)]:
        w = wl.to_bf16(wl.normal(shape, 99))
        got = vvc.pack_weight(w.cuda())
        np.testing.assert_array_equal(wl.bits(got.cpu()), oracle.pack_weight(wl.bits(w)))


BASE = mk("base", 1, 64, 3, 6, 150, 64, index=1)

# tuning: kernel 1 = pixel-major kernel, 2 = channel-major mode, 3 = pixel-major mode of
# the persistent kernel; halo 1 on, 2 off
PLAN_VARIANTS = [
    dict(kernel=2),
    dict(kernel=2, halo=1),
    dict(kernel=2, halo=2),
    dict(kernel=2, kc=32),
    dict(kernel=2, kc=16),
    dict(kernel=2, kc=32, halo=1),
    dict(kernel=2, tile_w=64, tile_h=3),
    dict(kernel=2, tile_w=128, halo=1),
    dict(kernel=2, tile_w=48, tile_h=3, halo=1),
    dict(kernel=2, tile_w=30, tile_h=4, halo=1),
    dict(kernel=2, k_splits=3),
    dict(kernel=2, halo=1, k_splits=2),
    dict(kernel=2, stages=2),
    dict(kernel=3),
    dict(kernel=3, halo=1),
    dict(kernel=3, halo=2),
    dict(kernel=3, kc=32),
    dict(kernel=3, kc=16),
    dict(kernel=3, tile_w=64, tile_h=3),
    dict(kernel=3, tile_w=48, tile_h=3, halo=1),
    dict(kernel=3, k_splits=3),
    dict(kernel=3, stages=2),
    dict(kernel=1, halo=2),
    dict(kernel=1, halo=1),
    dict(kernel=1, halo=2, kc=32),
    dict(kernel=1, halo=2, kc=16),
    dict(kernel=1, halo=1, kc=32),
    dict(kernel=1, halo=1, kc=16),
    dict(kernel=1, halo=2, R=2),
    dict(kernel=1, halo=1, R=3, BN=32),
    dict(kernel=1, halo=2, k_splits=3),
    dict(kernel=1, halo=1, k_splits=2),
    dict(kernel=1, halo=2, stages=2),
]


@pytest.mark.parametrize("tv", PLAN_VARIANTS, ids=lambda d: "-".join(f"{k}{v}" for k, v in d.items()))
def test_plan_variants(tv):
    tv = dict(tv)
    tv.setdefault("k_splits", 1)
    run_and_check(BASE, tuning=vvc.Tuning(**tv))


SHAPES = [
    mk("wide_halo_two_boxes", 1, 64, 2, 4, 250, 128, index=18),
    mk("cout200_two_channel_tiles", 1, 64, 2, 5, 90, 200, pads=CR, index=19),
    mk("wide_640_tiles", 1, 64, 3, 3, 642, 96, pads=VALID, index=20),
    mk("flat_h_zero_pad", 1, 64, 3, 7, 50, 64, pads=((2, 0, Z), (1, 1, Z), (0, 0, Z)), index=21),
    mk("flat_small_w_384", 1, 384, 3, 9, 22, 384, pads=VALID, index=22),
    mk("strip_reflect_small_w", 1, 64, 3, 12, 20, 128, pads=CR, index=23),
    mk("strip_reflect_128", 1, 128, 2, 6, 128, 96, pads=CR, index=24),
    mk("strip_zero_pad_odd", 2, 32, 2, 7, 37, 64, pads=P1, index=25),
    mk("t1_2d_tiles_h", 2, 32, 1, 9, 40, 48, kernel=(1, 3, 3), pads=P2D, index=2),
    mk("stride2_causal_reflect", 1, 32, 5, 11, 71, 32, stride=(2, 2, 2), pads=CR, index=3),
    mk("reflect_causal_wide", 1, 16, 4, 7, 133, 32, pads=CR, index=4),
    mk("narrow_cin3", 1, 3, 3, 10, 140, 96, pads=CR, index=5),
    mk("narrow_cout3", 1, 96, 1, 12, 130, 3, kernel=(1, 3, 3), pads=P2D, index=6),
    mk("pointwise", 2, 64, 2, 5, 37, 32, kernel=(1, 1, 1), pads=VALID, index=7),
    mk("down2d", 1, 32, 1, 65, 65, 32, kernel=(1, 3, 3), stride=(1, 2, 2), pads=VALID,
       zero_pad_br_input=True, index=8),
    mk("valid3d_small_w", 1, 96, 4, 10, 21, 96, pads=VALID, index=9),
    mk("stride_122", 1, 48, 3, 12, 260, 64, stride=(1, 2, 2), pads=CR, index=10),
    mk("cout48_cin1024ish", 1, 256, 2, 6, 20, 48, pads=CR, index=11),
]


@pytest.mark.parametrize("call", SHAPES, ids=lambda c: c.name)
def test_shapes(call):
    run_and_check(call)


@pytest.mark.parametrize("lay", [(wl.NCDHW, wl.NCDHW), (wl.NCDHW, wl.NDHWC), (wl.NDHWC, wl.NCDHW)])
def test_layouts_parity_and_bit_identity(lay):
    call = mk("layouts", 1, 40, 3, 7, 140, 32, pads=CR, epi=wl.EPI_BIAS, index=12)
    gc, _ = run_and_check(call, lay[0], lay[1])
    ref = GpuCall(call, wl.make_inputs("test", call, wl.NDHWC, wl.NDHWC))
    # same plan, same MMA order: the four layout combinations are bit-identical
    np.testing.assert_array_equal(oracle.from_layout(gc.y, lay[1]), ref.y)


# NCDHW output written from registers by row segments at every alignment (odd Wo:
# rows start at odd and even elements; 16-byte, 4-byte pair and 2-byte edge stores).
NCDHW_ROW_CASES = [
    mk("ncdhw_rows_odd_wo", 1, 32, 3, 6, 67, 64, pads=VALID,
       epi=wl.EPI_BIAS | wl.EPI_RESIDUAL | wl.EPI_RESIDUAL_BIAS | wl.EPI_SAVE_VALUE, index=42),
    mk("ncdhw_rows_wo_mod8_3", 1, 48, 2, 5, 77, 96, pads=CR, epi=wl.EPI_BIAS, index=43),
]


# NDHWC blocks on one output row go out through bulk tensor stores (y, value, conv);
# the rest (row ends, strip halo columns, channel tails) through the per-thread path.
TMA_STORE_CASES = [
    mk("bulk_store_bias_value", 1, 64, 3, 6, 150, 96, pads=P1,
       epi=wl.EPI_BIAS | wl.EPI_SAVE_VALUE, index=44),
    mk("bulk_store_cout200_strip", 1, 32, 2, 9, 61, 200, pads=CR, epi=wl.EPI_BIAS, index=45),
    mk("bulk_store_flat_valid", 2, 64, 3, 6, 90, 64, pads=VALID, index=46),
]


@pytest.mark.parametrize("call", TMA_STORE_CASES, ids=lambda c: c.name)
def test_bulk_store_epilogue(call):
    # one split: a split reduction writes through the separate reduction kernel
    gc, _ = run_and_check(call, wl.NDHWC, wl.NDHWC, tuning=vvc.Tuning(k_splits=1))
    assert gc.c.plan.bulk_store == 1


@pytest.mark.parametrize("call", NCDHW_ROW_CASES, ids=lambda c: c.name)
def test_ncdhw_rows(call):
    gc, _ = run_and_check(call, wl.NDHWC, wl.NCDHW)
    ref = GpuCall(call, wl.make_inputs("test", call, wl.NDHWC, wl.NDHWC))
    np.testing.assert_array_equal(oracle.from_layout(gc.y, wl.NCDHW), ref.y)


EPI_CASES = [
    mk("epi_bias_res_rbias", 1, 32, 3, 6, 140, 64, pads=P1,
       epi=wl.EPI_BIAS | wl.EPI_RESIDUAL | wl.EPI_RESIDUAL_BIAS, index=13),
    mk("epi_norm160", 1, 32, 3, 6, 140, 160, pads=P1, epi=wl.EPI_BIAS | wl.EPI_L2NORM_SILU,
       index=14),
    mk("epi_norm320_res", 1, 64, 3, 5, 70, 320, pads=P1,
       epi=wl.EPI_BIAS | wl.EPI_RESIDUAL | wl.EPI_L2NORM_SILU | wl.EPI_SAVE_VALUE, index=15),
    mk("epi_pad_br", 1, 64, 4, 9, 140, 64, pads=VALID,
       epi=wl.EPI_BIAS | wl.EPI_RESIDUAL | wl.EPI_RESIDUAL_BIAS | wl.EPI_OUT_PAD_BR, index=16),
]


@pytest.mark.parametrize("call", EPI_CASES, ids=lambda c: c.name)
@pytest.mark.parametrize("out_layout", [wl.NDHWC, wl.NCDHW])
def test_epilogues(call, out_layout):
    run_and_check(call, wl.NDHWC, out_layout)


# Fused L2 norm in the channel-major kernel (all channel tiles of a pixel tile on
# one CTA): flat, strip and direct pixel tiles; 1..4 channel tiles with a partial
# last tile; Cout not a multiple of 8; residual, residual bias and the saved value.
NORM_CM_CASES = [
    mk("norm_cm160_flat", 1, 32, 3, 7, 50, 160, pads=((2, 0, Z), (1, 1, Z), (0, 0, Z)),
       epi=wl.EPI_BIAS | wl.EPI_L2NORM_SILU, index=26),
    mk("norm_cm320_strip_res", 1, 64, 3, 5, 70, 320, pads=CR,
       epi=wl.EPI_BIAS | wl.EPI_RESIDUAL | wl.EPI_RESIDUAL_BIAS | wl.EPI_L2NORM_SILU |
       wl.EPI_SAVE_VALUE, index=27),
    mk("norm_cm200_direct_s2", 1, 32, 3, 9, 41, 200, stride=(1, 2, 2), pads=CR,
       epi=wl.EPI_BIAS | wl.EPI_L2NORM_SILU | wl.EPI_SAVE_VALUE, index=28),
    mk("norm_cm36_odd", 2, 24, 2, 5, 33, 36, pads=P1, epi=wl.EPI_RESIDUAL | wl.EPI_L2NORM_SILU,
       index=29),
    mk("norm_cm512_wide", 1, 64, 2, 3, 300, 512, pads=CR, epi=wl.EPI_BIAS | wl.EPI_L2NORM_SILU,
       index=30),
]


@pytest.mark.parametrize("call", NORM_CM_CASES, ids=lambda c: c.name)
@pytest.mark.parametrize("out_layout", [wl.NDHWC, wl.NCDHW])
def test_norm_channel_major(call, out_layout):
    run_and_check(call, wl.NDHWC, out_layout, tuning=vvc.Tuning(kernel=2, k_splits=1))


@pytest.mark.parametrize("call", [c for c in EPI_CASES if c.epi & wl.EPI_L2NORM_SILU],
                         ids=lambda c: c.name)
def test_norm_pixel_major(call):
    run_and_check(call, wl.NDHWC, wl.NDHWC, tuning=vvc.Tuning(kernel=1))


# Pixel-major mode of the persistent kernel (Cout <= 128): narrow and 96/128-channel
# outputs, every epilogue, both layouts, strip / flat / strided tiles, the fused norm.
PM_CASES = [
    mk("pm_cout3", 1, 96, 1, 12, 130, 3, kernel=(1, 3, 3), pads=P2D, index=36),
    mk("pm_cout96_strip_reflect", 1, 64, 3, 9, 70, 96, pads=CR,
       epi=wl.EPI_BIAS | wl.EPI_RESIDUAL | wl.EPI_RESIDUAL_BIAS | wl.EPI_SAVE_VALUE, index=37),
    mk("pm_cout128_flat", 1, 64, 3, 7, 50, 128, pads=((2, 0, Z), (1, 1, Z), (0, 0, Z)),
       epi=wl.EPI_BIAS, index=38),
    mk("pm_cout48_stride2", 1, 32, 3, 13, 29, 48, stride=(1, 2, 2), pads=CR, index=39),
    mk("pm_cout40_norm", 2, 24, 2, 5, 33, 40, pads=P1,
       epi=wl.EPI_BIAS | wl.EPI_RESIDUAL | wl.EPI_L2NORM_SILU | wl.EPI_SAVE_VALUE, index=40),
    mk("pm_cout64_pad_br", 1, 64, 4, 9, 140, 64, pads=VALID,
       epi=wl.EPI_BIAS | wl.EPI_RESIDUAL | wl.EPI_RESIDUAL_BIAS | wl.EPI_OUT_PAD_BR, index=41),
]


@pytest.mark.parametrize("call", PM_CASES, ids=lambda c: c.name)
@pytest.mark.parametrize("out_layout", [wl.NDHWC, wl.NCDHW])
def test_pixel_major_mode(call, out_layout):
    run_and_check(call, wl.NDHWC, out_layout, tuning=vvc.Tuning(kernel=3))


# Narrow inputs (Cin < 8, Cin * KR * KS <= 64): the spatial taps are gathered by the
# staging kernel and the convolution runs as (KT, 1, 1) over the gathered channels.
IM2COL_CASES = [
    mk("im2col_cin3_causal_reflect", 1, 3, 4, 9, 70, 96, pads=CR, index=31),
    mk("im2col_cin1_zero_bias", 2, 1, 3, 7, 33, 32, pads=P1, epi=wl.EPI_BIAS, index=32),
    mk("im2col_cin5_t1", 1, 5, 1, 17, 40, 48, kernel=(1, 3, 3), pads=P2D, index=33),
    mk("im2col_cin7_stride2", 1, 7, 3, 13, 29, 64, stride=(1, 2, 2), pads=CR, index=34),
    mk("im2col_cin3_valid_norm", 1, 3, 3, 8, 30, 160, pads=VALID,
       epi=wl.EPI_BIAS | wl.EPI_L2NORM_SILU, index=35),
]


@pytest.mark.parametrize("call", IM2COL_CASES, ids=lambda c: c.name)
@pytest.mark.parametrize("layout", [wl.NDHWC, wl.NCDHW])
def test_im2col_narrow_input(call, layout):
    gc, _ = run_and_check(call, layout, wl.NDHWC, tuning=vvc.Tuning(im2col=1))
    assert gc.c.launches >= 2  # the staged gather runs before the convolution
    assert gc.c.plan.im2col == 1


# In-kernel gather of narrow inputs (Cin * KR * KS <= 32, W stride 1): raw input rows
# copied by TMA, expanded in shared memory, resident weights; one launch.
GATHER_CASES = [
    mk("gather_cin3_causal_reflect", 1, 3, 4, 9, 64, 96, pads=CR, index=36),
    mk("gather_cin3_t1_zero", 1, 3, 1, 17, 40, 96, kernel=(1, 3, 3), pads=P2D, index=37),
    mk("gather_cin1_zero_bias", 2, 1, 3, 7, 32, 32, pads=P1, epi=wl.EPI_BIAS, index=38),
    mk("gather_cin3_wide_row", 1, 3, 3, 5, 600, 64, pads=CR, index=39),
    mk("gather_cin2_two_ctiles", 1, 2, 3, 6, 40, 200, pads=CR, epi=wl.EPI_BIAS, index=48),
    mk("gather_cin3_residual", 1, 3, 3, 8, 64, 128, pads=CR,
       epi=wl.EPI_BIAS | wl.EPI_RESIDUAL | wl.EPI_RESIDUAL_BIAS, index=49),
    mk("gather_cin3_stride_th", 1, 3, 7, 12, 48, 64, stride=(2, 2, 1), pads=CR, index=50),
    mk("gather_cin3_valid", 1, 3, 4, 8, 24, 48, pads=VALID, index=51),
    mk("gather_cin4_k322", 1, 4, 5, 9, 32, 64, kernel=(3, 2, 2),
       pads=((2, 0, Z), (1, 0, Z), (0, 1, Z)), index=52),
]


@pytest.mark.parametrize("call", GATHER_CASES, ids=lambda c: c.name)
@pytest.mark.parametrize("layout", [wl.NDHWC, wl.NCDHW])
@pytest.mark.parametrize("out_layout", [wl.NDHWC, wl.NCDHW])
def test_gather_narrow_input(call, layout, out_layout):
    # forced (automatic only with one temporal tap, where it is the faster path)
    gc, _ = run_and_check(call, layout, out_layout, tuning=vvc.Tuning(im2col=3))
    assert gc.c.launches == 1 and gc.c.plan.im2col == 2, (gc.c.launches, gc.c.plan.im2col)
    if call.kernel[0] == 1:
        auto, _ = run_and_check(call, layout, out_layout)
        assert auto.c.plan.im2col == 2


# Paired last chunks: Cin % 64 in 1..32, so the last 32-channel chunks of two tap
# pairs share a pipeline stage (odd and even pair counts, flat and strip tiles,
# reflect H, two channel tiles, three chunks, a single chunk, the fused norm).
RH = ((2, 0, Z), (1, 1, R), (0, 0, Z))    # causal T + reflect H, no W pad
ONE = vvc.Tuning(k_splits=1, pair=1)        # small cases would otherwise split the reduction
PAIR_CASES = [
    (mk("pair_96_flat_valid", 1, 96, 4, 9, 70, 96, pads=VALID, index=41), ONE),
    (mk("pair_96_strip_zero", 1, 96, 3, 11, 40, 64, index=42), ONE),
    (mk("pair_160_k2_two_ctiles", 1, 160, 3, 7, 37, 200, kernel=(2, 3, 3),
        pads=((1, 0, Z), (1, 1, Z), (1, 1, Z)), epi=wl.EPI_BIAS, index=43), ONE),
    (mk("pair_96_t1_residual", 2, 96, 1, 13, 50, 96, kernel=(1, 3, 3), pads=P2D,
        epi=wl.EPI_BIAS | wl.EPI_RESIDUAL | wl.EPI_RESIDUAL_BIAS, index=44), ONE),
    (mk("pair_96_reflect_h", 1, 96, 4, 10, 33, 96, pads=RH, index=45), ONE),
    (mk("pair_24_one_chunk", 1, 24, 3, 8, 45, 48, pads=VALID, index=46), vvc.Tuning(kc=64, k_splits=1, pair=1)),
    (mk("pair_96_norm", 1, 96, 3, 8, 40, 160, pads=VALID,
        epi=wl.EPI_BIAS | wl.EPI_L2NORM_SILU, index=47), ONE),
]


@pytest.mark.parametrize("case", PAIR_CASES, ids=lambda c: c[0].name)
@pytest.mark.parametrize("layout", [wl.NDHWC, wl.NCDHW])
def test_paired_last_chunks(case, layout):
    call, tuning = case
    gc, _ = run_and_check(call, layout, layout, tuning=tuning)
    assert gc.c.plan.kernel == 2 and gc.c.plan.paired == 1


def test_paired_off_matches_oracle():
    call = PAIR_CASES[0][0]
    gc, _ = run_and_check(call, tuning=vvc.Tuning(pair=2, k_splits=1))
    assert gc.c.plan.paired == 0


# The split reduction: 8 channels a thread with 16-byte stores when Cout % 8 == 0 (the
# partial sums of four splits loaded before they are added), 16 a thread otherwise; the
# sum always runs in split order, so the result is the same as one split's within the
# conv tolerance and deterministic.
SPLIT_CASES = [
    (mk("split_cout40_w8", 1, 64, 3, 6, 50, 40, pads=P1, epi=wl.EPI_BIAS | wl.EPI_RESIDUAL,
        index=60), 3),
    (mk("split_cout20_w16", 1, 64, 3, 6, 50, 20, pads=P1, epi=wl.EPI_BIAS, index=61), 2),
    (mk("split_cout136_six", 1, 128, 2, 5, 30, 136, pads=CR, epi=wl.EPI_BIAS, index=62), 6),
]


@pytest.mark.parametrize("case", SPLIT_CASES, ids=lambda c: c[0].name)
@pytest.mark.parametrize("out_layout", [wl.NDHWC, wl.NCDHW], ids=["ndhwc", "ncdhw"])
def test_split_reduction_widths(case, out_layout):
    call, k = case
    gc, _ = run_and_check(call, wl.NDHWC, out_layout, tuning=vvc.Tuning(k_splits=k))
    assert gc.c.plan.k_splits == k and gc.c.launches == 2
    # deterministic: the same call again gives the same bits
    rc = gc.c.run()
    assert rc == vvc.OK
    torch.cuda.synchronize()
    np.testing.assert_array_equal(wl.bits(gc.c.y.detach().cpu()), gc.y)


def test_epilogue_split_k_matches():
    call = mk("epi_split", 1, 64, 3, 5, 70, 160, pads=P1,
              epi=wl.EPI_BIAS | wl.EPI_RESIDUAL | wl.EPI_L2NORM_SILU, index=17)
    run_and_check(call, tuning=vvc.Tuning(k_splits=4))


def test_tiny_workload_full():
    for call in wl.tiny().calls:
        run_and_check(call)


def test_l2norm_silu_standalone():
    rng = np.random.default_rng(5)
    for C, rows in ((640, 1000), (160, 333), (24, 77)):
        x = wl.to_bf16(torch.from_numpy(rng.standard_normal((rows, C)).astype(np.float32)))
        res = wl.to_bf16(torch.from_numpy(rng.standard_normal((rows, C)).astype(np.float32)))
        b = torch.from_numpy((rng.standard_normal(C) * 0.1).astype(np.float32))
        rb = torch.from_numpy((rng.standard_normal(C) * 0.1).astype(np.float32))
        g = wl.to_bf16(torch.from_numpy((1 + 0.1 * rng.standard_normal(C)).astype(np.float32))).float()
        y, v = vvc.l2norm_silu(x.cuda(), g.cuda(), b.cuda(), res.cuda(), rb.cuda(), save_value=True)
        ry, rv = oracle.l2norm_silu(wl.bits(x), g.numpy(), b.numpy(), wl.bits(res), rb.numpy())
        assert ulp_dist(wl.bits(y.cpu()), ry).max() <= 3
        assert ulp_dist(wl.bits(v.cpu()), rv).max() <= 1
        y2 = vvc.l2norm_silu(x.cuda(), g.cuda())
        ry2, _ = oracle.l2norm_silu(wl.bits(x), g.numpy())
        assert ulp_dist(wl.bits(y2.cpu()), ry2).max() <= 3
