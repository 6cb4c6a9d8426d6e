"""The production epilogue paths, which run only without the debug conv store.

Every parity test in test_conv_gpu.py asks for the debug store of B(conv)
(CONV3D_EPI_DEBUG_STORE_CONV), which the oracle's epilogue check needs.  Some
store paths are taken only without it: the NDHWC bulk tensor store of y alone
(without the conv map), the NCDHW bulk tensor stores (blocks on one output row
starting at a column that is a multiple of 8) and the NCDHW 16-byte vector stores.  Here each call runs
twice on the same inputs and plan, with and without the debug store.  The debug
run is checked against the oracle as everywhere else.  The run without it must
give the same y and value bit for bit, since the arithmetic is the same.
"""

import numpy as np
import pytest

import video_vae_convolution_gb300 as vvc
import workloads as wl
from gpu_parity import GpuCall, check_conv, check_epilogue, full_reference

pytestmark = pytest.mark.gpu

Z, R = wl.ZERO, wl.REFLECT
CR = ((2, 0, Z), (1, 1, R), (1, 1, R))
P1 = ((1, 1, Z),) * 3
VALID = ((0, 0, Z),) * 3


def mk(name, N, Cin, D, H, W, Cout, pads=P1, epi=0, index=0, **kw):
    return wl.ConvCall(name, N, Cin, D, H, W, Cout, pads=pads, epi=epi, index=index, **kw)


ONE = vvc.Tuning(k_splits=1)  # bulk stores need one split (small cases would split)

# (call, output layout[, tuning]); names with "bulk" must plan bulk stores
CASES = [
    # NDHWC bulk stores (y only; with the saved value), strip and flat tiles
    (mk("prod_ndhwc_bulk_bias", 1, 64, 3, 6, 150, 96, epi=wl.EPI_BIAS, index=50), wl.NDHWC,
     ONE),
    (mk("prod_ndhwc_bulk_value", 1, 32, 2, 9, 61, 200, pads=CR,
        epi=wl.EPI_BIAS | wl.EPI_SAVE_VALUE, index=51), wl.NDHWC, ONE),
    (mk("prod_ndhwc_bulk_flat", 2, 64, 3, 6, 90, 64, pads=VALID, index=52), wl.NDHWC, ONE),
    # NDHWC per-thread path: residual and the bottom/right pad
    (mk("prod_ndhwc_res_pad", 1, 64, 4, 9, 140, 64, pads=VALID,
        epi=wl.EPI_BIAS | wl.EPI_RESIDUAL | wl.EPI_RESIDUAL_BIAS | wl.EPI_OUT_PAD_BR,
        index=53), wl.NDHWC),
    # NCDHW vector stores (W multiple of 8) and the per-pixel path (odd W)
    (mk("prod_ncdhw_aligned", 1, 48, 4, 6, 66, 64, pads=VALID,
        epi=wl.EPI_BIAS | wl.EPI_RESIDUAL | wl.EPI_SAVE_VALUE, index=54), wl.NCDHW),
    (mk("prod_ncdhw_odd", 1, 32, 3, 6, 67, 64, pads=VALID, epi=wl.EPI_BIAS, index=55),
     wl.NCDHW),
    # NCDHW bulk stores: flat tiles (Wo = 64), blocks across rows and a channel tile
    # past Cout (Wo = 88, Cout = 200) with the saved value, and strip tiles 36 columns
    # wide (w0 = 36 starts off the 8-column grid: per-pixel fallback; 0 and 72 on it)
    (mk("prod_ncdhw_bulk_flat", 1, 64, 3, 6, 66, 96, pads=VALID, epi=wl.EPI_BIAS, index=58),
     wl.NCDHW, ONE),
    (mk("prod_ncdhw_bulk_cout200", 1, 32, 3, 5, 90, 200, pads=VALID,
        epi=wl.EPI_BIAS | wl.EPI_SAVE_VALUE, index=59), wl.NCDHW, ONE),
    (mk("prod_ncdhw_bulk_strip_tw36", 1, 32, 2, 7, 112, 64, pads=CR, index=60), wl.NCDHW,
     vvc.Tuning(tile_w=36, tile_h=2, halo=1, k_splits=1)),
    # fused norm (channel-major passes), both layouts
    (mk("prod_norm_ndhwc", 1, 32, 3, 7, 50, 160, pads=((2, 0, Z), (1, 1, Z), (0, 0, Z)),
        epi=wl.EPI_BIAS | wl.EPI_L2NORM_SILU | wl.EPI_SAVE_VALUE, index=56), wl.NDHWC),
    (mk("prod_norm_ncdhw", 1, 64, 3, 5, 70, 320, pads=CR,
        epi=wl.EPI_BIAS | wl.EPI_L2NORM_SILU, index=57), wl.NCDHW),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0].name)
def test_production_path_matches_debug_run(case):
    call, out_layout = case[:2]
    tuning = case[2] if len(case) > 2 else None
    inp = wl.make_inputs("test", call, wl.NDHWC, out_layout)
    dbg = GpuCall(call, inp, wl.NDHWC, out_layout, tuning=tuning, debug_conv=True)
    check_conv(dbg.conv, full_reference(dbg), call.name)
    check_epilogue(dbg)
    prod = GpuCall(call, inp, wl.NDHWC, out_layout, tuning=tuning, debug_conv=False)
    assert prod.conv is None
    if "_bulk" in call.name:
        assert prod.c.plan.bulk_store == 1
        if out_layout == wl.NCDHW:  # not beside the NDHWC debug store
            assert dbg.c.plan.bulk_store == 0
    np.testing.assert_array_equal(prod.y, dbg.y)
    if dbg.value is not None:
        np.testing.assert_array_equal(prod.value, dbg.value)
