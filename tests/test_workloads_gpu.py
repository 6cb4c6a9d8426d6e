"""Full-size parity of every workload, in the plans bench.py and users get (no
overrides), against the oracle.

* Wan chain, T=1 image-VAE layers, fused 160 blocks and the tiny case: every
  element of B(conv) is compared with the oracle's fp32 accumulator (conv
  tolerance), in both layouts where the workload has two.  The oracle runs once
  per call; the second layout reuses it (the input values are the same).
* Encoder ladder: each output feeds the next call, in NDHWC and in NCDHW.  The
  two layouts must give bit-identical outputs call by call (same plans, same
  MMA order), and the NDHWC call is checked against the oracle on its actual
  input at every border pixel of every frame, the columns beside each 128-wide
  tile boundary, the first and last output frames whole, and 65536 random pixels
  (every pixel where the output holds fewer).
* The epilogue (stage 2) is checked on the whole output of every call by running
  the oracle epilogue on the GPU's own B(conv).
"""

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_parity import (GpuCall, border_and_random_points, check_conv, check_epilogue,
                        check_points)

pytestmark = pytest.mark.gpu

# oracle accumulator of the last call checked: the two layouts of one call are
# consecutive test cases with the same input values
_ACC = {}


def _oracle_acc(name, call):
    key = (name, call.name)
    if key not in _ACC:
        _ACC.clear()
        inp = wl.make_inputs(name, call, wl.NDHWC, wl.NDHWC)
        _ACC[key] = oracle.conv3d_acc(wl.bits(inp["x"]), oracle.NDHWC, wl.bits(inp["w"]),
                                      call.stride, call.pads)
    return _ACC[key]


def _cases(name):
    w = wl.all_workloads()[name]
    return [(name, c, lay) for c in w.calls for lay in w.layouts]


@pytest.mark.parametrize("case", _cases("tiny") + _cases("wan") + _cases("t1") +
                         _cases("fused160"),
                         ids=lambda c: f"{c[0]}-{c[1].name}-{'ndhwc' if c[2][0] else 'ncdhw'}")
def test_workload_call_full_output(case):
    name, call, (lay, out_lay) = case
    inp = wl.make_inputs(name, call, lay, out_lay)
    gc = GpuCall(call, inp, lay, out_lay)
    del inp
    check_conv(gc.conv, _oracle_acc(name, call), call.name)
    check_epilogue(gc)
    del gc
    torch.cuda.empty_cache()


def test_ladder_chained_both_layouts():
    """The 30-call causal encoder ladder, each output feeding the next call."""
    w = wl.ladder()
    x_cl = x_cf = None  # previous outputs, NDHWC and NCDHW
    for call in w.calls:
        inp = wl.make_inputs("ladder", call, wl.NDHWC, wl.NDHWC, x_override=x_cf)
        gc = GpuCall(call, inp, wl.NDHWC, wl.NDHWC)
        inp_cf = wl.make_inputs("ladder", call, wl.NCDHW, wl.NCDHW, x_override=x_cf)
        gf = GpuCall(call, inp_cf, wl.NCDHW, wl.NCDHW)
        y_cl = gc.c.y.detach().cpu()
        y_cf = gf.c.y.detach().cpu()
        assert np.array_equal(wl.bits(y_cl), wl.bits(y_cf.permute(0, 2, 3, 4, 1))), \
            f"{call.name}: NCDHW and NDHWC outputs differ"
        Do, Ho, Wo = gc.c.out_dims
        pts = border_and_random_points(call.N, Do, Ho, Wo, 65536, seed=call.index)
        check_points(gc, pts)
        check_epilogue(gf)
        # next input: this call's output (NCDHW bf16 on the CPU; the NDHWC call reads
        # the same values after make_inputs permutes them)
        x_cf = y_cf
        del gc, gf, inp, inp_cf
    torch.cuda.empty_cache()
