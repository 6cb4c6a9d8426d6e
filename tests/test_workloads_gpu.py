"""Full-size parity of every workload, in the plans bench.py and users get (no
overrides), against the oracle on sampled output pixels.

Sampled pixels: every border and W-tile-boundary pixel of the first and last
(n, d) planes plus random ones; at each, all output channels are compared with
the oracle's fp32 accumulator (conv tolerance).  The epilogue is checked on the
whole output by running the oracle epilogue on the GPU's own B(conv).  Chained
workloads (the encoder ladder) feed each call the previous GPU output and check
each call against the oracle on that actual input.
"""

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_parity import GpuCall, check_sampled

pytestmark = pytest.mark.gpu

# oracle MACs per sampled pixel = Cout * K: keep each call to ~2 GMAC
MAC_BUDGET = 2.0e9


def points_for(call):
    return int(max(48, min(768, MAC_BUDGET / (call.Cout * call.K))))


def _cases(name):
    w = wl.all_workloads()[name]
    return [(name, c, lay) for c in w.calls for lay in w.layouts]


@pytest.mark.parametrize("case", _cases("tiny") + _cases("wan") + _cases("fused160") +
                         _cases("t1"),
                         ids=lambda c: f"{c[0]}-{c[1].name}-{'ndhwc' if c[2][0] else 'ncdhw'}")
def test_workload_call(case):
    name, call, (lay, out_lay) = case
    inp = wl.make_inputs(name, call, lay, out_lay)
    gc = GpuCall(call, inp, lay, out_lay)
    check_sampled(gc, k=points_for(call), seed=call.index)
    del gc
    torch.cuda.empty_cache()


@pytest.mark.parametrize("lay", [wl.NDHWC, wl.NCDHW], ids=["ndhwc", "ncdhw"])
def test_ladder_chained(lay):
    """The 30-call causal encoder ladder, each output feeding the next call."""
    w = wl.ladder()
    x = None
    for call in w.calls:
        inp = wl.make_inputs("ladder", call, lay, lay, x_override=x)
        gc = GpuCall(call, inp, lay, lay)
        check_sampled(gc, k=points_for(call), seed=call.index)
        # next input: this call's output, in the same layout (bf16 on the CPU)
        y = gc.c.y.detach().cpu()
        x = y if lay == wl.NCDHW else y.permute(0, 4, 1, 2, 3).contiguous()
        del gc
    torch.cuda.empty_cache()
