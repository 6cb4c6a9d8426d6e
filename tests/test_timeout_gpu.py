"""Failure detection on the GPU without a fault: a bounded wait that runs out.

The test aid `conv3d_tuning.inject` makes the TMA producer leave one pipeline
stage unissued, so the MMA thread's wait on it can never complete.  With a
200 ms limit every affected CTA records CONV3D_ERR_DEVICE_TIMEOUT, drains its
copies and MMAs, frees its TMEM and returns; the host reads the status word,
and the context stays usable for the next call.
"""

import time

import numpy as np
import pytest
import torch

import video_vae_convolution_gb300 as vvc
import workloads as wl
from gpu_parity import GpuCall, check_conv, full_reference

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kernel", [1, 2], ids=["pixel_major", "channel_major"])
def test_bounded_wait_reports_timeout(kernel):
    call = wl.ConvCall("timeout_case", 1, 64, 2, 4, 64, 64, pads=((1, 1, wl.ZERO),) * 3, index=60)
    inp = wl.make_inputs("test", call)
    dev = torch.device("cuda")
    x = inp["x"].to(dev)
    wp = vvc.pack_weight(inp["w"].to(dev))
    assert vvc.device_status() == vvc.OK
    bad = vvc.Conv3d(x, wp, call.Cout, call.kernel, call.stride, call.pads,
                     tuning=vvc.Tuning(kernel=kernel, inject=1, timeout_ms=200, k_splits=1))
    t0 = time.time()
    assert bad.run() == vvc.OK            # the launch itself is valid
    status = vvc.device_status()          # synchronises, reads and clears the word
    assert time.time() - t0 < 20.0
    assert status == vvc.ERR_DEVICE_TIMEOUT
    assert vvc.device_status() == vvc.OK  # cleared
    # the context is still usable: a normal call completes with correct results
    gc = GpuCall(call, inp)
    check_conv(gc.conv, full_reference(gc), call.name)
