"""GPU test of vvc.Chain: a fixed sequence of calls recorded as one CUDA graph gives
the same outputs, bit for bit, as the calls issued one by one, and picks up new input
values written in place between replays."""

import numpy as np
import pytest
import torch

import video_vae_convolution_gb300 as vvc
import workloads as wl

pytestmark = pytest.mark.gpu

Z, R = wl.ZERO, wl.REFLECT
HALO = ((2, 0, Z), (1, 1, R), (1, 1, R))
VALID = ((0, 0, Z),) * 3


def _bits(t):
    return wl.bits(t.detach().cpu().contiguous())


def test_chain_graph_matches_eager():
    dev = torch.device("cuda")
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    x = torch.randn((1, 5, 12, 40, 32), generator=g, device=dev).to(torch.bfloat16)
    w1 = (torch.randn((64, 32, 3, 3, 3), generator=g, device=dev) * 0.05).to(torch.bfloat16)
    w2 = (torch.randn((48, 64, 3, 3, 3), generator=g, device=dev) * 0.05).to(torch.bfloat16)
    bias = 0.1 * torch.randn(48, generator=g, device=dev)
    c1 = vvc.Conv3d(x, vvc.pack_weight(w1), 64, (3, 3, 3), (1, 1, 1), HALO, wl.NDHWC,
                    wl.NDHWC, 0, out_halo=HALO)
    c2 = vvc.Conv3d(c1.y, vvc.pack_weight(w2), 48, (3, 3, 3), (1, 1, 1), VALID, wl.NDHWC,
                    wl.NDHWC, vvc.EPI_BIAS, bias=bias, tuning=vvc.Tuning(k_splits=2))
    chain = vvc.Chain([c1, c2])
    assert chain.launches == c1.launches + c2.launches >= 3   # c2 adds its split reduction
    for step in range(2):
        if step:
            x.copy_(torch.randn(x.shape, generator=g, device=dev).to(torch.bfloat16))
        c1()
        c2()
        torch.cuda.synchronize()
        ref1, ref2 = _bits(c1.y), _bits(c2.y)
        c1.y[:, 2:].fill_(3.0)       # the T halo frames stay zero (the next call's pad)
        c2.y.fill_(3.0)
        chain.run()
        torch.cuda.synchronize()
        assert vvc.device_status() == 0
        np.testing.assert_array_equal(_bits(c1.y), ref1)
        np.testing.assert_array_equal(_bits(c2.y), ref2)
