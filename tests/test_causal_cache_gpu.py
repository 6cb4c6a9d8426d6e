"""GPU tests of the streaming causal convolution (cuDNN frontend doc "Fused Conv3D +
Bias + Residual + RMSNorm + SiLU", section "Causal Conv3D with Cache", and the
CausalConv3dWithCacheSm100 row of its API table: input/history packing with
padding, then the 12 -> 160 convolution without bias).

* conv3d_causal_pack against oracle.causal_pack, bit for bit, on strided views of the
  chunk (the page takes strided NCTHW chunks) with 0, 1 and 2 history frames; every
  output element is written (the buffers start as a sentinel).
* A video run chunk by chunk through CausalConv3dWithCache (each chunk after the
  previous chunk's cache) against the oracle's causal convolution of the whole video,
  at the conv tolerance of gpu_parity; the caches are the video's last frames.
"""

import numpy as np
import pytest
import torch

import oracle
import video_vae_convolution_gb300 as vvc
import workloads as wl
from gpu_parity import bits, check_conv

pytestmark = pytest.mark.gpu

SENTINEL = 0x7F7F  # a bf16 value the packer never writes


def _rand_bf16(gen, shape, scale=1.0):
    return (torch.randn(shape, generator=gen) * scale).to(torch.bfloat16)


def _view(base_shape, kind, gen):
    """A chunk [N, C, T, H, W] as a strided view of a larger tensor."""
    N, C, T, H, W = base_shape
    dev = torch.device("cuda")
    if kind == "contiguous":
        return _rand_bf16(gen, (N, C, T, H, W)).to(dev)
    if kind == "t_slice":  # frames 1 .. T of a longer clip
        return _rand_bf16(gen, (N, C, T + 3, H, W)).to(dev)[:, :, 1:T + 1]
    if kind == "channels_last":  # an NTHWC tensor seen as NCTHW (channel stride 1)
        return _rand_bf16(gen, (N, T, H, W, C)).to(dev).permute(0, 4, 1, 2, 3)
    if kind == "w_step2":  # every other column
        return _rand_bf16(gen, (N, C, T, H, 2 * W)).to(dev)[..., ::2]
    raise ValueError(kind)


PACK_CASES = [
    # (N, C, T, H, W, P, Cp, view)
    (1, 12, 4, 10, 14, 0, 16, "contiguous"),
    (1, 12, 4, 10, 14, 1, 16, "t_slice"),
    (1, 12, 4, 10, 14, 2, 16, "channels_last"),
    (2, 12, 1, 7, 9, 2, 16, "w_step2"),
    (1, 12, 1, 6, 5, 1, 16, "contiguous"),
    (1, 3, 3, 8, 8, 2, 8, "t_slice"),
    (1, 12, 4, 104, 180, 2, 16, "contiguous"),
]


@pytest.mark.parametrize("case", PACK_CASES, ids=lambda c: "x".join(map(str, c[:5])) +
                         f"_P{c[5]}_{c[7]}")
def test_causal_pack_bit_exact(case):
    N, C, T, H, W, P, Cp, kind = case
    gen = torch.Generator().manual_seed(N * 1000 + C * 100 + T * 10 + P)
    x = _view((N, C, T, H, W), kind, gen)
    dev = x.device
    prev = _rand_bf16(gen, (N, P, H, W, C)).to(dev) if P else None
    K = min(2, T + P)
    padded = torch.full((N, T + 2, H + 2, W + 2, Cp), 0, dtype=torch.int16, device=dev)
    padded.fill_(SENTINEL)
    cache = torch.full((N, K, H, W, C), SENTINEL, dtype=torch.int16, device=dev)
    vvc.causal_pack(x, prev, Cp, padded.view(torch.bfloat16), cache.view(torch.bfloat16))
    torch.cuda.synchronize()
    ref_padded, ref_cache = oracle.causal_pack(bits(x), None if prev is None else bits(prev),
                                               Cp=Cp)
    got_padded = padded.cpu().numpy().view(np.uint16)
    got_cache = cache.cpu().numpy().view(np.uint16)
    np.testing.assert_array_equal(got_padded, ref_padded)
    np.testing.assert_array_equal(got_cache, ref_cache)


@pytest.mark.parametrize("chunks", [(1, 4, 4), (2, 1, 3)])
def test_streaming_conv_is_the_whole_causal_conv(chunks):
    # 12 -> 160 as on the page; each chunk after the previous chunk's cache
    N, C, H, W, Co = 1, 12, 10, 14, 160
    T = sum(chunks)
    gen = torch.Generator().manual_seed(7 + T)
    video = _rand_bf16(gen, (N, C, T, H, W)).cuda()
    w = _rand_bf16(gen, (Co, C, 3, 3, 3), (C * 27) ** -0.5).cuda()
    wp = vvc.pack_weight(w)
    outs, prev, t0 = [], None, 0
    for tc in chunks:
        P = 0 if prev is None else prev.shape[1]
        call = vvc.CausalConv3dWithCache((N, C, tc, H, W), wp, Co, history_frames=P)
        assert call.conv.plan.kernel == 2
        y, cache = call(video[:, :, t0:t0 + tc], prev)
        torch.cuda.synchronize()
        assert vvc.device_status() == 0
        outs.append(bits(y))
        t0 += tc
        K = min(2, t0)
        ref_cache = bits(video[:, :, t0 - K:t0].permute(0, 2, 3, 4, 1))
        np.testing.assert_array_equal(bits(cache), ref_cache)
        prev = cache.clone()
    got = np.concatenate(outs, axis=1)
    Z = oracle.PAD_ZERO
    ref = oracle.conv3d_acc(bits(video), oracle.NCDHW, bits(w), (1, 1, 1),
                            ((2, 0, Z), (1, 1, Z), (1, 1, Z)))
    check_conv(got, ref, f"streaming {chunks}")


def test_causal_conv_page_shape():
    # one 4-frame chunk with two history frames at [104, 180] (the 160-channel blocks'
    # plane), every output against the oracle's valid convolution of the packed input
    N, C, T, H, W, Co = 1, 12, 4, 104, 180, 160
    gen = torch.Generator().manual_seed(11)
    x = _rand_bf16(gen, (N, C, T, H, W)).cuda()
    prev = _rand_bf16(gen, (N, 2, H, W, C)).cuda()
    w = _rand_bf16(gen, (Co, C, 3, 3, 3), (C * 27) ** -0.5).cuda()
    call = vvc.CausalConv3dWithCache((N, C, T, H, W), vvc.pack_weight(w), Co, history_frames=2)
    y, cache = call(x, prev)
    torch.cuda.synchronize()
    assert vvc.device_status() == 0
    padded, ref_cache = oracle.causal_pack(bits(x), bits(prev), Cp=16)
    np.testing.assert_array_equal(bits(call.padded), padded)
    np.testing.assert_array_equal(bits(cache), ref_cache)
    w16 = np.zeros((Co, 16, 3, 3, 3), np.uint16)
    w16[:, :C] = bits(w)
    ref = oracle.conv3d_acc(padded, oracle.NDHWC, w16)
    check_conv(bits(y), ref, "causal 12->160 [4, 104, 180]")
