"""Pins of the CPU oracle against things other than itself.

Each check ties the oracle to a fact fixed outside it: numpy / torch library
routines (explicit padding + tap sums, torch fp64 conv3d, matmul, bf16
rounding, F.normalize, F.silu), closed forms, the T=1 causal identity from the
ROCm/FlyDSL PR "[Flydsl] Add Qwen-Image VAE classic conv shapes to conv3d
tests" ("T=1 degeneration"), the output-shape rules of the cuDNN frontend doc
"Fused Conv3D + Bias + Residual + RMSNorm + SiLU" ("Raw Conv3D Variant",
"Spatial Padding Variant") and hand-worked epilogue values
(tests/golden/epilogue_cases.txt).
"""

import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_bits_from_f32(a):
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def rand_bf16(rng, shape, scale=1.0):
    return bf16_bits_from_f32(rng.standard_normal(shape).astype(np.float32) * scale)


def to_f64(orc, bits):
    return orc.bf16_to_f32(bits).astype(np.float64)


# ---- brute force: explicit padding, then a tap-by-tap valid correlation --------------

def brute_conv(x_ncdhw, w, stride, pads):
    """float64 reference written without the oracle's index arithmetic:
    materialise the padded tensor with numpy.pad, then sum shifted slices."""
    xp = x_ncdhw
    for axis, (b, a, mode) in zip((2, 3, 4), pads):
        widths = [(0, 0)] * 5
        widths[axis] = (b, a)
        xp = np.pad(xp, widths, mode="reflect" if mode == wl.REFLECT else "constant")
    N, C, D, H, W = xp.shape
    Co, _, KT, KR, KS = w.shape
    st, sh, sw = stride
    Do = (D - KT) // st + 1
    Ho = (H - KR) // sh + 1
    Wo = (W - KS) // sw + 1
    out = np.zeros((N, Co, Do, Ho, Wo), dtype=np.float64)
    for t in range(KT):
        for r in range(KR):
            for s in range(KS):
                sl = xp[:, :, t:t + st * (Do - 1) + 1:st, r:r + sh * (Ho - 1) + 1:sh,
                        s:s + sw * (Wo - 1) + 1:sw]
                out += np.einsum("ncdhw,oc->nodhw", sl, w[:, :, t, r, s])
    return out.transpose(0, 2, 3, 4, 1)  # NDHWC


def torch_conv(x_ncdhw, w, stride, pads):
    """float64 torch.nn.functional.conv3d after F.pad (reflect and zero)."""
    x = torch.from_numpy(x_ncdhw)
    (tb, ta, tm), (hb, ha, hm), (wb, wa, wm) = pads
    # spatial pads first (reflect or zero), then the temporal pad
    if hm == wl.REFLECT or wm == wl.REFLECT:
        assert hm == wm
        x = F.pad(x, (wb, wa, hb, ha, 0, 0), mode="reflect")
    else:
        x = F.pad(x, (wb, wa, hb, ha, 0, 0))
    if tm == wl.REFLECT:
        x = F.pad(x, (0, 0, 0, 0, tb, ta), mode="reflect")
    else:
        x = F.pad(x, (0, 0, 0, 0, tb, ta))
    y = F.conv3d(x, torch.from_numpy(w), stride=stride)
    return y.numpy().transpose(0, 2, 3, 4, 1)


CASES = [
    # (N, C, D, H, W, Co, kernel, stride, pads)
    (1, 3, 3, 5, 6, 4, (3, 3, 3), (1, 1, 1), ((0, 0, 0),) * 3),
    (2, 5, 4, 6, 5, 3, (3, 3, 3), (1, 1, 1), ((1, 1, 0),) * 3),
    (1, 16, 5, 6, 6, 8, (3, 3, 3), (1, 1, 1), ((2, 0, 0), (1, 1, 1), (1, 1, 1))),
    (1, 1, 6, 5, 4, 2, (3, 3, 3), (2, 2, 2), ((2, 0, 0), (1, 1, 1), (1, 1, 1))),
    (1, 3, 2, 6, 6, 5, (1, 3, 3), (1, 2, 2), ((0, 0, 0), (0, 0, 0), (0, 0, 0))),
    (1, 5, 3, 7, 7, 2, (3, 3, 3), (1, 2, 2), ((2, 0, 0), (1, 1, 1), (1, 1, 1))),
    (2, 3, 1, 4, 4, 3, (1, 3, 3), (1, 1, 1), ((0, 0, 0), (1, 1, 0), (1, 1, 0))),
    (1, 4, 3, 3, 3, 4, (1, 1, 1), (1, 1, 1), ((0, 0, 0),) * 3),
    (1, 2, 4, 2, 2, 3, (3, 3, 3), (1, 1, 1), ((2, 0, 0), (1, 1, 1), (1, 1, 1))),
]


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("layout", [wl.NCDHW, wl.NDHWC])
def test_brute_force_and_torch(orc, case, layout):
    N, C, D, H, W, Co, k, stride, pads = case
    rng = np.random.default_rng(hash((case, layout)) % (2 ** 32))
    xb = rand_bf16(rng, (N, C, D, H, W))
    wb = rand_bf16(rng, (Co, C) + k, 0.3)
    x_in = xb if layout == wl.NCDHW else np.ascontiguousarray(xb.transpose(0, 2, 3, 4, 1))
    acc = orc.conv3d_acc(x_in, layout, wb, stride, pads)
    ref_b = brute_conv(to_f64(orc, xb), to_f64(orc, wb), stride, pads)
    ref_t = torch_conv(to_f64(orc, xb), to_f64(orc, wb), stride, pads)
    assert acc.shape == ref_b.shape
    # bf16 products are exact in fp64 and these sums stay far inside 53 bits,
    # so all three agree exactly once rounded to fp32.
    np.testing.assert_array_equal(acc, ref_b.astype(np.float32))
    np.testing.assert_array_equal(acc, ref_t.astype(np.float32))


def test_points_match_full(orc):
    rng = np.random.default_rng(7)
    xb = rand_bf16(rng, (2, 8, 5, 7, 9))
    wb = rand_bf16(rng, (6, 8, 3, 3, 3), 0.2)
    pads = ((2, 0, 0), (1, 1, 1), (1, 1, 1))
    full = orc.conv3d_acc(xb, wl.NCDHW, wb, (1, 1, 1), pads)
    pts = np.array([[0, 0, 0, 0], [1, 4, 6, 8], [0, 2, 3, 0], [1, 0, 6, 4]], dtype=np.int64)
    sel = orc.conv3d_acc_points(xb, wl.NCDHW, wb, pts, (1, 1, 1), pads)
    for i, (n, d, h, w) in enumerate(pts):
        np.testing.assert_array_equal(sel[i], full[n, d, h, w])


# ---- special cases and closed forms ---------------------------------------------------

def test_t1_causal_identity(orc):
    """CausalConv3d(x, W) == Conv2d(x.squeeze(T), W[:, :, 2], padding=1) at T=1."""
    rng = np.random.default_rng(11)
    x = rand_bf16(rng, (1, 6, 1, 9, 10))
    w = rand_bf16(rng, (5, 6, 3, 3, 3), 0.3)
    causal = ((2, 0, 0), (1, 1, 0), (1, 1, 0))
    y5 = orc.conv3d_acc(x, wl.NCDHW, w, (1, 1, 1), causal)
    w2 = np.ascontiguousarray(w[:, :, 2:3])
    y2 = orc.conv3d_acc(x, wl.NCDHW, w2, (1, 1, 1), ((0, 0, 0), (1, 1, 0), (1, 1, 0)))
    np.testing.assert_array_equal(y5, y2)
    # and a symmetric temporal pad is NOT that identity (it would use W[:, :, 1])
    ysym = orc.conv3d_acc(x, wl.NCDHW, w, (1, 1, 1), ((1, 1, 0), (1, 1, 0), (1, 1, 0)))
    assert not np.array_equal(ysym, y2)


def test_1x1x1_is_gemm(orc):
    rng = np.random.default_rng(3)
    x = rand_bf16(rng, (2, 3, 4, 5, 24))  # NDHWC
    w = rand_bf16(rng, (7, 24, 1, 1, 1), 0.2)
    y = orc.conv3d_acc(x, wl.NDHWC, w)
    ref = to_f64(orc, x).reshape(-1, 24) @ to_f64(orc, w).reshape(7, 24).T
    np.testing.assert_array_equal(y.reshape(-1, 7), ref.astype(np.float32))


def test_layout_round_trip(orc):
    rng = np.random.default_rng(5)
    xb = rand_bf16(rng, (1, 9, 4, 6, 7))
    wb = rand_bf16(rng, (4, 9, 3, 3, 3), 0.2)
    pads = ((2, 0, 0), (1, 1, 1), (1, 1, 1))
    a = orc.conv3d_acc(xb, wl.NCDHW, wb, (1, 1, 1), pads)
    b = orc.conv3d_acc(np.ascontiguousarray(xb.transpose(0, 2, 3, 4, 1)), wl.NDHWC, wb,
                       (1, 1, 1), pads)
    np.testing.assert_array_equal(a, b)
    y = orc.round_bf16(a)
    np.testing.assert_array_equal(orc.from_layout(orc.to_layout(y, wl.NCDHW), wl.NCDHW), y)


def _ones(shape):
    return np.full(shape, 0x3F80, dtype=np.uint16)  # bf16 1.0


def test_closed_form_ones_zero_pad(orc):
    C, D, H, W = 3, 4, 5, 6
    x = _ones((1, C, D, H, W))
    w = _ones((2, C, 3, 3, 3))
    y = orc.conv3d_acc(x, wl.NCDHW, w, (1, 1, 1), ((1, 1, 0),) * 3)
    # each output counts the in-bounds taps: prod over dims of the window overlap
    def cnt(o, L):
        return min(o + 1, L - 1) - max(o - 1, 0) + 1
    for d in range(D):
        for h in range(H):
            for ww in range(W):
                expect = C * cnt(d, D) * cnt(h, H) * cnt(ww, W)
                assert y[0, d, h, ww, 0] == expect and y[0, d, h, ww, 1] == expect
    assert y[0, 1, 1, 1, 0] == C * 27


def test_closed_form_ones_reflect(orc):
    x = _ones((1, 2, 3, 4, 5))
    w = _ones((1, 2, 3, 3, 3))
    y = orc.conv3d_acc(x, wl.NCDHW, w, (1, 1, 1), ((1, 1, 1),) * 3)
    assert np.all(y == 2 * 27)
    # causal temporal zero pad + reflect spatial: planes 0 and 1 see 1 and 2 frames
    y = orc.conv3d_acc(x, wl.NCDHW, w, (1, 1, 1), ((2, 0, 0), (1, 1, 1), (1, 1, 1)))
    assert np.all(y[0, 0] == 2 * 9) and np.all(y[0, 1] == 2 * 18) and np.all(y[0, 2] == 2 * 27)


def test_closed_form_one_hot(orc):
    """A one-hot input at (p, ci) gives out[p - tap + pad] = W[:, ci, tap]:
    pins the correlation orientation and the causal direction."""
    rng = np.random.default_rng(9)
    C, D, H, W = 4, 5, 6, 7
    w = rand_bf16(rng, (3, C, 3, 3, 3))
    x = np.zeros((1, C, D, H, W), dtype=np.uint16)
    p = (2, 3, 4)
    ci = 2
    x[0, ci, p[0], p[1], p[2]] = 0x3F80
    pads = ((2, 0, 0), (1, 1, 0), (1, 1, 0))
    y = orc.conv3d_acc(x, wl.NCDHW, w, (1, 1, 1), pads)
    wf = orc.bf16_to_f32(w)
    seen = 0
    for t in range(3):
        for r in range(3):
            for s in range(3):
                o = (p[0] - t + 2, p[1] - r + 1, p[2] - s + 1)
                if 0 <= o[0] < D and 0 <= o[1] < H and 0 <= o[2] < W:
                    np.testing.assert_array_equal(y[0, o[0], o[1], o[2]], wf[:, ci, t, r, s])
                    seen += 1
    assert seen == 27
    assert np.count_nonzero(np.any(y != 0, axis=-1)) == 27


@pytest.mark.parametrize("pads", [((0, 0, 0),) * 3, ((1, 1, 0),) * 3])
def test_stride_is_subsampling(orc, pads):
    rng = np.random.default_rng(13)
    x = rand_bf16(rng, (1, 3, 7, 9, 8))
    w = rand_bf16(rng, (2, 3, 3, 3, 3), 0.3)
    full = orc.conv3d_acc(x, wl.NCDHW, w, (1, 1, 1), pads)
    s2 = orc.conv3d_acc(x, wl.NCDHW, w, (2, 2, 2), pads)
    np.testing.assert_array_equal(s2, full[:, ::2, ::2, ::2][:, :s2.shape[1], :s2.shape[2],
                                                              :s2.shape[3]])


def test_output_shape_rules(orc):
    # valid 3x3x3: [N,T,H,W] -> [N,T-2,H-2,W-2] (cuDNN doc, "Raw Conv3D Variant")
    assert orc.out_dims(8, 106, 182, 3, 3, 3, (1, 1, 1), ((0, 0, 0),) * 3) == (6, 104, 180)
    # Wan dominant shapes with the pad applied outside (valid)
    assert orc.out_dims(6, 354, 642, 3, 3, 3, (1, 1, 1), ((0, 0, 0),) * 3) == (4, 352, 640)
    assert orc.out_dims(3, 46, 82, 3, 3, 3, (1, 1, 1), ((0, 0, 0),) * 3) == (1, 44, 80)
    # encoder ladder: causal T pad 2 + reflect 1 keeps size; stride 2 halves
    cr = ((2, 0, 0), (1, 1, 1), (1, 1, 1))
    assert orc.out_dims(17, 256, 256, 3, 3, 3, (1, 1, 1), cr) == (17, 256, 256)
    assert orc.out_dims(17, 256, 256, 3, 3, 3, (1, 2, 2), cr) == (17, 128, 128)
    assert orc.out_dims(17, 128, 128, 3, 3, 3, (2, 2, 2), cr) == (9, 64, 64)
    assert orc.out_dims(9, 64, 64, 3, 3, 3, (2, 2, 2), cr) == (5, 32, 32)
    # ZeroPad2d((0,1,0,1)) then k=3 s=2 p=0: 1025 -> 512
    assert orc.out_dims(1, 1025, 1025, 1, 3, 3, (1, 2, 2), ((0, 0, 0),) * 3) == (1, 512, 512)
    assert orc.out_dims(1, 257, 257, 1, 3, 3, (1, 2, 2), ((0, 0, 0),) * 3) == (1, 128, 128)
    with pytest.raises(ValueError):
        orc.out_dims(1, 4, 4, 1, 3, 3, (1, 1, 1), ((0, 0, 0), (4, 4, 1), (0, 0, 0)))


def test_pad_bottom_right(orc):
    y = np.arange(2 * 3 * 4 * 5, dtype=np.uint16).reshape(1, 2, 3, 4, 5)
    p = orc.pad_bottom_right(y)
    assert p.shape == (1, 2, 4, 5, 5)
    np.testing.assert_array_equal(p[:, :, :3, :4], y)
    assert np.all(p[:, :, 3] == 0) and np.all(p[:, :, :, 4] == 0)


# ---- bf16 rounding, pack ----------------------------------------------------------------

def test_round_bf16_matches_torch(orc):
    rng = np.random.default_rng(1)
    mags = (10.0 ** rng.integers(-30, 30, 200000)).astype(np.float32)
    vals = [rng.standard_normal(200000).astype(np.float32) * mags]
    # exact ties, subnormals, signed zero, infinities, near-overflow
    base = np.arange(0, 1 << 16, dtype=np.uint32) << 16
    vals.append((base | 0x8000).view(np.float32))
    vals.append((base | 0x7FFF).view(np.float32))
    vals.append((base | 0x8001).view(np.float32))
    vals.append(np.array([0.0, -0.0, np.inf, -np.inf, 3.3895e38, -3.3895e38, 1e-40, -1e-45],
                         dtype=np.float32))
    f = np.concatenate(vals)
    f = f[~np.isnan(f)]
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(orc.round_bf16(f), ref)
    nan = orc.round_bf16(np.array([np.nan], dtype=np.float32))
    assert np.isnan(orc.bf16_to_f32(nan))[0]


@pytest.mark.parametrize("shape", [(5, 3, 3, 3, 3), (4, 64, 3, 3, 3), (3, 96, 1, 3, 3),
                                   (2, 130, 1, 1, 1)])
def test_pack_weight(orc, shape):
    rng = np.random.default_rng(2)
    w = rand_bf16(rng, shape)
    p = orc.pack_weight(w)
    Co, Ci, KT, KR, KS = shape
    cp = -(-Ci // 64) * 64
    ref = np.zeros((Co, KT, KR, KS, cp), dtype=np.uint16)
    ref[..., :Ci] = np.transpose(w, (0, 2, 3, 4, 1))
    np.testing.assert_array_equal(p, ref)


# ---- epilogue -------------------------------------------------------------------------------

def _parse_sparse(spec, C, default=0.0):
    v = np.full(C, default, dtype=np.float32)
    if spec == "-":
        return None
    for item in spec.split(","):
        if item.startswith("all="):
            v[:] = float(item[4:])
        else:
            k, val = item.split(":")
            v[int(k)] = float(val)
    return v


def _golden_cases():
    cases = []
    with open(os.path.join(GOLDEN, "epilogue_cases.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            cases.append([c.strip() for c in line.split("|")])
    return cases


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c[0])
def test_epilogue_golden(orc, case):
    name, C, flags_s, conv_s, bias_s, res_s, rb_s, gamma_s, field, exp_s = case
    C = int(C)
    names = {"BIAS": orc.BIAS, "RESIDUAL": orc.RESIDUAL, "RESIDUAL_BIAS": orc.RESIDUAL_BIAS,
             "L2NORM": orc.L2NORM_SILU}
    flags = 0
    for f in flags_s.split(","):
        flags |= names[f]
    conv = _parse_sparse(conv_s, C)
    conv = np.zeros(C, np.float32) if conv is None else conv
    bias = _parse_sparse(bias_s, C)
    res = _parse_sparse(res_s, C)
    rb = _parse_sparse(rb_s, C)
    gamma = _parse_sparse(gamma_s, C)
    if flags & orc.BIAS and bias is None:
        bias = np.zeros(C, np.float32)
    out = orc.epilogue(orc.round_bf16(conv[None]), flags, bias,
                       None if res is None else orc.round_bf16(res[None]), rb, gamma)
    expect = _parse_sparse(exp_s, C)
    expect = np.zeros(C, np.float32) if expect is None else expect
    np.testing.assert_array_equal(orc.bf16_to_f32(out[field][0]), expect)


def _ulp_dist(orc, a, b):
    def ordinal(u):
        i = u.astype(np.int32)
        neg = (i & 0x8000) != 0
        mag = i & 0x7FFF
        return np.where(neg, -mag, mag)
    return np.abs(ordinal(a) - ordinal(b))


def test_norm_invariant_and_library(orc):
    """||normalized||_2 ~= 1 within bf16 rounding; normalized and SiLU agree with
    F.normalize / F.silu evaluated in float64 to within 1 bf16 ulp per step."""
    rng = np.random.default_rng(21)
    for C in (16, 32, 160, 320, 640):
        M = 300
        conv = rand_bf16(rng, (M, C))
        bias = rng.standard_normal(C).astype(np.float32) * 0.1
        gamma = orc.bf16_to_f32(rand_bf16(rng, (C,), 0.1)) + 1.0
        res = rand_bf16(rng, (M, C))
        flags = orc.BIAS | orc.RESIDUAL | orc.L2NORM_SILU
        out = orc.epilogue(conv, flags, bias, res, None, gamma)
        value = to_f64(orc, out["value"])
        nrm = F.normalize(torch.from_numpy(value), dim=1, eps=1e-12).numpy()
        n_bits = bf16_bits_from_f32(nrm.astype(np.float32))
        norms = np.linalg.norm(orc.bf16_to_f32(n_bits).astype(np.float64), axis=1)
        assert np.all(np.abs(norms - 1.0) <= 2.0 ** -8)
        # activated from the library: silu(B(B(n * sqrt C) * gamma))
        sc = orc.round_bf16((orc.bf16_to_f32(n_bits) * np.float32(np.sqrt(np.float32(C))))
                            .astype(np.float32))
        af = orc.round_bf16(orc.bf16_to_f32(sc) * gamma[None, :])
        act_lib = bf16_bits_from_f32(
            F.silu(torch.from_numpy(orc.bf16_to_f32(af).astype(np.float64))).numpy()
            .astype(np.float32))
        d = _ulp_dist(orc, out["act"], act_lib)
        assert d.max() <= 2, d.max()
        assert np.mean(d == 0) > 0.97


def test_zero_row_and_silu_zero(orc):
    C = 32
    conv = np.zeros((3, C), dtype=np.uint16)
    out = orc.epilogue(conv, orc.L2NORM_SILU, gamma=np.ones(C, np.float32))
    assert np.all(out["act"] == 0)


def test_l2norm_silu_standalone_matches_epilogue(orc):
    """The standalone variant with input_bias equals the fused contract applied
    to raw = conv ("main = B(raw + input_bias)")."""
    rng = np.random.default_rng(31)
    C = 64
    raw = rand_bf16(rng, (50, C))
    bias = rng.standard_normal(C).astype(np.float32) * 0.1
    res = rand_bf16(rng, (50, C))
    rb = rng.standard_normal(C).astype(np.float32) * 0.1
    gamma = np.ones(C, np.float32)
    y, v = orc.l2norm_silu(raw, gamma, bias, res, rb)
    e = orc.epilogue(raw, orc.BIAS | orc.RESIDUAL | orc.RESIDUAL_BIAS | orc.L2NORM_SILU,
                     bias, res, rb, gamma)
    np.testing.assert_array_equal(y, e["act"])
    np.testing.assert_array_equal(v, e["value"])
    # without input_bias, main is raw itself
    y2, v2 = orc.l2norm_silu(raw, gamma)
    np.testing.assert_array_equal(v2, raw)


def test_forward_small_workload_against_torch(orc):
    """The seeded tiny workload through oracle.forward: conv equals the bf16
    rounding of torch's fp64 conv3d."""
    w = wl.tiny()
    call = w.calls[0]
    inp = wl.make_inputs("tiny", call)
    xb = wl.bits(inp["x"])
    wb = wl.bits(inp["w"])
    out = orc.forward(xb, wl.NDHWC, wb, call.stride, call.pads, wl.NDHWC, orc.BIAS,
                      bias=inp["bias"].numpy())
    x64 = inp["x"].double().permute(0, 4, 1, 2, 3).numpy()
    ref = torch_conv(x64, inp["w"].double().numpy(), call.stride, call.pads)
    np.testing.assert_array_equal(out["conv"], bf16_bits_from_f32(ref.astype(np.float32)))


# ---- padded output + two-frame cache ([cuDNN-PO] "Normalization and Padding Variant",
#      "Standalone Normalization and Padding Variant") ------------------------------------

def _frames(N, T, H, W, C, seed):
    rng = np.random.default_rng(seed)
    # nonzero bf16 bit patterns (sign 0, exponent 1..254), so a stray zero shows
    return rng.integers(0x0080, 0x7F00, size=(N, T, H, W, C)).astype(np.uint16)


def test_pad_cache_worked_examples(orc):
    # one current frame, no history: planes 0 and 1 all zero, plane 2 = the frame
    # inside a zero border; the cache holds that single frame
    act = np.arange(1, 1 + 2 * 3 * 2, dtype=np.uint16).reshape(1, 1, 2, 3, 2)
    padded, cache = orc.pad_cache_fused(act, 0, np.full((1, 3, 4, 5, 2), 9, np.uint16),
                                        np.full((1, 1, 2, 3, 2), 9, np.uint16))
    assert not padded[:, :2].any()
    assert padded[0, 2, 1, 1].tolist() == [1, 2] and padded[0, 2, 2, 3].tolist() == [11, 12]
    assert not padded[0, 2, 0].any() and not padded[0, 2, 3].any()
    assert not padded[0, 2, :, 0].any() and not padded[0, 2, :, 4].any()
    assert np.array_equal(cache, act)
    # standalone, two history frames and one new one: the cache is the newest
    # history frame followed by the new frame
    prev = _frames(1, 2, 2, 3, 2, 1)
    padded, cache = orc.pad_cache_standalone(act, prev)
    assert padded.shape == (1, 3, 4, 5, 2) and cache.shape == (1, 2, 2, 3, 2)
    assert np.array_equal(padded[:, 0, 1:-1, 1:-1], prev[:, 0])
    assert np.array_equal(padded[:, 1, 1:-1, 1:-1], prev[:, 1])
    assert np.array_equal(cache[:, 0], prev[:, 1]) and np.array_equal(cache[:, 1], act[:, 0])


@pytest.mark.parametrize("P", [0, 1, 2])
@pytest.mark.parametrize("Tc", [1, 2, 3, 5])
def test_pad_cache_fused_leaves_history_and_borders(orc, P, Tc):
    N, H, W, C = 2, 3, 4, 8
    act = _frames(N, Tc, H, W, C, 10 + Tc)
    K = min(2, Tc + P)
    sentinel = 0x3F80  # bf16 1.0: not written by the kernel wherever it survives
    padded, cache = orc.pad_cache_fused(
        act, P, np.full((N, Tc + 2, H + 2, W + 2, C), sentinel, np.uint16),
        np.full((N, K, H, W, C), sentinel, np.uint16))
    border = np.ones((H + 2, W + 2), bool)
    border[1:-1, 1:-1] = False
    assert not padded[:, :, border].any()                  # every plane's border is zero
    assert not padded[:, :2 - P].any()                     # missing history planes are zero
    assert (padded[:, 2 - P:2, 1:-1, 1:-1] == sentinel).all()  # history interiors untouched
    assert np.array_equal(padded[:, 2:, 1:-1, 1:-1], act)  # current frames, in order
    kc = min(2, Tc)
    assert np.array_equal(cache[:, K - kc:], act[:, Tc - kc:])  # newest frames at the tail
    assert (cache[:, :K - kc] == sentinel).all()           # older frames are the caller's


@pytest.mark.parametrize("P", [0, 1, 2])
@pytest.mark.parametrize("Tc", [1, 2, 3])
def test_pad_cache_fused_plus_history_step_is_standalone(orc, P, Tc):
    # The page gives the fused variant plus a caller-side step (history frames into
    # the history planes' interiors, older cache frames from the previous cache) and
    # the standalone variant that does both itself: the two must produce the same.
    N, H, W, C = 1, 2, 3, 8
    act = _frames(N, Tc, H, W, C, 20 + P)
    prev = _frames(N, P, H, W, C, 30 + Tc) if P else None
    K = min(2, Tc + P)
    padded, cache = orc.pad_cache_fused(act, P, np.full((N, Tc + 2, H + 2, W + 2, C), 7, np.uint16),
                                        np.full((N, K, H, W, C), 7, np.uint16))
    for j in range(P):                         # history frame j of P -> plane 2 - P + j
        padded[:, 2 - P + j, 1:-1, 1:-1] = prev[:, j]
    older = max(K - Tc, 0)                     # cache slots the current frames do not fill
    for j in range(older):                     # the newest `older` history frames, in order
        cache[:, j] = prev[:, P - older + j]
    ref_padded, ref_cache = orc.pad_cache_standalone(act, prev)
    assert np.array_equal(padded, ref_padded)
    assert np.array_equal(cache, ref_cache)


# ---- streaming causal convolution: input packing with history (cuDNN frontend doc,
#      "Causal Conv3D with Cache") -----------------------------------------------------

def test_causal_pack_worked_example(orc):
    # a 1-frame chunk of 3 channels, no history: two zero planes (the causal padding),
    # then the frame channels-last inside a zero border, channels 3 .. 7 zero
    x = np.arange(1, 1 + 3 * 2 * 2, dtype=np.uint16).reshape(1, 3, 1, 2, 2)  # [N, C, T, H, W]
    padded, cache = orc.causal_pack(x, None, Cp=8)
    assert padded.shape == (1, 3, 4, 4, 8) and cache.shape == (1, 1, 2, 2, 3)
    assert not padded[:, :2].any()
    assert padded[0, 2, 1, 1].tolist() == [1, 5, 9, 0, 0, 0, 0, 0]    # pixel (0, 0)
    assert padded[0, 2, 2, 2].tolist() == [4, 8, 12, 0, 0, 0, 0, 0]   # pixel (1, 1)
    assert not padded[0, 2, 0].any() and not padded[0, 2, :, 3].any()
    assert cache[0, 0, 1, 0].tolist() == [3, 7, 11]
    # with one history frame: plane 1 holds it, plane 0 stays zero, and the cache is
    # [history, chunk frame]
    prev = np.full((1, 1, 2, 2, 3), 0x4000, np.uint16)
    padded, cache = orc.causal_pack(x, prev, Cp=8)
    assert not padded[:, 0].any()
    assert (padded[0, 1, 1:-1, 1:-1, :3] == 0x4000).all() and not padded[0, 1, 1:-1, 1:-1, 3:].any()
    assert cache.shape == (1, 2, 2, 2, 3) and (cache[:, 0] == 0x4000).all()


@pytest.mark.parametrize("chunks", [(1, 4, 4), (2, 1, 3), (5,), (1, 1, 1, 2)])
def test_causal_pack_streaming_is_the_whole_causal_conv(orc, chunks):
    # Chunk by chunk, each packed after the previous chunk's cache and convolved as a
    # valid 3x3x3 convolution, the outputs are the causal (T: 2 zero frames before) and
    # zero-padded (H, W: 1) convolution of the whole video: torch fp64 conv3d after
    # F.pad.  The caches are the last frames of the video so far.
    rng = np.random.default_rng(sum(chunks))
    N, C, H, W, Co, Cp = 1, 12, 4, 5, 6, 16
    T = sum(chunks)
    video = rand_bf16(rng, (N, C, T, H, W))
    w = rand_bf16(rng, (Co, C, 3, 3, 3), 0.2)
    w16 = np.zeros((Co, Cp, 3, 3, 3), np.uint16)
    w16[:, :C] = w
    outs, prev, t0 = [], None, 0
    for tc in chunks:
        chunk = np.ascontiguousarray(video[:, :, t0:t0 + tc])
        padded, cache = orc.causal_pack(chunk, prev, Cp=Cp)
        outs.append(orc.conv3d_acc(padded, orc.NDHWC, w16))
        t0 += tc
        K = min(2, t0)
        assert np.array_equal(cache, np.transpose(video[:, :, t0 - K:t0], (0, 2, 3, 4, 1)))
        prev = cache
    got = np.concatenate(outs, axis=1)
    Z = wl.ZERO
    ref = torch_conv(to_f64(orc, video), to_f64(orc, w), (1, 1, 1), ((2, 0, Z), (1, 1, Z), (1, 1, Z)))
    assert got.shape == ref.shape
    # (the oracle returns its fp64 sums rounded to fp32: half an fp32 ulp)
    np.testing.assert_allclose(got, ref, rtol=2.0 ** -24, atol=1e-12)


# ---- channels-last GroupNorm + SiLU (FlyDSL issue, MiniMax-H3 comment: the GroupNorm
#      between the encoder's convolutions, time-isolated groups) -------------------------

def _gn_inputs(orc, shape, C, seed):
    rng = np.random.default_rng(seed)
    x = orc.round_bf16(rng.standard_normal(shape).astype(np.float32) * 2 + 0.5)
    gamma = (1 + 0.2 * rng.standard_normal(C)).astype(np.float32)
    beta = (0.2 * rng.standard_normal(C)).astype(np.float32)
    return x, gamma, beta


@pytest.mark.parametrize("isolated", [True, False])
def test_group_norm_matches_torch(orc, isolated):
    # without the SiLU, the normalised value is torch's group_norm in fp64 over the
    # NCDHW view: per frame (frames as batch) when time-isolated, else per clip
    N, D, H, W, C, G = 2, 3, 4, 5, 24, 6
    x, gamma, beta = _gn_inputs(orc, (N, D, H, W, C), C, 3)
    got = orc.bf16_to_f32(orc.group_norm_silu(x, G, gamma, beta, eps=1e-6,
                                              time_isolated=isolated, silu=False))
    xt = torch.from_numpy(orc.bf16_to_f32(x).astype(np.float64))
    if isolated:
        v = xt.reshape(N * D, H, W, C).permute(0, 3, 1, 2)      # frames as batch, NCHW
    else:
        v = xt.permute(0, 4, 1, 2, 3)                          # NCDHW
    ref = torch.nn.functional.group_norm(v, G, torch.from_numpy(gamma.astype(np.float64)),
                                         torch.from_numpy(beta.astype(np.float64)), eps=1e-6)
    ref = (ref.permute(0, 2, 3, 1).reshape(N, D, H, W, C) if isolated
           else ref.permute(0, 2, 3, 4, 1))
    ref_b = orc.bf16_to_f32(orc.round_bf16(ref.numpy()))
    np.testing.assert_array_equal(got, ref_b)
    # the SiLU step: torch's silu in fp64 on the bf16 normalised values, rounded once
    with_silu = orc.group_norm_silu(x, G, gamma, beta, eps=1e-6, time_isolated=isolated)
    silu_ref = F.silu(torch.from_numpy(got.astype(np.float64))).numpy()
    np.testing.assert_array_equal(with_silu, orc.round_bf16(silu_ref))


def test_group_norm_closed_forms(orc):
    N, D, H, W, C, G = 1, 2, 3, 3, 16, 4
    _, gamma, beta = _gn_inputs(orc, (N, D, H, W, C), C, 4)
    # a constant group normalises to zero: the output is B(beta) (SiLU off), and with
    # the SiLU of beta = 0 it is 0
    x = np.full((N, D, H, W, C), orc.round_bf16(np.float32(1.75)), np.uint16)
    y = orc.bf16_to_f32(orc.group_norm_silu(x, G, gamma, beta, silu=False))
    np.testing.assert_array_equal(y, np.broadcast_to(orc.bf16_to_f32(orc.round_bf16(beta)), y.shape))
    y0 = orc.group_norm_silu(x, G, gamma, np.zeros(C, np.float32))
    assert not orc.bf16_to_f32(y0).any()
    # time isolation: rescaling one frame changes nothing anywhere
    x, gamma, beta = _gn_inputs(orc, (N, D, H, W, C), C, 5)
    # (frame 1 scaled by 2: exact in bf16; a group's normalised values do not change)
    xs = orc.bf16_to_f32(x).copy()
    xs[:, 1] *= 2.0
    xs_b = orc.round_bf16(xs)
    a = orc.group_norm_silu(x, G, gamma, beta, eps=0.0)   # eps = 0: the identity is exact
    b = orc.group_norm_silu(xs_b, G, gamma, beta, eps=0.0)
    assert np.array_equal(a[:, 0], b[:, 0])
    assert np.array_equal(a[:, 1], b[:, 1])
    # negating x and gamma negates the normalised value exactly
    n1 = orc.bf16_to_f32(orc.group_norm_silu(x, G, gamma, np.zeros(C, np.float32), silu=False))
    n2 = orc.bf16_to_f32(orc.group_norm_silu(x ^ np.uint16(0x8000), G, -gamma,
                                             np.zeros(C, np.float32), silu=False))
    np.testing.assert_array_equal(n1, n2)


# ---- x2 nearest upsampling before a 3x3 convolution (FlyDSL PR, "Upsample Conv2d") ------

def test_upsample2x_nearest_matches_torch(orc):
    rng = np.random.default_rng(11)
    x = orc.round_bf16(rng.standard_normal((2, 1, 5, 7, 8)).astype(np.float32))
    got = orc.upsample2x_nearest(x)
    xt = torch.from_numpy(orc.bf16_to_f32(x)).permute(0, 4, 1, 2, 3)[:, :, 0]   # NCHW
    ref = F.interpolate(xt, scale_factor=2, mode="nearest-exact")
    ref = ref.permute(0, 2, 3, 1).unsqueeze(1).numpy()
    np.testing.assert_array_equal(orc.bf16_to_f32(got), ref)


def test_upsample2x_conv_parity_classes(orc):
    # Output (2i + ph, 2j + pw) of the zero-pad-1 3x3 convolution of the x2 nearest
    # upsampled input reads upsampled rows 2i + ph + r - 1 (r = 0..2), i.e. low-res rows
    # i + (-1, 0, 0)[r] for ph = 0 and i + (0, 0, 1)[r] for ph = 1 (columns alike): each
    # parity class is a convolution of the low-res input with the same 9 weights and a
    # tap -> offset table.  The fused kernel computes exactly this.
    rng = np.random.default_rng(12)
    N, H, W, Ci, Co = 1, 5, 6, 8, 4
    x = orc.round_bf16(rng.standard_normal((N, 1, H, W, Ci)).astype(np.float32))
    w = orc.round_bf16((rng.standard_normal((Co, Ci, 1, 3, 3)) / 8).astype(np.float32))
    xf = orc.bf16_to_f32(x).astype(np.float64)[:, 0]            # [N, H, W, Ci]
    wf = orc.bf16_to_f32(w).astype(np.float64)[:, :, 0]         # [Co, Ci, 3, 3]
    up = np.repeat(np.repeat(xf, 2, axis=1), 2, axis=2)         # [N, 2H, 2W, Ci]
    upp = np.pad(up, ((0, 0), (1, 1), (1, 1), (0, 0)))
    direct = np.zeros((N, 2 * H, 2 * W, Co))
    for r in range(3):
        for s in range(3):
            direct += np.einsum("nhwc,oc->nhwo", upp[:, r:r + 2 * H, s:s + 2 * W], wf[:, :, r, s])
    off = ((-1, 0, 0), (0, 0, 1))
    xp = np.pad(xf, ((0, 0), (1, 1), (1, 1), (0, 0)))           # low-res, zero border
    for ph in range(2):
        for pw in range(2):
            cls = np.zeros((N, H, W, Co))
            for r in range(3):
                for s in range(3):
                    a, b = 1 + off[ph][r], 1 + off[pw][s]
                    cls += np.einsum("nhwc,oc->nhwo", xp[:, a:a + H, b:b + W], wf[:, :, r, s])
            np.testing.assert_allclose(direct[:, ph::2, pw::2], cls, rtol=1e-12, atol=1e-12)
    # the oracle's fp32 accumulator of the plain definition agrees with fp64
    acc = orc.upsample2x_conv_acc(x, w)[:, 0]
    np.testing.assert_allclose(acc, direct, rtol=1e-5, atol=1e-5)


# ---- FP8 e4m3fn operands (FlyDSL PR, "Summary" / "Test shapes": the FP8 suite) --------

def test_e4m3_decode_matches_torch_and_closed_forms(orc):
    codes = np.arange(256, dtype=np.uint8)
    got = orc.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert list(np.flatnonzero(nan)) == [0x7F, 0xFF]          # only S.1111.111
    np.testing.assert_array_equal(got[~nan], ref[~nan])
    # closed forms of the format: bias 7, 3 mantissa bits, subnormals m/8 * 2^-6
    assert got[0x38] == 1.0 and got[0xB8] == -1.0
    assert got[0x7E] == 448.0 and got[0xFE] == -448.0         # 1.75 * 2^8
    assert got[0x01] == 2.0 ** -9 and got[0x07] == 7 * 2.0 ** -9
    assert got[0x08] == 2.0 ** -6                              # smallest normal
    assert got[0x3C] == 1.5 and got[0x41] == 2.25
    assert got[0x00] == 0.0 and not np.signbit(got[0x00]) and np.signbit(got[0x80])


def test_e4m3_to_bf16_is_exact(orc):
    codes = np.arange(256, dtype=np.uint8)
    v = orc.e4m3_to_f64(codes)
    b = orc.e4m3_to_bf16(codes)
    ok = ~np.isnan(v)
    np.testing.assert_array_equal(orc.bf16_to_f32(b)[ok].astype(np.float64), v[ok])
    assert np.all(np.isnan(orc.bf16_to_f32(b)[~ok]))


@pytest.mark.parametrize("case", [CASES[2], CASES[3], CASES[5]])
def test_conv_e4m3_matches_torch(orc, case):
    # torch's own e4m3fn decode, fp64 conv3d, then the per-tensor scale
    N, C, D, H, W, Co, k, stride, pads = case
    rng = np.random.default_rng(31)
    x8 = rng.integers(0, 256, (N, D, H, W, C), dtype=np.uint8)
    w8 = rng.integers(0, 256, (Co, C) + k, dtype=np.uint8)
    x8[(x8 & 0x7F) == 0x7F] = 0x38                              # no NaN codes
    w8[(w8 & 0x7F) == 0x7F] = 0xB8
    scale = 2.0 ** -11
    acc = orc.conv3d_acc_e4m3(x8, wl.NDHWC, w8, scale, stride, pads)
    dec = lambda a: torch.from_numpy(a).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ref = torch_conv(np.ascontiguousarray(dec(x8).transpose(0, 4, 1, 2, 3)), dec(w8), stride,
                     pads) * scale
    np.testing.assert_allclose(acc, ref.astype(np.float32), rtol=2.0 ** -23, atol=0)


def test_pack_weight_e4m3(orc):
    rng = np.random.default_rng(32)
    w8 = rng.integers(0, 256, (5, 140, 3, 2, 3), dtype=np.uint8)
    p = orc.pack_weight_e4m3(w8)
    assert p.shape == (5, 3, 2, 3, 256)
    assert np.all(p[..., 140:] == 0)
    for co, t, r, s in [(0, 0, 0, 0), (4, 2, 1, 2), (2, 1, 0, 1)]:
        np.testing.assert_array_equal(p[co, t, r, s, :140], w8[co, :, t, r, s])
