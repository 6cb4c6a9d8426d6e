"""ORACLE — test infrastructure only.

A plain, slow CPU implementation of the video-VAE convolution path (direct
convolution with fp64 accumulation, the post-operation contract with every BF16
rounding point, the standalone L2-norm/SiLU and the weight pack).  It exists to
check the CUDA library.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` / ``--impl reference`` legs may import it; the
product package never does, and shares no code with it.

Sources (web pages, cited by title and section):

* ROCm/FlyDSL issue "[Feature]: conv3d_implicit — accept and emit NDHWC so
  chained convs skip the layout round-trip" — the op, its layouts, and the
  VAE's reflect + causal padding ("The call site is already a clean drop-in").
* ROCm/FlyDSL PR "[Flydsl] Add Qwen-Image VAE classic conv shapes to conv3d
  tests" — the T=1 causal identity ("T=1 degeneration") and the downsample
  ZeroPad2d((0,1,0,1)) + stride-2 conv ("Downsample Conv2d").
* [cuDNN-PO] cuDNN frontend doc "Fused Conv3D + Bias + Residual + RMSNorm +
  SiLU" — the Operation Contract (rounding points), "Weight Packing",
  "Normalization and Padding Variant", "Standalone Normalization and Padding
  Variant", "Spatial Padding Variant", "Causal Conv3D with Cache".

bf16 values are carried as ``numpy.uint16`` bit patterns throughout.

Pins: see ``tests/test_oracle_pins.py``.  The oracle's mainloop summation order
is the one thing left free ("parity unpinned" beyond +-1 bf16 ulp of ``conv``).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "conv3d_oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

# Epilogue flags (oracle-local numbering, independent of the CUDA ABI's).
BIAS = 1
RESIDUAL = 2
RESIDUAL_BIAS = 4
L2NORM_SILU = 8

NCDHW = 0
NDHWC = 1
PAD_ZERO = 0
PAD_REFLECT = 1


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (-O2, OpenMP, no FP contraction)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            p = ctypes.c_void_p
            i = ctypes.c_int
            lng = ctypes.c_long
            lib.orc_num_threads.argtypes = [i]
            lib.orc_num_threads.restype = i
            lib.orc_out_dims.argtypes = [i, i, i, i, i, i, i, i, i, p, p]
            lib.orc_out_dims.restype = i
            lib.orc_conv3d_acc.argtypes = [p, i, i, i, i, i, i, p, i, i, i, i, i, i, i, p, p, i]
            lib.orc_conv3d_acc.restype = i
            lib.orc_conv3d_acc_points.argtypes = [p, i, i, i, i, i, i, p, i, i, i, i, i, i, i,
                                                  p, p, lng, p, i]
            lib.orc_conv3d_acc_points.restype = i
            lib.orc_round_bf16.argtypes = [p, p, lng]
            lib.orc_round_bf16.restype = None
            lib.orc_epilogue.argtypes = [p, lng, i, ctypes.c_uint, p, p, p, p, p, p, p, i]
            lib.orc_epilogue.restype = i
            lib.orc_l2norm_silu.argtypes = [p, lng, i, p, p, p, p, p, p, i]
            lib.orc_l2norm_silu.restype = i
            lib.orc_pack_weight.argtypes = [p, i, i, i, i, i, p]
            lib.orc_pack_weight.restype = i
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u16(a):
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, a.dtype
    return a


def _f32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float32)


def num_threads(n: int = 0) -> int:
    """Set (n > 0) and return the OpenMP thread count the oracle uses."""
    return _load().orc_num_threads(int(n))


# ---- bf16 helpers -------------------------------------------------------------

def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def round_bf16(f: np.ndarray) -> np.ndarray:
    """B(x): fp32 -> bf16 bits, round to nearest even."""
    f = np.ascontiguousarray(f, dtype=np.float32)
    out = np.empty(f.shape, dtype=np.uint16)
    _load().orc_round_bf16(_ptr(f), _ptr(out), f.size)
    return out


# ---- geometry -------------------------------------------------------------------

def pads9(pads) -> np.ndarray:
    """pads: ((before, after, mode) for T, H, W) -> int32[9]."""
    flat = [int(v) for trip in pads for v in trip]
    assert len(flat) == 9
    return np.asarray(flat, dtype=np.int32)


def out_dims(D, H, W, KT, KR, KS, stride, pads):
    o = np.zeros(3, dtype=np.int32)
    p = pads9(pads)
    rc = _load().orc_out_dims(D, H, W, KT, KR, KS, stride[0], stride[1], stride[2],
                              _ptr(p), _ptr(o))
    if rc != 0:
        raise ValueError("invalid convolution geometry")
    return tuple(int(v) for v in o)


def _dims(x, layout):
    if layout == NCDHW:
        N, C, D, H, W = x.shape
    else:
        N, D, H, W, C = x.shape
    return N, C, D, H, W


# ---- convolution ------------------------------------------------------------------

def conv3d_acc(x, layout, w, stride=(1, 1, 1), pads=((0, 0, 0),) * 3, nthreads=0):
    """fp32 accumulator of the convolution, shape [N, Do, Ho, Wo, Co].

    x: uint16 bf16 bits, 5-D in `layout`; w: uint16 bf16 bits [Co, Ci, KT, KR, KS].
    """
    x = _u16(x)
    w = _u16(w)
    N, C, D, H, W = _dims(x, layout)
    Co, Ci, KT, KR, KS = w.shape
    assert Ci == C, (Ci, C)
    Do, Ho, Wo = out_dims(D, H, W, KT, KR, KS, stride, pads)
    acc = np.empty((N, Do, Ho, Wo, Co), dtype=np.float32)
    p = pads9(pads)
    rc = _load().orc_conv3d_acc(_ptr(x), layout, N, C, D, H, W, _ptr(w), Co, KT, KR, KS,
                                stride[0], stride[1], stride[2], _ptr(p), _ptr(acc), nthreads)
    if rc != 0:
        raise ValueError(f"orc_conv3d_acc failed ({rc})")
    return acc


def conv3d_acc_points(x, layout, w, points, stride=(1, 1, 1), pads=((0, 0, 0),) * 3,
                      nthreads=0):
    """fp32 accumulator at selected output pixels: points int64 [P, 4] (n, d, h, w)."""
    x = _u16(x)
    w = _u16(w)
    N, C, D, H, W = _dims(x, layout)
    Co, Ci, KT, KR, KS = w.shape
    assert Ci == C
    pts = np.ascontiguousarray(points, dtype=np.int64).reshape(-1, 4)
    acc = np.empty((pts.shape[0], Co), dtype=np.float32)
    p = pads9(pads)
    rc = _load().orc_conv3d_acc_points(_ptr(x), layout, N, C, D, H, W, _ptr(w), Co, KT, KR,
                                       KS, stride[0], stride[1], stride[2], _ptr(p),
                                       _ptr(pts), pts.shape[0], _ptr(acc), nthreads)
    if rc != 0:
        raise ValueError(f"orc_conv3d_acc_points failed ({rc})")
    return acc


def epilogue(conv, flags, bias=None, residual=None, residual_bias=None, gamma=None,
             nthreads=0):
    """Post-operations on conv rows (bf16 bits [..., C]); returns dict of bf16 bits.

    Keys: 'main', 'value', and 'act' when L2NORM_SILU is set.
    """
    conv = _u16(conv)
    C = conv.shape[-1]
    M = conv.size // C
    bias = _f32(bias)
    residual_bias = _f32(residual_bias)
    gamma = _f32(gamma)
    if residual is not None:
        residual = _u16(residual)
        assert residual.shape == conv.shape
    main = np.empty(conv.shape, dtype=np.uint16)
    value = np.empty(conv.shape, dtype=np.uint16)
    act = np.empty(conv.shape, dtype=np.uint16) if flags & L2NORM_SILU else None
    rc = _load().orc_epilogue(_ptr(conv), M, C, flags, _ptr(bias), _ptr(residual),
                              _ptr(residual_bias), _ptr(gamma), _ptr(main), _ptr(value),
                              _ptr(act), nthreads)
    if rc != 0:
        raise ValueError(f"orc_epilogue failed ({rc})")
    out = {"main": main, "value": value}
    if act is not None:
        out["act"] = act
    return out


def l2norm_silu(raw, gamma, input_bias=None, residual=None, residual_bias=None,
                nthreads=0):
    """Standalone post-operations on raw bf16 [..., C]; returns (y, value)."""
    raw = _u16(raw)
    C = raw.shape[-1]
    rows = raw.size // C
    if residual is not None:
        residual = _u16(residual)
    y = np.empty(raw.shape, dtype=np.uint16)
    value = np.empty(raw.shape, dtype=np.uint16)
    rc = _load().orc_l2norm_silu(_ptr(raw), rows, C, _ptr(_f32(input_bias)), _ptr(residual),
                                 _ptr(_f32(residual_bias)), _ptr(_f32(gamma)), _ptr(y),
                                 _ptr(value), nthreads)
    if rc != 0:
        raise ValueError(f"orc_l2norm_silu failed ({rc})")
    return y, value


def pack_weight(w):
    """OITRS -> OTRSI with Ci zero-padded to a multiple of 64 (bf16 bits)."""
    w = _u16(w)
    Co, Ci, KT, KR, KS = w.shape
    cp = (Ci + 63) // 64 * 64
    out = np.empty((Co, KT, KR, KS, cp), dtype=np.uint16)
    rc = _load().orc_pack_weight(_ptr(w), Co, Ci, KT, KR, KS, _ptr(out))
    if rc != 0:
        raise ValueError("orc_pack_weight failed")
    return out


# ---- whole forward pass, as the library defines its outputs ------------------------

def to_layout(t_ndhwc: np.ndarray, layout: int) -> np.ndarray:
    """[N, D, H, W, C] -> the requested layout (a plain permutation)."""
    if layout == NDHWC:
        return np.ascontiguousarray(t_ndhwc)
    return np.ascontiguousarray(np.transpose(t_ndhwc, (0, 4, 1, 2, 3)))


def from_layout(t: np.ndarray, layout: int) -> np.ndarray:
    if layout == NDHWC:
        return np.ascontiguousarray(t)
    return np.ascontiguousarray(np.transpose(t, (0, 2, 3, 4, 1)))


def pad_bottom_right(t_ndhwc: np.ndarray) -> np.ndarray:
    """Append a zero bottom row and right column ([cuDNN-PO], "Spatial Padding
    Variant": output [N, T-2, H-1, W-1, Co] from a valid conv)."""
    N, D, H, W, C = t_ndhwc.shape
    out = np.zeros((N, D, H + 1, W + 1, C), dtype=t_ndhwc.dtype)
    out[:, :, :H, :W, :] = t_ndhwc
    return out


def pad_cache_fused(act, history_frames, padded_init, cache_init):
    """What the fused normalization-and-padding convolution writes ([cuDNN-PO],
    "Normalization and Padding Variant"), applied to caller-supplied initial
    buffers so that the regions the kernel leaves alone keep their contents.

    act: the activated current frames [N, Tc, Hc, Wc, C] (bf16 bits), Tc = T - 2.
    padded_init: [N, Tc + 2, Hc + 2, Wc + 2, C]; cache_init: [N, K, Hc, Wc, C] with
    K = min(2, Tc + P), P = history_frames in 0..2.  Returns (padded, cache):
    * every plane's one-pixel spatial border is zero;
    * the planes before the P history planes (t < 2 - P) are zero;
    * the history planes' interiors (2 - P <= t < 2) are untouched;
    * the current frames fill the interiors of planes 2 .. Tc + 1;
    * the last min(2, Tc) current frames fill the tail of the cache; its head
      (older frames) is untouched.
    """
    act = _u16(act)
    N, Tc, Hc, Wc, C = act.shape
    P = int(history_frames)
    assert 0 <= P <= 2
    K = min(2, Tc + P)
    padded = _u16(padded_init).copy()
    cache = _u16(cache_init).copy()
    assert padded.shape == (N, Tc + 2, Hc + 2, Wc + 2, C)
    assert cache.shape == (N, K, Hc, Wc, C)
    padded[:, :, 0, :, :] = 0
    padded[:, :, -1, :, :] = 0
    padded[:, :, :, 0, :] = 0
    padded[:, :, :, -1, :] = 0
    padded[:, :2 - P] = 0
    padded[:, 2:, 1:-1, 1:-1, :] = act
    kc = min(2, Tc)
    cache[:, K - kc:] = act[:, Tc - kc:]
    return padded, cache


def pad_cache_standalone(act, previous=None):
    """Padded output and cache of the standalone post-operations ([cuDNN-PO],
    "Standalone Normalization and Padding Variant"), which also copy the history.

    act: activated frames [N, T, H, W, C] (bf16 bits); previous: None or the
    P = 1 or 2 prior activated frames [N, P, H, W, C].  Returns (padded
    [N, T + 2, H + 2, W + 2, C], cache [N, min(2, T + P), H, W, C]): the frames
    [previous..., act...] end at plane T + 1 of the padded tensor (history in
    planes 2 - P .. 1, zeros before it and on every spatial border), and the
    cache holds the last min(2, T + P) of them.
    """
    act = _u16(act)
    N, T, H, W, C = act.shape
    padded = np.zeros((N, T + 2, H + 2, W + 2, C), dtype=np.uint16)
    padded[:, 2:, 1:-1, 1:-1, :] = act
    seq = act
    if previous is not None:
        prev = _u16(previous)
        P = prev.shape[1]
        assert prev.shape == (N, P, H, W, C) and 1 <= P <= 2
        padded[:, 2 - P:2, 1:-1, 1:-1, :] = prev
        seq = np.concatenate([prev, act], axis=1)
    K = min(2, seq.shape[1])
    return padded, np.ascontiguousarray(seq[:, seq.shape[1] - K:])


def causal_pack(chunk_ncthw, previous=None, Cp=16):
    """Input packing of the streaming causal convolution ([cuDNN-PO], "Causal Conv3D
    with Cache": history frames inserted before the chunk, causal and spatial zeros,
    channels padded 12 -> 16; the raw history returned for the next chunk).

    chunk_ncthw: the chunk [N, C, T, H, W] (bf16 bits); previous: None or the P = 1 or
    2 raw history frames [N, P, H, W, C].  Returns (padded [N, T + 2, H + 2, W + 2, Cp],
    cache [N, min(2, T + P), H, W, C]): the frames [previous..., chunk...] channels-last
    end at plane T + 1 (zero planes before the history, a zero spatial border, channels
    C .. Cp - 1 zero), and the cache holds the last min(2, T + P) of them.  A valid
    3x3x3 convolution over padded is the chunk's causal (T: 2 before) and zero-padded
    (H, W: 1 each side) convolution continuing the earlier frames.
    """
    x = np.transpose(_u16(chunk_ncthw), (0, 2, 3, 4, 1))  # -> [N, T, H, W, C]
    N, T, H, W, C = x.shape
    assert C <= Cp
    seq = x
    if previous is not None:
        prev = _u16(previous)
        assert prev.shape[0] == N and prev.shape[2:] == (H, W, C) and 1 <= prev.shape[1] <= 2
        seq = np.concatenate([prev, x], axis=1)
    P = seq.shape[1] - T
    padded = np.zeros((N, T + 2, H + 2, W + 2, Cp), dtype=np.uint16)
    padded[:, 2 - P:, 1:-1, 1:-1, :C] = seq
    K = min(2, seq.shape[1])
    return padded, np.ascontiguousarray(seq[:, seq.shape[1] - K:])


def group_norm_silu(x, groups, gamma, beta, eps=1e-6, time_isolated=True, silu=True):
    """Channels-last GroupNorm followed by SiLU, as the MiniMax-H3 comment on the
    FlyDSL issue describes the layers between the encoder's convolutions: groups of
    C / groups contiguous channels, statistics per (n, d, group) over H x W x C/groups
    when time_isolated (the time-to-batch reshape), else per (n, group) over
    D x H x W x C/groups.

    x: bf16 bits [N, D, H, W, C]; gamma, beta: fp32 [C].  In fp64: mean and biased
    variance of each group, g = B((x - mean) / sqrt(var + eps) * gamma + beta), and
    with silu y = B(g / (1 + exp(-g))); returns y (bf16 bits).
    """
    xb = _u16(x)
    N, D, H, W, C = xb.shape
    assert C % groups == 0
    xf = bf16_to_f32(xb).astype(np.float64)
    cg = C // groups
    # (n, slice, positions, group, channel in group); one slice per frame when isolated
    v = xf.reshape(N, D, H * W, groups, cg) if time_isolated else \
        xf.reshape(N, 1, D * H * W, groups, cg)
    axes = (2, 4)
    mean = v.mean(axis=axes, keepdims=True)
    var = ((v - mean) ** 2).mean(axis=axes, keepdims=True)
    t = (v - mean) / np.sqrt(var + eps)
    t = t.reshape(xf.shape) * np.asarray(gamma, np.float64) + np.asarray(beta, np.float64)
    g = bf16_to_f32(round_bf16(t)).astype(np.float64)  # B() of the fp64 value via fp32
    if not silu:
        return round_bf16(g)
    return round_bf16(g / (1.0 + np.exp(-g)))


# ---- FP8 e4m3 operands ----------------------------------------------------------------
# ROCm/FlyDSL PR "[Flydsl] Add Qwen-Image VAE classic conv shapes to conv3d tests",
# "Summary" / "Test shapes": the FP8 suite feeds e4m3fn activations and weights and
# takes a bf16 output.  e4m3fn (the "fn" variant: finite, no infinities) packs a sign
# bit, a 4-bit exponent with bias 7 and a 3-bit mantissa; exponent 0 holds the
# subnormals m/8 * 2^-6, and only S.1111.111 is NaN (so the largest finite value is
# 1.75 * 2^8 = 448).  The pages give no scale convention; the library takes one
# per-tensor factor that multiplies the fp32 accumulator (conv = B(scale * acc)).

def e4m3_to_f64(codes) -> np.ndarray:
    """Values of e4m3fn codes (uint8), from the format's definition."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where((c & 0x80) != 0, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


def e4m3_to_bf16(codes) -> np.ndarray:
    """bf16 bits of e4m3fn values.  Exact: 3 mantissa bits and exponents 2^-9 .. 2^8
    fit bf16's 7 mantissa bits and 8-bit exponent, so the fp32 bit pattern of the value
    has 16 trailing zero bits.  (Looked up per code in the 256 decoded values.)"""
    f = e4m3_to_f64(np.arange(256, dtype=np.uint8)).astype(np.float32)
    u = f.view(np.uint32)
    finite = np.isfinite(f)
    assert np.all((u[finite] & 0xFFFF) == 0)
    table = (u >> 16).astype(np.uint16)
    return table[np.asarray(codes, dtype=np.uint8)]


def conv3d_acc_e4m3(x8, layout, w8, scale, stride=(1, 1, 1), pads=((0, 0, 0),) * 3,
                    nthreads=0):
    """fp32 accumulator of the convolution of e4m3fn operands times `scale`,
    [N, Do, Ho, Wo, Co]: the plain convolution of the (exact) values, then one
    fp32 rounding of scale * acc."""
    acc = conv3d_acc(e4m3_to_bf16(x8), layout, e4m3_to_bf16(w8), stride, pads, nthreads)
    return (acc.astype(np.float64) * float(np.float32(scale))).astype(np.float32)


def pack_weight_e4m3(w8):
    """OITRS e4m3fn bytes -> OTRSI with Ci zero-padded to a multiple of 128 (bytes)."""
    w8 = np.ascontiguousarray(w8, dtype=np.uint8)
    Co, Ci, KT, KR, KS = w8.shape
    cp = (Ci + 127) // 128 * 128
    out = np.zeros((Co, KT, KR, KS, cp), dtype=np.uint8)
    out[..., :Ci] = np.transpose(w8, (0, 2, 3, 4, 1))
    return out


def upsample2x_nearest(x):
    """Nearest-exact x2 spatial upsampling of NDHWC bf16 bits [N, D, H, W, C] (ROCm/FlyDSL
    PR "Add Qwen-Image VAE classic conv shapes ...", "Upsample Conv2d": the decoder's
    convolution runs at the doubled H x W after it).  At scale 2 the source of output
    (h, w) is (floor((h + 0.5) / 2), floor((w + 0.5) / 2)) = (h // 2, w // 2)."""
    xb = _u16(x)
    return np.ascontiguousarray(np.repeat(np.repeat(xb, 2, axis=2), 2, axis=3))


def upsample2x_conv_acc(x, w, nthreads=0):
    """fp32 accumulator of the 3x3 (KT = 1), zero-pad-1, stride-1 convolution of the x2
    nearest-upsampled NDHWC input: the plain definition, with the upsampled tensor
    written out."""
    return conv3d_acc(upsample2x_nearest(x), NDHWC, w, (1, 1, 1),
                      ((0, 0, PAD_ZERO), (1, 1, PAD_ZERO), (1, 1, PAD_ZERO)), nthreads)


def forward(x, layout, w, stride=(1, 1, 1), pads=((0, 0, 0),) * 3, out_layout=NDHWC,
            flags=0, bias=None, residual=None, residual_bias=None, gamma=None,
            out_pad_br=False, nthreads=0):
    """Reference outputs of one call, as bf16 bits.

    residual is given in `out_layout` with the unpadded output shape.  Returns a
    dict: 'acc' (fp32 NDHWC), 'conv', 'value' (NDHWC and unpadded), and 'y'
    (the call's output in out_layout: act with L2NORM_SILU, else value;
    bottom/right padded when out_pad_br).
    """
    acc = conv3d_acc(x, layout, w, stride, pads, nthreads)
    conv = round_bf16(acc)
    res = None if residual is None else from_layout(_u16(residual), out_layout)
    e = epilogue(conv, flags, bias, res, residual_bias, gamma, nthreads)
    y = e["act"] if flags & L2NORM_SILU else e["value"]
    if out_pad_br:
        y = pad_bottom_right(y)
    return {"acc": acc, "conv": conv, "value": e["value"], "main": e["main"],
            "y": to_layout(y, out_layout)}
