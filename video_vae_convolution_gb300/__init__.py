"""GB300 (sm_103a) video-VAE convolution: thin Python binding of the C ABI.

Everything here is argument marshalling: tensors are allocated with torch (device
memory and streams only) and every step of the computation runs in the CUDA
library ``libvvc_conv3d.so`` (see ``include/conv3d.h``).  There is no fallback:
if the library cannot be built or loaded, the calls raise.
"""

from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Sequence

import torch

from . import build as _build

NCDHW = 0
NDHWC = 1
PAD_ZERO = 0
PAD_REFLECT = 1
DTYPE_BF16 = 0
DTYPE_E4M3 = 1

EPI_BIAS = 1
EPI_RESIDUAL = 2
EPI_RESIDUAL_BIAS = 4
EPI_L2NORM_SILU = 8
EPI_SAVE_VALUE = 16
EPI_OUT_PAD_BR = 32
EPI_PAD_CACHE = 64
EPI_DEBUG_STORE_CONV = 1 << 30

OK = 0
ERR_INVALID_ARG = -1
ERR_UNSUPPORTED = -2
ERR_MISALIGNED = -3
ERR_OVERLAP = -4
ERR_WORKSPACE = -5
ERR_CUDA = -6
ERR_DEVICE_TIMEOUT = -7
ERR_SCRATCH_LIMIT = -8

# ABI version of the C library this binding mirrors (major * 100 + minor).
ABI_VERSION = 320

# Every function the C header declares (checked by the tests against include/conv3d.h).
EXPORTS = (
    "conv3d_packed_weight_bytes", "conv3d_pack_weight", "conv3d_workspace_bytes",
    "conv3d_workspace_bytes_ex", "conv3d_fwd", "conv3d_fwd_ex", "conv3d_launch_count",
    "l2norm_silu", "conv3d_get_device_status", "conv3d_status_string", "conv3d_version",
    "conv3d_struct_size", "conv3d_fwd_static_scratch", "conv3d_plan", "l2norm_silu_pad",
    "group_norm_workspace_bytes", "group_norm_silu", "conv3d_packed_weight_bytes_e4m3",
    "conv3d_pack_weight_e4m3", "conv3d_causal_pack",
)


class Conv3dError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = _lib().conv3d_status_string(status).decode() if _LIB is not None else str(status)
        super().__init__(f"{what}: {msg} ({status})" if what else f"{msg} ({status})")


class Pad(ctypes.Structure):
    _fields_ = [("before", ctypes.c_int32), ("after", ctypes.c_int32), ("mode", ctypes.c_int32)]


class Params(ctypes.Structure):
    _fields_ = [
        ("x", ctypes.c_void_p), ("layout", ctypes.c_int32),
        ("N", ctypes.c_int32), ("Cin", ctypes.c_int32), ("D", ctypes.c_int32),
        ("H", ctypes.c_int32), ("W", ctypes.c_int32),
        ("w_packed", ctypes.c_void_p),
        ("Cout", ctypes.c_int32), ("KT", ctypes.c_int32), ("KR", ctypes.c_int32),
        ("KS", ctypes.c_int32),
        ("stride", ctypes.c_int32 * 3),
        ("pad", Pad * 3),
        ("y", ctypes.c_void_p), ("out_layout", ctypes.c_int32), ("epi", ctypes.c_uint32),
        ("bias", ctypes.c_void_p), ("residual", ctypes.c_void_p),
        ("residual_bias", ctypes.c_void_p), ("gamma", ctypes.c_void_p),
        ("value_out", ctypes.c_void_p), ("conv_out", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("cache_out", ctypes.c_void_p), ("history_frames", ctypes.c_int32),
        ("out_halo", Pad * 3), ("input_upsample", ctypes.c_int32),
        ("dtype", ctypes.c_int32), ("fp8_scale", ctypes.c_float),
    ]


class Tuning(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "tile_w", "tile_h", "R", "kc", "BN", "halo", "stages", "k_splits", "kernel",
        "inject", "timeout_ms", "im2col", "pair", "prefetch", "compact")]

    def __init__(self, **kw):
        super().__init__()
        for k, v in kw.items():
            setattr(self, k, int(v))


class PlanInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "kernel", "mma_n", "stages_per_tile", "k_splits", "paired", "im2col", "launches",
        "grid", "bulk_store", "flat")]


_LIB = None
_lock = threading.Lock()


def _lib():
    global _LIB
    if _LIB is None:
        with _lock:
            if _LIB is None:
                path = _build.LIB_PATH
                if not _build.up_to_date():
                    path = _build.build()
                lib = ctypes.CDLL(path)
                P = ctypes.POINTER(Params)
                T = ctypes.POINTER(Tuning)
                vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
                lib.conv3d_packed_weight_bytes.argtypes = [i32] * 5
                lib.conv3d_packed_weight_bytes.restype = sz
                lib.conv3d_pack_weight.argtypes = [vp] + [i32] * 5 + [vp, vp]
                lib.conv3d_pack_weight.restype = ctypes.c_int
                lib.conv3d_packed_weight_bytes_e4m3.argtypes = [i32] * 5
                lib.conv3d_packed_weight_bytes_e4m3.restype = sz
                lib.conv3d_pack_weight_e4m3.argtypes = [vp] + [i32] * 5 + [vp, vp]
                lib.conv3d_pack_weight_e4m3.restype = ctypes.c_int
                lib.conv3d_workspace_bytes.argtypes = [P, ctypes.POINTER(sz)]
                lib.conv3d_workspace_bytes.restype = ctypes.c_int
                lib.conv3d_workspace_bytes_ex.argtypes = [P, T, ctypes.POINTER(sz)]
                lib.conv3d_workspace_bytes_ex.restype = ctypes.c_int
                lib.conv3d_fwd.argtypes = [P, vp]
                lib.conv3d_fwd.restype = ctypes.c_int
                lib.conv3d_fwd_ex.argtypes = [P, T, vp]
                lib.conv3d_fwd_ex.restype = ctypes.c_int
                lib.conv3d_fwd_static_scratch.argtypes = [P, vp]
                lib.conv3d_fwd_static_scratch.restype = ctypes.c_int
                lib.conv3d_launch_count.argtypes = [P, T]
                lib.conv3d_launch_count.restype = ctypes.c_int
                lib.conv3d_plan.argtypes = [P, T, ctypes.POINTER(PlanInfo)]
                lib.conv3d_plan.restype = ctypes.c_int
                lib.l2norm_silu.argtypes = [vp, i64, i32, vp, vp, vp, vp, vp, vp, vp]
                lib.l2norm_silu.restype = ctypes.c_int
                lib.l2norm_silu_pad.argtypes = [vp] + [i32] * 5 + [vp] * 5 + [i32] + [vp] * 4
                lib.l2norm_silu_pad.restype = ctypes.c_int
                lib.conv3d_causal_pack.argtypes = ([vp, ctypes.POINTER(i64)] + [i32] * 5 +
                                                   [vp, i32, vp, i32, vp, vp])
                lib.conv3d_causal_pack.restype = ctypes.c_int
                lib.group_norm_workspace_bytes.argtypes = [i32] * 7
                lib.group_norm_workspace_bytes.restype = sz
                lib.group_norm_silu.argtypes = ([vp] + [i32] * 7 + [ctypes.c_float, vp, vp, i32, vp,
                                                vp, sz, vp])
                lib.group_norm_silu.restype = ctypes.c_int
                lib.conv3d_get_device_status.argtypes = [ctypes.POINTER(i32), vp]
                lib.conv3d_get_device_status.restype = ctypes.c_int
                lib.conv3d_status_string.argtypes = [ctypes.c_int]
                lib.conv3d_status_string.restype = ctypes.c_char_p
                lib.conv3d_version.argtypes = []
                lib.conv3d_version.restype = ctypes.c_int
                lib.conv3d_struct_size.argtypes = [ctypes.c_int]
                lib.conv3d_struct_size.restype = sz
                if lib.conv3d_version() // 100 != ABI_VERSION // 100:
                    raise RuntimeError(f"library ABI {lib.conv3d_version()}, binding {ABI_VERSION}")
                for which, st in ((0, Params), (1, Tuning), (2, Pad), (3, PlanInfo)):
                    if lib.conv3d_struct_size(which) != ctypes.sizeof(st):
                        raise RuntimeError(f"ABI struct mismatch for {st.__name__}")
                _LIB = lib
    return _LIB


def library_path() -> str:
    _lib()
    return _build.LIB_PATH


def _check(rc: int, what: str):
    if rc != OK:
        raise Conv3dError(rc, what)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


# ---- weights -------------------------------------------------------------------------------

def packed_weight_shape(Cout, Cin, KT, KR, KS):
    return (Cout, KT, KR, KS, (Cin + 63) // 64 * 64)


def pack_weight(w: torch.Tensor, stream=None) -> torch.Tensor:
    """OITRS (or OIRS, read as KT = 1) bf16 CUDA weights -> packed OTRSI tensor."""
    if w.dim() == 4:
        w = w.unsqueeze(2)
    assert w.dim() == 5 and w.dtype == torch.bfloat16 and w.is_cuda
    w = w.contiguous()
    Cout, Cin, KT, KR, KS = w.shape
    out = torch.empty(packed_weight_shape(Cout, Cin, KT, KR, KS), dtype=torch.bfloat16,
                      device=w.device)
    _check(_lib().conv3d_pack_weight(_ptr(w), Cout, Cin, KT, KR, KS, _ptr(out), _stream(stream)),
           "conv3d_pack_weight")
    return out


def packed_weight_shape_e4m3(Cout, Cin, KT, KR, KS):
    return (Cout, KT, KR, KS, (Cin + 127) // 128 * 128)


def pack_weight_e4m3(w: torch.Tensor, stream=None) -> torch.Tensor:
    """OITRS (or OIRS) e4m3fn CUDA weights (torch.float8_e4m3fn, or their bytes as
    torch.uint8) -> packed OTRSI bytes (torch.uint8) for dtype=DTYPE_E4M3 calls."""
    if w.dim() == 4:
        w = w.unsqueeze(2)
    assert w.dim() == 5 and w.element_size() == 1 and w.is_cuda
    w = w.contiguous()
    Cout, Cin, KT, KR, KS = w.shape
    out = torch.empty(packed_weight_shape_e4m3(Cout, Cin, KT, KR, KS), dtype=torch.uint8,
                      device=w.device)
    _check(_lib().conv3d_pack_weight_e4m3(_ptr(w), Cout, Cin, KT, KR, KS, _ptr(out),
                                          _stream(stream)), "conv3d_pack_weight_e4m3")
    return out


# ---- convolution -----------------------------------------------------------------------------

def out_dims(D, H, W, kernel, stride, pads):
    L = (D, H, W)
    return tuple((L[i] + pads[i][0] + pads[i][1] - kernel[i]) // stride[i] + 1 for i in range(3))


def _dims(x: torch.Tensor, layout: int):
    if x.dim() == 4:  # rank-4 NCHW / NHWC: D = 1
        if layout == NCDHW:
            N, C, H, W = x.shape
        else:
            N, H, W, C = x.shape
        return N, C, 1, H, W
    if layout == NCDHW:
        N, C, D, H, W = x.shape
    else:
        N, D, H, W, C = x.shape
    return N, C, D, H, W


def out_shape(N, Cout, Do, Ho, Wo, layout, pad_br=False):
    if pad_br:
        Ho, Wo = Ho + 1, Wo + 1
    return (N, Cout, Do, Ho, Wo) if layout == NCDHW else (N, Do, Ho, Wo, Cout)


class Conv3d:
    """One prepared convolution call: builds the C parameter block once so that
    ``run()`` is a single C call (cheap enough for timing loops and CUDA graphs).

    x: bf16 CUDA tensor in `layout` (5-D, or 4-D with D = 1).  w_packed from
    pack_weight.  pads: ((before, after, mode) for T, H, W).  Outputs are allocated
    here unless given; the workspace is allocated here (torch) unless given.
    dtype=DTYPE_E4M3: x holds e4m3fn bytes (NDHWC), w_packed comes from
    pack_weight_e4m3 and the accumulator is multiplied by fp8_scale; y stays bf16.
    """

    def __init__(self, x, w_packed, Cout, kernel, stride=(1, 1, 1),
                 pads=((0, 0, PAD_ZERO),) * 3, layout=NDHWC, out_layout=NDHWC, epi=0,
                 bias=None, residual=None, residual_bias=None, gamma=None, y=None,
                 value_out=None, conv_out=None, workspace=None, tuning: Optional[Tuning] = None,
                 cache_out=None, history_frames=0, out_halo=None, input_upsample=0,
                 dtype=DTYPE_BF16, fp8_scale=1.0):
        N, C, D, H, W = _dims(x, layout)
        KT, KR, KS = kernel
        up = 2 if input_upsample == 2 else 1  # the convolution reads the x2 upsampled grid
        Do, Ho, Wo = out_dims(D, H * up, W * up, kernel, stride, pads)
        dev = x.device
        self.dims = (N, C, D, H, W)
        self.out_dims = (Do, Ho, Wo)
        pad_br = bool(epi & EPI_OUT_PAD_BR)
        if y is None and epi & EPI_PAD_CACHE:
            # padded output: two leading planes and a one-pixel spatial border
            y = torch.empty((N, Do + 2, Ho + 2, Wo + 2, Cout), dtype=torch.bfloat16, device=dev)
        if out_halo is not None and y is None:
            # haloed NDHWC output; zeros, so that the unwritten T halo frames read 0
            (tb, ta, _), (hb, ha, _), (wb, wa, _) = out_halo
            y = torch.zeros((N, Do + tb + ta, Ho + hb + ha, Wo + wb + wa, Cout),
                            dtype=torch.bfloat16, device=dev)
        if y is None:
            y = torch.empty(out_shape(N, Cout, Do, Ho, Wo, out_layout, pad_br),
                            dtype=torch.bfloat16, device=dev)
        if epi & EPI_PAD_CACHE and cache_out is None:
            cache_out = torch.empty((N, min(2, Do + history_frames), Ho, Wo, Cout),
                                    dtype=torch.bfloat16, device=dev)
        if epi & EPI_SAVE_VALUE and value_out is None:
            value_out = torch.empty(out_shape(N, Cout, Do, Ho, Wo, out_layout),
                                    dtype=torch.bfloat16, device=dev)
        if epi & EPI_DEBUG_STORE_CONV and conv_out is None:
            conv_out = torch.empty((N, Do, Ho, Wo, Cout), dtype=torch.bfloat16, device=dev)
        p = Params()
        p.x = x.data_ptr()
        p.layout = layout
        p.N, p.Cin, p.D, p.H, p.W = N, C, D, H, W
        p.w_packed = w_packed.data_ptr()
        p.Cout, p.KT, p.KR, p.KS = Cout, KT, KR, KS
        for i in range(3):
            p.stride[i] = stride[i]
            p.pad[i].before, p.pad[i].after, p.pad[i].mode = pads[i]
        p.y = y.data_ptr()
        p.out_layout = out_layout
        p.epi = epi
        p.bias = None if bias is None else bias.data_ptr()
        p.residual = None if residual is None else residual.data_ptr()
        p.residual_bias = None if residual_bias is None else residual_bias.data_ptr()
        p.gamma = None if gamma is None else gamma.data_ptr()
        p.value_out = None if value_out is None else value_out.data_ptr()
        p.conv_out = None if conv_out is None else conv_out.data_ptr()
        p.cache_out = None if cache_out is None else cache_out.data_ptr()
        p.history_frames = history_frames
        if out_halo is not None:
            for i in range(3):
                p.out_halo[i].before, p.out_halo[i].after, p.out_halo[i].mode = out_halo[i]
        p.input_upsample = input_upsample
        p.dtype = dtype
        p.fp8_scale = fp8_scale
        self.out_halo = out_halo
        self.cache_out = cache_out
        self.tuning = tuning
        tp = ctypes.byref(tuning) if tuning is not None else None
        nbytes = ctypes.c_size_t(0)
        _check(_lib().conv3d_workspace_bytes_ex(ctypes.byref(p), tp, ctypes.byref(nbytes)),
               "conv3d_workspace_bytes")
        self.workspace_bytes = nbytes.value
        if workspace is None and nbytes.value > 0:
            workspace = torch.empty(nbytes.value, dtype=torch.uint8, device=dev)
        p.workspace = None if workspace is None else workspace.data_ptr()
        p.workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        self.params = p
        # keep every buffer alive as long as the call object
        self.x, self.w_packed, self.y = x, w_packed, y
        self.value_out, self.conv_out, self.workspace = value_out, conv_out, workspace
        self.bias, self.residual, self.residual_bias, self.gamma = bias, residual, residual_bias, gamma
        self.launches = _lib().conv3d_launch_count(ctypes.byref(p), tp)
        self.plan = PlanInfo()
        _check(_lib().conv3d_plan(ctypes.byref(p), tp, ctypes.byref(self.plan)), "conv3d_plan")

    def run(self, stream=None) -> int:
        tp = ctypes.byref(self.tuning) if self.tuning is not None else None
        return _lib().conv3d_fwd_ex(ctypes.byref(self.params), tp, _stream(stream))

    def __call__(self, stream=None):
        _check(self.run(stream), "conv3d_fwd")
        return self.y


class Chain:
    """A fixed sequence of prepared calls (Conv3d objects, e.g. the layers of an
    encoder whose outputs feed the next call) recorded once as a CUDA graph: run()
    replays every kernel launch of the sequence with one graph launch, without the
    per-launch host and queue gaps of issuing the calls one by one.  The calls keep
    their buffers, tensor maps and plans from recording time; refill their inputs in
    place between runs.  Every call runs once eagerly first (kernel attributes, the
    first-call device set-up), then the sequence is captured on a side stream."""

    def __init__(self, calls, stream=None):
        self.calls = list(calls)
        s = stream if stream is not None else torch.cuda.current_stream()
        for c in self.calls:
            _check(c.run(s), "conv3d_fwd")
        side = torch.cuda.Stream(device=s.device)
        side.wait_stream(s)
        torch.cuda.synchronize(s.device)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=side):
            for c in self.calls:
                _check(c.run(side), "conv3d_fwd (graph capture)")
        torch.cuda.synchronize(s.device)
        self.launches = sum(c.launches for c in self.calls)

    def run(self, stream=None):
        """Replays the recorded launches on `stream` (default: the current stream)."""
        if stream is None:
            self.graph.replay()
        else:
            with torch.cuda.stream(stream):
                self.graph.replay()


def conv3d(x, w_packed, Cout, kernel, **kw):
    """Runs one convolution; returns y (and fills value_out / conv_out if asked)."""
    c = Conv3d(x, w_packed, Cout, kernel, **kw)
    c()
    if kw.get("epi", 0) & (EPI_SAVE_VALUE | EPI_DEBUG_STORE_CONV):
        return {"y": c.y, "value": c.value_out, "conv": c.conv_out}
    return c.y


def l2norm_silu(x: torch.Tensor, gamma: torch.Tensor, input_bias=None, residual=None,
                residual_bias=None, save_value=False, y=None, stream=None):
    """Standalone post-operations on channels-last bf16 x [..., C]; returns y
    (and the pre-normalisation value when save_value)."""
    C = x.shape[-1]
    rows = x.numel() // C
    if y is None:
        y = torch.empty_like(x)
    value = torch.empty_like(x) if save_value else None
    _check(_lib().l2norm_silu(_ptr(x), rows, C, _ptr(input_bias), _ptr(residual),
                              _ptr(residual_bias), _ptr(gamma), _ptr(y), _ptr(value),
                              _stream(stream)), "l2norm_silu")
    return (y, value) if save_value else y


def l2norm_silu_pad(x: torch.Tensor, gamma: torch.Tensor, input_bias=None, residual=None,
                    residual_bias=None, previous=None, save_value=False, padded=None,
                    cache=None, stream=None):
    """Standalone post-operations with padded output and cache on channels-last bf16
    x [N, T, H, W, C] (C % 8 == 0); previous: None or 1-2 prior activated frames
    [N, P, H, W, C].  Returns (padded [N, T+2, H+2, W+2, C], cache
    [N, min(2, T+P), H, W, C], value or None)."""
    N, T, H, W, C = x.shape
    P = 0 if previous is None else previous.shape[1]
    if padded is None:
        padded = torch.empty((N, T + 2, H + 2, W + 2, C), dtype=x.dtype, device=x.device)
    if cache is None:
        cache = torch.empty((N, min(2, T + P), H, W, C), dtype=x.dtype, device=x.device)
    value = torch.empty_like(x) if save_value else None
    _check(_lib().l2norm_silu_pad(_ptr(x), N, T, H, W, C, _ptr(input_bias), _ptr(residual),
                                  _ptr(residual_bias), _ptr(gamma), _ptr(previous), P,
                                  _ptr(padded), _ptr(cache), _ptr(value), _stream(stream)),
           "l2norm_silu_pad")
    return padded, cache, value


def causal_pack(x: torch.Tensor, previous=None, Cp=None, padded=None, cache=None, stream=None):
    """Input packing of a streaming causal 3x3x3 convolution (conv3d_causal_pack): x is
    the chunk [N, C, T, H, W] (any strided bf16 CUDA view), previous the raw history
    [N, P, H, W, C] (P <= 2) or None.  Returns (padded [N, T+2, H+2, W+2, Cp], cache
    [N, min(2, T+P), H, W, C]); Cp defaults to C rounded up to 16."""
    N, C, T, H, W = x.shape
    P = 0 if previous is None else previous.shape[1]
    if Cp is None:
        Cp = (C + 15) // 16 * 16
    if padded is None:
        padded = torch.empty((N, T + 2, H + 2, W + 2, Cp), dtype=x.dtype, device=x.device)
    if cache is None:
        cache = torch.empty((N, min(2, T + P), H, W, C), dtype=x.dtype, device=x.device)
    strides = (ctypes.c_int64 * 5)(*x.stride())
    _check(_lib().conv3d_causal_pack(_ptr(x), strides, N, C, T, H, W, _ptr(previous), P,
                                     _ptr(padded), Cp, _ptr(cache), _stream(stream)),
           "conv3d_causal_pack")
    return padded, cache


class CausalConv3dWithCache:
    """Streaming causal 3x3x3 convolution over chunks of an NCTHW video (cuDNN frontend
    doc, "Causal Conv3D with Cache"): each call packs the chunk after the history of the
    previous one (conv3d_causal_pack) and runs the valid convolution over the packed
    input (conv3d_fwd, no bias).  Buffers are sized for one chunk shape and reused, so
    the calls of a fixed shape can be captured in a CUDA graph.

    w_packed: pack_weight of the [Cout, C, 3, 3, 3] weights.  history_frames: P of the
    calls (0 for the first chunk of a video, then min(2, frames so far)).
    """

    def __init__(self, chunk_shape, w_packed, Cout, history_frames=0, Cp=None,
                 device="cuda", tuning: Optional[Tuning] = None):
        N, C, T, H, W = chunk_shape
        self.Cp = (C + 15) // 16 * 16 if Cp is None else Cp
        self.P = history_frames
        self.padded = torch.empty((N, T + 2, H + 2, W + 2, self.Cp), dtype=torch.bfloat16,
                                  device=device)
        self.cache = torch.empty((N, min(2, T + history_frames), H, W, C), dtype=torch.bfloat16,
                                 device=device)
        self.conv = Conv3d(self.padded, w_packed, Cout, (3, 3, 3), (1, 1, 1),
                           ((0, 0, PAD_ZERO),) * 3, NDHWC, NDHWC, 0, tuning=tuning)
        self.launches = 1 + self.conv.launches

    def __call__(self, x: torch.Tensor, previous=None, stream=None):
        """Returns (output [N, T, H, W, Cout], cache [N, min(2, T+P), H, W, C])."""
        if (0 if previous is None else previous.shape[1]) != self.P:
            raise Conv3dError(ERR_INVALID_ARG, "CausalConv3dWithCache: history frames")
        causal_pack(x, previous, self.Cp, self.padded, self.cache, stream)
        return self.conv(stream), self.cache


def group_norm_silu(x: torch.Tensor, groups: int, gamma=None, beta=None, eps=1e-6,
                    time_isolated=True, silu=True, y=None, workspace=None, stream=None):
    """Channels-last GroupNorm (+ SiLU) of bf16 x [N, D, H, W, C] (C % 8 == 0): per
    frame when time_isolated, else per clip; returns y (same shape)."""
    N, D, H, W, C = x.shape
    if y is None:
        y = torch.empty_like(x)
    nbytes = _lib().group_norm_workspace_bytes(N, D, H, W, C, groups, int(time_isolated))
    if nbytes == 0:
        raise Conv3dError(ERR_INVALID_ARG, "group_norm_silu")
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=x.device)
    _check(_lib().group_norm_silu(_ptr(x), N, D, H, W, C, groups, int(time_isolated), eps,
                                  _ptr(gamma), _ptr(beta), int(silu), _ptr(y), _ptr(workspace),
                                  workspace.numel(), _stream(stream)), "group_norm_silu")
    return y


def device_status(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device status word."""
    v = ctypes.c_int32(0)
    _check(_lib().conv3d_get_device_status(ctypes.byref(v), _stream(stream)),
           "conv3d_get_device_status")
    return v.value
