"""Host-side checks of the CUDA library that need no GPU: it builds, loads,
exports every function include/conv3d.h declares, its ABI structs match the
binding, and argument validation rejects bad calls before launching anything.
"""

import ctypes
import os
import re

import pytest

import video_vae_convolution_gb300 as vvc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    text = open(os.path.join(ROOT, "include", "conv3d.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(",
                       text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while", "sizeof")))


def test_library_loads_and_exports_header():
    lib = vvc._lib()
    declared = header_functions()
    assert len(declared) >= 10
    for name in declared:
        assert hasattr(lib, name), f"{name} declared in conv3d.h but not exported"
    assert sorted(declared) == sorted(vvc.EXPORTS)
    assert lib.conv3d_version() // 100 == vvc.ABI_VERSION // 100
    assert lib.conv3d_status_string(vvc.ERR_OVERLAP) == b"output or workspace overlaps another buffer"


def test_packed_weight_bytes():
    lib = vvc._lib()
    assert lib.conv3d_packed_weight_bytes(96, 96, 3, 3, 3) == 96 * 27 * 128 * 2
    assert lib.conv3d_packed_weight_bytes(128, 3, 3, 3, 3) == 128 * 27 * 64 * 2
    assert lib.conv3d_packed_weight_bytes(0, 3, 3, 3, 3) == 0


def _params(**kw):
    p = vvc.Params()
    p.x, p.w_packed, p.y = 0x100000, 0x200000, 0x10000000
    p.layout = p.out_layout = vvc.NDHWC
    p.N, p.Cin, p.D, p.H, p.W = 1, 16, 4, 12, 12
    p.Cout, p.KT, p.KR, p.KS = 32, 3, 3, 3
    for i in range(3):
        p.stride[i] = 1
        p.pad[i].before = p.pad[i].after = 1
        p.pad[i].mode = vvc.PAD_ZERO
    for k, v in kw.items():
        setattr(p, k, v)
    return p


def fwd(p, t=None):
    return vvc._lib().conv3d_fwd_ex(ctypes.byref(p), None if t is None else ctypes.byref(t), None)


def test_validation_rejects_before_launch():
    assert fwd(_params(Cin=0)) == vvc.ERR_INVALID_ARG
    assert fwd(_params(layout=7)) == vvc.ERR_INVALID_ARG
    assert fwd(_params(x=None)) == vvc.ERR_INVALID_ARG
    p = _params()
    p.stride[1] = 0
    assert fwd(p) == vvc.ERR_INVALID_ARG
    p = _params(epi=vvc.EPI_RESIDUAL_BIAS, residual_bias=0x300000)
    assert fwd(p) == vvc.ERR_INVALID_ARG                     # residual_bias needs residual
    p = _params(epi=vvc.EPI_L2NORM_SILU)
    assert fwd(p) == vvc.ERR_INVALID_ARG                     # gamma missing
    p = _params(epi=vvc.EPI_L2NORM_SILU | vvc.EPI_OUT_PAD_BR, gamma=0x300000)
    assert fwd(p) == vvc.ERR_INVALID_ARG                     # pad variant stops at value
    p = _params(W=2)
    p.pad[2].before = p.pad[2].after = 0
    assert fwd(p) == vvc.ERR_INVALID_ARG                     # output extent < 1
    p = _params()
    p.pad[1].mode = vvc.PAD_REFLECT
    p.pad[1].before = 12
    assert fwd(p) == vvc.ERR_INVALID_ARG                     # reflect pad >= extent
    p = _params()
    p.pad[0].mode = vvc.PAD_REFLECT
    assert fwd(p) == vvc.ERR_UNSUPPORTED                     # no reflect along T
    p = _params(epi=vvc.EPI_L2NORM_SILU, gamma=0x300000, Cout=640)
    assert fwd(p) == vvc.ERR_UNSUPPORTED


def test_alignment_overlap_workspace():
    one = vvc.Tuning(k_splits=1)
    assert fwd(_params(x=0x100008), one) == vvc.ERR_MISALIGNED
    assert fwd(_params(y=0x100000), one) == vvc.ERR_OVERLAP   # y on top of x
    p = _params(epi=vvc.EPI_SAVE_VALUE, value_out=0x10000010)
    assert fwd(p, one) == vvc.ERR_OVERLAP                     # value_out inside y
    p = _params(layout=vvc.NCDHW)                             # NCDHW input needs staging
    assert fwd(p, one) == vvc.ERR_WORKSPACE
    n = ctypes.c_size_t(0)
    assert vvc._lib().conv3d_workspace_bytes(ctypes.byref(p), ctypes.byref(n)) == vvc.OK
    assert n.value >= 1 * 16 * 4 * 12 * 12 * 2
    p.workspace, p.workspace_bytes = 0x100000, n.value         # workspace overlapping x
    assert fwd(p) == vvc.ERR_OVERLAP
    p.workspace, p.workspace_bytes = 0x40000000, n.value - 16  # too small
    assert fwd(p) == vvc.ERR_WORKSPACE


def test_workspace_and_launch_plan():
    lib = vvc._lib()
    p = _params()
    n = ctypes.c_size_t(1)
    assert lib.conv3d_workspace_bytes(ctypes.byref(p), ctypes.byref(n)) == vvc.OK
    t = vvc.Tuning(k_splits=3)
    assert lib.conv3d_workspace_bytes_ex(ctypes.byref(p), ctypes.byref(t), ctypes.byref(n)) == 0
    Do, Ho, Wo = 4, 12, 12
    assert n.value >= 3 * Do * Ho * Wo * 32 * 4
    assert lib.conv3d_launch_count(ctypes.byref(p), ctypes.byref(t)) == 2   # conv + reduce
    assert lib.conv3d_launch_count(ctypes.byref(_params(Cin=3)), None) >= 2  # staging
    assert lib.conv3d_launch_count(ctypes.byref(_params(Cin=64, Cout=64)),
                                   ctypes.byref(vvc.Tuning(k_splits=1))) == 1


def _plan(p, t=None):
    info = vvc.PlanInfo()
    rc = vvc._lib().conv3d_plan(ctypes.byref(p), None if t is None else ctypes.byref(t),
                                ctypes.byref(info))
    assert rc == vvc.OK
    return info


def _valid(**kw):
    p = _params(**kw)
    for i in range(3):
        p.pad[i].before = p.pad[i].after = 0
    return p


def test_plan_paired_last_chunks():
    # 96 input channels = one 64-channel chunk + 32: with paired last chunks a 3x3x3
    # tile runs 9 full stages + ceil(9 / 2) shared ones instead of 9 + 9
    p = _valid(Cin=96, Cout=96, D=6, H=354, W=642)
    on = _plan(p)
    off = _plan(p, vvc.Tuning(pair=2))
    assert (on.kernel, on.paired, on.stages_per_tile, on.k_splits) == (2, 1, 14, 1)
    assert (off.paired, off.stages_per_tile) == (0, 18)
    assert on.mma_n == off.mma_n == 256
    # 1x3x3 (T = 1): 3 tap pairs -> 2 full stages + ceil(3 / 2) shared ones
    t1 = _valid(N=4, Cin=96, Cout=96, D=1, H=353, W=641, KT=1)
    assert (_plan(t1).paired, _plan(t1).stages_per_tile) == (1, 5)
    assert (_plan(t1, vvc.Tuning(pair=2)).paired, _plan(t1, vvc.Tuning(pair=2)).stages_per_tile) == (0, 6)
    # 160 channels: two full chunks per pair + shared last chunks (9 * 2 + 5)
    assert _plan(_valid(Cin=160, Cout=160, D=8, H=106, W=182)).stages_per_tile == 23
    # not paired: whole chunks (128), last chunk over 32 channels (112), a split
    # reduction, reflect padding along W, a single tap pair (1x1x1)
    assert _plan(_valid(Cin=128, Cout=128, D=6, H=354, W=642)).paired == 0
    assert _plan(_valid(Cin=112, Cout=96, D=6, H=354, W=642)).paired == 0
    assert _plan(p, vvc.Tuning(k_splits=2)).paired == 0
    rw = _params(Cin=96, Cout=96, D=6, H=66, W=130)
    rw.pad[2].mode = vvc.PAD_REFLECT
    assert _plan(rw).paired == 0
    assert _plan(_valid(Cin=96, Cout=96, KT=1, KR=1, KS=1)).paired == 0


def _causal(**kw):
    p = _valid(**kw)
    p.pad[0].before = 2
    return p


def test_plan_compact_volume_tiles():
    # 256 -> 256 on [9, 64, 64] with a 1-pixel halo input and the causal T padding: the
    # per-frame flat tiles need 17 x 9 = 153 tiles of 256 positions per channel tile
    # (3 rounds of 306 work items on 152 SMs, so 208-wide tiles); the volume without the
    # two halo rows under each frame needs 149 (298 work items, 2 rounds)
    p = _causal(Cin=256, Cout=256, D=9, H=66, W=66)
    auto, off = _plan(p), _plan(p, vvc.Tuning(compact=2))
    assert (auto.flat, auto.mma_n, auto.k_splits) == (3, 256, 1)
    assert (off.flat, off.mma_n) == (1, 208)
    # 16x16 planes with a halo (the ladder's 512 -> 512 at [5, 16, 16]): 6 compact
    # tiles against 7 volume tiles that include the halo rows
    small = _causal(Cin=512, Cout=512, D=5, H=18, W=18)
    assert _plan(small).flat == 3
    assert _plan(small, vvc.Tuning(compact=2)).flat == 2
    # forced on where it saves nothing (256^2 planes: the same 258 tiles per frame)
    big = _causal(Cin=128, Cout=128, D=3, H=66, W=258)
    assert _plan(big).flat == 1
    assert _plan(big, vvc.Tuning(compact=1)).flat == 3
    # not applicable: H zero padding in the call (flat volume tiles need none), a T
    # padding outside the im2col corner range [-16, 15], one frame, NCDHW output, the
    # fused norm
    hp = _params(Cin=64, Cout=64, D=5, H=16, W=18)
    hp.pad[2].before = hp.pad[2].after = 0
    assert _plan(hp, vvc.Tuning(compact=1)).flat != 3
    far = _causal(Cin=64, Cout=64, D=40, H=18, W=18, KT=1)
    far.pad[0].before = 17
    assert _plan(far, vvc.Tuning(compact=1)).flat != 3
    # a partial last channel chunk (112 = 64 + 48 channels)
    assert _plan(_causal(Cin=112, Cout=64, D=5, H=18, W=18),
                 vvc.Tuning(compact=1, pair=2)).flat != 3
    # im2col offsets beyond the measured 0..2 (a 5-tap temporal kernel)
    assert _plan(_causal(Cin=64, Cout=64, D=9, H=18, W=18, KT=5),
                 vvc.Tuning(compact=1)).flat != 3
    assert _plan(_valid(Cin=64, Cout=64, D=1, H=18, W=18, KT=1),
                 vvc.Tuning(compact=1)).flat != 3
    nc = _causal(Cin=64, Cout=64, D=5, H=18, W=18)
    nc.out_layout = vvc.NCDHW
    assert _plan(nc, vvc.Tuning(compact=1)).flat != 3
    nm = _causal(Cin=64, Cout=64, D=5, H=18, W=18)
    nm.epi, nm.gamma = vvc.EPI_L2NORM_SILU, 0x300000
    assert _plan(nm, vvc.Tuning(compact=1)).flat != 3
    # e4m3 operands plan the same convolution over channel pairs: the same compact tiles
    f8 = _causal(Cin=256, Cout=256, D=9, H=66, W=66, dtype=vvc.DTYPE_E4M3, fp8_scale=1.0)
    assert (_plan(f8).flat, _plan(f8).mma_n) == (3, 256)
    # never with paired last chunks (their half-width copies use the tiled map): a
    # 96-channel input keeps the tiled volume tiles and pairs its last chunks
    pr = _causal(Cin=96, Cout=64, D=6, H=14, W=14)
    info = _plan(pr, vvc.Tuning(compact=1, k_splits=1))
    assert info.flat == 2 and info.paired == 1


def test_causal_pack_validation():
    lib = vvc._lib()
    st = (ctypes.c_int64 * 5)(12 * 4 * 8 * 10, 4 * 8 * 10, 8 * 10, 10, 1)  # contiguous NCTHW

    def call(x=0x100000, strides=st, N=1, C=12, T=4, H=8, W=10, prev=None, P=0,
             padded=0x200000, Cp=16, cache=0x300000):
        return lib.conv3d_causal_pack(x, strides, N, C, T, H, W, prev, P, padded, Cp, cache,
                                      None)

    assert call(x=None) == vvc.ERR_INVALID_ARG
    assert call(strides=None) == vvc.ERR_INVALID_ARG
    assert call(Cp=8) == vvc.ERR_INVALID_ARG                 # Cp < C
    assert call(Cp=20) == vvc.ERR_INVALID_ARG                # Cp not a multiple of 8
    assert call(P=3, prev=0x400000) == vvc.ERR_INVALID_ARG   # at most two history frames
    assert call(P=1) == vvc.ERR_INVALID_ARG                  # history frames without history
    assert call(prev=0x400000) == vvc.ERR_INVALID_ARG        # history without frames
    neg = (ctypes.c_int64 * 5)(0, 1, 0, 0, -1)
    assert call(strides=neg) == vvc.ERR_INVALID_ARG
    assert call(x=0x100001) == vvc.ERR_MISALIGNED
    assert call(prev=0x400004, P=2) == vvc.ERR_MISALIGNED    # history: 8-byte alignment
    assert call(padded=0x200008) == vvc.ERR_MISALIGNED
    assert call(cache=0x300008) == vvc.ERR_MISALIGNED
    assert call(padded=0x100000 + 4096) == vvc.ERR_OVERLAP   # padded over the chunk
    assert call(cache=0x200000 + 4096) == vvc.ERR_OVERLAP    # cache over padded


# The plans of the benchmark's chained ladder (spatially haloed inputs, causal T padding
# in each call, haloed outputs but for the last call) on 152 SMs, as measured: tile form
# (0 rows, 1 per-frame runs, 3 compact volume runs), MMA N, stages per tile, splits.
LADDER_PLANS = {
    "conv_in": (1, 256, 3, 1), "L0_0": (1, 256, 18, 1), "L0s": (0, 256, 54, 1),
    "L1a": (1, 256, 18, 1), "L1_0": (1, 256, 36, 1), "L1s": (0, 256, 108, 1),
    "L2_0": (3, 256, 36, 1), "L2s": (0, 256, 108, 3), "L3a": (3, 256, 36, 3),
    "L3_0": (3, 256, 72, 3), "L3s": (0, 256, 216, 7), "L4_0": (3, 256, 72, 6),
    "L5a": (3, 256, 72, 3), "L5_0": (3, 256, 144, 3), "conv_out": (3, 256, 144, 16),
}


def test_ladder_chain_plans():
    import workloads as wl
    calls = wl.ladder().calls
    causal_t = ((2, 0, vvc.PAD_ZERO), (0, 0, vvc.PAD_ZERO), (0, 0, vvc.PAD_ZERO))
    halo = ((0, 0, vvc.PAD_ZERO), (1, 1, vvc.PAD_REFLECT), (1, 1, vvc.PAD_REFLECT))
    seen = 0
    for i, call in enumerate(calls):
        first, last = i == 0, i == len(calls) - 1
        p = vvc.Params()
        p.x, p.w_packed, p.y = 0x100000000, 0x200000000, 0x400000000
        p.workspace, p.workspace_bytes = 0x800000000, 1 << 34
        p.layout = p.out_layout = vvc.NDHWC
        p.N, p.Cin, p.Cout = call.N, call.Cin, call.Cout
        p.D, p.H, p.W = call.D, call.H + (0 if first else 2), call.W + (0 if first else 2)
        p.KT, p.KR, p.KS = call.kernel
        pads = ([(b, a, vvc.PAD_ZERO if m == wl.ZERO else vvc.PAD_REFLECT)
                 for b, a, m in call.pads] if first else causal_t)
        for d in range(3):
            p.stride[d] = call.stride[d]
            p.pad[d].before, p.pad[d].after, p.pad[d].mode = pads[d]
            if not last:
                p.out_halo[d].before, p.out_halo[d].after, p.out_halo[d].mode = halo[d]
        info = _plan(p)
        assert info.kernel == 2, call.name
        if call.name in LADDER_PLANS:
            seen += 1
            got = (info.flat, info.mma_n, info.stages_per_tile, info.k_splits)
            assert got == LADDER_PLANS[call.name], (call.name, got)
    assert seen == len(LADDER_PLANS)


def test_plan_bulk_store():
    # NCDHW output takes bulk stores when its rows are 16-byte multiples (Wo % 8 == 0)
    # and no NDHWC debug store runs beside them; NDHWC when Cout % 8 == 0
    nc = _valid(Cin=96, Cout=96, D=6, H=354, W=642)
    nc.out_layout = vvc.NCDHW
    assert _plan(nc).bulk_store == 1
    assert _plan(_valid(Cin=96, Cout=96, D=6, H=354, W=642)).bulk_store == 1
    odd = _valid(Cin=96, Cout=96, N=4, D=1, H=353, W=641, KT=1)   # Wo = 639
    odd.out_layout = vvc.NCDHW
    assert _plan(odd).bulk_store == 0
    nc.epi, nc.conv_out = vvc.EPI_DEBUG_STORE_CONV, 0x40000000
    assert _plan(nc).bulk_store == 0
    nc.epi, nc.residual = vvc.EPI_RESIDUAL, 0x50000000
    assert _plan(nc).bulk_store == 0


def test_l2norm_validation():
    lib = vvc._lib()
    assert lib.l2norm_silu(None, 10, 16, None, None, None, 0x1000, 0x2000, None, None) == \
        vvc.ERR_INVALID_ARG
    assert lib.l2norm_silu(0x1000, 10, 16, None, None, 0x3000, 0x4000, 0x5000, None, None) == \
        vvc.ERR_INVALID_ARG
    assert lib.l2norm_silu(0x1000, 10, 16, None, None, None, 0x4000, 0x1010, None, None) == \
        vvc.ERR_OVERLAP
    assert lib.l2norm_silu(0x1002, 10, 16, None, None, None, 0x4000, 0x8000, None, None) == \
        vvc.ERR_MISALIGNED


def test_pad_cache_validation_and_plan():
    lib = vvc._lib()
    base = dict(Cin=32, Cout=40, D=5, H=7, W=9)
    p = _valid(**base)
    p.epi = vvc.EPI_L2NORM_SILU | vvc.EPI_PAD_CACHE
    p.gamma, p.cache_out, p.history_frames = 0x300000, 0x40000000, 1
    n_pc, n = ctypes.c_size_t(0), ctypes.c_size_t(0)
    assert lib.conv3d_workspace_bytes_ex(ctypes.byref(p), None, ctypes.byref(n_pc)) == vvc.OK
    q = _valid(**base)
    q.epi, q.gamma = vvc.EPI_L2NORM_SILU, 0x300000
    assert lib.conv3d_workspace_bytes_ex(ctypes.byref(q), None, ctypes.byref(n)) == vvc.OK
    # the contiguous activations [N, Do, Ho, Wo, Cout] sit after the call's own scratch
    assert n_pc.value >= n.value + 3 * 5 * 7 * 40 * 2
    assert _plan(p).launches == _plan(q).launches + 1
    for bad in (dict(epi=vvc.EPI_PAD_CACHE),                                 # no norm
                dict(history_frames=3), dict(history_frames=-1),
                dict(cache_out=None), dict(out_layout=vvc.NCDHW)):
        r = _valid(**base)
        r.epi = vvc.EPI_L2NORM_SILU | vvc.EPI_PAD_CACHE
        r.gamma, r.cache_out, r.history_frames = 0x300000, 0x40000000, 1
        for k, v in bad.items():
            setattr(r, k, v)
        assert lib.conv3d_launch_count(ctypes.byref(r), None) == vvc.ERR_INVALID_ARG, bad
    r = _valid(Cin=32, Cout=36, D=5, H=7, W=9)                              # Cout % 8 != 0
    r.epi = vvc.EPI_L2NORM_SILU | vvc.EPI_PAD_CACHE
    r.gamma, r.cache_out = 0x300000, 0x40000000
    assert lib.conv3d_launch_count(ctypes.byref(r), None) == vvc.ERR_INVALID_ARG


def test_l2norm_silu_pad_validation():
    lib = vvc._lib()
    a = dict(x=0x100000, g=0x200000, padded=0x10000000, cache=0x20000000)

    def call(N=1, T=2, H=3, W=4, C=16, prev=None, P=0, **kw):
        d = dict(a, **kw)
        return lib.l2norm_silu_pad(d["x"], N, T, H, W, C, None, None, None, d["g"], prev, P,
                                   d["padded"], d["cache"], None, None)
    assert call(C=12) == vvc.ERR_INVALID_ARG                 # C % 8 != 0
    assert call(P=1) == vvc.ERR_INVALID_ARG                  # history without frames
    assert call(prev=0x30000000, P=0) == vvc.ERR_INVALID_ARG  # frames without a count
    assert call(prev=0x30000000, P=3) == vvc.ERR_INVALID_ARG
    assert call(g=0) == vvc.ERR_INVALID_ARG
    assert call(x=0x100008) == vvc.ERR_MISALIGNED
    assert call(padded=0x100000 + 64) == vvc.ERR_OVERLAP    # padded output over the input
    assert call(cache=0x10000000 + 32) == vvc.ERR_OVERLAP   # cache over the padded output


def test_group_norm_validation():
    lib = vvc._lib()
    assert lib.group_norm_workspace_bytes(1, 2, 3, 4, 128, 32, 1) > 0
    assert lib.group_norm_workspace_bytes(1, 2, 3, 4, 120, 32, 1) == 0   # groups must divide C
    assert lib.group_norm_workspace_bytes(1, 2, 3, 4, 12, 4, 1) == 0     # C % 8 != 0
    assert lib.group_norm_workspace_bytes(1, 2, 3, 4, 4096, 32, 1) == 0  # C > 2048
    ws = lib.group_norm_workspace_bytes(1, 2, 3, 4, 128, 32, 1)

    def call(x=0x100000, y=0x200000, w=0x300000, wb=ws, C=128, G=32, eps=1e-6):
        return lib.group_norm_silu(x, 1, 2, 3, 4, C, G, 1, eps, None, None, 1, y, w, wb, None)
    assert call(C=96, G=7) == vvc.ERR_INVALID_ARG
    assert call(eps=-1.0) == vvc.ERR_INVALID_ARG
    assert call(y=0x200008) == vvc.ERR_MISALIGNED
    assert call(wb=ws - 16) == vvc.ERR_WORKSPACE
    assert call(y=0x100000 + 256) == vvc.ERR_OVERLAP   # y over x
    assert call(w=0x200000 + 64) == vvc.ERR_OVERLAP    # workspace over y


def test_ndhwc_calls_plan_no_transpose():
    # every call of the benchmark workloads in NDHWC runs the convolution alone (plus the
    # split reduction, or the spatial gather of a narrow input): no layout staging launch
    import workloads as wl
    lib = vvc._lib()
    for w in ("wan", "ladder", "fused160", "t1"):
        for call in wl.all_workloads()[w].calls:
            p = vvc.Params()
            p.x, p.w_packed, p.y = 0x100000, 0x200000, 0x10000000
            p.layout = p.out_layout = vvc.NDHWC
            p.N, p.Cin, p.D, p.H, p.W = call.N, call.Cin, call.D, call.H, call.W
            p.Cout = call.Cout
            p.KT, p.KR, p.KS = call.kernel
            for i in range(3):
                p.stride[i] = call.stride[i]
                b, a, m = call.pads[i]
                p.pad[i].before, p.pad[i].after = b, a
                p.pad[i].mode = vvc.PAD_ZERO if m == wl.ZERO else vvc.PAD_REFLECT
            p.epi = call.epi
            p.bias = p.residual_bias = p.gamma = 0x300000
            p.residual = 0x400000
            info = _plan(p)
            expected = 1 + (info.k_splits > 1) + (info.im2col == 1)
            assert info.launches == expected, (call.name, info.launches, expected)
            assert (info.im2col != 0) == (call.Cin < 8), call.name


def _halo(p, halo):
    for i, (b, a, m) in enumerate(halo):
        p.out_halo[i].before, p.out_halo[i].after, p.out_halo[i].mode = b, a, m
    return p


def test_output_halo_validation():
    R, Z = vvc.PAD_REFLECT, vvc.PAD_ZERO
    ok = ((2, 0, Z), (1, 1, R), (1, 1, R))
    info = vvc.PlanInfo()
    assert vvc._lib().conv3d_plan(ctypes.byref(_halo(_params(), ok)), None,
                                  ctypes.byref(info)) == vvc.OK
    bad = [
        dict(halo=((1, 0, R), (1, 1, R), (1, 1, R))),      # the T halo is never written
        dict(halo=((0, 0, Z), (2, 1, R), (1, 1, R))),      # at most one pixel a side
        dict(halo=((0, 0, Z), (1, 1, 5), (1, 1, R))),      # unknown mode
        dict(halo=ok, out_layout=vvc.NCDHW),               # NDHWC only
        dict(halo=ok, Cout=36),                            # 16-byte channel rows
        dict(halo=ok, epi=vvc.EPI_L2NORM_SILU, gamma=0x300000),
        dict(halo=ok, epi=vvc.EPI_OUT_PAD_BR | vvc.EPI_RESIDUAL, residual=0x300000),
        dict(halo=ok, H=2, KR=3, pad_h=0),                 # reflection needs Ho >= 2
    ]
    for case in bad:
        halo = case.pop("halo")
        pad_h = case.pop("pad_h", None)
        p = _params(**case)
        if pad_h is not None:
            p.pad[1].before = p.pad[1].after = pad_h
        assert fwd(_halo(p, halo)) == vvc.ERR_INVALID_ARG, case


def test_output_halo_overlap_counts_the_whole_tensor():
    # y [1, 6, 14, 14, 32] with the halo: a workspace or value_out that starts inside
    # it must be rejected, although it would lie past an unpadded output
    R, Z = vvc.PAD_REFLECT, vvc.PAD_ZERO
    p = _halo(_params(epi=vvc.EPI_SAVE_VALUE), ((2, 0, Z), (1, 1, R), (1, 1, R)))
    plain_bytes = 1 * 4 * 12 * 12 * 32 * 2
    p.value_out = p.y + plain_bytes + 1024  # past the plain output, inside the haloed y
    ws = ctypes.c_size_t(0)
    assert vvc._lib().conv3d_workspace_bytes(ctypes.byref(p), ctypes.byref(ws)) == vvc.OK
    p.workspace, p.workspace_bytes = 0x40000000, ws.value
    assert fwd(p) == vvc.ERR_OVERLAP


def test_e4m3_validation_and_plan():
    lib = vvc._lib()
    assert lib.conv3d_packed_weight_bytes_e4m3(96, 96, 3, 3, 3) == 96 * 27 * 128
    assert lib.conv3d_packed_weight_bytes_e4m3(8, 130, 1, 3, 3) == 8 * 9 * 256
    assert lib.conv3d_packed_weight_bytes_e4m3(0, 16, 3, 3, 3) == 0
    f8 = dict(dtype=vvc.DTYPE_E4M3, fp8_scale=1.0)
    info = _plan(_params(**f8))
    assert info.kernel == 2 and info.paired == 0 and info.im2col == 0
    # the same stage walk as the bf16 plan over Cin / 2 channel pairs
    assert info.stages_per_tile == _plan(_params(Cin=8)).stages_per_tile
    p = _params(Cin=96, Cout=96, **f8)
    # one chunk of 48 pairs per (kt, kr) with the three W taps in one stage, never
    # paired (bf16 96 channels pair the last chunks: 18 -> 14 stages)
    assert _plan(p).stages_per_tile == 9 and _plan(p).paired == 0
    bad = [
        dict(dtype=2),                                       # unknown element type
        dict(fp8_scale=0.0),                                 # scale must be nonzero
        dict(fp8_scale=float("inf")),                        # and finite
        dict(fp8_scale=float("nan")),
        dict(layout=vvc.NCDHW),                              # e4m3 input is NDHWC
        dict(Cin=24),                                        # 16-byte channel rows
        dict(input_upsample=2, pad=None),                    # no fused upsample
    ]
    for case in bad:
        kw = dict(f8)
        kw.update({k: v for k, v in case.items() if k != "pad"})
        assert fwd(_params(**kw)) == vvc.ERR_INVALID_ARG, case
    # outside the e4m3 instances: pixel-major kernels and tiny Cout
    p = _params(**f8)
    assert fwd(p, vvc.Tuning(kernel=1)) == vvc.ERR_UNSUPPORTED
    assert fwd(p, vvc.Tuning(kernel=3)) == vvc.ERR_UNSUPPORTED
    assert fwd(_params(Cout=8, **f8)) == vvc.ERR_UNSUPPORTED
    # buffer spans count one byte per e4m3 element: x right below y is no overlap
    p = _params(x=0x10000000 - 16 * 4 * 12 * 12, **f8)
    rc = fwd(p, vvc.Tuning(k_splits=1))
    assert rc != vvc.ERR_OVERLAP
    p = _params(x=0x10000000 - 16 * 4 * 12 * 12 + 16, **f8)
    assert fwd(p, vvc.Tuning(k_splits=1)) == vvc.ERR_OVERLAP
    # the bf16 call ignores the scale
    assert _plan(_params(fp8_scale=0.0)).kernel in (1, 2)
