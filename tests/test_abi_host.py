"""Host-side checks of the C ABI (no GPU needed).

The library must load, export every entry point include/tp.h declares, and
reject bad arguments with the documented status before touching the GPU:
every call here fails validation (or has P == 0), so nothing is launched and
the fake pointers are never dereferenced.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tp.h")

TP_OK, TP_ERR_NULL, TP_ERR_SHAPE, TP_ERR_ALIGN, TP_ERR_UNSUPPORTED = 0, 1, 2, 3, 4


@pytest.fixture(scope="module")
def tp():
    from backprojection_tp_project_gather_b300 import build
    build.build()
    import backprojection_tp_project_gather_b300 as m
    return m


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tp_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_operator_set():
    syms = declared_symbols()
    for name in ("tp_project_3d_2d", "tp_project_3d_2d_backward", "tp_backproject_2d_3d",
                 "tp_project_2d_2d", "tp_project_2d_2d_backward", "tp_project_3d_2d_save",
                 "tp_project_3d_2d_backward_saved", "tp_backproject_2d_3d_backward",
                 "tp_backproject_backward_scratch_bytes", "tp_project_3d_2d_l2", "tp_last_error",
                 "tp_version"):
        assert name in syms


def test_library_exports_every_declared_symbol(tp):
    lib = tp.lib()
    for name in declared_symbols():
        assert hasattr(lib, name), name
    assert re.fullmatch(r"\d+\.\d+\.\d+", tp.tp_version())


def test_bounds_checking_build_exports_the_same_symbols(tp):
    """libtp_b300_debug.so (-DTP_DEBUG_BOUNDS) is a drop-in for the normal
    library; the normal build reports no failed index checks."""
    from backprojection_tp_project_gather_b300 import build
    dbg = ctypes.CDLL(build.build(debug=True))
    for name in declared_symbols():
        assert hasattr(dbg, name), name
    assert tp.tp_debug_bounds_word() == 0
    assert tp.tp_debug_bounds_word(reset=True) == 0
    # The self-test exists only in the debug build; nothing is launched here.
    assert tp._fn("tp_debug_bounds_selftest")(3, None) == TP_ERR_UNSUPPORTED


# Fake, well-aligned device addresses: validation rejects each call first.
A = 0x10000
MIS = 0x10004      # 4-byte aligned, not 8-byte aligned (bad for complex64)


def opts(tp, interp=1, s=1.0, r=-1.0, flags=0):
    return tp.TPOptions(interp, s, r, flags)


WS = 0x20000       # fake workspace address
WSB = 1 << 30      # claimed workspace size


def proj3(tp, **kw):
    a = dict(vol=A, Bv=1, Nv=16, rot=A, Bp=1, P=4, shift=None, Bs=1, N=16, o=opts(tp), out=A,
             ws=WS, wsb=WSB)
    a.update(kw)
    return tp._fn("tp_project_3d_2d")(a["vol"], a["Bv"], a["Nv"], a["rot"], a["Bp"], a["P"],
                                     a["shift"], a["Bs"], a["N"], a["o"], a["out"], a["ws"],
                                     a["wsb"], None)


def test_forward_validation(tp):
    assert proj3(tp, vol=None) == TP_ERR_NULL
    assert proj3(tp, out=None) == TP_ERR_NULL
    assert proj3(tp, rot=None) == TP_ERR_NULL
    assert proj3(tp, N=15) == TP_ERR_SHAPE
    assert proj3(tp, Nv=17) == TP_ERR_SHAPE
    assert proj3(tp, Nv=0) == TP_ERR_SHAPE
    assert proj3(tp, P=-1) == TP_ERR_SHAPE
    assert proj3(tp, Bv=2, Bp=3) == TP_ERR_SHAPE
    assert proj3(tp, Bv=2, shift=A, Bs=3) == TP_ERR_SHAPE
    assert proj3(tp, Nv=8192) == TP_ERR_SHAPE
    assert proj3(tp, vol=MIS) == TP_ERR_ALIGN
    assert proj3(tp, out=MIS) == TP_ERR_ALIGN
    assert proj3(tp, rot=A + 2) == TP_ERR_ALIGN
    assert proj3(tp, o=opts(tp, interp=7)) == TP_ERR_UNSUPPORTED
    assert proj3(tp, o=opts(tp, s=0.0)) == TP_ERR_UNSUPPORTED
    assert proj3(tp, o=opts(tp, s=float("nan"))) == TP_ERR_UNSUPPORTED
    assert proj3(tp, o=opts(tp, r=float("inf"))) == TP_ERR_UNSUPPORTED
    assert proj3(tp, o=opts(tp, flags=1)) == TP_ERR_UNSUPPORTED
    assert "flags" in tp.tp_last_error()
    assert proj3(tp, ws=None) == TP_ERR_NULL
    assert proj3(tp, ws=WS + 4) == TP_ERR_ALIGN
    assert proj3(tp, wsb=16) == TP_ERR_SHAPE
    assert "workspace" in tp.tp_last_error()
    # An empty problem succeeds without launching anything.
    assert proj3(tp, P=0) == TP_OK
    assert tp.tp_last_error() == ""


def test_backward_validation(tp):
    lib = tp.lib()
    o = opts(tp)

    def bwd(go=A, vol=A, shift=None, gv=A, gr=A, gs=None, P=4):
        return tp._fn("tp_project_3d_2d_backward")(go, vol, 1, 16, A, 1, P, shift, 1, 16, o, gv, gr, gs,
                                             WS, WSB, None)
    assert bwd(go=None) == TP_ERR_NULL
    assert bwd(vol=None) == TP_ERR_NULL                 # needed for grad_rot
    assert bwd(gs=A) == TP_ERR_NULL                     # grad_shift without shift
    assert bwd(gv=MIS) == TP_ERR_ALIGN
    assert bwd(P=0) == TP_OK
    assert tp._fn("tp_project_2d_2d_backward")(A, A, 1, 15, A, 1, 4, None, 1, 16, o, A, A, None,
                                         None) == TP_ERR_SHAPE


def test_backprojection_validation(tp):
    lib = tp.lib()
    o = opts(tp)

    def bp(proj=A, B=2, Bp=1, Bv=1, data=A, wv=A, P=4, weights=None):
        return tp._fn("tp_backproject_2d_3d")(proj, weights, B, P, 16, A, Bp, None, 1, Bv, 16, o, data,
                                        wv, WS, WSB, None)
    assert bp(proj=None) == TP_ERR_NULL
    assert bp(data=None) == TP_ERR_NULL
    assert bp(Bv=3) == TP_ERR_SHAPE                     # Bv must be 1 or B
    assert bp(Bp=4) == TP_ERR_SHAPE                     # rotations batch larger than B
    assert bp(data=MIS) == TP_ERR_ALIGN
    assert bp(weights=A + 2) == TP_ERR_ALIGN
    assert bp(P=0) == TP_OK
    assert bp(wv=None, P=0) == TP_OK


def test_saved_forward_validation(tp):
    def save(dout=A, P=4, vol=A, ws=WS):
        return tp._fn("tp_project_3d_2d_save")(vol, 1, 16, A, 1, P, None, 1, 16, opts(tp), A, dout,
                                               ws, WSB, None)
    assert save(dout=None) == TP_ERR_NULL
    assert "dout" in tp.tp_last_error()
    assert save(dout=MIS) == TP_ERR_ALIGN
    assert save(vol=None) == TP_ERR_NULL
    assert save(ws=None) == TP_ERR_NULL
    assert save(P=0, dout=None) == TP_OK


def test_l2_forward_validation(tp):
    def l2(target=A, out=A, gout=A, gr=A, gs=None, shift=None, P=4, vol=A, ws=WS):
        return tp._fn("tp_project_3d_2d_l2")(vol, 1, 16, A, 1, P, shift, 1, 16, opts(tp), target, out,
                                             gout, gr, gs, ws, WSB, None)
    assert l2(target=None) == TP_ERR_NULL
    assert "target" in tp.tp_last_error()
    assert l2(gout=None) == TP_ERR_NULL
    assert l2(gs=A) == TP_ERR_NULL                       # grad_shift without shift
    assert l2(gout=MIS) == TP_ERR_ALIGN
    assert l2(target=MIS) == TP_ERR_ALIGN
    assert l2(gr=A + 2) == TP_ERR_ALIGN
    assert l2(ws=None) == TP_ERR_NULL
    assert l2(P=0, target=None, out=None, gout=None) == TP_OK


def test_saved_backward_validation(tp):
    def bs(go=A, out=A, dout=A, B=2, P=4, N=16, Bp=1, Bs=1, o=None, gr=A, gs=None):
        return tp._fn("tp_project_3d_2d_backward_saved")(go, out, dout, B, P, N, Bp, Bs,
                                                         o or opts(tp), gr, gs, None)
    assert bs(N=15) == TP_ERR_SHAPE
    assert bs(N=8192) == TP_ERR_SHAPE
    assert bs(B=0) == TP_ERR_SHAPE
    assert bs(Bp=3) == TP_ERR_SHAPE                     # rotations batch must be 1 or B
    assert bs(Bs=3) == TP_ERR_SHAPE
    assert bs(P=-1) == TP_ERR_SHAPE
    assert bs(o=opts(tp, flags=2)) == TP_ERR_UNSUPPORTED
    assert bs(o=opts(tp, s=-1.0)) == TP_ERR_UNSUPPORTED
    assert bs(go=None) == TP_ERR_NULL
    assert bs(dout=None) == TP_ERR_NULL
    assert bs(out=MIS) == TP_ERR_ALIGN
    assert bs(gr=A + 2) == TP_ERR_ALIGN
    assert bs(gr=None, gs=None, go=None) == TP_OK       # nothing requested: no work, no checks
    assert bs(P=0, go=None) == TP_OK


def test_backprojection_backward_validation(tp):
    SC = 0x40000

    def bb(G=A, GW=None, proj=A, B=2, P=4, Bv=1, Bp=1, shift=None, gp=A, gw=None, gr=A, gs=None,
           sc=SC, scb=WSB, ws=WS):
        return tp._fn("tp_backproject_2d_3d_backward")(G, GW, proj, None, B, P, 16, A, Bp, shift, 1,
                                                       Bv, 16, opts(tp), gp, gw, gr, gs, sc, scb,
                                                       ws, WSB, None)
    assert bb(G=None) == TP_ERR_NULL                    # grad_proj needs the data gradient
    assert bb(gw=A) == TP_ERR_NULL                      # grad_weights needs grad_weight_vol
    assert bb(proj=None) == TP_ERR_NULL                 # grad_rot needs the images
    assert bb(gs=A) == TP_ERR_NULL                      # grad_shift without a shift
    assert bb(sc=None) == TP_ERR_NULL
    assert "scratch" in tp.tp_last_error()
    assert bb(sc=SC + 8) == TP_ERR_ALIGN
    assert bb(scb=64) == TP_ERR_SHAPE
    assert bb(Bv=3) == TP_ERR_SHAPE
    assert bb(gp=MIS) == TP_ERR_ALIGN
    assert bb(gp=None, gr=None) == TP_OK                # nothing requested
    assert bb(P=0, G=None) == TP_OK
    small = tp.tp_backproject_backward_scratch_bytes(1, 2, 4, 16, 16, False)
    assert 0 < small < tp.tp_backproject_backward_scratch_bytes(1, 2, 4, 16, 16, True)
    assert tp.tp_backproject_backward_scratch_bytes(1, 2, 4, 15, 16, True) == 0


def test_workspace_size_query(tp):
    small = tp.tp_workspace_bytes(1, 1, 8, 32, "cubic")
    big = tp.tp_workspace_bytes(1, 1, 512, 256, "cubic")
    assert 0 < small < big
    assert tp.tp_workspace_bytes(1, 1, 8, 31, "cubic") == 0      # odd box
    assert tp.tp_workspace_bytes(2, 1, 8, 32, "cubic") == 0      # Bv > B
    assert tp.tp_workspace_bytes(1, 1, 8, 32, "cubic", N=31) == 0   # odd image box
    # The cubic scatter's sample lists: 4 bytes per output pixel.
    grow = tp.tp_workspace_bytes(1, 1, 8, 32, "cubic", N=64) - small
    assert grow >= 4 * 8 * (64 * 33 - 32 * 17)
    lin = tp.tp_workspace_bytes(1, 1, 8, 32, "linear")
    assert 0 < lin < tp.tp_workspace_bytes(1, 1, 8, 32, "linear", N=64)


def test_binding_rejects_cpu_tensors(tp):
    import torch
    vol = torch.zeros((1, 8, 8, 5), dtype=torch.complex64)
    rot = torch.eye(3).reshape(1, 1, 3, 3)
    with pytest.raises(ValueError, match="CUDA"):
        tp.tp_project_3d_2d(vol, rot)


TP_FLAG_HERMITIAN_X0 = 1


def test_hermitian_flag_acceptance(tp):
    """TP_FLAG_HERMITIAN_X0 is accepted where a spectrum is accumulated and
    refused by the forward calls, the saved-path backward and the
    backprojection's backward; other bits are refused everywhere.  Every
    call here stops at validation or has P == 0."""
    assert tp.FLAG_HERMITIAN_X0 == TP_FLAG_HERMITIAN_X0
    text = open(HEADER).read()
    assert re.search(r"#define\s+TP_FLAG_HERMITIAN_X0\s+1u", text)
    h = opts(tp, flags=TP_FLAG_HERMITIAN_X0)
    assert proj3(tp, o=h) == TP_ERR_UNSUPPORTED
    assert "TP_FLAG_HERMITIAN_X0" in tp.tp_last_error()
    assert tp._fn("tp_project_2d_2d")(A, 1, 16, A, 1, 4, None, 1, 16, h, A, None) == TP_ERR_UNSUPPORTED
    # accepted: the 3D and 2D backward (P == 0: nothing launched) and the backprojection
    assert tp._fn("tp_project_3d_2d_backward")(A, A, 1, 16, A, 1, 0, None, 1, 16, h, A, A, None,
                                               WS, WSB, None) == TP_OK
    assert tp._fn("tp_project_2d_2d_backward")(A, A, 1, 16, A, 1, 0, None, 1, 16, h, A, A, None,
                                               None) == TP_OK
    assert tp._fn("tp_backproject_2d_3d")(A, None, 1, 0, 16, A, 1, None, 1, 1, 16, h, A, A, WS,
                                          WSB, None) == TP_OK
    # a validation error still wins over the accepted flag
    assert tp._fn("tp_project_3d_2d_backward")(None, A, 1, 16, A, 1, 4, None, 1, 16, h, A, A,
                                               None, WS, WSB, None) == TP_ERR_NULL
    # refused
    bad = opts(tp, flags=TP_FLAG_HERMITIAN_X0 | 2)
    assert tp._fn("tp_project_3d_2d_backward")(A, A, 1, 16, A, 1, 0, None, 1, 16, bad, A, A, None,
                                               WS, WSB, None) == TP_ERR_UNSUPPORTED
    assert tp._fn("tp_project_3d_2d_backward_saved")(A, A, A, 1, 4, 16, 1, 1, h, A, None,
                                                     None) == TP_ERR_UNSUPPORTED
    assert tp._fn("tp_backproject_2d_3d_backward")(A, None, A, None, 2, 4, 16, A, 1, None, 1, 1,
                                                   16, h, A, None, A, None, 0x40000, WSB, WS,
                                                   WSB, None) == TP_ERR_UNSUPPORTED
    assert "tp_hermitian_x0" in tp.tp_last_error()


def test_hermitian_x0_validation(tp):
    f = tp._fn("tp_hermitian_x0")
    assert f(A, None, 1, 16, 4, None) == TP_ERR_UNSUPPORTED     # dim
    assert f(A, None, 1, 15, 3, None) == TP_ERR_SHAPE           # odd box
    assert f(A, None, 1, 8192, 3, None) == TP_ERR_SHAPE
    assert f(A, None, -1, 16, 3, None) == TP_ERR_SHAPE
    assert f(None, None, 1, 16, 3, None) == TP_ERR_NULL
    assert f(MIS, None, 1, 16, 3, None) == TP_ERR_ALIGN
    assert f(None, A + 2, 1, 16, 2, None) == TP_ERR_ALIGN
    assert f(A, A, 0, 16, 3, None) == TP_OK                     # B == 0: nothing to do


def test_package_imports_without_the_library_and_calls_fail_loudly(tmp_path):
    """On a fresh checkout the library file does not exist yet: the package
    (and its build module) must import, so that the build can run, while
    every call into the library raises ImportError."""
    import shutil
    import subprocess
    import sys
    src = os.path.join(ROOT, "backprojection_tp_project_gather_b300")
    dst = tmp_path / "backprojection_tp_project_gather_b300"
    dst.mkdir()
    for name in os.listdir(src):
        if name.endswith(".py"):
            shutil.copy(os.path.join(src, name), dst / name)
    code = ("import backprojection_tp_project_gather_b300 as tp\n"
            "import backprojection_tp_project_gather_b300.build as b\n"
            "assert b.LIB.endswith('libtp_b300.so')\n"
            "try:\n"
            "    tp.tp_version()\n"
            "except ImportError as e:\n"
            "    assert 'is missing' in str(e)\n"
            "    print('loud')\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=tmp_path, capture_output=True, text=True,
                       env=dict(os.environ, PYTHONPATH=str(tmp_path)), timeout=300)
    assert r.returncode == 0 and "loud" in r.stdout, r.stdout + r.stderr
