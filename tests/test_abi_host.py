"""The C-ABI library on the host: it loads, exports every declared symbol,
and rejects bad arguments with the page's status codes before touching any
device (no GPU needed; only failing calls are made)."""
import ctypes
import os
import re

import pytest

import causal_conv_backward_gb300 as m
from causal_conv_backward_gb300 import build as cbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
NULLPTR, INVALID, SHAPE, WORKSPACE = 161001, 161002, 561002, 561003


@pytest.fixture(scope="module")
def lib():
    cbuild.build()
    return m.load()


def declared_functions():
    names = []
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            with open(os.path.join(ROOT, "include", f)) as fh:
                src = fh.read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(mcc1d_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert "mcc1d_bwd" in names and "mcc1d_bwd_workspace_size" in names
    for n in names:
        assert hasattr(lib, n), n


def ws(S, B, H, W=3, dtype=0, has_mask=1, out=True):
    v = ctypes.c_uint64(12345)
    st = m.load().mcc1d_bwd_workspace_size(S, B, H, W, dtype, has_mask, ctypes.byref(v) if out else None)
    return st, v.value


def test_workspace_size_valid_shapes(lib):
    for (S, B, H) in [(1, 1, 384), (64, 2, 384), (4096, 8, 2048), (524288, 1, 384),
                      (16384, 32, 4096), (8192, 4, 24576), (16384, 32, 24576), (1, 32, 24576)]:
        for dt in (0, 1):
            st, n = ws(S, B, H, dtype=dt)
            assert st == 0 and n > 0
            assert ws(S, B, H, dtype=dt, has_mask=0) == (0, n)  # the mask does not change it
            assert ws(S, B, H, dtype=dt) == (0, n)              # deterministic


@pytest.mark.parametrize("S,B,H,W,dt,code", [
    (1, 1, 384, 3, 2, INVALID), (1, 1, 384, 3, -1, INVALID),
    (0, 1, 384, 3, 0, SHAPE), (1, 0, 384, 3, 0, SHAPE), (1, 33, 384, 3, 0, SHAPE),
    (524289, 1, 384, 3, 0, SHAPE), (16385, 32, 384, 3, 0, SHAPE), (1, 1, 320, 3, 0, SHAPE),
    (1, 1, 392, 3, 0, SHAPE), (1, 1, 24640, 3, 0, SHAPE), (1, 1, 384, 2, 0, SHAPE),
    (1, 1, 384, 4, 0, SHAPE), (-5, 1, 384, 3, 0, SHAPE), (1 << 40, 1, 384, 3, 0, SHAPE),
])
def test_workspace_size_rejects(lib, S, B, H, W, dt, code):
    st, v = ws(S, B, H, W, dt)
    assert st == code and v == 12345


def test_workspace_size_null_out(lib):
    assert ws(64, 2, 384, out=False)[0] == NULLPTR


def call(gy=0x1000, x=0x2000, w=0x3000, mask=None, gx=0x4000, gw=0x5000, wsp=0x6000,
         S=64, B=2, H=384, W=3, dt=0, wsb=None):
    if wsb is None:
        wsb = ws(S, B, H)[1] if ws(S, B, H)[0] == 0 else 0
    return m.load().mcc1d_bwd(gy, x, w, mask, gx, gw, wsp, None, S, B, H, W, dt, wsb)


@pytest.mark.parametrize("which", ["gy", "x", "w", "gx", "gw", "wsp"])
def test_bwd_null_pointer(lib, which):
    assert call(**{which: None}) == NULLPTR


@pytest.mark.parametrize("which", ["gy", "x", "w", "gx", "gw", "wsp"])
def test_bwd_misaligned_pointer(lib, which):
    base = {"gy": 0x1000, "x": 0x2000, "w": 0x3000, "gx": 0x4000, "gw": 0x5000, "wsp": 0x6000}
    assert call(**{which: base[which] + 2}) == INVALID


def test_bwd_bad_dtype_and_shape(lib):
    assert call(dt=7, wsb=1 << 30) == INVALID
    assert call(B=33, wsb=1 << 30) == SHAPE
    assert call(H=400, wsb=1 << 30) == SHAPE
    assert call(W=2, wsb=1 << 30) == SHAPE


def test_bwd_workspace_too_small(lib):
    need = ws(4096, 8, 2048)[1]
    assert call(S=4096, B=8, H=2048, wsb=need - 1) == WORKSPACE


def test_status_strings(lib):
    for code in (0, NULLPTR, INVALID, SHAPE, WORKSPACE, 561100, 561101, 561102):
        s = m.mcc1d_status_string(code)
        assert s.startswith("MCC1D_")
    assert m.mcc1d_status_string(42) == "unknown mcc1d status"
    assert m.mcc1d_version() >= 100


def test_sm_count_check_refuses_a_smaller_device(lib):
    """The plans cut every shape into 152 x (CTAs per SM) persistent CTAs; a
    device with fewer SMs would run part of each grid as a second wave, so
    every launching call refuses it with MCC1D_ERR_DEVICE. The rule, applied
    to fake counts (no device needed):"""
    assert m.PLAN_SMS == 152
    for n in (1, 76, 148, 151):
        assert m.mcc1d_check_sm_count(n) == 561102, n
        assert "fewer SMs" in m.mcc1d_status_string(m.mcc1d_check_sm_count(n))
    for n in (152, 160, 264):
        assert m.mcc1d_check_sm_count(n) == 0, n
    assert lib.mcc1d_device_sm_count(None) == NULLPTR


# ------------------------------------------------------------- strided calls
def desc(gy=0x10000, x=0x20000, w=0x30000, mask=None, gx=0x40000, gw=0x50000,
         gys=None, xs=None, ws_=None, ms=None, S=64, B=2, H=384):
    t = m.Mcc1dTensors()
    t.gradY, t.x, t.weight, t.mask, t.gradX, t.gradWeight = gy, x, w, mask, gx, gw
    t.gradY_strides[:] = gys or [B * H, H, 1]
    t.x_strides[:] = xs or [B * H, H, 1]
    t.weight_strides[:] = ws_ or [H, 1]
    t.mask_strides[:] = ms or [S, 1]
    return t


def ex_size(t, S=64, B=2, H=384, W=3, dt=0):
    v = ctypes.c_uint64(7)
    st = m.load().mcc1d_bwd_ex_workspace_size(ctypes.byref(t), S, B, H, W, dt, ctypes.byref(v))
    return st, v.value


def test_ex_workspace_dense_needs_no_copies(lib):
    st, n = ex_size(desc())
    base = ws(64, 2, 384)[1]
    assert st == 0 and base <= n < base + 256


def test_ex_workspace_counts_gathered_inputs(lib):
    S, B, H = 64, 2, 384
    E2 = S * B * H * 2
    base = ex_size(desc())[1]
    # a [B,S,H] buffer seen as [S,B,H] streams in place
    assert ex_size(desc(gys=[H, S * H, 1], xs=[H, S * H, 1]))[1] == base
    # H stride 2, or a base pointer off a 16-byte boundary, is gathered first
    assert ex_size(desc(gys=[2 * B * H, 2 * H, 2]))[1] == base + E2
    assert ex_size(desc(x=0x20002))[1] == base + E2
    assert ex_size(desc(gys=[B * H, H, 2], x=0x20002))[1] == base + 2 * E2
    # odd row strides break 16-byte row alignment
    assert ex_size(desc(xs=[B * H + 1, H, 1]))[1] == base + E2
    # weight and mask strides never cost workspace
    assert ex_size(desc(ws_=[1, 3], mask=0x60001, ms=[1, 2]))[1] == base


def test_ex_rejects(lib):
    assert m.load().mcc1d_bwd_ex_workspace_size(None, 64, 2, 384, 3, 0, ctypes.byref(ctypes.c_uint64())) == NULLPTR
    assert ex_size(desc(gy=None))[0] == NULLPTR
    assert ex_size(desc(gys=[-1, 384, 1]))[0] == INVALID
    assert ex_size(desc(ws_=[384, -1]))[0] == INVALID
    assert ex_size(desc(mask=0x60000, ms=[-64, 1]))[0] == INVALID
    assert ex_size(desc(gy=0x10001))[0] == INVALID        # not 2-byte aligned
    assert ex_size(desc(gx=0x40008))[0] == INVALID        # outputs stay 16-byte aligned
    assert ex_size(desc(), B=33)[0] == SHAPE
    assert ex_size(desc(), dt=3)[0] == INVALID
    t = desc()
    need = ex_size(t)[1]
    call = m.load().mcc1d_bwd_ex
    assert call(ctypes.byref(t), 64, 2, 384, 3, 0, None, need, None) == NULLPTR
    assert call(ctypes.byref(t), 64, 2, 384, 3, 0, 0x70008, need, None) == INVALID
    assert call(ctypes.byref(t), 64, 2, 384, 3, 0, 0x70000, need - 1, None) == WORKSPACE


def test_fwd_rejects_before_any_launch(lib):
    f = m.load().mcc1d_fwd
    ok = dict(x=0x1000, w=0x2000, y=0x3000)

    def call(S=64, B=2, H=384, W=3, dt=0, **kw):
        a = {**ok, **kw}
        return f(a["x"], a["w"], None, a["y"], None, S, B, H, W, dt, None)

    assert call(x=None) == NULLPTR and call(y=None) == NULLPTR and call(w=None) == NULLPTR
    assert call(x=0x1008) == INVALID and call(y=0x3002) == INVALID
    assert call(dt=2) == INVALID
    assert call(B=0) == SHAPE and call(H=4000) == SHAPE and call(W=0) == SHAPE and call(W=9) == SHAPE


def test_ex_accepts_widths_one_to_eight(lib):
    """The strided calls take any kernel width 1..8 (the page's calls keep W = 3)."""
    sizes = []
    for W in range(1, 9):
        t = desc(ws_=[384, 1])
        st, n = ex_size(t, W=W)
        assert st == 0, W
        sizes.append(n)
    assert sizes == sorted(sizes)  # W partial rows per slot
    assert ex_size(desc(), W=0)[0] == SHAPE
    assert ex_size(desc(), W=9)[0] == SHAPE
    assert ws(64, 2, 384, W=4)[0] == SHAPE   # page call: W must be 3


# ------------------------------------------------------- strided forward calls
def fdesc(x=0x20000, w=0x30000, mask=None, y=0x40000, xs=None, ws_=None, ms=None, S=64, B=2, H=384):
    t = m.Mcc1dFwdTensors()
    t.x, t.weight, t.mask, t.y = x, w, mask, y
    t.x_strides[:] = xs or [B * H, H, 1]
    t.weight_strides[:] = ws_ or [H, 1]
    t.mask_strides[:] = ms or [S, 1]
    return t


def fex_size(t, S=64, B=2, H=384, W=3, dt=0):
    v = ctypes.c_uint64(7)
    st = m.load().mcc1d_fwd_ex_workspace_size(ctypes.byref(t), S, B, H, W, dt, ctypes.byref(v))
    return st, v.value


def test_fwd_ex_workspace_sizes(lib):
    S, B, H = 64, 2, 384
    assert fex_size(fdesc()) == (0, 0)                                   # dense: streamed in place
    assert fex_size(fdesc(xs=[H, S * H, 1])) == (0, 0)                   # [B,S,H] memory: in place
    n = S * B * H * 2
    assert fex_size(fdesc(xs=[B * 2 * H, 2 * H, 2])) == (0, (n + 255) // 256 * 256)   # gathered
    assert fex_size(fdesc(x=0x20002)) == (0, (n + 255) // 256 * 256)    # rows off 16 B: gathered
    for W in range(1, 9):
        assert fex_size(fdesc(ws_=[H, 1]), W=W)[0] == 0


def test_fwd_ex_rejects_before_any_launch(lib):
    assert fex_size(fdesc(x=None))[0] == NULLPTR
    assert fex_size(fdesc(y=None))[0] == NULLPTR
    assert fex_size(fdesc(w=None))[0] == NULLPTR
    assert fex_size(fdesc(xs=[-768, 384, 1]))[0] == INVALID
    assert fex_size(fdesc(ws_=[384, -1]))[0] == INVALID
    assert fex_size(fdesc(mask=0x50000, ms=[-64, 1]))[0] == INVALID
    assert fex_size(fdesc(x=0x20001))[0] == INVALID                     # not 2-byte aligned
    assert fex_size(fdesc(y=0x40008))[0] == INVALID                     # output not 16-byte aligned
    assert fex_size(fdesc(), W=9)[0] == SHAPE and fex_size(fdesc(), W=0)[0] == SHAPE
    assert fex_size(fdesc(), dt=2)[0] == INVALID
    v = ctypes.c_uint64(0)
    assert m.load().mcc1d_fwd_ex_workspace_size(None, 64, 2, 384, 3, 0, ctypes.byref(v)) == NULLPTR
    assert m.load().mcc1d_fwd_ex_workspace_size(ctypes.byref(fdesc()), 64, 2, 384, 3, 0, None) == NULLPTR
    # a gathered x needs the workspace: missing or small is refused before any device work
    t = fdesc(xs=[2 * 2 * 384, 2 * 384, 2])
    f = m.load().mcc1d_fwd_ex
    assert f(ctypes.byref(t), 64, 2, 384, 3, 0, None, 0, None, None) == NULLPTR
    assert f(ctypes.byref(t), 64, 2, 384, 3, 0, 0x60000, 1024, None, None) == WORKSPACE
    assert f(ctypes.byref(t), 64, 2, 384, 3, 0, 0x60008, 1 << 20, None, None) == INVALID
