"""Kernel widths other than 3 through mcc1d_bwd_ex, against the oracle.

The page supports W = 3 only today ("当前W仅支持3" in its constraints); the
strided calls accept 1 <= W <= 8 with the same formulas (gradX sums W taps,
gradWeight has W rows). The oracle implements any W and is pinned for
W = 1..5 by the Jacobian and torch-autograd pins.
"""
import numpy as np
import pytest

import datagen
import oracle
from parity import GX_MAX_ULP, check_guards, gradw_ratio, guarded_full, max_ulp, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import causal_conv_backward_gb300 as m  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from causal_conv_backward_gb300 import build
    build.build()


def run_ex(inp, S, B, H, W, dt):
    gy, x, w = (to_device(inp[k], dt) for k in ("gy", "x", "w"))
    mask = None if inp["mask"] is None else torch.from_numpy(inp["mask"]).cuda()
    gx = guarded_full((S, B, H), gy.dtype, 0xFF)   # NaN patterns
    gw = guarded_full((W, H), gy.dtype, 0xFF)
    t = m.tensors(gy, x, w, mask, gx, gw)
    nb = m.mcc1d_bwd_ex_workspace_size(t, S, B, H, W, dt)
    ws = guarded_full((nb,), torch.uint8, 0xFF)
    m.mcc1d_bwd_ex(t, S, B, H, W, dt, ws, nb, torch.cuda.current_stream())
    assert m.mcc1d_bwd_device_status(ws, torch.cuda.current_stream()) == 0
    check_guards(gx, gw, ws, what="mcc1d_bwd_ex")
    return gx.view(torch.int16).cpu().numpy().view(np.uint16), gw.view(torch.int16).cpu().numpy().view(np.uint16)


CASES = []
for W in range(1, 9):
    for (S, B, H, dt) in [(1, 2, 384, "bf16"), (W + 1, 1, 1088, "fp16"), (77, 3, 448, "bf16"),
                          (1000, 2, 2048, "fp16"), (4096, 1, 384, "bf16")]:
        CASES.append((W, S, B, H, dt))


@pytest.mark.parametrize("W,S,B,H,dt", CASES, ids=[f"w{a}_s{b}_b{c}_h{d}_{e}" for a, b, c, d, e in CASES])
def test_width(W, S, B, H, dt):
    wl = datagen.Workload(f"w{W}", S, B, H, dt, W=W, mask=("bernoulli", 0.8))
    inp = datagen.generate(wl, seed=W * 100 + S)
    gx, gw = run_ex(inp, S, B, H, W, dt)
    ref = oracle.bwd(S, B, H, W, dt, inp["gy"], inp["x"], inp["w"], inp["mask"], want_exact=True)
    assert max_ulp(gx, ref["gx"]) <= GX_MAX_ULP
    assert gradw_ratio(gw, ref["gw_exact"], ref["gw_abs"], dt) <= 1.0


@pytest.mark.parametrize("W", [2, 4, 8])
def test_width_full_size_workload(W):
    """A full-size workload (4096 x 8 x 2048 bf16) at other widths."""
    wl = datagen.WORKLOADS["s4096_b8_h2048_bf16"].resized(W=W)
    inp = datagen.generate(wl, seed=W)
    gx, gw = run_ex(inp, wl.S, wl.B, wl.H, W, wl.dtype)
    ref = oracle.bwd(wl.S, wl.B, wl.H, W, wl.dtype, inp["gy"], inp["x"], inp["w"], inp["mask"],
                     want_exact=True)
    assert max_ulp(gx, ref["gx"]) <= GX_MAX_ULP
    assert gradw_ratio(gw, ref["gw_exact"], ref["gw_abs"], wl.dtype) <= 1.0


def test_width_three_matches_page_call():
    """W = 3 through the strided call equals mcc1d_bwd bit for bit."""
    wl = datagen.WORKLOADS["s524288_b1_h384_bf16"].resized(S=20000)
    inp = datagen.generate(wl, seed=1)
    gx, gw = run_ex(inp, wl.S, wl.B, wl.H, 3, wl.dtype)
    from parity import run_cuda
    gx2, gw2, st, _ = run_cuda(inp, wl.S, wl.B, wl.H, wl.dtype)
    assert st == 0 and np.array_equal(gx, gx2) and np.array_equal(gw, gw2)
