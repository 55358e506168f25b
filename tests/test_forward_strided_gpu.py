"""The forward on strided inputs (mcc1d_fwd_ex): every layout gives the same
bits as mcc1d_fwd on dense copies of the same values, within 1 ulp of the
oracle; x layouts that cannot stream in place are gathered through the
workspace first."""
import numpy as np
import pytest

import datagen
import oracle
from parity import GX_MAX_ULP, check_guards, guarded_full, max_ulp, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import causal_conv_backward_gb300 as m  # noqa: E402
from test_strided_gpu import make_view  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from causal_conv_backward_gb300 import build
    build.build()


def bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


CASES = []
for (S, B, H, dt, W) in [(777, 3, 1088, "bf16", 3), (1000, 1, 384, "fp16", 3), (130, 5, 2112, "fp16", 4),
                         (3000, 2, 640, "bf16", 1), (500, 4, 448, "bf16", 7)]:
    for lay in ("bsh", "hslice", "hslice_odd", "hstride2", "shb"):
        CASES.append((S, B, H, dt, W, lay))


@pytest.mark.parametrize("S,B,H,dt,W,layout", CASES,
                         ids=[f"s{a}_b{b}_h{c}_{d}_w{e}_{f}" for a, b, c, d, e, f in CASES])
def test_strided_forward_matches_dense(S, B, H, dt, W, layout):
    wl = datagen.Workload("fs", S, B, H, dt, W=W, mask=("bernoulli", 0.75))
    inp = datagen.generate(wl, seed=S + W)
    x, w = to_device(inp["x"], dt), to_device(inp["w"], dt)
    mask = torch.from_numpy(inp["mask"]).cuda()
    stream = torch.cuda.current_stream()
    y_dense = guarded_full(x.shape, x.dtype, 0xFF)
    m.mcc1d_fwd(x, w, mask, y_dense, stream, S, B, H, W, dt)
    # strided x, [H,W]-memory weight, [S,B]-memory mask
    xv = make_view(x, layout)
    wv = w.t().contiguous().t()
    mv = mask.t().contiguous().t()
    y = guarded_full((S, B, H), x.dtype, 0xFF)
    t = m.fwd_tensors(xv, wv, mv, y)
    nb = m.mcc1d_fwd_ex_workspace_size(t, S, B, H, W, dt)
    ws = guarded_full((max(nb, 16),), torch.uint8, 0xFF)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    m.mcc1d_fwd_ex(t, S, B, H, W, dt, ws, nb, stream, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    check_guards(y_dense, y, ws, what="mcc1d_fwd / mcc1d_fwd_ex")
    assert np.array_equal(bits(y), bits(y_dense))
    ref = oracle.fwd_bits(S, B, H, W, dt, inp["x"], inp["w"], inp["mask"])
    assert max_ulp(bits(y), ref) <= GX_MAX_ULP


def test_forward_convenience_routes_strided_views():
    """forward() takes a strided view through mcc1d_fwd_ex."""
    S, B, H, dt = 300, 3, 1024, "bf16"
    wl = datagen.Workload("fc", S, B, H, dt, W=4, mask=("bernoulli", 0.9))
    inp = datagen.generate(wl, seed=9)
    x, w = to_device(inp["x"], dt), to_device(inp["w"], dt)
    mask = torch.from_numpy(inp["mask"]).cuda()
    y1 = m.forward(x, w, mask)
    y2 = m.forward(make_view(x, "hstride2"), w, mask)
    torch.cuda.synchronize()
    assert np.array_equal(bits(y1), bits(y2))
