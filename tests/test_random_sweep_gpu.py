"""A seeded random sweep of shapes, widths, masks and layouts against the oracle.

Each case draws, from a fixed seed: the 16-bit type; the kernel width (3 half
of the time, else 1..8); H (a multiple of 64 in 384..24576, log-uniform); B
(1..32) and S with B*S <= 524288 (the page's shape envelope) and at most ~8M
elements so the oracle stays quick, three cases in ten in a long-sequence
regime (B <= 2, H <= 1024, S of thousands); a mask law (none, Bernoulli, padding
prefix, zero spans, all zeros); and the layout of gradY/x (dense, [B,S,H]
memory, an H-slice of a wider buffer, every other element along H), of the
weight ([H,W] memory) and of the mask ([S,B] memory). W = 3 on dense tensors
goes through mcc1d_bwd, everything else through mcc1d_bwd_ex. The plan's
edge cases (H-block splits, CTA ranges that end mid-sequence or mid-batch,
ragged stages, gathered inputs) are hit by chance many times over. Each case
runs twice with differently filled workspaces and must give the same bits.
"""
import numpy as np
import pytest

import datagen
from parity import GX_MAX_ULP, check_guards, gradw_ratio, guarded_full, max_ulp, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import causal_conv_backward_gb300 as m  # noqa: E402
import oracle  # noqa: E402

N_CASES = 160
MAX_ELEMENTS = 8 << 20


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from causal_conv_backward_gb300 import build
    build.build()


def draw_case(n):
    rng = np.random.default_rng(1000 + n)
    dt = ("bf16", "fp16")[rng.integers(2)]
    W = 3 if rng.random() < 0.5 else int(rng.integers(1, 9))
    if rng.random() < 0.3:
        # long sequences: few batches, narrow H, S in the thousands
        H = 64 * int(rng.integers(6, 17))
        B = int(rng.integers(1, 3))
        s_max = max(1, min(524288 // B, MAX_ELEMENTS // (B * H)))
        S = int(np.exp(rng.uniform(np.log(1000), np.log(s_max))))
    else:
        H = 64 * int(np.exp(rng.uniform(np.log(6), np.log(384))))
        H = min(max(H, 384), 24576)
        B = min(32, int(np.exp(rng.uniform(0, np.log(33)))))
        s_max = max(1, min(524288 // B, MAX_ELEMENTS // (B * H)))
        S = int(np.exp(rng.uniform(0, np.log(s_max)))) if s_max > 1 else 1
    S = max(1, min(S, s_max))
    laws = [("none",), ("bernoulli", float(rng.uniform(0.3, 1.0))), ("prefix",),
            ("spans", 0.2, 8, max(9, S // 4)), ("zeros",)]
    mask = laws[int(rng.choice(5, p=[0.2, 0.35, 0.2, 0.2, 0.05]))]
    layout = ("sbh", "bsh", "hslice", "hstride2")[int(rng.choice(4, p=[0.4, 0.25, 0.2, 0.15]))]
    w_t = bool(rng.random() < 0.25)
    m_t = bool(rng.random() < 0.25) and mask[0] != "none"
    return dict(dt=dt, W=W, S=S, B=B, H=H, mask=mask, layout=layout, w_t=w_t, m_t=m_t)


def view3(dense, layout):
    S, B, H = dense.shape
    if layout == "sbh":
        return dense
    if layout == "bsh":
        return dense.transpose(0, 1).contiguous().transpose(0, 1)
    if layout == "hslice":
        buf = torch.zeros((S, B, H + 64), dtype=dense.dtype, device=dense.device)
        buf[:, :, 32:32 + H] = dense
        return buf[:, :, 32:32 + H]
    buf = torch.zeros((S, B, 2 * H), dtype=dense.dtype, device=dense.device)
    buf[:, :, ::2] = dense
    return buf[:, :, ::2]


CASES = [draw_case(n) for n in range(N_CASES)]


def case_id(c):
    return (f"s{c['S']}_b{c['B']}_h{c['H']}_w{c['W']}_{c['dt']}_{c['mask'][0]}_{c['layout']}"
            + ("_wT" if c["w_t"] else "") + ("_mT" if c["m_t"] else ""))


@pytest.mark.parametrize("n", range(N_CASES), ids=[f"{n}-{case_id(c)}" for n, c in enumerate(CASES)])
def test_random_case(n):
    c = CASES[n]
    S, B, H, W, dt = c["S"], c["B"], c["H"], c["W"], c["dt"]
    wl = datagen.Workload("sweep", S, B, H, dt, W=W, mask=c["mask"])
    inp = datagen.generate(wl, seed=n)
    gy, x, w = (to_device(inp[k], dt) for k in ("gy", "x", "w"))
    mask = None if inp["mask"] is None else torch.from_numpy(inp["mask"]).cuda()
    if c["w_t"]:
        w = w.t().contiguous().t()          # [H,W] memory seen as [W,H]
    if c["m_t"]:
        mask = mask.t().contiguous().t()    # [S,B] memory seen as [B,S]
    gy_v, x_v = view3(gy, c["layout"]), view3(x, c["layout"])
    gx = guarded_full((S, B, H), gy.dtype, 0xFF)   # NaN patterns
    gw = guarded_full((W, H), gy.dtype, 0xFF)
    stream = torch.cuda.current_stream()
    dense = W == 3 and c["layout"] == "sbh" and not c["w_t"] and not c["m_t"]

    def call(fill):
        """One call with the workspace pre-filled with `fill` bytes."""
        if dense:
            nb = m.mcc1d_bwd_workspace_size(S, B, H, W, dt, mask is not None)
            ws = guarded_full((nb,), torch.uint8, fill)
            m.mcc1d_bwd(gy_v, x_v, w, mask, gx, gw, ws, stream, S, B, H, W, dt, nb)
        else:
            t = m.tensors(gy_v, x_v, w, mask, gx, gw)
            nb = m.mcc1d_bwd_ex_workspace_size(t, S, B, H, W, dt)
            ws = guarded_full((nb,), torch.uint8, fill)
            m.mcc1d_bwd_ex(t, S, B, H, W, dt, ws, nb, stream)
        assert m.mcc1d_bwd_device_status(ws, stream) == 0
        check_guards(gx, gw, ws, what="backward")
        return (gx.view(torch.int16).cpu().numpy().view(np.uint16).copy(),
                gw.view(torch.int16).cpu().numpy().view(np.uint16).copy())

    gxb, gwb = call(0xFF)
    gx2, gw2 = call(0x00)   # deterministic: a second call with other workspace garbage
    assert np.array_equal(gxb, gx2) and np.array_equal(gwb, gw2)
    ref = oracle.bwd(S, B, H, W, dt, inp["gy"], inp["x"], inp["w"], inp["mask"], want_exact=True)
    ulp = max_ulp(gxb, ref["gx"])
    assert ulp <= GX_MAX_ULP, f"gradX off by {ulp} ulp"
    ratio = gradw_ratio(gwb, ref["gw_exact"], ref["gw_abs"], dt)
    assert ratio <= 1.0, f"gradWeight error is {ratio:.3f} x tolerance"


N_FWD_CASES = 80


def draw_fwd_case(n):
    c = draw_case(20000 + n)
    c["W"] = int(np.random.default_rng(30000 + n).integers(1, 9))
    return c


FWD_CASES = [draw_fwd_case(n) for n in range(N_FWD_CASES)]


@pytest.mark.parametrize("n", range(N_FWD_CASES), ids=[f"{n}-{case_id(c)}" for n, c in enumerate(FWD_CASES)])
def test_random_forward_case(n):
    """The forward on the same kind of draws: the strided call (any layout of
    x, [H,W]-memory weight, [S,B]-memory mask) gives the same bits as the
    dense call, within 1 ulp of the oracle."""
    c = FWD_CASES[n]
    S, B, H, W, dt = c["S"], c["B"], c["H"], c["W"], c["dt"]
    wl = datagen.Workload("fsweep", S, B, H, dt, W=W, mask=c["mask"])
    inp = datagen.generate(wl, seed=n)
    x, w = to_device(inp["x"], dt), to_device(inp["w"], dt)
    mask = None if inp["mask"] is None else torch.from_numpy(inp["mask"]).cuda()
    stream = torch.cuda.current_stream()
    y = guarded_full((S, B, H), x.dtype, 0xFF)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    m.mcc1d_fwd(x, w, mask, y, stream, S, B, H, W, dt, status)
    wv = w.t().contiguous().t() if c["w_t"] else w
    mv = mask.t().contiguous().t() if (c["m_t"] and mask is not None) else mask
    y2 = guarded_full((S, B, H), x.dtype, 0xFF)
    xv = view3(x, c["layout"])          # held: the descriptor keeps only raw pointers
    t = m.fwd_tensors(xv, wv, mv, y2)
    nb = m.mcc1d_fwd_ex_workspace_size(t, S, B, H, W, dt)
    ws = guarded_full((max(nb, 16),), torch.uint8, 0xFF)
    m.mcc1d_fwd_ex(t, S, B, H, W, dt, ws, nb, stream, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    check_guards(y, y2, ws, what="forward")
    yb = y.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(yb, y2.view(torch.int16).cpu().numpy().view(np.uint16))
    ref = oracle.fwd_bits(S, B, H, W, dt, inp["x"], inp["w"], inp["mask"])
    assert max_ulp(yb, ref) <= GX_MAX_ULP
