"""Strided (non-contiguous) inputs through mcc1d_bwd_ex on the GPU.

The operator page accepts non-contiguous gradY, x, weight and mask (the
非连续Tensor column of its parameter table). Each layout below is a view a
caller would plausibly hold; the results must equal, bit for bit, those of
mcc1d_bwd on dense copies of the same values, and match the oracle.
"""
import numpy as np
import pytest

import datagen
from parity import GX_MAX_ULP, check_guards, gradw_ratio, guarded_empty, guarded_full, max_ulp, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import causal_conv_backward_gb300 as m  # noqa: E402
import oracle  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from causal_conv_backward_gb300 import build
    build.build()


def make_view(dense, layout):
    """A view of `dense` [S,B,H] with the same values and a different layout."""
    S, B, H = dense.shape
    if layout == "sbh":
        return dense
    if layout == "bsh":          # [B,S,H] memory seen as [S,B,H]
        return dense.transpose(0, 1).contiguous().transpose(0, 1)
    if layout == "hslice":       # H-slice of a wider buffer, 16-byte aligned rows
        buf = torch.zeros((S, B, H + 64), dtype=dense.dtype, device=dense.device)
        buf[:, :, 32:32 + H] = dense
        return buf[:, :, 32:32 + H]
    if layout == "hslice_odd":   # rows start 2 bytes off a 16-byte boundary
        buf = torch.zeros((S, B, H + 8), dtype=dense.dtype, device=dense.device)
        buf[:, :, 1:1 + H] = dense
        return buf[:, :, 1:1 + H]
    if layout == "hstride2":     # every other element along H
        buf = torch.zeros((S, B, 2 * H), dtype=dense.dtype, device=dense.device)
        buf[:, :, ::2] = dense
        return buf[:, :, ::2]
    if layout == "shb":          # [S,H,B] memory seen as [S,B,H] (H stride = B)
        return dense.transpose(1, 2).contiguous().transpose(1, 2)
    raise ValueError(layout)


def run_dense(gy, x, w, mask, S, B, H, dt):
    gx = guarded_empty((S, B, H), gy.dtype)
    gw = guarded_empty((3, H), gy.dtype)
    nb = m.mcc1d_bwd_workspace_size(S, B, H, 3, dt, mask is not None)
    ws = guarded_full((nb,), torch.uint8, 0xFF)
    m.mcc1d_bwd(gy, x, w, mask, gx, gw, ws, torch.cuda.current_stream(), S, B, H, 3, dt, nb)
    torch.cuda.synchronize()
    check_guards(gx, gw, ws, what="mcc1d_bwd")
    return gx, gw


def run_ex(gy, x, w, mask, S, B, H, dt):
    gx = guarded_full((S, B, H), gy.dtype, 0xFF)   # NaN patterns
    gw = guarded_full((3, H), gy.dtype, 0xFF)
    t = m.tensors(gy, x, w, mask, gx, gw)
    nb = m.mcc1d_bwd_ex_workspace_size(t, S, B, H, 3, dt)
    ws = guarded_full((nb,), torch.uint8, 0xFF)
    m.mcc1d_bwd_ex(t, S, B, H, 3, dt, ws, nb, torch.cuda.current_stream())
    torch.cuda.synchronize()
    check_guards(gx, gw, ws, what="mcc1d_bwd_ex")
    return gx, gw, nb


CASES = []
for shape in [(777, 3, 1088, "bf16"), (1000, 1, 384, "fp16"), (130, 5, 2112, "fp16")]:
    for lay in ("bsh", "hslice", "hslice_odd", "hstride2", "shb"):
        CASES.append((*shape, lay))


@pytest.mark.parametrize("S,B,H,dt,layout", CASES, ids=[f"s{a}_b{b}_h{c}_{d}_{e}" for a, b, c, d, e in CASES])
def test_strided_inputs_match_dense(S, B, H, dt, layout):
    wl = datagen.Workload("strided", S, B, H, dt, mask=("bernoulli", 0.75))
    inp = datagen.generate(wl, seed=S + H)
    gy, x, w = (to_device(inp[k], dt) for k in ("gy", "x", "w"))
    mask = torch.from_numpy(inp["mask"]).cuda()
    gx_d, gw_d = run_dense(gy, x, w, mask, S, B, H, dt)
    # strided gradY/x; weight as the transpose of an [H,W] buffer; mask as the
    # transpose of an [S,B] buffer
    wv = w.t().contiguous().t()
    mv = mask.t().contiguous().t()
    gx_s, gw_s, _ = run_ex(make_view(gy, layout), make_view(x, layout), wv, mv, S, B, H, dt)
    torch.cuda.synchronize()
    assert torch.equal(gx_s.view(torch.int16), gx_d.view(torch.int16)), layout
    assert torch.equal(gw_s.view(torch.int16), gw_d.view(torch.int16)), layout
    ref = oracle.bwd(S, B, H, 3, dt, inp["gy"], inp["x"], inp["w"], inp["mask"], want_exact=True)
    gxb = gx_s.view(torch.int16).cpu().numpy().view(np.uint16)
    gwb = gw_s.view(torch.int16).cpu().numpy().view(np.uint16)
    assert max_ulp(gxb, ref["gx"]) <= GX_MAX_ULP
    assert gradw_ratio(gwb, ref["gw_exact"], ref["gw_abs"], dt) <= 1.0


def test_broadcast_input_stride_zero():
    """x repeated over the batch (stride 0 along B) streams in place."""
    S, B, H, dt = 512, 4, 1024, "bf16"
    wl = datagen.Workload("bcast", S, 1, H, dt, mask=("bernoulli", 0.9))
    one = datagen.generate(wl, seed=9)
    wl4 = datagen.Workload("bcast4", S, B, H, dt, mask=("bernoulli", 0.9))
    full = datagen.generate(wl4, seed=10)
    x1 = to_device(one["x"], dt)                      # [S,1,H]
    xb = x1.expand(S, B, H)                           # stride 0 along B
    gy = to_device(full["gy"], dt)
    w = to_device(full["w"], dt)
    mask = torch.from_numpy(full["mask"]).cuda()
    gx_s, gw_s, nb = run_ex(gy, xb, w, mask, S, B, H, dt)
    gx_d, gw_d = run_dense(gy, xb.contiguous(), w, mask, S, B, H, dt)
    torch.cuda.synchronize()
    assert torch.equal(gx_s.view(torch.int16), gx_d.view(torch.int16))
    assert torch.equal(gw_s.view(torch.int16), gw_d.view(torch.int16))
    assert nb < S * B * H * 2  # no gathered copy was needed


def test_backward_helper_accepts_views():
    S, B, H, dt = 300, 2, 2048, "fp16"
    wl = datagen.Workload("helper", S, B, H, dt, mask=("bernoulli", 0.8))
    inp = datagen.generate(wl, seed=4)
    gy, x, w = (to_device(inp[k], dt) for k in ("gy", "x", "w"))
    mask = torch.from_numpy(inp["mask"]).cuda().bool()
    gx_d, gw_d = m.backward(gy, x, w, mask)
    gx_s, gw_s = m.backward(make_view(gy, "bsh"), make_view(x, "hstride2"), w.t().contiguous().t(),
                            mask.t().contiguous().t())
    torch.cuda.synchronize()
    assert torch.equal(gx_s.view(torch.int16), gx_d.view(torch.int16))
    assert torch.equal(gw_s.view(torch.int16), gw_d.view(torch.int16))


def test_strided_bulk_store_plan():
    """[B,S,H] memory seen as [S,B,H] on a plan whose gradX leaves by bulk
    copies (4 KB rows, long CTA ranges): the same bits as the dense call."""
    S, B, H, dt = 16384, 8, 4096, "fp16"
    p = m.mcc1d_plan_describe(S, B, H, 3, dt, m.PLAN_BWD_EX)
    assert p["hb_width"] == 2048 and p["rows_total"] // p["ncta"] >= 1024
    wl = datagen.Workload("sbulk", S, B, H, dt, mask=("bernoulli", 0.9))
    inp = datagen.generate(wl, seed=77)
    gy, x, w = (to_device(inp[k], dt) for k in ("gy", "x", "w"))
    mask = torch.from_numpy(inp["mask"]).cuda()
    gx_d, gw_d = run_dense(gy, x, w, mask, S, B, H, dt)
    gx_s, gw_s, _ = run_ex(make_view(gy, "bsh"), make_view(x, "bsh"), w, mask, S, B, H, dt)
    torch.cuda.synchronize()
    assert torch.equal(gx_s.view(torch.int16), gx_d.view(torch.int16))
    assert torch.equal(gw_s.view(torch.int16), gw_d.view(torch.int16))
