"""The forward kernel (mcc1d_fwd) against the oracle's forward.

y(t,j,h) = mask(j,t) * sum_k weight(k,h) * x(t-(W-1)+k, j, h), x zero before
t = 0: the map whose transpose is the page's backward. y must be within
1 ulp of the oracle's fp64 value rounded once, at full workload sizes and on
edge shapes, for W = 3 and every other width 1..8; masked rows are exactly
zero.
"""
import numpy as np
import pytest

import datagen
import oracle
from parity import GX_MAX_ULP, check_guards, guarded_full, max_ulp, to_device, values

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import causal_conv_backward_gb300 as m  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from causal_conv_backward_gb300 import build
    build.build()


def run_fwd(inp, S, B, H, dt, mask_override=None, use_override=False, W=3):
    x = to_device(inp["x"], dt)
    w = to_device(inp["w"], dt)
    mask = mask_override if use_override else inp["mask"]
    md = None if mask is None else torch.from_numpy(np.ascontiguousarray(mask)).cuda()
    y = guarded_full(x.shape, x.dtype, 0xFF)   # NaN patterns
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    m.mcc1d_fwd(x, w, md, y, torch.cuda.current_stream(), S, B, H, W, dt, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    check_guards(y, what="mcc1d_fwd y")
    return y.view(torch.int16).cpu().numpy().view(np.uint16)


CASES = [("s64_b2_h384_bf16", True), ("s64_b2_h384_bf16", False), ("s4096_b8_h2048_bf16", True),
         ("s524288_b1_h384_bf16", True), ("s8192_b4_h24576_bf16", True),
         ("s16384_b32_h4096_fp16", True), ("s16384_b32_h4096_fp16", False)]


@pytest.mark.parametrize("name,with_mask", CASES, ids=[f"{n}{'' if k else '_nomask'}" for n, k in CASES])
def test_forward_full(name, with_mask):
    wl = datagen.WORKLOADS[name]
    if not with_mask:
        wl = wl.without_mask()
    inp = datagen.generate(wl, seed=0)
    y = run_fwd(inp, wl.S, wl.B, wl.H, wl.dtype)
    ref = oracle.fwd_bits(wl.S, wl.B, wl.H, 3, wl.dtype, inp["x"], inp["w"], inp["mask"])
    ulp = max_ulp(y, ref)
    assert ulp <= GX_MAX_ULP, f"y off by {ulp} ulp"


EDGE = []
for dt in ("bf16", "fp16"):
    for S in (1, 2, 3, 4, 5, 9, 64, 65, 129):
        EDGE.append((S, 1, 384, dt))
    for (S, B, H) in ((3, 5, 1088), (33, 2, 2112), (7, 32, 1024), (9, 2, 24576), (1000, 3, 448),
                      (700, 3, 1920), (20000, 2, 768), (30000, 1, 640)):
        EDGE.append((S, B, H, dt))


@pytest.mark.parametrize("S,B,H,dt", EDGE, ids=[f"s{a}_b{b}_h{c}_{d}" for a, b, c, d in EDGE])
def test_forward_edge_shapes(S, B, H, dt):
    wl = datagen.Workload("fe", S, B, H, dt, mask=("bernoulli", 0.7))
    inp = datagen.generate(wl, seed=S * 7 + H)
    y = run_fwd(inp, S, B, H, dt)
    ref = oracle.fwd_bits(S, B, H, 3, dt, inp["x"], inp["w"], inp["mask"])
    assert max_ulp(y, ref) <= GX_MAX_ULP


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_forward_mask_semantics(dt):
    S, B, H = 300, 3, 1088
    wl = datagen.Workload("fm", S, B, H, dt, mask=("bernoulli", 0.6))
    inp = datagen.generate(wl, seed=1)
    y = run_fwd(inp, S, B, H, dt)
    assert np.all(values(y, dt)[inp["mask"].T == 0] == 0)      # masked rows are zero
    y0 = run_fwd(inp, S, B, H, dt, np.zeros((B, S), np.uint8), True)
    assert np.all(values(y0, dt) == 0)
    yn = run_fwd(inp, S, B, H, dt, None, True)
    y1 = run_fwd(inp, S, B, H, dt, np.ones((B, S), np.uint8), True)
    assert np.array_equal(yn, y1)


def test_forward_deterministic():
    wl = datagen.WORKLOADS["s4096_b8_h2048_bf16"]
    inp = datagen.generate(wl, seed=2)
    a = run_fwd(inp, wl.S, wl.B, wl.H, wl.dtype)
    for _ in range(3):
        assert np.array_equal(a, run_fwd(inp, wl.S, wl.B, wl.H, wl.dtype))


WIDTHS = []
for W in (1, 2, 4, 5, 6, 7, 8):
    for (S, B, H, dt) in ((1, 2, 384, "bf16"), (W, 1, 1088, "fp16"), (W + 1, 3, 448, "bf16"),
                          (77, 3, 2112, "fp16"), (5000, 2, 640, "bf16")):
        WIDTHS.append((W, S, B, H, dt))


@pytest.mark.parametrize("W,S,B,H,dt", WIDTHS, ids=[f"w{a}_s{b}_b{c}_h{d}_{e}" for a, b, c, d, e in WIDTHS])
def test_forward_widths(W, S, B, H, dt):
    wl = datagen.Workload("fw", S, B, H, dt, W=W, mask=("bernoulli", 0.8))
    inp = datagen.generate(wl, seed=W * 31 + S)
    y = run_fwd(inp, S, B, H, dt, W=W)
    ref = oracle.fwd_bits(S, B, H, W, dt, inp["x"], inp["w"], inp["mask"])
    assert max_ulp(y, ref) <= GX_MAX_ULP


@pytest.mark.parametrize("W", [2, 4, 8])
def test_forward_width_full_size(W):
    """4096 x 8 x 2048 bf16 (a full workload) at other widths."""
    wl = datagen.WORKLOADS["s4096_b8_h2048_bf16"].resized(W=W)
    inp = datagen.generate(wl, seed=W)
    y = run_fwd(inp, wl.S, wl.B, wl.H, wl.dtype, W=W)
    ref = oracle.fwd_bits(wl.S, wl.B, wl.H, W, wl.dtype, inp["x"], inp["w"], inp["mask"])
    assert max_ulp(y, ref) <= GX_MAX_ULP


# 4 KB rows over CTA ranges of at least 1024 rows: y leaves by bulk copies.
BULK = [(20000, 8, 4096, "bf16", ("spans", 0.2, 64, 1024)), (12000, 16, 6144, "fp16", ("bernoulli", 0.9)),
        (40001, 4, 4096, "fp16", ("prefix",))]


@pytest.mark.parametrize("S,B,H,dt,mask", BULK, ids=[f"s{a}_b{b}_h{c}_{d}_{e[0]}" for a, b, c, d, e in BULK])
def test_forward_bulk_store_plans(S, B, H, dt, mask):
    wl = datagen.Workload("fbulk", S, B, H, dt, mask=mask)
    inp = datagen.generate(wl, seed=S + 7)
    y = run_fwd(inp, S, B, H, dt)
    ref = oracle.fwd_bits(S, B, H, 3, dt, inp["x"], inp["w"], inp["mask"])
    assert max_ulp(y, ref) <= GX_MAX_ULP
