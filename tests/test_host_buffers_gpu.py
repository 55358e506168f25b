"""mcc1d_bwd_host: the backward on tensors in page-locked host memory.

The kernel reads gradY, x, weight and mask and writes gradX and gradWeight
in place over the host link. gradX must equal mcc1d_bwd's bit for bit (same
arithmetic per element); gradWeight must meet its tolerance against the
oracle (its partial sums are grouped differently).
"""
import numpy as np
import pytest

import datagen
import oracle
from parity import GX_MAX_ULP, check_guards, gradw_ratio, guarded_full, max_ulp, run_cuda

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import causal_conv_backward_gb300 as m  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from causal_conv_backward_gb300 import build
    build.build()


def pinned16(a):
    t = torch.empty(a.shape, dtype=torch.int16, pin_memory=True)
    t.copy_(torch.from_numpy(np.ascontiguousarray(a).view(np.int16)))
    return t


def run_host(inp, S, B, H, dt, outputs_on_device=False):
    gy, x, w = pinned16(inp["gy"]), pinned16(inp["x"]), pinned16(inp["w"])
    mask = None
    if inp["mask"] is not None:
        mask = torch.empty(inp["mask"].shape, dtype=torch.uint8, pin_memory=True)
        mask.copy_(torch.from_numpy(inp["mask"]))
    pin = not outputs_on_device
    gx = guarded_full((S, B, H), torch.int16, 0xFF, pin_memory=pin)
    gw = guarded_full((3, H), torch.int16, 0xFF, pin_memory=pin)
    nb = m.mcc1d_bwd_workspace_size(S, B, H, 3, dt, mask is not None)
    ws = guarded_full((nb,), torch.uint8, 0xFF)
    s = torch.cuda.current_stream()
    m.mcc1d_bwd_host(gy, x, w, mask, gx, gw, ws, s, S, B, H, 3, dt, nb)
    assert m.mcc1d_bwd_device_status(ws, s) == 0   # synchronises the stream
    check_guards(gx, gw, ws, what="mcc1d_bwd_host")
    return gx.cpu().numpy().view(np.uint16), gw.cpu().numpy().view(np.uint16)


CASES = [("s64_b2_h384_bf16", None), ("s4096_b8_h2048_bf16", None), ("s16384_b32_h4096_fp16", 2048),
         ("s524288_b1_h384_bf16", 65536), ("s8192_b4_h24576_bf16", 1024)]


@pytest.mark.parametrize("name,seq", CASES, ids=[f"{n}{'' if s is None else f'_s{s}'}" for n, s in CASES])
@pytest.mark.parametrize("mask", [True, False], ids=["mask", "nomask"])
def test_host_buffers_match_device_call(name, seq, mask):
    wl = datagen.WORKLOADS[name]
    if seq is not None:
        wl = wl.resized(S=seq)
    if not mask:
        wl = wl.without_mask()
    inp = datagen.generate(wl, seed=6)
    gx_h, gw_h = run_host(inp, wl.S, wl.B, wl.H, wl.dtype)
    gx_d, gw_d, st, _ = run_cuda(inp, wl.S, wl.B, wl.H, wl.dtype)
    assert st == 0
    assert np.array_equal(gx_h, gx_d)
    ref = oracle.bwd(wl.S, wl.B, wl.H, 3, wl.dtype, inp["gy"], inp["x"], inp["w"], inp["mask"],
                     want_exact=True)
    assert max_ulp(gx_h, ref["gx"]) <= GX_MAX_ULP
    assert gradw_ratio(gw_h, ref["gw_exact"], ref["gw_abs"], wl.dtype) <= 1.0


@pytest.mark.parametrize("S", [1, 2, 3, 9, 70])
def test_host_buffers_edge_and_device_outputs(S):
    wl = datagen.Workload("hb", S, 3, 1088, "fp16", mask=("bernoulli", 0.7))
    inp = datagen.generate(wl, seed=S)
    gx_h, gw_h = run_host(inp, S, 3, 1088, "fp16", outputs_on_device=True)
    ref = oracle.bwd(S, 3, 1088, 3, "fp16", inp["gy"], inp["x"], inp["w"], inp["mask"], want_exact=True)
    assert max_ulp(gx_h, ref["gx"]) <= GX_MAX_ULP
    assert gradw_ratio(gw_h, ref["gw_exact"], ref["gw_abs"], "fp16") <= 1.0


def test_pageable_host_memory_is_rejected():
    """Memory the device cannot reach is refused before any launch."""
    S, B, H = 64, 2, 384
    gy = np.zeros((S, B, H), np.uint16)      # pageable numpy buffers
    x = np.zeros((S, B, H), np.uint16)
    w = np.zeros((3, H), np.uint16)
    gx = np.zeros((S, B, H), np.uint16)
    gw = np.zeros((3, H), np.uint16)
    nb = m.mcc1d_bwd_workspace_size(S, B, H, 3, 0, False)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    rc = m.load().mcc1d_bwd_host(gy.ctypes.data, x.ctypes.data, w.ctypes.data, None, gx.ctypes.data,
                                 gw.ctypes.data, ws.data_ptr(), None, S, B, H, 3, 0, nb)
    assert rc == 161002
