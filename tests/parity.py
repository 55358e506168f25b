"""Shared helpers of the parity tests: run the CUDA path through the C ABI,
and compare its outputs with the oracle's under the stated tolerances.

Tolerances (the operation's acceptance bar):
* gradX: at most 1 unit in the last place of the output type from the oracle's
  fp64 value rounded once (distance between bit patterns, +0 == -0);
* gradWeight: |gpu - exact| <= 1e-5 * sum|terms| + ulp(exact) per (k, h),
  exact and sum|terms| being the oracle's fp64 values.
"""
from __future__ import annotations

import numpy as np

GX_MAX_ULP = 1
GW_REL = 1e-5

TORCH_DT = {"bf16": "bfloat16", "fp16": "float16"}


def ordinal(bits: np.ndarray) -> np.ndarray:
    b = bits.astype(np.int32)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def max_ulp(a: np.ndarray, b: np.ndarray, chunk: int = 1 << 26) -> int:
    a = a.reshape(-1)
    b = b.reshape(-1)
    m = 0
    for s in range(0, a.size, chunk):
        d = np.abs(ordinal(a[s:s + chunk]) - ordinal(b[s:s + chunk]))
        if d.size:
            m = max(m, int(d.max()))
    return m


def values(bits: np.ndarray, dtype: str) -> np.ndarray:
    b = np.asarray(bits, np.uint16)
    with np.errstate(invalid="ignore"):
        if dtype == "fp16":
            return b.view(np.float16).astype(np.float64)
        return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def ulp_of(v: np.ndarray, dtype: str) -> np.ndarray:
    """Spacing of the 16-bit grid at |v| (for v already representable or not)."""
    a = np.abs(np.asarray(v, np.float64))
    man, emin = (7, -126) if dtype == "bf16" else (10, -14)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, emin)
    return np.ldexp(1.0, (e - man).astype(np.int64))


def gradw_ratio(gpu_bits, exact, abs_sum, dtype) -> float:
    """max over (k,h) of |gpu - exact| / (1e-5 * sum|terms| + ulp(exact))."""
    g = values(gpu_bits, dtype)
    tol = GW_REL * abs_sum + ulp_of(exact, dtype)
    return float(np.max(np.abs(g - exact) / tol))


# ------------------------------------------------------------------ guard bands
# Every output and workspace a parity test hands to the library is carved out
# of a larger allocation with GUARD_BYTES of a fixed pattern before and after
# it. After the call, check_guards() asserts that the pattern is intact, so a
# store past either end of a buffer (which would otherwise land silently in
# the caching allocator's memory) fails the test.
GUARD_BYTES = 4096
GUARD_PATTERN = 0xC3


class _Guard:
    __slots__ = ("base", "nbytes")

    def __init__(self, base, nbytes):
        self.base = base
        self.nbytes = nbytes


def guarded_empty(shape, dtype, device="cuda", *, pin_memory=False):
    """An uninitialised tensor of `shape`/`dtype` (contiguous, 256-byte
    aligned) with guard regions around it; check it with check_guards()."""
    import torch
    shape = tuple(int(d) for d in shape)
    elem = torch.empty((), dtype=dtype).element_size()
    nbytes = int(np.prod(shape, dtype=np.int64)) * elem
    inner = (nbytes + 255) // 256 * 256
    if pin_memory:
        base = torch.empty(2 * GUARD_BYTES + inner, dtype=torch.uint8, pin_memory=True)
    else:
        base = torch.empty(2 * GUARD_BYTES + inner, dtype=torch.uint8, device=device)
    base.fill_(GUARD_PATTERN)
    t = base[GUARD_BYTES:GUARD_BYTES + nbytes].view(dtype).view(shape)
    t._mcc1d_guard = _Guard(base, nbytes)
    return t


def guarded_full(shape, dtype, fill_byte, device="cuda", *, pin_memory=False):
    """guarded_empty() with every byte of the tensor set to `fill_byte`."""
    import torch
    t = guarded_empty(shape, dtype, device, pin_memory=pin_memory)
    if t.numel():
        t.view(-1).view(torch.uint8).fill_(fill_byte)
    return t


def check_guards(*tensors, what=""):
    """Assert that the guard regions of every tensor made by guarded_empty()
    still hold the pattern (call after the work on them has completed)."""
    for k, t in enumerate(tensors):
        g = getattr(t, "_mcc1d_guard", None) if t is not None else None
        if g is None:
            continue
        head = g.base[:GUARD_BYTES]
        tail = g.base[GUARD_BYTES + g.nbytes:]
        bad_head = int((head != GUARD_PATTERN).sum())
        bad_tail = int((tail != GUARD_PATTERN).sum())
        assert bad_head == 0 and bad_tail == 0, (
            f"{what} buffer {k}: {bad_head} guard bytes before and {bad_tail} after it were overwritten")


def to_device(bits: np.ndarray, dtype: str, device="cuda"):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device)
    return t.view(getattr(torch, TORCH_DT[dtype]))


_KEEP = object()


def run_cuda(inp: dict, S, B, H, dtype, *, W=3, stream=None, workspace=None, fill_outputs=True,
             mask_override=_KEEP):
    """Run the CUDA path once through the C ABI; returns (gx_bits, gw_bits,
    device_status, workspace). Outputs are pre-filled with NaN patterns so an
    unwritten element cannot pass; outputs and workspace sit between guard
    regions that are checked after the call."""
    import torch
    import causal_conv_backward_gb300 as m

    gy = to_device(inp["gy"], dtype)
    x = to_device(inp["x"], dtype)
    w = to_device(inp["w"], dtype)
    mask = inp["mask"] if mask_override is _KEEP else mask_override
    md = None if mask is None else torch.from_numpy(np.ascontiguousarray(mask)).cuda()
    gx = guarded_empty(gy.shape, gy.dtype)
    gw = guarded_empty(w.shape, w.dtype)
    if fill_outputs:
        gx.view(torch.int16).fill_(-1)   # 0xFFFF: a NaN in both formats
        gw.view(torch.int16).fill_(-1)
    code = m.dtype_code(dtype)
    nbytes = m.mcc1d_bwd_workspace_size(S, B, H, W, code, md is not None)
    if workspace is None:
        workspace = guarded_full((nbytes,), torch.uint8, 0xFF)
    if stream is None:
        stream = torch.cuda.current_stream()
    else:
        stream.wait_stream(torch.cuda.current_stream())  # inputs were made on torch's stream
    m.mcc1d_bwd(gy, x, w, md, gx, gw, workspace, stream, S, B, H, W, code, workspace.numel())
    status = m.mcc1d_bwd_device_status(workspace, stream)  # synchronises `stream`
    check_guards(gx, gw, workspace, what="mcc1d_bwd gradX/gradWeight/workspace")
    gxb = gx.view(torch.int16).cpu().numpy().view(np.uint16)
    gwb = gw.view(torch.int16).cpu().numpy().view(np.uint16)
    return gxb, gwb, status, workspace
