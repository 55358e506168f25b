"""mcc1d_bwd_noalloc: the backward for callers that cannot allocate.

Some callers cannot allocate device memory when they call the backward
(code running inside a runtime or framework that owns every device
allocation, or whose memory budget is fixed to the tensors it is handed), so
they cannot supply the workspace that mcc1d_bwd asks for. mcc1d_bwd_noalloc
keeps that scratch in a fixed 8 MiB array inside the library instead.

The GPU test calls it twice in a row through the C ABI, on two different
shapes and dtypes (so the second call runs over what the first left in the
shared array). Each result must equal, bit for bit, mcc1d_bwd's on the same
inputs (same plan, same kernels, same summation order), and must meet the
acceptance bar against the oracle on its own: gradX within 1 ulp of the
oracle's value rounded once, gradWeight within 1e-5 * sum|terms| + 1 ulp of
the oracle's exact sum. The outputs sit between guard regions that must be
untouched afterwards. The file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest

import causal_conv_backward_gb300 as m
import datagen
import oracle
from causal_conv_backward_gb300 import build as cbuild
from parity import GX_MAX_ULP, check_guards, gradw_ratio, guarded_full, max_ulp, run_cuda, to_device


@pytest.fixture(scope="module")
def lib():
    cbuild.build()
    return m.load()


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_and_oracle_twice(lib):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cases = [datagen.WORKLOADS["s4096_b8_h2048_bf16"],
             datagen.Workload("noalloc_s3000_b3_h1088_fp16", 3000, 3, 1088, "fp16",
                              mask=("bernoulli", 0.8))]
    stream = torch.cuda.current_stream()
    for wl in cases:
        inp = datagen.generate(wl, seed=11)
        gx_ref, gw_ref, st, _ = run_cuda(inp, wl.S, wl.B, wl.H, wl.dtype)
        assert st == 0
        gy, x, w = (to_device(inp[k], wl.dtype) for k in ("gy", "x", "w"))
        mask = torch.from_numpy(inp["mask"]).cuda()
        gx = guarded_full(gy.shape, gy.dtype, 0xFF)   # NaN patterns
        gw = guarded_full(w.shape, w.dtype, 0xFF)
        rc = lib.mcc1d_bwd_noalloc(gy.data_ptr(), x.data_ptr(), w.data_ptr(), mask.data_ptr(),
                                   gx.data_ptr(), gw.data_ptr(), ctypes.c_void_p(stream.cuda_stream),
                                   wl.S, wl.B, wl.H, wl.W, m.dtype_code(wl.dtype))
        assert rc == 0, m.mcc1d_status_string(rc)
        stream.synchronize()
        check_guards(gx, gw, what="mcc1d_bwd_noalloc")
        gxb = gx.view(torch.int16).cpu().numpy().view(np.uint16)
        gwb = gw.view(torch.int16).cpu().numpy().view(np.uint16)
        # the same plan and kernels as mcc1d_bwd: the same bits
        assert np.array_equal(gxb, gx_ref), wl.name
        assert np.array_equal(gwb, gw_ref), wl.name
        # and the acceptance bar against the oracle
        ref = oracle.bwd(wl.S, wl.B, wl.H, wl.W, wl.dtype, inp["gy"], inp["x"], inp["w"], inp["mask"],
                         want_exact=True)
        assert max_ulp(gxb, ref["gx"]) <= GX_MAX_ULP, wl.name
        assert gradw_ratio(gwb, ref["gw_exact"], ref["gw_abs"], wl.dtype) <= 1.0, wl.name


def test_noalloc_rejects_bad_arguments_before_any_launch(lib):
    """Argument errors come back before any device work (fake, never
    dereferenced pointers)."""
    good = dict(gy=0x1000, x=0x2000, w=0x3000, gx=0x4000, gw=0x5000)

    def call(S=64, B=2, H=384, W=3, dt=0, **kw):
        a = {**good, **kw}
        return lib.mcc1d_bwd_noalloc(a["gy"], a["x"], a["w"], None, a["gx"], a["gw"], None,
                                     S, B, H, W, dt)

    assert call(gy=None) == 161001
    assert call(gw=None) == 161001
    assert call(x=0x2002) == 161002
    assert call(dt=5) == 161002
    assert call(B=33) == 561002
    assert call(H=390) == 561002


def test_every_valid_shape_fits_the_fixed_scratch(lib):
    """The workspace of every shape the operator accepts fits the 8 MiB array
    (worst cases: 1024-wide H-blocks whose boundaries fall inside CTA ranges)."""
    worst = 0
    for H in range(384, 24577, 64):
        for bs in (1, 7, 64, 100, 1000, 9728, 19456, 38912, 77824, 100000, 262144, 524288):
            for B in (1, 32):
                if bs % B:
                    continue
                n = m.mcc1d_bwd_workspace_size(bs // B, B, H, 3, 0, 1)
                worst = max(worst, n)
    assert worst <= m.NOALLOC_SCRATCH_BYTES, worst
