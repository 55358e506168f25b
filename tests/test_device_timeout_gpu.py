"""A device-side wait that runs out turns into a status code, not a hang.

Every wait in the library's kernels (on the ring's mbarriers) is bounded by
the global timer and reports MCC1D_ERR_DEVICE_TIMEOUT when it gives up. This
test runs the same bounded wait through mcc1d_selftest_wait on a barrier
that nothing ever signals, checks the status and the time it took, and then
runs a normal backward on the same context to show it is still usable. No
kernel here faults, traps or waits without a limit.
"""
import time

import numpy as np
import pytest

import datagen
import oracle
from parity import GX_MAX_ULP, gradw_ratio, max_ulp, run_cuda

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import causal_conv_backward_gb300 as m  # noqa: E402

TIMEOUT = 561101


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from causal_conv_backward_gb300 import build
    build.build()


def run_selftest(arrive):
    word = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    m.mcc1d_selftest_wait(word, arrive, stream)
    torch.cuda.synchronize()
    return int(word.item()), time.perf_counter() - t0


def test_wait_that_is_signalled_succeeds():
    status, dt = run_selftest(True)
    assert status == 0 and dt < 1.0


def test_wait_that_is_never_signalled_reports_timeout_and_context_survives():
    status, dt = run_selftest(False)
    assert status == TIMEOUT, m.mcc1d_status_string(status)
    assert 1.5 < dt < 20.0, dt      # the library's limit is about 2 s
    # the same context still runs the backward correctly
    wl = datagen.WORKLOADS["s64_b2_h384_bf16"]
    inp = datagen.generate(wl, seed=5)
    gx, gw, st, _ = run_cuda(inp, wl.S, wl.B, wl.H, wl.dtype)
    assert st == 0
    ref = oracle.bwd(wl.S, wl.B, wl.H, 3, wl.dtype, inp["gy"], inp["x"], inp["w"], inp["mask"],
                     want_exact=True)
    assert max_ulp(gx, ref["gx"]) <= GX_MAX_ULP
    assert gradw_ratio(gw, ref["gw_exact"], ref["gw_abs"], wl.dtype) <= 1.0
