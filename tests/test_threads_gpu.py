"""Calls from several host threads at once, each on its own stream and
workspace, give the same bits as the same calls made one after another.
ctypes releases the GIL during the C call, so the library's per-kernel setup
(shared-memory attributes, the forward's register query) really does run
concurrently; the first calls of each kernel happen inside the threads."""
import threading

import numpy as np
import pytest

import datagen
from parity import to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import causal_conv_backward_gb300 as m  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from causal_conv_backward_gb300 import build
    build.build()


SHAPES = [(301, 3, 448, "fp16"), (1000, 2, 1344, "bf16"), (77, 5, 2112, "bf16"), (2048, 1, 640, "fp16"),
          (500, 4, 960, "bf16"), (64, 2, 384, "fp16")]


def make(S, B, H, dt, seed):
    wl = datagen.Workload("thr", S, B, H, dt, mask=("bernoulli", 0.8))
    inp = datagen.generate(wl, seed=seed)
    return {k: (None if v is None else (to_device(v, dt) if v.dtype == np.uint16 else torch.from_numpy(v).cuda()))
            for k, v in inp.items()}


def run(S, B, H, dt, t, stream):
    with torch.cuda.stream(stream):
        gx = torch.empty_like(t["gy"])
        gw = torch.empty_like(t["w"])
        y = torch.empty_like(t["x"])
        nb = m.mcc1d_bwd_workspace_size(S, B, H, 3, dt, True)
        ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    for _ in range(3):
        m.mcc1d_bwd(t["gy"], t["x"], t["w"], t["mask"], gx, gw, ws, stream, S, B, H, 3, dt, nb)
        m.mcc1d_fwd(t["x"], t["w"], t["mask"], y, stream, S, B, H, 3, dt)
    stream.synchronize()
    return (gx.view(torch.int16).cpu().numpy(), gw.view(torch.int16).cpu().numpy(),
            y.view(torch.int16).cpu().numpy())


def test_concurrent_threads_match_sequential():
    inputs = [make(*shp, seed=i) for i, shp in enumerate(SHAPES)]
    torch.cuda.synchronize()
    results = [None] * len(SHAPES)
    errors = []

    def worker(i):
        try:
            results[i] = run(*SHAPES[i], inputs[i], torch.cuda.Stream())
        except Exception as e:  # noqa: BLE001
            errors.append((i, repr(e)))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(SHAPES))]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    for i, shp in enumerate(SHAPES):
        ref = run(*shp, inputs[i], torch.cuda.current_stream())
        for a, b in zip(results[i], ref):
            assert np.array_equal(a, b), shp
