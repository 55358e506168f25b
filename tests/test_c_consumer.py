"""The library used from plain C, with no Python or torch in the process.

A small C99 program includes ``include/mcc1d.h``, links ``libmcc1d.so`` and
calls it. On the CPU it checks the host-side contract (sizes, validation,
status strings); on the GPU (``-m gpu``) it allocates with the CUDA runtime,
runs the backward on all-ones inputs and compares with the closed form of the
operation for those inputs: gradX(i) = number of taps i+k < S (3, then 2 and
1 at the last two positions), gradWeight(k) = B * (S - (W-1-k)).
"""
import os
import shutil
import subprocess

import pytest

from causal_conv_backward_gb300 import build as cbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")
CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")

HOST_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "mcc1d.h"

#define CHECK(c) do { if (!(c)) { printf("FAIL line %d: %s\n", __LINE__, #c); return 1; } } while (0)

int main(void)
{
    uint64_t n = 0, n2 = 0;
    mcc1d_tensors t;
    CHECK(mcc1d_version() >= 100);
    CHECK(mcc1d_bwd_workspace_size(64, 2, 384, 3, MCC1D_BF16, 1, &n) == MCC1D_OK && n > 0);
    CHECK(mcc1d_bwd_workspace_size(64, 2, 384, 3, MCC1D_FP16, 0, &n2) == MCC1D_OK && n2 == n);
    CHECK(mcc1d_bwd_workspace_size(64, 2, 384, 4, MCC1D_BF16, 1, &n) == MCC1D_ERR_INNER_TILING_ERROR);
    CHECK(mcc1d_bwd_workspace_size(64, 33, 384, 3, MCC1D_BF16, 1, &n) == MCC1D_ERR_INNER_TILING_ERROR);
    CHECK(mcc1d_bwd_workspace_size(64, 2, 384, 3, 7, 1, &n) == MCC1D_ERR_PARAM_INVALID);
    CHECK(mcc1d_bwd_workspace_size(64, 2, 384, 3, MCC1D_BF16, 1, NULL) == MCC1D_ERR_PARAM_NULLPTR);
    /* validation happens before any device work: a null input is refused */
    CHECK(mcc1d_bwd(NULL, (void *)256, (void *)512, NULL, (void *)768, (void *)1024, (void *)4096, NULL,
                    64, 2, 384, 3, MCC1D_BF16, 1u << 20) == MCC1D_ERR_PARAM_NULLPTR);
    memset(&t, 0, sizeof t);
    t.gradY = (void *)0x10000; t.x = (void *)0x20000; t.weight = (void *)0x30000;
    t.gradX = (void *)0x40000; t.gradWeight = (void *)0x50000;
    t.gradY_strides[0] = 2 * 384; t.gradY_strides[1] = 384; t.gradY_strides[2] = 1;
    memcpy(t.x_strides, t.gradY_strides, sizeof t.x_strides);
    t.weight_strides[0] = 384; t.weight_strides[1] = 1;
    CHECK(mcc1d_bwd_ex_workspace_size(&t, 64, 2, 384, 8, MCC1D_BF16, &n) == MCC1D_OK && n > 0);
    CHECK(mcc1d_bwd_ex_workspace_size(&t, 64, 2, 384, 9, MCC1D_BF16, &n) == MCC1D_ERR_INNER_TILING_ERROR);
    CHECK(strncmp(mcc1d_status_string(MCC1D_OK), "MCC1D_", 6) == 0);
    printf("ok\n");
    return 0;
}
"""

GPU_PROGRAM = r"""
#include <stdio.h>
#include <stdlib.h>
#include <cuda_runtime_api.h>
#include "mcc1d.h"

#define CHECK(c) do { if (!(c)) { printf("FAIL line %d: %s\n", __LINE__, #c); return 1; } } while (0)

static float bf16_value(uint16_t b)
{
    union { uint32_t u; float f; } v;
    v.u = (uint32_t)b << 16;
    return v.f;
}

int main(void)
{
    const int64_t S = 64, B = 2, H = 384, W = 3;
    const size_t E = (size_t)(S * B * H);
    const uint16_t one = 0x3F80; /* 1.0 in bf16 */
    uint16_t *h_in = (uint16_t *)malloc(E * 2), *h_gx = (uint16_t *)malloc(E * 2);
    uint16_t h_w[3 * 384], h_gw[3 * 384];
    void *gy, *x, *w, *gx, *gw, *ws;
    uint64_t nbytes = 0;
    int32_t dev_status = -1;
    size_t e;
    int64_t i, j, h, k;
    CHECK(h_in && h_gx);
    for (e = 0; e < E; ++e) h_in[e] = one;
    for (e = 0; e < 3 * 384; ++e) h_w[e] = one;
    CHECK(mcc1d_bwd_workspace_size(S, B, H, W, MCC1D_BF16, 0, &nbytes) == MCC1D_OK);
    CHECK(cudaMalloc(&gy, E * 2) == cudaSuccess && cudaMalloc(&x, E * 2) == cudaSuccess);
    CHECK(cudaMalloc(&gx, E * 2) == cudaSuccess && cudaMalloc(&w, W * H * 2) == cudaSuccess);
    CHECK(cudaMalloc(&gw, W * H * 2) == cudaSuccess && cudaMalloc(&ws, nbytes) == cudaSuccess);
    CHECK(cudaMemcpy(gy, h_in, E * 2, cudaMemcpyHostToDevice) == cudaSuccess);
    CHECK(cudaMemcpy(x, h_in, E * 2, cudaMemcpyHostToDevice) == cudaSuccess);
    CHECK(cudaMemcpy(w, h_w, W * H * 2, cudaMemcpyHostToDevice) == cudaSuccess);
    CHECK(cudaMemset(gx, 0xFF, E * 2) == cudaSuccess && cudaMemset(gw, 0xFF, W * H * 2) == cudaSuccess);
    CHECK(mcc1d_bwd(gy, x, w, NULL, gx, gw, ws, NULL, S, B, H, W, MCC1D_BF16, nbytes) == MCC1D_OK);
    CHECK(mcc1d_bwd_device_status(ws, NULL, &dev_status) == MCC1D_OK && dev_status == MCC1D_OK);
    CHECK(cudaMemcpy(h_gx, gx, E * 2, cudaMemcpyDeviceToHost) == cudaSuccess);
    CHECK(cudaMemcpy(h_gw, gw, W * H * 2, cudaMemcpyDeviceToHost) == cudaSuccess);
    for (i = 0; i < S; ++i)
        for (j = 0; j < B; ++j)
            for (h = 0; h < H; ++h) {
                const float want = (float)(S - i < 3 ? S - i : 3);
                CHECK(bf16_value(h_gx[(i * B + j) * H + h]) == want);
            }
    for (k = 0; k < W; ++k)
        for (h = 0; h < H; ++h)
            CHECK(bf16_value(h_gw[k * H + h]) == (float)(B * (S - (W - 1 - k))));
    cudaFree(gy); cudaFree(x); cudaFree(w); cudaFree(gx); cudaFree(gw); cudaFree(ws);
    free(h_in); free(h_gx);
    printf("ok\n");
    return 0;
}
"""


def _compile_and_run(tmp_path, source, extra_flags=(), extra_libs=()):
    lib = cbuild.build()
    libdir = os.path.dirname(lib)
    src = tmp_path / "consumer.c"
    src.write_text(source)
    exe = tmp_path / "consumer"
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", f"-I{INCLUDE}", *extra_flags,
           str(src), "-o", str(exe), f"-L{libdir}", "-lmcc1d", f"-Wl,-rpath,{libdir}", *extra_libs]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no host C compiler")
def test_header_is_plain_c_and_host_contract_holds(tmp_path):
    _compile_and_run(tmp_path, HOST_PROGRAM)


@pytest.mark.skipif(shutil.which("g++") is None, reason="no host C++ compiler")
def test_header_compiles_as_cpp(tmp_path):
    src = tmp_path / "consumer.cpp"
    src.write_text('#include "mcc1d.h"\nint main() { return mcc1d_version() > 0 ? 0 : 1; }\n')
    subprocess.run(["g++", "-std=c++11", "-Wall", "-Werror", f"-I{INCLUDE}", "-fsyntax-only", str(src)],
                   check=True, capture_output=True, text=True)


@pytest.mark.gpu
def test_c_program_runs_the_backward(tmp_path):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _compile_and_run(tmp_path, GPU_PROGRAM, extra_flags=["-isystem", f"{CUDA_HOME}/include"],
                     extra_libs=[f"-L{CUDA_HOME}/lib64", "-lcudart", f"-Wl,-rpath,{CUDA_HOME}/lib64"])
