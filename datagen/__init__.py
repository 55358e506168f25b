"""Seeded synthetic inputs for the masked causal conv1d backward.

The one module that both sides of every parity check draw from: it writes
16-bit bit patterns and mask bytes, and holds none of the operation's
arithmetic. Generation is counter-based (see ``mcc1d_datagen.c``), so the
same (seed, workload) gives the same bits for any thread count.

Workloads (shapes and value laws of the operator page's supported envelope:
B 1..32, B*S up to 512K, H 384..24576 with H % 64 == 0, W = 3):

=========================  =====  ====  ======  =====  ================  ===========  ===========================
name                       S      B     H       dtype  x, gradY          weight       mask
=========================  =====  ====  ======  =====  ================  ===========  ===========================
s64_b2_h384_bf16           64     2     384     bf16   N(0,1)            U(-1,1)      Bernoulli(0.8)
s4096_b8_h2048_bf16        4096   8     2048    bf16   N(0,1)            U(-.5,.5)    prefix of ones, L~U{S/2..S}
s524288_b1_h384_bf16       524288 1     384     bf16   N(0,1)            U(-1,1)      Bernoulli(0.95)
s16384_b32_h4096_fp16      16384  32    4096    fp16   N(0,0.5^2)        U(-1,1)      Bernoulli(0.9)
s8192_b4_h24576_bf16       8192   4     24576   bf16   N(0,1)            U(-1,1)      zero spans, ~20% of tokens
=========================  =====  ====  ======  =====  ================  ===========  ===========================

Stream ids under one seed: x = 1, gradY = 2, weight = 3, mask = 4.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field, replace

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mcc1d_datagen.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libmcc1d_datagen.so")

DTYPE_CODE = {"bf16": 0, "fp16": 1}
STREAM_X, STREAM_GY, STREAM_W, STREAM_MASK = 1, 2, 3, 4

_lock = threading.Lock()
_lib = None


@dataclass(frozen=True)
class Workload:
    name: str
    S: int
    B: int
    H: int
    dtype: str
    W: int = 3
    x: tuple = ("normal", 0.0, 1.0)
    gy: tuple = ("normal", 0.0, 1.0)
    w: tuple = ("uniform", -1.0, 1.0)
    mask: tuple = ("bernoulli", 0.8)   # ("none",) for mask = nullptr
    note: str = field(default="", compare=False)

    @property
    def E(self) -> int:
        return self.S * self.B * self.H

    def algorithmic_bytes(self) -> int:
        """Minimum HBM bytes of one call: read gradY and x, write gradX (2 B
        each per element), read the mask (1 B per token, if any), read weight
        and write gradWeight (W*H 16-bit values each)."""
        has_mask = self.mask[0] != "none"
        return 6 * self.E + (self.B * self.S if has_mask else 0) + 2 * 2 * self.W * self.H

    def fwd_algorithmic_bytes(self) -> int:
        """Minimum HBM bytes of one forward call: read x and write y (2 B each
        per element), read the mask (1 B per token, if any) and the weight."""
        has_mask = self.mask[0] != "none"
        return 4 * self.E + (self.B * self.S if has_mask else 0) + 2 * self.W * self.H

    def without_mask(self) -> "Workload":
        return replace(self, name=self.name + "_nomask", mask=("none",))

    def resized(self, **kw) -> "Workload":
        w = replace(self, **kw)
        return replace(w, name=f"s{w.S}_b{w.B}_h{w.H}_{w.dtype}" + ("" if w.mask[0] != "none" else "_nomask"))


WORKLOADS = {
    w.name: w for w in [
        Workload("s64_b2_h384_bf16", 64, 2, 384, "bf16", mask=("bernoulli", 0.8),
                 note="small case; also run with mask = nullptr"),
        Workload("s4096_b8_h2048_bf16", 4096, 8, 2048, "bf16", w=("uniform", -0.5, 0.5),
                 mask=("prefix",), note="padding-style mask"),
        Workload("s524288_b1_h384_bf16", 524288, 1, 384, "bf16", mask=("bernoulli", 0.95),
                 note="long sequence, narrow H"),
        Workload("s16384_b32_h4096_fp16", 16384, 32, 4096, "fp16", x=("normal", 0.0, 0.5),
                 gy=("normal", 0.0, 0.5), mask=("bernoulli", 0.9),
                 note="512K tokens (B*S = 524288); also run with mask = nullptr"),
        Workload("s8192_b4_h24576_bf16", 8192, 4, 24576, "bf16", mask=("spans", 0.2, 64, 1024),
                 note="widest H"),
    ]
}


def build(force: bool = False) -> str:
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
                           "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i64, i32, u64, vp, d = (ctypes.c_int64, ctypes.c_int, ctypes.c_uint64,
                                ctypes.c_void_p, ctypes.c_double)
        lib.mcc1d_gen_normal.argtypes = [vp, i64, i32, d, d, u64, u64, i32]
        lib.mcc1d_gen_uniform.argtypes = [vp, i64, i32, d, d, u64, u64, i32]
        lib.mcc1d_gen_to16.argtypes = [d, i32]
        lib.mcc1d_gen_to16.restype = ctypes.c_uint16
        lib.mcc1d_gen_mask_bernoulli.argtypes = [vp, i64, i64, d, u64, u64]
        lib.mcc1d_gen_mask_prefix.argtypes = [vp, i64, i64, u64, u64, vp]
        lib.mcc1d_gen_mask_spans.argtypes = [vp, i64, i64, d, i64, i64, u64, u64]
        for f in ("mcc1d_gen_normal", "mcc1d_gen_uniform", "mcc1d_gen_mask_bernoulli",
                  "mcc1d_gen_mask_prefix", "mcc1d_gen_mask_spans"):
            getattr(lib, f).restype = None
        _lib = lib
        return lib


def _ptr(a):
    if isinstance(a, np.ndarray):
        assert a.flags["C_CONTIGUOUS"]
        return a.ctypes.data
    return a.data_ptr()  # CPU torch tensor (e.g. pinned)


def _numel(a) -> int:
    return a.size if isinstance(a, np.ndarray) else a.numel()


def to16(v: float, dtype: str) -> int:
    return int(_load().mcc1d_gen_to16(float(v), DTYPE_CODE[dtype]))


def fill_values(out, law: tuple, dtype: str, seed: int, stream: int, nthreads: int = 0):
    lib = _load()
    kind = law[0]
    if kind == "normal":
        lib.mcc1d_gen_normal(_ptr(out), _numel(out), DTYPE_CODE[dtype], law[1], law[2],
                             seed, stream, nthreads)
    elif kind == "uniform":
        lib.mcc1d_gen_uniform(_ptr(out), _numel(out), DTYPE_CODE[dtype], law[1], law[2],
                              seed, stream, nthreads)
    elif kind == "zeros":
        out[...] = 0
    elif kind == "ones":
        out[...] = to16(1.0, dtype)
    else:
        raise ValueError(f"unknown value law {law}")


def fill_mask(out, law: tuple, B: int, S: int, seed: int, stream: int = STREAM_MASK):
    lib = _load()
    kind = law[0]
    if kind == "bernoulli":
        lib.mcc1d_gen_mask_bernoulli(_ptr(out), B, S, law[1], seed, stream)
    elif kind == "prefix":
        lib.mcc1d_gen_mask_prefix(_ptr(out), B, S, seed, stream, None)
    elif kind == "spans":
        lib.mcc1d_gen_mask_spans(_ptr(out), B, S, law[1], law[2], law[3], seed, stream)
    elif kind == "zeros":
        out[...] = 0
    elif kind == "ones":
        out[...] = 1
    else:
        raise ValueError(f"unknown mask law {law}")


def prefix_lengths(B: int, S: int, seed: int, stream: int = STREAM_MASK) -> np.ndarray:
    lib = _load()
    m = np.empty((B, S), np.uint8)
    L = np.empty(B, np.int64)
    lib.mcc1d_gen_mask_prefix(m.ctypes.data, B, S, seed, stream, L.ctypes.data)
    return L


def generate(wl, seed: int = 0, *, alloc=None, nthreads: int = 0) -> dict:
    """Inputs of a workload (a ``Workload`` or a name in ``WORKLOADS``).

    Returns ``{"x", "gy", "w", "mask"}``: uint16 bit patterns [S,B,H] /
    [S,B,H] / [W,H] and uint8 [B,S] (None for mask = nullptr). ``alloc``,
    if given, is ``alloc(shape, numpy_dtype)`` returning a C-contiguous host
    buffer (numpy array or CPU torch tensor) to write into."""
    if isinstance(wl, str):
        wl = WORKLOADS[wl]
    if alloc is None:
        alloc = lambda shape, dt: np.empty(shape, dt)  # noqa: E731
    x = alloc((wl.S, wl.B, wl.H), np.uint16)
    gy = alloc((wl.S, wl.B, wl.H), np.uint16)
    w = alloc((wl.W, wl.H), np.uint16)
    fill_values(x, wl.x, wl.dtype, seed, STREAM_X, nthreads)
    fill_values(gy, wl.gy, wl.dtype, seed, STREAM_GY, nthreads)
    fill_values(w, wl.w, wl.dtype, seed, STREAM_W, nthreads)
    mask = None
    if wl.mask[0] != "none":
        mask = alloc((wl.B, wl.S), np.uint8)
        fill_mask(mask, wl.mask, wl.B, wl.S, seed)
    return {"x": x, "gy": gy, "w": w, "mask": mask}
