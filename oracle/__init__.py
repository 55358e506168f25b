"""CPU oracle for the masked causal depthwise conv1d backward (fp64, plain C).

TEST INFRASTRUCTURE ONLY. The oracle is the slow, obviously correct statement
of what the operation computes (CANN page "aclnnMaskedCausalConv1dBackward",
section 功能说明 / 计算公式). Only the tests, the package smoke check and the
benchmark's CPU-baseline leg may import it; the GPU library never does, and
the two share no code.

All arrays are numpy: 16-bit tensors are passed as their raw bit patterns
(``np.uint16``), the mask as ``np.uint8`` (nonzero = keep) or ``None``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "mcc1d_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libmcc1d_oracle.so")

DTYPES = {"bf16": 0, "fp16": 1}


def compile_oracle(src: str, out: str) -> str:
    """Compile an oracle source file to a shared library with the host C compiler."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
                           "-o", tmp, src, "-lm"])
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle (if stale); returns the .so path."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(SOURCE)):
        return _LIB
    return compile_oracle(SOURCE, _LIB)


def _ptr(a):
    if a is None:
        return None
    if isinstance(a, np.ndarray):
        assert a.flags["C_CONTIGUOUS"]
        return a.ctypes.data
    return a.data_ptr()  # a CPU torch tensor


def _dt(dtype) -> int:
    return DTYPES[dtype] if isinstance(dtype, str) else int(dtype)


class Oracle:
    """The oracle's entry points bound to one compiled copy of the source."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        lib.mcc1d_oracle_to_double.argtypes = [ctypes.c_uint16, i32]
        lib.mcc1d_oracle_to_double.restype = ctypes.c_double
        lib.mcc1d_oracle_from_double.argtypes = [ctypes.c_double, i32]
        lib.mcc1d_oracle_from_double.restype = ctypes.c_uint16
        lib.mcc1d_oracle_threads.argtypes = [i32]
        lib.mcc1d_oracle_threads.restype = i32
        lib.mcc1d_oracle_bwd.argtypes = [i64, i64, i64, i64, i32, vp, vp, vp, vp,
                                         vp, vp, vp, vp, vp, i32]
        lib.mcc1d_oracle_bwd.restype = i32
        lib.mcc1d_oracle_gradx_at.argtypes = [i64, i64, i64, i64, i32, vp, vp, vp,
                                              i64, vp, vp, vp]
        lib.mcc1d_oracle_gradx_at.restype = i32
        lib.mcc1d_oracle_fwd.argtypes = [i64, i64, i64, i64, i32, vp, vp, vp, vp, vp, i32]
        lib.mcc1d_oracle_fwd.restype = i32
        self.lib = lib
        self.path = lib_path
        self._tables = {}

    def to_double(self, bits: int, dtype) -> float:
        return self.lib.mcc1d_oracle_to_double(int(bits), _dt(dtype))

    def from_double(self, v: float, dtype) -> int:
        return int(self.lib.mcc1d_oracle_from_double(float(v), _dt(dtype)))

    def decode(self, bits, dtype) -> np.ndarray:
        """Exact fp64 values of 16-bit patterns (the oracle's own decoder)."""
        dt = _dt(dtype)
        if dt not in self._tables:
            f = self.lib.mcc1d_oracle_to_double
            self._tables[dt] = np.array([f(b, dt) for b in range(65536)])
        return self._tables[dt][np.asarray(bits, dtype=np.uint16)]

    def encode(self, values, dtype) -> np.ndarray:
        """Round fp64 values once to 16-bit patterns (the oracle's own rounding)."""
        f, dt = self.lib.mcc1d_oracle_from_double, _dt(dtype)
        v = np.asarray(values, dtype=np.float64)
        return np.array([f(float(a), dt) for a in v.ravel()], np.uint16).reshape(v.shape)

    def threads(self, nthreads: int = 0) -> int:
        return int(self.lib.mcc1d_oracle_threads(nthreads))

    def bwd(self, S, B, H, W, dtype, gy, x, w, mask=None, *, want_gx=True,
            want_exact=False, nthreads: int = 0) -> dict:
        """Full backward. Returns ``gx`` (uint16 [S,B,H], if want_gx), ``gw``
        (uint16 [W,H]), ``gw_abs`` (fp64 [W,H], the sum of |terms|) and, with
        want_exact, ``gx_exact`` / ``gw_exact`` (fp64, before rounding)."""
        out = {"gw": np.empty((W, H), np.uint16), "gw_abs": np.empty((W, H), np.float64)}
        if want_gx:
            out["gx"] = np.empty((S, B, H), np.uint16)
        if want_exact:
            out["gw_exact"] = np.empty((W, H), np.float64)
            if want_gx:
                out["gx_exact"] = np.empty((S, B, H), np.float64)
        rc = self.lib.mcc1d_oracle_bwd(
            S, B, H, W, _dt(dtype), _ptr(gy), _ptr(x), _ptr(w), _ptr(mask),
            _ptr(out.get("gx")), _ptr(out.get("gx_exact")),
            _ptr(out["gw"]), _ptr(out.get("gw_exact")), _ptr(out["gw_abs"]), nthreads)
        if rc != 0:
            raise ValueError("oracle rejected its arguments")
        return out

    def gradx_at(self, S, B, H, W, dtype, gy, w, mask, idx):
        """gradX at flat positions ``idx`` of [S,B,H]; returns (bits, exact)."""
        idx = np.ascontiguousarray(idx, dtype=np.int64)
        bits = np.empty(idx.shape, np.uint16)
        exact = np.empty(idx.shape, np.float64)
        rc = self.lib.mcc1d_oracle_gradx_at(S, B, H, W, _dt(dtype), _ptr(gy), _ptr(w),
                                            _ptr(mask), idx.size, _ptr(idx), _ptr(bits),
                                            _ptr(exact))
        if rc != 0:
            raise ValueError("oracle rejected its arguments")
        return bits, exact

    def fwd(self, S, B, H, W, dtype, x, w, mask=None, *, nthreads: int = 0) -> np.ndarray:
        """The forward y = mask * causal depthwise conv(x, w), fp64 [S,B,H]."""
        y = np.empty((S, B, H), np.float64)
        rc = self.lib.mcc1d_oracle_fwd(S, B, H, W, _dt(dtype), _ptr(x), _ptr(w), _ptr(mask),
                                       _ptr(y), None, nthreads)
        if rc != 0:
            raise ValueError("oracle rejected its arguments")
        return y

    def fwd_bits(self, S, B, H, W, dtype, x, w, mask=None, *, nthreads: int = 0) -> np.ndarray:
        """The forward rounded once to the 16-bit type, uint16 [S,B,H]."""
        yb = np.empty((S, B, H), np.uint16)
        rc = self.lib.mcc1d_oracle_fwd(S, B, H, W, _dt(dtype), _ptr(x), _ptr(w), _ptr(mask),
                                       None, _ptr(yb), nthreads)
        if rc != 0:
            raise ValueError("oracle rejected its arguments")
        return yb


_lock = threading.Lock()
_default = None


def get() -> Oracle:
    """The oracle built from this directory's source."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
        return _default


def to_double(bits, dtype):
    return get().to_double(bits, dtype)


def from_double(v, dtype):
    return get().from_double(v, dtype)


def decode(bits, dtype):
    return get().decode(bits, dtype)


def encode(values, dtype):
    return get().encode(values, dtype)


def threads(nthreads: int = 0) -> int:
    return get().threads(nthreads)


def bwd(*a, **k):
    return get().bwd(*a, **k)


def gradx_at(*a, **k):
    return get().gradx_at(*a, **k)


def fwd(*a, **k):
    return get().fwd(*a, **k)


def fwd_bits(*a, **k):
    return get().fwd_bits(*a, **k)
