"""ctypes binding of libmcc1d.so: argument marshalling only."""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

BF16, FP16 = 0, 1
STATUS = {
    0: "MCC1D_OK",
    161001: "MCC1D_ERR_PARAM_NULLPTR",
    161002: "MCC1D_ERR_PARAM_INVALID",
    561002: "MCC1D_ERR_INNER_TILING_ERROR",
    561003: "MCC1D_ERR_WORKSPACE",
    561100: "MCC1D_ERR_CUDA",
    561101: "MCC1D_ERR_DEVICE_TIMEOUT",
    561102: "MCC1D_ERR_DEVICE",
}
PLAN_SMS = 152

_lock = threading.Lock()
_lib = None


class Mcc1dTensors(ctypes.Structure):
    """Mirror of ``mcc1d_tensors``: pointers plus strides (elements; the
    mask's in bytes), outermost dimension first."""
    _fields_ = [("gradY", ctypes.c_void_p), ("gradY_strides", ctypes.c_int64 * 3),
                ("x", ctypes.c_void_p), ("x_strides", ctypes.c_int64 * 3),
                ("weight", ctypes.c_void_p), ("weight_strides", ctypes.c_int64 * 2),
                ("mask", ctypes.c_void_p), ("mask_strides", ctypes.c_int64 * 2),
                ("gradX", ctypes.c_void_p), ("gradWeight", ctypes.c_void_p)]


class Mcc1dFwdTensors(ctypes.Structure):
    """Mirror of ``mcc1d_fwd_tensors`` (the forward's strided inputs)."""
    _fields_ = [("x", ctypes.c_void_p), ("x_strides", ctypes.c_int64 * 3),
                ("weight", ctypes.c_void_p), ("weight_strides", ctypes.c_int64 * 2),
                ("mask", ctypes.c_void_p), ("mask_strides", ctypes.c_int64 * 2),
                ("y", ctypes.c_void_p)]


class Mcc1dError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {STATUS.get(self.status, 'unknown')} ({self.status})")


def lib_path() -> str:
    return _build.LIB


def load():
    """Load libmcc1d.so (it must have been built: ``__graft_entry__.build()``
    or ``python -m causal_conv_backward_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_build.LIB):
            raise RuntimeError(f"libmcc1d.so is not built ({_build.LIB}); "
                               "run causal_conv_backward_gb300.build.build() first")
        lib = ctypes.CDLL(_build.LIB)
        i64, i32, u64, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_uint64, ctypes.c_void_p
        lib.mcc1d_bwd_workspace_size.argtypes = [i64, i64, i64, i64, i32, i32, ctypes.POINTER(u64)]
        lib.mcc1d_bwd_workspace_size.restype = i32
        lib.mcc1d_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i32, u64]
        lib.mcc1d_bwd.restype = i32
        lib.mcc1d_bwd_ex_workspace_size.argtypes = [ctypes.POINTER(Mcc1dTensors), i64, i64, i64, i64,
                                                    i32, ctypes.POINTER(u64)]
        lib.mcc1d_bwd_ex_workspace_size.restype = i32
        lib.mcc1d_bwd_ex.argtypes = [ctypes.POINTER(Mcc1dTensors), i64, i64, i64, i64, i32, vp, u64, vp]
        lib.mcc1d_bwd_ex.restype = i32
        lib.mcc1d_bwd_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i32, u64]
        lib.mcc1d_bwd_host.restype = i32
        lib.mcc1d_fwd.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i32, vp]
        lib.mcc1d_fwd.restype = i32
        lib.mcc1d_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i32]
        lib.mcc1d_bwd_noalloc.restype = i32
        lib.mcc1d_bwd_device_status.argtypes = [vp, vp, ctypes.POINTER(i32)]
        lib.mcc1d_bwd_device_status.restype = i32
        lib.mcc1d_status_string.argtypes = [i32]
        lib.mcc1d_status_string.restype = ctypes.c_char_p
        lib.mcc1d_version.argtypes = []
        lib.mcc1d_version.restype = i32
        lib.mcc1d_plan_describe.argtypes = [i64, i64, i64, i64, i32, i32, ctypes.c_char_p, u64,
                                            ctypes.POINTER(u64)]
        lib.mcc1d_plan_describe.restype = i32
        lib.mcc1d_fwd_ex_workspace_size.argtypes = [ctypes.POINTER(Mcc1dFwdTensors), i64, i64, i64, i64,
                                                    i32, ctypes.POINTER(u64)]
        lib.mcc1d_fwd_ex_workspace_size.restype = i32
        lib.mcc1d_fwd_ex.argtypes = [ctypes.POINTER(Mcc1dFwdTensors), i64, i64, i64, i64, i32, vp, u64, vp, vp]
        lib.mcc1d_fwd_ex.restype = i32
        lib.mcc1d_check_sm_count.argtypes = [i32]
        lib.mcc1d_check_sm_count.restype = i32
        lib.mcc1d_device_sm_count.argtypes = [ctypes.POINTER(i32)]
        lib.mcc1d_device_sm_count.restype = i32
        lib.mcc1d_selftest_wait.argtypes = [vp, i32, vp]
        lib.mcc1d_selftest_wait.restype = i32
        _lib = lib
        return lib


def _ptr(a):
    if a is None:
        return None
    if isinstance(a, int):
        return a
    return a.data_ptr()


def dtype_code(dtype) -> int:
    if isinstance(dtype, int):
        return dtype
    name = str(dtype).replace("torch.", "")
    return {"bf16": BF16, "bfloat16": BF16, "fp16": FP16, "float16": FP16, "half": FP16}[name]


def mcc1d_bwd_workspace_size(S, B, H, W, dtype, has_mask) -> int:
    out = ctypes.c_uint64(0)
    st = load().mcc1d_bwd_workspace_size(S, B, H, W, dtype_code(dtype), int(bool(has_mask)),
                                         ctypes.byref(out))
    if st != 0:
        raise Mcc1dError(st, "mcc1d_bwd_workspace_size")
    return int(out.value)


def mcc1d_bwd(gradY, x, weight, mask_or_null, gradX, gradWeight, workspace, stream,
              S, B, H, W, dtype, workspace_bytes) -> None:
    """Enqueue the backward; buffers are device pointers (ints) or tensors,
    ``stream`` a cudaStream_t as int (0 = legacy default) or a torch stream."""
    if stream is not None and not isinstance(stream, int):
        stream = stream.cuda_stream
    st = load().mcc1d_bwd(_ptr(gradY), _ptr(x), _ptr(weight), _ptr(mask_or_null), _ptr(gradX),
                          _ptr(gradWeight), _ptr(workspace), stream or None, S, B, H, W,
                          dtype_code(dtype), int(workspace_bytes))
    if st != 0:
        raise Mcc1dError(st, "mcc1d_bwd")


def tensors(gradY, x, weight, mask, gradX, gradWeight) -> Mcc1dTensors:
    """Descriptor of torch tensors (their data pointers and element strides).
    It holds raw pointers only: keep the tensors (and any view's base) alive
    until the work enqueued with it has completed."""
    t = Mcc1dTensors()
    t.gradY, t.x, t.weight = gradY.data_ptr(), x.data_ptr(), weight.data_ptr()
    t.gradY_strides[:] = list(gradY.stride())
    t.x_strides[:] = list(x.stride())
    t.weight_strides[:] = list(weight.stride())
    if mask is not None:
        t.mask = mask.data_ptr()
        t.mask_strides[:] = [st * mask.element_size() for st in mask.stride()]
    t.gradX, t.gradWeight = gradX.data_ptr(), gradWeight.data_ptr()
    return t


def fwd_tensors(x, weight, mask, y) -> Mcc1dFwdTensors:
    """Forward descriptor of torch tensors (data pointers and element strides).
    It holds raw pointers only: keep the tensors (and any view's base) alive
    until the work enqueued with it has completed."""
    t = Mcc1dFwdTensors()
    t.x, t.weight, t.y = x.data_ptr(), weight.data_ptr(), y.data_ptr()
    t.x_strides[:] = list(x.stride())
    t.weight_strides[:] = list(weight.stride())
    if mask is not None:
        t.mask = mask.data_ptr()
        t.mask_strides[:] = [st * mask.element_size() for st in mask.stride()]
    return t


def mcc1d_fwd_ex_workspace_size(t: Mcc1dFwdTensors, S, B, H, W, dtype) -> int:
    v = ctypes.c_uint64(0)
    st = load().mcc1d_fwd_ex_workspace_size(ctypes.byref(t), S, B, H, W, dtype_code(dtype), ctypes.byref(v))
    if st != 0:
        raise Mcc1dError(st, "mcc1d_fwd_ex_workspace_size")
    return int(v.value)


def mcc1d_fwd_ex(t: Mcc1dFwdTensors, S, B, H, W, dtype, workspace, workspace_bytes, stream,
                 device_status=None) -> None:
    """Enqueue the forward on strided tensors described by ``t``."""
    if stream is not None and not isinstance(stream, int):
        stream = stream.cuda_stream
    st = load().mcc1d_fwd_ex(ctypes.byref(t), S, B, H, W, dtype_code(dtype), _ptr(workspace),
                             int(workspace_bytes), stream or None, _ptr(device_status))
    if st != 0:
        raise Mcc1dError(st, "mcc1d_fwd_ex")


def mcc1d_bwd_ex_workspace_size(t: Mcc1dTensors, S, B, H, W, dtype) -> int:
    out = ctypes.c_uint64(0)
    st = load().mcc1d_bwd_ex_workspace_size(ctypes.byref(t), S, B, H, W, dtype_code(dtype),
                                            ctypes.byref(out))
    if st != 0:
        raise Mcc1dError(st, "mcc1d_bwd_ex_workspace_size")
    return int(out.value)


def mcc1d_bwd_ex(t: Mcc1dTensors, S, B, H, W, dtype, workspace, workspace_bytes, stream) -> None:
    """Enqueue the backward on strided tensors described by ``t``."""
    if stream is not None and not isinstance(stream, int):
        stream = stream.cuda_stream
    st = load().mcc1d_bwd_ex(ctypes.byref(t), S, B, H, W, dtype_code(dtype), _ptr(workspace),
                             int(workspace_bytes), stream or None)
    if st != 0:
        raise Mcc1dError(st, "mcc1d_bwd_ex")


def mcc1d_bwd_host(gradY, x, weight, mask_or_null, gradX, gradWeight, workspace, stream,
                   S, B, H, W, dtype, workspace_bytes) -> None:
    """Enqueue the backward on tensors that may be page-locked host buffers
    (e.g. torch tensors made with pin_memory=True); workspace on the device."""
    if stream is not None and not isinstance(stream, int):
        stream = stream.cuda_stream
    st = load().mcc1d_bwd_host(_ptr(gradY), _ptr(x), _ptr(weight), _ptr(mask_or_null), _ptr(gradX),
                               _ptr(gradWeight), _ptr(workspace), stream or None, S, B, H, W,
                               dtype_code(dtype), int(workspace_bytes))
    if st != 0:
        raise Mcc1dError(st, "mcc1d_bwd_host")


def mcc1d_fwd(x, weight, mask_or_null, y, stream, S, B, H, W, dtype, device_status=None) -> None:
    """Enqueue the forward y = mask * causal depthwise conv(x, weight)."""
    if stream is not None and not isinstance(stream, int):
        stream = stream.cuda_stream
    st = load().mcc1d_fwd(_ptr(x), _ptr(weight), _ptr(mask_or_null), _ptr(y), stream or None,
                          S, B, H, W, dtype_code(dtype), _ptr(device_status))
    if st != 0:
        raise Mcc1dError(st, "mcc1d_fwd")


def forward(x, weight, mask=None, *, y=None, stream=None):
    """Convenience forward on torch CUDA tensors x [S,B,H], weight [W,H]
    (1 <= W <= 8), mask [B,S] or None; inputs may be strided views (they go
    through mcc1d_fwd_ex). Returns y (dense; allocated when not given)."""
    import torch
    S, B, H = x.shape
    W = weight.shape[0]
    if mask is not None and mask.dtype == torch.bool:
        mask = mask.view(torch.uint8)
    if y is None:
        y = torch.empty((S, B, H), dtype=x.dtype, device=x.device)
    if stream is None:
        stream = torch.cuda.current_stream(x.device)
    dense = x.is_contiguous() and weight.is_contiguous() and (mask is None or mask.is_contiguous())
    if dense:
        mcc1d_fwd(x, weight, mask, y, stream, S, B, H, W, dtype_code(x.dtype))
    else:
        t = fwd_tensors(x, weight, mask, y)
        nb = mcc1d_fwd_ex_workspace_size(t, S, B, H, W, x.dtype)
        ws = torch.empty(max(nb, 1), dtype=torch.uint8, device=x.device)
        if isinstance(stream, torch.cuda.Stream):
            ws.record_stream(stream)   # not reused before the call has run on `stream`
        mcc1d_fwd_ex(t, S, B, H, W, x.dtype, ws, nb, stream)
    return y


def mcc1d_bwd_noalloc(gradY, x, weight, mask_or_null, gradX, gradWeight, stream,
                      S, B, H, W, dtype) -> None:
    """Enqueue the backward with the library's fixed scratch array instead of a
    workspace (for callers that cannot allocate device memory)."""
    if stream is not None and not isinstance(stream, int):
        stream = stream.cuda_stream
    st = load().mcc1d_bwd_noalloc(_ptr(gradY), _ptr(x), _ptr(weight), _ptr(mask_or_null),
                                  _ptr(gradX), _ptr(gradWeight), stream or None, S, B, H, W,
                                  dtype_code(dtype))
    if st != 0:
        raise Mcc1dError(st, "mcc1d_bwd_noalloc")


NOALLOC_SCRATCH_BYTES = 8 * 1024 * 1024


def mcc1d_bwd_device_status(workspace, stream=None) -> int:
    if stream is not None and not isinstance(stream, int):
        stream = stream.cuda_stream
    out = ctypes.c_int32(-1)
    st = load().mcc1d_bwd_device_status(_ptr(workspace), stream or None, ctypes.byref(out))
    if st != 0:
        raise Mcc1dError(st, "mcc1d_bwd_device_status")
    return int(out.value)


def mcc1d_check_sm_count(sm_count: int) -> int:
    """The status every launching call returns for a device with this many
    SMs (MCC1D_OK, or MCC1D_ERR_DEVICE below the plans' 152)."""
    return int(load().mcc1d_check_sm_count(int(sm_count)))


def mcc1d_device_sm_count() -> int:
    """SM count of the current device, as the library reads it."""
    out = ctypes.c_int32(0)
    st = load().mcc1d_device_sm_count(ctypes.byref(out))
    if st != 0:
        raise Mcc1dError(st, "mcc1d_device_sm_count")
    return int(out.value)


def mcc1d_status_string(status: int) -> str:
    return load().mcc1d_status_string(int(status)).decode()


def mcc1d_version() -> int:
    return int(load().mcc1d_version())


def mcc1d_selftest_wait(device_status, arrive: bool, stream=None) -> None:
    """Enqueue the bounded-wait self-test; ``device_status`` is an int32 device
    word (a tensor or pointer) that receives MCC1D_OK or
    MCC1D_ERR_DEVICE_TIMEOUT."""
    if stream is not None and not isinstance(stream, int):
        stream = stream.cuda_stream
    st = load().mcc1d_selftest_wait(_ptr(device_status), 1 if arrive else 0, stream or None)
    if st != 0:
        raise Mcc1dError(st, "mcc1d_selftest_wait")


PLAN_BWD, PLAN_BWD_EX, PLAN_FWD = 0, 1, 2


def mcc1d_plan_describe(S, B, H, W, dtype, kind=PLAN_BWD) -> dict:
    """The execution plan the library would use for a shape, as a dict
    (per-H-block ranges ``c_lo``, ``c_hi``, ``slot_base`` as lists)."""
    lib = load()
    need = ctypes.c_uint64(0)
    st = lib.mcc1d_plan_describe(S, B, H, W, dtype_code(dtype), kind, None, 0, ctypes.byref(need))
    if st != 0:
        raise Mcc1dError(st, "mcc1d_plan_describe")
    buf = ctypes.create_string_buffer(need.value)
    lib.mcc1d_plan_describe(S, B, H, W, dtype_code(dtype), kind, buf, need.value, None)
    out = {}
    for line in buf.value.decode().splitlines():
        k, v = line.split("=", 1)
        out[k] = [int(a) for a in v.split(",")] if k in ("c_lo", "c_hi", "slot_base") else int(v)
    return out


def backward(gradY, x, weight, mask=None, *, gradX=None, gradWeight=None, workspace=None,
             stream=None):
    """Convenience call on torch CUDA tensors: gradY, x [S,B,H], weight [W,H]
    (bf16 or fp16; W = 3 on the dense call, 1..8 through the strided one),
    mask [B,S] bool/uint8 or None; inputs may be strided views. Allocates whatever output or workspace is not given (with torch)
    and returns (gradX, gradWeight)."""
    import torch

    S, B, H = gradY.shape
    W = weight.shape[0]
    code = dtype_code(gradY.dtype)
    for t in (gradY, x, weight):
        if not t.is_cuda:
            raise ValueError("gradY, x and weight must be CUDA tensors")
    if mask is not None and mask.dtype == torch.bool:
        mask = mask.view(torch.uint8)
    if gradX is None:
        gradX = torch.empty((S, B, H), dtype=gradY.dtype, device=gradY.device)
    if gradWeight is None:
        gradWeight = torch.empty((W, H), dtype=weight.dtype, device=weight.device)
    if stream is None:
        stream = torch.cuda.current_stream(gradY.device)
    dense = (W == 3 and all(t.is_contiguous() for t in (gradY, x, weight))
             and (mask is None or mask.is_contiguous()))
    if dense:
        nbytes = mcc1d_bwd_workspace_size(S, B, H, W, code, mask is not None)
    else:
        desc = tensors(gradY, x, weight, mask, gradX, gradWeight)
        nbytes = mcc1d_bwd_ex_workspace_size(desc, S, B, H, W, code)
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=gradY.device)
        if isinstance(stream, torch.cuda.Stream):
            workspace.record_stream(stream)   # not reused before the call has run on `stream`
    wsb = workspace.numel() * workspace.element_size()
    if dense:
        mcc1d_bwd(gradY, x, weight, mask, gradX, gradWeight, workspace, stream, S, B, H, W, code, wsb)
    else:
        mcc1d_bwd_ex(desc, S, B, H, W, code, workspace, wsb, stream)
    return gradX, gradWeight
