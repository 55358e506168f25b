"""Masked causal depthwise conv1d backward (and forward) for NVIDIA GB300.

Thin ctypes binding over ``libmcc1d.so`` (see ``include/mcc1d.h``). The names
mirror the C ABI; the binding only marshals arguments. Every step of the
computation runs in the library's CUDA kernels: there is no CPU or PyTorch
fallback, and a missing library is an error.

Torch tensors may be passed for device buffers; their ``data_ptr()`` is
handed to the C ABI, and torch is used for nothing else. ``backward`` is a
convenience wrapper that allocates outputs and workspace with torch.
"""
from __future__ import annotations

from ._lib import (  # noqa: F401
    BF16, FP16, Mcc1dError, STATUS, backward, dtype_code, lib_path, load,
    mcc1d_bwd, mcc1d_bwd_device_status, mcc1d_bwd_noalloc, NOALLOC_SCRATCH_BYTES, mcc1d_bwd_workspace_size, mcc1d_status_string,
    mcc1d_version, Mcc1dTensors, tensors, mcc1d_bwd_ex, mcc1d_bwd_ex_workspace_size,
    mcc1d_fwd, forward, mcc1d_bwd_host, mcc1d_plan_describe, PLAN_BWD, PLAN_BWD_EX, PLAN_FWD,
    mcc1d_selftest_wait, Mcc1dFwdTensors, fwd_tensors, mcc1d_fwd_ex, mcc1d_fwd_ex_workspace_size,
    PLAN_SMS, mcc1d_check_sm_count, mcc1d_device_sm_count,
)
