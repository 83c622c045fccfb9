"""Device-side drawing of the synthgen streams (bit-identical to the numpy functions).

Used by the benchmark and the GPU tests to make tensors of the large
workloads directly in device memory. ``tests/test_gpu_synth.py`` checks that
every function here equals its numpy counterpart on slices.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

from . import (TID_SE_W1, TID_SE_W2, TID_W1, TID_W2, TID_ROUTER, TID_X, TID_X_OUTLIER, Workload)
from .build import LIB_PATH

_lib = None


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built (synthgen.build.build())")
        lib = ctypes.CDLL(LIB_PATH)
        u64, f32, vp = ctypes.c_uint64, ctypes.c_float, ctypes.c_void_p
        lib.synth_normal_f32.argtypes = [u64, u64, u64, u64, f32, vp, vp]
        lib.synth_normal_f32.restype = ctypes.c_int
        lib.synth_normal_bf16.argtypes = [u64, u64, u64, ctypes.c_uint32, f32, u64, u64, f32, vp, vp]
        lib.synth_normal_bf16.restype = ctypes.c_int
        _lib = lib
    return _lib


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def normal_f32_(out: torch.Tensor, seed: int, tid: int, start: int, sigma: float) -> torch.Tensor:
    assert out.is_cuda and out.dtype == torch.float32 and out.is_contiguous()
    rc = _load().synth_normal_f32(seed, tid, start, out.numel(), float(np.float32(sigma)), out.data_ptr(), _stream())
    if rc != 0:
        raise RuntimeError(f"synth_normal_f32: cuda error {rc}")
    return out


def normal_bf16_(out: torch.Tensor, seed: int, tid: int, start: int, sigma: float, outlier_tid: int = 0,
                 outlier_p: float = 0.0, outlier_mult: float = 1.0) -> torch.Tensor:
    assert out.is_cuda and out.dtype == torch.bfloat16 and out.is_contiguous()
    thr = int(round(outlier_p * 2.0**32)) if outlier_p > 0 else 0
    rc = _load().synth_normal_bf16(seed, tid, outlier_tid, thr, float(np.float32(outlier_mult)), start, out.numel(),
                                   float(np.float32(sigma)), out.data_ptr(), _stream())
    if rc != 0:
        raise RuntimeError(f"synth_normal_bf16: cuda error {rc}")
    return out


def activations(wl: Workload, seed: int, T: int | None = None, out: torch.Tensor | None = None) -> torch.Tensor:
    T = wl.T if T is None else T
    if out is None:
        out = torch.empty(T, wl.H, dtype=torch.bfloat16, device="cuda")
    return normal_bf16_(out, seed, TID_X, 0, 1.0, TID_X_OUTLIER, wl.outlier_p, wl.outlier_mult)


def router(wl: Workload) -> torch.Tensor:
    out = torch.empty(wl.E, wl.H, dtype=torch.bfloat16, device="cuda")
    return normal_bf16_(out, wl.model_seed, TID_ROUTER, 0, wl.router_sigma)


def expert_w1(wl: Workload, e0: int, n: int, out: torch.Tensor | None = None) -> torch.Tensor:
    """W1 of experts [e0, e0+n) as fp32 [n, 2I, H] (gate rows first), same values as synthgen.expert_w1_f32."""
    per = 2 * wl.I_log * wl.H
    if out is None:
        out = torch.empty(n, 2 * wl.I_log, wl.H, dtype=torch.float32, device="cuda")
    return normal_f32_(out, wl.model_seed, TID_W1, e0 * per, wl.w_sigma)


def expert_w2(wl: Workload, e0: int, n: int, out: torch.Tensor | None = None) -> torch.Tensor:
    per = wl.H * wl.I_log
    if out is None:
        out = torch.empty(n, wl.H, wl.I_log, dtype=torch.float32, device="cuda")
    return normal_f32_(out, wl.model_seed, TID_W2, e0 * per, wl.w_sigma)


def shared_w1(wl: Workload) -> torch.Tensor:
    """W1 of the shared expert as fp32 [2 shared_I, H], same values as synthgen.shared_w1_f32."""
    out = torch.empty(2 * wl.shared_I, wl.H, dtype=torch.float32, device="cuda")
    return normal_f32_(out, wl.model_seed, TID_SE_W1, 0, wl.w_sigma)


def shared_w2(wl: Workload) -> torch.Tensor:
    out = torch.empty(wl.H, wl.shared_I, dtype=torch.float32, device="cuda")
    return normal_f32_(out, wl.model_seed, TID_SE_W2, 0, wl.w_sigma)
