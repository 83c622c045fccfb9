"""ctypes declarations of the libfp4moe C ABI (include/fp4moe.h).

Every exported symbol is declared here with its argument types. The binding
fails loudly when the library is missing: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfp4moe.so")

c_i32, c_u32, c_f32, c_sz, c_vp = ctypes.c_int32, ctypes.c_uint32, ctypes.c_float, ctypes.c_size_t, ctypes.c_void_p

OK, INVALID_ARG, MISALIGNED, CAPACITY, UNSUPPORTED, CUDA_ERROR = range(6)
ERR_TIMEOUT, ERR_EXPERT_ID, ERR_CAPACITY, ERR_NAN, ERR_SCALE_RANGE = 0x1, 0x2, 0x4, 0x8, 0x10
SAT_L1, SAT_L2 = 0x1, 0x2
W_NVFP4, W_MXFP4 = 0, 1


class Config(ctypes.Structure):
    _fields_ = [("hidden", c_i32), ("inter", c_i32), ("inter_logical", c_i32), ("num_experts", c_i32),
                ("top_k", c_i32), ("max_tokens", c_i32), ("swiglu_limit", c_f32), ("w_format", c_i32),
                ("ep_first", c_i32), ("ep_count", c_i32), ("shared_inter", c_i32)]


class SharedWeights(ctypes.Structure):
    """fp4moe_shared_weights: device pointers of the shared expert's block-FP8 weights."""
    _fields_ = [("w1", c_vp), ("w1_scales", c_vp), ("w2", c_vp), ("w2_scales", c_vp)]


CP = ctypes.POINTER(Config)
SWP = ctypes.POINTER(SharedWeights)

# name -> (restype, argtypes); pointers to device memory are passed as c_void_p
SIGNATURES = {
    "fp4moe_abi_version": (c_i32, []),
    "fp4moe_status_string": (ctypes.c_char_p, [c_i32]),
    "fp4moe_capacity_rows": (c_sz, [CP, c_i32]),
    "fp4moe_workspace_bytes": (c_sz, [CP]),
    "fp4moe_weight_bytes": (c_i32, [CP, ctypes.POINTER(c_sz), ctypes.POINTER(c_sz), ctypes.POINTER(c_sz),
                                    ctypes.POINTER(c_sz)]),
    "moe_route": (c_i32, [CP, c_i32] + [c_vp] * 13),
    "moe_route_noalloc": (c_i32, [CP, c_i32] + [c_vp] * 13),
    "moe_quantize_scatter": (c_i32, [CP, c_i32] + [c_vp] * 7),
    "moe_grouped_gemm_w1_swiglu": (c_i32, [CP, c_i32] + [c_vp] * 12),
    "moe_grouped_gemm_w2": (c_i32, [CP, c_i32] + [c_vp] * 10),
    "moe_combine": (c_i32, [CP, c_i32] + [c_vp] * 4),
    "moe_grouped_gemm_w2_combine": (c_i32, [CP, c_i32] + [c_vp] * 11),
    "moe_forward": (c_i32, [CP, c_i32] + [c_vp] * 16),
    "fp4moe_quantize_weights": (c_i32, [CP, c_i32, c_i32] + [c_vp] * 5),
    "fp4moe_mxfp4_as_nvfp4": (c_i32, [CP, c_i32, c_i32] + [c_vp] * 7),
    "fp4moe_tp_shard_units": (c_i32, [c_i32] * 6 + [ctypes.POINTER(c_i32)] * 3),
    "fp4moe_shard_mxfp4": (c_i32, [CP] + [c_i32] * 5 + [c_vp] * 5),
    "fp4moe_make_alpha": (c_i32, [c_i32] + [c_vp] * 4),
    "fp4moe_calibrate": (c_i32, [CP, c_i32] + [c_vp] * 10),
    "fp4moe_quantize_rows_f32": (c_i32, [c_i32, c_i32] + [c_vp] * 5),
    "fp4moe_tensor_peak_probe": (c_i32, [c_i32, c_i32, c_vp, c_vp]),
    "fp4moe_selftest_wait_timeout": (c_i32, [c_vp, ctypes.c_int64, c_vp, c_vp]),
    "fp4moe_batch_gs1": (c_i32, [CP, c_i32] + [c_vp] * 6),
    "fp4moe_read_error": (c_i32, [c_vp, ctypes.POINTER(c_u32), c_i32, c_vp]),
    "fp4moe_read_scale_status": (c_i32, [c_vp, ctypes.POINTER(c_u32), ctypes.POINTER(c_f32), c_i32, c_vp]),
    "fp4moe_refresh_gs2": (c_i32, [CP] + [c_vp] * 5),
    "fp4moe_shared_weight_bytes": (c_i32, [CP, ctypes.POINTER(c_sz), ctypes.POINTER(c_sz), ctypes.POINTER(c_sz),
                                           ctypes.POINTER(c_sz)]),
    "fp4moe_shared_quantize_weights": (c_i32, [CP, c_i32] + [c_vp] * 4),
    "moe_shared_expert": (c_i32, [CP, c_i32, c_vp, SWP, c_vp, c_vp, c_vp]),
    "moe_combine_shared": (c_i32, [CP, c_i32] + [c_vp] * 6),
    "moe_forward_shared": (c_i32, [CP, c_i32] + [c_vp] * 11 + [SWP] + [c_vp] * 5),
}

_lib = None


def load() -> ctypes.CDLL:
    """Load libfp4moe.so, declaring every signature. Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; "
                               "g.build()'` (no CPU fallback exists)")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib
