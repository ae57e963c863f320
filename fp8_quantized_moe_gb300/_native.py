"""ctypes loader for libmoefp8.so (the C ABI declared in include/moefp8.h).

The library is built in-tree by ``fp8_quantized_moe_gb300.build``.  Loading
never falls back to anything: if the shared library is missing or does not
load, the import of the op wrappers raises.
"""

from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

P = ctypes.c_void_p
i64 = ctypes.c_int64
i32 = ctypes.c_int
sz = ctypes.c_size_t

# name -> (argtypes, restype); restype i32 is a moe_status
SIGNATURES = {
    "moe_status_string": ([i32], ctypes.c_char_p),
    "moe_get_device_error": ([P, ctypes.POINTER(ctypes.c_int)], i32),
    "moe_num_sms": ([], i32),
    "moe_quantize_rows": ([P, i64, i64, i32, P, P, P, P], i32),
    "moe_quantize_weights": ([P, i64, i64, i64, i32, P, P, P, P], i32),
    "moe_ragged_sort_workspace_bytes": ([i64, i32, i32], sz),
    "moe_ragged_sort": ([P, i64, i32, i32, P, P, i64, i32, P, P, P, P, P, P, P, sz, P], i32),
    "moe_quantize_sort": ([P, P, i64, i32, i32, i64, i32, P, P, P, P, P, P, P, P, sz, P], i32),
    "gmm_fp8_ksplit": ([P, P, i32, P, P, i64, P, i32, i32, i32, i64, i64, i64, P, P], i32),
    "gmm_fp8": ([P, P, i32, P, P, i32, P, i32, i32, i32, i64, i64, i64, P, P], i32),
    "moe_swiglu_quant": ([P, i64, i64, i32, P, P, P, P], i32),
    "ragged_gather_reduce": ([P, P, P, i64, i32, i64, P, P], i32),
    "moe_gather_scale_quant": ([P, P, P, i64, i32, i64, P, P, P, P], i32),
    "moe_swiglu_bwd_quant": ([P, P, i64, i64, P, P, P, P], i32),
    "moe_quantize_group_cols": ([P, i64, i64, P, i32, i32, i32, P, P, P], i32),
    "tgmm_fp8_workspace_bytes": ([i64, i64, i64, i32], sz),
    "tgmm_fp8": ([P, P, i32, P, P, i32, P, i32, i32, i32, i64, i64, i64, P, P, sz, P], i32),
    "tgmm_fp8_gcq": ([P, P, i32, P, P, P, i32, i32, i32, i64, i64, i64, P, P, sz, P], i32),
    "moe_transpose_u8": ([P, i64, i64, i64, P, P], i32),
    "gmm_fp8_swiglu": ([P, P, i32, P, P, i32, P, i32, i32, i32, i64, i64, i64, i32, P, P, P, P, P, P], i32),
    "moe_ragged_sort_noalloc": ([P, i64, i32, i32, P, P, i64, i32, P, P, P, P, P, P, P], i32),
    "moe_router_topk": ([P, P, i64, i64, i32, i32, P, P, P, P], i32),
    "moe_test_stall_epilogue": ([ctypes.c_uint64], None),
    "moe_router_backward_workspace_bytes": ([i64, i64, i32], sz),
    "moe_router_backward": ([P, P, P, P, P, P, P, i64, i64, i32, i32, P, P, P, P, P, sz, P], i32),
    "moe_quantize_rows_mx": ([P, i64, i64, P, P, P], i32),
    "moe_quantize_sort_mx": ([P, P, i64, i32, i32, i64, P, P, P, P, P, P, P, sz, P], i32),
    "gmm_fp8_mx": ([P, P, P, P, P, i32, i32, i32, i64, i64, i64, P, P], i32),
    "gmm_fp8_mx_swiglu": ([P, P, P, P, P, i32, i32, i32, i64, i64, i64, P, P, P, P], i32),
    "moe_swiglu_quant_mx": ([P, i64, i64, P, P, P], i32),
    "moe_quantize_weights_int8": ([P, i64, i64, i64, i32, P, P, P, P], i32),
    "gmm_fp8_w8": ([P, P, i32, P, P, i32, P, i32, i32, i32, i64, i64, i64, P, P, sz, P], i32),
    "gmm_fp8_w8_workspace_bytes": ([i64, i64], sz),
}

_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load (building first if needed) and type the shared library."""
    global _lib
    with _lock:
        if _lib is None:
            if build_if_missing:
                _build.build()
            if not os.path.exists(_build.LIB):
                raise RuntimeError(f"libmoefp8.so not found at {_build.LIB}; run fp8_quantized_moe_gb300.build")
            L = ctypes.CDLL(_build.LIB)
            for name, (args, res) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = res
            _lib = L
    return _lib


class MoEError(RuntimeError):
    pass


def check(status: int, what: str) -> None:
    if status != 0:
        msg = load().moe_status_string(status).decode()
        raise MoEError(f"{what} failed: status {status} ({msg})")
