"""ctypes view of liblp.so (the C ABI declared in include/lp.h).

Loading is explicit and loud: if the library has not been built, ``load()``
raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os
import threading

from .build import LIB

c_i64, c_i32, c_u64, c_f32, c_vp = (ctypes.c_int64, ctypes.c_int32, ctypes.c_uint64,
                                    ctypes.c_float, ctypes.c_void_p)

LP_F32, LP_F16, LP_BF16 = 0, 1, 2
LP_OK, LP_ERR_INVALID_ARGUMENT, LP_ERR_UNSUPPORTED_DTYPE, LP_ERR_CUDA, LP_ERR_TOO_LARGE = range(5)

EXPORTS = ("lp_apply_token_bitmask", "lp_apply_token_bitmask_rows", "lp_apply_packed_bitmask",
           "lp_upload_bitmask",
           "lp_sample",
           "lp_mask_and_sample", "lp_mask_and_sample_slots", "lp_sample_workspace_bytes",
           "lp_mask_and_sample_noalloc",
           "lp_philox4x32_10", "lp_status_string")


class SamplingParams(ctypes.Structure):
    """lp_sampling_params: each array is a device pointer to B values or NULL."""

    _fields_ = [("temperature", c_vp), ("temperature_scalar", c_f32),
                ("top_k", c_vp), ("top_k_scalar", c_i32),
                ("top_p", c_vp), ("top_p_scalar", c_f32),
                ("min_p", c_vp), ("min_p_scalar", c_f32),
                ("seed", c_u64), ("offset", c_u64)]


class LPError(RuntimeError):
    def __init__(self, fn: str, status: int, message: str):
        super().__init__(f"{fn}: {message} (status {status})")
        self.status = status


_lib = None
_lock = threading.Lock()


def declare(lib) -> None:
    """Set the argument and result types of every exported entry point."""
    lib.lp_apply_token_bitmask.restype = c_i32
    lib.lp_apply_token_bitmask.argtypes = [c_vp, c_i32, c_i64, c_i64, c_i64, c_vp, c_i64, c_i64,
                                           c_i64, c_i64, c_vp, c_i64, c_vp]
    lib.lp_apply_token_bitmask_rows.restype = c_i32
    lib.lp_apply_token_bitmask_rows.argtypes = [c_vp, c_i32, c_i64, c_i64, c_i64, c_vp, c_i64,
                                                c_i64, c_i64, c_i64, c_vp, c_vp, c_vp]
    lib.lp_upload_bitmask.restype = c_i32
    lib.lp_upload_bitmask.argtypes = [c_vp, c_i64, c_vp, c_i64, c_i64, c_i64, c_vp, c_vp, c_vp,
                                      c_vp]
    lib.lp_apply_packed_bitmask.restype = c_i32
    lib.lp_apply_packed_bitmask.argtypes = [c_vp, c_i64, c_vp, c_i32, c_i64, c_i64, c_i64, c_vp,
                                            c_i64, c_i64, c_i64, c_f32, c_i64, c_vp, c_i64, c_vp]
    lib.lp_sample.restype = c_i32
    lib.lp_sample.argtypes = [c_vp, c_i32, c_i64, c_i64, c_i64, ctypes.POINTER(SamplingParams),
                              c_vp, c_vp, c_i64, c_vp]
    lib.lp_mask_and_sample.restype = c_i32
    lib.lp_mask_and_sample.argtypes = [c_vp, c_i32, c_i64, c_i64, c_i64, c_vp, c_i64, c_i64,
                                       c_i64, c_i64, c_vp, c_i64, ctypes.POINTER(SamplingParams),
                                       c_vp, c_vp, c_i64, c_vp]
    lib.lp_mask_and_sample_slots.restype = c_i32
    lib.lp_mask_and_sample_slots.argtypes = [c_vp, c_i32, c_i64, c_i64, c_i64, c_vp, c_i64,
                                             c_i64, c_i64, c_i64, c_vp, c_i64,
                                             ctypes.POINTER(SamplingParams), c_i64, c_vp, c_vp,
                                             c_vp, c_i64, c_vp]
    lib.lp_mask_and_sample_noalloc.restype = c_i32
    lib.lp_mask_and_sample_noalloc.argtypes = [c_vp, c_i32, c_i64, c_i64, c_i64, c_vp, c_i64,
                                               c_i64, c_i64, c_i64, c_vp, c_i64,
                                               ctypes.POINTER(SamplingParams), c_vp, c_vp]
    lib.lp_sample_workspace_bytes.restype = c_i64
    lib.lp_sample_workspace_bytes.argtypes = [c_i32, c_i64, c_i64]
    lib.lp_philox4x32_10.restype = c_i32
    lib.lp_philox4x32_10.argtypes = [c_vp, c_vp, c_vp, c_i64, c_vp]
    lib.lp_status_string.restype = ctypes.c_char_p
    lib.lp_status_string.argtypes = [c_i32]


def load(path: str | None = None):
    """Open liblp.so once per process; raise if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or LIB
            if not os.path.exists(p):
                raise RuntimeError(
                    f"{p} is not built: run `python -m grammar_constrained_logit_gb300.build` "
                    "(or __graft_entry__.build()) first; there is no fallback path")
            lib = ctypes.CDLL(p)
            declare(lib)
            _lib = lib
    return _lib


def check(fn: str, status: int) -> None:
    if status != LP_OK:
        msg = load().lp_status_string(status).decode()
        raise LPError(fn, status, msg)
