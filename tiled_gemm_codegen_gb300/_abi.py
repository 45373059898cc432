"""ctypes declarations of the C ABI in ``include/tg_gemm.h`` (same names).

Argument marshalling only: every step of the GEMM runs in the CUDA library.
Loading fails loudly when the library has not been built - there is no
fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

TG_OK = 0
TG_ERR_INVALID_ARG = 1
TG_ERR_UNSUPPORTED = 2
TG_ERR_CUDA = 3
TG_ERR_OOM = 4
TG_ERR_TIMEOUT = 5
TG_ERR_DEVICE_CHECK = 6

STATUS_NAMES = {
    TG_OK: "TG_OK",
    TG_ERR_INVALID_ARG: "TG_ERR_INVALID_ARG",
    TG_ERR_UNSUPPORTED: "TG_ERR_UNSUPPORTED",
    TG_ERR_CUDA: "TG_ERR_CUDA",
    TG_ERR_OOM: "TG_ERR_OOM",
    TG_ERR_TIMEOUT: "TG_ERR_TIMEOUT",
    TG_ERR_DEVICE_CHECK: "TG_ERR_DEVICE_CHECK",
}


class tg_options(ctypes.Structure):
    _fields_ = [
        ("block_n", ctypes.c_int32),
        ("stages", ctypes.c_int32),
        ("split_k", ctypes.c_int32),
        ("force_pack", ctypes.c_int32),
        ("epilogue", ctypes.c_int32),
        ("max_ctas", ctypes.c_int32),
        ("timeout_ns", ctypes.c_uint64),
        ("debug_stall", ctypes.c_int32),
        ("cta_pair", ctypes.c_int32),
        ("stream_k", ctypes.c_int32),
        ("operands", ctypes.c_int32),
        ("trace_buffer", ctypes.c_uint64),
        ("a_col_major", ctypes.c_int32),
        ("b_col_major", ctypes.c_int32),
        ("direct", ctypes.c_int32),
    ]


class tg_plan_info(ctypes.Structure):
    _fields_ = [
        ("block_m", ctypes.c_int32),
        ("block_n", ctypes.c_int32),
        ("block_k", ctypes.c_int32),
        ("stages", ctypes.c_int32),
        ("tiles_m", ctypes.c_int32),
        ("tiles_n", ctypes.c_int32),
        ("k_blocks", ctypes.c_int32),
        ("split_k", ctypes.c_int32),
        ("num_units", ctypes.c_int64),
        ("grid", ctypes.c_int32),
        ("pack_a", ctypes.c_int32),
        ("pack_b", ctypes.c_int32),
        ("epilogue", ctypes.c_int32),
        ("smem_bytes", ctypes.c_int32),
        ("tmem_cols", ctypes.c_int32),
        ("workspace_bytes", ctypes.c_int64),
        ("cta_pair", ctypes.c_int32),
        ("stream_k", ctypes.c_int32),
        ("sk_tiles", ctypes.c_int32),
        ("direct", ctypes.c_int32),
        ("reserved", ctypes.c_int32 * 2),
    ]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_ if name != "reserved"}


class tg_epilogue(ctypes.Structure):
    _fields_ = [
        ("alpha", ctypes.c_float),
        ("beta", ctypes.c_float),
        ("bias", ctypes.c_void_p),
        ("bias_stride", ctypes.c_int64),
        ("residual", ctypes.c_void_p),
        ("ldr", ctypes.c_int64),
        ("strideR", ctypes.c_int64),
        ("activation", ctypes.c_int32),
        ("out_type", ctypes.c_int32),
        ("reserved", ctypes.c_int32 * 6),
    ]


TG_ACT_NONE, TG_ACT_RELU, TG_ACT_GELU_TANH, TG_ACT_SILU = 0, 1, 2, 3
TG_F32, TG_BF16 = 0, 1
TG_FP8_E4M3, TG_FP8_E5M2 = 0, 1

_i64 = ctypes.c_int64
_vp = ctypes.c_void_p
_GEMM_ARGS = [_vp, _vp, _vp] + [_i64] * 10 + [_vp]

SIGNATURES = {
    "tg_gemm": (_GEMM_ARGS, ctypes.c_int),
    "tg_gemm_ex": (_GEMM_ARGS + [ctypes.POINTER(tg_options)], ctypes.c_int),
    "tg_gemm_host": (_GEMM_ARGS + [ctypes.POINTER(tg_options)], ctypes.c_int),
    "tg_plan": ([_vp, _vp, _vp] + [_i64] * 10 + [ctypes.c_int32, ctypes.POINTER(tg_options),
                                                   ctypes.POINTER(tg_plan_info)], ctypes.c_int),
    "tg_gemm_fused": ([_vp, _vp, _vp] + [_i64] * 10 + [ctypes.POINTER(tg_epilogue), _vp,
                                                         ctypes.POINTER(tg_options)], ctypes.c_int),
    "tg_gemm_splitk_static": ([_vp, _vp, _vp] + [_i64] * 10 + [ctypes.c_int32, _vp], ctypes.c_int),
    "tg_tune": (_GEMM_ARGS + [ctypes.POINTER(tg_options), ctypes.c_int32, ctypes.POINTER(tg_options),
                              ctypes.POINTER(ctypes.c_float)], ctypes.c_int),
    "tg_gemm_fp8": ([_vp, _vp, _vp] + [_i64] * 10 + [ctypes.c_int32, ctypes.c_int32,
                                                       ctypes.POINTER(tg_epilogue), _vp,
                                                       ctypes.POINTER(tg_options)], ctypes.c_int),
    "tg_gemm_mxfp8": ([_vp, _vp, _vp] + [_i64] * 10 + [ctypes.c_int32, ctypes.c_int32,
                                                         _vp, _i64, _i64, _vp, _i64, _i64,
                                                         ctypes.POINTER(tg_epilogue), _vp,
                                                         ctypes.POINTER(tg_options)], ctypes.c_int),
    "tg_gemm_mxfp4": ([_vp, _vp, _vp] + [_i64] * 10 + [_vp, _i64, _i64, _vp, _i64, _i64,
                                                         ctypes.POINTER(tg_epilogue), _vp,
                                                         ctypes.POINTER(tg_options)], ctypes.c_int),
    "tg_device_error": ([_vp], ctypes.c_int),
    "tg_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "tg_shutdown": ([], None),
}

_LOCK = threading.Lock()
_LIB = None
_LIB_CHECKS = None


def library_path() -> str:
    return _build.library_path()


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    for name, (args, res) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


def load_checks() -> ctypes.CDLL:
    """The TG_DEBUG_CHECKS build of the library (a separate handle with the
    same entry points), built on first use."""
    global _LIB_CHECKS
    with _LOCK:
        if _LIB_CHECKS is None:
            _LIB_CHECKS = _declare(ctypes.CDLL(_build.build(checks=True)))
        return _LIB_CHECKS


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """The loaded library.  Raises if it was never built (no fallback)."""
    global _LIB
    with _LOCK:
        if _LIB is not None:
            return _LIB
        path = library_path()
        if not os.path.exists(path):
            if not build_if_missing:
                raise RuntimeError(
                    f"tiled_gemm_codegen_gb300: CUDA library not built ({path} missing); "
                    "run tiled_gemm_codegen_gb300.build.build() first")
            _build.build()
        _LIB = _declare(ctypes.CDLL(path))
        return _LIB
