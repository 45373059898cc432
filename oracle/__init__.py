"""Reference oracle for the bf16 -> fp32 GEMM: TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (the CUDA library in
``tiled_gemm_codegen_gb300``) never imports it, and the two share no code.

Contents
--------
* ``gemm_f64`` / ``gemm_entries_f64`` - thin ctypes wrappers over the plain C
  fp64 triple loop in ``gemm_f64.c`` (the contraction C = sum_k A[:,k] B[k,:];
  LuisaCompute "Pipelines and stage boundaries", the k-tile example, and OCANNL
  "Module Ir.Schedule", Tensorize).
* ``layout`` - the TIRx layout calculus (TVM "Tensor Layout": TileLayout
  forward mapping, SwizzleLayout, bank/line of an element), used to pin the
  pages' worked tables and to check the library's shared-memory staging
  pattern on the host.

Parity status: every function here is pinned by ``tests/test_oracle.py`` and
``tests/test_layout.py``: brute force (exact rational sums of integer and of
random bf16 inputs, the latter within the textbook fp64 summation bound),
closed forms, invariants and planted mistakes for the GEMM, and the pages'
printed tables for the layout calculus.  The pages print no numeric GEMM
result, so no GEMM pin is a page value.
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_f64.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LOCK = threading.Lock()
_LIB = None


def library_path() -> str:
    return os.path.join(_BUILD_DIR, f"liboracle_gemm_{platform.machine()}.so")


def build(force: bool = False) -> str:
    """Compile ``gemm_f64.c`` with gcc (C99, OpenMP, no FMA contraction)."""
    out = library_path()
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    os.makedirs(_BUILD_DIR, exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c99", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-shared", "-fPIC", "-o", tmp, _SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _lib():
    global _LIB
    with _LOCK:
        if _LIB is None:
            lib = ctypes.CDLL(build())
            i64 = ctypes.c_int64
            vp = ctypes.c_void_p
            lib.oracle_gemm_f64.argtypes = [vp, vp, vp] + [i64] * 10
            lib.oracle_gemm_f64.restype = ctypes.c_int
            lib.oracle_gemm_entries_f64.argtypes = [vp, vp] + [i64] * 8 + [vp, vp, vp, i64, vp]
            lib.oracle_gemm_entries_f64.restype = ctypes.c_int
            lib.oracle_num_threads.argtypes = []
            lib.oracle_num_threads.restype = ctypes.c_int
            _LIB = lib
        return _LIB


def _u16(x) -> np.ndarray:
    """Accept a numpy uint16 array of bf16 bit patterns, or a torch bf16 tensor."""
    if isinstance(x, np.ndarray):
        if x.dtype != np.uint16:
            raise TypeError("oracle expects bf16 bit patterns as uint16")
        return np.ascontiguousarray(x)
    # torch tensor (bf16): reinterpret the bits without any arithmetic
    import torch  # local import: the oracle does not otherwise need torch

    if x.dtype != torch.bfloat16:
        raise TypeError("oracle expects a bf16 tensor")
    return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def num_threads() -> int:
    return int(_lib().oracle_num_threads())


def gemm_f64(A, B, M, N, K, lda=None, ldb=None, ldc=None, batch=1,
             strideA=None, strideB=None, strideC=None) -> np.ndarray:
    """Full product in fp64.  A, B: bf16 bit patterns (flat storage with the
    given element strides).  Returns C as a flat fp64 array of
    ``batch * strideC`` elements (``ldc``/``strideC`` default to dense)."""
    lda = K if lda is None else lda
    ldb = N if ldb is None else ldb
    ldc = N if ldc is None else ldc
    strideA = M * lda if strideA is None else strideA
    strideB = K * ldb if strideB is None else strideB
    strideC = M * ldc if strideC is None else strideC
    a = _u16(A).reshape(-1)
    b = _u16(B).reshape(-1)
    if batch > 0 and M > 0 and K > 0:
        need = (batch - 1) * strideA + (M - 1) * lda + K
        if a.size < need:
            raise ValueError(f"A has {a.size} elements, needs {need}")
    if batch > 0 and K > 0 and N > 0:
        need = (batch - 1) * strideB + (K - 1) * ldb + N
        if b.size < need:
            raise ValueError(f"B has {b.size} elements, needs {need}")
    c = np.zeros(max(batch * strideC, 1), dtype=np.float64)
    rc = _lib().oracle_gemm_f64(a.ctypes.data, b.ctypes.data, c.ctypes.data,
                                M, N, K, lda, ldb, ldc, batch, strideA, strideB, strideC)
    if rc != 0:
        raise ValueError("oracle_gemm_f64 rejected its arguments")
    return c[: batch * strideC]


def gemm_dense_f64(A, B) -> np.ndarray:
    """Convenience: A [batch?, M, K], B [batch?, K, N] dense (torch bf16 or
    uint16 numpy with shape).  Returns C [batch?, M, N] in fp64."""
    a = _u16(A)
    b = _u16(B)
    batched = a.ndim == 3
    if not batched:
        a = a[None]
        b = b[None]
    batch, M, K = a.shape
    _, K2, N = b.shape
    if K2 != K or b.shape[0] != batch:
        raise ValueError("shape mismatch")
    c = gemm_f64(a, b, M, N, K, batch=batch).reshape(batch, M, N)
    return c if batched else c[0]


def gemm_entries_f64(A, B, M, N, K, bi, ii, jj, lda=None, ldb=None, batch=1,
                     strideA=None, strideB=None) -> np.ndarray:
    """Selected entries C_b[i][j], each as one fp64 dot product (k ascending)."""
    lda = K if lda is None else lda
    ldb = N if ldb is None else ldb
    strideA = M * lda if strideA is None else strideA
    strideB = K * ldb if strideB is None else strideB
    a = _u16(A).reshape(-1)
    b = _u16(B).reshape(-1)
    bi = np.ascontiguousarray(bi, dtype=np.int64)
    ii = np.ascontiguousarray(ii, dtype=np.int64)
    jj = np.ascontiguousarray(jj, dtype=np.int64)
    if not (bi.shape == ii.shape == jj.shape):
        raise ValueError("index arrays differ in shape")
    out = np.zeros(bi.size, dtype=np.float64)
    rc = _lib().oracle_gemm_entries_f64(a.ctypes.data, b.ctypes.data, M, N, K, lda, ldb,
                                        batch, strideA, strideB, bi.ctypes.data,
                                        ii.ctypes.data, jj.ctypes.data, bi.size,
                                        out.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_gemm_entries_f64: index outside the problem")
    return out
