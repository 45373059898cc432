"""tiled_gemm_codegen_gb300 - a tiled bf16 -> fp32 GEMM for GB300 (sm_103a).

The product is the C-ABI CUDA library declared in ``include/tg_gemm.h``.
This package is its thin Python binding: the C functions under the same
names (``tg_gemm``, ``tg_gemm_ex``, ``tg_gemm_host``, ``tg_gemm_splitk_static``, ``tg_plan``,
``tg_gemm_fp8``, ``tg_gemm_mxfp8``, ``tg_gemm_mxfp4``, ``tg_tune``,
``tg_device_error``, ``tg_status_string``, ``tg_shutdown``) taking raw
pointers and sizes, plus conveniences that read pointers, shapes and
strides off torch tensors.  PyTorch only provides device memory and
streams; no arithmetic happens here.
"""
from __future__ import annotations

import ctypes

from ._abi import (TG_ACT_GELU_TANH, TG_ACT_NONE, TG_ACT_RELU, TG_ACT_SILU, TG_BF16, TG_ERR_CUDA,
                   TG_FP8_E4M3, TG_FP8_E5M2,
                   TG_ERR_DEVICE_CHECK, TG_ERR_INVALID_ARG, TG_ERR_OOM, TG_ERR_TIMEOUT, TG_ERR_UNSUPPORTED,
                   TG_F32, TG_OK, STATUS_NAMES, library_path, load, load_checks, tg_epilogue, tg_options,
                   tg_plan_info)

ACTIVATIONS = {"none": TG_ACT_NONE, "relu": TG_ACT_RELU, "gelu_tanh": TG_ACT_GELU_TANH,
               "silu": TG_ACT_SILU}

__all__ = [
    "TG_OK", "TG_ERR_INVALID_ARG", "TG_ERR_UNSUPPORTED", "TG_ERR_CUDA", "TG_ERR_OOM",
    "TG_ERR_TIMEOUT", "TG_ERR_DEVICE_CHECK", "TgError", "tg_options", "tg_plan_info", "load", "load_checks",
    "library_path",
    "tg_gemm", "tg_gemm_ex", "tg_gemm_host", "tg_gemm_fused", "tg_gemm_splitk_static", "tg_plan",
    "tg_gemm_fp8", "gemm_fp8", "TG_FP8_E4M3", "TG_FP8_E5M2",
    "tg_gemm_mxfp8", "gemm_mxfp8", "tg_gemm_mxfp4", "gemm_mxfp4", "tg_tune", "tune",
    "tg_epilogue", "gemm_fused", "ACTIVATIONS", "tg_device_error", "tg_status_string",
    "tg_shutdown", "make_options", "gemm", "gemm_host", "plan", "OPERAND_FAMILIES", "device_error",
]


class TgError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        name = STATUS_NAMES.get(status, str(status))
        super().__init__(f"{what}: {name} ({tg_status_string(status)})" if what else name)


# ---------------------------------------------------------------- raw C ABI
def tg_gemm(A, B, C, M, N, K, lda, ldb, ldc, batch, strideA, strideB, strideC, stream=None) -> int:
    return load().tg_gemm(A, B, C, M, N, K, lda, ldb, ldc, batch, strideA, strideB, strideC, stream)


def tg_gemm_ex(A, B, C, M, N, K, lda, ldb, ldc, batch, strideA, strideB, strideC, stream=None,
               opt=None) -> int:
    return load().tg_gemm_ex(A, B, C, M, N, K, lda, ldb, ldc, batch, strideA, strideB, strideC,
                             stream, ctypes.byref(opt) if opt is not None else None)


def tg_gemm_host(A, B, C, M, N, K, lda, ldb, ldc, batch, strideA, strideB, strideC, stream=None,
                 opt=None) -> int:
    return load().tg_gemm_host(A, B, C, M, N, K, lda, ldb, ldc, batch, strideA, strideB, strideC,
                               stream, ctypes.byref(opt) if opt is not None else None)


def tg_gemm_fused(A, B, D, M, N, K, lda, ldb, ldd, batch, strideA, strideB, strideD, ep,
                  stream=None, opt=None) -> int:
    return load().tg_gemm_fused(A, B, D, M, N, K, lda, ldb, ldd, batch, strideA, strideB, strideD,
                                ctypes.byref(ep), stream,
                                ctypes.byref(opt) if opt is not None else None)


def tg_gemm_splitk_static(A, B, C, M, N, K, lda, ldb, ldc, batch, strideA, strideB, strideC,
                          split_k, stream=None) -> int:
    return load().tg_gemm_splitk_static(A, B, C, M, N, K, lda, ldb, ldc, batch, strideA, strideB,
                                        strideC, split_k, stream)


def tg_gemm_fp8(A, B, D, M, N, K, lda, ldb, ldd, batch, strideA, strideB, strideD, a_format,
                b_format, ep=None, stream=None, opt=None) -> int:
    return load().tg_gemm_fp8(A, B, D, M, N, K, lda, ldb, ldd, batch, strideA, strideB, strideD,
                              a_format, b_format, ctypes.byref(ep) if ep is not None else None, stream,
                              ctypes.byref(opt) if opt is not None else None)


def tg_gemm_mxfp8(A, B, D, M, N, K, lda, ldb, ldd, batch, strideA, strideB, strideD, a_format,
                  b_format, SFA, ld_sfa, stride_sfa, SFB, ld_sfb, stride_sfb, ep=None, stream=None,
                  opt=None) -> int:
    return load().tg_gemm_mxfp8(A, B, D, M, N, K, lda, ldb, ldd, batch, strideA, strideB, strideD,
                                a_format, b_format, SFA, ld_sfa, stride_sfa, SFB, ld_sfb, stride_sfb,
                                ctypes.byref(ep) if ep is not None else None, stream,
                                ctypes.byref(opt) if opt is not None else None)


def tg_gemm_mxfp4(A, B, D, M, N, K, lda, ldb, ldd, batch, strideA, strideB, strideD, SFA, ld_sfa,
                  stride_sfa, SFB, ld_sfb, stride_sfb, ep=None, stream=None, opt=None) -> int:
    return load().tg_gemm_mxfp4(A, B, D, M, N, K, lda, ldb, ldd, batch, strideA, strideB, strideD,
                                SFA, ld_sfa, stride_sfa, SFB, ld_sfb, stride_sfb,
                                ctypes.byref(ep) if ep is not None else None, stream,
                                ctypes.byref(opt) if opt is not None else None)


def tg_tune(A, B, C, M, N, K, lda, ldb, ldc, batch, strideA, strideB, strideC, stream=None,
            base=None, reps=3, best=None, best_us=None) -> int:
    return load().tg_tune(A, B, C, M, N, K, lda, ldb, ldc, batch, strideA, strideB, strideC, stream,
                          ctypes.byref(base) if base is not None else None, reps,
                          ctypes.byref(best) if best is not None else None,
                          ctypes.byref(best_us) if best_us is not None else None)


def tg_plan(A, B, C, M, N, K, lda, ldb, ldc, batch, strideA, strideB, strideC, sm_count=0,
            opt=None, out=None):
    out = tg_plan_info() if out is None else out
    st = load().tg_plan(A, B, C, M, N, K, lda, ldb, ldc, batch, strideA, strideB, strideC,
                        sm_count, ctypes.byref(opt) if opt is not None else None, ctypes.byref(out))
    return st, out


def tg_device_error(stream=None) -> int:
    return load().tg_device_error(stream)


def tg_status_string(status: int) -> str:
    return load().tg_status_string(status).decode()


def tg_shutdown() -> None:
    load().tg_shutdown()


# ---------------------------------------------------------------- conveniences
def make_options(**kw) -> tg_options:
    o = tg_options()
    for k, v in kw.items():
        if not hasattr(o, k):
            raise TypeError(f"unknown option {k!r}")
        setattr(o, k, int(v))
    return o


def _stream_ptr(stream):
    import torch

    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _geometry(t, shape, st, what):
    """_operand_geometry on the tensor's shape and strides, read once (each
    read is a call into the framework)."""
    nd = len(shape)
    if nd not in (2, 3):
        raise ValueError(f"{what} must be 2-D or 3-D")
    rows, cols = shape[-2], shape[-1]
    if st[-1] != 1 and cols > 1:
        raise ValueError(f"{what} must have unit stride in its last dimension")
    ld = st[-2] if rows > 1 else max(cols, 1)
    if nd == 3:
        batch, sb = shape[0], (st[0] if shape[0] > 1 else 0)
    else:
        batch, sb = 1, 0
    return t.data_ptr(), rows, cols, max(ld, cols), batch, sb


def _operand_geometry(t, rows_dim, what):
    """(ptr, rows, cols, ld, batch, batch_stride) of a 2-D or 3-D tensor
    whose last dim has unit stride."""
    return _geometry(t, t.shape, t.stride(), what)


def _operand(t, what):
    """(ptr, rows, cols, ld, batch, batch_stride, col_major) of a logical
    rows x cols operand: row-major when its last dim has unit stride,
    column-major (a transposed view) when its second-last dim has."""
    shape, st = t.shape, t.stride()
    nd = len(shape)
    rows, cols = shape[-2], shape[-1]
    if nd in (2, 3) and cols > 1 and st[-1] != 1 and (st[-2] == 1 or rows == 1):
        ld = max(st[-1], rows, 1)
        batch, sb = (shape[0], st[0] if shape[0] > 1 else 0) if nd == 3 else (1, 0)
        return t.data_ptr(), rows, cols, ld, batch, sb, True
    return (*_geometry(t, shape, st, what), False)


def _with_layout(options, a_cm, b_cm):
    if not (a_cm or b_cm):
        return options
    o = tg_options()
    if options is not None:
        ctypes.memmove(ctypes.byref(o), ctypes.byref(options), ctypes.sizeof(o))
    o.a_col_major = int(a_cm)
    o.b_col_major = int(b_cm)
    return o


def gemm(A, B, C=None, *, options: tg_options | None = None, stream=None):
    """C = A @ B (per problem) for CUDA bf16 tensors A [.., M, K], B [.., K, N];
    C is an fp32 CUDA tensor [.., M, N] (allocated when None).  Asynchronous
    on ``stream`` (default: torch's current stream)."""
    import torch

    if A.dtype != torch.bfloat16 or B.dtype != torch.bfloat16:
        raise TypeError("A and B must be bf16")
    if not (A.is_cuda and B.is_cuda):
        raise ValueError("A and B must be CUDA tensors (use gemm_host for host buffers)")
    pa, M, K, lda, ba, sA, a_cm = _operand(A, "A")
    pb, K2, N, ldb, bb, sB, b_cm = _operand(B, "B")
    options = _with_layout(options, a_cm, b_cm)
    if K2 != K:
        raise ValueError(f"inner dimensions differ: {K} vs {K2}")
    batch = max(ba, bb)
    if ba not in (1, batch) or bb not in (1, batch):
        raise ValueError("batch sizes differ")
    if ba == 1:
        sA = 0
    if bb == 1:
        sB = 0
    if C is None:
        shape = (batch, M, N) if (A.dim() == 3 or B.dim() == 3) else (M, N)
        C = torch.empty(shape, dtype=torch.float32, device=A.device)
    if C.dtype != torch.float32 or not C.is_cuda:
        raise TypeError("C must be an fp32 CUDA tensor")
    pc, Mc, Nc, ldc, bc, sC = _operand_geometry(C, -2, "C")
    if (Mc, Nc) != (M, N) or bc != batch:
        raise ValueError("C has the wrong shape")
    st = tg_gemm_ex(pa, pb, pc, M, N, K, lda, ldb, ldc, batch, sA, sB, sC, _stream_ptr(stream),
                    options)
    if st != TG_OK:
        raise TgError(st, "tg_gemm_ex")
    return C


def gemm_fused(A, B, D=None, *, bias=None, residual=None, alpha: float = 1.0, beta: float = 1.0,
               activation: str = "none", out_dtype=None, options: tg_options | None = None,
               stream=None):
    """D = act(alpha * (A @ B) + bias) + beta * residual, fused into the GEMM's
    store-back.  bias: fp32 CUDA tensor [N] or [batch, N]; residual: CUDA
    tensor shaped like D; D: fp32 or bf16 (out_dtype, default fp32)."""
    import torch

    if A.dtype != torch.bfloat16 or B.dtype != torch.bfloat16:
        raise TypeError("A and B must be bf16")
    pa, M, K, lda, ba, sA, a_cm = _operand(A, "A")
    pb, K2, N, ldb, bb, sB, b_cm = _operand(B, "B")
    options = _with_layout(options, a_cm, b_cm)
    if K2 != K:
        raise ValueError(f"inner dimensions differ: {K} vs {K2}")
    batch = max(ba, bb)
    if ba == 1:
        sA = 0
    if bb == 1:
        sB = 0
    if D is None:
        dt = out_dtype if out_dtype is not None else torch.float32
        shape = (batch, M, N) if (A.dim() == 3 or B.dim() == 3) else (M, N)
        D = torch.empty(shape, dtype=dt, device=A.device)
    if D.dtype not in (torch.float32, torch.bfloat16) or not D.is_cuda:
        raise TypeError("D must be an fp32 or bf16 CUDA tensor")
    pd, Md, Nd, ldd, bd, sD = _operand_geometry(D, -2, "D")
    if (Md, Nd) != (M, N) or bd != batch:
        raise ValueError("D has the wrong shape")
    ep = tg_epilogue()
    ep.alpha = float(alpha)
    ep.beta = float(beta)
    ep.activation = ACTIVATIONS[activation]
    ep.out_type = TG_BF16 if D.dtype == torch.bfloat16 else TG_F32
    if bias is not None:
        if bias.dtype != torch.float32 or not bias.is_cuda or bias.stride(-1) != 1:
            raise TypeError("bias must be a contiguous fp32 CUDA tensor")
        ep.bias = bias.data_ptr()
        ep.bias_stride = bias.stride(0) if bias.dim() == 2 and bias.shape[0] > 1 else 0
    if residual is not None:
        if residual.dtype != D.dtype or not residual.is_cuda:
            raise TypeError("residual must have D's dtype and live on the GPU")
        pr, Mr, Nr, ldr, br, sR = _operand_geometry(residual, -2, "residual")
        if (Mr, Nr) != (M, N) or br not in (1, batch):
            raise ValueError("residual has the wrong shape")
        ep.residual = pr
        ep.ldr = ldr
        ep.strideR = sR if br > 1 else 0
    st = tg_gemm_fused(pa, pb, pd, M, N, K, lda, ldb, ldd, batch, sA, sB, sD, ep,
                       _stream_ptr(stream), options)
    if st != TG_OK:
        raise TgError(st, "tg_gemm_fused")
    return D


def _fp8_format(t, what):
    import torch

    if t.dtype == torch.float8_e4m3fn:
        return TG_FP8_E4M3
    if t.dtype == torch.float8_e5m2:
        return TG_FP8_E5M2
    raise TypeError(f"{what} must be float8_e4m3fn or float8_e5m2")


def _fp8_call(A, Bt, D, scale, bias, residual, beta, activation, out_dtype, fp4=False):
    """Shapes, D and the epilogue of the 8-bit entry points (fp4: packed
    4-bit operands, uint8 tensors of two elements a byte; K, the leading
    dimensions and the batch strides passed on count elements)."""
    import torch

    if fp4:
        if A.dtype != torch.uint8 or Bt.dtype != torch.uint8:
            raise TypeError("packed 4-bit A and Bt must be uint8 tensors (two E2M1 codes a byte)")
        fa = fb = 0
    else:
        fa, fb = _fp8_format(A, "A"), _fp8_format(Bt, "Bt")
    if not (A.is_cuda and Bt.is_cuda):
        raise ValueError("A and Bt must be CUDA tensors")
    pa, M, K, lda, ba, sA = _operand_geometry(A, -2, "A")
    pb, N, K2, ldb, bb, sB = _operand_geometry(Bt, -2, "Bt")
    if fp4:
        K, K2, lda, ldb, sA, sB = 2 * K, 2 * K2, 2 * lda, 2 * ldb, 2 * sA, 2 * sB
    if K2 != K:
        raise ValueError(f"inner dimensions differ: {K} vs {K2}")
    batch = max(ba, bb)
    if ba == 1:
        sA = 0
    if bb == 1:
        sB = 0
    if D is None:
        dt = out_dtype if out_dtype is not None else torch.float32
        shape = (batch, M, N) if (A.dim() == 3 or Bt.dim() == 3) else (M, N)
        D = torch.empty(shape, dtype=dt, device=A.device)
    if D.dtype not in (torch.float32, torch.bfloat16) or not D.is_cuda:
        raise TypeError("D must be an fp32 or bf16 CUDA tensor")
    pd, Md, Nd, ldd, bd, sD = _operand_geometry(D, -2, "D")
    if (Md, Nd) != (M, N) or bd != batch:
        raise ValueError("D has the wrong shape")
    ep = tg_epilogue()
    ep.alpha = float(scale)
    ep.beta = float(beta)
    ep.activation = ACTIVATIONS[activation]
    ep.out_type = TG_BF16 if D.dtype == torch.bfloat16 else TG_F32
    if bias is not None:
        if bias.dtype != torch.float32 or not bias.is_cuda or bias.stride(-1) != 1:
            raise TypeError("bias must be a contiguous fp32 CUDA tensor")
        ep.bias = bias.data_ptr()
        ep.bias_stride = bias.stride(0) if bias.dim() == 2 and bias.shape[0] > 1 else 0
    if residual is not None:
        if residual.dtype != D.dtype or not residual.is_cuda:
            raise TypeError("residual must have D's dtype and live on the GPU")
        pr, Mr, Nr, ldr, br, sR = _operand_geometry(residual, -2, "residual")
        if (Mr, Nr) != (M, N) or br not in (1, batch):
            raise ValueError("residual has the wrong shape")
        ep.residual = pr
        ep.ldr = ldr
        ep.strideR = sR if br > 1 else 0
    args = (pa, pb, pd, M, N, K, lda, ldb, ldd, batch, sA, sB, sD, fa, fb)
    return D, ep, args


def gemm_fp8(A, Bt, D=None, *, scale: float = 1.0, bias=None, residual=None, beta: float = 1.0,
             activation: str = "none", out_dtype=None, options: tg_options | None = None,
             stream=None):
    """D = act(scale * (A @ Bt^T) + bias) + beta * residual with 8-bit
    floating-point A [.., M, K] and Bt [.., N, K] (B column-major), both
    contiguous along K; scale carries the operands' per-tensor scales."""
    D, ep, args = _fp8_call(A, Bt, D, scale, bias, residual, beta, activation, out_dtype)
    st = tg_gemm_fp8(*args, ep, _stream_ptr(stream), options)
    if st != TG_OK:
        raise TgError(st, "tg_gemm_fp8")
    return D


def gemm_mxfp8(A, Bt, SFA, SFB, D=None, *, scale: float = 1.0, bias=None, residual=None,
               beta: float = 1.0, activation: str = "none", out_dtype=None,
               options: tg_options | None = None, stream=None):
    """Block-scaled (MXFP8) GEMM: as gemm_fp8, with every 32 consecutive
    elements along K of a row of A (of Bt) scaled by 2^(e - 127), e the
    uint8 E8M0 code in SFA [.., M, ceil(K/32)] (SFB [.., N, ceil(K/32)])."""
    import torch

    D, ep, args = _fp8_call(A, Bt, D, scale, bias, residual, beta, activation, out_dtype)
    M, N, K, batch = args[3], args[4], args[5], args[9]
    runs = -(-K // 32)
    geo = []
    for sf, rows, name in ((SFA, M, "SFA"), (SFB, N, "SFB")):
        if sf.dtype != torch.uint8 or not sf.is_cuda:
            raise TypeError(f"{name} must be a uint8 CUDA tensor")
        p, r, c, ld, b, sb = _operand_geometry(sf, -2, name)
        if (r, c) != (rows, runs) or b not in (1, batch):
            raise ValueError(f"{name} must have shape [.., {rows}, {runs}]")
        geo.append((p, ld, sb if b > 1 else 0))
    (pfa, ldfa, sfa_s), (pfb, ldfb, sfb_s) = geo
    st = tg_gemm_mxfp8(*args, pfa, ldfa, sfa_s, pfb, ldfb, sfb_s, ep, _stream_ptr(stream), options)
    if st != TG_OK:
        raise TgError(st, "tg_gemm_mxfp8")
    return D


def gemm_mxfp4(A, Bt, SFA, SFB, D=None, *, scale: float = 1.0, bias=None, residual=None,
               beta: float = 1.0, activation: str = "none", out_dtype=None,
               options: tg_options | None = None, stream=None):
    """Block-scaled 4-bit (MXFP4) GEMM: A [.., M, K/2] and Bt [.., N, K/2]
    are uint8 tensors of packed E2M1 codes (element k of a row in byte k // 2,
    the low nibble for even k), so K = 2 * A.shape[-1]; every 32 consecutive
    elements along K of a row of A (of Bt) are scaled by 2^(e - 127), e the
    uint8 E8M0 code in SFA [.., M, ceil(K/32)] (SFB [.., N, ceil(K/32)]).
    Epilogue arguments as gemm_fp8."""
    import torch

    D, ep, args = _fp8_call(A, Bt, D, scale, bias, residual, beta, activation, out_dtype, fp4=True)
    M, N, K, batch = args[3], args[4], args[5], args[9]
    runs = -(-K // 32)
    geo = []
    for sf, rows, name in ((SFA, M, "SFA"), (SFB, N, "SFB")):
        if sf.dtype != torch.uint8 or not sf.is_cuda:
            raise TypeError(f"{name} must be a uint8 CUDA tensor")
        p, r, c, ld, b, sb = _operand_geometry(sf, -2, name)
        if (r, c) != (rows, runs) or b not in (1, batch):
            raise ValueError(f"{name} must have shape [.., {rows}, {runs}]")
        geo.append((p, ld, sb if b > 1 else 0))
    (pfa, ldfa, sfa_s), (pfb, ldfb, sfb_s) = geo
    st = tg_gemm_mxfp4(*args[:13], pfa, ldfa, sfa_s, pfb, ldfb, sfb_s, ep, _stream_ptr(stream), options)
    if st != TG_OK:
        raise TgError(st, "tg_gemm_mxfp4")
    return D


def tune(A, B, C=None, *, options: tg_options | None = None, reps: int = 3, stream=None):
    """Run-time plan search on these CUDA tensors (tg_tune): returns
    (options of the fastest plan, its median time in microseconds).  C is
    written with the product."""
    import torch

    if A.dtype != torch.bfloat16 or B.dtype != torch.bfloat16:
        raise TypeError("A and B must be bf16")
    pa, M, K, lda, ba, sA, a_cm = _operand(A, "A")
    pb, K2, N, ldb, bb, sB, b_cm = _operand(B, "B")
    options = _with_layout(options, a_cm, b_cm)
    if K2 != K:
        raise ValueError(f"inner dimensions differ: {K} vs {K2}")
    batch = max(ba, bb)
    if ba == 1:
        sA = 0
    if bb == 1:
        sB = 0
    if C is None:
        shape = (batch, M, N) if (A.dim() == 3 or B.dim() == 3) else (M, N)
        C = torch.empty(shape, dtype=torch.float32, device=A.device)
    pc, Mc, Nc, ldc, bc, sC = _operand_geometry(C, -2, "C")
    best = tg_options()
    us = ctypes.c_float(0.0)
    st = tg_tune(pa, pb, pc, M, N, K, lda, ldb, ldc, batch, sA, sB, sC, _stream_ptr(stream), options,
                 reps, best, us)
    if st != TG_OK:
        raise TgError(st, "tg_tune")
    return best, us.value


def gemm_host(A, B, C=None, *, options: tg_options | None = None, stream=None):
    """The same product on HOST (CPU) tensors, through tg_gemm_host (copies in
    and out inside the call; synchronous)."""
    import torch

    if A.dtype != torch.bfloat16 or B.dtype != torch.bfloat16:
        raise TypeError("A and B must be bf16")
    if A.is_cuda or B.is_cuda:
        raise ValueError("gemm_host takes host tensors")
    pa, M, K, lda, ba, sA = _operand_geometry(A, -2, "A")
    pb, K2, N, ldb, bb, sB = _operand_geometry(B, -2, "B")
    if K2 != K:
        raise ValueError(f"inner dimensions differ: {K} vs {K2}")
    batch = max(ba, bb)
    if ba == 1:
        sA = 0
    if bb == 1:
        sB = 0
    if C is None:
        shape = (batch, M, N) if (A.dim() == 3 or B.dim() == 3) else (M, N)
        C = torch.empty(shape, dtype=torch.float32)
    pc, Mc, Nc, ldc, bc, sC = _operand_geometry(C, -2, "C")
    if (Mc, Nc) != (M, N) or bc != batch:
        raise ValueError("C has the wrong shape")
    st = tg_gemm_host(pa, pb, pc, M, N, K, lda, ldb, ldc, batch, sA, sB, sC,
                      _stream_ptr(stream), options)
    if st != TG_OK:
        raise TgError(st, "tg_gemm_host")
    return C


OPERAND_FAMILIES = {"bf16": 0, "fp8": 1, "mxfp8": 2, "mxfp4": 3}


def plan(M, N, K, batch=1, *, lda=None, ldb=None, ldc=None, strideA=None, strideB=None,
         strideC=None, A=0x1000, B=0x100000000, C=0x200000000, sm_count=0, options=None,
         operands: str = "bf16") -> dict:
    """The plan tg_gemm_ex would use (host-only when sm_count > 0); with
    operands="fp8" / "mxfp8" / "mxfp4" the plan of gemm_fp8 / gemm_mxfp8 /
    gemm_mxfp4 (B stored N x K, so ldb defaults to K; for mxfp4 K and the
    pitches count elements).  The default addresses are placeholders
    with 16-byte alignment; pass real or deliberately misaligned addresses
    to see the pack decisions."""
    family = OPERAND_FAMILIES[operands]
    if family:
        options = options if options is not None else tg_options()
        options.operands = family
    lda = K if lda is None else lda
    ldb = (K if family else N) if ldb is None else ldb
    ldc = N if ldc is None else ldc
    strideA = M * lda if strideA is None else strideA
    strideB = (N if family else K) * ldb if strideB is None else strideB
    strideC = M * ldc if strideC is None else strideC
    st, info = tg_plan(A, B, C, M, N, K, lda, ldb, ldc, batch, strideA, strideB, strideC,
                       sm_count, options)
    if st != TG_OK:
        raise TgError(st, "tg_plan")
    return info.as_dict()


def device_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) its watchdog status."""
    return tg_device_error(_stream_ptr(stream))
