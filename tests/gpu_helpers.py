"""Shared helpers of the GPU parity tests: tolerance checks and calls
through the C ABI on torch-allocated device memory."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import tiled_gemm_codegen_gb300 as tg

# The tolerance of the contract: relative Frobenius error <= 1e-5 over the
# whole output, and per element |err| <= 1e-5 * sqrt(K) * max|C_ref|.
REL_FRO = 1e-5
PER_ELEM = 1e-5


def assert_close(got: np.ndarray, ref: np.ndarray, K: int, what: str = ""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    nref = np.linalg.norm(ref)
    diff = got - ref
    if nref == 0:
        assert np.all(got == 0), f"{what}: expected exact zeros"
        return 0.0
    rel = np.linalg.norm(diff) / nref
    bound = PER_ELEM * np.sqrt(max(K, 1)) * np.abs(ref).max()
    worst = np.abs(diff).max()
    assert rel <= REL_FRO, f"{what}: relative Frobenius error {rel:.3e} > {REL_FRO}"
    assert worst <= bound, f"{what}: max |err| {worst:.3e} > {bound:.3e}"
    return rel


def dev():
    return torch.device("cuda:0")


def run(A_cpu, B_cpu, options=None, C=None):
    """Copy bf16 CPU operands to the GPU, run tg.gemm, return C on the CPU
    as float64 numpy (after checking the device error word)."""
    A = A_cpu.to(dev())
    B = B_cpu.to(dev())
    out = tg.gemm(A, B, C, options=options)
    st = tg.device_error()
    assert st == tg.TG_OK, f"device error {tg.STATUS_NAMES.get(st, st)}"
    return out.cpu().double().numpy()


def oracle_dense(A_cpu, B_cpu):
    return oracle.gemm_dense_f64(A_cpu, B_cpu)
