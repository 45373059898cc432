"""Parity at the five workloads' full sizes, in the launch configuration the
benchmark times (the default plan).

The oracle computes sampled entries one by one (every tile-fringe row and
column near the edges, plus random positions); a property that holds at any
size - row and column sums of C against A (B 1) and (1^T A) B in fp64 -
covers every output element.  With small-integer inputs of the same shapes
the sampled entries must match the oracle bit for bit.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
import tiled_gemm_codegen_gb300 as tg
from gpu_helpers import PER_ELEM, REL_FRO, assert_close, dev

pytestmark = pytest.mark.gpu

NAMES = list(synth.WORKLOADS)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    tg.load()
    yield
    torch.cuda.empty_cache()


def _run_default(A, B):
    C = tg.gemm(A.to(dev()), B.to(dev()))
    assert tg.device_error() == tg.TG_OK
    return C


def _sampled(w, A, B, C, count=3000, seed=0):
    bi, ii, jj = synth.sample_indices(w.batch, w.M, w.N, count, seed=seed, tile_m=128, tile_n=64)
    ref = oracle.gemm_entries_f64(A, B, w.M, w.N, w.K, bi, ii, jj, batch=w.batch)
    Cc = C if C.dim() == 3 else C.unsqueeze(0)
    idx = (torch.from_numpy(bi).to(dev()), torch.from_numpy(ii).to(dev()), torch.from_numpy(jj).to(dev()))
    got = Cc[idx].double().cpu().numpy()
    return got, ref


def _checksums(w, A, B, C):
    """Row sums and column sums of the GPU output against fp64 products of
    A with B's row sums and of A's column sums with B, problem by problem."""
    Cc = C if C.dim() == 3 else C.unsqueeze(0)
    Ac = A if A.dim() == 3 else A.unsqueeze(0)
    Bc = B if B.dim() == 3 else B.unsqueeze(0)
    worst = 0.0
    for b in range(w.batch):
        c64 = Cc[b].double()
        a64 = Ac[b].to(dev()).double()
        b64 = Bc[b].to(dev()).double()
        row_ref = a64 @ b64.sum(dim=1)
        col_ref = a64.sum(dim=0) @ b64
        scale = float(torch.max(torch.abs(c64)))
        row_tol = w.N * PER_ELEM * np.sqrt(w.K) * scale
        col_tol = w.M * PER_ELEM * np.sqrt(w.K) * scale
        rerr = float(torch.max(torch.abs(c64.sum(dim=1) - row_ref)))
        cerr = float(torch.max(torch.abs(c64.sum(dim=0) - col_ref)))
        assert rerr <= row_tol, (b, rerr, row_tol)
        assert cerr <= col_tol, (b, cerr, col_tol)
        worst = max(worst, rerr / row_tol, cerr / col_tol)
        del c64, a64, b64
    return worst


@pytest.mark.parametrize("name", NAMES)
def test_workload_float_parity(name):
    w = synth.WORKLOADS[name]
    A, B = synth.workload_inputs(w)
    C = _run_default(A, B)
    assert bool(torch.isfinite(C).all())
    if w.M * w.N * w.K * w.batch <= 10 ** 8:
        assert_close(C.cpu().double().numpy(), oracle.gemm_dense_f64(A, B), w.K, name)
        return
    got, ref = _sampled(w, A, B, C)
    # tolerance on the sampled entries: per element against the largest
    # sampled magnitude (stricter than the whole-output max), relative
    # Frobenius error over the sample
    diff = got - ref
    assert np.abs(diff).max() <= PER_ELEM * np.sqrt(w.K) * np.abs(ref).max(), name
    assert np.linalg.norm(diff) / np.linalg.norm(ref) <= REL_FRO, name
    _checksums(w, A, B, C)


@pytest.mark.parametrize("name", NAMES)
def test_workload_exact_integer(name):
    w = synth.WORKLOADS[name]
    A, B = synth.make_int_inputs(w.batch, w.M, w.N, w.K, seed=w.seed + 100)
    C = _run_default(A, B)
    got, ref = _sampled(w, A, B, C, count=2000, seed=1)
    assert np.array_equal(got, ref), name
