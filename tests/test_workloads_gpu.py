"""Parity at the five workloads' full sizes, in the launch configuration the
benchmark times (the default plan): every element of C against the fp64
oracle's full product (the oracle does 4096^3 in a few seconds on a
many-core host), within the contract's tolerance for random inputs and bit
for bit for small-integer inputs of the same shapes.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
import tiled_gemm_codegen_gb300 as tg
from gpu_helpers import assert_close, dev

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


@pytest.mark.parametrize("name", NAMES)
def test_workload_float_parity(name):
    """Every element of C against the fp64 oracle's full product, under the
    contract's bounds (relative Frobenius error over the whole output, and
    per element against the largest |C_ref|).  The one-by-one dot-product
    form of the oracle on sampled entries (every tile-fringe row and column
    near the edges, plus random positions) is checked as well."""
    w = synth.WORKLOADS[name]
    A, B = synth.workload_inputs(w)
    C = _run_default(A, B)
    got = C.cpu().double().numpy()
    assert np.all(np.isfinite(got))
    ref = oracle.gemm_dense_f64(A, B)
    assert_close(got, ref, w.K, name)
    g, r = _sampled(w, A, B, C)
    assert_close(g, r, w.K, name + " (sampled entries)")


@pytest.mark.parametrize("name", NAMES)
def test_workload_exact_integer(name):
    """Small-integer inputs of the same shapes: every partial sum is an exact
    fp32 integer, so every element of C must equal the oracle bit for bit."""
    w = synth.WORKLOADS[name]
    A, B = synth.make_int_inputs(w.batch, w.M, w.N, w.K, seed=w.seed + 100)
    C = _run_default(A, B)
    got = C.cpu().double().numpy()
    ref = oracle.gemm_dense_f64(A, B)
    bad = np.argwhere(got != ref)
    assert bad.size == 0, f"{name}: {len(bad)} elements differ, first at {bad[:4].tolist()}"
