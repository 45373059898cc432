"""GPU checks of the run-time plan search (tg_tune)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import synth
import tiled_gemm_codegen_gb300 as tg
from gpu_helpers import dev, oracle_dense

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,N,K,batch", [(1000, 1500, 2000, 1), (64, 4096, 4096, 1), (300, 200, 700, 4)])
def test_tune_returns_a_valid_faster_or_equal_plan(M, N, K, batch):
    A, B = synth.make_int_inputs(batch, M, N, K, seed=M + N)
    Ad, Bd = A.to(dev()), B.to(dev())
    best, us = tg.tune(Ad, Bd, reps=3)
    assert us > 0
    # the options form a valid plan, and the product with them is exact
    info = tg.plan(M, N, K, batch, A=Ad.data_ptr(), B=Bd.data_ptr(), C=Ad.data_ptr() + (1 << 32), options=best)
    if best.direct == 2:
        assert info["direct"] == 2 and info["block_n"] == 64
    else:
        assert info["block_n"] == best.block_n and info["stages"] == best.stages
    C = tg.gemm(Ad, Bd, options=best)
    assert tg.device_error() == tg.TG_OK
    assert np.array_equal(C.cpu().double().numpy(), oracle_dense(A, B))
    # the search includes the default plan's neighbourhood: its best is not
    # much slower than the default plan, timed the same way
    import statistics
    ts = []
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(); tg.gemm(Ad, Bd, C); e1.record(); e1.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e3)
    assert us <= 1.25 * statistics.median(ts) + 5.0


def test_tune_keeps_layout_fields():
    M, N, K = 200, 300, 400
    A, B = synth.make_int_inputs(1, M, N, K, seed=3)
    At = A.t().contiguous().to(dev()).t()  # column-major A (a transposed view)
    Bd = B.to(dev())
    best, us = tg.tune(At, Bd, reps=2)
    assert best.a_col_major == 1 and best.b_col_major == 0
    C = tg.gemm(At, Bd, options=best)
    assert np.array_equal(C.cpu().double().numpy(), oracle_dense(A, B))
