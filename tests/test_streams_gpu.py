"""Concurrency of the C ABI: calls on different streams may run at the same
time, each with its own scratch workspace (split-K partials, tile
counters, pack copies), and calls from several host threads are safe.
Integer-valued inputs make every result exact, so any cross-talk between
the workspaces shows up as a mismatch against the fp64 oracle."""
from __future__ import annotations

import threading

import numpy as np
import pytest
import torch

import synth
import tiled_gemm_codegen_gb300 as tg
from gpu_helpers import dev, oracle_dense

pytestmark = pytest.mark.gpu

# (M, N, K, options, misaligned): split-K, stream-K and the pack pass all
# use the per-stream workspace
CASES = [
    (300, 520, 1024, dict(split_k=3, cta_pair=1), False),
    (257, 389, 1040, dict(stream_k=2, block_n=256, cta_pair=2), False),
    (200, 300, 712, dict(split_k=2, block_n=128, cta_pair=1), True),
    (129, 640, 2048, dict(split_k=4, block_n=64), False),
]


def _operands(i, M, N, K, misaligned):
    A, B = synth.make_int_inputs(1, M, N, K, seed=100 + i)
    want = oracle_dense(A, B)
    Ad, Bd = A.to(dev()), B.to(dev())
    if misaligned:
        # rows of A one element longer than K: not 16-byte aligned -> pack
        Ap = torch.zeros(M, K + 1, dtype=torch.bfloat16, device=dev())
        Ap[:, :K] = Ad
        Ad = Ap[:, :K]
    return Ad, Bd, want


def test_streams_run_concurrently_with_separate_workspaces():
    streams = [torch.cuda.Stream() for _ in CASES]
    ops = [_operands(i, *c[:3], c[4]) for i, c in enumerate(CASES)]
    outs = [torch.full((c[0], c[1]), float("nan"), device=dev()) for c in CASES]
    torch.cuda.synchronize()
    for _ in range(6):
        # every stream's call enqueued before any finishes
        for (M, N, K, opt, _mis), (Ad, Bd, _w), C, s in zip(CASES, ops, outs, streams):
            tg.gemm(Ad, Bd, C, options=tg.make_options(**opt), stream=s)
    torch.cuda.synchronize()
    assert tg.device_error() == tg.TG_OK
    for (Ad, Bd, want), C, c in zip(ops, outs, CASES):
        assert np.array_equal(C.cpu().double().numpy(), want), c


def test_host_threads_on_their_own_streams():
    ops = [_operands(i, *c[:3], c[4]) for i, c in enumerate(CASES)]
    errors = []

    def worker(i):
        try:
            M, N, K, opt, _ = CASES[i]
            Ad, Bd, want = ops[i]
            s = torch.cuda.Stream()
            C = torch.empty(M, N, device=dev())
            with torch.cuda.stream(s):
                for _ in range(8):
                    tg.gemm(Ad, Bd, C, options=tg.make_options(**opt), stream=s)
            s.synchronize()
            if not np.array_equal(C.cpu().double().numpy(), want):
                errors.append(f"case {i}: mismatch")
        except Exception as e:  # reported below, on the main thread
            errors.append(f"case {i}: {e!r}")

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(CASES))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not any(t.is_alive() for t in threads)
    assert not errors, errors
