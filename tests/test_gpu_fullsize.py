"""GPU parity at the workloads' full sizes, in the launch configuration the benchmark uses
(automatic kernel and split choice), checked on sampled outputs the fp64 oracle computes one
sequence and a few heads at a time.

Workloads: 2 V2-shaped decode (64 x 4096), 3 ragged (128 x U[1024, 32768], permuted pages),
4 long context (8 x 131072), 5 two-token decode over an FP8 cache (128 x 8192).
Tolerance: |gpu - oracle| <= 1e-2 max|oracle| + 1e-3, on o, o_lat and lse.
"""
import numpy as np
import pytest
import torch

import workloads as W

from _support import Case, assert_close, gpu_rows

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

needs_cuda = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")

HEADS = np.array([0, 37, 64, 127])


def _sampled_sequences(wl, k=2):
    """The longest sequence and a seeded pick among the rest."""
    longest = int(np.argmax(wl.seq_lens))
    g = np.random.default_rng(wl.seed)
    others = [b for b in range(wl.B) if b != longest]
    return [longest] + [int(b) for b in g.choice(others, size=k - 1, replace=False)]


@needs_cuda
@pytest.mark.parametrize("n", [2, 3, 4, 5])
def test_full_size_decode_step(n):
    wl = W.config(n)
    case = Case(wl)
    case.run_step()
    assert case.step.status() == 0
    o_all = case.step.o
    assert bool(torch.isfinite(o_all).all())
    assert bool(torch.isfinite(case.step.lse).all())
    for b in _sampled_sequences(wl):
        o, o_lat, lse = case.oracle(b, heads=HEADS)
        got_o = gpu_rows(case.step.o, wl, b)[:, HEADS]
        got_lat = gpu_rows(case.step.o_lat, wl, b)[:, HEADS]
        got_lse = gpu_rows(case.step.lse, wl, b)[:, HEADS]
        assert_close(wl, got_o, o, f"cfg{n} o[b={b}]")
        assert_close(wl, got_lat, o_lat, f"cfg{n} o_lat[b={b}]")
        assert_close(wl, got_lse, lse, f"cfg{n} lse[b={b}]")
