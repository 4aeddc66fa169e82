"""GPU parity at the workloads' full sizes, in the launch configuration the benchmark uses
(automatic kernel and split choice).

Workloads: 2 V2-shaped decode (64 x 4096), 3 ragged (128 x U[1024, 32768], permuted pages),
4 long context (8 x 131072), 5 two-token decode over an FP8 cache (128 x 8192).

For four sequences of each (the longest, the shortest and two seeded picks) every head's
o_lat and lse are checked against the oracle's latent attention, fed with the oracle's own
absorbed queries rounded to bf16 (the type q_lat is stored in); for two of them the
unabsorbed o of a few heads is checked against the non-absorbed definition as well.
Tolerance: |gpu - oracle| <= 1e-2 max|oracle| + 1e-3.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import mla_oracle as O

from _support import Case, assert_close, gpu_rows, tau_of, theta_of

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

needs_cuda = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")

HEADS = np.array([0, 37, 64, 127])


def _sampled_sequences(wl, k=4):
    """The longest and the shortest sequence, then seeded picks among the rest."""
    longest = int(np.argmax(wl.seq_lens))
    shortest = int(np.argmin(wl.seq_lens))
    picked = [longest] + ([shortest] if shortest != longest else [])
    g = np.random.default_rng(wl.seed)
    others = [b for b in range(wl.B) if b not in picked]
    picked += [int(b) for b in g.choice(others, size=k - len(picked), replace=False)]
    return picked


@needs_cuda
@pytest.mark.parametrize("n", [2, 3, 4, 5])
def test_full_size_decode_step(n):
    wl = W.config(n)
    case = Case(wl)
    case.run_step()
    assert case.step.status() == 0
    assert bool(torch.isfinite(case.step.o).all())
    assert bool(torch.isfinite(case.step.lse).all())
    tau = tau_of(wl)
    seqs = _sampled_sequences(wl)
    for k, b in enumerate(seqs):
        pos = wl.positions(b)
        ce = case.cache_of(b)
        q_lat = O.round_bf16(O.absorb_q(case.q_c_np[b], case.q_r_np[b], pos, case.w_uk_np, wl.rope_base, theta_of(wl)))
        ref_lat, ref_lse = O.latent_attention(q_lat, ce["c"], ce["k_r"], pos, tau)
        assert_close(wl, gpu_rows(case.step.o_lat, wl, b), ref_lat, f"cfg{n} o_lat[b={b}] (all heads)")
        assert_close(wl, gpu_rows(case.step.lse, wl, b), ref_lse, f"cfg{n} lse[b={b}] (all heads)")
        if k < 2:
            o, o_lat, lse = case.oracle(b, heads=HEADS)
            assert_close(wl, gpu_rows(case.step.o, wl, b)[:, HEADS], o, f"cfg{n} o[b={b}]")
            assert_close(wl, gpu_rows(case.step.o_lat, wl, b)[:, HEADS], o_lat, f"cfg{n} naive o_lat[b={b}]")
            assert_close(wl, gpu_rows(case.step.lse, wl, b)[:, HEADS], lse, f"cfg{n} naive lse[b={b}]")


@needs_cuda
def test_full_size_two_token_decode_with_fp8_scores():
    """Workload 5 (two-token decode, 128 x 8192, FP8 cache) through MLA_KERNEL_TC_FP8_SCORES:
    every head of four sampled sequences against the oracle's FP8-scores reading (q_lat's
    latent part quantised per 1x128 group, then the ordinary latent attention)."""
    import mla_latent_kv_78_b300 as M
    wl = W.config(5)
    case = Case(wl, kernel=M.MLA_KERNEL_TC_FP8_SCORES)
    case.run_step()
    assert case.step.status() == 0
    tau = tau_of(wl)
    for b in _sampled_sequences(wl):
        pos = wl.positions(b)
        ce = case.cache_of(b)
        q_lat = O.round_bf16(O.absorb_q(case.q_c_np[b], case.q_r_np[b], pos, case.w_uk_np, wl.rope_base, theta_of(wl)))
        q8 = O.quantize_q_latent(q_lat, wl.C)[0]
        ref_lat, ref_lse = O.latent_attention(q8, ce["c"], ce["k_r"], pos, tau)
        assert_close(wl, gpu_rows(case.step.o_lat, wl, b), ref_lat, f"fp8-scores o_lat[b={b}] (all heads)")
        assert_close(wl, gpu_rows(case.step.lse, wl, b), ref_lse, f"fp8-scores lse[b={b}] (all heads)")


@needs_cuda
def test_full_size_two_token_decode_staged():
    """Workload 5 (two-token decode, 128 x 8192, FP8 cache) through MLA_KERNEL_TC_FP8_STAGED
    (the cache converted once to bf16 in the workspace, then the bf16 tensor-core decode):
    every head of four sampled sequences against the oracle."""
    import mla_latent_kv_78_b300 as M
    wl = W.config(5)
    case = Case(wl, kernel=M.MLA_KERNEL_TC_FP8_STAGED)
    case.run_step()
    assert case.step.status() == 0
    tau = tau_of(wl)
    for b in _sampled_sequences(wl):
        pos = wl.positions(b)
        ce = case.cache_of(b)
        q_lat = O.round_bf16(O.absorb_q(case.q_c_np[b], case.q_r_np[b], pos, case.w_uk_np, wl.rope_base, theta_of(wl)))
        ref_lat, ref_lse = O.latent_attention(q_lat, ce["c"], ce["k_r"], pos, tau)
        assert_close(wl, gpu_rows(case.step.o_lat, wl, b), ref_lat, f"staged o_lat[b={b}] (all heads)")
        assert_close(wl, gpu_rows(case.step.lse, wl, b), ref_lse, f"staged lse[b={b}] (all heads)")
