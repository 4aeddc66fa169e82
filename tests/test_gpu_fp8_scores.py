"""The decode over an FP8 cache with its scores on FP8 tensor cores (MLA_KERNEL_TC_FP8_SCORES)
against the oracle's FP8-scores reading (reading 8 of the oracle): q_lat's latent part is
quantised per (query row, head) in 1x128 groups exactly as the cache's latents are
(「Deepseek系列从v3到R易背面经版」 F8量化策略), each group's code product is scaled by the two
group scales, the bf16 RoPE part is added, and the softmax and P.V are the ordinary ones.

The reference is ``latent_attention`` on the query that ``quantize_q_latent`` returns, at the
FP8 cache's tolerance (1e-2 max|oracle| + 1e-3). The wide-spread case also checks that this
reference and the unquantised one are further apart than that tolerance, so the test tells
the two definitions apart.
"""
import numpy as np
import pytest
import torch

import mla_latent_kv_78_b300 as M
import workloads as W
from oracle import mla_oracle as O

from _support import ACT, Case, assert_close, dev, gpu_rows, tau_of, theta_of, tolerance

pytestmark = pytest.mark.gpu

needs_cuda = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")

K8 = M.MLA_KERNEL_TC_FP8_SCORES

FP8_SMALL = W.small_v2(3, [129, 64, 70], n_q=2, cache="fp8", seed=41)
FP8_LONG = W.small_v2(4, [700, 257, 1000, 64], n_q=1, cache="fp8", seed=42)
FP8_LONG_MTP = W.small_v2(3, [513, 256, 900], n_q=2, cache="fp8", seed=43)
FP8_YARN = W.small_v2(2, [300, 129], n_q=2, cache="fp8", seed=44, rope_scaling=40.0)
FP8_GROUPS = W.small_v2(3, [300, 700, 64], n_q=2, cache="fp8", seed=45, group_scales=(1.0, 1e-3, 1e-5, 1.0))


def _reference(wl, q_lat_b, ce, b):
    q8 = O.quantize_q_latent(q_lat_b, wl.C)[0]
    return O.latent_attention(q8, ce["c"], ce["k_r"], wl.positions(b), tau_of(wl))


def _run(wl, q_lat, num_splits=0):
    case = Case(wl, kernel=K8, num_splits=num_splits)
    case.step.append(case.new_c, case.new_r)
    case.step.decode(dev(q_lat.reshape(-1, wl.H, wl.C + wl.R), ACT[wl.act]))
    torch.cuda.synchronize()
    assert case.step.status() == 0
    return case


@needs_cuda
@pytest.mark.parametrize("wl", [FP8_SMALL, FP8_LONG, FP8_LONG_MTP, FP8_YARN], ids=lambda w: w.name)
def test_fp8_scores_decode_matches_the_oracle(wl):
    q_lat = wl.latent_queries()
    case = _run(wl, q_lat)
    for b in range(wl.B):
        ref_o, ref_lse = _reference(wl, q_lat[b], case.cache_of(b), b)
        assert_close(wl, gpu_rows(case.step.o_lat, wl, b), ref_o, f"o_lat[b={b}]")
        assert_close(wl, gpu_rows(case.step.lse, wl, b), ref_lse, f"lse[b={b}]")


@needs_cuda
@pytest.mark.parametrize("splits", [2, 3])
def test_fp8_scores_split_kv_matches_the_oracle(splits):
    wl = FP8_LONG
    q_lat = wl.latent_queries()
    case = _run(wl, q_lat, num_splits=splits)
    for b in range(wl.B):
        ref_o, ref_lse = _reference(wl, q_lat[b], case.cache_of(b), b)
        assert_close(wl, gpu_rows(case.step.o_lat, wl, b), ref_o, f"o_lat[b={b}]")
        assert_close(wl, gpu_rows(case.step.lse, wl, b), ref_lse, f"lse[b={b}]")


@needs_cuda
def test_fp8_scores_wide_spread_follows_the_quantised_definition():
    """Queries scaled by 10: scores spanning more than 40 nats. The GPU matches the FP8-scores
    reference, and that reference differs from the unquantised one by more than the tolerance
    somewhere, so the comparison distinguishes the two."""
    wl = FP8_LONG_MTP
    q_lat = W.round_to_storage(wl.latent_queries() * np.float32(10.0), wl.act)
    case = _run(wl, q_lat)
    apart = False
    for b in range(wl.B):
        ce = case.cache_of(b)
        ref_o, ref_lse = _reference(wl, q_lat[b], ce, b)
        exact_o, _ = O.latent_attention(q_lat[b], ce["c"], ce["k_r"], wl.positions(b), tau_of(wl))
        apart |= bool(np.any(np.abs(exact_o - ref_o) > tolerance(wl, ref_o)))
        assert_close(wl, gpu_rows(case.step.o_lat, wl, b), ref_o, f"o_lat[b={b}]")
        assert_close(wl, gpu_rows(case.step.lse, wl, b), ref_lse, f"lse[b={b}]")
    assert apart, "the quantised and exact references agree everywhere: the test cannot tell them apart"


def _spike(X, Y, pos=600):
    """q_lat = X e_0 for every row and head (its quantisation is exact: one nonzero per group
    0, the rest zero), token `pos` of sequence 0 appended again with latent column 0 = Y."""
    wl = FP8_LONG
    case = Case(wl, kernel=K8, num_splits=1)
    case.step.append(case.new_c, case.new_r)
    lat = ACT[wl.latent_storage]
    c0, r0 = wl.latents(0)
    c0 = c0.copy()
    c0[pos, 0] = Y
    case.step.prefill(dev(c0[pos:pos + 1], lat), dev(r0[pos:pos + 1], lat),
                      torch.zeros(1, dtype=torch.int32, device="cuda"),
                      torch.full((1,), pos, dtype=torch.int32, device="cuda"))
    q_lat = np.zeros((wl.B, wl.n_q, wl.H, wl.C + wl.R), np.float32)
    q_lat[..., 0] = X
    case.step.decode(dev(q_lat.reshape(-1, wl.H, wl.C + wl.R), ACT[wl.act]))
    torch.cuda.synchronize()
    assert case.step.status() == 0
    tau = tau_of(wl)
    for b in range(wl.B):
        c, r = wl.latents(b)
        if b == 0:
            c = c.copy()
            c[pos, 0] = Y
        ce = O.cache_entries(c, r, np.arange(wl.seq_lens[b]), wl.cache, wl.rope_base, theta_of(wl))
        ref_o, ref_lse = _reference(wl, q_lat[b], ce, b)
        if b == 0:
            jump = X * ce["c"][pos, 0] * tau - np.delete(X * ce["c"][:, 0] * tau, pos).max()
        assert_close(wl, gpu_rows(case.step.o_lat, wl, b), ref_o, f"o_lat[b={b}]")
        assert_close(wl, gpu_rows(case.step.lse, wl, b), ref_lse, f"lse[b={b}]")
    return jump


@needs_cuda
def test_fp8_scores_late_spike():
    """A late token ~30 nats above the rest: absorbed by the lagging softmax reference."""
    assert _spike(30.0, 17.0) > 28.0


@needs_cuda
def test_fp8_scores_spike_beyond_the_weight_range():
    """~80 nats: the first pass clamps, the unit runs again with exact maxima (both extra
    passes quantise Q again and go through the FP8 scores)."""
    assert _spike(30.0, 40.0) > 75.0


@needs_cuda
def test_fp8_scores_groups_far_below_unit_scale():
    """Cache groups drawn 1e-3 and 1e-5 times smaller: the key scales enter the scores in fp32
    after each group's code product, so small groups keep their precision. Each latent group
    of o_lat is checked at a tolerance scaled to that group."""
    wl = FP8_GROUPS
    q_lat = wl.latent_queries()
    case = _run(wl, q_lat)
    for b in range(wl.B):
        ref_o, ref_lse = _reference(wl, q_lat[b], case.cache_of(b), b)
        got = gpu_rows(case.step.o_lat, wl, b)
        for g in range(wl.C // 128):
            sl = slice(128 * g, 128 * (g + 1))
            assert_close(wl, got[..., sl], ref_o[..., sl], f"o_lat[b={b}] group {g}")
        assert_close(wl, gpu_rows(case.step.lse, wl, b), ref_lse, f"lse[b={b}]")
