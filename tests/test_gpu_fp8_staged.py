"""The decode over an FP8 cache through MLA_KERNEL_TC_FP8_STAGED: a streaming kernel converts
every visible token once into a bf16 pool in the workspace (code * group scale in fp32,
rounded once to bf16; 「Deepseek系列从v3到R易背面经版」 F8量化策略: E4M3 codes, one scale per
1x128 group), and the bf16 tensor-core decode runs over it through an identity block table.

Against the oracle at the FP8 cache's tolerance (1e-2 max|oracle| + 1e-3), and against the
fused FP8 kernel (MLA_KERNEL_TC), which builds the same bf16 operands inside the decode and
issues the same MMAs in the same order: the two agree to the rounding of the softmax's row
sums, which the bf16 kernel adds up in another order (one bf16 ulp of o_lat, 1e-6 of lse).
"""
import numpy as np
import pytest
import torch

import mla_latent_kv_78_b300 as M
import workloads as W
from oracle import mla_oracle as O

from _support import ACT, Case, assert_close, dev, gpu_rows, tau_of, theta_of

pytestmark = pytest.mark.gpu

needs_cuda = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")

KS = M.MLA_KERNEL_TC_FP8_STAGED

FP8_SMALL = W.small_v2(3, [129, 64, 70], n_q=2, cache="fp8", seed=61)
FP8_LONG = W.small_v2(4, [700, 257, 1000, 64], n_q=1, cache="fp8", seed=62)
FP8_LONG_MTP = W.small_v2(3, [513, 256, 900], n_q=2, cache="fp8", seed=63)
FP8_YARN = W.small_v2(2, [300, 129], n_q=2, cache="fp8", seed=64, rope_scaling=40.0)
FP8_SEQ = W.small_v2(3, [400, 131, 777], n_q=1, cache="fp8", seed=65, permute_pages=False)
FP8_GROUPS = W.small_v2(3, [300, 700, 64], n_q=2, cache="fp8", seed=66, group_scales=(1.0, 1e-3, 1e-5, 1.0))
_lens = [int(x) for x in np.random.default_rng(67).integers(2, 600, size=45)]
FP8_MANY_MTP = W.small_v2(45, _lens, n_q=2, cache="fp8", seed=68)


def _decode(wl, kernel, num_splits=0, q_lat=None):
    case = Case(wl, kernel=kernel, num_splits=num_splits)
    case.step.append(case.new_c, case.new_r)
    q = wl.latent_queries() if q_lat is None else q_lat
    case.q_dev = dev(q.reshape(-1, wl.H, wl.C + wl.R), ACT[wl.act])
    case.step.decode(case.q_dev)
    torch.cuda.synchronize()
    return case, q


def _check_oracle(case, wl, q_lat):
    tau = tau_of(wl)
    for b in range(wl.B):
        ce = case.cache_of(b)
        ref_o, ref_lse = O.latent_attention(q_lat[b], ce["c"], ce["k_r"], wl.positions(b), tau)
        assert_close(wl, gpu_rows(case.step.o_lat, wl, b), ref_o, f"o_lat[b={b}]")
        assert_close(wl, gpu_rows(case.step.lse, wl, b), ref_lse, f"lse[b={b}]")


@needs_cuda
@pytest.mark.parametrize("wl", [FP8_SMALL, FP8_LONG, FP8_LONG_MTP, FP8_YARN, FP8_SEQ, FP8_MANY_MTP],
                         ids=lambda w: w.name + ("-perm" if w.permute_pages else "-seq") + f"-L{max(w.seq_lens)}")
def test_staged_decode_matches_the_oracle(wl):
    case, q = _decode(wl, KS)
    assert M.mla_decode_kernel(case.cfg, wl.B, wl.n_q) == KS
    assert case.step.status() == 0
    _check_oracle(case, wl, q)


@needs_cuda
@pytest.mark.parametrize("wl", [FP8_LONG_MTP, FP8_SEQ, FP8_MANY_MTP], ids=lambda w: w.name + ("-perm" if w.permute_pages else "-seq") + f"-L{max(w.seq_lens)}")
@pytest.mark.parametrize("splits", [0, 3])
def test_staged_equals_the_fused_kernel(wl, splits):
    """Same operands, same MMA order: the staged and the fused FP8 decodes agree up to the
    order in which the softmax's row sums are added (o_lat within one bf16 ulp of its
    largest element, lse within 1e-6 relative), with the automatic and a forced split."""
    staged, _ = _decode(wl, KS, splits)
    fused, _ = _decode(wl, M.MLA_KERNEL_TC, splits)
    assert staged.step.status() == 0 and fused.step.status() == 0
    a, b = staged.step.o_lat.float(), fused.step.o_lat.float()
    assert float((a - b).abs().max()) <= 2.0 ** -8 * float(b.abs().max())
    la, lb = staged.step.lse, fused.step.lse
    assert float((la - lb).abs().max()) <= 1e-6 * float(lb.abs().max()) + 1e-6


@needs_cuda
@pytest.mark.parametrize("splits", [2, 3])
def test_staged_split_kv_matches_the_oracle(splits):
    case, q = _decode(FP8_LONG, KS, splits)
    assert case.step.status() == 0
    _check_oracle(case, FP8_LONG, q)


@needs_cuda
def test_staged_wide_score_spread():
    """Queries scaled by 10 (scores spanning more than 40 nats)."""
    wl = FP8_LONG_MTP
    q = W.round_to_storage(wl.latent_queries() * np.float32(10.0), wl.act)
    case, _ = _decode(wl, KS, q_lat=q)
    assert case.step.status() == 0
    _check_oracle(case, wl, q)


@needs_cuda
@pytest.mark.parametrize("X, Y, least", [(30.0, 17.0, 28.0), (30.0, 40.0, 75.0)], ids=["30nat", "80nat"])
def test_staged_score_spikes(X, Y, least):
    """One late token X*Y/13.9 nats above the rest: ~30 nats (absorbed by the lagging
    reference) and ~80 nats (beyond the weight range: the unit runs again with exact
    maxima)."""
    wl, pos = FP8_LONG, 600
    case = Case(wl, kernel=KS, num_splits=1)
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
        ref_o, ref_lse = O.latent_attention(q_lat[b], ce["c"], ce["k_r"], wl.positions(b), tau)
        if b == 0:
            jump = X * ce["c"][pos, 0] * tau - np.delete(X * ce["c"][:, 0] * tau, pos).max()
        assert_close(wl, gpu_rows(case.step.o_lat, wl, b), ref_o, f"o_lat[b={b}]")
        assert_close(wl, gpu_rows(case.step.lse, wl, b), ref_lse, f"lse[b={b}]")
    assert jump > least


@needs_cuda
def test_staged_groups_far_below_unit_scale():
    """Groups drawn 1e-3 and 1e-5 times smaller: the staged bf16 values keep each group's
    precision (the scale is applied in fp32). Each group of o_lat at a tolerance scaled to it."""
    wl = FP8_GROUPS
    case, q = _decode(wl, KS)
    assert case.step.status() == 0
    tau = tau_of(wl)
    for b in range(wl.B):
        ce = case.cache_of(b)
        ref_o, _ = O.latent_attention(q[b], ce["c"], ce["k_r"], wl.positions(b), tau)
        got = gpu_rows(case.step.o_lat, wl, b)
        for k, m in enumerate(wl.group_scales):
            cols = slice(128 * k, 128 * (k + 1))
            err = float(np.max(np.abs(got[..., cols] - ref_o[..., cols])))
            tol = 1e-2 * float(np.max(np.abs(ref_o[..., cols]))) + 1e-3 * m
            assert err <= tol, f"b={b} group {k} (x{m:g}): {err:.3e} > {tol:.3e}"


@needs_cuda
def test_staged_bad_page_id_is_flagged_like_the_fused_kernel():
    """A page id outside the pool: MLA_DEV_INDEX_OUT_OF_RANGE, the page reads as zeros (as in
    the fused kernel, whose result it must equal), the other sequences are unaffected."""
    wl = FP8_LONG
    outs = []
    for kernel in (KS, M.MLA_KERNEL_TC):
        case, _ = _decode(wl, kernel)
        good = case.step.o_lat.clone()
        bt = case.step.block_table.clone()
        bt[2, 1] = wl.num_pages + 5
        case.step.block_table.copy_(bt)
        case.step.dev_status.zero_()
        case.step.decode(case.q_dev)
        torch.cuda.synchronize()
        assert case.step.status() & M.MLA_DEV_INDEX_OUT_OF_RANGE
        for b in (0, 1, 3):
            assert torch.equal(case.step.o_lat[b], good[b])
        outs.append(case.step.o_lat.clone())
    assert torch.equal(outs[0], outs[1])


@needs_cuda
def test_staged_short_sequence_is_flagged():
    """seq_lens[b] < n_q: MLA_DEV_BAD_SEQLEN, that row's output is zero, the others exact."""
    wl = FP8_SMALL
    case, q = _decode(wl, KS)
    sl = case.step.seq_lens.clone()
    sl[0] = 1
    case.step.seq_lens.copy_(sl)
    case.step.dev_status.zero_()
    case.step.decode(case.q_dev)
    torch.cuda.synchronize()
    assert case.step.status() & M.MLA_DEV_BAD_SEQLEN
    assert not bool(case.step.o_lat[:wl.n_q].any())
    tau = tau_of(wl)
    for b in range(1, wl.B):
        ce = case.cache_of(b)
        ref_o, _ = O.latent_attention(q[b], ce["c"], ce["k_r"], wl.positions(b), tau)
        assert_close(wl, gpu_rows(case.step.o_lat, wl, b), ref_o, f"o_lat[b={b}]")
