"""GPU parity at sizes the oracle finishes in seconds: every call of the C ABI
against the fp64 oracle on the same seeded inputs.

Tolerance (both o_lat and o): |gpu - oracle| <= 1e-2 max|oracle| + 1e-3 for bf16 and
FP8 caches, <= 1e-5 max|oracle| for the fp32 workload. Page placement and FP8
codes are compared bit for bit.
"""
import numpy as np
import pytest
import torch

import mla_latent_kv_78_b300 as M
import workloads as W
from oracle import mla_oracle as O

from _support import ACT, Case, assert_close, config_of, dev, gpu_rows, tau_of, theta_of

pytestmark = pytest.mark.gpu

needs_cuda = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")

# V2 head shapes, sequences that span several 64-token pages with ragged tails
SMALL_BF16 = W.small_v2(4, [65, 200, 7, 130], n_q=1, cache="bf16", seed=11)
SMALL_FP8 = W.small_v2(3, [129, 64, 70], n_q=2, cache="fp8", seed=12)
SMALL_BF16_MTP = W.small_v2(3, [2, 100, 191], n_q=2, cache="bf16", seed=13)
SMALL_BF16_LONG = W.small_v2(4, [700, 257, 1000, 64], n_q=1, cache="bf16", seed=14)
SMALL_BF16_LONG_MTP = W.small_v2(3, [513, 256, 900], n_q=2, cache="bf16", seed=15)
SMALL_FP8_LONG = W.small_v2(4, [700, 257, 1000, 64], n_q=1, cache="fp8", seed=17)
SMALL_FP8_LONG_MTP = W.small_v2(3, [513, 256, 900], n_q=2, cache="fp8", seed=18)
# 200 query rows: token tiles of the absorb kernels (128 / 64) with a ragged tail
SMALL_BF16_T200 = W.small_v2(100, [3] * 100, n_q=2, cache="bf16", seed=16)
TINY = W.config(1)
TINY_PERM = W.config(1).with_(permute_pages=True)
# YaRN on the decoupled RoPE (「一文通透DeepSeek-V2」 §3.1.3: s = 40), short and long sequences;
# the long one puts the query near position 150K of the 160K the extension targets
SMALL_YARN = W.small_v2(3, [700, 257, 1000], n_q=1, cache="bf16", seed=31, rope_scaling=40.0)
SMALL_YARN_FP8 = W.small_v2(2, [300, 129], n_q=2, cache="fp8", seed=32, rope_scaling=40.0)
LONG_YARN = W.small_v2(2, [150000, 3000], n_q=1, cache="bf16", seed=33, rope_scaling=40.0)
TINY_YARN = W.config(1).with_(rope_scaling=40.0)


def _rope_tol(ref: np.ndarray, k_r: np.ndarray) -> np.ndarray:
    """Bound on a bf16-stored rotated k^R value: one bf16 ulp of the oracle's value, plus
    the fp32 arithmetic error of the rotation, which scales with the pair's magnitude
    |x_2k| + |x_2k+1| rather than with the result (a rotation that nearly cancels)."""
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(ref), 1e-30))) - 7)
    pair = np.abs(k_r[:, 0::2]) + np.abs(k_r[:, 1::2])
    return ulp + 2.0 ** -20 * np.repeat(pair, 2, axis=1)


def _bits_equal(a: np.ndarray, b: np.ndarray) -> bool:
    return a.shape == b.shape and np.array_equal(a.view(np.uint8), b.view(np.uint8))


@needs_cuda
@pytest.mark.parametrize("wl", [TINY, TINY_PERM, SMALL_BF16, SMALL_FP8, SMALL_YARN, TINY_YARN],
                         ids=lambda w: w.name + ("-perm" if w.permute_pages else "") + ("-yarn" if w.rope_scaling > 1 else ""))
def test_append_writes_each_token_to_its_slot(wl):
    """Every cached token lands in pool[block_table[b][pos // P]][pos % P] and nowhere else
    (bit-exact); c_KV is copied (or E4M3-coded, bit-exact), k^R is RoPE'd (<= 1 ulp)."""
    case = Case(wl, prefill=True)
    case.step.append(case.new_c, case.new_r)
    torch.cuda.synchronize()
    assert case.step.status() == 0
    pool = case.step.pool.cpu().numpy()  # [num_pages, P, entry]
    touched = np.zeros(pool.shape[:2], dtype=bool)
    for b in range(wl.B):
        L = wl.seq_lens[b]
        c, r = wl.latents(b)
        ce = O.cache_entries(c, r, np.arange(L), wl.cache, wl.rope_base, theta_of(wl))
        pg, sl = O.page_slots(np.full(L, b), np.arange(L), case.bt_np, wl.P)
        ent = pool[pg, sl]                       # [L, entry]
        touched[pg, sl] = True
        if wl.cache == "f32":
            got_c = ent[:, :4 * wl.C].copy().view(np.float32)
            got_r = ent[:, 4 * wl.C:].copy().view(np.float32).astype(np.float64)
            assert _bits_equal(got_c, c.astype(np.float32))
            np.testing.assert_allclose(got_r, ce["k_r"], rtol=2 ** -23, atol=1e-30)
        elif wl.cache == "bf16":
            got_c = ent[:, :2 * wl.C].copy().view(np.uint16)
            assert np.array_equal(got_c, W.to_bf16_bits(c))
            got_r = W.bf16_bits_to_f32(ent[:, 2 * wl.C:].copy().view(np.uint16)).astype(np.float64)
            assert np.all(np.abs(got_r - ce["k_r"]) <= _rope_tol(ce["k_r"], r))
        else:
            codes = ent[:, :wl.C]
            got_r = W.bf16_bits_to_f32(ent[:, wl.C:wl.C + 2 * wl.R].copy().view(np.uint16)).astype(np.float64)
            scales = ent[:, wl.C + 2 * wl.R:].copy().view(np.float32)
            assert np.array_equal(codes, ce["codes"]), "E4M3 codes differ"
            assert _bits_equal(scales, ce["scales"].astype(np.float32)), "group scales differ"
            assert np.all(np.abs(got_r - ce["k_r"]) <= _rope_tol(ce["k_r"], r))
    # slots no token maps to stay untouched (the pool starts zeroed)
    assert not pool[~touched].any()


@needs_cuda
@pytest.mark.parametrize("wl", [TINY, SMALL_BF16, SMALL_FP8, SMALL_BF16_LONG_MTP, SMALL_BF16_T200, SMALL_YARN,
                                TINY_YARN],
                         ids=lambda w: w.name + f"-T{w.B * w.n_q}" + ("-yarn" if w.rope_scaling > 1 else ""))
@pytest.mark.parametrize("kernel", [M.MLA_KERNEL_SIMT, M.MLA_KERNEL_AUTO], ids=["simt", "auto"])
def test_absorb_q(wl, kernel):
    case = Case(wl, kernel=kernel, prefill=False)
    case.step.absorb(case.q_c, case.q_r)
    torch.cuda.synchronize()
    pos = np.concatenate([wl.positions(b) for b in range(wl.B)])
    ref = O.absorb_q(case.q_c_np.reshape(-1, wl.H, wl.D), case.q_r_np.reshape(-1, wl.H, wl.R), pos,
                     case.w_uk_np, wl.rope_base, theta_of(wl))
    got = case.step.q_lat.float().cpu().numpy()
    assert_close(wl, got[..., :wl.C], ref[..., :wl.C], "q_lat latent part")
    assert_close(wl, got[..., wl.C:], ref[..., wl.C:], "q_lat RoPE part")


@needs_cuda
@pytest.mark.parametrize("wl", [TINY, SMALL_BF16, SMALL_BF16_T200], ids=lambda w: w.name + f"-T{w.B * w.n_q}")
@pytest.mark.parametrize("kernel", [M.MLA_KERNEL_SIMT, M.MLA_KERNEL_AUTO], ids=["simt", "auto"])
def test_unabsorb(wl, kernel):
    case = Case(wl, kernel=kernel, prefill=False)
    g = np.random.default_rng(5)
    o_lat = W.round_to_storage(g.standard_normal((wl.B * wl.n_q, wl.H, wl.C)).astype(np.float32) * 0.1, wl.act)
    case.step.o_lat.copy_(dev(o_lat, ACT[wl.act]))
    case.step.unabsorb()
    torch.cuda.synchronize()
    ref = O.unabsorb(o_lat, case.w_uv_np)
    assert_close(wl, case.step.o.cpu().numpy(), ref, "o")


def _decode_only(wl, kernel, num_splits=0):
    case = Case(wl, kernel=kernel, num_splits=num_splits)
    case.step.append(case.new_c, case.new_r)
    q_lat = wl.latent_queries()
    case.step.decode(dev(q_lat.reshape(-1, wl.H, wl.C + wl.R), ACT[wl.act]))
    torch.cuda.synchronize()
    assert case.step.status() == 0
    tau = tau_of(wl)
    for b in range(wl.B):
        ce = case.cache_of(b)
        ref_o, ref_lse = O.latent_attention(q_lat[b], ce["c"], ce["k_r"], wl.positions(b), tau)
        assert_close(wl, gpu_rows(case.step.o_lat, wl, b), ref_o, f"o_lat[b={b}]")
        assert_close(wl, gpu_rows(case.step.lse, wl, b), ref_lse, f"lse[b={b}]")
    return case


@needs_cuda
@pytest.mark.parametrize("wl", [TINY, TINY_PERM, SMALL_BF16, SMALL_FP8, SMALL_BF16_MTP,
                                SMALL_BF16_LONG, SMALL_BF16_LONG_MTP, SMALL_FP8_LONG,
                                SMALL_FP8_LONG_MTP],
                         ids=lambda w: w.name + ("-perm" if w.permute_pages else "") + f"-L{max(w.seq_lens)}")
@pytest.mark.parametrize("kernel", [M.MLA_KERNEL_SIMT, M.MLA_KERNEL_AUTO], ids=["simt", "auto"])
def test_decode_latent_attention(wl, kernel):
    _decode_only(wl, kernel)


@needs_cuda
@pytest.mark.parametrize("splits", [2, 3, 7])
@pytest.mark.parametrize("kernel", [M.MLA_KERNEL_SIMT, M.MLA_KERNEL_AUTO], ids=["simt", "auto"])
@pytest.mark.parametrize("wl", [SMALL_BF16_LONG, SMALL_FP8_LONG], ids=["bf16", "fp8"])
def test_decode_splits_agree(splits, kernel, wl):
    base = _decode_only(wl, kernel, 1)
    other = _decode_only(wl, kernel, splits)
    a = base.step.o_lat.float().cpu().numpy()
    b = other.step.o_lat.float().cpu().numpy()
    # split partials are fp32; the final bf16 rounding may differ by one ulp, and the
    # tensor-core kernel sums P after rounding it to bf16 relative to each split's own
    # reference maximum, so lse may move by up to one bf16 rounding (2^-9 relative in l)
    assert np.max(np.abs(a - b)) <= 2.0 ** -8 * np.max(np.abs(a))
    np.testing.assert_allclose(other.step.lse.cpu().numpy(), base.step.lse.cpu().numpy(),
                               rtol=0, atol=2.0 ** -9)


# more query rows than the 74 CTA pairs, lengths spread from 1 to 900 tokens: the tensor-core
# decode takes its rows longest first (a device-side plan); every row must still be exact
_lens = [int(x) for x in np.random.default_rng(51).integers(1, 900, size=96)]
MANY_RAGGED = W.small_v2(96, _lens, n_q=1, cache="bf16", seed=52)
MANY_RAGGED_FP8_MTP = W.small_v2(45, [max(2, x // 2) for x in _lens[:45]], n_q=2, cache="fp8", seed=53)


@needs_cuda
@pytest.mark.parametrize("wl", [MANY_RAGGED, MANY_RAGGED_FP8_MTP], ids=["bf16", "fp8-mtp"])
def test_decode_many_ragged_rows(wl):
    _decode_only(wl, M.MLA_KERNEL_AUTO)


# 90 query rows of one length: two full rounds of the 74 CTA pairs would leave 16 rows for a
# third; those (the plan's last 16) run instead as two half-range units each, merged after
EQUAL_MTP = W.small_v2(45, [700] * 45, n_q=2, cache="bf16", seed=54)


@needs_cuda
def test_tail_rows_split_in_two_are_exact_and_deterministic():
    """Every row, split or not, against the oracle; then the same decode three more times
    with bit-identical results (which rows form the split tail depends on the lengths only)."""
    wl = EQUAL_MTP
    case = _decode_only(wl, M.MLA_KERNEL_AUTO)
    # the 16 tail rows' two fp32 partials per head (148 SMs: 74 pairs)
    assert M.mla_decode_workspace_size(case.cfg, wl.B, wl.n_q, wl.max_seq_len, 0) >= 16 * 128 * 2 * 513 * 4
    q = dev(wl.latent_queries().reshape(-1, wl.H, wl.C + wl.R), ACT[wl.act])
    first_o, first_lse = case.step.o_lat.clone(), case.step.lse.clone()
    for _ in range(3):
        case.step.decode(q)
        torch.cuda.synchronize()
        assert torch.equal(case.step.o_lat, first_o) and torch.equal(case.step.lse, first_lse)


@needs_cuda
def test_tensor_core_kernel_is_selected_for_v2_shapes():
    for wl in (SMALL_BF16, SMALL_BF16_MTP, SMALL_FP8, SMALL_FP8_LONG):
        assert M.mla_decode_kernel(config_of(wl), wl.B, wl.n_q) == M.MLA_KERNEL_TC
    assert M.mla_decode_kernel(config_of(TINY), TINY.B, 1) == M.MLA_KERNEL_SIMT


@needs_cuda
@pytest.mark.parametrize("wl", [TINY, TINY_PERM, SMALL_BF16, SMALL_FP8, SMALL_BF16_MTP, SMALL_BF16_LONG,
                                SMALL_FP8_LONG_MTP, SMALL_YARN, SMALL_YARN_FP8, TINY_YARN],
                         ids=lambda w: w.name + ("-perm" if w.permute_pages else "") + f"-L{max(w.seq_lens)}"
                         + ("-yarn" if w.rope_scaling > 1 else ""))
def test_decode_step_end_to_end(wl):
    """append -> absorb -> decode -> unabsorb against the non-absorbed oracle."""
    case = Case(wl)
    case.run_step()
    assert case.step.status() == 0
    for b in range(wl.B):
        o, o_lat, lse = case.oracle(b)
        assert_close(wl, gpu_rows(case.step.o, wl, b), o, f"o[b={b}]")
        assert_close(wl, gpu_rows(case.step.o_lat, wl, b), o_lat, f"o_lat[b={b}]")
        assert_close(wl, gpu_rows(case.step.lse, wl, b), lse, f"lse[b={b}]")


@needs_cuda
@pytest.mark.parametrize("branches", [False, True], ids=["series", "branches"])
def test_captured_step_matches_the_eager_step(branches):
    """The step recorded as one CUDA graph (append and absorb in series, or as parallel
    branches) computes what the four calls do eagerly, bit for bit, replay after replay, and
    matches the oracle."""
    wl = SMALL_BF16_LONG
    case = Case(wl)
    case.run_step()
    eager = case.step.o.clone()
    case.step.capture(case.new_c, case.new_r, case.q_c, case.q_r, branches=branches)
    for _ in range(3):
        case.step.o.zero_()
        case.step.replay()
        torch.cuda.synchronize()
        assert torch.equal(case.step.o, eager)
    assert case.step.status() == 0
    for b in range(wl.B):
        o, _, _ = case.oracle(b)
        assert_close(wl, gpu_rows(case.step.o, wl, b), o, f"o[b={b}]")


@needs_cuda
@pytest.mark.parametrize("wl", [TINY, SMALL_BF16, SMALL_FP8, SMALL_BF16_T200], ids=lambda w: w.name + f"-T{w.B * w.n_q}")
def test_append_absorb_equals_the_two_calls(wl):
    """mla_append_absorb (the absorption overlapping the append) leaves the pool and q_lat
    exactly as mla_append_cache followed by mla_absorb_q."""
    sep = Case(wl)
    sep.step.append(sep.new_c, sep.new_r)
    sep.step.absorb(sep.q_c, sep.q_r)
    fused = Case(wl)
    fused.step.append_absorb(fused.new_c, fused.new_r, fused.q_c, fused.q_r)
    torch.cuda.synchronize()
    assert torch.equal(sep.step.pool, fused.step.pool)
    assert torch.equal(sep.step.q_lat, fused.step.q_lat)
    assert fused.step.status() == 0


@needs_cuda
@pytest.mark.parametrize("splits", [1, 3])
def test_decode_is_deterministic(splits):
    wl = SMALL_BF16_LONG
    case = Case(wl, num_splits=splits)
    case.run_step()
    first = case.step.o_lat.clone()
    for _ in range(3):
        case.step.decode()
    torch.cuda.synchronize()
    assert torch.equal(first, case.step.o_lat)


@needs_cuda
@pytest.mark.parametrize("kernel", [M.MLA_KERNEL_SIMT, M.MLA_KERNEL_AUTO], ids=["simt", "auto"])
def test_bad_page_id_is_flagged_and_skipped(kernel):
    """A page id outside the pool sets MLA_DEV_INDEX_OUT_OF_RANGE; the other sequences'
    results are unaffected and nothing outside the pool is touched."""
    wl = SMALL_BF16
    case = Case(wl, kernel=kernel)
    case.run_step()
    good = case.step.o_lat.clone()
    bt = case.step.block_table.clone()
    bt[2, 0] = wl.num_pages + 5
    case.step.block_table.copy_(bt)
    case.step.dev_status.zero_()
    case.step.decode()
    torch.cuda.synchronize()
    assert case.step.status() & M.MLA_DEV_INDEX_OUT_OF_RANGE
    for b in (0, 1, 3):
        assert torch.equal(case.step.o_lat[b], good[b])


@needs_cuda
@pytest.mark.parametrize("kernel", [M.MLA_KERNEL_SIMT, M.MLA_KERNEL_AUTO], ids=["simt", "auto"])
def test_short_sequence_is_flagged(kernel):
    """seq_lens[b] < n_q cannot hold this step's tokens: MLA_DEV_BAD_SEQLEN."""
    wl = SMALL_BF16_MTP
    case = Case(wl, kernel=kernel)
    case.run_step()
    sl = case.step.seq_lens.clone()
    sl[0] = 1
    case.step.seq_lens.copy_(sl)
    case.step.dev_status.zero_()
    case.step.decode()
    torch.cuda.synchronize()
    assert case.step.status() & M.MLA_DEV_BAD_SEQLEN


@needs_cuda
def test_empty_batch_and_empty_token_lists_are_noops():
    wl = SMALL_BF16
    cfg = config_of(wl)
    z = torch.zeros(0, device="cuda")
    lib = M.lib()
    assert lib.mla_decode(cfg, None, None, None, 1, 1, None, 0, 1, 1, 0, None, 0, None, None, None, None) == 0
    assert lib.mla_append_cache(cfg, None, None, None, None, 0, None, 1, 1, 1, None, None, None) == 0
    assert lib.mla_unabsorb(cfg, None, 0, None, None, None) == 0
    assert z.numel() == 0


def _spike_case(wl, X, Y, pos):
    """Decode with q_lat = X e_0 for every row and head, after token `pos` of sequence 0 was
    appended again (through the library) with latent column 0 set to Y. The scores are then
    X c_n[0] / sqrt(192): N(0, (X/13.9)^2) nats for ordinary tokens and X Y / 13.9 for the
    spike. One split, so the spike falls in a later tile than the one that sets the tensor-core
    kernel's first reference."""
    case = Case(wl, num_splits=1)
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
            others = np.delete(X * ce["c"][:, 0] * tau, pos)
            jump = X * ce["c"][pos, 0] * tau - others.max()
        assert_close(wl, gpu_rows(case.step.o_lat, wl, b), ref_o, f"o_lat[b={b}]")
        assert_close(wl, gpu_rows(case.step.lse, wl, b), ref_lse, f"lse[b={b}]")
    return jump


@needs_cuda
@pytest.mark.parametrize("wl", [SMALL_BF16_LONG, SMALL_FP8_LONG], ids=["bf16", "fp8"])
def test_late_score_spike_matches_oracle(wl):
    """One cached token in a late tile scores ~30 nats above every earlier token
    (「deepseek(2)——deepseek 關鍵技術」 §1: the softmax is exact, whatever the spread). The
    tensor-core kernel's lagging reference absorbs it without clamping."""
    jump = _spike_case(wl, X=30.0, Y=17.0, pos=600)
    assert jump > 28.0


@needs_cuda
@pytest.mark.parametrize("wl", [SMALL_BF16_LONG, SMALL_FP8_LONG], ids=["bf16", "fp8"])
def test_score_spike_beyond_the_weight_range_matches_oracle(wl):
    """A token ~80 nats above the earlier tokens, far beyond the 2^96 weight range the lagging
    reference leaves (66.5 nats): the kernel clamps in its first pass, notices, and runs the
    unit again with the exact per-head maxima as the reference. The result must still be the
    oracle's."""
    jump = _spike_case(wl, X=30.0, Y=40.0, pos=600)
    assert jump > 75.0


@needs_cuda
@pytest.mark.parametrize("wl", [SMALL_BF16_LONG, SMALL_FP8_LONG, SMALL_BF16_LONG_MTP],
                         ids=["bf16", "fp8", "bf16-mtp"])
@pytest.mark.parametrize("kernel", [M.MLA_KERNEL_SIMT, M.MLA_KERNEL_AUTO], ids=["simt", "auto"])
def test_decode_wide_score_spread(wl, kernel):
    """Queries scaled by 10: the scaled scores of a row span more than 40 nats and the weights
    are close to one-hot; every head must still match the oracle."""
    case = Case(wl, kernel=kernel)
    case.step.append(case.new_c, case.new_r)
    q_lat = W.round_to_storage(wl.latent_queries() * np.float32(10.0), wl.act)
    case.step.decode(dev(q_lat.reshape(-1, wl.H, wl.C + wl.R), ACT[wl.act]))
    torch.cuda.synchronize()
    assert case.step.status() == 0
    tau = tau_of(wl)
    spread = 0.0
    for b in range(wl.B):
        ce = case.cache_of(b)
        ref_o, ref_lse = O.latent_attention(q_lat[b], ce["c"], ce["k_r"], wl.positions(b), tau)
        n = int(wl.positions(b)[-1]) + 1
        s = (q_lat[b, -1] @ np.concatenate([ce["c"], ce["k_r"]], axis=1)[:n].T) * tau
        spread = max(spread, float(np.max(s.max(axis=1) - s.min(axis=1))))
        assert_close(wl, gpu_rows(case.step.o_lat, wl, b), ref_o, f"o_lat[b={b}]")
        assert_close(wl, gpu_rows(case.step.lse, wl, b), ref_lse, f"lse[b={b}]")
    assert spread > 40.0


SMALL_FP8_GROUPS = W.small_v2(3, [300, 700, 64], n_q=2, cache="fp8", seed=19,
                              group_scales=(1.0, 1e-3, 1e-5, 1.0))


@needs_cuda
@pytest.mark.parametrize("kernel", [M.MLA_KERNEL_SIMT, M.MLA_KERNEL_AUTO], ids=["simt", "auto"])
def test_fp8_groups_far_below_unit_scale(kernel):
    """FP8 cache whose second and third 1x128 groups are drawn 1e-3 and 1e-5 times smaller
    (group scales amax/448 of about 8e-6 and 8e-8). Each group of o_lat is checked against the
    oracle at the usual tolerance scaled to that group's own magnitude, so a group whose scale
    lost precision, or flushed to zero, fails even though its values are tiny next to the
    others (「Deepseek系列从v3到R易背面经版」 F8量化策略: one scale per 1x128 group)."""
    wl = SMALL_FP8_GROUPS
    case = _decode_only(wl, kernel)
    tau = tau_of(wl)
    q_lat = wl.latent_queries()
    for b in range(wl.B):
        ce = case.cache_of(b)
        ref_o, _ = O.latent_attention(q_lat[b], ce["c"], ce["k_r"], wl.positions(b), tau)
        got = gpu_rows(case.step.o_lat, wl, b)
        for k, m in enumerate(wl.group_scales):
            cols = slice(128 * k, 128 * (k + 1))
            ref_g = ref_o[..., cols]
            err = float(np.max(np.abs(got[..., cols] - ref_g)))
            tol = 1e-2 * float(np.max(np.abs(ref_g))) + 1e-3 * m
            assert err <= tol, f"b={b} group {k} (x{m:g}): {err:.3e} > {tol:.3e}"


@needs_cuda
def test_bounded_wait_runs_out_and_the_next_call_is_exact():
    """The device-side failure path, made on purpose without a fault: through the test hook
    the even CTA of every pair never issues the loads of one latent chunk whose bytes it has
    registered, and every wait gives up after 2e5 cycles (about 0.1 ms) instead of about 2 s.
    The decode must return with MLA_DEV_TIMEOUT set, and the next ordinary call on the same
    stream must match the oracle (the context is still usable)."""
    wl = SMALL_BF16_LONG
    case = Case(wl, num_splits=1)
    case.step.append(case.new_c, case.new_r)
    assert M.mla_decode_kernel(case.cfg, wl.B, wl.n_q) == M.MLA_KERNEL_TC
    q_lat = wl.latent_queries()
    q_dev = dev(q_lat.reshape(-1, wl.H, wl.C + wl.R), ACT[wl.act])
    lib = M.lib()
    try:
        assert lib.mla_debug_decode_fault(200_000, 3) == 0
        case.step.dev_status.zero_()
        case.step.decode(q_dev)
        torch.cuda.synchronize()
        assert case.step.status() & M.MLA_DEV_TIMEOUT
    finally:
        assert lib.mla_debug_decode_fault(0, -1) == 0
    assert lib.mla_debug_decode_fault(-1, -1) == M.MLA_ERR_INVALID_ARG
    case.step.dev_status.zero_()
    case.step.decode(q_dev)
    torch.cuda.synchronize()
    assert case.step.status() == 0
    tau = tau_of(wl)
    for b in range(wl.B):
        ce = case.cache_of(b)
        ref_o, ref_lse = O.latent_attention(q_lat[b], ce["c"], ce["k_r"], wl.positions(b), tau)
        assert_close(wl, gpu_rows(case.step.o_lat, wl, b), ref_o, f"o_lat[b={b}]")
        assert_close(wl, gpu_rows(case.step.lse, wl, b), ref_lse, f"lse[b={b}]")


@needs_cuda
def test_yarn_long_context_step():
    """YaRN at long context (「一文通透DeepSeek-V2」 §3.1.3: 4K -> 128K, target 160K): a query
    near position 150K. Every head's o_lat and lse against the oracle's latent attention, and
    o of a few heads against the non-absorbed definition."""
    wl = LONG_YARN
    case = Case(wl)
    case.run_step()
    assert case.step.status() == 0
    heads = np.array([0, 63, 127])
    for b in range(wl.B):
        pos = wl.positions(b)
        ce = case.cache_of(b)
        q_lat = O.round_bf16(O.absorb_q(case.q_c_np[b], case.q_r_np[b], pos, case.w_uk_np, wl.rope_base,
                                        theta_of(wl)))
        ref_lat, ref_lse = O.latent_attention(q_lat, ce["c"], ce["k_r"], pos, tau_of(wl))
        assert_close(wl, gpu_rows(case.step.o_lat, wl, b), ref_lat, f"o_lat[b={b}]")
        assert_close(wl, gpu_rows(case.step.lse, wl, b), ref_lse, f"lse[b={b}]")
        o, _, _ = case.oracle(b, heads=heads)
        assert_close(wl, gpu_rows(case.step.o, wl, b)[:, heads], o, f"o[b={b}]")
