"""Pins for the fp64 oracle: values it must reproduce that do not come from itself.

Each test names the passage of the pages, or the mathematical fact, it checks.
Everything here runs on the CPU.
"""
import json
import math
import os
from decimal import Decimal, getcontext

import numpy as np
import pytest

from oracle import mla_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed=0):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- textbook case
def test_textbook_three_tokens_golden():
    """Hand-worked single-head case (tests/golden/textbook_three_tokens.json).

    With W_UK, W_UV selecting key / value halves, H = 1 and zero RoPE parts,
    MLA reduces to textbook causal attention with scale 1/sqrt(D + R).
    A scale of 1/sqrt(D) (the MHA one) would give other weights.
    """
    g = json.load(open(os.path.join(GOLDEN, "textbook_three_tokens.json")))
    c = np.array(g["c_kv"])
    w_uk = np.array(g["w_uk"])[None]
    w_uv = np.array(g["w_uv"])[None]
    q_c = np.array(g["q_c"])[None, None]
    q_r = np.zeros((1, 1, 2))
    k_r = np.zeros((3, 2))
    o, o_lat, lse = O.mla_decode_naive(c, k_r, q_c, q_r, w_uk, w_uv, np.array([2]), 10000.0)
    np.testing.assert_allclose(o[0, 0], g["o"], rtol=0, atol=1e-15)
    assert abs(lse[0, 0] - g["lse"]) < 1e-15
    # o_lat is the same weights applied to the latents themselves
    np.testing.assert_allclose(o_lat[0, 0], np.array(g["p"]) @ c, atol=1e-15)
    # position 1: the causal mask hides token 3
    o1, _, lse1 = O.mla_decode_naive(c, k_r, q_c, q_r, w_uk, w_uv, np.array([1]), 10000.0)
    np.testing.assert_allclose(o1[0, 0], [1 / 3, 2 / 3], atol=1e-15)
    assert abs(lse1[0, 0] - math.log(3)) < 1e-15


# ---------------------------------------------------------------- RoPE
def test_rope_closed_forms():
    """RoPE rotates pair k by pos * base^(-2k/R) (reading 1 of the oracle header)."""
    # R = 2: theta_0 = 1, so position p rotates (1, 0) to (cos p, sin p).
    for p in [0, 1, 2, 7, 1000, 131071]:
        y = O.apply_rope(np.array([1.0, 0.0]), np.int64(p), 10000.0)
        np.testing.assert_allclose(y, [math.cos(p), math.sin(p)], atol=1e-12)
    # R = 4, base = 10000: theta_1 = 10000^(-1/2) = 0.01, so position 100 turns pair 1 by 1 rad.
    y = O.apply_rope(np.array([0.0, 0.0, 0.0, 1.0]), np.int64(100), 10000.0)
    np.testing.assert_allclose(y, [0.0, 0.0, -math.sin(1.0), math.cos(1.0)], atol=1e-12)
    # position 0 is the identity
    x = _rng(1).standard_normal(64)
    np.testing.assert_array_equal(O.apply_rope(x, np.int64(0), 10000.0), x)


def test_rope_norm_and_relative_position():
    """Rotations keep the norm, and RoPE_m(q).RoPE_n(k) depends only on n - m
    (「一文通透DeepSeek-V2」 §2.2.2: S = R_m^T Q^T R_n K)."""
    g = _rng(2)
    q, k = g.standard_normal(64), g.standard_normal(64)
    for m in [0, 5, 4095, 131000]:
        qm = O.apply_rope(q, np.int64(m), 10000.0)
        assert abs(np.linalg.norm(qm) - np.linalg.norm(q)) < 1e-12
    d = 17
    ref = O.apply_rope(q, np.int64(3), 10000.0) @ O.apply_rope(k, np.int64(3 + d), 10000.0)
    for m in [0, 100, 4096, 65536]:
        v = O.apply_rope(q, np.int64(m), 10000.0) @ O.apply_rope(k, np.int64(m + d), 10000.0)
        assert abs(v - ref) < 1e-9


def test_decoupled_rope_shift_invariance():
    """Shifting every position by the same amount leaves MLA's output unchanged: the
    decoupled q^R/k^R carry only relative position (「一文通透DeepSeek-V2」 §2.2.2)."""
    g = _rng(3)
    H, D, C, R, L = 2, 8, 16, 4, 6
    c = g.standard_normal((L, C))
    k_r = g.standard_normal((L, R))
    q_c, q_r = g.standard_normal((1, H, D)), g.standard_normal((1, H, R))
    w_uk, w_uv = g.standard_normal((H, D, C)), g.standard_normal((H, D, C))
    o, o_lat, lse = O.mla_decode_naive(c, O.apply_rope(k_r, np.arange(L), 10000.0), q_c, q_r,
                                       w_uk, w_uv, np.array([L - 1]), 10000.0)
    for shift in [11, 5000, 131000]:
        # the same tokens cached at positions shift .. shift+L-1, queried from shift+L-1
        k_rot = O.apply_rope(k_r, np.arange(L) + shift, 10000.0)
        q_lat = O.absorb_q(q_c, q_r, np.array([L - 1 + shift]), w_uk, 10000.0)
        ol, ls = O.latent_attention(q_lat, c, k_rot, np.array([L - 1]), O.softmax_scale(D, R))
        np.testing.assert_allclose(ol, o_lat, rtol=1e-9, atol=1e-10)
        np.testing.assert_allclose(ls, lse, rtol=1e-9, atol=1e-10)
        np.testing.assert_allclose(O.unabsorb(ol, w_uv), o, rtol=1e-9, atol=1e-10)
    # and the RoPE part is not inert: dropping q^R changes the result
    o0, _, _ = O.mla_decode_naive(c, O.apply_rope(k_r, np.arange(L), 10000.0), q_c, 0 * q_r,
                                  w_uk, w_uv, np.array([L - 1]), 10000.0)
    assert np.max(np.abs(o0 - o)) > 1e-3


# ---------------------------------------------------------------- absorption
@pytest.mark.parametrize("n_q", [1, 2])
def test_absorbed_equals_naive(n_q):
    """Absorbing W^{UK} into the query and W^{UV} into the output is exact algebra
    (「一文通透DeepSeek-V2」 §2.2.1-2.2.2; 「Deepseek系列从v3到R易背面经版」 MLA)."""
    g = _rng(4)
    H, D, C, R, L = 3, 8, 24, 6, 9
    c = g.standard_normal((L, C))
    k_r = O.apply_rope(g.standard_normal((L, R)), np.arange(L), 10000.0)
    q_c, q_r = g.standard_normal((n_q, H, D)), g.standard_normal((n_q, H, R))
    w_uk, w_uv = g.standard_normal((H, D, C)) * 0.3, g.standard_normal((H, D, C)) * 0.3
    pos = np.arange(L - n_q, L)
    o, o_lat, lse = O.mla_decode_naive(c, k_r, q_c, q_r, w_uk, w_uv, pos, 10000.0)
    q_lat = np.stack([O.absorb_q(q_c[j][None], q_r[j][None], pos[j:j + 1], w_uk, 10000.0)[0]
                      for j in range(n_q)])
    o_lat2, lse2 = O.latent_attention(q_lat, c, k_r, pos, O.softmax_scale(D, R))
    o2 = O.unabsorb(o_lat2, w_uv)
    np.testing.assert_allclose(o_lat2, o_lat, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse2, lse, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(o2, o, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- softmax invariants
def test_softmax_rows_sum_to_one():
    """A latent column that is 1 for every token reads back sum_n p_n = 1."""
    g = _rng(5)
    H, D, C, R, L = 4, 8, 16, 4, 33
    c = g.standard_normal((L, C)) * 3
    c[:, 5] = 1.0
    k_r = g.standard_normal((L, R))
    q_lat = g.standard_normal((2, H, C + R)) * 2
    o_lat, _ = O.latent_attention(q_lat, c, k_r, np.array([L - 2, L - 1]), 0.2)
    np.testing.assert_allclose(o_lat[..., 5], 1.0, atol=1e-14)


def test_single_token_closed_form():
    """L = 1: the only weight is 1, so o_i = W^{UV}_i c_0. With W^{UV}_i = (i+1)[I | 0]
    that is (i+1) times the first D latent coordinates."""
    g = _rng(6)
    H, D, C, R = 3, 4, 8, 2
    c = g.standard_normal((1, C))
    w_uv = np.zeros((H, D, C))
    for i in range(H):
        w_uv[i, :, :D] = (i + 1) * np.eye(D)
    o, o_lat, lse = O.mla_decode_naive(c, g.standard_normal((1, R)), g.standard_normal((1, H, D)),
                                       g.standard_normal((1, H, R)), g.standard_normal((H, D, C)),
                                       w_uv, np.array([0]), 10000.0)
    for i in range(H):
        np.testing.assert_allclose(o[0, i], (i + 1) * c[0, :D], atol=1e-14)
        np.testing.assert_allclose(o_lat[0, i], c[0], atol=1e-14)


def test_zero_query_is_uniform_average():
    """q = 0 gives equal scores, so o is the plain mean of v^C over the visible tokens
    and lse = log(number of visible tokens)."""
    g = _rng(7)
    H, D, C, R, L = 2, 4, 8, 2, 7
    c = g.standard_normal((L, C))
    w_uv = g.standard_normal((H, D, C))
    o, o_lat, lse = O.mla_decode_naive(c, g.standard_normal((L, R)), np.zeros((1, H, D)),
                                       np.zeros((1, H, R)), g.standard_normal((H, D, C)), w_uv,
                                       np.array([4]), 10000.0)
    mean_c = c[:5].mean(axis=0)
    np.testing.assert_allclose(o_lat[0, 0], mean_c, atol=1e-14)
    for i in range(H):
        # mean of W c_n over n equals W (mean c): a property of the mean, not a retyped formula
        np.testing.assert_allclose(o[0, i], np.array([w_uv[i][d] @ mean_c for d in range(D)]),
                                   atol=1e-13)
    np.testing.assert_allclose(lse, math.log(5), atol=1e-14)


def test_mtp_causal_mask_between_new_tokens():
    """Two-token decode: query 0 must not see the last token, query 1 must."""
    g = _rng(8)
    H, D, C, R, L = 2, 4, 8, 2, 6
    c = g.standard_normal((L, C))
    k_r = g.standard_normal((L, R))
    args = (g.standard_normal((2, H, D)), g.standard_normal((2, H, R)),
            g.standard_normal((H, D, C)), g.standard_normal((H, D, C)), np.array([L - 2, L - 1]), 1e4)
    o, _, _ = O.mla_decode_naive(c, k_r, *args)
    c2, k2 = c.copy(), k_r.copy()
    c2[-1] += 5.0
    k2[-1] -= 3.0
    o2, _, _ = O.mla_decode_naive(c2, k2, *args)
    np.testing.assert_array_equal(o[0], o2[0])
    assert np.max(np.abs(o[1] - o2[1])) > 1e-3


# ---------------------------------------------------------------- brute force
def _brute_force_decimal(c, k_r_rot, q_c, q_r, w_uk, w_uv, pos, base):
    """Pure-Python loops at 50 significant digits (RoPE angles via math.cos/sin)."""
    getcontext().prec = 50
    n_q, H, D = q_c.shape
    R = q_r.shape[-1]
    C = c.shape[1]
    tau = Decimal(1) / Decimal(D + R).sqrt()
    out = np.zeros((n_q, H, D))
    lses = np.zeros((n_q, H))
    for j in range(n_q):
        for i in range(H):
            qr = []
            for k in range(R // 2):
                ang = float(pos[j]) * float(base) ** (-2.0 * k / R)
                a, b = float(q_r[j, i, 2 * k]), float(q_r[j, i, 2 * k + 1])
                qr += [a * math.cos(ang) - b * math.sin(ang), a * math.sin(ang) + b * math.cos(ang)]
            scores = []
            for n in range(int(pos[j]) + 1):
                s = Decimal(0)
                for d in range(D):
                    kd = sum(Decimal(float(w_uk[i, d, x])) * Decimal(float(c[n, x])) for x in range(C))
                    s += Decimal(float(q_c[j, i, d])) * kd
                for r in range(R):
                    s += Decimal(qr[r]) * Decimal(float(k_r_rot[n, r]))
                scores.append(s * tau)
            mx = max(scores)
            ex = [(s - mx).exp() for s in scores]
            z = sum(ex)
            for d in range(D):
                acc = Decimal(0)
                for n, e in enumerate(ex):
                    v = sum(Decimal(float(w_uv[i, d, x])) * Decimal(float(c[n, x])) for x in range(C))
                    acc += e / z * v
                out[j, i, d] = float(acc)
            lses[j, i] = float(mx + z.ln())
    return out, lses


@pytest.mark.parametrize("H,L,n_q", [(1, 1, 1), (2, 3, 1), (2, 4, 2), (1, 4, 2)])
def test_brute_force_tiny(H, L, n_q):
    g = _rng(100 + H * 10 + L)
    D, C, R = 3, 5, 4
    c = g.standard_normal((L, C))
    k_r = O.apply_rope(g.standard_normal((L, R)), np.arange(L), 10000.0)
    q_c, q_r = g.standard_normal((n_q, H, D)), g.standard_normal((n_q, H, R))
    w_uk, w_uv = g.standard_normal((H, D, C)), g.standard_normal((H, D, C))
    pos = np.arange(L - n_q, L)
    o, _, lse = O.mla_decode_naive(c, k_r, q_c, q_r, w_uk, w_uv, pos, 10000.0)
    o_bf, lse_bf = _brute_force_decimal(c, k_r, q_c, q_r, w_uk, w_uv, pos, 10000.0)
    np.testing.assert_allclose(o, o_bf, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, lse_bf, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- split-KV combine
def test_combine_of_ranges_equals_whole():
    """Attention over disjoint token ranges merged by log-sum-exp weights equals
    attention over the union (exact algebra of softmax normalisation)."""
    g = _rng(9)
    H, C, R, L = 4, 16, 4, 40
    c = g.standard_normal((L, C))
    k_r = g.standard_normal((L, R))
    q_lat = g.standard_normal((1, H, C + R))
    pos = np.array([L - 1])
    whole, lse_whole = O.latent_attention(q_lat, c, k_r, pos, 0.3)
    cuts = [0, 7, 8, 25, 40]
    parts, lses = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        ol, ls = O.latent_attention(q_lat, c[a:b], k_r[a:b], np.array([b - a - 1]), 0.3)
        parts.append(ol)
        lses.append(ls)
    # an empty range contributes lse = -inf and must carry no weight
    parts.append(np.full_like(parts[0], 123.0))
    lses.append(np.full_like(lses[0], -np.inf))
    o, lse = O.combine_partials(np.stack(parts), np.stack(lses))
    np.testing.assert_allclose(o, whole, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, lse_whole, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- cache sizes
def test_cache_size_counts():
    """MHA caches 2 n_h d_h l elements per token (「一文通透DeepSeek-V2」 §2.1.2); MLA caches
    (d_c + d_h^R) l (§2.2.2); with d_c = 4 d_h and d_h^R = d_h/2 that equals GQA with 2.25
    groups (§2.2.2, last paragraph). V2 sizes from §3.1.1."""
    n_h, d_h, d_c, d_r, layers = 128, 128, 512, 64, 60
    assert O.mha_cache_elements(n_h, d_h, 1) == 32768
    assert O.mla_cache_elements(d_c, d_r, 1) == 576
    assert d_c == 4 * d_h and d_r == d_h // 2
    assert O.mla_cache_elements(d_c, d_r, layers) == O.gqa_cache_elements(2.25, d_h, layers)
    assert O.mla_cache_elements(4 * 64, 32, 1) == 4.5 * 64
    # 576 / 32768 = 1.7578 %
    assert abs(O.mla_cache_elements(d_c, d_r, 1) / O.mha_cache_elements(n_h, d_h, 1) - 0.017578125) < 1e-15


# ---------------------------------------------------------------- FP8 E4M3
def test_e4m3_table_points():
    """Points of the E4M3 format fixed by its definition (1 sign, 4 exponent bits with
    bias 7, 3 mantissa bits, no infinity, S.1111.111 = NaN)."""
    v = O.e4m3_values()
    assert v[0x7E] == 448.0 and v[0xFE] == -448.0
    assert v[0x38] == 1.0 and v[0x08] == 2.0 ** -6 and v[0x01] == 2.0 ** -9
    assert v[0x07] == 7 / 8 * 2.0 ** -6
    assert v[0x00] == 0.0 and math.isnan(v[0x7F]) and math.isnan(v[0xFF])
    assert v[0x40] == 2.0 and v[0x3C] == 1.5 and v[0x78] == 256.0


def test_e4m3_table_matches_independent_decoder():
    """Cross-check every code against torch's float8_e4m3fn decoder (an independent
    implementation of the same format)."""
    torch = pytest.importorskip("torch")
    codes = np.arange(256, dtype=np.uint8)
    t = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    v = O.e4m3_values()
    assert np.all((t == v) | (np.isnan(t) & np.isnan(v)))


def test_e4m3_encode_rounding():
    v = O.e4m3_values()
    finite = [c for c in range(256) if not math.isnan(v[c])]
    # every finite code round-trips (negative zero included)
    enc = O.e4m3_encode(np.array([v[c] for c in finite], dtype=np.float32))
    dec = O.e4m3_decode(enc)
    np.testing.assert_array_equal(dec, [v[c] for c in finite])
    # ties go to the even mantissa: 1.0625 lies halfway between 1.0 (0x38) and 1.125 (0x39)
    assert O.e4m3_encode(np.float32(1.0625)) == 0x38
    assert O.e4m3_encode(np.float32(1.1875)) == 0x3A      # between 0x39 and 0x3A -> 0x3A
    assert O.e4m3_encode(np.float32(2.0 ** -10)) == 0x00  # half the smallest subnormal -> 0
    assert O.e4m3_encode(np.float32(3 * 2.0 ** -10)) == 0x02
    # saturation
    assert O.e4m3_encode(np.float32(1000.0)) == 0x7E
    assert O.e4m3_encode(np.float32(-460.0)) == 0xFE
    assert O.e4m3_encode(np.float32(447.9)) == 0x7E


def test_e4m3_encode_matches_independent_encoder():
    """In-range values: compare with torch's float -> float8_e4m3fn conversion."""
    torch = pytest.importorskip("torch")
    x = (_rng(10).standard_normal(200000) * 60).astype(np.float32)
    x = np.clip(x, -448, 448)
    x[:1000] = x[:1000] * 1e-4  # subnormal range
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(O.e4m3_encode(x), ref)


def test_fp8_group_quantiser():
    """1x128 groups per token (「Deepseek系列从v3到R易背面经版」 F8量化策略 (1)): each group's
    largest magnitude lands on 448, and dequantised values are within half a mantissa step
    (2^-4 relative) of the input in the normal range."""
    g = _rng(11)
    c = g.standard_normal((37, 512)).astype(np.float32)
    c[3, 128:256] = 0.0  # an all-zero group gets scale 1
    codes, scales = O.quantize_fp8_groups(c)
    assert codes.shape == (37, 512) and scales.shape == (37, 4)
    assert scales[3, 1] == 1.0 and np.all(codes[3, 128:256] == 0)
    deq = O.dequantize_fp8_groups(codes, scales)
    grp = np.abs(c.reshape(37, 4, 128)).max(-1)
    # the element holding each group's max encodes as +-448 (code 0x7E / 0xFE)
    for n in range(37):
        for k in range(4):
            if grp[n, k] > 0:
                idx = k * 128 + int(np.argmax(np.abs(c[n, k * 128:(k + 1) * 128])))
                assert codes[n, idx] & 0x7F == 0x7E
    big = np.abs(c) >= (scales.repeat(128, axis=1) * 2.0 ** -6)
    rel = np.abs(deq - c)[big] / np.abs(c)[big]
    assert rel.max() <= 2.0 ** -4 + 1e-7


def test_query_quantiser_against_torch_codec():
    """FP8 scores (reading 8): q_lat's latent part is quantised per (row, head) in 1x128
    groups. The codes equal torch's independent float -> float8_e4m3fn conversion of the
    fp32 quotient by the group scale, the scale is the group's amax / 448 in fp32, and the
    RoPE part passes through untouched."""
    torch = pytest.importorskip("torch")
    g = _rng(12)
    q = g.standard_normal((3, 5, 576)).astype(np.float32) * np.float32(0.15)
    q[1, 2, 256:384] = 0.0            # an all-zero group: scale 1, codes 0
    q8, codes, scales = O.quantize_q_latent(q, 512)
    assert codes.shape == (3, 5, 512) and scales.shape == (3, 5, 4)
    grp = q[..., :512].reshape(3, 5, 4, 128)
    amax = np.abs(grp).max(-1)
    np.testing.assert_array_equal(scales, np.where(amax > 0, amax / np.float32(448.0), 1.0).astype(np.float32))
    quot = (grp / scales[..., None]).astype(np.float32)
    ref = torch.from_numpy(np.ascontiguousarray(quot)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(codes, ref.reshape(3, 5, 512))
    np.testing.assert_array_equal(q8[..., 512:], q[..., 512:].astype(np.float64))
    back = torch.from_numpy(ref).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(q8[..., :512], (back * scales[..., None]).reshape(3, 5, 512))


def test_query_quantiser_is_exact_on_representable_groups():
    """A group whose values are E4M3 values times a power of two, with its largest magnitude
    at 448 times that power, quantises without error (scale = the power of two exactly), so
    the FP8 scores equal the exact scores; a general group moves by at most half an E4M3
    step (2^-4 relative) per element."""
    vals = O.e4m3_values()
    fin = vals[np.isfinite(vals) & (np.abs(vals) <= 448)]
    g = _rng(13)
    grp = g.choice(fin, size=(2, 128))
    grp[:, 0] = 448.0
    grp *= np.array([[2.0 ** -5], [2.0 ** 3]])
    q = np.zeros((2, 576))
    q[:, :128] = grp
    q[:, 128:512] = g.standard_normal((2, 384))
    q8, _, scales = O.quantize_q_latent(q, 512)
    assert scales[0, 0] == 2.0 ** -5 and scales[1, 0] == 2.0 ** 3
    np.testing.assert_array_equal(q8[:, :128], grp)
    rel = np.abs(q8[:, 128:512] - q[:, 128:512]) / np.abs(q[:, 128:512])
    big = np.abs(q[:, 128:512]) >= np.repeat(scales[:, 1:], 128, axis=1) * 2.0 ** -6
    assert rel[big].max() <= 2.0 ** -4 + 1e-7


# ---------------------------------------------------------------- page / slot mapping
def test_page_slot_mapping():
    bt = np.array([[5, 2, -1], [0, 4, 1]], dtype=np.int32)
    pg, sl = O.page_slots(np.array([0, 0, 1, 1, 1]), np.array([0, 17, 15, 16, 40]), bt, 16)
    np.testing.assert_array_equal(pg, [5, 2, 0, 4, 1])
    np.testing.assert_array_equal(sl, [0, 1, 15, 0, 8])


# ---------------------------------------------------------------- storage rounding
def _torch_bf16(x_f32: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 -> fp64 through torch's own conversion (an implementation independent of
    the oracle's bit arithmetic)."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x_f32, dtype=np.float32))
    return t.to(torch.bfloat16).to(torch.float64).numpy()


def test_round_bf16_matches_an_independent_rounding():
    """round_bf16 is round-to-nearest-even from fp32 to bf16, the rounding every bf16 value of
    the cache and of the activations goes through. Checked against torch's converter on random
    fp32 values over a wide exponent range, both signs."""
    g = _rng(40)
    x = (g.standard_normal(200_000) * np.exp2(g.integers(-60, 60, 200_000))).astype(np.float32)
    np.testing.assert_array_equal(O.round_bf16(x.astype(np.float64)), _torch_bf16(x))


def test_round_bf16_ties_go_to_even():
    """Exact halfway cases: the fp32 value's 16 dropped bits are exactly 0x8000. bf16 keeps 7
    stored mantissa bits, so 1 + 2^-8 lies halfway between 1 and 1 + 2^-7 (keeps the even 1),
    and 1 + 3 * 2^-8 halfway between 1 + 2^-7 and 1 + 2^-6 (keeps the even 1 + 2^-6). One ulp
    of fp32 to either side of a tie is not a tie. Worked by hand, then the same constructed
    ties checked against torch over many exponents and mantissas."""
    assert O.round_bf16(np.array([1 + 2.0 ** -8]))[0] == 1.0
    assert O.round_bf16(np.array([1 + 3 * 2.0 ** -8]))[0] == 1 + 2.0 ** -6
    assert O.round_bf16(np.array([-(1 + 2.0 ** -8)]))[0] == -1.0
    assert O.round_bf16(np.array([1 + 2.0 ** -8 + 2.0 ** -23]))[0] == 1 + 2.0 ** -7
    assert O.round_bf16(np.array([1 + 2.0 ** -8 - 2.0 ** -23]))[0] == 1.0
    # a value that fp64 -> fp32 rounding moves onto a tie is rounded as the fp32 value says
    assert O.round_bf16(np.array([1 + 2.0 ** -8 + 2.0 ** -40]))[0] == 1.0
    g = _rng(41)
    hi = g.integers(0, 1 << 16, 50_000, dtype=np.uint64) & np.uint64(0x7F7F)   # finite, any mantissa parity
    bits = ((hi << np.uint64(16)) | np.uint64(0x8000)).astype(np.uint32)
    ties = bits.view(np.float32)
    got = O.round_bf16(ties.astype(np.float64))
    np.testing.assert_array_equal(got, _torch_bf16(ties))
    # every tie went to the neighbour whose last kept bit is 0
    kept = (got.astype(np.float32).view(np.uint32) >> np.uint32(16)) & np.uint32(1)
    assert not kept[np.abs(got) > 0].any()


def test_cache_entries_hand_worked():
    """What the cache holds for a token (「一文通透DeepSeek-V2」 §2.2.2: k^R_t = RoPE(W^{KR}h_t)
    is cached, rotated at the token's own position, beside c^{KV}_t), worked by hand for
    R = 4, base 10000 (theta_0 = 1, theta_1 = 0.01) at positions 0, 1 and 100.

    bf16 and fp32 caches: c is the stored value of c^{KV}; k^R = (x0 cos a0 - x1 sin a0,
    x0 sin a0 + x1 cos a0, x2 cos a1 - x3 sin a1, x2 sin a1 + x3 cos a1) with a0 = pos,
    a1 = 0.01 pos, then rounded to the cache's storage type."""
    c = np.array([[0.5, -1.25, 3.0, 0.0]] * 3)
    k = np.array([[1.0, 2.0, -0.5, 0.25]] * 3)
    pos = np.array([0, 1, 100])
    expect = []
    for p in pos:
        a0, a1 = float(p), 0.01 * float(p)
        expect.append([1.0 * math.cos(a0) - 2.0 * math.sin(a0), 1.0 * math.sin(a0) + 2.0 * math.cos(a0),
                       -0.5 * math.cos(a1) - 0.25 * math.sin(a1), -0.5 * math.sin(a1) + 0.25 * math.cos(a1)])
    expect = np.array(expect)
    bf = O.cache_entries(c, k, pos, "bf16", 10000.0)
    np.testing.assert_array_equal(bf["c"], c)                       # exact in bf16
    np.testing.assert_array_equal(bf["k_r"], _torch_bf16(expect.astype(np.float32)))
    np.testing.assert_array_equal(bf["k_r"][0], [1.0, 2.0, -0.5, 0.25])   # position 0: identity
    f32 = O.cache_entries(c, k, pos, "f32", 10000.0)
    np.testing.assert_allclose(f32["k_r"], expect, rtol=2.0 ** -23, atol=0)
    assert f32["k_r"].dtype == np.float64 and np.all(f32["k_r"] == f32["k_r"].astype(np.float32))


def test_cache_entries_fp8_group_hand_worked():
    """One 1x128 group quantised by hand (「Deepseek系列从v3到R易背面经版」 F8量化策略).

    Group x = (1, -2, 0.5, 3, 0, ..., 0): amax = 3, scale = 3/448. x / scale = 149.33, -298.67,
    74.67, 448, 0. E4M3 spacing is 16 on [128, 256), 32 on [256, 448], 8 on [64, 128):
    149.33 -> 144 = 1.125 * 2^7 (code 0 1110 001 = 0x71); -298.67 -> -288 = -1.125 * 2^8
    (1 1111 001 = 0xF9); 74.67 -> 72 = 1.125 * 2^6 (0 1101 001 = 0x69); 448 = 1.75 * 2^8
    (0 1111 110 = 0x7E). The cache then reads code value * scale. The second group is all
    zeros: scale 1, every code 0. k^R stays bf16."""
    C = 256
    c = np.zeros((1, C))
    c[0, :4] = [1.0, -2.0, 0.5, 3.0]
    k = np.array([[1.0, 2.0, -0.5, 0.25]])
    e = O.cache_entries(c, k, np.array([0]), "fp8", 10000.0)
    scale = np.float32(3.0) / np.float32(448.0)
    np.testing.assert_array_equal(e["scales"][0], [scale, np.float32(1.0)])
    codes = np.zeros(C, dtype=np.uint8)
    codes[:4] = [0x71, 0xF9, 0x69, 0x7E]
    np.testing.assert_array_equal(e["codes"][0], codes)
    want = np.zeros(C)
    want[:4] = np.array([144.0, -288.0, 72.0, 448.0]) * float(scale)
    np.testing.assert_array_equal(e["c"][0], want)
    np.testing.assert_array_equal(e["k_r"][0], [1.0, 2.0, -0.5, 0.25])


# ---------------------------------------------------------------- YaRN (§3.1.3)
YARN = dict(s=40.0, alpha=1.0, beta=32.0, orig_context=4096)   # 「一文通透DeepSeek-V2」 §3.1.3


def test_yarn_reduces_to_plain_rope_at_scale_one():
    """s = 1 extends nothing: every frequency is base^(-2k/R) and the logit factor is 1."""
    np.testing.assert_allclose(O.yarn_theta(64, 10000.0, 1.0), O.rope_theta(64, 10000.0), rtol=1e-15, atol=0)
    assert O.yarn_attention_factor(1.0) == 1.0


def test_yarn_ramp_ends_hand_counted():
    """V2's decoupled RoPE (R = 64, base 10000) with the page's s = 40, alpha = 1, beta = 32
    over a 4096-token original context. Worked by hand: pair k keeps its frequency while
    4096 theta_k / 2pi > 32, i.e. k < 32 ln(4096 / 64pi) / ln 10000 = 10.47, so k = 0..10;
    it is divided by s while 4096 theta_k / 2pi < 1, i.e. k > 32 ln(4096 / 2pi) / ln 10000
    = 22.51, so k = 23..31; the 12 pairs between move part of the way."""
    th = O.rope_theta(64, 10000.0)
    y = O.yarn_theta(64, 10000.0, **YARN)
    np.testing.assert_array_equal(y[:11], th[:11])
    np.testing.assert_allclose(y[23:], th[23:] / 40.0, rtol=1e-15, atol=0)
    mid = y[11:23] / th[11:23]
    assert np.all((mid < 1.0) & (mid > 1.0 / 40.0))
    # the ratio falls monotonically from 1 to 1/s, and the frequencies stay ordered
    ratio = y / th
    assert np.all(np.diff(ratio) <= 1e-15) and np.all(np.diff(y) < 0)


def test_yarn_hand_worked_middle_pair():
    """Pair k = 16 of the same setting, by hand: theta = 10000^(-1/2) = 0.01, wavelength
    2pi / 0.01 = 628.3185, r = 4096 / 628.3185 = 6.51897, gamma = (6.51897 - 1) / 31 =
    0.178031, new theta = 0.01 ((1 - 0.178031) / 40 + 0.178031) = 0.00198580."""
    y = O.yarn_theta(64, 10000.0, **YARN)
    assert abs(y[16] - 0.00198580) < 2e-8


def test_yarn_attention_factor_value():
    """sqrt(t) = 0.0707 ln 40 + 1 = 0.0707 * 3.688879 + 1 = 1.260804, t = 1.589627."""
    assert abs(O.yarn_attention_factor(40.0) - 1.589627) < 2e-6


def test_yarn_keeps_the_relative_position_property():
    """With the interpolated frequencies on both sides, RoPE_m(q) . RoPE_n(k) still depends
    only on n - m (what lets the decoupled key be cached rotated), at positions up to 160K."""
    g = _rng(42)
    q, k = g.standard_normal(64), g.standard_normal(64)
    th = O.yarn_theta(64, 10000.0, **YARN)
    d = 1234
    ref = O.apply_rope(q, np.int64(0), 10000.0, th) @ O.apply_rope(k, np.int64(d), 10000.0, th)
    for m in [1, 4096, 100000, 160000 - d]:
        v = O.apply_rope(q, np.int64(m), 10000.0, th) @ O.apply_rope(k, np.int64(m + d), 10000.0, th)
        assert abs(v - ref) < 1e-8


def test_yarn_absorbed_equals_naive():
    """The absorbed path with YaRN frequencies and the scaled logits equals the naive form."""
    g = _rng(43)
    H, D, C, R, L = 3, 8, 16, 8, 40
    c = g.standard_normal((L, C))
    k_r = g.standard_normal((L, R))
    w_uk, w_uv = g.standard_normal((2, H, D, C)) * 0.3
    q_c, q_r = g.standard_normal((1, H, D)), g.standard_normal((1, H, R))
    th = O.yarn_theta(R, 10000.0, 40.0, 1.0, 32.0, 16)
    tau = O.softmax_scale(D, R) * O.yarn_attention_factor(40.0)
    pos = np.array([L - 1])
    ce = O.cache_entries(c, k_r, np.arange(L), "f32", 10000.0, th)
    o, o_lat, lse = O.mla_decode_naive(ce["c"], ce["k_r"], q_c, q_r, w_uk, w_uv, pos, 10000.0,
                                        theta=th, scale=tau)
    q_lat = O.absorb_q(q_c, q_r, pos, w_uk, 10000.0, th)
    o_lat2, lse2 = O.latent_attention(q_lat, ce["c"], ce["k_r"], pos, tau)
    np.testing.assert_allclose(o_lat2[0], o_lat[0], atol=1e-12)
    np.testing.assert_allclose(O.unabsorb(o_lat2, w_uv)[0], o[0], atol=1e-12)
    np.testing.assert_allclose(lse2[0], lse[0], atol=1e-12)


# ---------------------------------------------------------------- upstream / downstream
def test_rms_norm_closed_forms():
    """RMSNorm of the compressed latent (「一文通透DeepSeek-V2」 §3.1.4), eps = 0 here:
    x = (3, 4) has mean square 12.5, so it maps to (3, 4) / sqrt(12.5) = (0.848528, 1.131371);
    a gain multiplies elementwise; the output's root mean square is the gain's magnitude; a
    positive factor on the input changes nothing."""
    np.testing.assert_allclose(O.rms_norm(np.array([3.0, 4.0]), np.ones(2), eps=0.0),
                               [0.848528137423857, 1.131370849898476], rtol=1e-14)
    np.testing.assert_allclose(O.rms_norm(np.array([3.0, 4.0]), np.array([2.0, -1.0]), eps=0.0),
                               [1.697056274847714, -1.131370849898476], rtol=1e-14)
    g = _rng(50)
    x = g.standard_normal((5, 512))
    y = O.rms_norm(x, np.full(512, 0.7), eps=0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=-1)), 0.7, rtol=1e-13)
    np.testing.assert_allclose(O.rms_norm(37.5 * x, np.ones(512), eps=0.0), O.rms_norm(x, np.ones(512), eps=0.0), rtol=1e-13)
    # eps bounds the gain on tiny inputs: x * g / sqrt(eps) when mean(x^2) << eps
    t = np.full(4, 1e-9)
    np.testing.assert_allclose(O.rms_norm(t, np.ones(4), eps=1e-6), t / 1e-3, rtol=1e-6)


def test_project_latent_selects_and_normalises():
    """c^{KV} = RMSNorm(W^{DKV} h), k^R = W^{KR} h (「deepseek(2)——deepseek 關鍵技術」 §1,
    「一文通透DeepSeek-V2」 §2.2.1-2.2.2): with W^{DKV} and W^{KR} selecting disjoint slices of
    h, the latent is the normalised first slice and k^R the raw second one."""
    g = _rng(51)
    d, C, R = 40, 16, 8
    h = g.standard_normal((3, d))
    w_dkv = np.zeros((C, d)); w_dkv[:, :C] = np.eye(C)
    w_kr = np.zeros((R, d)); w_kr[:, C:C + R] = np.eye(R)
    gain = g.uniform(0.5, 1.5, C)
    c, k = O.project_latent(h, w_dkv, w_kr, gain)
    np.testing.assert_allclose(c, O.rms_norm(h[:, :C], gain), rtol=1e-14)
    np.testing.assert_array_equal(k, h[:, C:C + R])


def test_output_projection_hand_worked():
    """u_t = W^O [o_{t,1}; o_{t,2}] with n_h = 2, d_h = 2, d = 3, worked by hand:
    o = ((1, 2), (3, 4)) concatenates to (1, 2, 3, 4); the rows of W^O pick element 1,
    element 3 and the sum: u = (1, 3, 10). It also equals the per-head sum
    sum_i W^O[:, i d_h:(i+1) d_h] o_{t,i}."""
    o = np.array([[[1.0, 2.0], [3.0, 4.0]]])
    w_o = np.array([[1.0, 0, 0, 0], [0, 0, 1.0, 0], [1.0, 1.0, 1.0, 1.0]])
    np.testing.assert_array_equal(O.output_projection(o, w_o), [[1.0, 3.0, 10.0]])
    g = _rng(52)
    o = g.standard_normal((4, 3, 5))
    w_o = g.standard_normal((7, 15))
    per_head = sum(o[:, i] @ w_o[:, 5 * i:5 * (i + 1)].T for i in range(3))
    np.testing.assert_allclose(O.output_projection(o, w_o), per_head, rtol=1e-13, atol=1e-13)


def test_prefill_is_causal_attention_over_the_prompt():
    """The non-absorbed prefill path (「一文通透DeepSeek-V2」 §2.2.1: the naive formula restores
    k^C, v^C from the cached latent) is the naive decode with every prompt position as a query:
    query t sees tokens 0..t. Checked against one-query decodes at each position."""
    g = _rng(53)
    H, D, C, R, L = 2, 4, 8, 4, 6
    c, k_r = g.standard_normal((L, C)), g.standard_normal((L, R))
    w_uk, w_uv = g.standard_normal((2, H, D, C)) * 0.5
    q_c, q_r = g.standard_normal((L, H, D)), g.standard_normal((L, H, R))
    ce = O.cache_entries(c, k_r, np.arange(L), "f32", 10000.0)
    o, o_lat, lse = O.mla_decode_naive(ce["c"], ce["k_r"], q_c, q_r, w_uk, w_uv, np.arange(L), 10000.0)
    for t in range(L):
        o1, _, lse1 = O.mla_decode_naive(ce["c"][:t + 1], ce["k_r"][:t + 1], q_c[t:t + 1], q_r[t:t + 1],
                                          w_uk, w_uv, np.array([t]), 10000.0)
        np.testing.assert_allclose(o[t], o1[0], atol=1e-13)
        np.testing.assert_allclose(lse[t], lse1[0], atol=1e-13)
    # the first token attends to itself only
    np.testing.assert_allclose(o[0], np.einsum("hdc,c->hd", w_uv, ce["c"][0]), atol=1e-13)
