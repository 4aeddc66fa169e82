"""fp64 CPU oracle for DeepSeek-V2 Multi-head Latent Attention (MLA) decode.

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module. The CUDA library
never calls it and shares no code with it.

What it computes, and where the pages define it
-----------------------------------------------
Sources are five web pages on DeepSeek-V2; they are cited by title:

* [V2-explainer]  「一文通透DeepSeek-V2(改造Transformer的中文模型)」,
  community.sslcode.com.cn — §2.1.1 (causal masked attention), §2.1.2 (MHA and
  its 2·n_h·d_h·l cache), §2.2.1 (low-rank joint KV compression, absorption),
  §2.2.2 (decoupled RoPE, the (d_c + d_h^R)·l cache), §3.1.1 (V2 sizes).
* [key-tech]  「deepseek(2)——deepseek 關鍵技術」, hk.pswp.cn — §1 MLA, the
  equations for k_{t,i} = [k^C_{t,i}; k^R_t], q_{t,i} = [q^C_{t,i}; q^R_{t,i}]
  and o_{t,i} with the 1/sqrt(d_h + d_h^R) softmax scale.
* [v3-notes]  「Deepseek系列从v3到R易背面经版」, www.coreui.cn — "MLA"
  (W^{UK} fused into the query side turns MHA into MQA) and "F8量化策略"
  (E4M3, per-token 1x128 activation groups).
* [V2-explainer] §3.1.3 (长上下文扩展): YaRN on the decoupled RoPE for the 4K -> 128K
  extension, scale s = 40, alpha = 1, beta = 32, target 160K, and a length factor
  sqrt(t) = 0.0707 ln s + 1 that regulates the attention entropy.

The reference function ``mla_decode_naive`` is the plain, non-absorbed
definition: it decompresses k^C = W^{UK} c and v^C = W^{UV} c for every cached
token and every head and runs textbook causal softmax attention. The
absorbed-form steps (``absorb_q``, ``latent_attention``, ``unabsorb``,
``combine_partials``) restate the GPU path's step boundaries in plain fp64 so
each step can be checked on its own; the tests pin them to the naive form.

Readings where the pages are silent or garbled (each is also listed in the
design notes):

1. RoPE form: rotation matrices R_m are named ([V2-explainer] §2.2.2) but not
   spelled out. Reading: block-diagonal 2x2 rotations of interleaved pairs
   (x_{2k}, x_{2k+1}) by the angle pos * base^(-2k/d_h^R), base 10000.
2. Softmax scale: 1/sqrt(d_h + d_h^R) ([key-tech] §1), not the MHA 1/sqrt(d_h).
3. Positions: seq_len counts the cached tokens including this step's n_q new
   ones; query j sits at position seq_len - n_q + j and sees tokens 0..pos
   (causal mask of [V2-explainer] §2.1.1; two-token MTP decode masks the two
   new tokens causally against each other).
4. Cache contents: the stored k^R is RoPE(k_R) at the token's position,
   rounded to the cache's storage type; an FP8 cache stores c_KV as E4M3 codes
   with one fp32 scale per 128-element group, scale = amax/448 (fp32, IEEE
   division), scale = 1 for an all-zero group, code = E4M3(x / scale) with
   round-to-nearest-even and saturation; the cached value is code * scale.
5. W^{UK}, W^{UV} in R^{(n_h d_h) x d_c} are held as [H][D][C]: head i owns
   rows i*D .. i*D + D - 1.
6. YaRN ([V2-explainer] §3.1.3 names the method and its parameters but not its
   formula). Reading, the published "by parts" interpolation: for RoPE pair k with
   frequency theta_k and wavelength lambda_k = 2 pi / theta_k, r_k = L / lambda_k with L
   the original context (4096: the 4K the extension starts from; 4096 s = 160K is the
   target the page names); gamma_k = clip((r_k - alpha) / (beta - alpha), 0, 1); the new
   frequency is (1 - gamma_k) theta_k / s + gamma_k theta_k. q^R and k^R both rotate by
   it (the relative-position property needs the same frequencies on both sides). The
   factor sqrt(t) multiplies q and k alike, so every logit is scaled by t = sqrt(t)^2.
7. The latent's RMSNorm ([V2-explainer] §3.1.4: an extra RMSNorm after the compressed
   latent, and extra scaling factors at the width bottlenecks). Reading: c^{KV} =
   g * x / sqrt(mean(x^2) + eps) with x = W^{DKV} h, a learned gain g per latent
   dimension that also carries the bottleneck's scaling factor, eps = 1e-6 (not on the
   pages); k^R = W^{KR} h is not normalised. The projected c^{KV} and k^R are stored in
   the activation type before they are cached, as when the projection and the cache
   write are separate calls.
8. FP8 scores ([v3-notes] F8量化策略: E4M3 operands with 1x128 activation groups, partial
   sums promoted to fp32 every 128 products). Reading for the decode's scores over an FP8
   cache: q_lat's latent part (its first d_c dims) is quantised per (query row, head) in
   1x128 groups exactly as the cache's c_KV is (reading 4); each group's product of codes is
   scaled by the two groups' scales and summed in fp32, and the bf16 RoPE part is added as
   in the bf16 path. The exact value of that sum is q8 . [c; k^R] with q8 = q_lat whose
   latent part is replaced by code * scale, which is what ``quantize_q_latent`` returns; the
   softmax and P . V are unchanged.

Parity status: every function here is pinned by tests/test_oracle.py
(closed forms, special cases, brute force in 50-digit decimal arithmetic,
the absorbed/naive equivalence, invariants, and a cross-check of the E4M3
table against an independent library decoder). No function is unpinned.
"""
from __future__ import annotations

import math
from typing import Optional, Tuple

import numpy as np

E4M3_MAX = 448.0
FP8_GROUP = 128


# --------------------------------------------------------------------------
# Decoupled RoPE  ([V2-explainer] §2.2.2; [key-tech] §1 q^R, k^R equations)
# --------------------------------------------------------------------------
def rope_theta(R: int, base: float) -> np.ndarray:
    """theta_k = base^(-2k/R), k = 0 .. R/2 - 1, in fp64."""
    k = np.arange(R // 2, dtype=np.float64)
    return np.power(np.float64(base), -2.0 * k / R)


def yarn_theta(R: int, base: float, s: float, alpha: float = 1.0, beta: float = 32.0,
               orig_context: int = 4096) -> np.ndarray:
    """YaRN frequencies of the decoupled RoPE ([V2-explainer] §3.1.3; reading 6).

    Pairs whose wavelength fits in the original context fewer than alpha times are
    interpolated fully (theta / s), pairs that fit more than beta times keep theta, and the
    ones between move linearly in r = orig_context / wavelength.
    """
    theta = rope_theta(R, base)
    r = orig_context / (2.0 * math.pi / theta)
    gamma = np.clip((r - alpha) / (beta - alpha), 0.0, 1.0)
    return (1.0 - gamma) * theta / s + gamma * theta


def yarn_attention_factor(s: float, coef: float = 0.0707) -> float:
    """t with sqrt(t) = coef ln s + 1 ([V2-explainer] §3.1.3): every logit is scaled by t."""
    return (coef * math.log(s) + 1.0) ** 2


def rope_angles(pos: np.ndarray, R: int, base: float, theta: Optional[np.ndarray] = None) -> np.ndarray:
    """angle[..., k] = pos * theta_k (theta_k = base^(-2k/R) unless given), in fp64."""
    if theta is None:
        theta = rope_theta(R, base)
    return np.asarray(pos, dtype=np.float64)[..., None] * np.asarray(theta, dtype=np.float64)


def apply_rope(x: np.ndarray, pos: np.ndarray, base: float, theta: Optional[np.ndarray] = None) -> np.ndarray:
    """Rotate interleaved pairs of the last axis of x by the position's angles.

    x: [..., R]; pos broadcasts against x's leading axes.
    y_{2k}   = x_{2k} cos(a_k) - x_{2k+1} sin(a_k)
    y_{2k+1} = x_{2k} sin(a_k) + x_{2k+1} cos(a_k)
    """
    x = np.asarray(x, dtype=np.float64)
    R = x.shape[-1]
    a = rope_angles(pos, R, base, theta)
    c, s = np.cos(a), np.sin(a)
    x0, x1 = x[..., 0::2], x[..., 1::2]
    y = np.empty(np.broadcast_shapes(x.shape, a.shape[:-1] + (R,)), dtype=np.float64)
    y[..., 0::2] = x0 * c - x1 * s
    y[..., 1::2] = x0 * s + x1 * c
    return y


# --------------------------------------------------------------------------
# Storage types
# --------------------------------------------------------------------------
def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round to the nearest bf16 value (ties to even), via fp32; returns fp64."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)  # fp64 -> fp32: RNE
    b = f.view(np.uint32).astype(np.uint64)
    # Rounding fp32 -> bf16 directly from fp64 would differ from rounding
    # twice only on values within 2^-24 relative of a bf16 tie; take the
    # fp32 route on purpose, which is what a device does with fp32 math.
    lsb = (b >> np.uint64(16)) & np.uint64(1)
    r = ((b + np.uint64(0x7FFF) + lsb) >> np.uint64(16)) << np.uint64(16)
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def round_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)
    if dtype == "bf16":
        return round_bf16(x)
    raise ValueError(dtype)


def e4m3_values() -> np.ndarray:
    """Value of every E4M3 code 0..255 (OCP 'FN' flavour, fp64).

    Sign bit, 4 exponent bits with bias 7, 3 mantissa bits. Exponent field 0
    holds subnormals m/8 * 2^-6; exponent field 15 with mantissa 7 is NaN
    (there is no infinity), so the largest finite value is 1.75 * 2^8 = 448.
    """
    out = np.empty(256, dtype=np.float64)
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        e = (code >> 3) & 0xF
        m = code & 0x7
        if e == 0xF and m == 0x7:
            out[code] = math.nan
        elif e == 0:
            out[code] = sign * (m / 8.0) * 2.0 ** -6
        else:
            out[code] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return out


_E4M3 = e4m3_values()
_E4M3_POS = _E4M3[:0x7F]  # codes 0x00..0x7E: 0 and the 126 positive finite values, ascending


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """Encode fp32 values as E4M3 codes: round to nearest, ties to even, saturate at 448.

    Works on magnitudes: finds the two representable neighbours of |x| in the
    ascending code table and keeps the nearer one; on an exact tie it keeps
    the code with an even mantissa (least significant bit 0). |x| >= 448 maps
    to 448. Zero maps to +0 or -0 by the sign of x.
    """
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    a = np.abs(x)
    hi = np.searchsorted(_E4M3_POS, a, side="left")       # first code with value >= a
    hi = np.minimum(hi, 0x7E)
    lo = np.maximum(hi - 1, 0)
    vhi, vlo = _E4M3_POS[hi], _E4M3_POS[lo]
    dhi, dlo = vhi - a, a - vlo
    pick_hi = (dhi < dlo) | ((dhi == dlo) & ((hi & 1) == 0))
    code = np.where(a >= vhi, hi, np.where(pick_hi, hi, lo))
    code = np.where(a >= E4M3_MAX, 0x7E, code)
    sign = np.signbit(x).astype(np.int64) << 7
    return (code | sign).astype(np.uint8)


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    return _E4M3[np.asarray(codes, dtype=np.uint8)]


def quantize_fp8_groups(c: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Per-token 1x128-group E4M3 quantisation ([v3-notes] F8量化策略 (1)).

    c: [n, C] values that fp32 holds exactly (C a multiple of 128).
    Returns (codes uint8 [n, C], scales fp32 [n, C/128]). Both the scale and
    the division are taken in fp32 (IEEE, correctly rounded), which is the
    precision the device takes the same integer decision in.
    """
    c32 = np.asarray(c, dtype=np.float32)
    n, C = c32.shape
    g = c32.reshape(n, C // FP8_GROUP, FP8_GROUP)
    amax = np.max(np.abs(g), axis=-1)
    scale = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    q = (g / scale[..., None]).astype(np.float32)
    codes = e4m3_encode(q).reshape(n, C)
    return codes, scale


def dequantize_fp8_groups(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    n, C = codes.shape
    v = e4m3_decode(codes).reshape(n, C // FP8_GROUP, FP8_GROUP)
    return (v * np.asarray(scales, dtype=np.float64)[..., None]).reshape(n, C)


def quantize_q_latent(q_lat: np.ndarray, C: int):
    """The query side of FP8 scores (reading 8): q_lat [..., C + R] with its latent part
    (first C dims) quantised per (row, head) in 1x128 groups like the cache (reading 4).

    Returns (q8 [..., C + R] fp64 with the latent part replaced by code * scale and the RoPE
    part unchanged, codes uint8 [..., C], scales fp32 [..., C / 128]).
    """
    q = np.asarray(q_lat, dtype=np.float64)
    lead = q.shape[:-1]
    codes, scales = quantize_fp8_groups(q[..., :C].reshape(-1, C))
    q8 = q.copy()
    q8[..., :C] = dequantize_fp8_groups(codes, scales).reshape(lead + (C,))
    return q8, codes.reshape(lead + (C,)), scales.reshape(lead + (C // FP8_GROUP,))


# --------------------------------------------------------------------------
# Cache write (step a1): what the latent cache holds for each token
# ([V2-explainer] §2.2.2: only c^{KV}_t and k^R_t are cached)
# --------------------------------------------------------------------------
def cache_entries(c_kv: np.ndarray, k_r: np.ndarray, pos: np.ndarray, cache: str,
                  rope_base: float, theta: Optional[np.ndarray] = None):
    """Values of the cached (c_KV, k^R) for tokens at positions pos.

    Returns a dict with fp64 'c' [n, C] and 'k_r' [n, R] (the values attention
    sees), and for an FP8 cache also 'codes' and 'scales'.
    """
    k_rot = apply_rope(k_r, pos, rope_base, theta)
    if cache == "f32":
        return {"c": round_storage(c_kv, "f32"), "k_r": round_storage(k_rot, "f32")}
    if cache == "bf16":
        return {"c": round_storage(c_kv, "bf16"), "k_r": round_storage(k_rot, "bf16")}
    if cache == "fp8":
        codes, scales = quantize_fp8_groups(c_kv)
        return {"c": dequantize_fp8_groups(codes, scales), "k_r": round_storage(k_rot, "bf16"),
                "codes": codes, "scales": scales}
    raise ValueError(cache)


def page_slots(seq_idx: np.ndarray, pos: np.ndarray, block_table: np.ndarray, P: int):
    """(page id, slot in page) of each token: page = block_table[b][pos // P], slot = pos % P."""
    seq_idx = np.asarray(seq_idx, dtype=np.int64)
    pos = np.asarray(pos, dtype=np.int64)
    return block_table[seq_idx, pos // P].astype(np.int64), pos % P


# --------------------------------------------------------------------------
# The plain definition (non-absorbed), [V2-explainer] §2.2.1-2.2.2, [key-tech] §1
# --------------------------------------------------------------------------
def softmax_scale(D: int, R: int) -> float:
    return 1.0 / math.sqrt(D + R)


def mla_decode_naive(c: np.ndarray, k_r_cached: np.ndarray, q_c: np.ndarray, q_r: np.ndarray,
                     w_uk: np.ndarray, w_uv: np.ndarray, positions: np.ndarray,
                     rope_base: float, heads: Optional[np.ndarray] = None,
                     theta: Optional[np.ndarray] = None, scale: Optional[float] = None):
    """One sequence's MLA decode, computed the long way.

    c          [L, C]    cached latents c^{KV}_n (values attention sees)
    k_r_cached [L, R]    cached RoPE keys k^R_n (already rotated at position n)
    q_c        [n_q, H, D]  q^C of this step's query tokens
    q_r        [n_q, H, R]  q^R before RoPE
    w_uk, w_uv [H, D, C]
    positions  [n_q]     position of each query token (query j sees n <= positions[j])
    heads      optional subset of head indices to compute
    theta      RoPE frequencies (default base^(-2k/R); YaRN's from yarn_theta)
    scale      softmax scale (default 1/sqrt(D + R); with YaRN times yarn_attention_factor)

    For each head i: k^C_{n,i} = W^{UK}_i c_n, v^C_{n,i} = W^{UV}_i c_n,
    k_{n,i} = [k^C_{n,i}; k^R_n], q_{j,i} = [q^C_{j,i}; RoPE_{pos_j}(q^R_{j,i})],
    s_n = q_{j,i}^T k_{n,i} / sqrt(D + R) for n <= pos_j,
    o_{j,i} = sum_n softmax(s)_n v^C_{n,i}.

    Returns (o [n_q, h, D], o_lat [n_q, h, C], lse [n_q, h]) for the h
    computed heads; o_lat = sum_n softmax(s)_n c_n and lse = log sum_n e^{s_n}
    are the latent-space by-products the decode step also reports.
    """
    c = np.asarray(c, dtype=np.float64)
    k_r_cached = np.asarray(k_r_cached, dtype=np.float64)
    n_q, H, D = q_c.shape
    R = q_r.shape[-1]
    C = c.shape[1]
    heads = np.arange(H) if heads is None else np.asarray(heads)
    tau = softmax_scale(D, R) if scale is None else scale
    o = np.zeros((n_q, len(heads), D))
    o_lat = np.zeros((n_q, len(heads), C))
    lse = np.zeros((n_q, len(heads)))
    for hi, i in enumerate(heads):
        k_c = c @ np.asarray(w_uk[i], dtype=np.float64).T        # [L, D]
        v_c = c @ np.asarray(w_uv[i], dtype=np.float64).T        # [L, D]
        k = np.concatenate([k_c, k_r_cached], axis=1)           # [L, D + R]
        for j in range(n_q):
            p_j = int(positions[j])
            q_rot = apply_rope(q_r[j, i], np.int64(p_j), rope_base, theta)
            q = np.concatenate([np.asarray(q_c[j, i], dtype=np.float64), q_rot])
            s = (k[:p_j + 1] @ q) * tau
            m = np.max(s)
            e = np.exp(s - m)
            z = np.sum(e)
            p = e / z
            o[j, hi] = p @ v_c[:p_j + 1]
            o_lat[j, hi] = p @ c[:p_j + 1]
            lse[j, hi] = m + math.log(z)
    return o, o_lat, lse


# --------------------------------------------------------------------------
# Absorbed-form steps ([V2-explainer] §2.2.1 "W^{UK} absorbed into W^Q, W^{UV}
# into W^O"; [v3-notes] MLA: the query-side fusion turns MHA into MQA)
# --------------------------------------------------------------------------
def absorb_q(q_c: np.ndarray, q_r: np.ndarray, pos: np.ndarray, w_uk: np.ndarray,
             rope_base: float, theta: Optional[np.ndarray] = None) -> np.ndarray:
    """q_lat[t, i] = [q^C_{t,i}^T W^{UK}_i ; RoPE_{pos_t}(q^R_{t,i})]   (step a2).

    q_c [T, H, D], q_r [T, H, R], pos [T], w_uk [H, D, C] -> [T, H, C + R].
    """
    q_c = np.asarray(q_c, dtype=np.float64)
    lat = np.einsum("thd,hdc->thc", q_c, np.asarray(w_uk, dtype=np.float64))
    rot = apply_rope(q_r, np.asarray(pos)[:, None], rope_base, theta)
    return np.concatenate([lat, rot], axis=-1)


def latent_attention(q_lat: np.ndarray, c: np.ndarray, k_r_cached: np.ndarray,
                     positions: np.ndarray, scale: float):
    """Scores against the shared 576-d latent key, softmax, weighted latents (step a3).

    q_lat [n_q, H, C + R]; c [L, C]; k_r_cached [L, R]; query j sees n <= positions[j].
    s_n = q_lat . [c_n; k^R_n] * scale;  o_lat = sum_n softmax(s)_n c_n;  lse = log sum e^{s}.
    Returns (o_lat [n_q, H, C], lse [n_q, H]).
    """
    q_lat = np.asarray(q_lat, dtype=np.float64)
    kv = np.concatenate([np.asarray(c, dtype=np.float64),
                         np.asarray(k_r_cached, dtype=np.float64)], axis=1)  # [L, C + R]
    n_q, H, _ = q_lat.shape
    C = c.shape[1]
    o_lat = np.zeros((n_q, H, C))
    lse = np.zeros((n_q, H))
    for j in range(n_q):
        n = int(positions[j]) + 1
        s = (q_lat[j] @ kv[:n].T) * scale                        # [H, n]
        m = np.max(s, axis=1, keepdims=True)
        e = np.exp(s - m)
        z = np.sum(e, axis=1, keepdims=True)
        o_lat[j] = (e / z) @ kv[:n, :C]
        lse[j] = (m + np.log(z))[:, 0]
    return o_lat, lse


def unabsorb(o_lat: np.ndarray, w_uv: np.ndarray) -> np.ndarray:
    """o[t, i] = W^{UV}_i o_lat[t, i]   (step a6): [T, H, C] x [H, D, C] -> [T, H, D]."""
    return np.einsum("thc,hdc->thd", np.asarray(o_lat, dtype=np.float64),
                     np.asarray(w_uv, dtype=np.float64))


def combine_partials(o_parts: np.ndarray, lse_parts: np.ndarray):
    """Merge attention over disjoint token ranges (step a5).

    o_parts [S, ...]: each range's softmax-normalised output; lse_parts [S, ...].
    m = max_s lse_s; w_s = e^{lse_s - m}; o = sum_s w_s o_s / sum_s w_s;
    lse = m + log sum_s w_s. Ranges with lse = -inf carry no weight.
    """
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    m = np.max(lse_parts, axis=0)
    w = np.exp(lse_parts - m)
    z = np.sum(w, axis=0)
    o = np.sum(w[..., None] * np.asarray(o_parts, dtype=np.float64), axis=0) / z[..., None]
    return o, m + np.log(z)


# --------------------------------------------------------------------------
# Upstream of the cache and downstream of the attention
# ([V2-explainer] §2.2.1 c^{KV} = W^{DKV} h, §2.2.2 k^R = RoPE(W^{KR} h), §3.1.4 the
# latent's RMSNorm; §2.1.2 and [key-tech] §1 u_t = W^O [o_{t,1}; ...; o_{t,n_h}])
# --------------------------------------------------------------------------
def rms_norm(x: np.ndarray, gain: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    """gain * x / sqrt(mean(x^2 over the last axis) + eps) (reading 7)."""
    x = np.asarray(x, dtype=np.float64)
    return np.asarray(gain, dtype=np.float64) * x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)


def project_latent(h: np.ndarray, w_dkv: np.ndarray, w_kr: np.ndarray, gain: np.ndarray,
                   eps: float = 1e-6):
    """The cached quantities of tokens with hidden states h [T, d], before RoPE:
    c^{KV} = RMSNorm(W^{DKV} h) [T, C] and k^R = W^{KR} h [T, R] (W^{DKV} [C, d], W^{KR}
    [R, d], gain [C]). cache_entries() then rotates k^R and stores both."""
    h = np.asarray(h, dtype=np.float64)
    c = rms_norm(h @ np.asarray(w_dkv, dtype=np.float64).T, gain, eps)
    k = h @ np.asarray(w_kr, dtype=np.float64).T
    return c, k


def output_projection(o: np.ndarray, w_o: np.ndarray) -> np.ndarray:
    """u_t = W^O [o_{t,1}; ...; o_{t,n_h}]: o [T, H, D] (heads concatenated in order),
    W^O [d, H D] -> u [T, d]."""
    o = np.asarray(o, dtype=np.float64)
    return o.reshape(o.shape[0], -1) @ np.asarray(w_o, dtype=np.float64).T


# --------------------------------------------------------------------------
# Cache sizes ([V2-explainer] §2.1.2 MHA: 2 n_h d_h l; §2.2.2 MLA: (d_c + d_h^R) l)
# --------------------------------------------------------------------------
def mha_cache_elements(n_h: int, d_h: int, layers: int) -> int:
    return 2 * n_h * d_h * layers


def mla_cache_elements(d_c: int, d_rope: int, layers: int) -> int:
    return (d_c + d_rope) * layers


def gqa_cache_elements(n_groups: float, d_h: int, layers: int) -> float:
    return 2 * n_groups * d_h * layers
