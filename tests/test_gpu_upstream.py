"""GPU parity of the steps either side of the latent cache, against the fp64 oracle:

* mla_project_append, the fused upstream append (「一文通透DeepSeek-V2」 §2.2.1 c^{KV} = W^{DKV} h,
  §3.1.4 the RMSNorm after the compressed latent, §2.2.2 k^R = RoPE(W^{KR} h));
* mla_output_projection, u_t = W^O [o_{t,1}; ...; o_{t,n_h}] (§2.1.2; 「deepseek(2)——deepseek
  關鍵技術」 §1).

Sizes are DeepSeek-V2's (d = 5120, n_h = 128, d_h = 128, d_c = 512, d_h^R = 64; §3.1.1) for
a decode step's 64 tokens and a 200-token prompt, plus a small shape with a ragged tail.
"""
import numpy as np
import pytest
import torch

import mla_latent_kv_78_b300 as M
import workloads as W
from oracle import mla_oracle as O

from _support import assert_close, dev

pytestmark = pytest.mark.gpu

needs_cuda = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")

BF = torch.bfloat16


def _bf16(x: np.ndarray) -> np.ndarray:
    return W.round_to_storage(np.asarray(x, dtype=np.float32), "bf16")


def _rng(seed):
    return np.random.default_rng([9100, seed])


@needs_cuda
@pytest.mark.parametrize("H,D,d_model,T", [(128, 128, 5120, 64), (128, 128, 5120, 200), (4, 32, 64, 37)],
                         ids=["v2-T64", "v2-T200", "small-T37"])
def test_output_projection(H, D, d_model, T):
    g = _rng(H + T)
    o = _bf16(g.standard_normal((T, H, D)) * 0.05)
    w_o = _bf16(g.standard_normal((d_model, H * D)) * 0.006)   # the pages' init std (§3.1.1)
    cfg = M.make_config(H, D, 512 if H == 128 else 64, 64 if H == 128 else 16, 64)
    ws_n = M.mla_output_projection_workspace_size(cfg, d_model, T)
    ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device="cuda")
    u = torch.full((T, d_model), float("nan"), device="cuda")
    M.mla_output_projection(cfg, dev(o.reshape(T, H * D), BF), dev(w_o, BF), u, ws)
    torch.cuda.synchronize()
    ref = O.output_projection(o, w_o)
    wl = W.small_v2(1, [1])   # bf16 tolerance: 1e-2 max|oracle| + 1e-3
    assert_close(wl, u.cpu().numpy(), ref, f"u (T={T}, d={d_model})")


def _project_inputs(T, d_model, C, R, seed):
    g = _rng(seed)
    h = _bf16(g.standard_normal((T, d_model)))
    w = _bf16(g.standard_normal((C + R, d_model)) * 0.02)
    gain = g.uniform(0.5, 1.5, C).astype(np.float32)
    return h, w, gain


def _oracle_cached(h, w, gain, pos, C, cache, eps):
    """The cached (c, k^R) the oracle derives: projection and RMSNorm in fp64, rounded to bf16
    (the activation type the projected values are stored in before caching), then cached."""
    c, k = O.project_latent(h, w[:C], w[C:], gain, eps)
    return O.cache_entries(O.round_bf16(c), O.round_bf16(k), pos, cache, 10000.0)


@needs_cuda
@pytest.mark.parametrize("cache", ["bf16", "fp8"])
@pytest.mark.parametrize("T", [64, 200])
def test_project_append_writes_the_projected_entries(cache, T):
    """Every token's cache entry from mla_project_append against the oracle: bf16 latents within
    one bf16 ulp plus the fp32 error of the projection's sums (they may round the other way near
    a rounding boundary); FP8 codes identical for all but a few elements whose values sit on a
    rounding boundary (those one step apart); rotated k^R within the rotation bound."""
    H, D, C, R, P, d_model, eps = 128, 128, 512, 64, 64, 5120, 1e-6
    h, w, gain = _project_inputs(T, d_model, C, R, seed=T)
    B = 4
    seq = np.arange(T, dtype=np.int32) % B
    pos = (np.arange(T, dtype=np.int32) // B) * 3 + 5       # positions spread over pages
    maxp = int(pos.max()) // P + 1
    bt = (np.arange(B * maxp, dtype=np.int32).reshape(B, maxp) * 7) % (B * maxp)   # a permutation
    cfg = M.make_config(H, D, C, R, P, cache=cache)
    eb = M.mla_cache_entry_bytes(cfg)
    pool = torch.zeros((B * maxp, P, eb), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(M.mla_project_append_workspace_size(cfg, d_model, T), dtype=torch.uint8, device="cuda")
    M.mla_project_append(cfg, dev(h, BF), dev(w, BF), torch.from_numpy(gain).cuda(), eps,
                         torch.from_numpy(seq).cuda(), torch.from_numpy(pos).cuda(),
                         torch.from_numpy(bt).cuda(), pool, ws, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = _oracle_cached(h, w, gain, pos, C, cache, eps)
    ent = pool.cpu().numpy()[bt[seq, pos // P], pos % P]
    if cache == "bf16":
        got_c = W.bf16_bits_to_f32(ent[:, :2 * C].copy().view(np.uint16)).astype(np.float64)
        ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(ref["c"]), 1e-30))) - 7)
        # plus the fp32 error of a 5120-term sum, which scales with the row (RMS = gain after
        # the norm), not with an element that happens to lie near zero
        assert np.all(np.abs(got_c - ref["c"]) <= ulp + 2.0 ** -14 * gain)
        got_r = W.bf16_bits_to_f32(ent[:, 2 * C:].copy().view(np.uint16)).astype(np.float64)
    else:
        codes = ent[:, :C]
        same = codes == ref["codes"]
        assert same.mean() > 0.99, f"only {same.mean():.4f} of the E4M3 codes agree"
        scales = ent[:, C + 2 * R:].copy().view(np.float32).astype(np.float64)
        np.testing.assert_allclose(scales, ref["scales"], rtol=2.0 ** -7)
        got_c = O.dequantize_fp8_groups(codes, scales)
        step = np.repeat(ref["scales"], 128, axis=1) * 32.0   # the widest E4M3 step (values in [256, 448])
        assert np.all(np.abs(got_c - ref["c"]) <= step)
        got_r = W.bf16_bits_to_f32(ent[:, C:C + 2 * R].copy().view(np.uint16)).astype(np.float64)
    k = O.project_latent(h, w[:C], w[C:], gain, eps)[1]
    pair = np.repeat(np.abs(k[:, 0::2]) + np.abs(k[:, 1::2]), 2, axis=1)
    ulp_r = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(ref["k_r"]), 1e-30))) - 7)
    assert np.all(np.abs(got_r - ref["k_r"]) <= ulp_r + 2.0 ** -7 * pair)


@needs_cuda
@pytest.mark.parametrize("cache", ["bf16", "fp8"])
def test_project_append_then_decode_matches_the_chain(cache):
    """A 300-token prompt and this step's token projected into the cache by
    mla_project_append, then absorb -> decode -> unabsorb; o against the oracle's chain
    (projection, RMSNorm, bf16 storage, cache, non-absorbed attention)."""
    H, D, C, R, P, d_model, eps = 128, 128, 512, 64, 64, 5120, 1e-6
    L = 301
    h, w, gain = _project_inputs(L, d_model, C, R, seed=77)
    wl = W.small_v2(1, [L], n_q=1, cache=cache, seed=78)
    cfg = M.make_config(H, D, C, R, P, cache=cache)
    w_uk, w_uv = wl.weights()
    step = M.DecodeStep(cfg, torch.from_numpy(wl.block_table()), wl.seq_lens, 1, wl.num_pages,
                        dev(w_uk, BF), dev(w_uv, BF))
    ws = torch.empty(M.mla_project_append_workspace_size(cfg, d_model, L), dtype=torch.uint8, device="cuda")
    M.mla_project_append(cfg, dev(h, BF), dev(w, BF), torch.from_numpy(gain).cuda(), eps,
                         torch.zeros(L, dtype=torch.int32, device="cuda"),
                         torch.arange(L, dtype=torch.int32, device="cuda"), step.block_table, step.pool, ws,
                         num_pages=wl.num_pages, dev_status=step.dev_status)
    q_c, q_r = wl.queries()
    step.absorb(dev(q_c.reshape(1, H, D), BF), dev(q_r.reshape(1, H, R), BF))
    step.decode()
    step.unabsorb()
    torch.cuda.synchronize()
    assert step.status() == 0
    ref = _oracle_cached(h, w, gain, np.arange(L), C, cache, eps)
    o, o_lat, lse = O.mla_decode_naive(ref["c"], ref["k_r"], q_c[0], q_r[0], w_uk, w_uv,
                                       np.array([L - 1]), 10000.0)
    assert_close(wl, step.o.cpu().numpy(), o, "o")
    assert_close(wl, step.o_lat.float().cpu().numpy(), o_lat, "o_lat")


@needs_cuda
@pytest.mark.parametrize("L,yarn", [(200, False), (1, False), (64, False), (300, True)],
                         ids=["L200", "L1", "L64", "L300-yarn"])
def test_prefill_matches_the_naive_definition(L, yarn):
    """mla_prefill (k^C, v^C restored from the latents, causal attention over the prompt)
    against the oracle's non-absorbed definition with every prompt position as a query
    (「一文通透DeepSeek-V2」 §2.2.1; 「deepseek(2)——deepseek 關鍵技術」 §1), on a subset of the 128
    heads; L = 200 leaves a ragged 72-query block and a partly masked key block."""
    from _support import tau_of, theta_of
    wl = W.small_v2(1, [L], n_q=1, cache="bf16", seed=200 + L, rope_scaling=40.0 if yarn else 1.0)
    H, D, C, R = wl.H, wl.D, wl.C, wl.R
    cfg = M.make_config(H, D, C, R, wl.P, rope_scaling=wl.rope_scaling if yarn else 0.0)
    g = _rng(300 + L)
    c = _bf16(g.standard_normal((L, C)))
    k_r = _bf16(g.standard_normal((L, R)))
    q_c = _bf16(g.standard_normal((L, H, D)))
    q_r = _bf16(g.standard_normal((L, H, R)))
    w_uk, w_uv = wl.weights()
    ce = O.cache_entries(c, k_r, np.arange(L), "bf16", wl.rope_base, theta_of(wl))
    o = torch.full((L, H, D), float("nan"), device="cuda")
    ws = torch.empty(M.mla_prefill_workspace_size(cfg, L), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    M.mla_prefill(cfg, dev(ce["c"], BF), dev(ce["k_r"], BF), dev(q_c, BF), dev(q_r, BF), dev(w_uk, BF),
                  dev(w_uv, BF), o, ws, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    heads = np.array([0, 1, 63, 64, 127])
    ref, _, _ = O.mla_decode_naive(ce["c"], ce["k_r"], q_c, q_r, w_uk, w_uv, np.arange(L), wl.rope_base,
                                   heads=heads, theta=theta_of(wl), scale=tau_of(wl))
    got = o.cpu().numpy()[:, heads]
    assert np.all(np.isfinite(o.cpu().numpy()))
    assert_close(wl, got, ref, f"prefill o (L={L})")
