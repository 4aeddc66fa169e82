"""Shared helpers of the GPU parity tests: upload a workload, run the library's
calls, and compute the oracle's answer for chosen sequences and heads."""
from __future__ import annotations

import numpy as np
import torch

import mla_latent_kv_78_b300 as M
from oracle import mla_oracle as O
from workloads import Workload

ACT = {"f32": torch.float32, "bf16": torch.bfloat16}


def dev(x: np.ndarray, dtype: torch.dtype) -> torch.Tensor:
    """numpy values (already representable in dtype) -> contiguous CUDA tensor."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to("cuda").to(dtype).contiguous()


def config_of(wl: Workload, kernel: int = M.MLA_KERNEL_AUTO) -> M.mla_config:
    return M.make_config(wl.H, wl.D, wl.C, wl.R, wl.P, cache=wl.cache, act=wl.act, kernel=kernel,
                         rope_scaling=wl.rope_scaling if wl.rope_scaling > 1 else 0.0)


def theta_of(wl: Workload):
    """The oracle's RoPE frequencies for a workload (None: plain RoPE)."""
    if wl.rope_scaling > 1:
        return O.yarn_theta(wl.R, wl.rope_base, wl.rope_scaling)
    return None


def tau_of(wl: Workload) -> float:
    """The oracle's softmax scale for a workload (YaRN's logit factor included)."""
    tau = O.softmax_scale(wl.D, wl.R)
    return tau * O.yarn_attention_factor(wl.rope_scaling) if wl.rope_scaling > 1 else tau


def tolerance(wl: Workload, ref: np.ndarray):
    """|gpu - oracle| bound, elementwise.

    bf16 / FP8 caches: 1e-2 max|oracle| + 1e-3 over the compared array (the bound the task
    states; bf16 inputs and weights carry 2^-9 relative rounding each, so a per-element bound
    would fail on elements that cancel to near zero).
    fp32 workload: 1e-5 relative per element, |oracle| * 1e-5, plus a floor of 1e-6 max|oracle|
    for elements that cancel to near zero (fp32 accumulation error scales with the magnitude
    of the summed terms, not with their sum)."""
    m = float(np.max(np.abs(ref))) if ref.size else 0.0
    if wl.cache == "f32":
        return 1e-5 * np.abs(ref) + 1e-6 * m
    return 1e-2 * m + 1e-3


def assert_close(wl: Workload, gpu: np.ndarray, ref: np.ndarray, what: str) -> float:
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite GPU values"
    if not ref.size:
        return 0.0
    diff = np.abs(gpu - ref)
    tol = tolerance(wl, ref)
    bad = diff > tol
    if np.any(bad):
        i = np.unravel_index(int(np.argmax(diff - tol)), diff.shape)
        raise AssertionError(f"{what}: |gpu - oracle| = {diff[i]:.3e} > {np.broadcast_to(tol, diff.shape)[i]:.3e} "
                             f"at {i} (oracle {ref[i]:.6e}, {int(bad.sum())} of {bad.size} elements)")
    return float(np.max(diff))


class Case:
    """A workload resident on the GPU: weights, pool filled by mla_append_cache with every
    cached token except this step's n_q new ones, and a DecodeStep around it."""

    def __init__(self, wl: Workload, kernel: int = M.MLA_KERNEL_AUTO, num_splits: int = 0,
                 prefill: bool = True, chunk_tokens: int = 1 << 20):
        self.wl = wl
        self.cfg = config_of(wl, kernel)
        act = ACT[wl.act]
        self.w_uk_np, self.w_uv_np = wl.weights()
        self.bt_np = wl.block_table()
        self.step = M.DecodeStep(self.cfg, torch.from_numpy(self.bt_np), wl.seq_lens, wl.n_q,
                                 wl.num_pages, dev(self.w_uk_np, act), dev(self.w_uv_np, act),
                                 num_splits=num_splits)
        lat = ACT[wl.latent_storage]
        # this step's inputs, t = b * n_q + j, collected while the cache is filled
        new_c, new_r = [], []
        buf_c, buf_r, buf_s, buf_p, n = [], [], [], [], 0
        for b in range(wl.B):
            c, r = wl.latents(b)
            new_c.append(c[-wl.n_q:]); new_r.append(r[-wl.n_q:])
            if not prefill:
                continue
            keep = wl.seq_lens[b] - wl.n_q
            if keep > 0:
                buf_c.append(c[:keep]); buf_r.append(r[:keep])
                buf_s.append(np.full(keep, b, np.int32)); buf_p.append(np.arange(keep, dtype=np.int32))
                n += keep
            # upload in chunks of whole sequences to bound host memory
            if n >= chunk_tokens or (b == wl.B - 1 and n):
                self.step.prefill(dev(np.concatenate(buf_c), lat), dev(np.concatenate(buf_r), lat),
                                  torch.from_numpy(np.concatenate(buf_s)).cuda(),
                                  torch.from_numpy(np.concatenate(buf_p)).cuda())
                buf_c, buf_r, buf_s, buf_p, n = [], [], [], [], 0
        self.new_c = dev(np.concatenate(new_c), lat)
        self.new_r = dev(np.concatenate(new_r), lat)
        q_c, q_r = wl.queries()
        self.q_c_np, self.q_r_np = q_c, q_r
        self.q_c = dev(q_c.reshape(wl.B * wl.n_q, wl.H, wl.D), act)
        self.q_r = dev(q_r.reshape(wl.B * wl.n_q, wl.H, wl.R), act)

    def run_step(self) -> None:
        self.step.step(self.new_c, self.new_r, self.q_c, self.q_r)
        torch.cuda.synchronize()

    # ---- oracle side -------------------------------------------------------
    def cache_of(self, b: int):
        wl = self.wl
        c, r = wl.latents(b)
        return O.cache_entries(c, r, np.arange(wl.seq_lens[b]), wl.cache, wl.rope_base, theta_of(wl))

    def oracle(self, b: int, heads=None):
        """(o, o_lat, lse) of sequence b from the naive definition."""
        wl = self.wl
        ce = self.cache_of(b)
        return O.mla_decode_naive(ce["c"], ce["k_r"], self.q_c_np[b], self.q_r_np[b], self.w_uk_np,
                                  self.w_uv_np, wl.positions(b), wl.rope_base, heads=heads,
                                  theta=theta_of(wl), scale=tau_of(wl))


def gpu_rows(t: torch.Tensor, wl: Workload, b: int) -> np.ndarray:
    """Rows t = b * n_q + j of a [B * n_q, ...] output, as fp64 numpy."""
    return t[b * wl.n_q:(b + 1) * wl.n_q].float().cpu().numpy().astype(np.float64)
