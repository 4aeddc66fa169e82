"""Seeded synthetic inputs for MLA decode workloads.

This module only draws random numbers and encodes them in the storage types
the kernels read (fp32 values, bf16 bit patterns, int32 page tables). It
holds none of the attention arithmetic: no RoPE, no projection, no softmax
and no FP8 quantisation. The fp64 oracle and the CUDA path both take their
inputs from here and from nowhere else.

Shapes follow DeepSeek-V2's MLA hyper-parameters (n_h = 128 heads,
d_h = 128, d_c = 512, d_h^R = 64), as listed in 「一文通透DeepSeek-V2」
§3.1.1 (模型超参数). Every random stream is keyed by (seed, purpose[, b]) so
that any one sequence can be regenerated on its own, which is how the
full-size parity tests give the oracle a single sequence to check.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence, Tuple

import numpy as np

# Purpose keys of the random streams.
_K_LATENT = 1
_K_WEIGHT = 2
_K_QUERY = 3
_K_PAGES = 4
_K_SEQLEN = 5
_K_QLAT = 6


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 array -> bf16 bit patterns (uint16), round to nearest even.

    Inputs here are finite draws, so no NaN handling is needed.
    """
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    r = (b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> the fp32 values they encode (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def round_to_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round fp32 draws to the values a storage type can hold (returned as fp32)."""
    if dtype == "f32":
        return np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "bf16":
        return bf16_bits_to_f32(to_bf16_bits(x))
    raise ValueError(dtype)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic MLA decode problem.

    Attributes follow the pages' notation: H = n_h heads, D = d_h per-head
    dim, C = d_c latent dim, R = d_h^R decoupled-RoPE dim, P = page size in
    tokens, n_q = query tokens per sequence in this step. ``seq_lens[b]``
    counts the cached tokens *including* this step's n_q new ones; query j
    of sequence b sits at position seq_lens[b] - n_q + j.
    """

    name: str
    B: int
    H: int
    D: int
    C: int
    R: int
    n_q: int
    P: int
    seq_lens: Tuple[int, ...]
    cache: str          # pool entry format: "f32" | "bf16" | "fp8"
    act: str            # q, weights, q_lat, o_lat storage: "f32" | "bf16"
    latent_std: float = 1.0
    w_std: float = 0.02
    q_std: float = 1.0
    permute_pages: bool = False
    seed: int = 0
    rope_base: float = 10000.0
    # optional per-128-column multipliers of the c_KV draws (groups of very different
    # magnitude, e.g. to exercise FP8 group scales far below 1)
    group_scales: Optional[Tuple[float, ...]] = None
    # YaRN factor s of the decoupled RoPE (1: plain RoPE); the method itself lives in the
    # library and the oracle, this only names the setting
    rope_scaling: float = 1.0

    # ---- derived sizes -------------------------------------------------
    @property
    def pages_per_seq(self) -> Tuple[int, ...]:
        return tuple(-(-L // self.P) for L in self.seq_lens)

    @property
    def max_pages(self) -> int:
        return max(self.pages_per_seq)

    @property
    def num_pages(self) -> int:
        return sum(self.pages_per_seq)

    @property
    def max_seq_len(self) -> int:
        return max(self.seq_lens)

    @property
    def total_tokens(self) -> int:
        return sum(self.seq_lens)

    @property
    def latent_storage(self) -> str:
        """Storage type of the raw c_KV / k_R inputs handed to the append."""
        return "f32" if self.cache == "f32" else "bf16"

    def positions(self, b: int) -> np.ndarray:
        """Positions of sequence b's query tokens in this step."""
        L = self.seq_lens[b]
        return np.arange(L - self.n_q, L, dtype=np.int32)

    # ---- random streams -------------------------------------------------
    def _rng(self, *key: int) -> np.random.Generator:
        return np.random.default_rng([self.seed, *key])

    def block_table(self) -> np.ndarray:
        """int32 [B, max_pages]: page ids of each sequence; unused slots = -1.

        Sequential: sequence b owns a contiguous run of pages. Permuted: the
        pool's page ids are shuffled (numpy's Fisher-Yates ``permutation``)
        before they are handed out in sequence order.
        """
        ids = np.arange(self.num_pages, dtype=np.int64)
        if self.permute_pages:
            ids = self._rng(_K_PAGES).permutation(self.num_pages)
        bt = np.full((self.B, self.max_pages), -1, dtype=np.int32)
        k = 0
        for b, n in enumerate(self.pages_per_seq):
            bt[b, :n] = ids[k:k + n]
            k += n
        return bt

    def latents(self, b: int) -> Tuple[np.ndarray, np.ndarray]:
        """(c_KV [L_b, C], k_R [L_b, R]) of sequence b, pre-RoPE, storage-rounded fp32."""
        L = self.seq_lens[b]
        g = self._rng(_K_LATENT, b)
        x = g.standard_normal((L, self.C + self.R), dtype=np.float32) * np.float32(self.latent_std)
        if self.group_scales is not None:
            for k, m in enumerate(self.group_scales):
                x[:, 128 * k:128 * (k + 1)] *= np.float32(m)
        x = round_to_storage(x, self.latent_storage)
        return np.ascontiguousarray(x[:, :self.C]), np.ascontiguousarray(x[:, self.C:])

    def weights(self) -> Tuple[np.ndarray, np.ndarray]:
        """(W_UK, W_UV), each [H, D, C]: head i's rows of W^{UK}, W^{UV} in R^{(H D) x C}."""
        g = self._rng(_K_WEIGHT)
        w = g.standard_normal((2, self.H, self.D, self.C), dtype=np.float32) * np.float32(self.w_std)
        w = round_to_storage(w, self.act)
        return np.ascontiguousarray(w[0]), np.ascontiguousarray(w[1])

    def queries(self) -> Tuple[np.ndarray, np.ndarray]:
        """(q_C [B, n_q, H, D], q_R [B, n_q, H, R]), q_R before RoPE."""
        g = self._rng(_K_QUERY)
        q = g.standard_normal((self.B, self.n_q, self.H, self.D + self.R), dtype=np.float32)
        q = round_to_storage(q * np.float32(self.q_std), self.act)
        return np.ascontiguousarray(q[..., :self.D]), np.ascontiguousarray(q[..., self.D:])

    def latent_queries(self) -> np.ndarray:
        """q_lat [B, n_q, H, C + R] drawn directly, for testing the decode step alone.

        The latent part has the spread an absorbed query would have
        (std = sqrt(D) * w_std * q_std); the RoPE part has std q_std.
        """
        g = self._rng(_K_QLAT)
        q = g.standard_normal((self.B, self.n_q, self.H, self.C + self.R), dtype=np.float32)
        q[..., :self.C] *= np.float32(math.sqrt(self.D) * self.w_std * self.q_std)
        q[..., self.C:] *= np.float32(self.q_std)
        return round_to_storage(q, self.act)

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def _uniform_lens(B: int, lo: int, hi: int, seed: int) -> Tuple[int, ...]:
    g = np.random.default_rng([seed, _K_SEQLEN])
    return tuple(int(v) for v in g.integers(lo, hi + 1, size=B))


def config(n: int) -> Workload:
    """The five workloads: 1 tiny fp32, 2 V2-shaped 4K decode, 3 ragged,
    4 128K long context, 5 two-token (MTP) decode over an FP8 cache.

    Seeds are 7800 + n.
    """
    seed = 7800 + n
    v2 = dict(H=128, D=128, C=512, R=64, P=64, act="bf16", latent_std=1.0,
              w_std=0.02, q_std=1.0, seed=seed)
    if n == 1:
        return Workload(name="tiny-fp32", B=2, H=4, D=32, C=64, R=16, n_q=1, P=16,
                        seq_lens=(37, 64), cache="f32", act="f32", latent_std=1.0,
                        w_std=math.sqrt(1.0 / 64), q_std=1.0, seed=seed)
    if n == 2:
        return Workload(name="v2-decode-b64-l4096", B=64, n_q=1, seq_lens=(4096,) * 64,
                        cache="bf16", **v2)
    if n == 3:
        return Workload(name="v2-ragged-b128-l1k-32k", B=128, n_q=1,
                        seq_lens=_uniform_lens(128, 1024, 32768, seed), cache="bf16",
                        permute_pages=True, **v2)
    if n == 4:
        return Workload(name="v2-long-b8-l128k", B=8, n_q=1, seq_lens=(131072,) * 8,
                        cache="bf16", **v2)
    if n == 5:
        return Workload(name="v2-mtp2-fp8-b128-l8192", B=128, n_q=2, seq_lens=(8192,) * 128,
                        cache="fp8", **v2)
    raise ValueError(f"no workload {n}")


def small_v2(B: int, seq_lens: Sequence[int], n_q: int = 1, cache: str = "bf16",
             permute_pages: bool = True, seed: int = 1234, H: int = 128,
             group_scales: Optional[Tuple[float, ...]] = None, rope_scaling: float = 1.0) -> Workload:
    """A V2-shaped workload small enough for the oracle to finish in seconds."""
    assert len(seq_lens) == B
    return Workload(name=f"v2-small-b{B}", B=B, H=H, D=128, C=512, R=64, n_q=n_q, P=64,
                    seq_lens=tuple(int(x) for x in seq_lens), cache=cache, act="bf16",
                    latent_std=1.0, w_std=0.02, q_std=1.0, permute_pages=permute_pages,
                    seed=seed, group_scales=group_scales, rope_scaling=rope_scaling)
