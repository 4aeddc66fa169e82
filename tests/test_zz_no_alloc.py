"""mla_decode_noalloc: the decode for callers that cannot allocate device memory.

It runs the same decode as mla_decode but takes its scratch from a fixed array inside the
library instead of a caller-provided workspace. This file sorts last so that a run that stops
at the first failure has already run every other test; it also passes on its own in a fresh
process.
"""
import ctypes

import numpy as np
import pytest
import torch

import mla_latent_kv_78_b300 as M
import workloads as W
from mla_latent_kv_78_b300 import _lib as L

from oracle import mla_oracle as O

from _support import ACT, Case, assert_close, dev, gpu_rows

pytestmark = pytest.mark.gpu

needs_cuda = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")


def _both(wl, kernel, num_splits):
    """Run mla_decode (torch workspace) and mla_decode_noalloc on the same inputs."""
    case = Case(wl, kernel=kernel, num_splits=num_splits)
    case.step.append(case.new_c, case.new_r)
    q_lat = dev(wl.latent_queries().reshape(-1, wl.H, wl.C + wl.R), ACT[wl.act])
    st = case.step
    st.decode(q_lat)
    ref_o, ref_lse = st.o_lat.clone(), st.lse.clone()
    o = torch.full_like(st.o_lat, float("nan"))
    lse = torch.full_like(st.lse, float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    M.mla_decode_noalloc(st.cfg, q_lat, st.pool, st.block_table, st.seq_lens, wl.n_q,
                         st.max_seq_len, o, lse, num_splits=num_splits, num_pages=st.num_pages,
                         dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and st.status() == 0
    return ref_o, ref_lse, o, lse


@needs_cuda
@pytest.mark.parametrize("kernel", [M.MLA_KERNEL_AUTO, M.MLA_KERNEL_SIMT], ids=["tc", "simt"])
def test_noalloc_matches_decode_on_consecutive_calls(kernel):
    # two calls in a row with different sizes and split counts: the second must not depend on
    # what the first left in the shared scratch
    calls = [
        (W.small_v2(3, [700, 257, 64], n_q=1, cache="bf16", seed=21), 3),
        (W.small_v2(2, [300, 1000], n_q=2, cache="bf16", seed=22), 0),
    ]
    for wl, splits in calls:
        ref_o, ref_lse, o, lse = _both(wl, kernel, splits)
        assert_close(wl, o.float().cpu().numpy(), ref_o.float().cpu().numpy(), "o_lat noalloc")
        assert_close(wl, lse.cpu().numpy(), ref_lse.cpu().numpy(), "lse noalloc")
        # and against the oracle directly
        q_lat = wl.latent_queries()
        tau = O.softmax_scale(wl.D, wl.R)
        for b in range(wl.B):
            c, r = wl.latents(b)
            ce = O.cache_entries(c, r, np.arange(wl.seq_lens[b]), wl.cache, wl.rope_base)
            ref_ob, ref_lb = O.latent_attention(q_lat[b], ce["c"], ce["k_r"], wl.positions(b), tau)
            assert_close(wl, gpu_rows(o, wl, b), ref_ob, f"o_lat noalloc vs oracle [b={b}]")
            assert_close(wl, gpu_rows(lse, wl, b), ref_lb, f"lse noalloc vs oracle [b={b}]")


@needs_cuda
def test_noalloc_staged_fp8_decode():
    """MLA_KERNEL_TC_FP8_STAGED keeps its bf16 copy of the cache in the scratch: a small batch
    fits and matches mla_decode bit for bit; the two-token 128 x 8192 batch (1.2 GB staged)
    is refused before anything is launched."""
    wl = W.small_v2(3, [300, 129, 700], n_q=2, cache="fp8", seed=24)
    ref_o, ref_lse, o, lse = _both(wl, M.MLA_KERNEL_TC_FP8_STAGED, 0)
    assert torch.equal(o, ref_o) and torch.equal(lse, ref_lse)
    cfg = M.make_config(128, 128, 512, 64, 64, cache="fp8", kernel=M.MLA_KERNEL_TC_FP8_STAGED)
    assert M.mla_decode_workspace_size(cfg, 128, 2, 8192, 0) > L.NOALLOC_SCRATCH_BYTES
    rc = M.lib().mla_decode_noalloc(ctypes.byref(cfg), 16, 16, 16, 128, 16384, 16, 128, 2, 8192, 0,
                                    16, None, None, None)
    assert rc == L.MLA_ERR_SCRATCH_LIMIT


@needs_cuda
def test_noalloc_rejects_sizes_beyond_its_scratch():
    wl = W.small_v2(2, [64, 64], n_q=1, cache="bf16", seed=23)
    cfg = M.make_config(wl.H, wl.D, wl.C, wl.R, wl.P, cache=wl.cache, act=wl.act)
    batch, splits = 64, 4   # fp32 split partials: 64 x 128 heads x 4 x 513 x 4 B = 67 MB
    assert M.mla_decode_workspace_size(cfg, batch, 1, 4096, splits) > L.NOALLOC_SCRATCH_BYTES
    lib = M.lib()
    rc = lib.mla_decode_noalloc(ctypes.byref(cfg), 16, 16, 16, 64, 64, 16, batch, 1, 4096, splits,
                                16, None, None, None)
    assert rc == L.MLA_ERR_SCRATCH_LIMIT
    assert "scratch" in M.mla_status_string(rc)


@needs_cuda
def test_noalloc_at_the_edge_of_its_scratch():
    """Sizes whose split-KV partials fill the fixed scratch to within 10 % of its size: the
    no-alloc call accepts them and matches mla_decode on the same inputs bit for bit (same
    kernels, same split), so the scratch is usable up to its end."""
    wl = W.small_v2(8, [4096] * 8, n_q=1, cache="bf16", seed=24)
    cfg = M.make_config(wl.H, wl.D, wl.C, wl.R, wl.P, cache=wl.cache, act=wl.act)
    splits = 15   # fp32 partials: 8 x 128 heads x 15 x 513 x 4 B = 31.5 MB of 32 MiB
    need = M.mla_decode_workspace_size(cfg, wl.B, wl.n_q, max(wl.seq_lens), splits)
    assert 0.9 * L.NOALLOC_SCRATCH_BYTES < need <= L.NOALLOC_SCRATCH_BYTES
    ref_o, ref_lse, o, lse = _both(wl, M.MLA_KERNEL_AUTO, splits)
    assert torch.equal(o, ref_o) and torch.equal(lse, ref_lse)
