"""The C-ABI library builds, loads and exports what include/mla.h declares;
host-side argument checks answer without a GPU."""
import ctypes
import os
import re

import pytest

import mla_latent_kv_78_b300 as M
from mla_latent_kv_78_b300 import _lib as L

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "mla.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    lib = M.lib()
    names = _declared()
    assert "mla_decode" in names and "mla_append_cache" in names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/mla.h but not exported"
    # the binding wraps exactly the declared calls
    assert set(L.EXPORTED) <= set(names)


def test_entry_bytes():
    v2 = dict(H=128, D=128, C=512, R=64, P=64)
    assert M.mla_cache_entry_bytes(M.make_config(**v2, cache="bf16")) == 1152
    assert M.mla_cache_entry_bytes(M.make_config(**v2, cache="fp8")) == 656
    assert M.mla_cache_entry_bytes(M.make_config(4, 32, 64, 16, 16, cache="f32", act="f32")) == 320
    # invalid: odd RoPE width
    assert M.mla_cache_entry_bytes(M.make_config(4, 32, 64, 15, 16, cache="f32", act="f32")) == 0


def test_host_argument_checks_return_codes():
    lib = M.lib()
    cfg = M.make_config(128, 128, 512, 64, 64)
    bad = M.make_config(128, 128, 512, 63, 64)
    by = ctypes.byref
    # invalid config
    assert lib.mla_decode(by(bad), 1, 1, 1, 1, 1, 1, 1, 1, 1, 0, None, 0, 1, None, None, None) == L.MLA_ERR_INVALID_ARG
    # null pointers
    assert lib.mla_decode(by(cfg), None, 1, 1, 1, 1, 1, 1, 1, 1, 0, None, 0, 1, None, None, None) == L.MLA_ERR_INVALID_ARG
    assert lib.mla_append_cache(by(cfg), None, None, None, None, 4, None, 1, 1, 1, None, None, None) == L.MLA_ERR_INVALID_ARG
    assert lib.mla_absorb_q(by(cfg), None, None, None, 4, None, None, None) == L.MLA_ERR_INVALID_ARG
    assert lib.mla_unabsorb(by(cfg), None, 4, None, None, None) == L.MLA_ERR_INVALID_ARG
    assert lib.mla_append_absorb(by(cfg), None, None, None, None, 4, None, 1, 1, 1, None, None, None, None,
                                 None, None, None) == L.MLA_ERR_INVALID_ARG
    # empty work is a no-op that launches nothing
    assert lib.mla_append_cache(by(cfg), None, None, None, None, 0, None, 1, 1, 1, None, None, None) == L.MLA_OK
    assert lib.mla_append_absorb(by(cfg), None, None, None, None, 0, None, 1, 1, 1, None, None, None, None,
                                 None, None, None) == L.MLA_OK
    assert lib.mla_decode(by(cfg), None, None, None, 1, 1, None, 0, 1, 1, 0, None, 0, None, None, None, None) == L.MLA_OK
    # max_seq_len beyond the page table's reach
    assert lib.mla_decode(by(cfg), 16, 16, 16, 2, 4, 16, 1, 1, 129, 0, None, 0, 16, None, None, None) == L.MLA_ERR_INVALID_ARG
    # n_q larger than max_seq_len
    assert lib.mla_decode(by(cfg), 16, 16, 16, 2, 4, 16, 1, 3, 2, 0, None, 0, 16, None, None, None) == L.MLA_ERR_INVALID_ARG
    # FP8 cache needs bf16 activations
    assert lib.mla_decode_kernel(by(M.make_config(128, 128, 512, 64, 64, cache="fp8", act="f32")), 1, 1) == L.MLA_ERR_UNSUPPORTED
    assert M.mla_status_string(L.MLA_ERR_WORKSPACE) == "workspace too small"


def test_kernel_selection():
    v2 = M.make_config(128, 128, 512, 64, 64)
    tiny = M.make_config(4, 32, 64, 16, 16, cache="f32", act="f32")
    assert M.mla_decode_kernel(tiny, 2, 1) == M.MLA_KERNEL_SIMT
    forced = M.make_config(128, 128, 512, 64, 64, kernel=M.MLA_KERNEL_SIMT)
    assert M.mla_decode_kernel(forced, 64, 1) == M.MLA_KERNEL_SIMT
    k = M.mla_decode_kernel(v2, 64, 1)
    assert k in (M.MLA_KERNEL_SIMT, M.MLA_KERNEL_TC)


def test_fp8_scores_kernel_selection():
    """MLA_KERNEL_TC_FP8_SCORES runs only over an FP8 cache with the tensor-core shapes."""
    fp8 = M.make_config(128, 128, 512, 64, 64, cache="fp8", kernel=M.MLA_KERNEL_TC_FP8_SCORES)
    assert M.mla_decode_kernel(fp8, 64, 1) == M.MLA_KERNEL_TC_FP8_SCORES
    assert M.mla_decode_kernel(fp8, 64, 2) == M.MLA_KERNEL_TC_FP8_SCORES
    bf16 = M.make_config(128, 128, 512, 64, 64, cache="bf16", kernel=M.MLA_KERNEL_TC_FP8_SCORES)
    assert M.mla_decode_kernel(bf16, 64, 1) == L.MLA_ERR_UNSUPPORTED
    small = M.make_config(4, 32, 128, 16, 16, cache="fp8", kernel=M.MLA_KERNEL_TC_FP8_SCORES)
    assert M.mla_decode_kernel(small, 2, 1) == L.MLA_ERR_UNSUPPORTED
    assert M.mla_decode_workspace_size(fp8, 8, 1, 4096, 3) == 8 * 1 * 128 * 3 * (512 + 1) * 4
    bad = M.make_config(128, 128, 512, 64, 64, cache="fp8", kernel=5)
    assert M.mla_decode_kernel(bad, 1, 1) == L.MLA_ERR_INVALID_ARG


def test_fp8_staged_kernel_selection_and_workspace():
    """MLA_KERNEL_TC_FP8_STAGED runs only over an FP8 cache with the tensor-core shapes; its
    workspace is the staged bf16 pool (ceil(max_seq_len / 64) pages of 64 x 1152 bytes per
    sequence), the staged block table (rounded up to 256 bytes), then the tensor-core kernel's
    own workspace."""
    st = M.make_config(128, 128, 512, 64, 64, cache="fp8", kernel=M.MLA_KERNEL_TC_FP8_STAGED)
    assert M.mla_decode_kernel(st, 64, 1) == M.MLA_KERNEL_TC_FP8_STAGED
    assert M.mla_decode_kernel(st, 64, 2) == M.MLA_KERNEL_TC_FP8_STAGED
    bf16 = M.make_config(128, 128, 512, 64, 64, cache="bf16", kernel=M.MLA_KERNEL_TC_FP8_STAGED)
    assert M.mla_decode_kernel(bf16, 64, 1) == L.MLA_ERR_UNSUPPORTED
    small = M.make_config(4, 32, 128, 16, 16, cache="fp8", kernel=M.MLA_KERNEL_TC_FP8_STAGED)
    assert M.mla_decode_kernel(small, 2, 1) == L.MLA_ERR_UNSUPPORTED
    tc = M.make_config(128, 128, 512, 64, 64, cache="fp8", kernel=M.MLA_KERNEL_TC)
    for B, n_q, L_max, splits in ((8, 1, 4096, 3), (5, 2, 1000, 1), (128, 2, 8192, 0)):
        ppr = -(-L_max // 64)
        staged = B * ppr * 64 * 1152 + -(-(B * ppr * 4) // 256) * 256
        assert (M.mla_decode_workspace_size(st, B, n_q, L_max, splits)
                == staged + M.mla_decode_workspace_size(tc, B, n_q, L_max, splits))


def test_tensor_core_workspace_holds_the_plan_and_the_split_tail():
    """Automatic schedule of the tensor-core decode on 148 SMs (74 CTA pairs; the CPU build
    assumes that count): more query rows than pairs need the plan (one int32 per row, rounded
    up to 256 bytes); when the rows left for the last round fill at most half the pairs, those
    rows are split in two and their fp32 partials (2 x (512 + 1) floats per head) come first."""
    cfg = M.make_config(128, 128, 512, 64, 64)

    def up(x):
        return -(-x // 256) * 256

    part = 128 * 2 * (512 + 1) * 4   # one split row's partials, all heads
    assert M.mla_decode_workspace_size(cfg, 64, 1, 4096, 0) == 0                      # 64 rows: one round
    assert M.mla_decode_workspace_size(cfg, 128, 1, 32768, 0) == up(128 * 4)          # 54 left > 37: no split
    assert M.mla_decode_workspace_size(cfg, 45, 2, 700, 0) == up(16 * part) + up(90 * 4)
    assert M.mla_decode_workspace_size(cfg, 128, 2, 8192, 0) == up(34 * part) + up(256 * 4)
    # an explicit split count turns the tail off
    assert M.mla_decode_workspace_size(cfg, 128, 2, 8192, 1) == up(256 * 4)


def test_workspace_size_grows_with_splits():
    cfg = M.make_config(128, 128, 512, 64, 64, kernel=M.MLA_KERNEL_SIMT)
    assert M.mla_decode_workspace_size(cfg, 2, 1, 4096, 1) == 0
    w2 = M.mla_decode_workspace_size(cfg, 2, 1, 4096, 2)
    w4 = M.mla_decode_workspace_size(cfg, 2, 1, 4096, 4)
    assert w2 == 2 * 1 * 128 * 2 * (512 + 1) * 4 and w4 == 2 * w2
