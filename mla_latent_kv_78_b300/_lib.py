"""ctypes binding of libmla_b300.so: argument marshalling only.

Every function here has the name of the C entry point it calls and does
nothing but turn tensors into pointers and sizes; all arithmetic runs in the
library's CUDA kernels. Tensors must already live on the CUDA device (the
library takes device pointers) and be contiguous. There is no fallback: if
the library is missing, loading it raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmla_b300.so")

MLA_OK = 0
MLA_ERR_INVALID_ARG = -1
MLA_ERR_UNSUPPORTED = -2
MLA_ERR_WORKSPACE = -3
MLA_ERR_ALIGNMENT = -4
MLA_ERR_CUDA = -5
MLA_ERR_SCRATCH_LIMIT = -6
NOALLOC_SCRATCH_BYTES = 32 << 20

MLA_DEV_INDEX_OUT_OF_RANGE = 1
MLA_DEV_BAD_SEQLEN = 2
MLA_DEV_TIMEOUT = 4

MLA_F32, MLA_BF16, MLA_FP8_E4M3 = 0, 1, 2
MLA_KERNEL_AUTO, MLA_KERNEL_SIMT, MLA_KERNEL_TC, MLA_KERNEL_TC_FP8_SCORES = 0, 1, 2, 3
MLA_KERNEL_TC_FP8_STAGED = 4

_DTYPES = {"f32": MLA_F32, "bf16": MLA_BF16, "fp8": MLA_FP8_E4M3}
TORCH_ACT = {MLA_F32: torch.float32, MLA_BF16: torch.bfloat16}


class MlaError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} returned {code} ({mla_status_string(code)})")
        self.code = code


class mla_config(ctypes.Structure):
    _fields_ = [
        ("n_heads", ctypes.c_int32),
        ("d_head", ctypes.c_int32),
        ("d_latent", ctypes.c_int32),
        ("d_rope", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("cache_dtype", ctypes.c_int32),
        ("act_dtype", ctypes.c_int32),
        ("kernel", ctypes.c_int32),
        ("softmax_scale", ctypes.c_float),
        ("rope_base", ctypes.c_float),
        ("rope_scaling", ctypes.c_float),
        ("rope_orig_context", ctypes.c_int32),
        ("rope_yarn_alpha", ctypes.c_float),
        ("rope_yarn_beta", ctypes.c_float),
        ("rope_mscale_coef", ctypes.c_float),
    ]


def make_config(H: int, D: int, C: int, R: int, P: int, cache: str = "bf16", act: str = "bf16",
                kernel: int = MLA_KERNEL_AUTO, softmax_scale: float = 0.0,
                rope_base: float = 10000.0, rope_scaling: float = 0.0,
                rope_orig_context: int = 0, rope_yarn_alpha: float = 0.0,
                rope_yarn_beta: float = 0.0, rope_mscale_coef: float = 0.0) -> mla_config:
    """A filled mla_config; the rope_* YaRN fields stay 0 (plain RoPE) unless given."""
    return mla_config(H, D, C, R, P, _DTYPES[cache], _DTYPES[act], kernel, softmax_scale, rope_base,
                      rope_scaling, rope_orig_context, rope_yarn_alpha, rope_yarn_beta,
                      rope_mscale_coef)


_lib: Optional[ctypes.CDLL] = None

_P = ctypes.c_void_p
_I = ctypes.c_int32
_SIGS = {
    "mla_cache_entry_bytes": (ctypes.c_size_t, [ctypes.POINTER(mla_config)]),
    "mla_append_cache": (ctypes.c_int, [ctypes.POINTER(mla_config), _P, _P, _P, _P, _I, _P, _I, _I,
                                        _I, _P, _P, _P]),
    "mla_absorb_q": (ctypes.c_int, [ctypes.POINTER(mla_config), _P, _P, _P, _I, _P, _P, _P]),
    "mla_append_absorb": (ctypes.c_int, [ctypes.POINTER(mla_config), _P, _P, _P, _P, _I, _P, _I, _I,
                                         _I, _P, _P, _P, _P, _P, _P, _P]),
    "mla_decode_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(mla_config), _I, _I, _I, _I]),
    "mla_decode_kernel": (ctypes.c_int, [ctypes.POINTER(mla_config), _I, _I]),
    "mla_decode": (ctypes.c_int, [ctypes.POINTER(mla_config), _P, _P, _P, _I, _I, _P, _I, _I, _I,
                                  _I, _P, ctypes.c_size_t, _P, _P, _P, _P]),
    "mla_unabsorb": (ctypes.c_int, [ctypes.POINTER(mla_config), _P, _I, _P, _P, _P]),
    "mla_decode_noalloc": (ctypes.c_int, [ctypes.POINTER(mla_config), _P, _P, _P, _I, _I, _P, _I,
                                          _I, _I, _I, _P, _P, _P, _P]),
    "mla_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "mla_project_append_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(mla_config), _I, _I]),
    "mla_project_append": (ctypes.c_int, [ctypes.POINTER(mla_config), _P, _I, _I, _P, _P, ctypes.c_float,
                                          _P, _P, _P, _I, _I, _I, _P, _P, ctypes.c_size_t, _P, _P]),
    "mla_output_projection_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(mla_config), _I, _I]),
    "mla_prefill_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(mla_config), _I]),
    "mla_prefill": (ctypes.c_int, [ctypes.POINTER(mla_config), _P, _P, _I, _P, _P, _P, _P, _P, _P,
                                   ctypes.c_size_t, _P, _P]),
    "mla_output_projection": (ctypes.c_int, [ctypes.POINTER(mla_config), _P, _I, _P, _I, _P, _P,
                                             ctypes.c_size_t, _P, _P]),
    "mla_debug_decode_fault": (ctypes.c_int, [ctypes.c_longlong, ctypes.c_int32]),
}
EXPORTED = tuple(_SIGS)


def lib() -> ctypes.CDLL:
    """Load libmla_b300.so from this package directory (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: run `python -m mla_latent_kv_78_b300.build`")
        l = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(l, name)
            f.restype = res
            f.argtypes = args
        _lib = l
    return _lib


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libmla_b300 takes device tensors")
    if not t.is_contiguous():
        raise ValueError("libmla_b300 takes contiguous tensors")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(fn: str, rc: int) -> None:
    if rc != MLA_OK:
        raise MlaError(fn, rc)


def mla_status_string(code: int) -> str:
    return lib().mla_status_string(code).decode()


def mla_cache_entry_bytes(cfg: mla_config) -> int:
    return int(lib().mla_cache_entry_bytes(ctypes.byref(cfg)))


def mla_append_cache(cfg: mla_config, c_kv, k_r, seq_idx, pos, block_table, kv_pool,
                     num_pages: Optional[int] = None, dev_status=None, stream=None) -> None:
    T = c_kv.shape[0]
    batch, maxp = block_table.shape
    if num_pages is None:
        num_pages = kv_pool.shape[0]
    _check("mla_append_cache", lib().mla_append_cache(
        ctypes.byref(cfg), _ptr(c_kv), _ptr(k_r), _ptr(seq_idx), _ptr(pos), T, _ptr(block_table),
        batch, maxp, num_pages, _ptr(kv_pool), _ptr(dev_status), _stream(stream)))


def mla_absorb_q(cfg: mla_config, q_c, q_r, pos, w_uk, q_lat, stream=None) -> None:
    T = q_c.shape[0]
    _check("mla_absorb_q", lib().mla_absorb_q(ctypes.byref(cfg), _ptr(q_c), _ptr(q_r), _ptr(pos),
                                              T, _ptr(w_uk), _ptr(q_lat), _stream(stream)))


def mla_append_absorb(cfg: mla_config, c_kv, k_r, seq_idx, pos, block_table, kv_pool, q_c, q_r,
                      w_uk, q_lat, num_pages: Optional[int] = None, dev_status=None,
                      stream=None) -> None:
    T = c_kv.shape[0]
    if q_c.shape[0] != T:
        raise ValueError("c_kv and q_c must hold the same tokens")
    batch, maxp = block_table.shape
    if num_pages is None:
        num_pages = kv_pool.shape[0]
    _check("mla_append_absorb", lib().mla_append_absorb(
        ctypes.byref(cfg), _ptr(c_kv), _ptr(k_r), _ptr(seq_idx), _ptr(pos), T, _ptr(block_table),
        batch, maxp, num_pages, _ptr(kv_pool), _ptr(dev_status), _ptr(q_c), _ptr(q_r),
        _ptr(w_uk), _ptr(q_lat), _stream(stream)))


def mla_decode_workspace_size(cfg: mla_config, batch: int, n_q: int, max_seq_len: int,
                              num_splits: int = 0) -> int:
    return int(lib().mla_decode_workspace_size(ctypes.byref(cfg), batch, n_q, max_seq_len,
                                               num_splits))


def mla_decode_kernel(cfg: mla_config, batch: int, n_q: int) -> int:
    return int(lib().mla_decode_kernel(ctypes.byref(cfg), batch, n_q))


def mla_decode(cfg: mla_config, q_lat, kv_pool, block_table, seq_lens, n_q: int,
               max_seq_len: int, o_lat, lse=None, workspace=None, num_splits: int = 0,
               num_pages: Optional[int] = None, dev_status=None, stream=None) -> None:
    batch, maxp = block_table.shape
    if num_pages is None:
        num_pages = kv_pool.shape[0]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("mla_decode", lib().mla_decode(
        ctypes.byref(cfg), _ptr(q_lat), _ptr(kv_pool), _ptr(block_table), maxp, num_pages,
        _ptr(seq_lens), batch, n_q, max_seq_len, num_splits, _ptr(workspace), ws_bytes,
        _ptr(o_lat), _ptr(lse), _ptr(dev_status), _stream(stream)))


def mla_decode_noalloc(cfg: mla_config, q_lat, kv_pool, block_table, seq_lens, n_q: int,
                       max_seq_len: int, o_lat, lse=None, num_splits: int = 0,
                       num_pages: Optional[int] = None, dev_status=None, stream=None) -> None:
    """mla_decode with the library's fixed device scratch instead of a workspace argument
    (for callers that cannot allocate device memory)."""
    batch, maxp = block_table.shape
    if num_pages is None:
        num_pages = kv_pool.shape[0]
    _check("mla_decode_noalloc", lib().mla_decode_noalloc(
        ctypes.byref(cfg), _ptr(q_lat), _ptr(kv_pool), _ptr(block_table), maxp, num_pages,
        _ptr(seq_lens), batch, n_q, max_seq_len, num_splits, _ptr(o_lat), _ptr(lse),
        _ptr(dev_status), _stream(stream)))


def mla_project_append_workspace_size(cfg: mla_config, d_model: int, num_tokens: int) -> int:
    return int(lib().mla_project_append_workspace_size(ctypes.byref(cfg), d_model, num_tokens))


def mla_project_append(cfg: mla_config, h, w_dkv_kr, gain, eps: float, seq_idx, pos, block_table,
                       kv_pool, workspace, num_pages: Optional[int] = None, dev_status=None,
                       stream=None) -> None:
    T, d_model = h.shape
    batch, maxp = block_table.shape
    if num_pages is None:
        num_pages = kv_pool.shape[0]
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("mla_project_append", lib().mla_project_append(
        ctypes.byref(cfg), _ptr(h), d_model, T, _ptr(w_dkv_kr), _ptr(gain), eps, _ptr(seq_idx),
        _ptr(pos), _ptr(block_table), batch, maxp, num_pages, _ptr(kv_pool), _ptr(workspace),
        ws_bytes, _ptr(dev_status), _stream(stream)))


def mla_output_projection_workspace_size(cfg: mla_config, d_model: int, num_tokens: int) -> int:
    return int(lib().mla_output_projection_workspace_size(ctypes.byref(cfg), d_model, num_tokens))


def mla_output_projection(cfg: mla_config, o, w_o, u, workspace=None, dev_status=None,
                          stream=None) -> None:
    T = o.shape[0]
    d_model = w_o.shape[0]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("mla_output_projection", lib().mla_output_projection(
        ctypes.byref(cfg), _ptr(o), T, _ptr(w_o), d_model, _ptr(u), _ptr(workspace), ws_bytes,
        _ptr(dev_status), _stream(stream)))


def mla_prefill_workspace_size(cfg: mla_config, prompt_len: int) -> int:
    return int(lib().mla_prefill_workspace_size(ctypes.byref(cfg), prompt_len))


def mla_prefill(cfg: mla_config, c_kv, k_r, q_c, q_r, w_uk, w_uv, o, workspace, dev_status=None,
                stream=None) -> None:
    L = c_kv.shape[0]
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("mla_prefill", lib().mla_prefill(
        ctypes.byref(cfg), _ptr(c_kv), _ptr(k_r), L, _ptr(q_c), _ptr(q_r), _ptr(w_uk), _ptr(w_uv),
        _ptr(o), _ptr(workspace), ws_bytes, _ptr(dev_status), _stream(stream)))


def mla_unabsorb(cfg: mla_config, o_lat, w_uv, o, stream=None) -> None:
    T = o_lat.shape[0]
    _check("mla_unabsorb", lib().mla_unabsorb(ctypes.byref(cfg), _ptr(o_lat), T, _ptr(w_uv),
                                              _ptr(o), _stream(stream)))
