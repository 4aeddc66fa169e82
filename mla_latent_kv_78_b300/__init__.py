"""B300-native DeepSeek-V2 Multi-head Latent Attention (MLA) decode.

The compute lives in libmla_b300.so (CUDA for sm_103a, C ABI in
include/mla.h); this package is its Python binding plus a small helper that
owns the device buffers of one decode step.
"""
from ._lib import (  # noqa: F401
    EXPORTED,
    MLA_BF16,
    MLA_DEV_BAD_SEQLEN,
    MLA_DEV_INDEX_OUT_OF_RANGE,
    MLA_DEV_TIMEOUT,
    MLA_ERR_INVALID_ARG,
    MLA_F32,
    MLA_FP8_E4M3,
    MLA_KERNEL_AUTO,
    MLA_KERNEL_SIMT,
    MLA_KERNEL_TC,
    MLA_KERNEL_TC_FP8_SCORES,
    MLA_KERNEL_TC_FP8_STAGED,
    MlaError,
    lib,
    make_config,
    mla_absorb_q,
    mla_append_absorb,
    mla_append_cache,
    mla_cache_entry_bytes,
    mla_config,
    mla_decode,
    mla_decode_kernel,
    mla_decode_noalloc,
    mla_decode_workspace_size,
    mla_output_projection,
    mla_output_projection_workspace_size,
    mla_prefill,
    mla_prefill_workspace_size,
    mla_project_append,
    mla_project_append_workspace_size,
    mla_status_string,
    mla_unabsorb,
)
from .step import DecodeStep  # noqa: F401
