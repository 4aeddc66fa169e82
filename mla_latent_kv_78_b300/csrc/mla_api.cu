// C-ABI front end of libmla_b300.so: argument checks on the host, then one
// launch sequence per call on the caller's stream. Nothing here allocates.
#include <math.h>
#include <stdio.h>

#include "mla_internal.cuh"

using mla::Dims;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t entry_bytes(const mla_config* c) {
  switch (c->cache_dtype) {
    case MLA_F32: return (size_t)(c->d_latent + c->d_rope) * 4;
    case MLA_BF16: return (size_t)(c->d_latent + c->d_rope) * 2;
    case MLA_FP8_E4M3:
      return (size_t)c->d_latent + 2 * (size_t)c->d_rope + 4 * (size_t)(c->d_latent / mla::kFp8Group);
    default: return 0;
  }
}

// Validates the config and fills Dims. Returns MLA_OK or an error code.
int make_dims(const mla_config* c, Dims* d) {
  if (!c) return MLA_ERR_INVALID_ARG;
  if (c->n_heads < 1 || c->d_head < 1 || c->d_latent < 1 || c->d_rope < 0 || (c->d_rope & 1) ||
      c->page_size < 1)
    return MLA_ERR_INVALID_ARG;
  if (c->act_dtype != MLA_F32 && c->act_dtype != MLA_BF16) return MLA_ERR_INVALID_ARG;
  if (c->cache_dtype != MLA_F32 && c->cache_dtype != MLA_BF16 && c->cache_dtype != MLA_FP8_E4M3)
    return MLA_ERR_INVALID_ARG;
  if (c->kernel < MLA_KERNEL_AUTO || c->kernel > MLA_KERNEL_TC_FP8_STAGED) return MLA_ERR_INVALID_ARG;
  if (c->d_latent > 512) return MLA_ERR_UNSUPPORTED;   // SIMT register tile bound
  // the cache input type follows the cache: fp32 cache <- fp32 latents, else bf16
  if (c->cache_dtype == MLA_FP8_E4M3) {
    if (c->d_latent % mla::kFp8Group) return MLA_ERR_UNSUPPORTED;
    if (c->act_dtype != MLA_BF16) return MLA_ERR_UNSUPPORTED;
  }
  d->H = c->n_heads;
  d->D = c->d_head;
  d->C = c->d_latent;
  d->R = c->d_rope;
  d->P = c->page_size;
  d->cache_dtype = c->cache_dtype;
  d->act_dtype = c->act_dtype;
  d->scale = c->softmax_scale > 0.f ? c->softmax_scale : 1.0f / sqrtf((float)(c->d_head + c->d_rope));
  d->rope_base = c->rope_base > 0.f ? c->rope_base : 10000.0f;
  d->entry_bytes = (int)entry_bytes(c);
  d->fp8_scores = false;
  // YaRN (「一文通透DeepSeek-V2」 §3.1.3): defaults are the page's values
  d->yarn_s = c->rope_scaling > 1.f ? c->rope_scaling : 1.f;
  d->yarn_orig = c->rope_orig_context > 0 ? c->rope_orig_context : 4096;
  d->yarn_alpha = c->rope_yarn_alpha > 0.f ? c->rope_yarn_alpha : 1.f;
  d->yarn_beta = c->rope_yarn_beta > 0.f ? c->rope_yarn_beta : 32.f;
  if (d->yarn_s > 1.f) {
    if (!(d->yarn_beta > d->yarn_alpha) || c->rope_orig_context < 0) return MLA_ERR_INVALID_ARG;
    if (d->R / 2 > mla::kMaxRopePairs) return MLA_ERR_UNSUPPORTED;
    const float coef = c->rope_mscale_coef > 0.f ? c->rope_mscale_coef : 0.0707f;
    const float sqrt_t = coef * logf(d->yarn_s) + 1.f;
    d->scale *= sqrt_t * sqrt_t;
  }
  if (c->cache_dtype == MLA_FP8_E4M3 && (d->entry_bytes % 16)) return MLA_ERR_UNSUPPORTED;
  return MLA_OK;
}

int num_sms() {
  int dev = 0, n = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n;
}

int cuda_rc(cudaError_t e) {
  if (e == cudaSuccess) return MLA_OK;
  fprintf(stderr, "libmla_b300: CUDA error %d (%s)\n", (int)e, cudaGetErrorString(e));
  return MLA_ERR_CUDA;
}

// Which decode kernel runs for this config and shape.
int pick_kernel(const mla_config* c, const Dims& d, int n_q) {
  const bool tc_ok = mla::tc_supported(d, n_q);
  if (c->kernel == MLA_KERNEL_SIMT) return MLA_KERNEL_SIMT;
  if (c->kernel == MLA_KERNEL_TC) return tc_ok ? MLA_KERNEL_TC : MLA_ERR_UNSUPPORTED;
  if (c->kernel == MLA_KERNEL_TC_FP8_SCORES)
    return tc_ok && d.cache_dtype == MLA_FP8_E4M3 ? MLA_KERNEL_TC_FP8_SCORES : MLA_ERR_UNSUPPORTED;
  if (c->kernel == MLA_KERNEL_TC_FP8_STAGED)
    return tc_ok && d.cache_dtype == MLA_FP8_E4M3 ? MLA_KERNEL_TC_FP8_STAGED : MLA_ERR_UNSUPPORTED;
  return tc_ok ? MLA_KERNEL_TC : MLA_KERNEL_SIMT;
}

}  // namespace

extern "C" {

size_t mla_cache_entry_bytes(const mla_config* cfg) {
  Dims d;
  if (make_dims(cfg, &d) != MLA_OK) return 0;
  return (size_t)d.entry_bytes;
}

const char* mla_status_string(int code) {
  switch (code) {
    case MLA_OK: return "ok";
    case MLA_ERR_INVALID_ARG: return "invalid argument";
    case MLA_ERR_UNSUPPORTED: return "unsupported configuration";
    case MLA_ERR_WORKSPACE: return "workspace too small";
    case MLA_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case MLA_ERR_CUDA: return "CUDA error";
    case MLA_ERR_SCRATCH_LIMIT: return "sizes exceed the fixed scratch of mla_decode_noalloc";
    default: return "unknown status";
  }
}

int mla_append_cache(const mla_config* cfg, const void* c_kv, const void* k_r,
                     const int32_t* seq_idx, const int32_t* pos, int32_t num_tokens,
                     const int32_t* block_table, int32_t batch, int32_t max_pages_per_seq,
                     int32_t num_pages, void* kv_pool, int32_t* dev_status, void* stream) {
  Dims d;
  int rc = make_dims(cfg, &d);
  if (rc != MLA_OK) return rc;
  if (num_tokens < 0 || batch < 0 || max_pages_per_seq < 0 || num_pages < 0)
    return MLA_ERR_INVALID_ARG;
  if (num_tokens == 0) return MLA_OK;
  if (!c_kv || !k_r || !seq_idx || !pos || !block_table || !kv_pool || batch < 1 ||
      max_pages_per_seq < 1 || num_pages < 1)
    return MLA_ERR_INVALID_ARG;
  if (d.cache_dtype == MLA_FP8_E4M3 && !aligned16(kv_pool)) return MLA_ERR_ALIGNMENT;
  return cuda_rc(mla::launch_append(d, c_kv, k_r, seq_idx, pos, num_tokens, block_table, batch,
                                    max_pages_per_seq, num_pages, kv_pool, dev_status,
                                    (cudaStream_t)stream));
}

int mla_absorb_q(const mla_config* cfg, const void* q_c, const void* q_r, const int32_t* pos,
                 int32_t num_tokens, const void* w_uk, void* q_lat, void* stream) {
  Dims d;
  int rc = make_dims(cfg, &d);
  if (rc != MLA_OK) return rc;
  if (num_tokens < 0) return MLA_ERR_INVALID_ARG;
  if (num_tokens == 0) return MLA_OK;
  if (!q_c || (!q_r && d.R > 0) || !pos || !w_uk || !q_lat) return MLA_ERR_INVALID_ARG;
  if (mla::absorb_tc_supported(d) && cfg->kernel != MLA_KERNEL_SIMT) {
    if (!aligned16(q_c) || !aligned16(q_r) || !aligned16(w_uk) || !aligned16(q_lat))
      return MLA_ERR_ALIGNMENT;
    return cuda_rc(mla::launch_absorb_tc(d, q_c, q_r, pos, num_tokens, w_uk, q_lat, (cudaStream_t)stream));
  }
  return cuda_rc(mla::launch_absorb(d, q_c, q_r, pos, num_tokens, w_uk, q_lat, (cudaStream_t)stream));
}

int mla_append_absorb(const mla_config* cfg, const void* c_kv, const void* k_r,
                      const int32_t* seq_idx, const int32_t* pos, int32_t num_tokens,
                      const int32_t* block_table, int32_t batch, int32_t max_pages_per_seq,
                      int32_t num_pages, void* kv_pool, int32_t* dev_status, const void* q_c,
                      const void* q_r, const void* w_uk, void* q_lat, void* stream) {
  Dims d;
  int rc = make_dims(cfg, &d);
  if (rc != MLA_OK) return rc;
  if (num_tokens < 0 || batch < 0 || max_pages_per_seq < 0 || num_pages < 0)
    return MLA_ERR_INVALID_ARG;
  if (num_tokens == 0) return MLA_OK;
  // every argument of both halves is checked before anything is launched
  if (!c_kv || !k_r || !seq_idx || !pos || !block_table || !kv_pool || batch < 1 ||
      max_pages_per_seq < 1 || num_pages < 1)
    return MLA_ERR_INVALID_ARG;
  if (!q_c || (!q_r && d.R > 0) || !w_uk || !q_lat) return MLA_ERR_INVALID_ARG;
  if (d.cache_dtype == MLA_FP8_E4M3 && !aligned16(kv_pool)) return MLA_ERR_ALIGNMENT;
  const bool tc = mla::absorb_tc_supported(d) && cfg->kernel != MLA_KERNEL_SIMT;
  if (tc && (!aligned16(q_c) || !aligned16(q_r) || !aligned16(w_uk) || !aligned16(q_lat)))
    return MLA_ERR_ALIGNMENT;
  const cudaStream_t s = (cudaStream_t)stream;
  rc = cuda_rc(mla::launch_append(d, c_kv, k_r, seq_idx, pos, num_tokens, block_table, batch,
                                  max_pages_per_seq, num_pages, kv_pool, dev_status, s));
  if (rc != MLA_OK) return rc;
  // the append is an ordinary launch (everything before it on the stream has completed when
  // it starts) and writes only the cache, so the absorption behind it may read its inputs at
  // once; it still completes only after the append has
  if (tc) return cuda_rc(mla::launch_absorb_tc(d, q_c, q_r, pos, num_tokens, w_uk, q_lat, s, true));
  return cuda_rc(mla::launch_absorb(d, q_c, q_r, pos, num_tokens, w_uk, q_lat, s));
}

size_t mla_decode_workspace_size(const mla_config* cfg, int32_t batch, int32_t n_q,
                                 int32_t max_seq_len, int32_t num_splits) {
  Dims d;
  if (make_dims(cfg, &d) != MLA_OK || batch < 1 || n_q < 1 || max_seq_len < 1 || num_splits < 0)
    return 0;
  const int k = pick_kernel(cfg, d, n_q);
  if (k == MLA_KERNEL_TC || k == MLA_KERNEL_TC_FP8_SCORES)
    return mla::tc_workspace_bytes(d, batch, n_q, max_seq_len, num_splits, num_sms());
  if (k == MLA_KERNEL_TC_FP8_STAGED)
    return mla::fp8_staged_bytes(batch, max_seq_len) +
           mla::tc_workspace_bytes(d, batch, n_q, max_seq_len, num_splits, num_sms());
  if (k != MLA_KERNEL_SIMT) return 0;
  const int S = mla::simt_pick_splits(d, batch, n_q, max_seq_len, num_splits, num_sms());
  return mla::simt_workspace_bytes(d, batch, n_q, S);
}

int mla_decode_kernel(const mla_config* cfg, int32_t batch, int32_t n_q) {
  Dims d;
  int rc = make_dims(cfg, &d);
  if (rc != MLA_OK) return rc;
  if (batch < 0 || n_q < 1) return MLA_ERR_INVALID_ARG;
  return pick_kernel(cfg, d, n_q);
}

int mla_decode(const mla_config* cfg, const void* q_lat, const void* kv_pool,
               const int32_t* block_table, int32_t max_pages_per_seq, int32_t num_pages,
               const int32_t* seq_lens, int32_t batch, int32_t n_q, int32_t max_seq_len,
               int32_t num_splits, void* workspace, size_t workspace_bytes, void* o_lat,
               float* lse, int32_t* dev_status, void* stream) {
  Dims d;
  int rc = make_dims(cfg, &d);
  if (rc != MLA_OK) return rc;
  if (batch < 0 || n_q < 1 || max_seq_len < 0 || num_splits < 0 || max_pages_per_seq < 0 ||
      num_pages < 0)
    return MLA_ERR_INVALID_ARG;
  if (batch == 0) return MLA_OK;
  if (!q_lat || !kv_pool || !block_table || !seq_lens || !o_lat || max_seq_len < n_q ||
      max_pages_per_seq < 1 || num_pages < 1)
    return MLA_ERR_INVALID_ARG;
  if ((long)max_pages_per_seq * d.P < (long)max_seq_len) return MLA_ERR_INVALID_ARG;
  const int k = pick_kernel(cfg, d, n_q);
  if (k < 0) return k;
  if (k == MLA_KERNEL_TC || k == MLA_KERNEL_TC_FP8_SCORES) {
    d.fp8_scores = k == MLA_KERNEL_TC_FP8_SCORES;
    const size_t need = mla::tc_workspace_bytes(d, batch, n_q, max_seq_len, num_splits, num_sms());
    if (workspace_bytes < need || (need && !workspace)) return MLA_ERR_WORKSPACE;
    if (!aligned16(q_lat) || !aligned16(kv_pool) || !aligned16(o_lat) || !aligned16(workspace))
      return MLA_ERR_ALIGNMENT;
    return cuda_rc(mla::launch_decode_tc(d, q_lat, kv_pool, block_table, max_pages_per_seq,
                                         num_pages, seq_lens, batch, n_q, max_seq_len, num_splits,
                                         workspace, workspace_bytes, o_lat, lse, dev_status,
                                         (cudaStream_t)stream));
  }
  if (k == MLA_KERNEL_TC_FP8_STAGED) {
    // the staging grid is (pages per row, batch); the staged pool's rows must fit an int
    if (batch > 65535 || (long)batch * ((max_seq_len + d.P - 1) / d.P) * d.P > 0x7fffffffL)
      return MLA_ERR_UNSUPPORTED;
    const size_t need = mla::fp8_staged_bytes(batch, max_seq_len) +
                        mla::tc_workspace_bytes(d, batch, n_q, max_seq_len, num_splits, num_sms());
    if (workspace_bytes < need || !workspace) return MLA_ERR_WORKSPACE;
    if (!aligned16(q_lat) || !aligned16(kv_pool) || !aligned16(o_lat) || !aligned16(workspace))
      return MLA_ERR_ALIGNMENT;
    return cuda_rc(mla::launch_decode_tc_fp8_staged(d, q_lat, kv_pool, block_table, max_pages_per_seq,
                                                    num_pages, seq_lens, batch, n_q, max_seq_len,
                                                    num_splits, workspace, workspace_bytes, o_lat, lse,
                                                    dev_status, (cudaStream_t)stream));
  }
  const int S = mla::simt_pick_splits(d, batch, n_q, max_seq_len, num_splits, num_sms());
  const size_t need = mla::simt_workspace_bytes(d, batch, n_q, S);
  if (workspace_bytes < need || (need && !workspace)) return MLA_ERR_WORKSPACE;
  if (need && !aligned16(workspace)) return MLA_ERR_ALIGNMENT;
  return cuda_rc(mla::launch_decode_simt(d, q_lat, kv_pool, block_table, max_pages_per_seq,
                                         num_pages, seq_lens, batch, n_q, max_seq_len, S, workspace,
                                         o_lat, lse, dev_status, (cudaStream_t)stream));
}

size_t mla_project_append_workspace_size(const mla_config* cfg, int32_t d_model, int32_t num_tokens) {
  Dims d;
  if (make_dims(cfg, &d) != MLA_OK || d_model < 1 || num_tokens < 1) return 0;
  const int N = d.C + d.R;
  const int s = mla::gemm_pick_splits(num_tokens, N, d_model, num_sms());
  return ((size_t)s * num_tokens * N * sizeof(float) + 255) / 256 * 256;
}

int mla_project_append(const mla_config* cfg, const void* h, int32_t d_model, int32_t num_tokens,
                       const void* w_dkv_kr, const float* gain, float eps, const int32_t* seq_idx,
                       const int32_t* pos, const int32_t* block_table, int32_t batch,
                       int32_t max_pages_per_seq, int32_t num_pages, void* kv_pool,
                       void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream) {
  Dims d;
  int rc = make_dims(cfg, &d);
  if (rc != MLA_OK) return rc;
  if (num_tokens < 0 || d_model < 1 || batch < 0 || max_pages_per_seq < 0 || num_pages < 0 || !(eps > 0.f))
    return MLA_ERR_INVALID_ARG;
  if (num_tokens == 0) return MLA_OK;
  if (d.act_dtype != MLA_BF16 || d.cache_dtype == MLA_F32) return MLA_ERR_UNSUPPORTED;
  if (d_model % 8 || d.C % 8 || d.R % 2) return MLA_ERR_UNSUPPORTED;
  if (!h || !w_dkv_kr || !gain || !seq_idx || !pos || !block_table || !kv_pool || batch < 1 ||
      max_pages_per_seq < 1 || num_pages < 1)
    return MLA_ERR_INVALID_ARG;
  if (!aligned16(h) || !aligned16(w_dkv_kr) || !aligned16(kv_pool)) return MLA_ERR_ALIGNMENT;
  const size_t need = mla_project_append_workspace_size(cfg, d_model, num_tokens);
  if (workspace_bytes < need || !workspace) return MLA_ERR_WORKSPACE;
  if (!aligned16(workspace)) return MLA_ERR_ALIGNMENT;
  const int splits = mla::gemm_pick_splits(num_tokens, d.C + d.R, d_model, num_sms());
  return cuda_rc(mla::launch_project_append(d, h, d_model, w_dkv_kr, num_tokens, gain, eps, seq_idx,
                                            pos, block_table, batch, max_pages_per_seq, num_pages,
                                            kv_pool, workspace, splits, dev_status,
                                            (cudaStream_t)stream));
}

size_t mla_output_projection_workspace_size(const mla_config* cfg, int32_t d_model, int32_t num_tokens) {
  Dims d;
  if (make_dims(cfg, &d) != MLA_OK || d_model < 1 || num_tokens < 1) return 0;
  return mla::gemm_workspace_bytes(num_tokens, d_model, d.H * d.D, MLA_F32, num_sms());
}

int mla_output_projection(const mla_config* cfg, const void* o, int32_t num_tokens, const void* w_o,
                          int32_t d_model, float* u, void* workspace, size_t workspace_bytes,
                          int32_t* dev_status, void* stream) {
  Dims d;
  int rc = make_dims(cfg, &d);
  if (rc != MLA_OK) return rc;
  if (num_tokens < 0 || d_model < 1) return MLA_ERR_INVALID_ARG;
  if (num_tokens == 0) return MLA_OK;
  if (d.act_dtype != MLA_BF16) return MLA_ERR_UNSUPPORTED;
  const int K = d.H * d.D;
  if (K % 8 || d_model % 8) return MLA_ERR_UNSUPPORTED;
  if (!o || !w_o || !u) return MLA_ERR_INVALID_ARG;
  if (!aligned16(o) || !aligned16(w_o)) return MLA_ERR_ALIGNMENT;
  const size_t need = mla_output_projection_workspace_size(cfg, d_model, num_tokens);
  if (workspace_bytes < need || (need && !workspace)) return MLA_ERR_WORKSPACE;
  if (need && !aligned16(workspace)) return MLA_ERR_ALIGNMENT;
  const int splits = mla::gemm_pick_splits(num_tokens, d_model, K, num_sms());
  return cuda_rc(mla::launch_gemm(o, w_o, num_tokens, d_model, K, splits, static_cast<float*>(workspace),
                                  u, MLA_F32, dev_status, (cudaStream_t)stream));
}

size_t mla_prefill_workspace_size(const mla_config* cfg, int32_t prompt_len) {
  Dims d;
  if (make_dims(cfg, &d) != MLA_OK || prompt_len < 1 || !mla::prefill_supported(d)) return 0;
  return mla::prefill_workspace_bytes(d, prompt_len);
}

int mla_prefill(const mla_config* cfg, const void* c_kv, const void* k_r, int32_t prompt_len,
                const void* q_c, const void* q_r, const void* w_uk, const void* w_uv, float* o,
                void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream) {
  Dims d;
  int rc = make_dims(cfg, &d);
  if (rc != MLA_OK) return rc;
  if (prompt_len < 0) return MLA_ERR_INVALID_ARG;
  if (prompt_len == 0) return MLA_OK;
  if (!mla::prefill_supported(d)) return MLA_ERR_UNSUPPORTED;
  if (!c_kv || !k_r || !q_c || !q_r || !w_uk || !w_uv || !o) return MLA_ERR_INVALID_ARG;
  if (!aligned16(c_kv) || !aligned16(k_r) || !aligned16(q_c) || !aligned16(q_r) || !aligned16(w_uk) ||
      !aligned16(w_uv) || !aligned16(o))
    return MLA_ERR_ALIGNMENT;
  if (workspace_bytes < mla::prefill_workspace_bytes(d, prompt_len) || !workspace) return MLA_ERR_WORKSPACE;
  if (!aligned16(workspace)) return MLA_ERR_ALIGNMENT;
  return cuda_rc(mla::launch_prefill(d, c_kv, k_r, prompt_len, q_c, q_r, w_uk, w_uv, o, workspace,
                                     dev_status, (cudaStream_t)stream));
}

int mla_unabsorb(const mla_config* cfg, const void* o_lat, int32_t num_tokens, const void* w_uv,
                 float* o, void* stream) {
  Dims d;
  int rc = make_dims(cfg, &d);
  if (rc != MLA_OK) return rc;
  if (num_tokens < 0) return MLA_ERR_INVALID_ARG;
  if (num_tokens == 0) return MLA_OK;
  if (!o_lat || !w_uv || !o) return MLA_ERR_INVALID_ARG;
  if (mla::absorb_tc_supported(d) && cfg->kernel != MLA_KERNEL_SIMT) {
    if (!aligned16(o_lat) || !aligned16(w_uv)) return MLA_ERR_ALIGNMENT;
    return cuda_rc(mla::launch_unabsorb_tc(d, o_lat, num_tokens, w_uv, o, (cudaStream_t)stream));
  }
  return cuda_rc(mla::launch_unabsorb(d, o_lat, num_tokens, w_uv, o, (cudaStream_t)stream));
}

}  // extern "C"
