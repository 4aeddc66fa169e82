/*
 * mla.h — C ABI of the B300 (sm_103a) DeepSeek-V2 Multi-head Latent Attention
 * decode library (libmla_b300.so).
 *
 * The method. Each token caches only a compressed latent c^{KV} (d_c values)
 * and one decoupled RoPE key k^R (d_h^R values) shared by all heads
 * (「一文通透DeepSeek-V2」 §2.2.1 low-rank joint KV compression, §2.2.2 decoupled
 * RoPE and the (d_c + d_h^R)·l cache). At decode time W^{UK} is absorbed into
 * the query and W^{UV} into the output, so every head scores against the
 * shared [c^{KV}; k^R] vector (§2.2.1 last paragraph; 「Deepseek系列从v3到R易
 * 背面经版」 MLA: MHA becomes MQA) with the scale 1/sqrt(d_h + d_h^R)
 * (「deepseek(2)——deepseek 關鍵技術」 §1).
 *
 * One decode step is four calls, all asynchronous on the caller's stream:
 *   mla_append_cache  write this step's c^{KV}, RoPE(k^R) into the paged pool
 *   mla_absorb_q      q_lat = [q^C W^{UK}_i ; RoPE(q^R)] per head
 *   mla_decode        paged latent attention (+ split-KV log-sum-exp combine)
 *   mla_unabsorb      o = W^{UV}_i o_lat per head
 *
 * Conventions for every call
 *   - All array pointers are DEVICE pointers, allocated and owned by the
 *     caller. Apart from the fixed scratch array of mla_decode_noalloc (see
 *     there) the library allocates no device memory and keeps no state
 *     between calls. `stream` is a cudaStream_t (NULL = legacy default stream).
 *   - Arrays are dense, row-major, with the shapes given below; element
 *     types follow cfg->act_dtype / cfg->cache_dtype.
 *   - Return value: MLA_OK (0) or a negative MLA_ERR_* code. Arguments are
 *     checked on the host before anything is launched; on an error nothing
 *     is launched. Faults only the device can see (a page id outside the
 *     pool, a sequence shorter than its query count, a bounded wait that
 *     ran out) are OR-ed as MLA_DEV_* bits into *dev_status (device int32,
 *     may be NULL), which the caller reads after synchronising. A flagged
 *     item is skipped, never accessed out of bounds.
 *   - Sequence b's cached length seq_lens[b] includes this step's n_q new
 *     tokens; query j of sequence b is at position seq_lens[b] - n_q + j and
 *     attends to positions 0 .. seq_lens[b] - n_q + j (causal mask,
 *     「一文通透DeepSeek-V2」 §2.1.1; two-token MTP decode masks the two new
 *     tokens against each other).
 *   - Token t of page-table row b at position p lives in page
 *     block_table[b * max_pages_per_seq + p / page_size], slot p % page_size.
 */
#ifndef MLA_B300_H
#define MLA_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- return codes ------------------------------------------------------ */
#define MLA_OK 0
#define MLA_ERR_INVALID_ARG -1   /* null pointer, negative size, inconsistent shape */
#define MLA_ERR_UNSUPPORTED -2   /* valid but not implemented (e.g. FP8 with fp32 act) */
#define MLA_ERR_WORKSPACE -3     /* workspace_bytes < mla_decode_workspace_size() */
#define MLA_ERR_ALIGNMENT -4     /* a pointer misses the 16-byte alignment a kernel needs */
#define MLA_ERR_CUDA -5          /* a CUDA runtime/driver call failed */
#define MLA_ERR_SCRATCH_LIMIT -6 /* mla_decode_noalloc: the sizes need more than its fixed scratch */

/* ---- device status bits (OR-ed into *dev_status) ----------------------- */
#define MLA_DEV_INDEX_OUT_OF_RANGE 1  /* page id / sequence id / position outside its table */
#define MLA_DEV_BAD_SEQLEN 2          /* seq_lens[b] < n_q or > max_seq_len */
#define MLA_DEV_TIMEOUT 4             /* a bounded barrier wait gave up; outputs invalid */

/* ---- element types ----------------------------------------------------- */
#define MLA_F32 0
#define MLA_BF16 1
#define MLA_FP8_E4M3 2   /* cache only */

/* ---- decode kernel choice ---------------------------------------------- */
#define MLA_KERNEL_AUTO 0   /* tensor-core kernel when the shape allows, else SIMT */
#define MLA_KERNEL_SIMT 1   /* generic CUDA-core kernel, any shape */
#define MLA_KERNEL_TC 2     /* tcgen05/TMEM kernel: n_heads=128, d_latent=512, d_rope=64,
                               page_size=64, bf16 act, bf16 or FP8 cache, n_q in {1,2}.
                               Operands are bf16 (an FP8 cache is dequantised as
                               code * scale in fp32, rounded once to bf16), accumulation
                               fp32. The softmax is exact for any spread of finite scores:
                               a unit whose scores jump beyond the kernel's running
                               reference by more than 2^96 is computed again with the
                               exact per-head maxima as the reference. Non-finite inputs
                               give non-finite outputs. */
#define MLA_KERNEL_TC_FP8_SCORES 3  /* the tensor-core kernel over an FP8 cache with the
                               scores on FP8 tensor cores (「Deepseek系列从v3到R易背面经版」
                               F8量化策略): in the kernel q_lat's latent part is quantised
                               per (query row, head) in 1x128 groups to E4M3 exactly as the
                               cache's latents are (scale = amax/448 in fp32), each group's
                               code product (tcgen05 kind::f8f6f4, fp32 accumulation) is
                               scaled by the two group scales and summed in fp32, and the
                               bf16 RoPE part is added. Softmax and P.V as MLA_KERNEL_TC.
                               FP8 cache, same shapes as MLA_KERNEL_TC; else
                               MLA_ERR_UNSUPPORTED. */
#define MLA_KERNEL_TC_FP8_STAGED 4  /* FP8 cache, same shapes as MLA_KERNEL_TC (else
                               MLA_ERR_UNSUPPORTED): one streaming kernel converts every
                               visible token of the batch once into a bf16 pool in the
                               workspace (code * group scale in fp32, rounded once to bf16,
                               the same operand values MLA_KERNEL_TC builds inside the
                               decode; RoPE keys copied), then the bf16 tensor-core decode
                               runs over that pool. Trades workspace for speed: the
                               workspace grows by batch * ceil(max_seq_len/64) * 64 * 1152
                               bytes (plus the staged block table), and each visible token
                               costs 1152 more bytes written and read back; in exchange no
                               token is converted more than once (MLA_KERNEL_TC converts it
                               once per query row) and the conversion runs on every SM.
                               mla_decode returns MLA_ERR_UNSUPPORTED for batch > 65535 or
                               batch * ceil(max_seq_len/64) * 64 >= 2^31 staged rows. */

typedef struct mla_config {
  int32_t n_heads;      /* H  = n_h                                               */
  int32_t d_head;       /* D  = d_h  (per-head q^C / k^C / v^C width)              */
  int32_t d_latent;     /* C  = d_c  (latent c^{KV} width)                         */
  int32_t d_rope;       /* R  = d_h^R (decoupled RoPE width, even)                 */
  int32_t page_size;    /* P  tokens per page of the latent pool                   */
  int32_t cache_dtype;  /* MLA_F32 | MLA_BF16 | MLA_FP8_E4M3                       */
  int32_t act_dtype;    /* MLA_F32 | MLA_BF16: q, weights, q_lat, o_lat storage    */
  int32_t kernel;       /* MLA_KERNEL_*                                           */
  float softmax_scale;  /* 0 -> 1/sqrt(d_head + d_rope)                            */
  float rope_base;      /* 0 -> 10000                                             */
  /* YaRN on the decoupled RoPE (「一文通透DeepSeek-V2」 §3.1.3, the 4K -> 128K extension).
   * rope_scaling = s <= 1 leaves plain RoPE. With s > 1, RoPE pair k (frequency
   * theta_k = base^(-2k/R), wavelength 2pi/theta_k) gets the frequency
   * (1 - g) theta_k / s + g theta_k, g = clip((r - alpha) / (beta - alpha), 0, 1),
   * r = rope_orig_context / wavelength, for q^R (mla_absorb_q) and k^R (mla_append_cache)
   * alike; and every logit of mla_decode is scaled by t = (mscale_coef ln s + 1)^2 on top of
   * softmax_scale. Zero fields take the page's values. */
  float rope_scaling;         /* s (0 or <= 1: off; the page uses 40)                  */
  int32_t rope_orig_context;  /* original context length (0 -> 4096)                   */
  float rope_yarn_alpha;      /* 0 -> 1                                                */
  float rope_yarn_beta;       /* 0 -> 32                                               */
  float rope_mscale_coef;     /* sqrt(t) = coef ln s + 1 (0 -> 0.0707)                 */
} mla_config;

/*
 * Bytes of one token's pool entry.
 *   MLA_F32 / MLA_BF16 cache: [c^{KV} (C) ; RoPE(k^R) (R)] elements of that type.
 *   MLA_FP8_E4M3 cache: C bytes of E4M3 codes, then 2R bytes of bf16 RoPE(k^R),
 *   then C/128 fp32 scales, one per 1x128 group (「Deepseek系列从v3到R易背面经版」
 *   F8量化策略: per-token 1x128 activation groups). 656 bytes at V2 sizes.
 * Returns 0 for an invalid config.
 */
size_t mla_cache_entry_bytes(const mla_config* cfg);

/*
 * mla_append_cache — cache write (「一文通透DeepSeek-V2」 §2.2.1 c^{KV}_t = W^{DKV} h_t is
 * cached; §2.2.2 k^R_t = RoPE(W^{KR} h_t) is cached). The projections themselves are
 * upstream: this call receives c^{KV} and the un-rotated k^R.
 *
 *   c_kv        [T][C]   latents (fp32 for an fp32 cache, else bf16)
 *   k_r         [T][R]   RoPE keys before rotation (same type as c_kv)
 *   seq_idx     [T]      int32 page-table row of each token, 0 <= seq_idx < batch
 *   pos         [T]      int32 position of each token in its sequence
 *   block_table [batch][max_pages_per_seq] int32 page ids
 *   kv_pool     [num_pages][page_size] entries of mla_cache_entry_bytes()
 * For each token: k^R is rotated by its position (interleaved pairs, angle
 * pos * base^(-2k/R), computed in fp64), then [c ; RoPE(k^R)] is written to its
 * slot; an FP8 cache stores c as E4M3 codes with scale = amax/448 per 128-group
 * (IEEE fp32 division, round-to-nearest-even, saturating). A token whose row,
 * position or page id is out of range is skipped and flagged.
 */
int mla_append_cache(const mla_config* cfg, const void* c_kv, const void* k_r,
                     const int32_t* seq_idx, const int32_t* pos, int32_t num_tokens,
                     const int32_t* block_table, int32_t batch, int32_t max_pages_per_seq,
                     int32_t num_pages, void* kv_pool, int32_t* dev_status, void* stream);

/*
 * mla_absorb_q — query-side absorption (「一文通透DeepSeek-V2」 §2.2.1: W^{UK} is absorbed
 * into the query; 「Deepseek系列从v3到R易背面经版」 MLA: (W^{UQ})^T W^{UK} fused).
 *
 *   q_c   [T][H][D]  q^C;   q_r [T][H][R] q^R before rotation;   pos [T] int32
 *   w_uk  [H][D][C]  head i's rows of W^{UK} in R^{(H D) x C}
 *   q_lat [T][H][C+R] out:  q_lat[t][i][0:C] = sum_d q_c[t][i][d] w_uk[i][d][:]  (fp32 accum.)
 *                           q_lat[t][i][C: ] = RoPE_pos[t](q_r[t][i])
 * All in cfg->act_dtype. Decode orders tokens as t = b * n_q + j.
 */
int mla_absorb_q(const mla_config* cfg, const void* q_c, const void* q_r, const int32_t* pos,
                 int32_t num_tokens, const void* w_uk, void* q_lat, void* stream);

/*
 * mla_append_absorb — the two inputs of a decode step in one call: mla_append_cache of the
 * step's new tokens, then mla_absorb_q of its queries, with the same pos [T] for both (each
 * token's position). Arguments, layouts and results exactly as those two calls; every
 * argument of both is checked before anything is launched, and MLA_OK means both were
 * queued. The absorption reads none of what the append writes, so the tensor-core absorption
 * reads its own inputs without waiting for the append to finish, and the two overlap on the
 * device. A kernel queued after this call still finds both the cache entries and q_lat
 * complete. The buffers of the two halves must not overlap.
 */
int mla_append_absorb(const mla_config* cfg, const void* c_kv, const void* k_r,
                      const int32_t* seq_idx, const int32_t* pos, int32_t num_tokens,
                      const int32_t* block_table, int32_t batch, int32_t max_pages_per_seq,
                      int32_t num_pages, void* kv_pool, int32_t* dev_status, const void* q_c,
                      const void* q_r, const void* w_uk, void* q_lat, void* stream);

/*
 * Workspace bytes mla_decode needs for these sizes: the fp32 split partials (one [C] output
 * and one log-sum-exp per query row, head and split) when the rows are split over several
 * ranges (num_splits, or the automatic choice, above 1). The tensor-core kernels also keep
 * there, with more query rows than CTA pairs, the order in which the pairs take the rows
 * (longest first), and with the automatic choice the two partials of each row in a last,
 * partly filled round of pairs that it splits in two. 0 when none of this applies. With
 * MLA_KERNEL_TC_FP8_STAGED also the staged bf16 pool and its block table, which come first.
 * num_splits as for mla_decode; max_seq_len bounds every seq_lens[b].
 */
size_t mla_decode_workspace_size(const mla_config* cfg, int32_t batch, int32_t n_q,
                                 int32_t max_seq_len, int32_t num_splits);

/*
 * Which decode kernel mla_decode would launch for these sizes: one of the MLA_KERNEL_*
 * values other than MLA_KERNEL_AUTO, or a negative MLA_ERR_* code.
 */
int mla_decode_kernel(const mla_config* cfg, int32_t batch, int32_t n_q);

/*
 * mla_decode — paged latent attention, absorbed form (「deepseek(2)——deepseek 關鍵技術」
 * §1 o_{t,i} = sum_j softmax_j(q_{t,i}^T k_{j,i} / sqrt(d_h + d_h^R)) v^C_{j,i}, with W^{UK},
 * W^{UV} moved to the query / output side):
 *   s_n  = (q_lat[b][j][i] . [c_n ; k^R_n]) * scale   for n <= seq_lens[b] - n_q + j
 *   o_lat[b][j][i] = sum_n softmax(s)_n c_n,   lse[b][j][i] = ln sum_n e^{s_n}
 *
 *   q_lat       [batch][n_q][H][C+R]   act dtype
 *   kv_pool     as written by mla_append_cache
 *   block_table [batch][max_pages_per_seq] int32;  seq_lens [batch] int32 (device)
 *   max_seq_len host-side bound on seq_lens (sizes the split-KV schedule)
 *   num_splits  0 = automatic; otherwise the SIMT kernel splits each sequence's
 *               tokens into num_splits ranges and the tensor-core kernel
 *               spreads the batch's pages over num_splits CTA pairs per query
 *               row; partial results are merged with log-sum-exp weights.
 *   workspace   device scratch of >= mla_decode_workspace_size() bytes (may be
 *               NULL when that size is 0); contents need no initialisation.
 *   o_lat       [batch][n_q][H][C] act dtype;   lse [batch][n_q][H] fp32 or NULL
 * The result for a fixed num_splits is deterministic (no floating-point atomics). With
 * num_splits = 0 the split schedule follows the device's SM count, so results are repeatable
 * on one kind of GPU and may differ by rounding between GPUs with different SM counts.
 */
int mla_decode(const mla_config* cfg, const void* q_lat, const void* kv_pool,
               const int32_t* block_table, int32_t max_pages_per_seq, int32_t num_pages,
               const int32_t* seq_lens, int32_t batch, int32_t n_q, int32_t max_seq_len,
               int32_t num_splits, void* workspace, size_t workspace_bytes, void* o_lat,
               float* lse, int32_t* dev_status, void* stream);

/*
 * mla_unabsorb — output-side absorption (「一文通透DeepSeek-V2」 §2.2.1: W^{UV} is absorbed
 * into W^O):  o[t][i][r] = sum_k w_uv[i][r][k] * o_lat[t][i][k]   (fp32 accumulation)
 *   o_lat [T][H][C] act dtype;  w_uv [H][D][C] act dtype;  o [T][H][D] fp32.
 */
int mla_unabsorb(const mla_config* cfg, const void* o_lat, int32_t num_tokens, const void* w_uv,
                 float* o, void* stream);

/*
 * mla_project_append — the fused upstream append: this step's hidden states to their cache
 * entries in one call (「一文通透DeepSeek-V2」 §2.2.1 c^{KV}_t = W^{DKV} h_t, §3.1.4 the extra
 * RMSNorm after the compressed latent, §2.2.2 k^R_t = RoPE(W^{KR} h_t)).
 *
 *   h          [T][d_model] bf16 hidden states (d_model a multiple of 8, 16-byte aligned)
 *   w_dkv_kr   [C + R][d_model] bf16: rows 0..C-1 hold W^{DKV}, rows C..C+R-1 hold W^{KR}
 *   gain       [C] fp32 gain of the latent's RMSNorm (it also carries the bottleneck's scaling)
 *   eps        RMSNorm epsilon (> 0)
 *   seq_idx, pos, block_table, batch, max_pages_per_seq, num_pages, kv_pool: as
 *              mla_append_cache (bf16 or FP8 cache)
 *   workspace  >= mla_project_append_workspace_size() bytes of device scratch
 * x = W^{DKV} h and k^R = W^{KR} h are formed on the tensor cores with fp32 accumulation;
 * c^{KV} = gain * x / sqrt(mean(x^2) + eps) in fp32; both are rounded to bf16 (the type a
 * separate projection would store) and then cached exactly as mla_append_cache caches them
 * (RoPE of k^R at the token's position, optional E4M3 groups). Errors as mla_append_cache;
 * MLA_ERR_UNSUPPORTED for an fp32 cache or activations.
 */
size_t mla_project_append_workspace_size(const mla_config* cfg, int32_t d_model, int32_t num_tokens);
int mla_project_append(const mla_config* cfg, const void* h, int32_t d_model, int32_t num_tokens,
                       const void* w_dkv_kr, const float* gain, float eps, const int32_t* seq_idx,
                       const int32_t* pos, const int32_t* block_table, int32_t batch,
                       int32_t max_pages_per_seq, int32_t num_pages, void* kv_pool,
                       void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream);

/*
 * mla_output_projection — u_t = W^O [o_{t,1}; ...; o_{t,n_h}] (「一文通透DeepSeek-V2」 §2.1.2,
 * W^O in R^{d x d_h n_h}; 「deepseek(2)——deepseek 關鍵技術」 §1).
 *   o     [T][H * D] bf16: the heads' outputs, concatenated in head order
 *   w_o   [d_model][H * D] bf16 (H * D and d_model multiples of 8; 16-byte aligned)
 *   u     [T][d_model] fp32
 *   workspace >= mla_output_projection_workspace_size() bytes (fp32 split partials; may be 0)
 * fp32 accumulation on the tensor cores; partial sums over K ranges are added in a fixed order,
 * so the result does not depend on scheduling.
 */
size_t mla_output_projection_workspace_size(const mla_config* cfg, int32_t d_model, int32_t num_tokens);
int mla_output_projection(const mla_config* cfg, const void* o, int32_t num_tokens, const void* w_o,
                          int32_t d_model, float* u, void* workspace, size_t workspace_bytes,
                          int32_t* dev_status, void* stream);

/*
 * mla_prefill — the non-absorbed path over a prompt (「一文通透DeepSeek-V2」 §2.2.1: the naive
 * formula restores k^C_{n,i} = W^{UK}_i c^{KV}_n and v^C_{n,i} = W^{UV}_i c^{KV}_n;
 * 「deepseek(2)——deepseek 關鍵技術」 §1 for q, k and o), causal over positions 0 .. L-1:
 *   o[t][i] = sum_{n <= t} softmax_n([q^C_{t,i}; RoPE_t(q^R_{t,i})] . [k^C_{n,i}; k^R_n] * scale) v^C_{n,i}
 *   c_kv   [L][C] bf16   the prompt's latents as cached
 *   k_r    [L][R] bf16   the prompt's RoPE keys, already rotated (as cached)
 *   q_c    [L][H][D], q_r [L][H][R] bf16 (q^R before rotation)
 *   w_uk, w_uv [H][D][C] bf16;  o [L][H][D] fp32
 *   workspace >= mla_prefill_workspace_size() bytes (K^C, V^C and the assembled queries)
 * Tensor-core path for d_head = 128, d_rope = 64, bf16 activations (MLA_ERR_UNSUPPORTED
 * otherwise); RoPE and the softmax scale follow cfg (YaRN included).
 */
size_t mla_prefill_workspace_size(const mla_config* cfg, int32_t prompt_len);
int mla_prefill(const mla_config* cfg, const void* c_kv, const void* k_r, int32_t prompt_len,
                const void* q_c, const void* q_r, const void* w_uk, const void* w_uv, float* o,
                void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream);

/*
 * mla_decode_noalloc — mla_decode for callers that cannot allocate device memory. The pages
 * have no counterpart to this call; it is a convenience of this library.
 *
 * Who needs it: hosts that give the library only the tensors they own and no way to get more
 * device memory (a serving framework's plugin interface whose memory pool is managed
 * elsewhere), processes that must not have a library call cudaMalloc in the middle of a decode
 * loop (it may block on the device or fail under memory pressure), and callers from runtimes
 * that have no CUDA allocator binding.
 *
 * Arguments and results are those of mla_decode, without workspace / workspace_bytes: the
 * scratch is a fixed MLA_NOALLOC_SCRATCH_BYTES array in the library's device image, which every
 * GPU that loads the library holds until the process exits. The call allocates nothing.
 *   - If mla_decode_workspace_size() for these sizes exceeds MLA_NOALLOC_SCRATCH_BYTES the call
 *     returns MLA_ERR_SCRATCH_LIMIT and launches nothing.
 *   - The first call on a device looks up the scratch's device address on that device (with
 *     it current); make that first call before any stream capture. The lookup is repeated
 *     when the device's context has changed since (after cudaDeviceReset).
 *   - Every call on a device shares the one array and leaves its contents behind. Nothing in it
 *     needs to start at zero (each call writes what it later reads), but calls whose work
 *     overlaps on the GPU (different streams, or different host threads) race on it: keep them
 *     ordered, for example on one stream.
 */
#define MLA_NOALLOC_SCRATCH_BYTES (32u << 20)
int mla_decode_noalloc(const mla_config* cfg, const void* q_lat, const void* kv_pool,
                       const int32_t* block_table, int32_t max_pages_per_seq, int32_t num_pages,
                       const int32_t* seq_lens, int32_t batch, int32_t n_q, int32_t max_seq_len,
                       int32_t num_splits, void* o_lat, float* lse, int32_t* dev_status,
                       void* stream);

/*
 * mla_debug_decode_fault — test hook for the device-side failure path (no counterpart on the
 * pages). wait_cycles > 0 sets the limit, in SM clock cycles, after which every bounded wait of
 * the tensor-core decode gives up (0 restores the default, about 2 s); withhold_chunk >= 0
 * makes the bf16 kernel's latent producer in the even CTA of every pair register that latent
 * chunk's bytes (chunks count 32-token, 256-column loads from the start of a pair's range)
 * without issuing its loads, so the P.V issuer's wait for it runs out with nothing in flight:
 * the decode then sets MLA_DEV_TIMEOUT, abandons its outputs and returns. -1 turns it off.
 * Process-wide; affects launches made after the call. Returns MLA_OK or MLA_ERR_INVALID_ARG.
 */
int mla_debug_decode_fault(long long wait_cycles, int32_t withhold_chunk);

/* Human-readable text of a return code (static storage). */
const char* mla_status_string(int code);

#ifdef __cplusplus
}
#endif
#endif /* MLA_B300_H */
