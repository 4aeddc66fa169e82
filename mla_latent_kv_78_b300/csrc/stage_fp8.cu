// FP8 cache staged to bf16 for the tensor-core decode (MLA_KERNEL_TC_FP8_STAGED).
//
// The FP8 cache's latents are E4M3 codes with one fp32 scale per 1x128 group
// (「Deepseek系列从v3到R易背面经版」 F8量化策略); the tensor-core decode takes them as bf16
// operands, code * scale in fp32 rounded once to bf16. The fused FP8 kernel does that
// conversion inside the decode, once per query row that reads a token (twice per token for
// two-token decode), on the few warps that sit between the loads and the MMAs, and it is
// bound by them. This path converts every visible token once, in a streaming pass over all
// SMs, into a bf16 pool in the workspace (the same conversion, the bf16 RoPE keys copied), and
// then runs the bf16 decode over that pool through an identity block table: row b's page p
// is staged page b * ppr + p, ppr = ceil(max_seq_len / 64). The decode sees the operand values
// the fused kernel builds, so it computes the same reading of the method.
//
// Costs: workspace of B * ppr * 64 * 1152 bytes (the batch's visible cache in bf16) and,
// per visible token, 656 bytes read plus 1152 bytes written before the decode reads them back.
#include "mla_internal.cuh"
#include "tc_ptx.cuh"

namespace mla {
namespace stg {

constexpr int kP = 64;                 // tokens per page
constexpr int kIn = 656 / 16;          // 16-byte words of an FP8 entry: 32 codes, 8 RoPE, 1 scales
constexpr int kOut = 1152 / 16;        // 16-byte words of a bf16 entry: 64 latent, 8 RoPE
constexpr int kWords = kP * kIn;       // input words of a page
constexpr int kThreads = 256;
constexpr int kPer = (kWords + kThreads - 1) / kThreads;   // words per thread (11)

__global__ void __launch_bounds__(kThreads)
    stage_fp8_kernel(const uint4* __restrict__ pool, const int32_t* __restrict__ bt, int maxp,
                     int num_pages, const int32_t* __restrict__ seq_lens, int n_q, int max_seq_len,
                     int ppr, uint4* __restrict__ spool, int32_t* __restrict__ sbt,
                     int32_t* status) {
  const int p = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  // launched programmatically: nothing is read before the preceding kernel has completed
  ptx::griddep_wait();
  const size_t sp = (size_t)b * ppr + p;
  if (tid == 0) sbt[sp] = (int32_t)sp;
  const int L = __ldg(seq_lens + b);
  // a row the decode rejects (and flags) reads nothing; pages past the row are never read
  if (L < n_q || L > max_seq_len || p * kP >= L) return;
  const int pg = __ldg(bt + (size_t)b * maxp + p);
  const bool bad = pg < 0 || pg >= num_pages;
  if (bad && tid == 0) flag_status(status, MLA_DEV_INDEX_OUT_OF_RANGE);
  const int ntok = min(kP, L - p * kP);   // live slots; the rest are written as zeros
  const uint4* src = pool + (size_t)(bad ? 0 : pg) * kWords;
  uint4* dst = spool + sp * (size_t)(kP * kOut);

  // all of this thread's loads first (11 words in flight), then convert and store
  uint4 w[kPer];
  float sc[kPer];
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int i = tid + u * kThreads;
    const int tok = i / kIn, k = i - tok * kIn;
    w[u] = make_uint4(0, 0, 0, 0);
    sc[u] = 0.f;
    if (i < kWords && !bad && tok < ntok && k < kIn - 1) {
      w[u] = __ldg(src + i);
      if (k < 32) sc[u] = __ldg(reinterpret_cast<const float*>(src + tok * kIn + kIn - 1) + (k >> 3));
    }
  }
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int i = tid + u * kThreads;
    const int tok = i / kIn, k = i - tok * kIn;
    if (i >= kWords || k == kIn - 1) continue;
    uint4* out = dst + tok * kOut;
    if (k < 32) {
      // 16 codes of group k / 8 -> 16 bf16 (two words)
      const uint4 c = w[u];
      const float s = sc[u];
      out[2 * k] = make_uint4(ptx::e4m3x2_scaled_bf16x2(c.x, s), ptx::e4m3x2_scaled_bf16x2(c.x >> 16, s),
                              ptx::e4m3x2_scaled_bf16x2(c.y, s), ptx::e4m3x2_scaled_bf16x2(c.y >> 16, s));
      out[2 * k + 1] = make_uint4(ptx::e4m3x2_scaled_bf16x2(c.z, s), ptx::e4m3x2_scaled_bf16x2(c.z >> 16, s),
                                  ptx::e4m3x2_scaled_bf16x2(c.w, s), ptx::e4m3x2_scaled_bf16x2(c.w >> 16, s));
    } else {
      out[64 + (k - 32)] = w[u];   // bf16 RoPE keys as stored
    }
  }
}

}  // namespace stg

size_t fp8_staged_bytes(int B, int max_seq_len) {
  const size_t ppr = ((size_t)max_seq_len + stg::kP - 1) / stg::kP;
  const size_t pool = (size_t)B * ppr * stg::kP * 1152;
  const size_t table = ((size_t)B * ppr * sizeof(int32_t) + 255) / 256 * 256;
  return pool + table;
}

cudaError_t launch_decode_tc_fp8_staged(const Dims& d, const void* q_lat, const void* pool,
                                        const int32_t* bt, int maxp, int num_pages,
                                        const int32_t* seq_lens, int B, int n_q, int max_seq_len,
                                        int num_splits, void* ws, size_t ws_bytes, void* o_lat,
                                        float* lse, int32_t* status, cudaStream_t stream) {
  if (d.entry_bytes != stg::kIn * 16 || d.P != stg::kP || d.C != 512 || d.R != 64)
    return cudaErrorInvalidValue;
  const int ppr = (max_seq_len + stg::kP - 1) / stg::kP;
  if (B > 65535 || (size_t)B * ppr > (size_t)0x7fffffff / stg::kP) return cudaErrorInvalidValue;
  const size_t staged = fp8_staged_bytes(B, max_seq_len);
  if (ws_bytes < staged) return cudaErrorInvalidValue;
  uint8_t* base = static_cast<uint8_t*>(ws);
  uint4* spool = reinterpret_cast<uint4*>(base);
  int32_t* sbt = reinterpret_cast<int32_t*>(base + (size_t)B * ppr * stg::kP * 1152);
  cudaError_t e = launch_programmatic(stg::stage_fp8_kernel, dim3(ppr, B), dim3(stg::kThreads), 0,
                                      stream, static_cast<const uint4*>(pool), bt, maxp, num_pages,
                                      seq_lens, n_q, max_seq_len, ppr, spool, sbt, status);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  Dims db = d;
  db.cache_dtype = MLA_BF16;
  db.entry_bytes = 1152;
  db.fp8_scores = false;
  return launch_decode_tc(db, q_lat, spool, sbt, ppr, B * ppr, seq_lens, B, n_q, max_seq_len,
                          num_splits, base + staged, ws_bytes - staged, o_lat, lse, status, stream);
}

}  // namespace mla
