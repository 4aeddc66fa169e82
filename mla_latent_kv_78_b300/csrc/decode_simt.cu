// Generic CUDA-core MLA decode over the paged latent cache (any head shape, any
// cache type), plus the log-sum-exp combine of split-KV partials.
//
// Absorbed form (「一文通透DeepSeek-V2」 §2.2.1-2.2.2; 「deepseek(2)——deepseek 關鍵技術」 §1):
//   s_n = q_lat . [c_n ; k^R_n] * scale,  o_lat = sum_n softmax(s)_n c_n,  lse = ln sum e^{s}
// for n <= seq_len - n_q + j (causal, 「一文通透DeepSeek-V2」 §2.1.1).
//
// One CTA per (head, query row, sequence, split); each warp walks every 4th
// token with its own online softmax (scores in log2 units), and the four
// warps merge at the end. This kernel re-reads the cache once per head, so
// it is the reference-quality path for small or unusual shapes; the V2 shapes
// run on the tensor-core kernel.
#include <math_constants.h>

#include "mla_internal.cuh"

namespace mla {

constexpr int kMaxC = 512;                 // latent width bound of this kernel
constexpr int kMaxU = kMaxC / 32;          // latent elements per lane
constexpr int kWarps = 4;

template <int CACHE>
struct KvRow {
  const uint8_t* row;
  int C, R;
  __device__ __forceinline__ float get(int k) const {
    if constexpr (CACHE == MLA_F32) {
      return reinterpret_cast<const float*>(row)[k];
    } else if constexpr (CACHE == MLA_BF16) {
      return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(row)[k]);
    } else {
      if (k < C) {
        const float s = reinterpret_cast<const float*>(row + C + 2 * R)[k / kFp8Group];
        return e4m3_decode(row[k]) * s;
      }
      return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(row + C)[k - C]);
    }
  }
};

template <typename Act, int CACHE>
__global__ void __launch_bounds__(kWarps * 32) decode_simt_kernel(
    Dims d, const Act* __restrict__ q_lat, const uint8_t* __restrict__ pool,
    const int32_t* __restrict__ bt, int maxp, int num_pages, const int32_t* __restrict__ seq_lens,
    int B, int n_q, int max_seq_len, int S, float* __restrict__ ws_o, float* __restrict__ ws_lse,
    Act* __restrict__ o_lat, float* __restrict__ lse_out, int32_t* status) {
  extern __shared__ float sm[];
  float* q = sm;                                    // [C + R], pre-scaled to log2 units
  float* red_o = sm + d.C + d.R;                    // [kWarps][C]
  float* red_ml = red_o + kWarps * d.C;             // [kWarps][2]

  const int i = blockIdx.x, j = blockIdx.y;
  const int b = blockIdx.z / S, split = blockIdx.z % S;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int CR = d.C + d.R;
  const size_t row_id = ((size_t)b * n_q + j) * d.H + i;   // (b, j, i)

  const int L = seq_lens[b];
  const bool bad_len = (L < n_q || L > max_seq_len);
  if (bad_len && threadIdx.x == 0) flag_status(status, MLA_DEV_BAD_SEQLEN);
  const int visible = bad_len ? 0 : L - n_q + j + 1;
  const int chunk = (visible + S - 1) / S;
  const int lo = min(visible, split * chunk);
  const int hi = min(visible, lo + chunk);

  const float qs = d.scale * 1.4426950408889634f;   // scale * log2(e)
  for (int k = threadIdx.x; k < CR; k += blockDim.x) q[k] = ld_act(q_lat, row_id * CR + k) * qs;
  __syncthreads();

  float m = -CUDART_INF_F, l = 0.f;
  float acc[kMaxU];
#pragma unroll
  for (int u = 0; u < kMaxU; ++u) acc[u] = 0.f;

  for (int n = lo + warp; n < hi; n += kWarps) {
    const int page = bt[(size_t)b * maxp + n / d.P];
    if (page < 0 || page >= num_pages) {
      if (lane == 0) flag_status(status, MLA_DEV_INDEX_OUT_OF_RANGE);
      continue;
    }
    KvRow<CACHE> kv{pool + ((size_t)page * d.P + n % d.P) * (size_t)d.entry_bytes, d.C, d.R};
    float part = 0.f;
    for (int k = lane; k < CR; k += 32) part = fmaf(q[k], kv.get(k), part);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
    const float m_new = fmaxf(m, part);
    const float corr = exp2f(m - m_new);
    const float p = exp2f(part - m_new);
    l = l * corr + p;
#pragma unroll
    for (int u = 0; u < kMaxU; ++u) {
      const int k = lane + 32 * u;
      if (k < d.C) acc[u] = fmaf(p, kv.get(k), acc[u] * corr);
    }
    m = m_new;
  }

  // merge the warps
#pragma unroll
  for (int u = 0; u < kMaxU; ++u) {
    const int k = lane + 32 * u;
    if (k < d.C) red_o[warp * d.C + k] = acc[u];
  }
  if (lane == 0) {
    red_ml[warp * 2] = m;
    red_ml[warp * 2 + 1] = l;
  }
  __syncthreads();
  float M = -CUDART_INF_F;
  for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red_ml[w * 2]);
  float Lsum = 0.f;
  float wgt[kWarps];
  for (int w = 0; w < kWarps; ++w) {
    wgt[w] = red_ml[w * 2] == -CUDART_INF_F ? 0.f : exp2f(red_ml[w * 2] - M);
    Lsum += red_ml[w * 2 + 1] * wgt[w];
  }
  const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
  const float lse = Lsum > 0.f ? (M + log2f(Lsum)) * 0.6931471805599453f : -CUDART_INF_F;
  for (int k = threadIdx.x; k < d.C; k += blockDim.x) {
    float v = 0.f;
    for (int w = 0; w < kWarps; ++w) v = fmaf(red_o[w * d.C + k], wgt[w], v);
    v *= inv;
    if (S == 1)
      st_act(o_lat, row_id * d.C + k, v);
    else
      ws_o[(row_id * S + split) * d.C + k] = v;
  }
  if (threadIdx.x == 0) {
    if (S == 1) {
      if (lse_out) lse_out[row_id] = lse;
    } else {
      ws_lse[row_id * S + split] = lse;
    }
  }
}

// One CTA per (b, j, i) row: o = sum_s w_s o_s / sum_s w_s, w_s = e^{lse_s - max lse}.
template <typename Act>
__global__ void __launch_bounds__(128) combine_kernel(int C, int S, const float* __restrict__ ws_o,
                                                      const float* __restrict__ ws_lse,
                                                      Act* __restrict__ o_lat,
                                                      float* __restrict__ lse_out,
                                                      const int32_t* __restrict__ row_of, int H) {
  const size_t r = blockIdx.x;
  // output row: r itself, or (partials of some query rows only) head r % H of query row
  // row_of[r / H]
  const size_t out = row_of ? (size_t)__ldg(row_of + r / H) * H + r % H : r;
  float M = -CUDART_INF_F;
  for (int s = 0; s < S; ++s) M = fmaxf(M, ws_lse[r * S + s]);
  float z = 0.f;
  for (int s = 0; s < S; ++s) {
    const float ls = ws_lse[r * S + s];
    z += ls == -CUDART_INF_F ? 0.f : __expf(ls - M);
  }
  const float inv = z > 0.f ? 1.f / z : 0.f;
  for (int k = threadIdx.x; k < C; k += blockDim.x) {
    float v = 0.f;
    for (int s = 0; s < S; ++s) {
      const float ls = ws_lse[r * S + s];
      if (ls != -CUDART_INF_F) v = fmaf(__expf(ls - M), ws_o[(r * S + s) * C + k], v);
    }
    st_act(o_lat, out * C + k, v * inv);
  }
  if (threadIdx.x == 0 && lse_out) lse_out[out] = z > 0.f ? M + logf(z) : -CUDART_INF_F;
}

size_t simt_workspace_bytes(const Dims& d, int B, int n_q, int S) {
  if (S <= 1) return 0;
  const size_t rows = (size_t)B * n_q * d.H;
  return rows * S * ((size_t)d.C + 1) * sizeof(float);
}

int simt_pick_splits(const Dims& d, int B, int n_q, int max_seq_len, int num_splits, int num_sms) {
  if (num_splits > 0) return num_splits;
  const long ctas = (long)B * n_q * d.H;
  int S = 1;
  // keep at least ~4 CTAs per SM in flight and at least 256 tokens per split
  while (ctas * S < 4L * num_sms && (long)max_seq_len / (S * 2) >= 256 && S < 64) S *= 2;
  return S;
}

template <typename Act, int CACHE>
static cudaError_t launch_t(const Dims& d, const void* q_lat, const void* pool, const int32_t* bt,
                            int maxp, int num_pages, const int32_t* seq_lens, int B, int n_q,
                            int max_seq_len, int S, void* ws, void* o_lat, float* lse,
                            int32_t* status, cudaStream_t stream) {
  dim3 grid(d.H, n_q, B * S);
  const size_t smem = sizeof(float) * ((size_t)d.C + d.R + (size_t)kWarps * d.C + 2 * kWarps);
  auto kern = decode_simt_kernel<Act, CACHE>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  float* ws_o = static_cast<float*>(ws);
  const size_t rows = (size_t)B * n_q * d.H;
  float* ws_lse = S > 1 ? ws_o + rows * S * d.C : nullptr;
  kern<<<grid, kWarps * 32, smem, stream>>>(d, (const Act*)q_lat, (const uint8_t*)pool, bt, maxp,
                                            num_pages, seq_lens, B, n_q, max_seq_len, S, ws_o,
                                            ws_lse, (Act*)o_lat, lse, status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || S == 1) return e;
  combine_kernel<Act><<<(unsigned)rows, 128, 0, stream>>>(d.C, S, ws_o, ws_lse, (Act*)o_lat, lse,
                                                           nullptr, 1);
  return cudaGetLastError();
}

cudaError_t launch_combine(int C, int S, const float* ws_o, const float* ws_lse, void* o_lat,
                           int act_dtype, float* lse, size_t rows, cudaStream_t stream,
                           const int32_t* row_of, int H) {
  if (act_dtype == MLA_F32)
    combine_kernel<float><<<(unsigned)rows, 128, 0, stream>>>(C, S, ws_o, ws_lse, (float*)o_lat, lse,
                                                              row_of, H);
  else
    combine_kernel<__nv_bfloat16><<<(unsigned)rows, 128, 0, stream>>>(C, S, ws_o, ws_lse,
                                                                      (__nv_bfloat16*)o_lat, lse,
                                                                      row_of, H);
  return cudaGetLastError();
}

cudaError_t launch_decode_simt(const Dims& d, const void* q_lat, const void* pool,
                               const int32_t* bt, int maxp, int num_pages, const int32_t* seq_lens,
                               int B, int n_q, int max_seq_len, int S, void* ws, void* o_lat,
                               float* lse, int32_t* status, cudaStream_t stream) {
  if (d.act_dtype == MLA_F32) {
    if (d.cache_dtype == MLA_F32)
      return launch_t<float, MLA_F32>(d, q_lat, pool, bt, maxp, num_pages, seq_lens, B, n_q,
                                      max_seq_len, S, ws, o_lat, lse, status, stream);
    if (d.cache_dtype == MLA_BF16)
      return launch_t<float, MLA_BF16>(d, q_lat, pool, bt, maxp, num_pages, seq_lens, B, n_q,
                                       max_seq_len, S, ws, o_lat, lse, status, stream);
    return cudaErrorInvalidValue;
  }
  if (d.cache_dtype == MLA_F32)
    return launch_t<__nv_bfloat16, MLA_F32>(d, q_lat, pool, bt, maxp, num_pages, seq_lens, B, n_q,
                                            max_seq_len, S, ws, o_lat, lse, status, stream);
  if (d.cache_dtype == MLA_BF16)
    return launch_t<__nv_bfloat16, MLA_BF16>(d, q_lat, pool, bt, maxp, num_pages, seq_lens, B, n_q,
                                             max_seq_len, S, ws, o_lat, lse, status, stream);
  return launch_t<__nv_bfloat16, MLA_FP8_E4M3>(d, q_lat, pool, bt, maxp, num_pages, seq_lens, B,
                                               n_q, max_seq_len, S, ws, o_lat, lse, status, stream);
}

}  // namespace mla
