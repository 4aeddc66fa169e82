// K1: latent-cache write with decoupled RoPE on k^R (and optional E4M3 quantisation).
//
// 「一文通透DeepSeek-V2」 §2.2.1: only c^{KV}_t is cached; §2.2.2: k^R_t = RoPE(W^{KR} h_t)
// is cached beside it. 「Deepseek系列从v3到R易背面经版」 F8量化策略: activations are
// quantised per token in 1x128 groups, E4M3.
//
// One warp per token. The page/slot mapping is integer-exact; RoPE runs in fp64
// and is rounded once to the cache type; the FP8 scale and the per-element
// division are IEEE fp32 (__fdiv_rn), so the integer codes match a CPU encoder
// that takes the same fp32 decisions.
#include "mla_internal.cuh"

namespace mla {

template <typename In, int CACHE>
__global__ void __launch_bounds__(128) append_kernel(Dims d, const In* __restrict__ c_kv,
                                                     const In* __restrict__ k_r,
                                                     const int32_t* __restrict__ seq_idx,
                                                     const int32_t* __restrict__ pos, int T,
                                                     const int32_t* __restrict__ bt, int batch,
                                                     int maxp, int num_pages,
                                                     uint8_t* __restrict__ pool,
                                                     int32_t* status) {
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const int b = seq_idx[t];
  const int p = pos[t];
  if (b < 0 || b >= batch || p < 0 || p / d.P >= maxp) {
    if (lane == 0) flag_status(status, MLA_DEV_INDEX_OUT_OF_RANGE);
    return;
  }
  const int page = bt[(size_t)b * maxp + p / d.P];
  if (page < 0 || page >= num_pages) {
    if (lane == 0) flag_status(status, MLA_DEV_INDEX_OUT_OF_RANGE);
    return;
  }
  uint8_t* dst = pool + ((size_t)page * d.P + (p % d.P)) * (size_t)d.entry_bytes;
  const In* src_c = c_kv + (size_t)t * d.C;
  const In* src_r = k_r + (size_t)t * d.R;
  const double base = (double)d.rope_base;

  if constexpr (CACHE != MLA_FP8_E4M3) {
    In* out = reinterpret_cast<In*>(dst);
    for (int k = lane; k < d.C; k += 32) out[k] = src_c[k];
    for (int k = lane; k < d.R / 2; k += 32) {
      double cs, sn;
      rope_cos_sin(p, k, d.R, base, &cs, &sn);
      const double x0 = (double)ld_act(src_r, 2 * k), x1 = (double)ld_act(src_r, 2 * k + 1);
      st_act(out, d.C + 2 * k, (float)(x0 * cs - x1 * sn));
      st_act(out, d.C + 2 * k + 1, (float)(x0 * sn + x1 * cs));
    }
  } else {
    uint8_t* codes = dst;
    __nv_bfloat16* kr = reinterpret_cast<__nv_bfloat16*>(dst + d.C);
    float* scales = reinterpret_cast<float*>(dst + d.C + 2 * d.R);
    // each lane owns 4 consecutive elements of every 128-group
    for (int g = 0; g < d.C / kFp8Group; ++g) {
      float x[4];
      float amax = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        x[e] = ld_act(src_c, g * kFp8Group + lane * 4 + e);
        amax = fmaxf(amax, fabsf(x[e]));
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
      const float s = amax > 0.f ? __fdiv_rn(amax, kE4M3Max) : 1.0f;
      uint32_t packed = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) packed |= (uint32_t)e4m3_encode(__fdiv_rn(x[e], s)) << (8 * e);
      reinterpret_cast<uint32_t*>(codes + g * kFp8Group)[lane] = packed;
      if (lane == 0) scales[g] = s;
    }
    for (int k = lane; k < d.R / 2; k += 32) {
      double cs, sn;
      rope_cos_sin(p, k, d.R, base, &cs, &sn);
      const double x0 = (double)ld_act(src_r, 2 * k), x1 = (double)ld_act(src_r, 2 * k + 1);
      kr[2 * k] = __float2bfloat16_rn((float)(x0 * cs - x1 * sn));
      kr[2 * k + 1] = __float2bfloat16_rn((float)(x0 * sn + x1 * cs));
    }
  }
}

cudaError_t launch_append(const Dims& d, const void* c_kv, const void* k_r, const int32_t* seq_idx,
                          const int32_t* pos, int T, const int32_t* bt, int batch, int maxp,
                          int num_pages, void* pool, int32_t* status, cudaStream_t stream) {
  const int threads = 128;
  const int blocks = (T * 32 + threads - 1) / threads;
  uint8_t* out = static_cast<uint8_t*>(pool);
  switch (d.cache_dtype) {
    case MLA_F32:
      append_kernel<float, MLA_F32><<<blocks, threads, 0, stream>>>(
          d, (const float*)c_kv, (const float*)k_r, seq_idx, pos, T, bt, batch, maxp, num_pages,
          out, status);
      break;
    case MLA_BF16:
      append_kernel<__nv_bfloat16, MLA_BF16><<<blocks, threads, 0, stream>>>(
          d, (const __nv_bfloat16*)c_kv, (const __nv_bfloat16*)k_r, seq_idx, pos, T, bt, batch,
          maxp, num_pages, out, status);
      break;
    default:
      append_kernel<__nv_bfloat16, MLA_FP8_E4M3><<<blocks, threads, 0, stream>>>(
          d, (const __nv_bfloat16*)c_kv, (const __nv_bfloat16*)k_r, seq_idx, pos, T, bt, batch,
          maxp, num_pages, out, status);
      break;
  }
  return cudaGetLastError();
}

}  // namespace mla
