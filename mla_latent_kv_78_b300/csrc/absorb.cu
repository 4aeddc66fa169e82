// K2 / K5: query-side and output-side absorption on CUDA cores.
//
// 「一文通透DeepSeek-V2」 §2.2.1 (last paragraph): by associativity W^{UK} can be absorbed
// into the query side and W^{UV} into the output side, so keys and values are never
// decompressed. 「Deepseek系列从v3到R易背面经版」 MLA: fusing (W^{UQ})^T W^{UK} turns MHA
// into MQA over the shared latent.
//
//   absorb:   q_lat[t][i][0:C] = q_c[t][i][:] . W_UK[i][:][0:C];  q_lat[t][i][C:] = RoPE(q_r)
//   unabsorb: o[t][i][r]       = W_UV[i][r][:] . o_lat[t][i][:]
//
// Both read each head's weight block once per token tile (kTok tokens) and
// accumulate in fp32.
#include "mla_internal.cuh"

namespace mla {

constexpr int kTok = 16;  // tokens per CTA

// grid: (H + rope_blocks, ceil(T / kTok)); blocks x >= H rotate q^R for 32 heads each.
template <typename Act>
__global__ void __launch_bounds__(128) absorb_kernel(Dims d, const Act* __restrict__ q_c,
                                                     const Act* __restrict__ q_r,
                                                     const int32_t* __restrict__ pos, int T,
                                                     const Act* __restrict__ w_uk,
                                                     Act* __restrict__ q_lat, const RopeTable rt) {
  extern __shared__ float sm[];
  const int t0 = blockIdx.y * kTok;
  const int nt = min(kTok, T - t0);
  const int CR = d.C + d.R;
  if ((int)blockIdx.x < d.H) {
    const int i = blockIdx.x;
    // q_c rows of this head for the tile: sm[t * D + k]
    for (int idx = threadIdx.x; idx < kTok * d.D; idx += blockDim.x) {
      const int t = idx / d.D, k = idx % d.D;
      sm[idx] = t < nt ? ld_act(q_c, ((size_t)(t0 + t) * d.H + i) * d.D + k) : 0.f;
    }
    __syncthreads();
    const Act* w = w_uk + (size_t)i * d.D * d.C;
    for (int c = threadIdx.x; c < d.C; c += blockDim.x) {
      float acc[kTok];
#pragma unroll
      for (int t = 0; t < kTok; ++t) acc[t] = 0.f;
      for (int k = 0; k < d.D; ++k) {
        const float wv = ld_act(w, (size_t)k * d.C + c);
#pragma unroll
        for (int t = 0; t < kTok; ++t) acc[t] = fmaf(sm[t * d.D + k], wv, acc[t]);
      }
      for (int t = 0; t < nt; ++t) st_act(q_lat, ((size_t)(t0 + t) * d.H + i) * CR + c, acc[t]);
    }
  } else {
    // RoPE of q^R: cos/sin per (token, pair) once in fp64, then rotate 32 heads.
    const int h0 = (blockIdx.x - d.H) * 32;
    const int h1 = min(d.H, h0 + 32);
    const int R2 = d.R / 2;
    float* cs = sm;               // [kTok][R2]
    float* sn = sm + kTok * R2;   // [kTok][R2]
    for (int idx = threadIdx.x; idx < nt * R2; idx += blockDim.x) {
      const int t = idx / R2, k = idx % R2;
      double c, s;
      if (k < kMaxRopePairs)
        sincos((double)pos[t0 + t] * rt.th[k], &s, &c);
      else
        rope_cos_sin(pos[t0 + t], k, d.R, (double)d.rope_base, &c, &s);
      cs[idx] = (float)c;
      sn[idx] = (float)s;
    }
    __syncthreads();
    const int nh = h1 - h0;
    for (int idx = threadIdx.x; idx < nt * nh * R2; idx += blockDim.x) {
      const int k = idx % R2;
      const int h = h0 + (idx / R2) % nh;
      const int t = idx / (R2 * nh);
      const size_t src = ((size_t)(t0 + t) * d.H + h) * d.R + 2 * k;
      const float x0 = ld_act(q_r, src), x1 = ld_act(q_r, src + 1);
      const float c = cs[t * R2 + k], s = sn[t * R2 + k];
      const size_t dst = ((size_t)(t0 + t) * d.H + h) * CR + d.C + 2 * k;
      st_act(q_lat, dst, x0 * c - x1 * s);
      st_act(q_lat, dst + 1, x0 * s + x1 * c);
    }
  }
}

// grid: (H, ceil(T / kTok)); 4 warps; warp w computes rows r = w, w + 4, ...
template <typename Act>
__global__ void __launch_bounds__(128) unabsorb_kernel(Dims d, const Act* __restrict__ o_lat,
                                                       int T, const Act* __restrict__ w_uv,
                                                       float* __restrict__ o) {
  extern __shared__ float sm[];  // [kTok][C]
  const int i = blockIdx.x;
  const int t0 = blockIdx.y * kTok;
  const int nt = min(kTok, T - t0);
  for (int idx = threadIdx.x; idx < kTok * d.C; idx += blockDim.x) {
    const int t = idx / d.C, k = idx % d.C;
    sm[idx] = t < nt ? ld_act(o_lat, ((size_t)(t0 + t) * d.H + i) * d.C + k) : 0.f;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Act* w = w_uv + (size_t)i * d.D * d.C;
  for (int r = warp; r < d.D; r += 4) {
    float acc[kTok];
#pragma unroll
    for (int t = 0; t < kTok; ++t) acc[t] = 0.f;
    for (int k = lane; k < d.C; k += 32) {
      const float wv = ld_act(w, (size_t)r * d.C + k);
#pragma unroll
      for (int t = 0; t < kTok; ++t) acc[t] = fmaf(wv, sm[t * d.C + k], acc[t]);
    }
#pragma unroll
    for (int t = 0; t < kTok; ++t) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], off);
    }
    if (lane == 0)
      for (int t = 0; t < nt; ++t) o[((size_t)(t0 + t) * d.H + i) * d.D + r] = acc[t];
  }
}

cudaError_t launch_absorb(const Dims& d, const void* q_c, const void* q_r, const int32_t* pos,
                          int T, const void* w_uk, void* q_lat, cudaStream_t stream) {
  const int rope_blocks = (d.H + 31) / 32;
  dim3 grid(d.H + rope_blocks, (T + kTok - 1) / kTok);
  const size_t smem = sizeof(float) * (size_t)kTok * (d.D > d.R ? d.D : d.R);
  RopeTable rt;
  fill_rope_table(&rt, d);
  if (d.act_dtype == MLA_F32)
    absorb_kernel<float><<<grid, 128, smem, stream>>>(d, (const float*)q_c, (const float*)q_r, pos,
                                                      T, (const float*)w_uk, (float*)q_lat, rt);
  else
    absorb_kernel<__nv_bfloat16><<<grid, 128, smem, stream>>>(
        d, (const __nv_bfloat16*)q_c, (const __nv_bfloat16*)q_r, pos, T,
        (const __nv_bfloat16*)w_uk, (__nv_bfloat16*)q_lat, rt);
  return cudaGetLastError();
}

cudaError_t launch_unabsorb(const Dims& d, const void* o_lat, int T, const void* w_uv, float* o,
                            cudaStream_t stream) {
  dim3 grid(d.H, (T + kTok - 1) / kTok);
  const size_t smem = sizeof(float) * (size_t)kTok * d.C;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaSuccess;
    if (d.act_dtype == MLA_F32)
      e = cudaFuncSetAttribute(unabsorb_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem);
    else
      e = cudaFuncSetAttribute(unabsorb_kernel<__nv_bfloat16>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  if (d.act_dtype == MLA_F32)
    unabsorb_kernel<float><<<grid, 128, smem, stream>>>(d, (const float*)o_lat, T,
                                                        (const float*)w_uv, o);
  else
    unabsorb_kernel<__nv_bfloat16><<<grid, 128, smem, stream>>>(
        d, (const __nv_bfloat16*)o_lat, T, (const __nv_bfloat16*)w_uv, o);
  return cudaGetLastError();
}

}  // namespace mla
