// K1: latent-cache write with decoupled RoPE on k^R (and optional E4M3 quantisation).
//
// 「一文通透DeepSeek-V2」 §2.2.1: only c^{KV}_t is cached; §2.2.2: k^R_t = RoPE(W^{KR} h_t)
// is cached beside it. 「Deepseek系列从v3到R易背面经版」 F8量化策略: activations are
// quantised per token in 1x128 groups, E4M3.
//
// One warp per token. The page/slot mapping is integer-exact; RoPE frequencies come from the
// host in fp64; the rotation runs in fp64 for an fp32 cache and in fp32 with a double-float
// angle reduction for bf16 / FP8 caches (both far below one ulp of the stored type), rounded
// once; the FP8 scale and the per-element division are IEEE fp32 (__fdiv_rn), so the integer
// codes match a CPU encoder that takes the same fp32 decisions.
#include "mla_internal.cuh"
#include "tc_ptx.cuh"

namespace mla {

// rotated pair k of one token: (x0, x1) -> (x0 c - x1 s, x0 s + x1 c). bf16 and FP8 caches
// keep k^R in bf16, so fp32 with a double-float angle reduction is exact to well below one
// bf16 ulp; the fp32 cache uses fp64 (fp32 accuracy is what it stores).
template <int CACHE>
__device__ __forceinline__ void rope_pair(const RopeTable& rt, int pos, int k, int R, double base,
                                          float x0, float x1, float* y0, float* y1) {
  if constexpr (CACHE == MLA_F32) {
    double cs, sn;
    if (k < kMaxRopePairs) {
      sincos((double)pos * rt.th[k], &sn, &cs);
    } else {
      rope_cos_sin(pos, k, R, base, &cs, &sn);
    }
    *y0 = (float)((double)x0 * cs - (double)x1 * sn);
    *y1 = (float)((double)x0 * sn + (double)x1 * cs);
  } else {
    float cs, sn;
    if (k < kMaxRopePairs) {
      rope_cs(pos, rt.hi[k], rt.lo[k], &cs, &sn);
      *y0 = x0 * cs - x1 * sn;
      *y1 = x0 * sn + x1 * cs;
    } else {
      double c2, s2;
      rope_cos_sin(pos, k, R, base, &c2, &s2);
      *y0 = (float)((double)x0 * c2 - (double)x1 * s2);
      *y1 = (float)((double)x0 * s2 + (double)x1 * c2);
    }
  }
}

// One token's cache entry (one warp): [c ; RoPE_pos(k^R)] into its slot, c as E4M3 codes with
// per-group fp32 scales for an FP8 cache. src_c / src_r may point to global or shared memory.
template <typename In, int CACHE>
__device__ __forceinline__ void write_entry(const Dims& d, const In* src_c, const In* src_r, int p,
                                            uint8_t* dst, const RopeTable& rt, int lane) {
  const double base = (double)d.rope_base;
  if constexpr (CACHE != MLA_FP8_E4M3) {
    In* out = reinterpret_cast<In*>(dst);
    // the latent row: 16-byte vectors when the row and both ends are 16-byte aligned
    const size_t row_bytes = (size_t)d.C * sizeof(In);
    if ((row_bytes & 15) == 0 && ((reinterpret_cast<uintptr_t>(src_c) | reinterpret_cast<uintptr_t>(out)) & 15) == 0) {
      const uint4* s4 = reinterpret_cast<const uint4*>(src_c);
      uint4* o4 = reinterpret_cast<uint4*>(out);
      for (int k = lane; k < (int)(row_bytes / 16); k += 32) o4[k] = s4[k];
    } else {
      for (int k = lane; k < d.C; k += 32) out[k] = src_c[k];
    }
    for (int k = lane; k < d.R / 2; k += 32) {
      float y0, y1;
      rope_pair<CACHE>(rt, p, k, d.R, base, ld_act(src_r, 2 * k), ld_act(src_r, 2 * k + 1), &y0, &y1);
      st_act(out, d.C + 2 * k, y0);
      st_act(out, d.C + 2 * k + 1, y1);
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
      float y0, y1;
      rope_pair<CACHE>(rt, p, k, d.R, base, ld_act(src_r, 2 * k), ld_act(src_r, 2 * k + 1), &y0, &y1);
      kr[2 * k] = __float2bfloat16_rn(y0);
      kr[2 * k + 1] = __float2bfloat16_rn(y1);
    }
  }
}

// The pool entry of token (b, p), or nullptr (flagged) when an index is out of range.
__device__ __forceinline__ uint8_t* entry_of(const Dims& d, int b, int p, const int32_t* bt, int batch,
                                             int maxp, int num_pages, uint8_t* pool, int32_t* status,
                                             int lane) {
  if (b < 0 || b >= batch || p < 0 || p / d.P >= maxp) {
    if (lane == 0) flag_status(status, MLA_DEV_INDEX_OUT_OF_RANGE);
    return nullptr;
  }
  const int page = bt[(size_t)b * maxp + p / d.P];
  if (page < 0 || page >= num_pages) {
    if (lane == 0) flag_status(status, MLA_DEV_INDEX_OUT_OF_RANGE);
    return nullptr;
  }
  return pool + ((size_t)page * d.P + (p % d.P)) * (size_t)d.entry_bytes;
}

template <typename In, int CACHE>
__global__ void __launch_bounds__(128) append_kernel(Dims d, const In* __restrict__ c_kv,
                                                     const In* __restrict__ k_r,
                                                     const int32_t* __restrict__ seq_idx,
                                                     const int32_t* __restrict__ pos, int T,
                                                     const int32_t* __restrict__ bt, int batch,
                                                     int maxp, int num_pages,
                                                     uint8_t* __restrict__ pool,
                                                     int32_t* status, const RopeTable rt) {
  // a kernel launched programmatically after this one (the query absorption of a decode step)
  // may start its own set-up now; it reads its inputs only once this grid has completed
  ptx::griddep_launch_dependents();
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const int p = pos[t];
  uint8_t* dst = entry_of(d, seq_idx[t], p, bt, batch, maxp, num_pages, pool, status, lane);
  if (!dst) return;
  write_entry<In, CACHE>(d, c_kv + (size_t)t * d.C, k_r + (size_t)t * d.R, p, dst, rt, lane);
}

// Epilogue of the fused upstream append (「一文通透DeepSeek-V2」 §2.2.1 c^{KV} = W^{DKV} h, §3.1.4
// the RMSNorm after the compressed latent, §2.2.2 k^R = RoPE(W^{KR} h)), one 256-thread block per
// token: the projection's split partials [splits][T][C + R] are summed in split order (each
// thread a few elements, so many loads are in flight), the latent is normalised
// (gain * x / sqrt(mean(x^2) + eps), fp32, a block-wide sum of squares), both parts are rounded
// to bf16 in shared memory (the activation type a separate projection would have produced) and
// warp 0 writes the entry as mla_append_cache writes it.
template <int CACHE>
__global__ void __launch_bounds__(256) project_append_kernel(
    Dims d, const float* __restrict__ part, int splits, const float* __restrict__ gain, float eps,
    const int32_t* __restrict__ seq_idx, const int32_t* __restrict__ pos, int T,
    const int32_t* __restrict__ bt, int batch, int maxp, int num_pages, uint8_t* __restrict__ pool,
    int32_t* status, const RopeTable rt) {
  // the latent's fp32 sums [C], the bf16 row [C + R], 8 warp partial sums of squares
  extern __shared__ __align__(16) float stage[];
  ptx::griddep_wait();
  const int t = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int CR = d.C + d.R;
  float* xs = stage;
  __nv_bfloat16* row = reinterpret_cast<__nv_bfloat16*>(stage + d.C);
  float* red = stage + d.C + (CR + 1) / 2 + 3;
  const size_t count = (size_t)T * CR;
  const float* src = part + (size_t)t * CR;
  float sq = 0.f;
  for (int k = threadIdx.x; k < CR; k += blockDim.x) {
    float acc = 0.f;
    for (int s = 0; s < splits; ++s) acc += src[(size_t)s * count + k];
    if (k < d.C) {
      xs[k] = acc;
      sq += acc * acc;
    } else {
      row[k] = __float2bfloat16_rn(acc);   // k^R: no norm
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off);
  if (lane == 0) red[warp] = sq;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) tot += red[w];
  const float inv = 1.0f / sqrtf(tot / (float)d.C + eps);
  for (int k = threadIdx.x; k < d.C; k += blockDim.x) row[k] = __float2bfloat16_rn(xs[k] * inv * gain[k]);
  __syncthreads();
  if (warp != 0) return;
  const int p = pos[t];
  uint8_t* dst = entry_of(d, seq_idx[t], p, bt, batch, maxp, num_pages, pool, status, lane);
  if (!dst) return;
  write_entry<__nv_bfloat16, CACHE>(d, row, row + d.C, p, dst, rt, lane);
}

// Shared-memory bytes of project_append_kernel's block.
inline size_t project_append_smem(const Dims& d) {
  return sizeof(float) * ((size_t)d.C + (size_t)(d.C + d.R + 1) / 2 + 3 + 8 + 4);
}

cudaError_t launch_append(const Dims& d, const void* c_kv, const void* k_r, const int32_t* seq_idx,
                          const int32_t* pos, int T, const int32_t* bt, int batch, int maxp,
                          int num_pages, void* pool, int32_t* status, cudaStream_t stream) {
  const int threads = 128;
  const int blocks = (T * 32 + threads - 1) / threads;
  uint8_t* out = static_cast<uint8_t*>(pool);
  RopeTable rt;
  fill_rope_table(&rt, d);
  switch (d.cache_dtype) {
    case MLA_F32:
      append_kernel<float, MLA_F32><<<blocks, threads, 0, stream>>>(
          d, (const float*)c_kv, (const float*)k_r, seq_idx, pos, T, bt, batch, maxp, num_pages,
          out, status, rt);
      break;
    case MLA_BF16:
      append_kernel<__nv_bfloat16, MLA_BF16><<<blocks, threads, 0, stream>>>(
          d, (const __nv_bfloat16*)c_kv, (const __nv_bfloat16*)k_r, seq_idx, pos, T, bt, batch,
          maxp, num_pages, out, status, rt);
      break;
    default:
      append_kernel<__nv_bfloat16, MLA_FP8_E4M3><<<blocks, threads, 0, stream>>>(
          d, (const __nv_bfloat16*)c_kv, (const __nv_bfloat16*)k_r, seq_idx, pos, T, bt, batch,
          maxp, num_pages, out, status, rt);
      break;
  }
  return cudaGetLastError();
}

cudaError_t launch_project_append(const Dims& d, const void* h, int d_model, const void* w, int T,
                                  const float* gain, float eps, const int32_t* seq_idx,
                                  const int32_t* pos, const int32_t* bt, int batch, int maxp,
                                  int num_pages, void* pool, void* ws, int splits, int32_t* status,
                                  cudaStream_t stream) {
  const int CR = d.C + d.R;
  float* part = static_cast<float*>(ws);
  // [c^{KV}; k^R] pre-norm, as split partials: X = h [T][d_model], W = [W^{DKV}; W^{KR}] [CR][d_model]
  cudaError_t e = launch_gemm(h, w, T, CR, d_model, splits, part, nullptr, kGemmPartials, status, stream);
  if (e != cudaSuccess) return e;
  RopeTable rt;
  fill_rope_table(&rt, d);
  const size_t smem = project_append_smem(d);
  uint8_t* out = static_cast<uint8_t*>(pool);
  if (d.cache_dtype == MLA_FP8_E4M3)
    e = launch_programmatic(project_append_kernel<MLA_FP8_E4M3>, dim3(T), dim3(256), smem, stream, d,
                            (const float*)part, splits, gain, eps, seq_idx, pos, T, bt, batch, maxp,
                            num_pages, out, status, rt);
  else
    e = launch_programmatic(project_append_kernel<MLA_BF16>, dim3(T), dim3(256), smem, stream, d,
                            (const float*)part, splits, gain, eps, seq_idx, pos, T, bt, batch, maxp,
                            num_pages, out, status, rt);
  return e == cudaSuccess ? cudaGetLastError() : e;
}

}  // namespace mla
