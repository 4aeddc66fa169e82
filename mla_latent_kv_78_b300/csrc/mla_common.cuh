// Shared device helpers for the MLA decode kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mla.h"

namespace mla {

constexpr int kFp8Group = 128;
constexpr float kE4M3Max = 448.0f;

struct Dims {
  int H, D, C, R, P;
  int cache_dtype, act_dtype;
  float scale;       // softmax scale
  float rope_base;
  int entry_bytes;   // bytes of one pool entry
};

__device__ __forceinline__ void flag_status(int32_t* st, int bits) {
  if (st) atomicOr(st, bits);
}

__device__ __forceinline__ float ld_act(const float* p, size_t i) { return p[i]; }
__device__ __forceinline__ float ld_act(const __nv_bfloat16* p, size_t i) {
  return __bfloat162float(p[i]);
}
__device__ __forceinline__ void st_act(float* p, size_t i, float v) { p[i] = v; }
__device__ __forceinline__ void st_act(__nv_bfloat16* p, size_t i, float v) {
  p[i] = __float2bfloat16_rn(v);
}

// RoPE angle of pair k at position pos: pos * base^(-2k/R), in fp64 so positions
// near 2^17 keep full accuracy.
__device__ __forceinline__ void rope_cos_sin(int pos, int k, int R, double base, double* c,
                                             double* s) {
  double theta = pow(base, -2.0 * (double)k / (double)R);
  sincos((double)pos * theta, s, c);
}

// E4M3 encode of one fp32 value: round to nearest even, saturate to +-448.
__device__ __forceinline__ uint8_t e4m3_encode(float x) {
  __nv_fp8_storage_t v = __nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
  return (uint8_t)v;
}

__device__ __forceinline__ float e4m3_decode(uint8_t code) {
  __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)code, __NV_E4M3);
  return __half2float(__half(h));
}

}  // namespace mla
