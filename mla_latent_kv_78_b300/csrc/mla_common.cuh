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
  float scale;       // softmax scale (YaRN's logit factor included)
  float rope_base;
  int entry_bytes;   // bytes of one pool entry
  // YaRN on the decoupled RoPE (yarn_s <= 1: plain RoPE)
  float yarn_s, yarn_alpha, yarn_beta;
  int yarn_orig;
  // FP8 cache: scores on FP8 tensor cores (q_lat's latent part quantised per 1x128 group)
  bool fp8_scores;
};

// RoPE frequency of pair k, computed on the host in fp64: base^(-2k/R), or with YaRN
// (「一文通透DeepSeek-V2」 §3.1.3) the by-parts interpolation between theta/s and theta over
// r = original context / wavelength.
inline double rope_theta_host(const Dims& d, int k) {
  const double th = pow((double)d.rope_base, -2.0 * (double)k / (double)d.R);
  if (!(d.yarn_s > 1.f)) return th;
  const double r = (double)d.yarn_orig * th / (2.0 * 3.14159265358979323846);
  double g = (r - (double)d.yarn_alpha) / ((double)d.yarn_beta - (double)d.yarn_alpha);
  g = g < 0.0 ? 0.0 : (g > 1.0 ? 1.0 : g);
  return (1.0 - g) * th / (double)d.yarn_s + g * th;
}

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

// RoPE frequencies theta_k = base^(-2k/R), computed on the host in fp64 and passed as a
// float pair (hi + lo) and as a double.
constexpr int kMaxRopePairs = 64;
struct RopeTable {
  float hi[kMaxRopePairs], lo[kMaxRopePairs];
  double th[kMaxRopePairs];
};

inline void fill_rope_table(RopeTable* t, const Dims& d) {
  for (int k = 0; k < d.R / 2 && k < kMaxRopePairs; ++k) {
    const double th = rope_theta_host(d, k);
    t->th[k] = th;
    t->hi[k] = (float)th;
    t->lo[k] = (float)(th - (double)t->hi[k]);
  }
}

// cos/sin of pos * theta without fp64: the angle is carried as a float pair (exact product of
// the integer position with theta_hi via FMA, plus pos * theta_lo), reduced by 2*pi with a
// three-part Cody-Waite split (6.28125 + 0.0019350051879882812 + 3.0199160e-07; the first two
// products are exact for |n| < 2^15, i.e. positions up to ~2e5), then evaluated with sincosf.
__device__ __forceinline__ void rope_cs(int pos, float th_hi, float th_lo, float* c, float* s) {
  const float p = (float)pos;
  const float a_hi = p * th_hi;
  const float a_lo = fmaf(p, th_hi, -a_hi) + p * th_lo;
  const float n = rintf(a_hi * 0.15915493667125702f);
  float r = fmaf(-n, 6.28125f, a_hi);
  r = fmaf(-n, 0.0019350051879882812f, r);
  r = fmaf(-n, 3.019916050561733e-07f, r);
  r += a_lo;
  sincosf(r, s, c);
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
