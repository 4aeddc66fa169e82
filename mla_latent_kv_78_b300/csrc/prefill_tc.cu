// Non-absorbed MLA over a prompt (prefill), on tensor cores.
//
// 「一文通透DeepSeek-V2」 §2.2.1: the naive formula restores k^C = W^{UK} c^{KV} and
// v^C = W^{UV} c^{KV} for every head, and §2.2.2 / 「deepseek(2)——deepseek 關鍵技術」 §1 give
//   k_{n,i} = [k^C_{n,i}; k^R_n],  q_{t,i} = [q^C_{t,i}; RoPE_t(q^R_{t,i})],
//   o_{t,i} = sum_{n <= t} softmax_n(q_{t,i} . k_{n,i} / sqrt(d_h + d_h^R)) v^C_{n,i}.
// For a prompt the decompression is cheaper than attending in the 576-d latent space, so this
// path forms K^C, V^C with the projection GEMM (bf16, [L][H d_h]), assembles Q = [q^C; RoPE(q^R)]
// ([L][H][d_h + d_h^R]) and runs causal attention per head:
//   one CTA per (head, 256 queries) as two 128-query tiles that share every key and value
//   block; 64-key blocks; per tile S = Q K^T (M = 128 queries, N = 64 keys, K = 192) into one of
//   two TMEM buffers; a softmax thread per query row (a reference maximum that moves when a
//   block's maximum exceeds it by more than 2^8, O rescaled in TMEM then); P (bf16) through
//   shared memory; O += P V (M = 128, N = 128, K = 64) in TMEM; TMA loads of both tiles' Q
//   once, of K^C, k^R and V^C in 2-stage rings. Warp 0 loads, warp 1 issues the MMAs, warps 2-5
//   and 6-9 run the two tiles' softmax (TMEM lane quadrant = warp % 4), so each scheduler
//   interleaves two softmax warps. Every wait is bounded.
#include <math_constants.h>

#include "mla_internal.cuh"
#include "tc_ptx.cuh"
#include "tma_host.cuh"

namespace mla {
namespace pf {

using namespace ptx;

constexpr int kD = 128, kR = 64, kDQ = kD + kR;   // per-head qk width 192, v width 128
constexpr int kBQ = 128, kBK = 64;               // queries per tile, keys per block
constexpr int kTiles = 2;                        // query tiles per CTA, each with its softmax group
constexpr int kNK = 3, kNV = 3;                  // ring stages
constexpr int kThreads = 64 + 128 * kTiles;      // loader warp, MMA warp, 4 softmax warps per tile
constexpr long long kTimeout = 4000000000LL;

// shared-memory layout (bytes from the 1024-aligned base)
constexpr int Q_OFF = 0;                             // per tile 3 boxes [128 q x 64] = 48 KB
constexpr int K_OFF = Q_OFF + kTiles * 3 * 16384;    // kNK stages of 3 boxes [64 keys x 64] = 24 KB
constexpr int V_OFF = K_OFF + kNK * 3 * 8192;        // kNV stages of 2 boxes [64 keys x 64 dv] = 16 KB
constexpr int BAR_OFF = V_OFF + kNV * 2 * 8192;      // (P lives in tensor memory)
constexpr int kSmem = BAR_OFF + 256 + 1024;

struct Bars {
  uint64_t q_full;
  uint64_t k_full[kNK], k_empty[kNK];
  uint64_t v_full[kNV], v_empty[kNV];
  uint64_t s_full[kTiles][2], p_full[kTiles][2], pv_done[kTiles][2];   // by S / P buffer
  uint32_t tmem;
};
static_assert(sizeof(Bars) <= 256, "barriers");

struct Params {
  int L, H;
  float scale_log2;
  float* o;   // [L][H][D] fp32
  int32_t* status;
};

__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, int32_t* status) {
  const uint32_t a = smem_u32(bar);
  const long long t0 = clock64();
  while (!mbar_try_wait(a, parity)) {
    if (clock64() - t0 > kTimeout) {
      flag_status(status, MLA_DEV_TIMEOUT);
      return false;
    }
  }
  return true;
}

// grid (H, ceil(L / 256)), 320 threads. Two query tiles share every key and value block: the
// MMA warp issues S(j) of both tiles from one K stage and P.V(j - 1) of both from one V stage,
// and while one tile's softmax group works the tensor core serves the other.
__global__ void __launch_bounds__(kThreads, 1)
    prefill_attn_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmKR, const __grid_constant__ CUtensorMap tmV,
                        const Params p) {
  extern __shared__ __align__(1024) uint8_t raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(sm + BAR_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the query blocks in decreasing order: the last ones attend to the most keys and start first
  const int h = blockIdx.x, q0 = (gridDim.y - 1 - blockIdx.y) * (kTiles * kBQ);
  // key blocks each tile needs (causal: up to its last query); 0 for a tile past the prompt
  const int nkb_all = (p.L + kBK - 1) / kBK;
  auto nkb_of = [&](int t) -> int {
    const int qs = q0 + t * kBQ;
    return qs < p.L ? min(nkb_all, (min(qs + kBQ, p.L) - 1) / kBK + 1) : 0;
  };
  const int nkb0 = nkb_of(0), nkb1 = nkb_of(1);
  const int nkb = max(nkb0, nkb1);
  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < kNK; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
    }
    for (int s = 0; s < kNV; ++s) {
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    for (int t = 0; t < kTiles; ++t) {
      for (int s = 0; s < 2; ++s) {
        mbar_init(&bars->s_full[t][s], 1);
        mbar_init(&bars->p_full[t][s], 4);   // the tile's 4 softmax warps
        mbar_init(&bars->pv_done[t][s], 1);
      }
    }
    fence_mbarrier_init_cluster();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem, 512);   // tile t: S / P buffers at 256t and 256t + 64, O at 256t + 128
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem;
  griddep_launch_dependents();
  griddep_wait();

  if (warp == 0) {
    // ---------------------------------------------------------------- loads (one box per lane)
    const uint64_t pol = policy_evict_normal();
    if (lane < 3 * kTiles) {   // both tiles' Q (rows past the prompt read as zeros)
      if (lane == 0) mbar_arrive_expect_tx(&bars->q_full, 3 * kTiles * 16384);
      __syncwarp((1u << (3 * kTiles)) - 1u);
      const int t = lane / 3, c = lane % 3;
      tma_load_3d(sm + Q_OFF + t * 3 * 16384 + c * 16384, &tmQ, c * 64, h, q0 + t * kBQ, &bars->q_full, pol);
    }
    bool ok = true;
    for (int j = 0; j < nkb && ok; ++j) {
      const int k0 = j * kBK;
      // K block: lanes 8*(j%3)+{0,1,2}; V block: lanes 8*(j%3)+{3,4}
      const int q = lane - 8 * (j % 3);
      bool r = true;
      if (q >= 0 && q < 5) {
        if (q < 3) {
          const int st = j % kNK;
          if (j >= kNK) r = wait_bounded(&bars->k_empty[st], ((j / kNK) - 1) & 1, p.status);
          if (r) {
            if (q == 0) mbar_arrive_expect_tx(&bars->k_full[st], 3 * 8192);
            uint8_t* dst = sm + K_OFF + st * 3 * 8192 + q * 8192;
            if (q < 2)
              tma_load_3d(dst, &tmK, q * 64, h, k0, &bars->k_full[st], pol);
            else
              tma_load_2d(dst, &tmKR, 0, k0, &bars->k_full[st], pol);
          }
        } else {
          const int st = j % kNV, b = q - 3;
          if (j >= kNV) r = wait_bounded(&bars->v_empty[st], ((j / kNV) - 1) & 1, p.status);
          if (r) {
            if (b == 0) mbar_arrive_expect_tx(&bars->v_full[st], 2 * 8192);
            tma_load_3d(sm + V_OFF + st * 2 * 8192 + b * 8192, &tmV, b * 64, h, k0, &bars->v_full[st], pol);
          }
        }
      }
      ok = __all_sync(0xffffffffu, r);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idS = idesc_bf16_f32(kBQ, kBK, 0, 0);
      const uint32_t idPV = idesc_bf16_f32(kBQ, kD, 0, 1);   // P K-major, V MN-major
      bool ok = wait_bounded(&bars->q_full, 0, p.status);
      auto issue_pv = [&](int jj) -> bool {
        const int st = jj % kNV;
        if (!wait_bounded(&bars->v_full[st], (jj / kNV) & 1, p.status)) return false;
        const uint32_t va = smem_u32(sm + V_OFF + st * 2 * 8192);
        const int bb = jj & 1;
        for (int t = 0; t < kTiles; ++t) {
          if (jj >= (t ? nkb1 : nkb0)) continue;
          if (!wait_bounded(&bars->p_full[t][bb], (jj >> 1) & 1, p.status)) return false;
          tc_fence_after();
          // A = P in tensor memory: the bf16 weights the softmax wrote over S buffer bb
          const uint32_t pa = tmem + (uint32_t)t * 256 + (uint32_t)bb * 64;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            mma_bf16_ta(tmem + (uint32_t)t * 256 + 128, pa + (uint32_t)k * 8,
                        smem_desc(va + k * 2048, 8192, 1024, kSw128), idPV, (jj | k) != 0);
          mma_commit(&bars->pv_done[t][bb]);
        }
        mma_commit(&bars->v_empty[st]);
        return true;
      };
      for (int j = 0; j < nkb && ok; ++j) {
        const int st = j % kNK, b = j & 1;
        ok = wait_bounded(&bars->k_full[st], (j / kNK) & 1, p.status);
        if (!ok) break;
        const uint32_t ka = smem_u32(sm + K_OFF + st * 3 * 8192);
        for (int t = 0; t < kTiles && ok; ++t) {
          if (j >= (t ? nkb1 : nkb0)) continue;
          // S / P buffer b is free once P.V of block j - 2 has read its weights
          if (j >= 2) ok = wait_bounded(&bars->pv_done[t][b], ((j >> 1) - 1) & 1, p.status);
          if (!ok) break;
          tc_fence_after();
          const uint32_t qa = smem_u32(sm + Q_OFF + t * 3 * 16384);
#pragma unroll
          for (int c = 0; c < 3; ++c)
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_bf16(tmem + (uint32_t)t * 256 + (uint32_t)b * 64, smem_desc(qa + c * 16384 + k * 32, 16, 1024, kSw128),
                       smem_desc(ka + c * 8192 + k * 32, 16, 1024, kSw128), idS, (c | k) != 0);
          mma_commit(&bars->s_full[t][b]);
        }
        mma_commit(&bars->k_empty[st]);
        if (ok && j >= 1) ok = issue_pv(j - 1);
      }
      if (ok && nkb > 0) issue_pv(nkb - 1);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- softmax (query rows)
    const int t = (warp - 2) >> 2;          // query tile of this softmax group
    const int nkbt = t ? nkb1 : nkb0;
    const int qd = warp & 3;
    const int r = qd * 32 + lane;           // query row of the tile = TMEM lane
    const int qt = q0 + t * kBQ;            // the tile's first query
    const int qi = qt + r;                  // query position
    const uint32_t lane_addr = tmem + (uint32_t)t * 256 + ((uint32_t)(qd * 32) << 16);
    float m = -CUDART_INF_F, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nkbt && ok; ++j) {
      const int b = j & 1;
      ok = wait_bounded(&bars->s_full[t][b], (j >> 1) & 1, p.status);
      if (!ok) break;
      tc_fence_after();
      float s[64];
      tmem_ld32(lane_addr + b * 64, s);
      tmem_ld32(lane_addr + b * 64 + 32, s + 32);
      tmem_ld_wait();
      const int k0 = j * kBK;
      float mx = -CUDART_INF_F;
      if (k0 + kBK - 1 > qt || k0 + kBK > p.L) {
        // a block on the tile's diagonal or at the prompt's end: mask keys past the query
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const bool valid = k0 + c <= qi && k0 + c < p.L;
          s[c] = valid ? s[c] * p.scale_log2 : -CUDART_INF_F;
          mx = fmaxf(mx, s[c]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          s[c] *= p.scale_log2;
          mx = fmaxf(mx, s[c]);
        }
      }
      // Lazy reference: the row keeps m while this block's maximum exceeds it by at most 8
      // (log2 units; weights up to 2^8 are exact in bf16 and fp32), so most blocks need no
      // rescale of O. A larger maximum moves m here, before any weight is formed, so no weight
      // is ever clamped.
      const bool move = mx > m + 8.f;
      const float m_new = move ? mx : m;
      const float alpha = move ? (m == -CUDART_INF_F ? 0.f : ex2(m - m_new)) : 1.f;
      m = m_new;
      uint32_t pk[32];
      float sum = 0.f;
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float p0 = m == -CUDART_INF_F ? 0.f : ex2(s[2 * c] - m);
        const float p1 = m == -CUDART_INF_F ? 0.f : ex2(s[2 * c + 1] - m);
        pk[c] = pack_bf16x2(p0, p1);
        sum += __uint_as_float(pk[c] << 16) + __uint_as_float(pk[c] & 0xFFFF0000u);
      }
      l = l * alpha + sum;
      // O is stable to rescale once P.V of block j - 1 is done (only then is it waited for)
      if (j >= 1 && __any_sync(0xffffffffu, alpha != 1.f)) {
        ok = wait_bounded(&bars->pv_done[t][(j - 1) & 1], ((j - 1) >> 1) & 1, p.status);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < kD; c += 32) {
          float o[32];
          tmem_ld32(lane_addr + 128 + c, o);
          tmem_ld_wait();
#pragma unroll
          for (int x = 0; x < 32; ++x) o[x] *= alpha;
          tmem_st32(lane_addr + 128 + c, o);
        }
        tmem_st_wait();
      }
      // P row r over the S columns just read (bf16 pairs, one 32-bit column per two keys)
      {
        float pf[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) pf[c] = __uint_as_float(pk[c]);
        tmem_st32(lane_addr + b * 64, pf);
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full[t][b]);
    }
    if (ok && nkbt > 0) ok = wait_bounded(&bars->pv_done[t][(nkbt - 1) & 1], ((nkbt - 1) >> 1) & 1, p.status);
    ok = __all_sync(0xffffffffu, ok);
    if (ok && nkbt > 0) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
      for (int c = 0; c < kD; c += 32) {
        float o[32];
        tmem_ld32(lane_addr + 128 + c, o);
        tmem_ld_wait();
        if (qi < p.L) {
          float4* dst = reinterpret_cast<float4*>(p.o + ((size_t)qi * p.H + h) * kD + c);
#pragma unroll
          for (int x = 0; x < 8; ++x)
            dst[x] = make_float4(o[4 * x] * inv, o[4 * x + 1] * inv, o[4 * x + 2] * inv, o[4 * x + 3] * inv);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// Q[t][i] = [q^C[t][i] ; RoPE_t(q^R[t][i])] (bf16), one block per token: the token's cos/sin
// pairs once in shared memory (they do not depend on the head), then one thread per
// (head, 16 bytes) of the output row.
__global__ void __launch_bounds__(256) prefill_q_kernel(const __nv_bfloat16* __restrict__ q_c,
                                                         const __nv_bfloat16* __restrict__ q_r, int L, int H,
                                                         __nv_bfloat16* __restrict__ q, const RopeTable rt) {
  __shared__ float cs[kR / 2], sn[kR / 2];
  griddep_wait();
  const int t = blockIdx.x;
  if (threadIdx.x < kR / 2) rope_cs(t, rt.hi[threadIdx.x], rt.lo[threadIdx.x], &cs[threadIdx.x], &sn[threadIdx.x]);
  __syncthreads();
  for (int idx = threadIdx.x; idx < H * (kDQ / 8); idx += blockDim.x) {
    const int h = idx / (kDQ / 8), u = idx % (kDQ / 8);
    const size_t th = (size_t)t * H + h;
    uint4* dst = reinterpret_cast<uint4*>(q + th * kDQ) + u;
    if (u < kD / 8) {
      *dst = reinterpret_cast<const uint4*>(q_c + th * kD)[u];
      continue;
    }
    const uint4 x = reinterpret_cast<const uint4*>(q_r + th * kR)[u - kD / 8];
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int k = (u - kD / 8) * 4 + e;   // RoPE pair
      const float c = cs[k], s = sn[k];
      const float x0 = __uint_as_float(w[e] << 16), x1 = __uint_as_float(w[e] & 0xFFFF0000u);
      o[e] = pack_bf16x2(x0 * c - x1 * s, x0 * s + x1 * c);
    }
    *dst = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

}  // namespace pf

bool prefill_supported(const Dims& d) {
  return d.act_dtype == MLA_BF16 && d.D == pf::kD && d.R == pf::kR && d.C % 8 == 0;
}

size_t prefill_workspace_bytes(const Dims& d, int L) {
  // K^C and V^C [L][H D] and Q [L][H][D + R], bf16, each 256-byte aligned
  auto al = [](size_t b) { return (b + 255) / 256 * 256; };
  return 2 * al((size_t)L * d.H * d.D * 2) + al((size_t)L * d.H * (d.D + d.R) * 2);
}

cudaError_t launch_prefill(const Dims& d, const void* c_kv, const void* k_r, int L, const void* q_c,
                           const void* q_r, const void* w_uk, const void* w_uv, float* o, void* ws,
                           int32_t* status, cudaStream_t stream) {
  auto al = [](size_t b) { return (b + 255) / 256 * 256; };
  uint8_t* base = static_cast<uint8_t*>(ws);
  __nv_bfloat16* kc = reinterpret_cast<__nv_bfloat16*>(base);
  __nv_bfloat16* vc = reinterpret_cast<__nv_bfloat16*>(base + al((size_t)L * d.H * d.D * 2));
  __nv_bfloat16* q = reinterpret_cast<__nv_bfloat16*>(base + 2 * al((size_t)L * d.H * d.D * 2));
  const int HD = d.H * d.D;
  // K^C = c . W^{UK}^T and V^C = c . W^{UV}^T: W viewed as [H D][C] (head i's rows i D ..)
  cudaError_t e = launch_gemm(c_kv, w_uk, L, HD, d.C, 1, nullptr, kc, MLA_BF16, status, stream);
  if (e == cudaSuccess) e = launch_gemm(c_kv, w_uv, L, HD, d.C, 1, nullptr, vc, MLA_BF16, status, stream);
  if (e != cudaSuccess) return e;
  RopeTable rt;
  fill_rope_table(&rt, d);
  e = launch_programmatic(pf::prefill_q_kernel, dim3((unsigned)L), dim3(256), 0, stream,
                          (const __nv_bfloat16*)q_c, (const __nv_bfloat16*)q_r, L, d.H, q, rt);
  if (e != cudaSuccess) return e;
  CUtensorMap tmQ, tmK, tmKR, tmV;
  {
    const uint64_t dims[3] = {(uint64_t)pf::kDQ, (uint64_t)d.H, (uint64_t)L};
    const uint64_t st[2] = {(uint64_t)pf::kDQ * 2, (uint64_t)d.H * pf::kDQ * 2};
    const uint32_t box[3] = {64, 1, pf::kBQ};
    if (!encode_bf16_map(&tmQ, q, 3, dims, st, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[3] = {(uint64_t)pf::kD, (uint64_t)d.H, (uint64_t)L};
    const uint64_t st[2] = {(uint64_t)pf::kD * 2, (uint64_t)HD * 2};
    const uint32_t box[3] = {64, 1, pf::kBK};
    if (!encode_bf16_map(&tmK, kc, 3, dims, st, box)) return cudaErrorInvalidValue;
    if (!encode_bf16_map(&tmV, vc, 3, dims, st, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[2] = {(uint64_t)pf::kR, (uint64_t)L};
    const uint64_t st[1] = {(uint64_t)pf::kR * 2};
    const uint32_t box[2] = {64, pf::kBK};
    if (!encode_bf16_map(&tmKR, k_r, 2, dims, st, box)) return cudaErrorInvalidValue;
  }
  pf::Params p;
  p.L = L;
  p.H = d.H;
  p.scale_log2 = d.scale * 1.4426950408889634f;
  p.o = o;
  p.status = status;
  static std::atomic<bool> attr[kMaxDevices];
  e = set_smem_limit_once(pf::prefill_attn_kernel, pf::kSmem, attr);
  if (e != cudaSuccess) return e;
  dim3 grid(d.H, (L + pf::kTiles * pf::kBQ - 1) / (pf::kTiles * pf::kBQ));
  e = launch_programmatic(pf::prefill_attn_kernel, grid, dim3(pf::kThreads), pf::kSmem, stream, tmQ, tmK,
                          tmKR, tmV, p);
  return e == cudaSuccess ? cudaGetLastError() : e;
}

}  // namespace mla
