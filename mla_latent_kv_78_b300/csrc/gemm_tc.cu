// Projections on tensor cores: Y[t][n] = sum_k X[t][k] W[n][k] (bf16 operands, fp32 accumulation).
//
// Used by the steps either side of the latent cache:
//   * the upstream projection of the cached quantities, [c^{KV}; k^R] = [W^{DKV}; W^{KR}] h
//     (「一文通透DeepSeek-V2」 §2.2.1, §2.2.2), finished by project_append's epilogue kernel;
//   * the output projection u_t = W^O [o_{t,1}; ...; o_{t,n_h}] (「一文通透DeepSeek-V2」 §2.1.2,
//     「deepseek(2)——deepseek 關鍵技術」 §1);
//   * the decompression k^C = W^{UK} c, v^C = W^{UV} c of the non-absorbed prefill.
// For decode-sized T the weights dominate the bytes, so a CTA owns 128 rows of W (the MMA's M,
// TMEM lane = output feature) for a tile of 64 or 128 tokens (N) and streams its share of K
// through a TMA ring (9 stages for 64 tokens, 6 for 128); K is split over CTAs when the (row,
// token) tiles alone leave SMs idle, and the fp32 partials are summed in a fixed order by
// gemm_reduce_kernel (the result does not depend on scheduling). Every wait is bounded.
#include "mla_internal.cuh"
#include "tc_ptx.cuh"
#include "tma_host.cuh"

namespace mla {
namespace gemm {

using namespace ptx;

constexpr int kBM = 128;       // rows of W per CTA
constexpr int kBK = 64;        // K per stage: one 128-byte swizzle atom of bf16
constexpr int kGroup = 3;   // stages refilled per producer step (every ring depth is a multiple)
constexpr long long kTimeout = 4000000000LL;

template <int BN>
struct GLay {
  static constexpr int kStages = BN <= 64 ? 9 : 6;   // as deep as shared memory allows
  static constexpr int A = kBM * kBK * 2;       // 16 KB
  static constexpr int B = BN * kBK * 2;        // 8 or 16 KB
  static constexpr int STAGE = A + B;
  static constexpr int BARS = kStages * STAGE;
  static constexpr int SMEM = BARS + (2 * kStages + 1) * 8 + 16 + 1024;
};

struct GemmParams {
  int T, N, K;
  int k_steps;     // 64-wide K steps per split
  float* out;      // [T][N] when splits == 1, else partials [splits][T][N]
  __nv_bfloat16* out_bf16;   // non-null: Y [T][N] in bf16 directly (splits == 1)
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

// grid (ceil(N / 128), ceil(T / BN), splits), 128 threads.
template <int BN>
__global__ void __launch_bounds__(128, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                const GemmParams p) {
  using Ly = GLay<BN>;
  constexpr int kStages = Ly::kStages;
  extern __shared__ __align__(1024) uint8_t raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + Ly::BARS);
  uint64_t* freeb = full + kStages;
  uint64_t* done = freeb + kStages;
  uint32_t* slot = reinterpret_cast<uint32_t*>(done + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * kBM, t0 = blockIdx.y * BN, split = blockIdx.z;
  const int k0 = split * p.k_steps * kBK;
  const int nk = max(0, min(p.k_steps, (p.K - k0 + kBK - 1) / kBK));
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&freeb[s], 1);
    }
    mbar_init(done, 1);
    fence_mbarrier_init_cluster();
  }
  if (warp == 1) {
    tmem_alloc(slot, BN < 32 ? 32 : BN);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;
  griddep_launch_dependents();
  griddep_wait();
  bool ok = true;
  if (warp == 0) {
    // ---- producer: stages are refilled kGroup at a time, stage g * kGroup + j by lane j, so
    // one instruction issues kGroup boxes (a warp's TMA loads issued by separate instructions
    // complete one after another on this part; the boxes of one instruction overlap)
    const uint64_t pol_w = policy_evict_first();   // weights are read once
    const uint64_t pol_x = policy_evict_last();    // activations are shared by the row tiles
    for (int g = 0; g * kGroup < nk && ok; ++g) {
      const int ks = g * kGroup + lane;
      const bool mine = lane < kGroup && ks < nk;
      const int st = ks % kStages;
      bool r = true;
      if (mine && ks >= kStages) r = wait_bounded(&freeb[st], ((ks / kStages) - 1) & 1, p.status);
      ok = __all_sync(0xffffffffu, r);
      if (!ok) break;
      if (mine) {
        uint8_t* dst = sm + st * Ly::STAGE;
        mbar_arrive_expect_tx(&full[st], Ly::STAGE);
        tma_load_2d(dst, &tmW, k0 + ks * kBK, n0, &full[st], pol_w);
        tma_load_2d(dst + Ly::A, &tmX, k0 + ks * kBK, t0, &full[st], pol_x);
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer: D[row][token] += W[row][k] . X[token][k]
    if (lane == 0) {
      const uint32_t id = idesc_bf16_f32(kBM, BN, 0, 0);
      for (int ks = 0; ks < nk && ok; ++ks) {
        const int st = ks % kStages;
        ok = wait_bounded(&full[st], (ks / kStages) & 1, p.status);
        if (!ok) break;
        tc_fence_after();
        const uint32_t a = smem_u32(sm + st * Ly::STAGE), b = a + Ly::A;
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k)
          mma_bf16(tmem, smem_desc(a + k * 32, 16, 1024, kSw128), smem_desc(b + k * 32, 16, 1024, kSw128),
                   id, (ks | k) != 0);
        mma_commit(&freeb[st]);
      }
      mma_commit(done);
    }
    __syncwarp();
  }
  // ---- epilogue: thread = output row n0 + threadIdx.x; coalesced stores along n per token
  const bool any = nk > 0 && wait_bounded(done, 0, p.status);
  tc_fence_after();
  const int n = n0 + (int)threadIdx.x;
  float* out = p.out + (size_t)split * p.T * p.N;
  const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
#pragma unroll 1
  for (int c = 0; c < BN; c += 32) {
    float v[32];
    if (any) {
      tmem_ld32(lane_base + c, v);
      tmem_ld_wait();
    } else {
#pragma unroll
      for (int x = 0; x < 32; ++x) v[x] = 0.f;
    }
    if (n < p.N) {
#pragma unroll
      for (int x = 0; x < 32; ++x) {
        const int t = t0 + c + x;
        if (t < p.T) {
          if (p.out_bf16)
            p.out_bf16[(size_t)t * p.N + n] = __float2bfloat16_rn(v[x]);
          else
            out[(size_t)t * p.N + n] = v[x];
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, BN < 32 ? 32 : BN);
}

// ---------------------------------------------------------------- persistent, prompt-sized
// Y [T][N] in bf16 for large T (the prefill's k^C = W^{UK} c, v^C = W^{UV} c): one CTA per SM
// loops over 128 x 128 output tiles (row tile fastest, so neighbouring CTAs share an X tile in
// L2). The K stages stream through one ring across tiles; the MMA warp accumulates tile i into
// TMEM buffer i % 2 while the epilogue warps drain buffer (i - 1) % 2: thread = output feature,
// bf16 values staged in shared memory (128-byte swizzle, two staging tiles) and stored with TMA.
constexpr int kPStages = 4;
constexpr int kPBN = 128;
constexpr int kPStage = kBM * kBK * 2 + kPBN * kBK * 2;   // 32 KB
constexpr int kPStageOut = kPBN * kBM * 2;                // 32 KB: [128 tokens][128 features]
constexpr int kPBars = kPStages * kPStage + 2 * kPStageOut;
constexpr int kPSmem = kPBars + (2 * kPStages + 4) * 8 + 16 + 1024;

__global__ void __launch_bounds__(192, 1)
    gemm_persistent_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                           const __grid_constant__ CUtensorMap tmY, const GemmParams p) {
  extern __shared__ __align__(1024) uint8_t raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + kPBars);
  uint64_t* freeb = full + kPStages;
  uint64_t* acc_full = freeb + kPStages;   // [2]
  uint64_t* acc_empty = acc_full + 2;      // [2]
  uint32_t* slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tiles = (p.N + kBM - 1) / kBM, t_tiles = (p.T + kPBN - 1) / kPBN;
  const int tiles = n_tiles * t_tiles;
  const int nk = (p.K + kBK - 1) / kBK;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kPStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&freeb[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);   // the 4 epilogue warps
    }
    fence_mbarrier_init_cluster();
  }
  if (warp == 1) {
    tmem_alloc(slot, 2 * kPBN);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;
  griddep_launch_dependents();
  griddep_wait();
  if (warp == 0) {
    // ---- producer: W rows and X tokens of each K step, the two boxes from two lanes
    const uint64_t pol_w = policy_evict_normal();   // W is re-read by every token tile
    const uint64_t pol_x = policy_evict_normal();
    int it = 0;
    bool ok = true;
    for (int i = blockIdx.x; i < tiles && ok; i += gridDim.x) {
      const int n0 = (i % n_tiles) * kBM, t0 = (i / n_tiles) * kPBN;
      for (int ks = 0; ks < nk && ok; ++ks, ++it) {
        const int st = it % kPStages;
        bool r = true;
        if (lane == 0 && it >= kPStages) r = wait_bounded(&freeb[st], ((it / kPStages) - 1) & 1, p.status);
        ok = __shfl_sync(0xffffffffu, r, 0);
        if (!ok) break;
        if (lane == 0) mbar_arrive_expect_tx(&full[st], kPStage);
        __syncwarp();
        if (lane < 2) {
          uint8_t* dst = sm + st * kPStage + lane * (kBM * kBK * 2);
          tma_load_2d(dst, lane ? &tmX : &tmW, ks * kBK, lane ? t0 : n0, &full[st], lane ? pol_x : pol_w);
        }
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer: D[feature][token] of tile i in TMEM buffer i % 2
    if (lane == 0) {
      const uint32_t id = idesc_bf16_f32(kBM, kPBN, 0, 0);
      int it = 0, lt = 0;
      bool ok = true;
      for (int i = blockIdx.x; i < tiles && ok; i += gridDim.x, ++lt) {
        const int b = lt & 1;
        if (lt >= 2) ok = wait_bounded(&acc_empty[b], ((lt >> 1) - 1) & 1, p.status);
        if (!ok) break;
        tc_fence_after();
        for (int ks = 0; ks < nk && ok; ++ks, ++it) {
          const int st = it % kPStages;
          ok = wait_bounded(&full[st], (it / kPStages) & 1, p.status);
          if (!ok) break;
          tc_fence_after();
          const uint32_t a = smem_u32(sm + st * kPStage), bb = a + kBM * kBK * 2;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            mma_bf16(tmem + (uint32_t)b * kPBN, smem_desc(a + k * 32, 16, 1024, kSw128),
                     smem_desc(bb + k * 32, 16, 1024, kSw128), id, (ks | k) != 0);
          mma_commit(&freeb[st]);
        }
        if (ok) mma_commit(&acc_full[b]);
      }
    }
    __syncwarp();
  } else {
    // ---- epilogue: thread = feature row r of the tile (TMEM lane quadrant = warp % 4)
    const int qd = warp & 3, r = qd * 32 + lane, et = threadIdx.x - 64;   // et: 0..127
    const uint32_t lane_base = tmem + ((uint32_t)(qd * 32) << 16);
    int lt = 0;
    bool ok = true;
    for (int i = blockIdx.x; i < tiles && ok; i += gridDim.x, ++lt) {
      const int n0 = (i % n_tiles) * kBM, t0 = (i / n_tiles) * kPBN;
      const int b = lt & 1;
      if (lane == 0) ok = wait_bounded(&acc_full[b], (lt >> 1) & 1, p.status);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      // the staging tile of tile lt - 2 has been read by its TMA stores
      if (et == 0) bulk_wait_read_1();
      asm volatile("bar.sync 1, 128;" ::: "memory");
      uint8_t* stg = sm + kPStages * kPStage + b * kPStageOut;
      // staging: two boxes [128 tokens][64 features] (128-byte rows, 16-byte unit u of token t at
      // u ^ (t & 7)); feature r goes to box r / 64, unit (r % 64) / 8, element r % 8
      uint8_t* col = stg + (r >> 6) * (kPBN * 128) + ((r & 63) & 7) * 2;
      const uint32_t u = (uint32_t)((r & 63) >> 3);
#pragma unroll 1
      for (int c = 0; c < kPBN; c += 32) {
        float v[32];
        tmem_ld32(lane_base + (uint32_t)b * kPBN + c, v);
        tmem_ld_wait();
#pragma unroll
        for (int x = 0; x < 32; ++x) {
          const int t = c + x;
          *reinterpret_cast<__nv_bfloat16*>(col + t * 128 + ((u ^ (uint32_t)(t & 7)) << 4)) = __float2bfloat16_rn(v[x]);
        }
      }
      // TMEM buffer b may take the next tile
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[b]);
      fence_proxy_async_smem();
      asm volatile("bar.sync 1, 128;" ::: "memory");
      if (et == 0) {
        tma_store_2d(&tmY, stg, n0, t0);
        tma_store_2d(&tmY, stg + kPBN * 128, n0 + 64, t0);
        bulk_commit_group();
      }
    }
    if (et == 0) bulk_wait_all();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 2 * kPBN);
}

// Y[t][n] = sum over the splits, in split order; fp32 or bf16 out (with a row stride).
template <typename Out>
__global__ void __launch_bounds__(256) gemm_reduce_kernel(const float* __restrict__ part, int splits,
                                                          size_t count, Out* __restrict__ y) {
  griddep_wait();
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < count;
       i += (size_t)gridDim.x * blockDim.x) {
    float acc = 0.f;
    for (int s = 0; s < splits; ++s) acc += part[(size_t)s * count + i];
    st_act(y, i, acc);
  }
}

}  // namespace gemm

// How many ways K is split: enough (row, token) x split tiles to cover the SMs once, each
// split keeping at least 8 K steps.
int gemm_pick_splits(int T, int N, int K, int num_sms) {
  const int bn = T <= 64 ? 64 : 128;
  const int tiles = ((N + gemm::kBM - 1) / gemm::kBM) * ((T + bn - 1) / bn);
  const int steps = (K + gemm::kBK - 1) / gemm::kBK;
  int s = num_sms / (tiles > 0 ? tiles : 1);
  if (s > steps / 8) s = steps / 8;
  return s < 1 ? 1 : s;
}

// Partial-sum bytes launch_gemm needs for these sizes and output type.
size_t gemm_workspace_bytes(int T, int N, int K, int out_dtype, int num_sms) {
  const int s = gemm_pick_splits(T, N, K, num_sms);
  return s > 1 ? ((size_t)s * T * N * sizeof(float) + 255) / 256 * 256 : 0;
}

// Y = X . W^T: X [T][K] bf16, W [N][K] bf16, Y [T][N] of out_dtype (MLA_F32 or MLA_BF16).
// With splits > 1 (or a bf16 Y) the fp32 partials go to `part` ([splits][T][N]) and a second
// kernel sums them. K must be a multiple of 8 and both operands 16-byte aligned (TMA).
cudaError_t launch_gemm(const void* x, const void* w, int T, int N, int K, int splits, float* part,
                        void* y, int out_dtype, int32_t* status, cudaStream_t stream) {
  const int bn = T <= 64 ? 64 : 128;
  CUtensorMap tmW, tmX;
  {
    const uint64_t dims[2] = {(uint64_t)K, (uint64_t)N};
    const uint64_t st[1] = {(uint64_t)K * 2};
    const uint32_t box[2] = {gemm::kBK, gemm::kBM};
    if (!encode_bf16_map(&tmW, w, 2, dims, st, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[2] = {(uint64_t)K, (uint64_t)T};
    const uint64_t st[1] = {(uint64_t)K * 2};
    const uint32_t box[2] = {gemm::kBK, (uint32_t)bn};
    if (!encode_bf16_map(&tmX, x, 2, dims, st, box)) return cudaErrorInvalidValue;
  }
  const int steps = (K + gemm::kBK - 1) / gemm::kBK;
  gemm::GemmParams p;
  p.T = T;
  p.N = N;
  p.K = K;
  p.k_steps = (steps + splits - 1) / splits;
  p.status = status;
  const bool direct = splits == 1 && (out_dtype == MLA_F32 || out_dtype == MLA_BF16);
  p.out = direct && out_dtype == MLA_F32 ? static_cast<float*>(y) : part;
  p.out_bf16 = direct && out_dtype == MLA_BF16 ? static_cast<__nv_bfloat16*>(y) : nullptr;
  const bool reduce = !direct && out_dtype != kGemmPartials;
  if (direct && p.out_bf16 && T > 128) {
    // prompt-sized bf16 output: the persistent kernel, one CTA per SM
    CUtensorMap tmY;
    {
      const uint64_t dims[2] = {(uint64_t)N, (uint64_t)T};
      const uint64_t st[1] = {(uint64_t)N * 2};
      const uint32_t box[2] = {64, gemm::kPBN};
      if (!encode_bf16_map(&tmY, y, 2, dims, st, box)) return cudaErrorInvalidValue;
    }
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int tiles = ((N + gemm::kBM - 1) / gemm::kBM) * ((T + gemm::kPBN - 1) / gemm::kPBN);
    static std::atomic<bool> attr[kMaxDevices];
    cudaError_t e = set_smem_limit_once(gemm::gemm_persistent_kernel, gemm::kPSmem, attr);
    if (e == cudaSuccess)
      e = launch_programmatic(gemm::gemm_persistent_kernel, dim3(tiles < sms ? tiles : sms), dim3(192),
                              gemm::kPSmem, stream, tmW, tmX, tmY, p);
    return e == cudaSuccess ? cudaGetLastError() : e;
  }
  dim3 grid((N + gemm::kBM - 1) / gemm::kBM, (T + bn - 1) / bn, splits);
  cudaError_t e;
  if (bn == 64) {
    static std::atomic<bool> attr[kMaxDevices];
    e = set_smem_limit_once(gemm::gemm_kernel<64>, gemm::GLay<64>::SMEM, attr);
    if (e == cudaSuccess)
      e = launch_programmatic(gemm::gemm_kernel<64>, grid, dim3(128), gemm::GLay<64>::SMEM, stream, tmW, tmX, p);
  } else {
    static std::atomic<bool> attr[kMaxDevices];
    e = set_smem_limit_once(gemm::gemm_kernel<128>, gemm::GLay<128>::SMEM, attr);
    if (e == cudaSuccess)
      e = launch_programmatic(gemm::gemm_kernel<128>, grid, dim3(128), gemm::GLay<128>::SMEM, stream, tmW, tmX, p);
  }
  if (e != cudaSuccess) return e;
  if (!reduce) return cudaGetLastError();
  const size_t count = (size_t)T * N;
  const int blocks = (int)((count + 255) / 256 < 1184 ? (count + 255) / 256 : 1184);
  if (out_dtype == MLA_F32)
    e = launch_programmatic(gemm::gemm_reduce_kernel<float>, dim3(blocks), dim3(256), 0, stream,
                            (const float*)part, splits, count, static_cast<float*>(y));
  else
    e = launch_programmatic(gemm::gemm_reduce_kernel<__nv_bfloat16>, dim3(blocks), dim3(256), 0, stream,
                            (const float*)part, splits, count, static_cast<__nv_bfloat16*>(y));
  return e == cudaSuccess ? cudaGetLastError() : e;
}

}  // namespace mla
