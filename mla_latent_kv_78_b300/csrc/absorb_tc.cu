// K2 / K5 on tensor cores: query-side and output-side absorption for the V2 head shapes
// (d_h = 128, d_c = 512, d_h^R = 64, bf16), one CTA per (head, token tile).
//
// 「一文通透DeepSeek-V2」 §2.2.1 (last paragraph): W^{UK} is absorbed into the query side and
// W^{UV} into the output side. Per head i these are small GEMMs whose cost is reading the
// head's 128 KB weight block once:
//   absorb:   q_lat[t][i][0:512]  = q_c[t][i][:] . W_UK[i]      (D = q_c . W_UK[i] per half of
//             the latent columns: M = 128 tokens, N = 256, K = 128; W_UK[i] is the MN-major B
//             operand), q_lat[t][i][512:576] = RoPE_pos[t](q_r[t][i])
//   unabsorb: o[t][i][0:128]      = W_UV[i] . o_lat[t][i][:]    (D = W_UV[i] . o_lat^T: M = 128,
//             N = tokens, K = 512)
// Operands arrive by TMA (128-byte swizzle) and the MMAs are tcgen05 kind::f16 with fp32 TMEM
// accumulators. The absorb epilogue (TMEM lane = token) stages q_lat rows in shared memory for
// TMA stores; the unabsorb epilogue (TMEM lane = output column) stores straight from registers.
#include "mla_internal.cuh"
#include "tc_ptx.cuh"
#include "tma_host.cuh"

namespace mla {
namespace tca {

using namespace ptx;

constexpr int kD = 128, kC = 512, kR = 64;
constexpr long long kTimeout = 4000000000LL;

struct AbsorbParams {
  int T, H;
  const __nv_bfloat16* q_r;
  const int32_t* pos;
  __nv_bfloat16* q_lat;
  int32_t* status;
  // 1: launched right behind a cache append, which writes none of this kernel's inputs, so
  // they are read at once and the append is waited for only before exiting (a kernel that
  // waits for this grid then also finds the append complete); 0: every input is read after
  // the preceding kernel has completed
  int early_inputs;
  float theta_hi[kR / 2], theta_lo[kR / 2];   // RoPE frequencies base^(-2k/R) as hi + lo floats
};

struct UnabsorbParams {
  int T, H;
  float* o;
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

// ------------------------------------------------------------------ absorb
// D[token][c] = q_c[token] . W_UK[i][:, c] for one half (256) of the latent columns per CTA:
// M = 128 tokens (TMEM lane = token), N = 256, K = 128. A = q_c tile, 2 boxes [128 t x 64 d]
// (K-major); B = the half of W_UK[i] as 4 boxes [128 d x 64 c] (MN-major). Two CTAs per head
// (and two per SM) keep enough weight bytes in flight; the first also rotates q^R.
constexpr int kAbsNT = 128;
constexpr int kAbsSmem = 2 * 16384 + 4 * 16384 + 64 + 1024;

__global__ void __launch_bounds__(128, 2)
    absorb_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmQ,
                     const __grid_constant__ CUtensorMap tmL, const AbsorbParams p) {
  extern __shared__ __align__(1024) uint8_t raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = sm;                 // q_c
  uint8_t* sB = sm + 2 * 16384;     // this CTA's half of W_UK[i]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + 4 * 16384);   // [0] loads, [1] mma
  uint32_t* slot = reinterpret_cast<uint32_t*>(bars + 2);
  const int i = blockIdx.x, half = blockIdx.y, t0 = blockIdx.z * kAbsNT;
  const int nt = min(kAbsNT, p.T - t0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbarrier_init_cluster();
  }
  if (warp == 0) {
    tmem_alloc(slot, 256);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;
  const int t = warp * 32 + lane;   // this thread's token (TMEM lane) in the tile
  griddep_launch_dependents();   // the decode may start its set-up while this grid finishes
  // launched programmatically: the set-up above and the weight loads overlap the preceding
  // kernel (in a decode step, the cache append), which never writes W^{UK}; q_c, q^R and the
  // positions are read after that kernel has completed unless early_inputs says they may be
  // read at once, and this grid completes after that kernel either way.
  // The six boxes come from six lanes of warp 0: a warp's TMA loads issued by separate
  // instructions complete one after another on this part, those of one instruction overlap.
  const uint64_t pol = policy_evict_first();
  if (warp == 0) {
    if (lane == 0) mbar_arrive_expect_tx(&bars[0], 6 * 16384);
    __syncwarp();
    if (lane >= 2 && lane < 6)
      tma_load_2d(sB + (lane - 2) * 16384, &tmW, (4 * half + lane - 2) * 64, i * kD, &bars[0], pol);
  }
  if (!p.early_inputs) griddep_wait();
  if (warp == 0 && lane < 2) tma_load_3d(sA + lane * 16384, &tmQ, lane * 64, i, t0, &bars[0], pol);
  // the first half's CTA also rotates q^R while the operands land: two threads per token,
  // 16 RoPE pairs each, all four 16-byte loads issued before any is used
  const uint32_t rsw = (uint32_t)(t & 7);
  if (half == 0) {
    const int tt = threadIdx.x >> 1, part = threadIdx.x & 1;
    for (int tb = 0; tb < kAbsNT; tb += 64) {
      const int tok = tb + tt;
      if (tok >= nt) break;
      const size_t row = (size_t)(t0 + tok) * p.H + i;
      const uint4* src = reinterpret_cast<const uint4*>(p.q_r + row * kR) + part * 4;
      uint4* dst = reinterpret_cast<uint4*>(p.q_lat + row * (kC + kR) + kC) + part * 4;
      const int pos = p.pos[t0 + tok];
      uint4 x[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) x[q] = src[q];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t w[4] = {x[q].x, x[q].y, x[q].z, x[q].w};
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int k = (part * 4 + q) * 4 + e;
          float c, s;
          rope_cs(pos, p.theta_hi[k], p.theta_lo[k], &c, &s);
          const float x0 = __uint_as_float(w[e] << 16), x1 = __uint_as_float(w[e] & 0xFFFF0000u);
          o[e] = pack_bf16x2(x0 * c - x1 * s, x0 * s + x1 * c);
        }
        dst[q] = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
  }
  if (threadIdx.x == 0) {
    if (wait_bounded(&bars[0], 0, p.status)) {
      tc_fence_after();
      const uint32_t id = idesc_bf16_f32(128, 256, 0, 1);
      const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
      for (int kk = 0; kk < 8; ++kk) {
        const uint64_t a = smem_desc(a0 + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024, kSw128);
        const uint64_t b = smem_desc(b0 + kk * 2048, 16384, 1024, kSw128);
        mma_bf16(tmem, a, b, id, kk > 0);
      }
    }
    mma_commit(&bars[1]);
  }
  wait_bounded(&bars[1], 0, p.status);
  tc_fence_after();
  // The MMAs have read the W half's buffer: each thread writes its token's row of each
  // 64-column box into it (128-byte swizzle), and as soon as a box is complete one thread
  // sends it to q_lat with a TMA store (whole 128-byte row segments) while the next is staged.
  const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
#pragma unroll 1
  for (int cc = 0; cc < 256 / 64; ++cc) {
    float v[64];
    tmem_ld32(lane_base + cc * 64, v);
    tmem_ld32(lane_base + cc * 64 + 32, v + 32);
    tmem_ld_wait();
    uint8_t* rowp = sB + cc * 16384 + t * 128;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      *reinterpret_cast<uint4*>(rowp + ((uint32_t)q ^ rsw) * 16) =
          make_uint4(pack_bf16x2(v[8 * q], v[8 * q + 1]), pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                     pack_bf16x2(v[8 * q + 4], v[8 * q + 5]), pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (threadIdx.x == 0) {
      tma_store_3d(&tmL, sB + cc * 16384, half * 256 + cc * 64, i, t0);
      bulk_commit_group();
    }
  }
  tc_fence_before();
  if (threadIdx.x == 0) bulk_wait_read_all();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 256);
  if (p.early_inputs) griddep_wait();
}

// ------------------------------------------------------------------ unabsorb
// smem: A = W_UV[i] as 8 boxes [128 r x 64 c] (16 KB) | B = o_lat tile as 8 boxes [64 t x 64 c]
// (8 KB). Box pair j (64 latent columns) has its own barrier, so the MMAs of K-slice j start
// as soon as it lands while later slices are still in flight.
constexpr int kUnNT = 64;
constexpr int kUnSmem = 8 * 16384 + 8 * 8192 + 128 + 1024;

__global__ void __launch_bounds__(128, 1)
    unabsorb_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmO,
                       const UnabsorbParams p) {
  extern __shared__ __align__(1024) uint8_t raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = sm;
  uint8_t* sB = sm + 8 * 16384;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + 8 * 8192);   // [0..7] slices, [8] mma
  uint32_t* slot = reinterpret_cast<uint32_t*>(bars + 9);
  const int i = blockIdx.x, t0 = blockIdx.y * kUnNT;
  const int nt = min(kUnNT, p.T - t0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int j = 0; j < 9; ++j) mbar_init(&bars[j], 1);
    fence_mbarrier_init_cluster();
  }
  if (warp == 0) {
    tmem_alloc(slot, 64);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;
  // launched programmatically after the decode: the set-up above and the loads of W^{UV} (which
  // the decode never writes) overlap its tail; o_lat is read only once it has completed.
  // Slice j's two boxes from lane j of warp 0 (one instruction per box kind for all slices).
  const uint64_t pol = policy_evict_first();
  if (warp == 0 && lane < 8) {
    mbar_arrive_expect_tx(&bars[lane], 16384 + 8192);
    tma_load_2d(sA + lane * 16384, &tmW, lane * 64, i * kD, &bars[lane], pol);
  }
  griddep_wait();
  if (warp == 0 && lane < 8) tma_load_3d(sB + lane * 8192, &tmO, lane * 64, i, t0, &bars[lane], pol);
  __syncwarp();
  if (threadIdx.x == 0) {
    const uint32_t id = idesc_bf16_f32(128, kUnNT, 0, 0);
    const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
    for (int j = 0; j < 8; ++j) {
      if (!wait_bounded(&bars[j], 0, p.status)) break;
      tc_fence_after();
      for (int k = 0; k < 4; ++k) {
        const uint64_t a = smem_desc(a0 + j * 16384 + k * 32, 16, 1024, kSw128);
        const uint64_t b = smem_desc(b0 + j * 8192 + k * 32, 16, 1024, kSw128);
        mma_bf16(tmem, a, b, id, (j | k) != 0);
      }
    }
    mma_commit(&bars[8]);
  }
  wait_bounded(&bars[8], 0, p.status);
  tc_fence_after();
  const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
  const int r = warp * 32 + lane;
  float v[kUnNT];
  tmem_ld32(lane_base, v);
  tmem_ld32(lane_base + 32, v + 32);
  tmem_ld_wait();
#pragma unroll
  for (int t = 0; t < kUnNT; ++t)
    if (t < nt) p.o[((size_t)(t0 + t) * p.H + i) * kD + r] = v[t];
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 64);
}

}  // namespace tca

bool absorb_tc_supported(const Dims& d) {
  return d.act_dtype == MLA_BF16 && d.D == tca::kD && d.C == tca::kC && d.R == tca::kR;
}

cudaError_t launch_absorb_tc(const Dims& d, const void* q_c, const void* q_r, const int32_t* pos,
                             int T, const void* w_uk, void* q_lat, cudaStream_t stream,
                             bool early_inputs) {
  CUtensorMap tmW, tmQ, tmL;
  {
    const uint64_t dims[2] = {(uint64_t)tca::kC, (uint64_t)d.H * tca::kD};
    const uint64_t st[1] = {(uint64_t)tca::kC * 2};
    const uint32_t box[2] = {64, 128};
    if (!encode_bf16_map(&tmW, w_uk, 2, dims, st, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[3] = {(uint64_t)(tca::kC + tca::kR), (uint64_t)d.H, (uint64_t)T};
    const uint64_t st[2] = {(uint64_t)(tca::kC + tca::kR) * 2, (uint64_t)d.H * (tca::kC + tca::kR) * 2};
    const uint32_t box[3] = {64, 1, tca::kAbsNT};
    if (!encode_bf16_map(&tmL, q_lat, 3, dims, st, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[3] = {(uint64_t)tca::kD, (uint64_t)d.H, (uint64_t)T};
    const uint64_t st[2] = {(uint64_t)tca::kD * 2, (uint64_t)d.H * tca::kD * 2};
    const uint32_t box[3] = {64, 1, tca::kAbsNT};
    if (!encode_bf16_map(&tmQ, q_c, 3, dims, st, box)) return cudaErrorInvalidValue;
  }
  tca::AbsorbParams p;
  p.T = T;
  p.H = d.H;
  p.q_r = static_cast<const __nv_bfloat16*>(q_r);
  p.pos = pos;
  p.q_lat = static_cast<__nv_bfloat16*>(q_lat);
  p.status = nullptr;
  p.early_inputs = early_inputs ? 1 : 0;
  for (int k = 0; k < tca::kR / 2; ++k) {
    const double th = rope_theta_host(d, k);
    p.theta_hi[k] = (float)th;
    p.theta_lo[k] = (float)(th - (double)p.theta_hi[k]);
  }
  static std::atomic<bool> attr[kMaxDevices];
  {
    cudaError_t e = set_smem_limit_once(tca::absorb_tc_kernel, tca::kAbsSmem, attr);
    if (e != cudaSuccess) return e;
  }
  dim3 grid(d.H, 2, (T + tca::kAbsNT - 1) / tca::kAbsNT);
  cudaError_t e = launch_programmatic(tca::absorb_tc_kernel, grid, dim3(128), tca::kAbsSmem, stream,
                                      tmW, tmQ, tmL, p);
  return e == cudaSuccess ? cudaGetLastError() : e;
}

cudaError_t launch_unabsorb_tc(const Dims& d, const void* o_lat, int T, const void* w_uv, float* o,
                               cudaStream_t stream) {
  CUtensorMap tmW, tmO;
  {
    const uint64_t dims[2] = {(uint64_t)tca::kC, (uint64_t)d.H * tca::kD};
    const uint64_t st[1] = {(uint64_t)tca::kC * 2};
    const uint32_t box[2] = {64, 128};
    if (!encode_bf16_map(&tmW, w_uv, 2, dims, st, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[3] = {(uint64_t)tca::kC, (uint64_t)d.H, (uint64_t)T};
    const uint64_t st[2] = {(uint64_t)tca::kC * 2, (uint64_t)d.H * tca::kC * 2};
    const uint32_t box[3] = {64, 1, tca::kUnNT};
    if (!encode_bf16_map(&tmO, o_lat, 3, dims, st, box)) return cudaErrorInvalidValue;
  }
  tca::UnabsorbParams p;
  p.T = T;
  p.H = d.H;
  p.o = o;
  p.status = nullptr;
  static std::atomic<bool> attr[kMaxDevices];
  {
    cudaError_t e = set_smem_limit_once(tca::unabsorb_tc_kernel, tca::kUnSmem, attr);
    if (e != cudaSuccess) return e;
  }
  dim3 grid(d.H, (T + tca::kUnNT - 1) / tca::kUnNT);
  cudaError_t e = launch_programmatic(tca::unabsorb_tc_kernel, grid, dim3(128), tca::kUnSmem, stream,
                                      tmW, tmO, p);
  return e == cudaSuccess ? cudaGetLastError() : e;
}

}  // namespace mla
