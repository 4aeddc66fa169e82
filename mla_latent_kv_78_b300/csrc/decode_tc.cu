// Tensor-core MLA decode (tcgen05 / TMEM / TMA) for DeepSeek-V2 head shapes:
// n_h = 128 heads, d_c = 512, d_h^R = 64, page size 64, bf16 latent cache.
//
// What it computes (「deepseek(2)——deepseek 關鍵技術」 §1, absorbed form of
// 「一文通透DeepSeek-V2」 §2.2.1-2.2.2): for one query row of one sequence,
//   s[n][h] = q_lat[h] . [c_n ; k^R_n] * scale,   o_lat[h] = sum_n softmax_n(s[:, h]) c_n,
// with all 128 heads sharing the 576-d latent key of each cached token.
//
// Design (B300-first; no design on the pages is followed):
//  * A CTA pair (cluster of 2) owns one (sequence, query row, split). Tiles are 256
//    tokens = 4 pages. Scores are computed transposed, S^T[token][head] = K . Q^T, with a
//    2-SM MMA (cta_group::2, M = 256 tokens, N = 128 heads): each CTA supplies its 128
//    tokens' 576-d keys and HALF of Q (its 64 heads), and every MMA runs at full rate
//    (N = 128). With a bf16 cache the Q half is not resident: each [128 tokens x 64 dims]
//    key chunk has its matching [64 heads x 64 dims] Q chunk (an L2 hit after the first
//    tile) streamed through a 3-slot ring that trails the 4-deep key ring by one step, which
//    leaves shared memory for a 4-deep latent ring and two P^T buffers.
//  * The output is accumulated transposed, O^T[d_c][head] = V^T . P^T, again 2-SM
//    (M = 256 latent rows per MMA, two MMAs per K step): each CTA holds half of O^T,
//    256 TMEM columns, which leaves room for a double-buffered S^T (2 x 128 columns).
//  * P^T is split by head: the CTA that computed a token's scores keeps its own head half and
//    stores the other half (16 KB per tile) straight into the peer's shared memory (st.async),
//    with the tile's per-head maxima when it publishes them. Both CTAs take identical
//    online-softmax decisions from the same data: the reference maximum of a head moves only
//    when a tile's published maximum exceeds it by more than 2^8, two tiles later, so the
//    common tile needs no cross-thread reduction. A unit in which a weight ran beyond the
//    range this lag leaves (2^96) is computed again with the exact maxima, so the result is
//    exact for any spread of scores.
//  * The key tile is read from HBM once, as [128 tokens x 64 dims] chunks for S^T; the
//    latent part is read a second time, about a tile later, as [32 tokens x 256 d_c]
//    chunks for O^T, normally from L2.
//  * Two threads issue MMAs: one thread cannot issue 2-SM MMAs as fast as the tensor pipe
//    retires them (~85 cycles per instruction against 64), two can.
//  * Warp roles: w0 key-chunk TMA producer (+Q), w1 S^T issuer (even CTA) + TMEM owner,
//    w2 latent-chunk producer (+ zeroing of rows past the range on the last tile),
//    w3 P^T relay, w4..w11 softmax / epilogue (thread = TMEM lane; warps 4-7 heads 0-63,
//    8-11 heads 64-127), w12 P.V issuer (even CTA); FP8 cache: w13..w15 convert the codes.
//  * Every wait is bounded; a timeout sets MLA_DEV_TIMEOUT and every role winds down.
#include <math_constants.h>
#include <string.h>

#include "mla_internal.cuh"
#include "tc_ptx.cuh"

namespace mla {
namespace tc {

using namespace ptx;

constexpr int kH = 128, kC = 512, kR = 64, kCR = 576, kP = 64;
constexpr int kTile = 256;           // tokens per tile (4 pages)
constexpr int kKCh = kCR / 64;       // 9 dim chunks per tile
constexpr int kVCh = kTile / 32;     // 8 latent chunks per tile
constexpr int kPvWarp = 12;             // the P.V issuer
constexpr int kCvtWarp0 = 13;           // FP8 cache: warps 13-15 convert codes to bf16 tiles
constexpr long long kTimeout = 4000000000LL;   // clock cycles (~2 s)
constexpr int kXSlots = 4;    // slots for the peer's published tile maxima: tile t uses t % 4
// Bytes the peer stores into this CTA's shared memory per tile (st.async, counted on
// p_landed): its 128 token rows of this CTA's head half of P^T, and its per-head tile maxima.
constexpr uint32_t kXBytes = 128 * 128 + kH * 4;
constexpr float kLazy = 8.f;    // log2 units a score may exceed the reference before it moves
// Weights above 2^kRange relative to the lagging reference are clamped (P and the fp32 sums
// would otherwise run out of range); a unit in which that happened runs again exactly (two
// more passes: the exact per-head maxima, then the softmax with them as the reference).
constexpr float kRange = 96.f;
constexpr int kRawS = 8192 + 2048;   // FP8 key chunk: [128 tok x 64 codes] + [128 tok x 4 scales]
constexpr int kRawV = 8192 + 512;    // FP8 latent chunk: 4 x [32 tok x 64 codes] + [32 tok x 4 scales]

constexpr int F_COL = 0;       // [8 warps][64]   column max / column sum partials
constexpr int F_CMLOC = 512;   // [2][128] this CTA's published per-head tile maxima
constexpr int F_RCV = 768;     // [4][128] the peer's per-head tile maxima by slot (-inf: none)
constexpr int F_M = F_RCV + kXSlots * kH;   // [128] reference (log2 units), same in both CTAs
constexpr int F_ALPHA = F_M + 128;   // [128]
constexpr int F_LLOC = F_ALPHA + 128;  // [128]
constexpr int F_LRCV = F_LLOC + 128;   // [128]
constexpr int F_INV = F_LRCV + 128;    // [128]
constexpr int F_X0 = F_INV + 128;     // [128] the peer's tile-0 per-head maxima
constexpr int F_FLAG = F_X0 + 128;    // ints, see FL_*
constexpr int FL_RESCALE = 0;  // [2] by tile parity: the reference moved for this tile
constexpr int FL_ABORT = 2;    // a bounded wait gave up
constexpr int FL_PUB = 3;      // [2] by tile parity: this CTA published the tile's maxima
constexpr int FL_TICKET = 5;   // FP8 converters: the next job allowed to acquire its slots
constexpr int FL_CLAMP = 6;    // this pass clamped a weight of this CTA's tokens (see kRange)
constexpr int FL_REPLAY = 7;   // the unit runs again exactly (set in both CTAs alike)
constexpr int FL_PEER_CLAMP = 8;   // the peer's FL_CLAMP, received with its epilogue sums
constexpr int FL_PEER_ABORT = 9;   // the peer's FL_ABORT at the end of a pass
constexpr int F_FLAGS_END = F_FLAG + 10;
constexpr int F_SQ = F_FLAGS_END;    // [128 heads][4] FP8 scores: query group scales (both CTAs')
// bf16: [128] the rescale factors of odd tiles (even tiles' at F_ALPHA): the relay warp folds a
// tile's column sums of P into the running sums after the softmax has moved on to later tiles
constexpr int F_ALPHA_ODD = F_FLAGS_END;
// end of the fp32 scratch (even: the barriers that follow need 8-byte alignment); only the FP8
// instantiations keep the query group scales, only the bf16 one the odd tiles' factors
template <bool F8>
constexpr int F_END = F8 ? F_SQ + 4 * kH : F_ALPHA_ODD + kH;
// Shared-memory layout. bf16 cache: keys and latents arrive by TMA in their MMA layout.
// FP8 cache: raw codes and scales arrive by TMA in staging rings (RS, RV slots) and the
// converter warps write bf16 operand tiles into the S and V rings.
template <bool F8>
struct Lay {
  // bf16: Q is streamed, chunk by chunk, next to the key chunks (a [64 heads x 64 dims] box
  // read from L2 per [128 tokens x 64 dims] key box), which frees 72 KB for deeper rings and
  // two P^T buffers; its own NQ-slot ring (NQ <= NS) trails the key ring by NS - NQ chunks,
  // so a Q slot is always free once the key slot of the same producer step is, and each Q
  // chunk is requested NQ steps before its MMAs. FP8: Q stays resident.
  static constexpr bool QRES = F8;
  static constexpr int SSTAGE = 16384;      // S-phase stage bytes (key chunk)
  static constexpr int NS = F8 ? 2 : 4;     // S-phase ring
  static constexpr int NQ = F8 ? 0 : 3;     // streamed Q chunks (bf16) [64 heads x 64 dims]
  static constexpr int NV = F8 ? 2 : 4;     // V-phase ring: [32 tok x 256 d_c] 16-bit = 16 KB
  static constexpr int PB = F8 ? 1 : 2;     // P^T buffers [256 tok x 64 heads] = 32 KB each
  static constexpr int RS = F8 ? 3 : 0;     // raw key-chunk slots (kRawS bytes)
  static constexpr int RV = F8 ? 2 : 0;     // raw latent-chunk slots (kRawV bytes)
  static constexpr int THREADS = F8 ? 512 : 416;
  static constexpr int OFF_Q = 0;                        // 9 x [64 heads x 64 dims] (8 KB each)
  static constexpr int OFF_S = OFF_Q + (QRES ? kKCh * 8192 : 0);
  static constexpr int OFF_QS = OFF_S + NS * SSTAGE;
  static constexpr int OFF_V = OFF_QS + NQ * 8192;
  static constexpr int OFF_P = OFF_V + NV * 16384;
  static constexpr int OFF_RS = OFF_P + PB * 32768;
  static constexpr int OFF_RV = OFF_RS + RS * kRawS;
  static constexpr int OFF_F = OFF_RV + RV * kRawV;      // fp32 scratch
  static constexpr int OFF_BAR = OFF_F + F_END<F8> * 4;
};

template <bool F8>
struct BarsT {
  static constexpr int NS = Lay<F8>::NS, NV = Lay<F8>::NV;
  static constexpr int RS = Lay<F8>::RS > 0 ? Lay<F8>::RS : 1;
  static constexpr int RV = Lay<F8>::RV > 0 ? Lay<F8>::RV : 1;
  uint64_t q_ready;
  uint64_t q_conv;       // FP8: both CTAs' resident Q halves have landed (even CTA, 2 arrivals)
  uint64_t s_ready[NS], s_free[NS];
  uint64_t qs_ready[Lay<F8>::NQ > 0 ? Lay<F8>::NQ : 1];  // bf16: streamed Q chunks (even CTA)
  uint64_t v_landed[NV], v_ready[NV], v_free[NV];
  uint64_t rs_ready[RS], rs_free[RS], rv_ready[RV], rv_free[RV];
  uint64_t s_full[2], s_empty[2];
  uint64_t p_landed[2], p_ready[2], o_done[2];
  uint64_t l_done[2];    // bf16: the relay has folded the tile's column sums of P in
  uint64_t gs_ready[2], gs_free[2];   // FP8 scores: latent code groups (even CTA / both)
  uint64_t q8_done;      // FP8 scores: Q quantised (the group ring may overwrite its bf16 rows)
  uint64_t sq_ready;     // FP8 scores: the peer's query group scales have landed
  uint64_t x0_ready;     // the peer's tile-0 maxima have landed
  uint64_t l_landed;
  uint64_t teardown;
  uint32_t tmem_base;
};
template <bool F8>
constexpr int kSmemBytes = Lay<F8>::OFF_BAR + (int)sizeof(BarsT<F8>) + 1024;   // + alignment slack
static_assert(kSmemBytes<false> <= 232448 && kSmemBytes<true> <= 232448, "shared memory");
static_assert(Lay<false>::OFF_BAR % 8 == 0 && Lay<true>::OFF_BAR % 8 == 0, "mbarrier alignment");

// Tensor maps of one launch (bf16 cache: q, k, v; FP8 cache: q and the raw maps).
struct Maps {
  CUtensorMap q;     // q_lat rows of 576 bf16, box 64 x 64, 128-byte swizzle
  CUtensorMap k;     // bf16 pool rows, box 64 x 64, swizzled
  CUtensorMap v;     // bf16 pool rows, box 64 x 32, swizzled
  CUtensorMap cs;    // FP8 pool rows of 656 bytes, box 64 B x 64 rows
  CUtensorMap cv;    // box 64 B x 32 rows
  CUtensorMap ss;    // box 16 B x 64 rows (the 4 scales of a token)
  CUtensorMap sv;    // box 16 B x 32 rows
  CUtensorMap kr;    // box 128 B x 64 rows (bf16 RoPE keys)
  CUtensorMap c8;    // box 128 B x 64 rows, 128-byte swizzle: one latent group's codes as an
                     // FP8 MMA operand (FP8 scores)
};

struct Params {
  long long wait_limit;   // clock cycles a bounded wait gives up after
  int withhold;           // test hook: latent chunk the even CTA never loads (-1: none)
  const int32_t* bt;
  const int32_t* order;    // rows by decreasing visible length (nullptr: launch order)
  const uint8_t* pool;     // FP8 scores: the key scales are read from the entries
  int q8;                  // FP8 scores (MLA_KERNEL_TC_FP8_SCORES)
  int maxp, num_pages;
  const int32_t* seq_lens;
  int B, n_q, max_seq_len, S;
  int tail;                // rows of the plan's tail run as two half-range units each (S == 1)
  float scale_log2;
  __nv_bfloat16* o_lat;
  float* lse;
  float* ws_o;
  float* ws_lse;
  int32_t* status;
#ifdef MLA_TC_TRACE
  unsigned long long* trace;
#endif
};

struct Ctx {
  volatile int* abort_flag;
  int32_t* status;
  long long limit;   // clock cycles
};

#ifdef MLA_TC_TRACE
// Debug builds only: per-event %globaltimer stamps for the first kTraceUnits units.
constexpr int kTraceUnits = 2, kTraceEvents = 24, kTraceTiles = 1024;
static void* g_tc_trace_host = nullptr;
__device__ __forceinline__ void trace(unsigned long long* buf, int unit, uint32_t rank, int ev,
                                      int t) {
  if (buf && unit < kTraceUnits && t < kTraceTiles) {
    unsigned long long ns;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(ns));
    buf[(((size_t)unit * 2 + rank) * kTraceEvents + ev) * kTraceTiles + t] = ns;
  }
}
#ifdef MLA_TC_PROF_ONLY
#define TRACE(ev, t) ((void)0)
#else
#define TRACE(ev, t) trace(prm.trace, unit, rank, ev, t)
#endif
// cycle totals of one thread's activities (slot < 8), stored at the end of event row 15
#define PROF(slot, stmt)                    \
  do {                                      \
    const long long p0_ = clock64();        \
    stmt;                                   \
    prof[slot] += clock64() - p0_;          \
  } while (0)
#define PROF_STORE(base)                                                                   \
  do {                                                                                      \
    if (prm.trace && unit < kTraceUnits)                                                    \
      for (int q = 0; q < 8; ++q)                                                           \
        prm.trace[(((size_t)unit * 2 + rank) * kTraceEvents + 15) * kTraceTiles + (base) + q] = \
            (unsigned long long)prof[q];                                                    \
  } while (0)
#else
#define TRACE(ev, t) ((void)0)
#define PROF(slot, stmt) stmt
#define PROF_STORE(base) ((void)0)
#endif

// One bf16 weight -> fp32, exactly.
__device__ __forceinline__ float p16_to_f32(uint32_t h) { return __uint_as_float(h << 16); }
// lo += low bf16 of w, hi += high bf16 of w, each an fp32 add of the exact bf16 value
__device__ __forceinline__ void add_bf16x2_f32(float& lo, float& hi, uint32_t w) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tadd.rn.f32.bf16 %0, l, %0;\n\tadd.rn.f32.bf16 %1, h, %1;\n\t}"
      : "+f"(lo), "+f"(hi)
      : "r"(w));
}

// Sum over the warp's 32 lanes of each of 32 values per lane; lane j returns the sum of
// value j. Halving exchange: at each step a lane keeps one half of its values, sends the
// other half to its partner and adds what it receives (31 shuffles in all).
// Lane j gets the maximum over the warp's lanes of v[j] (a transposing butterfly: 31
// shuffles for the 32 columns instead of 5 per column). Exact: max does not round.
__device__ __forceinline__ float warp_transpose_max32(float (&v)[32], int lane) {
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const bool hi = (lane & w) != 0;
#pragma unroll
    for (int q = 0; q < w; ++q) {
      const float keep = hi ? v[q + w] : v[q];
      const float send = hi ? v[q] : v[q + w];
      v[q] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, w));
    }
  }
  return v[0];
}

__device__ __forceinline__ float warp_transpose_sum32(float (&v)[32], int lane) {
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const bool hi = (lane & w) != 0;
#pragma unroll
    for (int q = 0; q < w; ++q) {
      const float keep = hi ? v[q + w] : v[q];
      const float send = hi ? v[q] : v[q + w];
      v[q] = keep + __shfl_xor_sync(0xffffffffu, send, w);
    }
  }
  return v[0];
}

// Bounded wait by one thread, polling (a suspended thread resumed measurably later than a
// polling one). kCluster: the arrivals carry data written by the other CTA's threads, so the
// acquire is at cluster scope; otherwise at CTA scope.
template <bool kCluster = false>
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, const Ctx& cx) {
  const uint32_t a = smem_u32(bar);
  auto test = [&]() { return kCluster ? mbar_test_cluster(a, parity) : mbar_test_cta(a, parity); };
  if (test()) return true;
  const long long t0 = clock64();
  while (true) {
    if (*cx.abort_flag) return false;
    if (test()) return true;
    if (clock64() - t0 > cx.limit) {
      *cx.abort_flag = 1;
      flag_status(cx.status, MLA_DEV_TIMEOUT);
      return false;
    }
  }
}

// Wait ignoring the abort flag (used while draining before exit), still bounded.
__device__ __forceinline__ void wait_drain(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const long long t0 = clock64();
  while (!mbar_try_wait(a, parity)) {
    if (clock64() - t0 > kTimeout) return;
  }
}

__device__ __forceinline__ void arrive_even(uint64_t* bar, uint32_t rank) {
  if (rank == 0)
    mbar_arrive(bar);
  else
    mbar_arrive_remote(mapa(smem_u32(bar), 0));
}

// Barrier set-up of one pass (one thread of each CTA).
template <bool F8>
__device__ __forceinline__ void init_barriers(BarsT<F8>* bars) {
  constexpr int kNS = Lay<F8>::NS, kNV = Lay<F8>::NV;
  using Ly = Lay<F8>;
    // *_ready live in the even CTA: one arrival (its producer registers both CTAs' bytes)
    // plus the bytes of both CTAs' loads, which signal it directly
    // (FP8 cache: each CTA's converter warps arrive once on the even CTA's s_ready / v_ready
    // after writing their f16 tile; the raw staging rings are CTA-local)
    mbar_init(&bars->q_ready, 1);
    mbar_init(&bars->q_conv, 2);
    for (int s = 0; s < kNS; ++s) {
      mbar_init(&bars->s_ready[s], F8 ? 2 : 1);
      mbar_init(&bars->s_free[s], 1);
    }
    for (int s = 0; s < Ly::NQ; ++s) mbar_init(&bars->qs_ready[s], 1);
    for (int s = 0; s < kNV; ++s) {
      mbar_init(&bars->v_landed[s], 1);
      mbar_init(&bars->v_ready[s], F8 ? 2 : 1);
      mbar_init(&bars->v_free[s], 1);
    }
    for (int s = 0; s < Ly::RS; ++s) {
      mbar_init(&bars->rs_ready[s], 1);
      mbar_init(&bars->rs_free[s], 1);
    }
    for (int s = 0; s < Ly::RV; ++s) {
      mbar_init(&bars->rv_ready[s], 1);
      mbar_init(&bars->rv_free[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->s_full[s], 1);
      mbar_init(&bars->s_empty[s], 16);
      mbar_init(&bars->p_landed[s], 8);
      mbar_init(&bars->p_ready[s], 2);
      mbar_init(&bars->l_done[s], 1);
      mbar_init(&bars->o_done[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->gs_ready[s], 1);
      mbar_init(&bars->gs_free[s], 1);
    }
    mbar_init(&bars->q8_done, 1);
    mbar_init(&bars->sq_ready, 1);
    mbar_init(&bars->x0_ready, 1);
    mbar_init(&bars->l_landed, 1);
    mbar_init(&bars->teardown, 2);   // both issuing threads' last commits
    fence_mbarrier_init_cluster();
}

// One pass over this pair's unit. mode 0 is the ordinary pass; modes 1 and 2 run only when
// mode 0 had to clamp a weight (see kRange): 1 computes the scores alone, for the exact
// per-head maxima, 2 is the ordinary pass with those maxima as the reference.
// Q8: the FP8 cache with the scores on FP8 tensor cores (MLA_KERNEL_TC_FP8_SCORES).
template <bool F8, bool Q8 = false>
__device__ __forceinline__ void decode_pass(const Maps& maps, const Params& prm, uint8_t* sm, const int mode) {
  using Ly = Lay<F8>;
  using Bars = BarsT<F8>;
  constexpr int kNS = Ly::NS, kNV = Ly::NV, kThreads = Ly::THREADS;
  constexpr int OFF_Q = Ly::OFF_Q, OFF_S = Ly::OFF_S, OFF_V = Ly::OFF_V, OFF_P = Ly::OFF_P;
  constexpr int kSStage = Ly::SSTAGE, kPB = Ly::PB;
  constexpr int OFF_F = Ly::OFF_F, OFF_BAR = Ly::OFF_BAR;
  const CUtensorMap& tmQ = maps.q;
  const CUtensorMap& tmK = maps.k;
  const CUtensorMap& tmV = maps.v;
  float* fs = reinterpret_cast<float*>(sm + OFF_F);
  int* flags = reinterpret_cast<int*>(fs + F_FLAG);
  Bars* bars = reinterpret_cast<Bars*>(sm + OFF_BAR);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;

  // ---- which (sequence, query row, split) this pair owns
  const int unit = blockIdx.x >> 1;
  // row = b * n_q + j; with more rows than CTA pairs the longest rows go first (see
  // plan_order_kernel), and the last `tail` rows of the plan each run as two units (split 0 and
  // 1 of 2) whose partials sit at the row's place in the tail. Head h's result goes to entry
  // obase + h * ostride of o_lat / lse rows (ostride 1) or of the partials (ostride = splits).
  int row, split, nsplit, obase, ostride;
  {
    const int rows = prm.B * prm.n_q;
    int prow;
    if (prm.tail > 0 && unit >= rows - prm.tail) {
      const int k = unit - (rows - prm.tail);
      prow = k >> 1;
      split = k & 1;
      nsplit = 2;
      row = __ldg(prm.order + rows - prm.tail + prow);
    } else {
      split = unit % prm.S;
      nsplit = prm.S;
      row = prm.order ? __ldg(prm.order + unit / prm.S) : unit / prm.S;
      prow = row;
    }
    obase = nsplit == 1 ? row * kH : prow * kH * nsplit + split;
    ostride = nsplit;
  }
  const int b = row / prm.n_q, j = row % prm.n_q;
  Ctx cx{reinterpret_cast<volatile int*>(&flags[FL_ABORT]), prm.status, prm.wait_limit};
  const uint32_t tmem = bars->tmem_base;
  const int L = prm.seq_lens[b];
  const bool bad_len = (L < prm.n_q || L > prm.max_seq_len);
  const int visible = bad_len ? 0 : L - prm.n_q + j + 1;
  int chunk = (visible + nsplit - 1) / nsplit;
  chunk = (chunk + kTile - 1) / kTile * kTile;
  const int lo = min(visible, split * chunk);
  const int hi = min(visible, lo + chunk);
  const int nt = (hi - lo + kTile - 1) / kTile;
  const int valid_pages = (hi + kP - 1) / kP;   // pages holding tokens < hi

  // Page ids of this unit's range, read by a whole producer warp 32 pages at a time (lane j
  // holds page 32*batch + j of the range) one batch ahead of use, so no TMA issue waits on a
  // block-table load. Pages past the range, or with an id outside the pool (flagged), map to
  // the row one past the pool, which TMA fills with zeros.
  auto fetch_pid = [&](int batch) -> int {
    const int pidx = lo / kP + batch * 32 + lane;
    if (pidx >= valid_pages) return -1;
    const int pg = __ldg(prm.bt + (size_t)b * prm.maxp + pidx);
    if (pg < 0 || pg >= prm.num_pages) {
      flag_status(prm.status, MLA_DEV_INDEX_OUT_OF_RANGE);
      return -1;
    }
    return pg;
  };
  int pid_batch = 0, pid_cur = 0, pid_next = 0;
  // first row of page idx_in_unit (warp-uniform, non-decreasing across calls)
  auto page_y = [&](int idx_in_unit) -> int {
    while ((idx_in_unit >> 5) > pid_batch) {
      ++pid_batch;
      pid_cur = pid_next;
      pid_next = fetch_pid(pid_batch + 1);
    }
    const int pg = __shfl_sync(0xffffffffu, pid_cur, idx_in_unit & 31);
    return pg < 0 ? prm.num_pages * kP : pg * kP;
  };

  if (nt == 0) {
    // nothing visible in this range: zero output, lse = -inf
    if (bad_len && tid == 0 && rank == 0 && split == 0) flag_status(prm.status, MLA_DEV_BAD_SEQLEN);
    for (int idx = tid; idx < kH * 256; idx += kThreads) {
      const int h = idx >> 8, q = idx & 255;
      const int dc = (q >> 7) * 256 + rank * 128 + (q & 127);
      const size_t o = (size_t)obase + (size_t)h * ostride;
      if (ostride == 1)
        prm.o_lat[o * kC + dc] = __float2bfloat16_rn(0.f);
      else
        prm.ws_o[o * kC + dc] = 0.f;
    }
    if (rank == 0 && tid < kH) {
      const size_t o = (size_t)obase + (size_t)tid * ostride;
      if (ostride == 1) {
        if (prm.lse) prm.lse[o] = -CUDART_INF_F;
      } else {
        prm.ws_lse[o] = -CUDART_INF_F;
      }
    }
  } else if (warp == 0) {
    // ================================================================ TMA producer
    // Q once, then every tile's key chunks in order (lane 0 issues; the warp keeps page ids)
    pid_cur = fetch_pid(0);
    pid_next = fetch_pid(1);
    const bool leader = lane == 0;
    const uint64_t pol_s = policy_evict_normal();  // re-read soon for the V phase
    const bool even = rank == 0;
    auto at_even = [&](uint64_t* bar) { return mapa(smem_u32(bar), 0); };
    if (leader) {
      prefetch_tensormap(&tmQ);
      if constexpr (F8) {
        prefetch_tensormap(&maps.cs);
        prefetch_tensormap(&maps.ss);
        prefetch_tensormap(&maps.kr);
        prefetch_tensormap(&maps.cv);
        prefetch_tensormap(&maps.sv);
        // each CTA's resident Q half: a CTA-local barrier, relayed to the even CTA's q_conv
        mbar_arrive_expect_tx(&bars->q_ready, kKCh * 8192);
      } else {
        prefetch_tensormap(&tmK);
        prefetch_tensormap(&tmV);
      }
    }
    if constexpr (F8) {
      // one box per lane: TMA loads issued by one thread complete one after another, which
      // the FP8 cache's many small boxes (codes, scales, RoPE keys) feel most
      __syncwarp();
      if (lane < kKCh)
        tma_load_2d(sm + OFF_Q + lane * 8192, &tmQ, lane * 64, row * kH + (int)rank * 64, &bars->q_ready,
                    policy_evict_last());
    }
    int s_cnt = 0;
#ifdef MLA_TC_TRACE
    long long prof[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    const long long prof_start = clock64();
#endif
    const uint64_t pol_q = policy_evict_last();   // Q chunks are read again every tile
    // Q chunk of S-phase step m into slot m % NQ. Issued after the key chunk of step
    // m + NS - NQ, whose slot was free only once the MMAs of step m - NQ completed, the last
    // of them reading the slot's previous Q.
    constexpr int kNQ = Ly::NQ;
    static_assert(F8 || (kNQ >= 1 && kNQ <= kNS), "Q ring deeper than the key ring");
    constexpr int kLag = kNS - kNQ;
    auto load_q_chunk = [&](int m) {
      const int qs = m % (kNQ > 0 ? kNQ : 1);
      if (even) mbar_arrive_expect_tx(&bars->qs_ready[qs], 2 * 8192);
      tma_load_2d_pair(sm + Ly::OFF_QS + qs * 8192, &tmQ, (m % kKCh) * 64, row * kH + (int)rank * 64,
                       at_even(&bars->qs_ready[qs]), pol_q);
    };
    auto load_s_chunk = [&](int c, int y0, int y1) -> bool {
      const int st = s_cnt % kNS;
      bool r = true;
      if (s_cnt >= kNS) PROF(0, r = wait_bar(&bars->s_free[st], ((s_cnt / kNS) - 1) & 1, cx));
      if (!r) return false;
      if (even) mbar_arrive_expect_tx(&bars->s_ready[st], 2 * kSStage);
      const uint32_t bar = at_even(&bars->s_ready[st]);
      uint8_t* dst = sm + OFF_S + st * kSStage;
      tma_load_2d_pair(dst, &tmK, c * 64, y0, bar, pol_s);
      tma_load_2d_pair(dst + 8192, &tmK, c * 64, y1, bar, pol_s);
      if (s_cnt >= kLag) load_q_chunk(s_cnt - kLag);
      TRACE(16, s_cnt);
      ++s_cnt;
      return true;
    };
    // FP8 cache: raw key chunks (codes + scales of this CTA's 128 tokens, or one page of
    // bf16 RoPE keys) into the staging ring, for the converter warps
    int m_cnt = 0;
    auto load_raw_s = [&](bool rope, int c, int y0, int y1) -> bool {   // whole warp
      constexpr int RS = Bars::RS;   // >= 1 (the bf16 cache never calls this)
      const int st = m_cnt % RS;
      const int q = lane - 4 * (m_cnt & 7);   // the chunk's boxes, one lane each
      bool r = true;
      if (q >= 0 && q < (rope ? 1 : 4)) {
        if (m_cnt >= RS) PROF(0, r = wait_bar(&bars->rs_free[st], ((m_cnt / RS) - 1) & 1, cx));
        if (r) {
          uint8_t* dst = sm + Ly::OFF_RS + st * kRawS;
          uint64_t* bar = &bars->rs_ready[st];
          if (q == 0) mbar_arrive_expect_tx(bar, rope ? 8192 : kRawS);
          if (rope)
            tma_load_2d(dst, &maps.kr, kC, y0, bar, pol_s);
          else if (q < 2)
            tma_load_2d(dst + q * 4096, &maps.cs, c * 64, q ? y1 : y0, bar, pol_s);
          else
            tma_load_2d(dst + 8192 + (q - 2) * 1024, &maps.ss, kC + 2 * kR, q == 3 ? y1 : y0, bar, pol_s);
        }
      }
      ++m_cnt;
      return __all_sync(0xffffffffu, r);
    };
    // FP8 scores: one latent group's codes of this CTA's 128 tokens (two pages), the MMA's A
    // operand as loaded, into a 2-slot ring over the bf16 Q rows 4-7 (free once Q is
    // quantised); both boxes from one instruction, both CTAs' bytes on the even CTA's barrier
    int g_cnt = 0;
    auto load_group = [&](int g, int y0, int y1) -> bool {   // whole warp
      const int st = g_cnt & 1;
      bool r = true;
      if (leader && g_cnt >= 2) r = wait_bar(&bars->gs_free[st], ((g_cnt >> 1) - 1) & 1, cx);
      if (!__shfl_sync(0xffffffffu, r, 0)) return false;
      if (leader && even) mbar_arrive_expect_tx(&bars->gs_ready[st], 2 * 16384);
      __syncwarp();
      if (lane < 2)
        tma_load_2d_pair(sm + OFF_Q + 32768 + st * 16384 + lane * 8192, &maps.c8, g * 128, lane ? y1 : y0,
                         at_even(&bars->gs_ready[st]), pol_s);
      ++g_cnt;
      return true;
    };
    // key chunks of every tile in order (the latent chunks have their own producer)
    bool ok = true;
    if (F8 && Q8) {
      if (leader) ok = wait_bar(&bars->q8_done, 0, cx);
      ok = __shfl_sync(0xffffffffu, ok, 0);
    }
    for (int k = 0; k < nt && ok; ++k) {
      const int ys0 = page_y(4 * k + 2 * (int)rank);
      const int ys1 = page_y(4 * k + 2 * (int)rank + 1);
      if (F8 && Q8) {
        for (int g = 0; g < 4 && ok; ++g) ok = load_group(g, ys0, ys1);
        if (ok) ok = load_raw_s(true, 0, ys0, 0);
        if (ok) ok = load_raw_s(true, 0, ys1, 0);
      } else if constexpr (F8) {
        for (int c = 0; c < kKCh + 1 && ok; ++c) {   // 8 latent chunks, 2 RoPE half chunks
          ok = c < 8 ? load_raw_s(false, c, ys0, ys1) : load_raw_s(true, 0, c == 8 ? ys0 : ys1, 0);
        }
      } else {
        for (int c = 0; c < kKCh && ok; ++c) {
          if (leader) {
            if (c == 4) TRACE(15, k);
            ok = load_s_chunk(c, ys0, ys1);
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
        }
      }
    }
    // the Q chunks of the last NS - NQ steps, each once the MMAs of step m - NQ (the previous
    // user of its slot) have completed
    if constexpr (!F8) {
      if (ok && leader) {
        for (int m = max(s_cnt - kLag, 0); m < s_cnt && ok; ++m) {
          const int x = m - kNQ;
          if (x >= 0) ok = wait_bar(&bars->s_free[x % kNS], (uint32_t)(x / kNS) & 1u, cx);
          if (ok) load_q_chunk(m);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
    }
#ifdef MLA_TC_TRACE
    prof[7] = clock64() - prof_start;
    if (leader) PROF_STORE(520);
#endif
    if (!ok && leader) {
      // drain this CTA's loads still in flight: wait until the even CTA's MMA issuer has
      // stopped and enough time has passed for any issued load to land
      const long long t0 = clock64();
      while (clock64() - t0 < 2000000) {
      }
    }
  } else if (warp == 1) {
    // ================================================================ S^T issuer (even CTA)
    // Scores of every tile: S^T(t) = K(t) . Q^T into TMEM buffer t % 2. The P.V products have
    // their own issuing thread (warp 12): one thread cannot issue 2-SM MMAs as fast as the
    // tensor pipe retires them, two can.
    if (rank == 0 && lane == 0) {
      const uint32_t idS = idesc_bf16_f32(256, 128, 0, 0);
      // operand descriptors; an operand's start moves by adding (byte offset >> 4)
      const uint64_t dS = smem_desc(smem_u32(sm + OFF_S), 16, 1024, kSw128);
      // bf16: the streamed Q chunk of each step in its own 2-slot ring; FP8: Q is resident
      const uint64_t dQ = F8 ? smem_desc(smem_u32(sm + OFF_Q), 16, 1024, kSw128)
                             : smem_desc(smem_u32(sm + Ly::OFF_QS), 16, 1024, kSw128);
      uint32_t s_st = 0, s_ph = 0;
#ifdef MLA_TC_TRACE
      int s_cnt = 0;
      long long prof[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      const long long prof_start = clock64();
#endif
      // bf16: Q travels with the key chunks; FP8: both CTAs' resident Q halves have landed
      bool ok = F8 ? wait_bar<true>(&bars->q_conv, 0, cx) : true;
      if (F8 && Q8) {
        // FP8 scores: per tile five partial products, one per TMEM buffer use (partial n of
        // the unit in buffer n % 2): the four latent groups on FP8 tensor cores (codes of the
        // CTA's tokens . codes of its Q half, K = 128) and the bf16 RoPE part. The softmax
        // warps promote them to fp32 with the group scales; the fifth lands in buffer t % 2.
        const uint32_t id8 = idesc_e4m3_f32(256, 128);
        const uint64_t dG = smem_desc(smem_u32(sm + OFF_Q + 32768), 16, 1024, kSw128);
        const uint64_t dQ8 = smem_desc(smem_u32(sm + OFF_Q), 16, 1024, kSw128);
        uint32_t g_st = 0, g_ph = 0;
        int n = 0;
        for (int t = 0; t < nt && ok; ++t) {
          for (int p = 0; p < 5 && ok; ++p, ++n) {
            const int b = n & 1, u = n >> 1;
            if (u >= 1) ok = wait_bar(&bars->s_empty[b], (u - 1) & 1, cx);
            if (!ok) break;
            const uint32_t d = tmem + (uint32_t)b * 128u;
            if (p < 4) {
              ok = wait_bar<true>(&bars->gs_ready[g_st], g_ph, cx);
              if (!ok) break;
              tc_fence_after();
              const uint64_t a0 = dG + g_st * (16384u >> 4), b0 = dQ8 + (uint32_t)p * (8192u >> 4);
              mma_e4m3_pair(d, a0, b0, id8, 0);
              mma_e4m3_pair(d, a0 + 2, b0 + 2, id8, 1);
              mma_e4m3_pair(d, a0 + 4, b0 + 4, id8, 1);
              mma_e4m3_pair(d, a0 + 6, b0 + 6, id8, 1);
              mma_commit_pair(&bars->gs_free[g_st], 0x3);
              if (++g_st == 2) {
                g_st = 0;
                g_ph ^= 1u;
              }
            } else {
              // the RoPE keys, converted into operand slot t % kNS by the converter warps
              const int st = t % kNS;
              ok = wait_bar<true>(&bars->s_ready[st], (t / kNS) & 1, cx);
              if (!ok) break;
              tc_fence_after();
              const uint64_t a0 = dS + (uint32_t)st * (uint32_t)(kSStage >> 4), b0 = dQ + 8u * 512u;
              mma_bf16_pair(d, a0, b0, idS, 0);
              mma_bf16_pair(d, a0 + 2, b0 + 2, idS, 1);
              mma_bf16_pair(d, a0 + 4, b0 + 4, idS, 1);
              mma_bf16_pair(d, a0 + 6, b0 + 6, idS, 1);
              mma_commit_pair(&bars->s_free[st], 0x3);
            }
            mma_commit_pair(&bars->s_full[b], 0x3);
          }
        }
      } else
      for (int t = 0; t < nt && ok; ++t) {
        TRACE(22, t);
        // TMEM buffer t % 2 is free once the softmax has read S^T(t-2)
        if (t >= 2) PROF(6, ok = wait_bar(&bars->s_empty[t & 1], ((t >> 1) - 1) & 1, cx));
        if (!ok) break;
        TRACE(9, t);
        const uint32_t d = tmem + (uint32_t)(t & 1) * 128u;
        for (int c = 0; c < kKCh && ok; ++c) {
          TRACE(17, s_cnt);
          PROF(0, ok = wait_bar<F8>(&bars->s_ready[s_st], s_ph, cx));
          // bf16: step m's Q chunk, slot m % NQ, the (m / NQ)-th use of that slot
          const int m = t * kKCh + c;
          constexpr int kNQ = Ly::NQ > 0 ? Ly::NQ : 1;
          const uint32_t qslot = (uint32_t)(m % kNQ);
          if (!F8 && ok) PROF(0, ok = wait_bar(&bars->qs_ready[qslot], (uint32_t)(m / kNQ) & 1u, cx));
          if (!ok) break;
          TRACE(18, s_cnt);
          PROF(2, tc_fence_after());
          // K chunk c (128 tokens x 64 dims per CTA) . Q chunk c^T, four K=16 steps
          const uint64_t a0 = dS + s_st * (uint32_t)(kSStage >> 4);
          const uint64_t b0 = F8 ? dQ + (uint32_t)c * 512u : dQ + qslot * (8192u >> 4);
          PROF(1, {
            mma_bf16_pair(d, a0, b0, idS, c != 0);
            mma_bf16_pair(d, a0 + 2, b0 + 2, idS, 1);
            mma_bf16_pair(d, a0 + 4, b0 + 4, idS, 1);
            mma_bf16_pair(d, a0 + 6, b0 + 6, idS, 1);
          });
          PROF(2, mma_commit_pair(&bars->s_free[s_st], 0x3));
          if (++s_st == kNS) {
            s_st = 0;
            s_ph ^= 1u;
          }
#ifdef MLA_TC_TRACE
          ++s_cnt;
#endif
          if (c == 4) TRACE(13, t);
        }
        if (!ok) break;
        mma_commit_pair(&bars->s_full[t & 1], 0x3);
        TRACE(0, t);
      }
#ifdef MLA_TC_TRACE
      prof[7] = clock64() - prof_start;
      PROF_STORE(512);
#endif
      // every MMA this thread issued (they write both CTAs' TMEM) completes before teardown
      mma_commit_pair(&bars->teardown, 0x1);
      wait_drain(&bars->teardown, 0);
    }
  } else if (warp == kPvWarp) {
    // ================================================================ P.V issuer (even CTA)
    // O^T += V^T(t) . P^T(t) for every tile once both CTAs' P^T halves are in place.
    if (rank == 0 && lane == 0) {
      const uint32_t idPV = idesc_bf16_f32(256, 128, 1, 1);
      const uint64_t dV = smem_desc(smem_u32(sm + OFF_V), 4096, 1024, kSw128);
      const uint64_t dP = smem_desc(smem_u32(sm + OFF_P), 8192, 1024, kSw128);
      uint32_t v_st = 0, v_ph = 0;
#ifdef MLA_TC_TRACE
      int v_cnt = 0;
      long long prof[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      const long long prof_start = clock64();
#endif
      bool ok = true;
      const int nt_pv = mode == 1 ? 0 : nt;   // the scores-only pass issues no P.V
      for (int t = 0; t < nt_pv && ok; ++t) {
        TRACE(23, t);
        PROF(6, ok = wait_bar<true>(&bars->p_ready[t & 1], (t >> 1) & 1, cx));
        if (!ok) break;
        TRACE(1, t);
        tc_fence_after();
        for (int v = 0; v < kVCh && ok; ++v) {
          TRACE(20, v_cnt);
          PROF(3, ok = wait_bar<F8>(&bars->v_ready[v_st], v_ph, cx));
          if (!ok) break;
          TRACE(21, v_cnt);
          PROF(5, tc_fence_after());
          // this CTA's 2 x 128 latent rows x 32 tokens (V^T) . P^T rows v of tile t
          const uint64_t a0 = dV + v_st * 1024u;
          const uint64_t b0 = dP + (uint32_t)(t % kPB) * 2048u + (uint32_t)v * 256u;
          const uint32_t acc = (t | v) != 0;
          PROF(4, {
            mma_bf16_pair(tmem + 256, a0, b0, idPV, acc);
            mma_bf16_pair(tmem + 256, a0 + 128, b0 + 128, idPV, 1);
            mma_bf16_pair(tmem + 384, a0 + 512, b0, idPV, acc);
            mma_bf16_pair(tmem + 384, a0 + 640, b0 + 128, idPV, 1);
          });
          PROF(5, mma_commit_pair(&bars->v_free[v_st], 0x3));
          if (++v_st == kNV) {
            v_st = 0;
            v_ph ^= 1u;
          }
#ifdef MLA_TC_TRACE
          ++v_cnt;
#endif
        }
        if (!ok) break;
        mma_commit_pair(&bars->o_done[t & 1], 0x3);
        TRACE(2, t);
      }
#ifdef MLA_TC_TRACE
      prof[7] = clock64() - prof_start;
      PROF_STORE(536);
#endif
      mma_commit_pair(&bars->teardown, 0x1);
      wait_drain(&bars->teardown, 0);
    }
  } else if (warp == 2 && mode != 1) {
    // ================================================================ latent-chunk producer
    // Loads each tile's latent rows (this CTA's 256 d_c columns, 32 tokens per chunk) in the
    // MMA issuer's order. On the last tile the rows past the range may hold anything (P is 0
    // there): those chunks land on this CTA's own barrier, the warp zeroes the rows, and only
    // then are the bytes counted on the even CTA's barrier.
    pid_cur = fetch_pid(0);
    pid_next = fetch_pid(1);
    const uint64_t pol_v = policy_evict_first();
    const bool even = rank == 0;
    const uint32_t even_v0 = mapa(smem_u32(&bars->v_ready[0]), 0);
    int v_cnt = 0;
    bool ok = true;
#ifdef MLA_TC_TRACE
    long long prof[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    const long long prof_start = clock64();
#endif
    // Chunks of the last tile that hold rows past the range (a suffix from v_part on) land on
    // this CTA's own barrier first; the others go straight to the even CTA's barrier.
    const int base_last = (nt - 1) * kVCh;   // chunk count before the last tile
    int v_part = kVCh;
    for (int v = kVCh - 1; v >= 0; --v)
      if (lo + (nt - 1) * kTile + v * 32 + 32 > hi) v_part = v;
    auto landing = [&](int v) { return v >= v_part; };
    auto finish_last = [&](int v) -> bool {   // zero + count chunk v of the last tile
      const int st = (base_last + v) % kNV;
      // the first landing chunk in slot st, and so the phase of v_landed[st] for chunk v
      const int first = v_part + ((st - (base_last + v_part)) % kNV + kNV) % kNV;
      bool r = true;
      if (lane == 0) r = wait_bar(&bars->v_landed[st], ((v - first) / kNV) & 1, cx);
      if (!__shfl_sync(0xffffffffu, r, 0)) return false;
      const int tok0 = lo + (nt - 1) * kTile + v * 32;
      const int nvalid = max(0, min(32, hi - tok0));
      if (nvalid < 32) {
        uint4* base = reinterpret_cast<uint4*>(sm + OFF_V + st * 16384);
        const int nrow = 32 - nvalid;
        for (int idx = lane; idx < 4 * nrow * 8; idx += 32) {
          const int sub = idx / (nrow * 8);
          const int rr = nvalid + (idx / 8) % nrow;
          base[sub * 256 + rr * 8 + (idx & 7)] = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0) {
        fence_acq_rel_cluster();
        mbar_complete_tx(even_v0 + st * 8, 16384);
      }
      return true;
    };
    if constexpr (!F8) {
      for (int t = 0; t < nt && ok; ++t) {
        const bool last = t == nt - 1;
        for (int v = 0; v < kVCh && ok; ++v, ++v_cnt) {
          const int st = v_cnt % kNV;
          // before a slot is reused on the last tile, the chunk that held it must be counted
          if (last && v >= kNV && landing(v - kNV)) ok = finish_last(v - kNV);
          if (!ok) break;
          const int y = page_y(4 * t + (v >> 1)) + (v & 1) * 32;   // whole warp
          if (lane == 0) {
            if (v_cnt >= kNV) PROF(0, ok = wait_bar(&bars->v_free[st], ((v_cnt / kNV) - 1) & 1, cx));
            if (ok) {
              if (even) mbar_arrive_expect_tx(&bars->v_ready[st], 2 * 16384);
              uint32_t bar;
              if (last && landing(v)) {
                mbar_arrive_expect_tx(&bars->v_landed[st], 16384);
                bar = smem_u32(&bars->v_landed[st]);
              } else {
                bar = mapa(smem_u32(&bars->v_ready[st]), 0);
              }
              // (test hook: the even CTA registers a withheld chunk's bytes but never loads
              // them, so the P.V issuer's wait for it runs out; nothing is left in flight)
              if (!(even && v_cnt == prm.withhold))
                for (int q4 = 0; q4 < 4; ++q4)
                  tma_load_2d_pair(sm + OFF_V + st * 16384 + q4 * 4096, &tmV,
                                   (q4 >> 1) * 256 + (int)rank * 128 + (q4 & 1) * 64, y, bar, pol_v);
              TRACE(19, v_cnt);
            }
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
        }
        if (last && ok)
          for (int v = max(kVCh - kNV, 0); v < kVCh && ok; ++v)
            if (landing(v)) ok = finish_last(v);
      }
    } else {
      // FP8 cache: raw codes of this CTA's 256 d_c columns (4 boxes of 64) and the 4 scales
      // of each of 32 tokens into the staging ring; the converter warp makes the f16 tile
      int k_cnt = 0;
      for (int t = 0; t < nt && ok; ++t) {
        for (int v = 0; v < kVCh && ok; ++v) {
          const int y = page_y(4 * t + (v >> 1)) + (v & 1) * 32;   // whole warp
          const int q = lane - 5 * (k_cnt % 6);   // four code boxes and the scales, one lane each
          bool r = true;
          if (q >= 0 && q < 5) {
            const int st = k_cnt % Ly::RV;
            if (k_cnt >= Ly::RV) r = wait_bar(&bars->rv_free[st], ((k_cnt / Ly::RV) - 1) & 1, cx);
            if (r) {
              uint8_t* dst = sm + Ly::OFF_RV + st * kRawV;
              uint64_t* bar = &bars->rv_ready[st];
              if (q == 0) mbar_arrive_expect_tx(bar, kRawV);
              if (q < 4)
                tma_load_2d(dst + q * 2048, &maps.cv, (q >> 1) * 256 + (int)rank * 128 + (q & 1) * 64, y,
                            bar, pol_v);
              else
                tma_load_2d(dst + 8192, &maps.sv, kC + 2 * kR, y, bar, pol_v);
            }
          }
          ++k_cnt;
          ok = __all_sync(0xffffffffu, r);
        }
      }
    }
#ifdef MLA_TC_TRACE
    prof[7] = clock64() - prof_start;
    if (lane == 0) PROF_STORE(528);
#endif
  } else if (warp >= kCvtWarp0) {
    // ================================================================ FP8 converters
    // Dequantisation of the FP8 cache, 「Deepseek系列从v3到R易背面经版」 F8量化策略 (per-token
    // 1x128 groups): value = code * scale of its group, taken in fp32 and rounded once to bf16,
    // produced here as bf16 operand tiles in the MMA's swizzled layout (bf16 keeps fp32's
    // exponent range, so no scale or value is limited to a narrower range). The three warps
    // share the key chunks of every tile in order (9 per tile, the ninth being the bf16 RoPE
    // keys, copied into the swizzled layout): warp w takes every third chunk alone. Chunks acquire their slots
    // (the staging chunk and the free operand slot) strictly in order, through a ticket: a
    // barrier is then never waited on more than one phase ahead of the phase it is in, which
    // its parity test could not tell from the phase before; the conversions themselves
    // overlap. The latent chunks for P.V are converted by the softmax warps.
    if constexpr (F8) {
      const int cw = warp - kCvtWarp0;      // 0..2
      const int ct = tid - kCvtWarp0 * 32;   // 0..95
      // codes (8 per item) x one fp32 scale -> 8 bf16
      auto cvt8 = [](uint2 codes, float sc) -> uint4 {
        return make_uint4(e4m3x2_scaled_bf16x2(codes.x, sc), e4m3x2_scaled_bf16x2(codes.x >> 16, sc),
                          e4m3x2_scaled_bf16x2(codes.y, sc), e4m3x2_scaled_bf16x2(codes.y >> 16, sc));
      };
#ifdef MLA_TC_TRACE
      long long prof[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      const long long prof_start = clock64();
#endif
      bool ok = true;
      if (ct == 0) ok = wait_bar(&bars->q_ready, 0, cx);
      ok = bar_and(10, 96, ok);
      // Q needs no conversion (bf16 already): report this CTA's half as landed (with FP8
      // scores the softmax warps quantise Q and report it)
      if (ok && ct == 0 && !Q8) arrive_even(&bars->q_conv, rank);
      // lane 0: wait until job J is next to acquire its slots
      volatile int* ticket = &flags[FL_TICKET];
      auto my_turn = [&](int J) -> bool {
        const long long t0 = clock64();
        while (*ticket != J) {
          if (*cx.abort_flag) return false;
          if (clock64() - t0 > cx.limit) {
            *cx.abort_flag = 1;
            flag_status(cx.status, MLA_DEV_TIMEOUT);
            return false;
          }
        }
        return true;
      };
      auto pass_turn = [&](int J) {
        __threadfence_block();
        *ticket = J + 1;
      };
      // Key chunk job n (tile n / 9, chunk n % 9), raw key chunks m .. m (+1 for the RoPE keys).
      // (FP8 scores: job n is tile n's RoPE keys alone, raw chunks 2n and 2n + 1; the latent
      // groups go to the tensor cores as loaded)
      auto key_job = [&](int J, int n) -> bool {
        const int c = Q8 ? kKCh - 1 : n % kKCh;
        const int m = Q8 ? 2 * n : (n / kKCh) * (kKCh + 1) + c;   // 10 raw key chunks per tile
        const int st = n % kNS;
        uint8_t* dst = sm + OFF_S + st * kSStage;
        bool r = true;
        if (lane == 0) {
          r = my_turn(J);
          if (r && n >= kNS) PROF(0, r = wait_bar(&bars->s_free[st], ((n / kNS) - 1) & 1, cx));
          for (int h = 0; h < (c < 8 ? 1 : 2) && r; ++h)
            PROF(1, r = wait_bar(&bars->rs_ready[(m + h) % Ly::RS], ((m + h) / Ly::RS) & 1, cx));
          if (r) pass_turn(J);
        }
        if (!__shfl_sync(0xffffffffu, r, 0)) return false;
        if (c < 8) {
          // latent dims 64c .. 64c+63 of the CTA's 128 tokens; lane = rows lane + 32k.
          // 16-byte loads of the 64-byte staging rows start at a per-row rotation and the
          // tile's 128-byte swizzle spreads the stores over all banks.
          const uint8_t* src = sm + Ly::OFF_RS + (m % Ly::RS) * kRawS;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int rr = lane + 32 * k;
            const float s2 = *reinterpret_cast<const float*>(src + 8192 + rr * 16 + (c >> 1) * 4);
            uint4 in[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
              in[j] = *reinterpret_cast<const uint4*>(src + rr * 64 + (((j + rr) & 3) << 4));
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int u0 = 2 * ((j + rr) & 3);
              *reinterpret_cast<uint4*>(dst + rr * 128 + ((u0 ^ (rr & 7)) << 4)) =
                  cvt8(make_uint2(in[j].x, in[j].y), s2);
              *reinterpret_cast<uint4*>(dst + rr * 128 + (((u0 + 1) ^ (rr & 7)) << 4)) =
                  cvt8(make_uint2(in[j].z, in[j].w), s2);
            }
          }
        } else {
          // RoPE keys, bf16 -> f16: rows 0-63 from the first page's staging slot, 64-127 from
          // the second's
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int rr = lane + 32 * k;
            const uint8_t* src = sm + Ly::OFF_RS + ((m + (k >> 1)) % Ly::RS) * kRawS + (rr & 63) * 128;
            uint4 w[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) w[j] = *reinterpret_cast<const uint4*>(src + (((j + rr) & 7) << 4));
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int u = (j + rr) & 7;
              *reinterpret_cast<uint4*>(dst + rr * 128 + ((u ^ (rr & 7)) << 4)) = w[j];
            }
          }
        }
        __syncwarp();   // every lane has read the staging slot(s)
        if (lane == 0)
          for (int h = 0; h < (c < 8 ? 1 : 2); ++h) mbar_arrive(&bars->rs_free[(m + h) % Ly::RS]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) arrive_even(&bars->s_ready[st], rank);
        return true;
      };
      for (int n = cw; n < (Q8 ? nt : nt * kKCh) && ok; n += 3) ok = key_job(n, n);
#ifdef MLA_TC_TRACE
      prof[7] = clock64() - prof_start;
      if (lane == 0) PROF_STORE(544 + 8 * cw);
#endif
    }
  } else if (warp == 3 && mode != 1) {
    // ================================================================ P^T relay
    // This CTA's P^T buffer of tile t is complete once its own softmax warps have written their
    // rows and the peer's rows and maxima have landed (p_landed); the relay makes the peer's
    // stores visible to the tensor core and reports the buffer to the even CTA's P.V issuer.
    // bf16: then the whole warp sums the buffer's columns (each head of this CTA's half over
    // the tile's 256 tokens) into running sums of P, scaled by the tile's factor when the
    // reference moved; the softmax threads then need no cross-thread sum per tile.
    bool ok = true;
    float l0 = 0.f, l1 = 0.f;   // bf16: sums of P for heads 64 rank + 2 lane, + 1
    for (int t = 0; t < nt && ok; ++t) {
      const int par = t & 1;
      if (lane == 0) {
        ok = wait_bar<true>(&bars->p_landed[par], (t >> 1) & 1, cx);
        TRACE(7, t);
        if (ok) {
          fence_proxy_async_smem();
          arrive_even(&bars->p_ready[par], rank);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if constexpr (!F8) {
        if (!ok) break;
        // row r: 64 bf16 weights in 16-byte chunks, chunk c at (c ^ (r % 8)) * 16; lane j
        // reads word j % 4 of chunk j / 4, i.e. heads 2j and 2j + 1
        const uint8_t* buf = sm + OFF_P + (t % kPB) * 32768 + (lane & 3) * 4;
        // (even and odd rows in separate chains; each bf16 half enters its fp32 add directly)
        const int cc = lane >> 2;
        float c0 = 0.f, c1 = 0.f, d0 = 0.f, d1 = 0.f;
#pragma unroll 8
        for (int r = 0; r < 256; r += 2) {
          const uint32_t w = *reinterpret_cast<const uint32_t*>(buf + r * 128 + ((cc ^ (r & 7)) << 4));
          const uint32_t x = *reinterpret_cast<const uint32_t*>(buf + (r + 1) * 128 + ((cc ^ ((r + 1) & 7)) << 4));
          add_bf16x2_f32(c0, c1, w);
          add_bf16x2_f32(d0, d1, x);
        }
        c0 += d0;
        c1 += d1;
        // the reference moves from tile 2 on, with the factor the softmax stored for tile t
        if (t >= 2) {
          const float* a = fs + (par ? F_ALPHA_ODD : F_ALPHA) + 64 * (int)rank + 2 * lane;
          l0 *= a[0];
          l1 *= a[1];
        }
        l0 += c0;
        l1 += c1;
        if (t == nt - 1) {
          // the finished sums: kept, and sent to the peer (which holds the other 64 heads) while
          // the last P.V still runs, together with this CTA's clamp flag (final: the softmax set
          // it before its last P^T rows landed)
          const int h = 64 * (int)rank + 2 * lane;
          fs[F_LLOC + h] = l0;
          fs[F_LLOC + h + 1] = l1;
          const uint32_t peer_l = mapa(smem_u32(fs + F_LRCV + h), peer);
          const uint32_t peer_l_bar = mapa(smem_u32(&bars->l_landed), peer);
          st_async_b32(peer_l, __float_as_uint(l0), peer_l_bar);
          st_async_b32(peer_l + 4, __float_as_uint(l1), peer_l_bar);
          if (lane == 0) {
            st_async_b32(mapa(smem_u32(&flags[FL_PEER_CLAMP]), peer), (uint32_t)flags[FL_CLAMP], peer_l_bar);
            mbar_arrive_expect_tx(&bars->l_landed, 64 * 4 + 4);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->l_done[par]);
      }
    }
  } else if (warp >= 4 && warp < 12) {
    // ================================================================ softmax / epilogue
    // Thread = one TMEM lane: token i of this CTA's half tile for the scores, latent row i for
    // the output. Each thread handles one head group (64 heads) of its token.
    //
    // Online softmax with a lazy reference (log2 units) M[h], identical in both CTAs: tile 0
    // sets it from both CTAs' maxima; afterwards a tile whose scores exceed M by more than
    // kLazy publishes its per-head maxima, and two tiles later both CTAs move M (and rescale
    // O and the running sums) from the same published data. Tiles in between use the old
    // reference, so their weights may exceed 1 (up to 2^kRange, which fp32 sums and bf16 P
    // hold without loss); the common tile needs no cross-thread reduction at all.
    const int sw = warp - 4;           // 0..7
    const int g = sw >> 2;             // head group: heads [64g, 64g + 64)
    const int qd = warp & 3;           // TMEM lane quadrant
    const int i = qd * 32 + lane;      // this CTA's token row (S^T) / latent row (O^T)
    const int stid = tid - 128;        // 0..255
    const uint32_t lane_addr = tmem + ((uint32_t)(qd * 32) << 16);
    const float* Mg = fs + F_M + 64 * g;
    const uint32_t peer_rcv = mapa(smem_u32(fs + F_RCV), peer);
    uint32_t peer_landed = 0;
    float l_w[2] = {0.f, 0.f};   // sums of P of this warp's tokens for heads 64g + 32 h2 + lane
#ifdef MLA_TC_TRACE
    long long prof[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    const long long prof_start = clock64();
#endif
    bool ok = true;
    // ---- FP8 scores (「Deepseek系列从v3到R易背面经版」 F8量化策略: E4M3 with 1x128 activation
    // groups, partial sums promoted to fp32 every 128 products). This CTA's Q half is quantised
    // per (head, 128-dim group) as the cache's latents are: thread = (head hq, group gq); the
    // codes replace bf16 rows 0-3 of the resident Q in the FP8 operand layout (128-byte rows,
    // 128-byte swizzle) and the scale goes to both CTAs' F_SQ. Every pass does it, as every
    // pass loads Q again.
    float skv[4] = {0.f, 0.f, 0.f, 0.f}, skn[4] = {0.f, 0.f, 0.f, 0.f};
    // the four key group scales of this thread's token of tile t (0 past the range)
    auto key_scales = [&](int t, float* out) {
      const int tok = lo + t * kTile + (int)rank * 128 + i;
      out[0] = out[1] = out[2] = out[3] = 0.f;
      if (tok < hi) {
        const int pg = __ldg(prm.bt + (size_t)b * prm.maxp + tok / kP);
        if (pg >= 0 && pg < prm.num_pages) {
          const float4 v = __ldg(reinterpret_cast<const float4*>(
              prm.pool + ((size_t)pg * kP + (size_t)(tok % kP)) * (size_t)(kC + 2 * kR + 16) + kC + 2 * kR));
          out[0] = v.x;
          out[1] = v.y;
          out[2] = v.z;
          out[3] = v.w;
        }
      }
    };
    if (F8 && Q8) {
      bool okq = true;
      if (stid == 0) okq = wait_bar(&bars->q_ready, 0, cx);
      okq = bar_and(1, 256, okq);
      const int hq = stid >> 2, gq = stid & 3;
      const uint32_t swq = (uint32_t)(hq & 7);
      uint4 cw8[8];
      float sq = 1.f;
      if (okq) {
        // group gq = bf16 rows 2gq and 2gq + 1 of head hq; logical 16-byte unit u of a row is at
        // u ^ (hq & 7)
        float amax = 0.f;
#pragma unroll
        for (int uu = 0; uu < 16; ++uu) {
          const uint4 x = *reinterpret_cast<const uint4*>(sm + OFF_Q + (2 * gq + (uu >> 3)) * 8192 + hq * 128 +
                                                          ((((uint32_t)uu & 7u) ^ swq) << 4));
          const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            amax = fmaxf(amax, fmaxf(fabsf(p16_to_f32(w[e] & 0xFFFFu)), fabsf(p16_to_f32(w[e] >> 16))));
        }
        sq = amax > 0.f ? __fdiv_rn(amax, kE4M3Max) : 1.f;
        // code unit cu (codes 16cu .. 16cu + 15) comes from bf16 units 2cu, 2cu + 1 of the group
#pragma unroll
        for (int cu = 0; cu < 8; ++cu) {
          uint32_t c4[4];
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int uu = 2 * cu + k;
            const uint4 x = *reinterpret_cast<const uint4*>(sm + OFF_Q + (2 * gq + (uu >> 3)) * 8192 + hq * 128 +
                                                            ((((uint32_t)uu & 7u) ^ swq) << 4));
            const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const uint32_t a = w[2 * e], bb = w[2 * e + 1];
              c4[2 * k + e] = (uint32_t)e4m3_encode(__fdiv_rn(p16_to_f32(a & 0xFFFFu), sq)) |
                              ((uint32_t)e4m3_encode(__fdiv_rn(p16_to_f32(a >> 16), sq)) << 8) |
                              ((uint32_t)e4m3_encode(__fdiv_rn(p16_to_f32(bb & 0xFFFFu), sq)) << 16) |
                              ((uint32_t)e4m3_encode(__fdiv_rn(p16_to_f32(bb >> 16), sq)) << 24);
            }
          }
          cw8[cu] = make_uint4(c4[0], c4[1], c4[2], c4[3]);
        }
      }
      bar_sync(2, 256);   // every bf16 row has been read before any is overwritten
      if (okq) {
        uint8_t* dst = sm + OFF_Q + gq * 8192 + hq * 128;
#pragma unroll
        for (int cu = 0; cu < 8; ++cu) *reinterpret_cast<uint4*>(dst + ((((uint32_t)cu) ^ swq) << 4)) = cw8[cu];
        const int hh = (int)rank * 64 + hq;
        fs[F_SQ + hh * 4 + gq] = sq;
        st_async_b32(mapa(smem_u32(fs + F_SQ + hh * 4 + gq), peer), __float_as_uint(sq),
                     mapa(smem_u32(&bars->sq_ready), peer));
        fence_proxy_async_smem();
      }
      bar_sync(3, 256);   // all codes written and fenced for the tensor core
      bool okx = okq;
      if (stid == 0 && okq) {
        mbar_arrive(&bars->q8_done);          // the group ring may overwrite bf16 rows 4-7
        arrive_even(&bars->q_conv, rank);     // this CTA's Q half is ready for the MMAs
        mbar_arrive_expect_tx(&bars->sq_ready, 64 * 4 * 4);
        okx = wait_bar<true>(&bars->sq_ready, 0, cx);
      }
      ok = bar_and(4, 256, okx);
      key_scales(0, skn);
    }
    // the five partial products of tile t promoted to fp32 (x key scale x query scale per
    // latent group, x 1 for the RoPE part), written into buffer par for the softmax below
    auto promote = [&](int t, int par) -> bool {
#pragma unroll
      for (int k = 0; k < 4; ++k) skv[k] = skn[k];
      if (t + 1 < nt) key_scales(t + 1, skn);
      float acc[64];
#pragma unroll
      for (int c = 0; c < 64; ++c) acc[c] = 0.f;
#pragma unroll 1
      for (int p = 0; p < 5; ++p) {
        const int n = 5 * t + p, bb = n & 1, u = n >> 1;
        // each warp reads only its own TMEM lanes: one lane polls for the warp
        bool okp = true;
        if (lane == 0) okp = wait_bar(&bars->s_full[bb], (uint32_t)(u & 1), cx);
        if (!__shfl_sync(0xffffffffu, okp, 0)) return false;
        tc_fence_after();
        const float f = p == 0 ? skv[0] : p == 1 ? skv[1] : p == 2 ? skv[2] : p == 3 ? skv[3] : 1.f;
#pragma unroll
        for (int h4 = 0; h4 < 4; ++h4) {
          float x[16];
          tmem_ld16(lane_addr + (uint32_t)bb * 128u + 64 * g + 16 * h4, x);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const float qs = p < 4 ? fs[F_SQ + (64 * g + 16 * h4 + c) * 4 + p] : 1.f;
            acc[16 * h4 + c] = fmaf(f * qs, x[c], acc[16 * h4 + c]);
          }
        }
        if (p < 4) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if (rank == 0)
              mbar_arrive(&bars->s_empty[bb]);
            else
              mbar_arrive_remote_relaxed(mapa(smem_u32(&bars->s_empty[bb]), 0));
          }
        }
      }
      tmem_st32(lane_addr + (uint32_t)par * 128u + 64 * g, acc);
      tmem_st32(lane_addr + (uint32_t)par * 128u + 64 * g + 32, acc + 32);
      tmem_st_wait();
      return true;
    };
    if (!ok) {
    } else if (mode == 1) {
      // ---- scores only: the exact per-head maxima of this range. Lane j of each warp keeps
      // the running maxima of heads 64g + j and 64g + 32 + j over the warp's tokens; the
      // warps, then the two CTAs, combine them into F_M, which the next pass uses as its
      // reference from the first tile on.
      float run[2] = {-CUDART_INF_F, -CUDART_INF_F};
      for (int t = 0; t < nt; ++t) {
        const int par = t & 1;
        bool ok1 = true;
        if (F8 && Q8)
          ok1 = promote(t, par);
        else if (stid == 0)
          ok1 = wait_bar(&bars->s_full[par], (t >> 1) & 1, cx);
        ok = bar_and(1, 256, ok1);
        if (!ok) break;
        tc_fence_after();
        const uint32_t s_addr = lane_addr + par * 128 + 64 * g;
        const bool valid = lo + t * kTile + (int)rank * 128 + i < hi;
#pragma unroll 1
        for (int h2 = 0; h2 < 2; ++h2) {
          float sv[32];
          tmem_ld32(s_addr + 32 * h2, sv);
          tmem_ld_wait();
          if (h2 == 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
              if (rank == 0)
                mbar_arrive(&bars->s_empty[par]);
              else
                mbar_arrive_remote_relaxed(mapa(smem_u32(&bars->s_empty[par]), 0));
            }
          }
          if constexpr (!F8) {
            float v[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) v[c] = valid ? sv[c] * prm.scale_log2 : -CUDART_INF_F;
            run[h2] = fmaxf(run[h2], warp_transpose_max32(v, lane));
          } else {
            // (the FP8 instantiations keep one reduction per column: the transposing form
            // measured slower there, through their register allocation)
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              const float mx = warp_max_f32(valid ? sv[c] * prm.scale_log2 : -CUDART_INF_F);
              if (lane == c) run[h2] = fmaxf(run[h2], mx);
            }
          }
        }
      }
      if (ok) {
        fs[F_COL + sw * 64 + lane] = run[0];
        fs[F_COL + sw * 64 + 32 + lane] = run[1];
        bar_sync(2, 256);
        float my_max = -CUDART_INF_F;
        if (stid < kH) {
          const int h = stid, gg = h >> 6, cc = h & 63;
#pragma unroll
          for (int q = 0; q < 4; ++q) my_max = fmaxf(my_max, fs[F_COL + (gg * 4 + q) * 64 + cc]);
          st_async_b32(mapa(smem_u32(fs + F_X0 + h), peer), __float_as_uint(my_max),
                       mapa(smem_u32(&bars->x0_ready), peer));
        }
        bool okx = true;
        if (stid == 0) {
          mbar_arrive_expect_tx(&bars->x0_ready, kH * 4);
          okx = wait_bar<true>(&bars->x0_ready, 0, cx);
        }
        ok = bar_and(13, 256, okx);
        if (ok && stid < kH) fs[F_M + stid] = fmaxf(my_max, fs[F_X0 + stid]);
      }
    } else {
    for (int t = 0; t < nt; ++t) {
      const int par = t & 1, slot = t & (kXSlots - 1);
      peer_landed = mapa(smem_u32(&bars->p_landed[par]), peer);
      // ---- reference for tile t, from tile t-2's published maxima (both CTAs). One thread
      // waits on each barrier; the others sleep in the named barrier, so no warp spins.
      bool ok1 = true;
      // bf16: this tile's rescale factors overwrite tile t - 2's, which the relay must have read
      const int f_alpha = (!F8 && par) ? F_ALPHA_ODD : F_ALPHA;
      if (t >= 2) {
        if (stid == 0) PROF(3, ok1 = wait_bar<true>(&bars->p_landed[par], ((t - 2) >> 1) & 1, cx));
        if (!F8 && stid == 0 && ok1) PROF(3, ok1 = wait_bar(&bars->l_done[par], ((t - 2) >> 1) & 1, cx));
        ok = bar_and(12, 256, ok1);
        if (!ok) break;
      }
      if (t >= 2 && stid < kH) {
        const int h = stid;
        const float* rcv = fs + F_RCV + ((t - 2) & (kXSlots - 1)) * kH;
        float cand = rcv[h];
        if (flags[FL_PUB + par]) cand = fmaxf(cand, fs[F_CMLOC + par * kH + h]);
        const float mo = fs[F_M + h];
        float alpha = 1.f;
        if (cand > mo + kLazy) {
          alpha = ex2(mo - cand);
          fs[F_M + h] = cand;
          flags[FL_RESCALE + par] = 1;
        }
        fs[f_alpha + h] = alpha;
      }
      if (F8 && Q8)
        ok1 = promote(t, par);
      else if (stid == 0)
        PROF(4, ok1 = wait_bar(&bars->s_full[par], (t >> 1) & 1, cx));
      ok = bar_and(1, 256, ok1);
      if (!ok) break;
      if (stid == 0) TRACE(3, t);
      const bool rescale = flags[FL_RESCALE + par] != 0;
      tc_fence_after();
      const uint32_t s_addr = lane_addr + par * 128 + 64 * g;
      const int tok = lo + t * kTile + (int)rank * 128 + i;
      const bool valid = tok < hi;
      if (t == 0 && mode == 0) {
        // ---- the first reference: per-head maxima over both CTAs' tokens of tile 0
#pragma unroll 1
        for (int h2 = 0; h2 < 2; ++h2) {
          float s[32];
          tmem_ld32(s_addr + 32 * h2, s);
          tmem_ld_wait();
          if constexpr (!F8) {
#pragma unroll
            for (int c = 0; c < 32; ++c) s[c] = valid ? s[c] * prm.scale_log2 : -CUDART_INF_F;
            fs[F_COL + sw * 64 + 32 * h2 + lane] = warp_transpose_max32(s, lane);
          } else {
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              const float mx = warp_max_f32(valid ? s[c] * prm.scale_log2 : -CUDART_INF_F);
              if (lane == c) fs[F_COL + sw * 64 + 32 * h2 + c] = mx;
            }
          }
        }
        bar_sync(2, 256);
        // this CTA's per-head maxima go straight into the peer's shared memory (st.async,
        // counted on the peer's x0_ready), the peer's arrive the same way
        float my_max = -CUDART_INF_F;
        if (stid < kH) {
          const int h = stid, gg = h >> 6, cc = h & 63;
#pragma unroll
          for (int q = 0; q < 4; ++q) my_max = fmaxf(my_max, fs[F_COL + (gg * 4 + q) * 64 + cc]);
          st_async_b32(mapa(smem_u32(fs + F_X0 + h), peer), __float_as_uint(my_max),
                       mapa(smem_u32(&bars->x0_ready), peer));
        }
        bool okx = true;
        if (stid == 0) {
          mbar_arrive_expect_tx(&bars->x0_ready, kH * 4);
          okx = wait_bar<true>(&bars->x0_ready, 0, cx);
        }
        ok = bar_and(13, 256, okx);
        if (!ok) break;
        if (stid < kH) {
          const int h = stid;
          fs[F_M + h] = fmaxf(my_max, fs[F_X0 + h]);
          fs[F_ALPHA + h] = 1.f;
        }
        bar_sync(4, 256);
      }
      if (stid == 0) TRACE(4, t);
      // ---- weights p = 2^(s - M) in bf16 (32 heads at a time), the overshoot checks, and
      // the running per-head sums of this warp's tokens (lane j keeps head 32 h2 + j)
      uint32_t pk[32];
      bool over = false, extreme = false;
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        float s[32];
        tmem_ld32(s_addr + 32 * h2, s);
        tmem_ld_wait();
        if (h2 == 1) {
          tc_fence_before();
          __syncwarp();
          // (the loads are complete; the arrival publishes nothing, so it need not wait for
          // this thread's outstanding P^T stores to the exchange ring)
          if (lane == 0) {
            if (rank == 0)
              mbar_arrive(&bars->s_empty[par]);
            else
              mbar_arrive_remote_relaxed(mapa(smem_u32(&bars->s_empty[par]), 0));
          }
          if (stid == 0) TRACE(12, t);
        }
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 m4 = *reinterpret_cast<const float4*>(Mg + 32 * h2 + 4 * c4);
          const float m[4] = {m4.x, m4.y, m4.z, m4.w};
          float p[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float d = (valid ? s[4 * c4 + e] * prm.scale_log2 : -CUDART_INF_F) - m[e];
            over |= d > kLazy;
            extreme |= d > kRange;
            d = fminf(d, kRange);
            p[e] = ex2(d);
          }
          pk[16 * h2 + 2 * c4] = pack_bf16x2(p[0], p[1]);
          pk[16 * h2 + 2 * c4 + 1] = pack_bf16x2(p[2], p[3]);
        }
        if constexpr (F8) {
          float v[32];
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            v[2 * c] = p16_to_f32(pk[16 * h2 + c] & 0xFFFFu);
            v[2 * c + 1] = p16_to_f32(pk[16 * h2 + c] >> 16);
          }
          const float lsum = warp_transpose_sum32(v, lane);
          if (rescale) l_w[h2] *= fs[F_ALPHA + 64 * g + 32 * h2 + lane];
          l_w[h2] += lsum;
        }
      }
      if (extreme) flags[FL_CLAMP] = 1;
      if (stid == 0) TRACE(14, t);
      // P^T's buffer (in both CTAs) is free once P.V of tile t - kPB is done; O is stable to
      // rescale once P.V of the previous tile is
      bool ok3 = true;
      {
        const int wt = rescale ? t - 1 : t - kPB;   // (a rescale needs t >= 2)
        if (wt >= 0 && stid == 0) PROF(5, ok3 = wait_bar(&bars->o_done[wt & 1], (wt >> 1) & 1, cx));
      }
      bool any_over = false;
      if (bar_or(5, 256, over || !ok3)) {
        ok = bar_and(6, 256, ok3);
        if (!ok) break;
        any_over = true;
        // ---- this tile's per-head maxima, published for the reference two tiles on: the
        // largest weight of each head (all relative to the same M) gives max s = M + log2(p)
        if constexpr (!F8) {
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            float v[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              const uint32_t w = pk[16 * h2 + (c >> 1)];
              v[c] = p16_to_f32((c & 1) ? (w >> 16) : (w & 0xFFFFu));
            }
            fs[F_COL + sw * 64 + 32 * h2 + lane] = warp_transpose_max32(v, lane);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const uint32_t w = pk[c >> 1];
            const float pv = p16_to_f32((c & 1) ? (w >> 16) : (w & 0xFFFFu));
            const float mx = warp_max_f32(pv);
            if (lane == (c & 31)) fs[F_COL + sw * 64 + c] = mx;
          }
        }
        bar_sync(2, 256);
        if (stid < kH) {
          const int h = stid, gg = h >> 6, cc = h & 63;
          float pmax = 0.f;
#pragma unroll
          for (int q = 0; q < 4; ++q) pmax = fmaxf(pmax, fs[F_COL + (gg * 4 + q) * 64 + cc]);
          const float my_max = pmax > 0.f ? fs[F_M + h] + log2f(pmax) : -CUDART_INF_F;
          fs[F_CMLOC + par * kH + h] = my_max;
          st_async_b32(peer_rcv + (uint32_t)(slot * kH + h) * 4u, __float_as_uint(my_max), peer_landed);
        }
        bar_sync(3, 256);
      } else if (stid < kH) {
        // nothing published: the peer's slot reads -inf
        st_async_b32(peer_rcv + (uint32_t)(slot * kH + stid) * 4u, __float_as_uint(-CUDART_INF_F),
                     peer_landed);
      }
      if (stid == 0) {
        flags[FL_PUB + par] = any_over ? 1 : 0;
        flags[FL_RESCALE + par] = 0;   // every thread has read it (barrier 5)
        TRACE(5, t);
      }
      tc_fence_after();
      if (rescale) {
#pragma unroll 1
        for (int blk = 0; blk < 2; ++blk)
#pragma unroll 1
          for (int hh = 0; hh < 2; ++hh) {
            float o[32];
            const uint32_t ta = lane_addr + 256 + blk * 128 + 64 * g + hh * 32;
            tmem_ld32(ta, o);
            tmem_ld_wait();
#pragma unroll
            for (int x = 0; x < 32; ++x) o[x] *= fs[f_alpha + 64 * g + hh * 32 + x];
            tmem_st32(ta, o);
          }
        tmem_st_wait();
      }
      // ---- P^T rows of this CTA's tokens: its own head half into its buffer, the peer's half
      // straight into the peer's buffer (same offsets, 128-byte swizzle)
      {
        const uint32_t sw_off = (uint32_t)((i & 7) * 16);
        const uint32_t off = (uint32_t)(OFF_P + (t % kPB) * 32768 + ((int)rank * 128 + i) * 128);
        if (g == (int)rank) {
#pragma unroll
          for (int cc = 0; cc < 8; ++cc)
            *reinterpret_cast<uint4*>(sm + off + ((cc * 16) ^ sw_off)) =
                make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
          fence_proxy_async_smem();
        } else {
          const uint32_t dst = mapa(smem_u32(sm + off), peer);
#pragma unroll
          for (int cc = 0; cc < 8; ++cc)
            st_async_v4_b32(dst + ((cc * 16) ^ sw_off),
                            make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]),
                            peer_landed);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (sw == 0) {
          mbar_arrive_expect_tx(&bars->p_landed[par], kXBytes);   // the peer's rows + maxima
          TRACE(6, t);
        } else {
          mbar_arrive(&bars->p_landed[par]);
        }
      }
      if constexpr (F8) {
        // ---- FP8 cache: this tile's latent chunks for P.V, dequantised by the 256 softmax
        // threads (chunk = 32 tokens x this CTA's 256 d_c columns; thread = token rr, 32 codes
        // of sub-tile q4 = part / 2). Rows past the range become zeros, so that P = 0 never
        // meets stale data.
        const int rr = stid & 31, part = stid >> 5, q4 = part >> 1, half = part & 1;
#ifdef MLA_TC_TRACE
        const long long pv0 = clock64();
#endif
#pragma unroll 1
        for (int v = 0; v < kVCh && ok; ++v) {
          const int n = t * kVCh + v;
          const int st = n % kNV, rv = n % Ly::RV;
          bool r = true;
          if (stid == 0) {
            if (n >= kNV) PROF(0, r = wait_bar(&bars->v_free[st], ((n / kNV) - 1) & 1, cx));
            if (r) PROF(1, r = wait_bar(&bars->rv_ready[rv], (n / Ly::RV) & 1, cx));
          }
          ok = bar_and(15, 256, r);
          if (!ok) break;
          const uint8_t* src = sm + Ly::OFF_RV + rv * kRawV;
          uint8_t* dst = sm + OFF_V + st * 16384 + q4 * 4096 + rr * 128;
          const bool valid = lo + t * kTile + v * 32 + rr < hi;
          const float sc = *reinterpret_cast<const float*>(src + 8192 + rr * 16 +
                                                           ((q4 < 2 ? 0 : 2) + (int)rank) * 4);
          const uint4* in = reinterpret_cast<const uint4*>(src + q4 * 2048 + rr * 64 + half * 32);
          const uint4 a0 = in[0], a1 = in[1];
          const uint4 z = make_uint4(0, 0, 0, 0);
          const uint32_t w[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t u = (uint32_t)(half * 4 + k) ^ (uint32_t)(rr & 7);
            const uint4 o = make_uint4(e4m3x2_scaled_bf16x2(w[2 * k], sc),
                                       e4m3x2_scaled_bf16x2(w[2 * k] >> 16, sc),
                                       e4m3x2_scaled_bf16x2(w[2 * k + 1], sc),
                                       e4m3x2_scaled_bf16x2(w[2 * k + 1] >> 16, sc));
            *reinterpret_cast<uint4*>(dst + u * 16) = valid ? o : z;
          }
          fence_proxy_async_smem();
          bar_sync(15, 256);
          if (stid == 0) {
            mbar_arrive(&bars->rv_free[rv]);
            arrive_even(&bars->v_ready[st], rank);
          }
        }
#ifdef MLA_TC_TRACE
        prof[2] += clock64() - pv0;
#endif
        if (!ok) break;
      }
    }
#ifdef MLA_TC_TRACE
    prof[7] = clock64() - prof_start;
    if (stid == 0) PROF_STORE(568);
#endif
    if (ok) {
      // ------------------------------------------------------------ epilogue
      if (stid == 0) ok = wait_bar(&bars->o_done[(nt - 1) & 1], ((nt - 1) >> 1) & 1, cx);
      ok = bar_and(7, 256, ok);
      if (ok) {
        tc_fence_after();
        const uint32_t peer_l = mapa(smem_u32(fs + F_LRCV), peer);
        const uint32_t peer_l_bar = mapa(smem_u32(&bars->l_landed), peer);
        bool ok4 = true;
        if constexpr (F8) {
          // per-head sums of P over this warp's tokens, then over this CTA's tokens
          fs[F_COL + sw * 64 + lane] = l_w[0];
          fs[F_COL + sw * 64 + 32 + lane] = l_w[1];
          bar_and(8, 256, true);
          if (stid < kH) {
            const int h = stid, gg = h >> 6, cc = h & 63;
            float sum = 0.f;
#pragma unroll
            for (int q = 0; q < 4; ++q) sum += fs[F_COL + (gg * 4 + q) * 64 + cc];
            fs[F_LLOC + h] = sum;
            st_async_b32(peer_l + (uint32_t)(h * 4), __float_as_uint(sum), peer_l_bar);
          }
        }
        if (stid == 0 && ok4) {
          if constexpr (F8) {
            // with the sums goes this CTA's clamp flag, so that both CTAs take the same decision
            st_async_b32(mapa(smem_u32(&flags[FL_PEER_CLAMP]), peer), (uint32_t)flags[FL_CLAMP],
                         peer_l_bar);
            mbar_arrive_expect_tx(&bars->l_landed, kH * 4 + 4);
          } else {
            // bf16: the relay sent this CTA's sums and flag after the last tile; its own
            // sums are in F_LLOC once that has happened
            ok4 = wait_bar(&bars->l_done[(nt - 1) & 1], ((nt - 1) >> 1) & 1, cx);
          }
          if (ok4) ok4 = wait_bar<true>(&bars->l_landed, 0, cx);
        }
        ok4 = bar_and(14, 256, ok4);
        // a clamped weight in either CTA: the outputs of this pass are not written, the unit
        // runs again exactly
        const bool replay = mode == 0 && (flags[FL_CLAMP] | flags[FL_PEER_CLAMP]) != 0;
        if (replay && stid == 0) flags[FL_REPLAY] = 1;
        if (ok4 && !replay && stid < kH) {
          const int h = stid;
          const float mine = fs[F_LLOC + h], other = fs[F_LRCV + h];
          // FP8: both CTAs' tokens summed here; bf16: each half's sum is whole in one CTA
          const float Lsum = F8 ? (rank == 0 ? mine + other : other + mine)
                                : ((h >> 6) == (int)rank ? mine : other);
          fs[F_INV + h] = Lsum > 0.f ? 1.f / Lsum : 0.f;
          if (rank == 0) {
            const float lse = Lsum > 0.f ? (fs[F_M + h] + log2f(Lsum)) * 0.6931471805599453f
                                         : -CUDART_INF_F;
            const size_t o = (size_t)obase + (size_t)h * ostride;
            if (ostride == 1) {
              if (prm.lse) prm.lse[o] = lse;
            } else {
              prm.ws_lse[o] = lse;
            }
          }
        }
        ok = bar_and(9, 256, ok4);
        if (ok && !replay) {
#pragma unroll 1
          for (int blk = 0; blk < 2; ++blk) {
            const int dc = blk * 256 + (int)rank * 128 + i;
#pragma unroll 1
            for (int hh = 0; hh < 2; ++hh) {
              float o[32];
              tmem_ld32(lane_addr + 256 + blk * 128 + 64 * g + hh * 32, o);
              tmem_ld_wait();
#pragma unroll
              for (int x = 0; x < 32; ++x) {
                const int h = 64 * g + hh * 32 + x;
                const float val = o[x] * fs[F_INV + h];
                const size_t o = (size_t)obase + (size_t)h * ostride;
                if (ostride == 1)
                  prm.o_lat[o * kC + dc] = __float2bfloat16_rn(val);
                else
                  prm.ws_o[o * kC + dc] = val;
              }
            }
          }
        }
      }
    }
    }
  }

}

// End of a pass. Both CTAs decide from both CTAs' abort flags and from the replay flag (which
// both derived from the same exchanged data), so they always meet at the same cluster barriers.
// Returns whether another pass follows; if so, the barriers and flags are set up for it.
template <bool F8>
__device__ __forceinline__ bool end_of_pass(int mode, uint8_t* sm) {
  float* fs = reinterpret_cast<float*>(sm + Lay<F8>::OFF_F);
  int* flags = reinterpret_cast<int*>(fs + F_FLAG);
  BarsT<F8>* bars = reinterpret_cast<BarsT<F8>*>(sm + Lay<F8>::OFF_BAR);
  const int tid = threadIdx.x;
  tc_fence_before();
  __syncthreads();
  if (tid == 0) st_cluster_u32(mapa(smem_u32(&flags[FL_PEER_ABORT]), cluster_ctarank() ^ 1u), (uint32_t)flags[FL_ABORT]);
  cluster_sync();
  const bool again = flags[FL_ABORT] == 0 && flags[FL_PEER_ABORT] == 0 &&
                     (mode == 1 || (mode == 0 && flags[FL_REPLAY] != 0));
  if (!again) return false;
  __syncthreads();   // every thread has read the flags
  if (tid == 0) {
    // every operation of the pass has completed and been waited for, except the arrivals that
    // MMA commits make on barriers nobody waits on at the end (the last stages' "free"
    // signals): give those a moment to land before the barriers are initialised again
    const long long t0 = clock64();
    while (clock64() - t0 < 4000) {
    }
    init_barriers<F8>(bars);
  }
  if (tid < F_FLAGS_END - F_FLAG) flags[tid] = 0;
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  return true;
}

// The same pass as an out-of-line function (the FP8 cache's passes run through it: measured
// faster there than the pass inlined into the kernel).
template <bool F8, bool Q8 = false>
__device__ __noinline__ void decode_pass_ool(const Maps& maps, const Params& prm, uint8_t* sm, int mode) {
  decode_pass<F8, Q8>(maps, prm, sm, mode);
}

// The two extra passes of a unit whose first pass clamped a weight, out of line so that the
// bf16 cache's ordinary pass stays straight-line code in the kernel.
template <bool F8>
__device__ __noinline__ void replay_passes(const Maps& maps, const Params& prm, uint8_t* sm) {
  decode_pass<F8>(maps, prm, sm, 1);
  if (end_of_pass<F8>(1, sm)) {
    decode_pass<F8>(maps, prm, sm, 2);
    end_of_pass<F8>(2, sm);
  }
}

template <bool F8, bool Q8 = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Lay<F8>::THREADS, 1)
    decode_kernel(const __grid_constant__ Maps maps, const __grid_constant__ Params prm) {
  using Ly = Lay<F8>;
  using Bars = BarsT<F8>;
  constexpr int kNS = Ly::NS, kNV = Ly::NV, kThreads = Ly::THREADS;
  constexpr int OFF_Q = Ly::OFF_Q, OFF_S = Ly::OFF_S, OFF_V = Ly::OFF_V, OFF_P = Ly::OFF_P;
  constexpr int kSStage = Ly::SSTAGE, kPB = Ly::PB;
  constexpr int OFF_F = Ly::OFF_F, OFF_BAR = Ly::OFF_BAR;
  const CUtensorMap& tmQ = maps.q;
  const CUtensorMap& tmK = maps.k;
  const CUtensorMap& tmV = maps.v;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  float* fs = reinterpret_cast<float*>(sm + OFF_F);
  int* flags = reinterpret_cast<int*>(fs + F_FLAG);
  Bars* bars = reinterpret_cast<Bars*>(sm + OFF_BAR);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;

  const int unit = blockIdx.x >> 1;
  // ---- set-up
  if (tid == 0) TRACE(11, 0);
  if (tid == 0) init_barriers<F8>(bars);
  if (tid < kH) fs[F_M + tid] = -CUDART_INF_F;
  if (tid < F_FLAGS_END - F_FLAG) flags[tid] = 0;
  if (warp == 1) {
    tmem_alloc_pair(&bars->tmem_base, 512);
    tmem_relinquish_pair();
  }
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  // Everything above touches only this pair's own shared memory and TMEM, so with a
  // programmatic launch it overlaps the tail of the preceding kernel on the stream; every
  // read of the inputs comes after that kernel has completed.
  griddep_launch_dependents();
  griddep_wait();

  // A unit normally takes one pass (mode 0). If a weight had to be clamped in it, both CTAs
  // run it again: mode 1 computes only the scores, for the exact per-head maxima over the
  // whole range, and mode 2 is the ordinary pass with those maxima as the reference (so every
  // weight is at most 1 and none is clamped).
  if constexpr (F8) {
    for (int mode = 0; mode < 3; ++mode) {
      decode_pass_ool<F8, Q8>(maps, prm, sm, mode);
      if (!end_of_pass<F8>(mode, sm)) break;
    }
  } else {
    decode_pass<F8>(maps, prm, sm, 0);
    if (end_of_pass<F8>(0, sm)) replay_passes<F8>(maps, prm, sm);
  }

  // ---- teardown
  if (tid == 128) TRACE(10, 0);
  if (warp == 1) tmem_dealloc_pair(bars->tmem_base, 512);
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 2-D bf16 map over a [rows][576] row-major array, 64 x box_rows boxes, 128-byte swizzle.
static bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kCR, rows};
  cuuint64_t strides[1] = {(cuuint64_t)kCR * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D byte map over the FP8 pool, rows of `entry` bytes, box_bytes x box_rows boxes, no swizzle.
static bool make_map_u8(CUtensorMap* m, const void* base, uint64_t rows, uint32_t entry,
                        uint32_t box_bytes, uint32_t box_rows, bool swizzle128 = false) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)entry, rows};
  cuuint64_t strides[1] = {(cuuint64_t)entry};
  cuuint32_t box[2] = {box_bytes, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The plan: query rows sorted by decreasing visible length (a stable counting sort on the
// number of 256-token tiles, rows past kPlanBins - 1 tiles sharing the top bin), so that the
// longest rows start first. The order is a function of the lengths alone (equal keys keep
// their row order), so the rows that end up in the split tail, and with them every result,
// are the same on every call. The decode that follows reads q_lat from the kernel before this
// one, so this kernel waits for that kernel before it completes.
constexpr int kPlanBins = 1024;
__global__ void __launch_bounds__(1024) plan_order_kernel(const int32_t* __restrict__ seq_lens, int B, int n_q,
                                                          int max_seq_len, int32_t* __restrict__ order) {
  __shared__ int hist[kPlanBins];
  griddep_launch_dependents();
  const int rows = B * n_q, tid = threadIdx.x;
  auto key_of = [&](int r) {
    const int L = seq_lens[r / n_q];
    const int vis = (L < n_q || L > max_seq_len) ? 0 : L - n_q + r % n_q + 1;
    return min((vis + kTile - 1) / kTile, kPlanBins - 1);
  };
  hist[tid] = 0;
  __syncthreads();
  for (int r = tid; r < rows; r += blockDim.x) atomicAdd(&hist[key_of(r)], 1);
  __syncthreads();
  // start of bin k = rows in bins above k: an inclusive scan from the top bin down, shifted
  const int mine = hist[kPlanBins - 1 - tid];
  __syncthreads();
  hist[tid] = mine;   // hist[i] = count of bin kPlanBins - 1 - i
  __syncthreads();
  for (int off = 1; off < kPlanBins; off <<= 1) {
    const int add = tid >= off ? hist[tid - off] : 0;
    __syncthreads();
    hist[tid] += add;
    __syncthreads();
  }
  const int incl = hist[tid];
  __syncthreads();
  hist[kPlanBins - 1 - tid] = incl - mine;   // exclusive start of bin kPlanBins - 1 - tid
  __syncthreads();
  // scatter in row order by one warp, 32 rows per step: lanes with equal keys take
  // consecutive places in lane order, and one of them advances the bin's next place
  if (tid < 32) {
    for (int base = 0; base < rows; base += 32) {
      const int r = base + tid;
      const int k = r < rows ? key_of(r) : -1;
      const unsigned same = __match_any_sync(0xffffffffu, k);
      const int first = __ffs(same) - 1;
      const int rank = __popc(same & ((1u << tid) - 1u));
      int at = 0;
      if (tid == first && k >= 0) at = hist[k];
      at = __shfl_sync(0xffffffffu, at, first);
      if (k >= 0) order[at + rank] = r;
      __syncwarp();
      if (tid == first && k >= 0) hist[k] = at + __popc(same);
      __syncwarp();
    }
  }
  griddep_wait();
}

// Test hook state (mla_debug_decode_fault): the limit of every bounded wait and a latent
// chunk the bf16 kernel withholds.
static std::atomic<long long> g_wait_limit{0};
static std::atomic<int> g_withhold{-1};

static int pick_splits(int B, int n_q, int max_seq_len, int num_splits, int num_sms) {
  if (num_splits > 0) return num_splits;
  const int units = B * n_q;
  const int pairs = num_sms / 2;
  const int tiles = (max_seq_len + kTile - 1) / kTile;
  if (units * 4 >= pairs * 3) return 1;   // the batch alone fills >= 3/4 of the pairs
  int S = pairs / units;
  if (S > tiles) S = tiles;
  return S < 1 ? 1 : S;
}

}  // namespace tc

bool tc_supported(const Dims& d, int n_q) {
  return d.H == tc::kH && d.C == tc::kC && d.R == tc::kR && d.P == tc::kP &&
         d.act_dtype == MLA_BF16 && (d.cache_dtype == MLA_BF16 || d.cache_dtype == MLA_FP8_E4M3) &&
         n_q >= 1 && n_q <= 2;
}

// With more query rows than CTA pairs the pairs take rows in the order of a plan (a
// permutation of the rows by decreasing visible length, the longest-first rule for
// scheduling unequal jobs on identical machines), kept in the workspace after the partials.
static bool use_plan(int B, int n_q, int num_sms) { return B * n_q > num_sms / 2; }
static size_t plan_bytes(int B, int n_q, int num_sms) {
  return use_plan(B, n_q, num_sms) ? ((size_t)B * n_q * sizeof(int32_t) + 255) / 256 * 256 : 0;
}

// With one split and more rows than CTA pairs, the rows of the last, partly filled round of
// pairs (in the plan's order the shortest) are each split in two when that round would keep
// at most half of the pairs busy: their halves then take that round in half the time.
static int pick_tail(int B, int n_q, int num_splits, int S, int num_sms) {
  const int rows = B * n_q, pairs = num_sms / 2;
  if (num_splits > 0 || S != 1 || !use_plan(B, n_q, num_sms) || rows <= pairs) return 0;
  const int r = rows % pairs;
  return 2 * r <= pairs ? r : 0;
}

// fp32 partial outputs and log-sum-exps: every row's S ranges, or the tail rows' two halves
static size_t partial_bytes(const Dims& d, int B, int n_q, int S, int tail) {
  const size_t rows = S > 1 ? (size_t)B * n_q : (size_t)tail;
  const int n = S > 1 ? S : 2;
  if (rows == 0) return 0;
  return rows * d.H * n * ((size_t)d.C + 1) * sizeof(float);
}

size_t tc_workspace_bytes(const Dims& d, int B, int n_q, int max_seq_len, int num_splits,
                          int num_sms) {
  const int S = tc::pick_splits(B, n_q, max_seq_len, num_splits, num_sms);
  const int tail = pick_tail(B, n_q, num_splits, S, num_sms);
  const size_t part = (partial_bytes(d, B, n_q, S, tail) + 255) / 256 * 256;
  return part + plan_bytes(B, n_q, num_sms);
}

cudaError_t launch_decode_tc(const Dims& d, const void* q_lat, const void* pool, const int32_t* bt,
                             int maxp, int num_pages, const int32_t* seq_lens, int B, int n_q,
                             int max_seq_len, int num_splits, void* ws, size_t ws_bytes,
                             void* o_lat, float* lse, int32_t* status, cudaStream_t stream) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int S = tc::pick_splits(B, n_q, max_seq_len, num_splits, sms);
  const bool f8 = d.cache_dtype == MLA_FP8_E4M3;
  const uint64_t prow = (uint64_t)num_pages * d.P;
  tc::Maps maps;
  memset(&maps, 0, sizeof(maps));
  if (!tc::make_map(&maps.q, q_lat, (uint64_t)B * n_q * d.H, 64)) return cudaErrorInvalidValue;
  if (f8) {
    const uint32_t eb = (uint32_t)d.entry_bytes;   // 656: codes, bf16 RoPE keys, scales
    if (!tc::make_map_u8(&maps.cs, pool, prow, eb, 64, 64) ||
        !tc::make_map_u8(&maps.cv, pool, prow, eb, 64, 32) ||
        !tc::make_map_u8(&maps.ss, pool, prow, eb, 16, 64) ||
        !tc::make_map_u8(&maps.sv, pool, prow, eb, 16, 32) ||
        !tc::make_map_u8(&maps.kr, pool, prow, eb, 128, 64) ||
        (d.fp8_scores && !tc::make_map_u8(&maps.c8, pool, prow, eb, 128, 64, true)))
      return cudaErrorInvalidValue;
  } else {
    if (!tc::make_map(&maps.k, pool, prow, 64)) return cudaErrorInvalidValue;
    if (!tc::make_map(&maps.v, pool, prow, 32)) return cudaErrorInvalidValue;
  }
  static std::atomic<bool> attr_bf16[kMaxDevices], attr_f8[kMaxDevices], attr_q8[kMaxDevices];
  {
    cudaError_t e = !f8 ? set_smem_limit_once(tc::decode_kernel<false>, tc::kSmemBytes<false>, attr_bf16)
                    : d.fp8_scores ? set_smem_limit_once(tc::decode_kernel<true, true>, tc::kSmemBytes<true>, attr_q8)
                                   : set_smem_limit_once(tc::decode_kernel<true>, tc::kSmemBytes<true>, attr_f8);
    if (e != cudaSuccess) return e;
  }
  const int tail = pick_tail(B, n_q, num_splits, S, sms);
  const size_t prows = (S > 1 ? (size_t)B * n_q : (size_t)tail) * d.H;   // partial rows
  const int pn = S > 1 ? S : 2;                                         // partials per row
  const size_t part = (partial_bytes(d, B, n_q, S, tail) + 255) / 256 * 256;
  if (ws_bytes < part + plan_bytes(B, n_q, sms)) return cudaErrorInvalidValue;
  int32_t* order = use_plan(B, n_q, sms) ? reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + part) : nullptr;
  tc::Params prm;
  const long long lim = tc::g_wait_limit.load();
  prm.wait_limit = lim > 0 ? lim : tc::kTimeout;
  prm.withhold = tc::g_withhold.load();
  prm.bt = bt;
  prm.order = order;
  prm.pool = static_cast<const uint8_t*>(pool);
  prm.q8 = d.fp8_scores ? 1 : 0;
  prm.maxp = maxp;
  prm.num_pages = num_pages;
  prm.seq_lens = seq_lens;
  prm.B = B;
  prm.n_q = n_q;
  prm.max_seq_len = max_seq_len;
  prm.S = S;
  prm.tail = tail;
  prm.scale_log2 = d.scale * 1.4426950408889634f;
  prm.o_lat = static_cast<__nv_bfloat16*>(o_lat);
  prm.lse = lse;
  prm.ws_o = part ? static_cast<float*>(ws) : nullptr;
  prm.ws_lse = part ? static_cast<float*>(ws) + prows * pn * d.C : nullptr;
  prm.status = status;
#ifdef MLA_TC_TRACE
  prm.trace = static_cast<unsigned long long*>(tc::g_tc_trace_host);
#endif
  const unsigned grid = 2u * (unsigned)(B * n_q * S + tail);
  if (order) {
    cudaError_t e = launch_programmatic(tc::plan_order_kernel, dim3(1), dim3(1024), 0, stream, seq_lens, B,
                                        n_q, max_seq_len, order);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e =
      !f8 ? launch_programmatic(tc::decode_kernel<false>, dim3(grid), dim3(tc::Lay<false>::THREADS),
                                tc::kSmemBytes<false>, stream, maps, prm)
      : d.fp8_scores ? launch_programmatic(tc::decode_kernel<true, true>, dim3(grid), dim3(tc::Lay<true>::THREADS),
                                           tc::kSmemBytes<true>, stream, maps, prm)
                     : launch_programmatic(tc::decode_kernel<true>, dim3(grid), dim3(tc::Lay<true>::THREADS),
                                           tc::kSmemBytes<true>, stream, maps, prm);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess || (S == 1 && tail == 0)) return e;
  // the tail's partial row p belongs to query row order[rows - tail + p]
  return launch_combine(d.C, pn, prm.ws_o, prm.ws_lse, o_lat, MLA_BF16, lse, prows, stream,
                        S > 1 ? nullptr : order + (B * n_q - tail), d.H);
}

}  // namespace mla

extern "C" int mla_debug_decode_fault(long long wait_cycles, int withhold_chunk) {
  if (wait_cycles < 0 || withhold_chunk < -1) return MLA_ERR_INVALID_ARG;
  mla::tc::g_wait_limit.store(wait_cycles);
  mla::tc::g_withhold.store(withhold_chunk);
  return MLA_OK;
}

#ifdef MLA_TC_TRACE
extern "C" int mla_debug_set_tc_trace(void* p) {
  mla::tc::g_tc_trace_host = p;
  return 0;
}
#endif
