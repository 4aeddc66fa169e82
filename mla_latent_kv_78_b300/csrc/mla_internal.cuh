// Launchers shared between the C-ABI front end and the kernel files.
#pragma once

#include <atomic>

#include "mla_common.cuh"

namespace mla {

constexpr int kMaxDevices = 64;

// A kernel's dynamic shared-memory limit belongs to the device it runs on, so the attribute
// is set once per device: `done` is the call site's per-device record. Two host threads that
// race here both set the same value, which is harmless.
template <typename Kern>
cudaError_t set_smem_limit_once(Kern kernel, int bytes, std::atomic<bool> (&done)[kMaxDevices]) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kMaxDevices && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && dev >= 0 && dev < kMaxDevices) done[dev].store(true, std::memory_order_release);
  return e;
}

// Launch with programmatic stream serialization: the kernel may begin while the preceding
// kernel on `stream` is still running, so it must read no input before griddepcontrol.wait.
template <typename... KArgs, typename... Args>
cudaError_t launch_programmatic(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

cudaError_t launch_append(const Dims& d, const void* c_kv, const void* k_r, const int32_t* seq_idx,
                          const int32_t* pos, int T, const int32_t* bt, int batch, int maxp,
                          int num_pages, void* pool, int32_t* status, cudaStream_t stream);

cudaError_t launch_absorb(const Dims& d, const void* q_c, const void* q_r, const int32_t* pos,
                          int T, const void* w_uk, void* q_lat, cudaStream_t stream);

cudaError_t launch_unabsorb(const Dims& d, const void* o_lat, int T, const void* w_uv, float* o,
                            cudaStream_t stream);

// Tensor-core absorb / unabsorb (d_h = 128, d_c = 512, d_h^R = 64, bf16).
bool absorb_tc_supported(const Dims& d);
// early_inputs: launched right behind launch_append on the same stream (which writes none of
// q_c, q_r, pos, w_uk); the inputs are then read before the append has completed.
cudaError_t launch_absorb_tc(const Dims& d, const void* q_c, const void* q_r, const int32_t* pos,
                             int T, const void* w_uk, void* q_lat, cudaStream_t stream,
                             bool early_inputs = false);
cudaError_t launch_unabsorb_tc(const Dims& d, const void* o_lat, int T, const void* w_uv, float* o,
                               cudaStream_t stream);

// Generic CUDA-core decode: grid (H, n_q, B * S). With S > 1 it writes
// normalised partials to the workspace and a combine kernel merges them.
size_t simt_workspace_bytes(const Dims& d, int B, int n_q, int S);
int simt_pick_splits(const Dims& d, int B, int n_q, int max_seq_len, int num_splits, int num_sms);
cudaError_t launch_decode_simt(const Dims& d, const void* q_lat, const void* pool,
                               const int32_t* bt, int maxp, int num_pages, const int32_t* seq_lens,
                               int B, int n_q, int max_seq_len, int S, void* ws, void* o_lat,
                               float* lse, int32_t* status, cudaStream_t stream);

// Log-sum-exp merge of split partials ws_o [rows][S][C], ws_lse [rows][S] into o_lat, lse.
// Partial row r goes to output row r, or with row_of to head r % H of query row row_of[r / H].
cudaError_t launch_combine(int C, int S, const float* ws_o, const float* ws_lse, void* o_lat,
                           int act_dtype, float* lse, size_t rows, cudaStream_t stream,
                           const int32_t* row_of = nullptr, int H = 1);

// Tensor-core projection Y = X . W^T (X [T][K], W [N][K] bf16; K a multiple of 8). Y is fp32 or
// bf16 (out_dtype); kGemmPartials leaves the fp32 split partials [splits][T][N] in `part`.
constexpr int kGemmPartials = -1;
int gemm_pick_splits(int T, int N, int K, int num_sms);
size_t gemm_workspace_bytes(int T, int N, int K, int out_dtype, int num_sms);
cudaError_t launch_gemm(const void* x, const void* w, int T, int N, int K, int splits, float* part,
                        void* y, int out_dtype, int32_t* status, cudaStream_t stream);

// Fused upstream append: [W^{DKV}; W^{KR}] h as split partials in ws, then RMSNorm, RoPE and the
// cache write in one epilogue kernel.
cudaError_t launch_project_append(const Dims& d, const void* h, int d_model, const void* w, int T,
                                  const float* gain, float eps, const int32_t* seq_idx,
                                  const int32_t* pos, const int32_t* bt, int batch, int maxp,
                                  int num_pages, void* pool, void* ws, int splits, int32_t* status,
                                  cudaStream_t stream);

// Non-absorbed prefill (K^C, V^C by the projection GEMM, causal tcgen05 attention).
bool prefill_supported(const Dims& d);
size_t prefill_workspace_bytes(const Dims& d, int L);
cudaError_t launch_prefill(const Dims& d, const void* c_kv, const void* k_r, int L, const void* q_c,
                           const void* q_r, const void* w_uk, const void* w_uv, float* o, void* ws,
                           int32_t* status, cudaStream_t stream);

// Tensor-core decode (tcgen05 + TMEM + TMA), V2 head shapes only.
bool tc_supported(const Dims& d, int n_q);
size_t tc_workspace_bytes(const Dims& d, int B, int n_q, int max_seq_len, int num_splits,
                          int num_sms);
cudaError_t launch_decode_tc(const Dims& d, const void* q_lat, const void* pool, const int32_t* bt,
                             int maxp, int num_pages, const int32_t* seq_lens, int B, int n_q,
                             int max_seq_len, int num_splits, void* ws, size_t ws_bytes,
                             void* o_lat, float* lse, int32_t* status, cudaStream_t stream);

// FP8 cache staged to bf16 (every visible token converted once into the workspace), then the
// bf16 tensor-core decode over the staged pool. The workspace holds fp8_staged_bytes() first,
// then the bf16 decode's own workspace.
size_t fp8_staged_bytes(int B, int max_seq_len);
cudaError_t launch_decode_tc_fp8_staged(const Dims& d, const void* q_lat, const void* pool,
                                        const int32_t* bt, int maxp, int num_pages,
                                        const int32_t* seq_lens, int B, int n_q, int max_seq_len,
                                        int num_splits, void* ws, size_t ws_bytes, void* o_lat,
                                        float* lse, int32_t* status, cudaStream_t stream);

}  // namespace mla
