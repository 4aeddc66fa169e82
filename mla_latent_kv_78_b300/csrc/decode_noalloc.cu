// mla_decode_noalloc: mla_decode for callers that cannot allocate device memory.
//
// Some hosts of this library hand it only the tensors they own and give it no way to obtain
// more device memory: an inference server's plugin interface whose memory pool is managed
// elsewhere, a process that must not let a library call into cudaMalloc (which may block on the
// device or fail under memory pressure in the middle of a decode loop), or a caller from a
// runtime with no CUDA allocator binding at all. For them the decode's scratch (the split-KV
// partial outputs and log-sum-exps, which the decode needs only when it spreads a query row over
// several CTA pairs) lives in a fixed array that is part of this library's device image: every
// GPU that loads the library holds it until the process exits.
#include <cuda.h>
#include <mutex>

#include "mla_internal.cuh"

namespace {

constexpr size_t kScratchBytes = MLA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDev = 64;

// The scratch itself. Host code never touches it by name: its device address is looked up per
// device below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

// The driver's cuCtxGetCurrent, reached through the runtime (no link to libcuda needed).
CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<CtxGetCurrentFn>(p);
  }();
  return fn;
}

std::mutex g_setup_mu;
struct ScratchEntry {
  CUcontext ctx;   // the context the address belongs to
  void* addr;
};
ScratchEntry g_scratch[kMaxDev] = {};

// Device address of the scratch in the current device's context. It is looked up on the first
// call in a context and again whenever the context has changed since (a device reset tears
// down the context the cached address belonged to).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return MLA_ERR_CUDA;
  CtxGetCurrentFn get = ctx_get_current();
  if (!get) return MLA_ERR_CUDA;
  CUcontext ctx = nullptr;
  if (get(&ctx) != CUDA_SUCCESS) return MLA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  ScratchEntry& e = g_scratch[dev];
  if (!ctx || !e.addr || e.ctx != ctx) {
    // (the lookup also makes the device's primary context current if none was yet)
    void* p = nullptr;
    const cudaError_t rc = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (rc != cudaSuccess || !p) return MLA_ERR_CUDA;
    if (get(&ctx) != CUDA_SUCCESS || !ctx) return MLA_ERR_CUDA;
    e.ctx = ctx;
    e.addr = p;
  }
  *out = e.addr;
  return MLA_OK;
}

}  // namespace

extern "C" int mla_decode_noalloc(const mla_config* cfg, const void* q_lat, const void* kv_pool,
                                  const int32_t* block_table, int32_t max_pages_per_seq,
                                  int32_t num_pages, const int32_t* seq_lens, int32_t batch,
                                  int32_t n_q, int32_t max_seq_len, int32_t num_splits, void* o_lat,
                                  float* lse, int32_t* dev_status, void* stream) {
  if (batch > 0 && n_q >= 1 && max_seq_len >= 1 && num_splits >= 0) {
    const size_t need = mla_decode_workspace_size(cfg, batch, n_q, max_seq_len, num_splits);
    if (need > kScratchBytes) return MLA_ERR_SCRATCH_LIMIT;
  }
  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != MLA_OK) return rc;
  return mla_decode(cfg, q_lat, kv_pool, block_table, max_pages_per_seq, num_pages, seq_lens, batch,
                    n_q, max_seq_len, num_splits, scratch, kScratchBytes, o_lat, lse, dev_status,
                    stream);
}
