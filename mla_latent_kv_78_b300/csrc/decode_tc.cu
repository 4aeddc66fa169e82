// Tensor-core MLA decode (tcgen05 / TMEM / TMA) — not yet enabled.
#include "mla_internal.cuh"

namespace mla {

bool tc_supported(const Dims&, int) { return false; }

size_t tc_workspace_bytes(const Dims&, int, int, int, int, int) { return 0; }

cudaError_t launch_decode_tc(const Dims&, const void*, const void*, const int32_t*, int, int,
                             const int32_t*, int, int, int, int, void*, size_t, void*, float*,
                             int32_t*, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace mla
