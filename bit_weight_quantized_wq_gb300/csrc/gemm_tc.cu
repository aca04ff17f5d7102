// Prefill kernel (tcgen05 / TMEM tensor cores): under construction.
#include "internal.h"

namespace wq {

__device__ uint32_t g_gemm_err;

uint32_t gemm_tc_read_and_clear_error() {
  uint32_t v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, g_gemm_err, sizeof(v));
  cudaMemcpyToSymbol(g_gemm_err, &z, sizeof(z));
  return v;
}

size_t gemm_tc_workspace_bytes(int, int64_t, int64_t, int64_t) { return 0; }

cudaError_t launch_gemm_tc(int, const uint16_t*, int64_t, int64_t, int64_t, const int32_t*, const void*,
                           const uint16_t*, uint16_t*, void*, size_t, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace wq
