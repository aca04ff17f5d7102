// Diagnostic: exercises the bounded-wait path every kernel of the library relies on.  One CTA
// waits on an mbarrier phase that nothing completes; the wait gives up after its limit,
// records its code in the error word read by wq_read_error_flags and the kernel returns, so
// the context stays usable.  No fault, trap or endless loop is involved.
#include "internal.h"

namespace wq {

__device__ uint32_t g_selftest_err;

uint32_t selftest_read_and_clear_error() {
  uint32_t v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, g_selftest_err, sizeof(v));
  cudaMemcpyToSymbol(g_selftest_err, &z, sizeof(z));
  return v;
}

namespace {

__device__ uint32_t g_selftest_out;

__global__ void k_selftest_wait(uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  const bool ok = mbar_wait_for(&bar, 0, &g_selftest_err, kErrSelftestWait, limit_ns);   // nobody arrives
  if (threadIdx.x == 0) g_selftest_out = ok ? 0u : 1u;
}

}  // namespace

cudaError_t run_selftest_wait(uint64_t limit_ns, uint32_t* timed_out_host, cudaStream_t stream) {
  k_selftest_wait<<<1, 32, 0, stream>>>(limit_ns);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess)
    e = cudaMemcpyFromSymbolAsync(timed_out_host, g_selftest_out, sizeof(uint32_t), 0, cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  return e;
}

}  // namespace wq
