// Row re-layout of the stacked gate+up weight for the SwiGLU epilogue.
//
// 推理优化与量化算子深度技术调研 §4.6 stacks the two projections as [W_gate; W_up] and runs
// them as one GEMM whose epilogue applies SiLU(gate) * up in registers.  For that, the
// kernels need gate row j and up row j in one thread's accumulators.  Both kernels hold rows
// r and r + 8 of a 16-row block in one thread (decode: the two row halves of an m16n8k16
// fragment; prefill: TMEM lanes l and l ^ 8 of one warp), so the weight is stored with gate
// and up rows alternating in blocks of 8:
//   interleaved row 16 q + 8 h + i  <-  stacked row h F + 8 q + i      (h = 0 gate, 1 up)
// A permutation of whole rows, done once offline -- the weight re-layout step of
// 第 6 课：量化源码走读 §2 -- and applied alike to the packed codes and their scales / zeros
// (quantization is row-wise, so it commutes with the permutation).
#include "internal.h"

namespace wq {

namespace {

__device__ __forceinline__ long long stacked_row(long long r, long long F) {
  const long long q = r >> 4, h = (r >> 3) & 1, i = r & 7;
  return h * F + 8 * q + i;
}

// One CTA per destination row (grid-stride); 16-byte copies when rows are 16-byte multiples
// and both bases are 16-byte aligned, bytes otherwise.
__global__ void __launch_bounds__(256) k_interleave_rows(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                                                         long long F, long long row_bytes, int vec16) {
  const long long rows = 2 * F;
  for (long long r = blockIdx.x; r < rows; r += gridDim.x) {
    const uint8_t* s = src + stacked_row(r, F) * row_bytes;
    uint8_t* d = dst + r * row_bytes;
    if (vec16) {
      const long long nv = row_bytes >> 4;
      for (long long v = threadIdx.x; v < nv; v += blockDim.x)
        reinterpret_cast<uint4*>(d)[v] = __ldg(reinterpret_cast<const uint4*>(s) + v);
    } else {
      for (long long b = threadIdx.x; b < row_bytes; b += blockDim.x) d[b] = s[b];
    }
  }
}

}  // namespace

cudaError_t launch_interleave_gate_up(const void* src, void* dst, int64_t F, int64_t row_bytes, cudaStream_t stream) {
  const bool vec16 = row_bytes % 16 == 0 && (reinterpret_cast<uintptr_t>(src) & 15u) == 0 &&
                     (reinterpret_cast<uintptr_t>(dst) & 15u) == 0;
  const long long rows = 2 * static_cast<long long>(F);
  const long long cap = static_cast<long long>(device_sm_count()) * 16;
  const unsigned grid = static_cast<unsigned>(rows < cap ? rows : cap);
  k_interleave_rows<<<grid, 256, 0, stream>>>(static_cast<const uint8_t*>(src), static_cast<uint8_t*>(dst), F,
                                              row_bytes, vec16 ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace wq
