// Declarations shared between the C-ABI layer (api.cu) and the kernel translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace wq {

// Format codes (same values as wq_fmt in include/wq.h).
enum Fmt : int { kInt4G128 = 0, kMxfp4 = 1 };

// Epilogue of the linear layer.  kEpiSwiglu: the weight is the fused gate+up projection of
// 2F rows with gate and up rows interleaved in blocks of 8 (row 16q + i is gate row 8q + i,
// row 16q + 8 + i the matching up row), and the kernel writes Y[M, F] = SiLU(gate) * up,
// applied to the fp32 accumulators before the one bf16 rounding.  kEpiSplit3: the output
// columns go to three tensors by column range (OutSplit), e.g. the Q, K and V of a fused QKV
// projection.
enum Epi : int { kEpiNone = 0, kEpiSwiglu = 1, kEpiSplit3 = 2 };

// Three row-major bf16 output tensors by column range: column n < n1 goes to
// y[0][m * ld[0] + n], n1 <= n < n2 to y[1][m * ld[1] + n - n1], n >= n2 to y[2][m * ld[2] + n - n2].
struct OutSplit {
  uint16_t* y[3];
  long long ld[3];
  int n1, n2;
};

__device__ __forceinline__ void store_split3(const OutSplit& s, int m, int n, uint16_t v) {
  if (n < s.n1) s.y[0][static_cast<long long>(m) * s.ld[0] + n] = v;
  else if (n < s.n2) s.y[1][static_cast<long long>(m) * s.ld[1] + (n - s.n1)] = v;
  else s.y[2][static_cast<long long>(m) * s.ld[2] + (n - s.n2)] = v;
}

// Encodes a 2-D tiled TMA descriptor through the driver entry point (no libcuda link).
// dims/strides in elements/bytes, innermost first.
cudaError_t make_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t dim0,
                         uint64_t dim1, uint64_t stride1_bytes, uint32_t box0, uint32_t box1,
                         CUtensorMapSwizzle swizzle, CUtensorMapL2promotion promo);

int device_sm_count();

// The calling thread's current CUDA context (driver entry point, no libcuda link), or
// nullptr when none is current or the entry point is unavailable.
CUcontext current_context();

// Raises a kernel's dynamic shared-memory limit on the current device, once per (kernel,
// device); thread-safe.
cudaError_t set_smem_attr_once(const void* kern, size_t smem_bytes);

// Every workspace layout starts with the same fixed header:
//   [0, kWsCounterBytes)               split-K counters of the tensor-core kernel's split
//                                      last-wave tiles
//   [kWsCounterBytes, kWsHeaderBytes)  the decode kernel's split-K exchange area (tagged
//                                      partial sums: at most two tiles for each of 160 CTAs,
//                                      32 rows x 256 columns of 4 bytes each)
// and the tensor-core kernel's other scratch follows it.  Every call that completes leaves
// the header at zero, so one workspace zeroed once can be shared by calls of any shape and
// by both kernels.
constexpr size_t kWsCounterBytes = 64 * 1024;
constexpr int64_t kWsMaxCounters = kWsCounterBytes / 4;
constexpr size_t kWsDecodeBytes = static_cast<size_t>(2) * 160 * 32 * 256 * 4;
constexpr size_t kWsHeaderBytes = kWsCounterBytes + kWsDecodeBytes;
// The decode entry points accept N <= kWsMaxCounters * kDecodeBand (2097152 weight rows).
constexpr int64_t kDecodeBand = 128;
// Activation rows the decode kernel accepts (tiles of 8, 16, 32 or 64 rows).
constexpr int64_t kDecodeMaxM = 64;

// quantize.cu
cudaError_t launch_quant_int4_g128(const float* W, int64_t N, int64_t K, int32_t* Wq, uint16_t* scales,
                                   uint16_t* zeros, cudaStream_t stream);
cudaError_t launch_quant_mxfp4(const float* W, int64_t N, int64_t K, int32_t* Wq, uint8_t* scales,
                               cudaStream_t stream);

// gemv.cu -- decode kernel, M <= 16
size_t gemv_workspace_bytes(int fmt, int64_t M, int64_t K, int64_t N);
cudaError_t launch_gemv(int fmt, const uint16_t* X, int64_t M, int64_t K, int64_t N, const int32_t* Wq,
                        const void* scales, const uint16_t* zeros, uint16_t* Y, void* ws, size_t ws_bytes,
                        cudaStream_t stream, int epi = kEpiNone, const OutSplit* split = nullptr);
uint32_t gemv_read_and_clear_error();
size_t gemv_noalloc_scratch_bytes();
cudaError_t launch_gemv_noalloc(int fmt, const uint16_t* X, int64_t M, int64_t K, int64_t N, const int32_t* Wq,
                                const void* scales, const uint16_t* zeros, uint16_t* Y, cudaStream_t stream);


// gemm_tc.cu -- tcgen05 kernel, any M
size_t gemm_tc_workspace_bytes(int fmt, int64_t M, int64_t K, int64_t N);
cudaError_t launch_gemm_tc(int fmt, const uint16_t* X, int64_t M, int64_t K, int64_t N, const int32_t* Wq,
                           const void* scales, const uint16_t* zeros, uint16_t* Y, void* ws, size_t ws_bytes,
                           cudaStream_t stream, int epi = kEpiNone, const OutSplit* split = nullptr);
uint32_t gemm_tc_read_and_clear_error();

// gptq.cu -- GPTQ sweep (INT4 g128) with a caller-provided inverse-Hessian Cholesky factor
int gptq_rows_per_cta(int64_t K);
uint32_t gptq_read_and_clear_error();
cudaError_t launch_gptq_int4_g128(const float* W, int64_t N, int64_t K, const float* U, int32_t* Wq,
                                  uint16_t* scales, uint16_t* zeros, cudaStream_t stream);

// gptq_factor.cu -- U (H^-1 = U^T U, H = 2 X^T X + lambda I) from calibration activations, float64
size_t gptq_factor_workspace_bytes(int64_t K);
cudaError_t launch_gptq_factor(const float* X, int64_t n, int64_t K, float* U, void* ws, cudaStream_t stream);
uint32_t gptq_factor_read_and_clear_error();

// awq.cu -- AWQ scale search + INT4 g128 quantize of the scaled weight
size_t awq_workspace_bytes(int64_t N, int64_t K, int64_t n);
cudaError_t launch_awq_int4_g128(const float* W, int64_t N, int64_t K, const float* X, int64_t n, int32_t* Wq,
                                 uint16_t* scales, uint16_t* zeros, float* s_out, int32_t* a_out, double* losses_out,
                                 void* ws, size_t ws_bytes, cudaStream_t stream);

// selftest.cu -- the bounded-wait path, exercised on demand
uint32_t selftest_read_and_clear_error();

// FP8 E4M3 W8A8 (gemm_fp8.cu): per-row quantization (fp32 weights or bf16 activations) and
// the GEMM with per-token and per-channel scales in the epilogue.
cudaError_t launch_quant_fp8_rows(bool bf16_in, const void* in, int64_t R, int64_t K, uint8_t* Q, float* scales,
                                  cudaStream_t stream);
cudaError_t launch_gemm_fp8(const uint8_t* Xq, const float* sx, int64_t M, int64_t K, int64_t N, const uint8_t* Wq,
                            const float* sw, uint16_t* Y, cudaStream_t stream);
uint32_t fp8_read_and_clear_error();

// W4A4 MXFP4 on the FP8 path (w4a4.cu): MXFP4 weights re-encoded as E4M3 against a per-row
// power of two; bf16 activations quantized to MXFP4 and re-encoded the same way.
cudaError_t launch_mx_weights_to_e4m3(const int32_t* Wq, const uint8_t* scales, int64_t N, int64_t K, uint8_t* W8,
                                      float* sw, cudaStream_t stream);
cudaError_t launch_quant_w4a4_act(const uint16_t* X, int64_t M, int64_t K, uint8_t* X8, float* sx,
                                  cudaStream_t stream);
cudaError_t run_selftest_wait(uint64_t limit_ns, uint32_t* timed_out_host, cudaStream_t stream);

// layout.cu -- row re-layout of the stacked gate+up weight
cudaError_t launch_interleave_gate_up(const void* src, void* dst, int64_t F, int64_t row_bytes, cudaStream_t stream);

}  // namespace wq
