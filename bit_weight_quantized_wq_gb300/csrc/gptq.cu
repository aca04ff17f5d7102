// GPTQ sweep: INT4 g128 quantization column by column with inverse-Hessian error
// compensation (第 1 章：推理加速全景 §4.2; 推理优化与量化算子深度技术调研 §1.3).
//
// For column i = 0 .. K-1 of every weight row w:
//   at a group start (i % 128 == 0): scale and zero point of the group from the row's
//     current values of its 128 columns, by the INT4 g128 rules of the quantize kernel;
//   q_i = clamp(rint(w_i / s) + z, 0, 15),  w_hat_i = (q_i - z) s;
//   e_i = (w_i - w_hat_i) / U[i, i];   w_j := w_j - e_i U[i, j] for every j > i,
// with U the upper Cholesky factor of H^-1 (H^-1 = U^T U, H = 2 X^T X + lambda I), which the
// caller provides.  Each operation is rounded on its own (no contraction), so every code is
// reproducible bit for bit.
//
// Rows are independent: one CTA owns R rows and keeps their current values (fp32) and codes
// (one byte each) in shared memory for the whole sweep -- the pages' lazy block update exists
// to avoid re-streaming W, which residency in shared memory avoids altogether.  Per column:
// R threads take the decisions, then all threads apply the compensation to the later
// columns, reading row i of U once (coalesced) for all R rows.
#include "internal.h"

namespace wq {

namespace {

constexpr int kGptqThreads = 512;
constexpr int kGptqMaxRows = 8;
constexpr int kGptqSmem = 227 * 1024 - 1024;

__global__ void __launch_bounds__(kGptqThreads, 1)
    k_gptq_int4_g128(const float* __restrict__ W, int N, int K, int R, const float* __restrict__ U,
                     uint32_t* __restrict__ Wq, __half* __restrict__ scales, __half* __restrict__ zeros) {
  extern __shared__ __align__(16) uint8_t smem[];
  float* w = reinterpret_cast<float*>(smem);                                   // [R][K]
  uint8_t* code = smem + static_cast<size_t>(R) * K * sizeof(float);           // [R][K]
  __shared__ float s_err[kGptqMaxRows], s_scale[kGptqMaxRows], s_zero[kGptqMaxRows];

  const int row0 = blockIdx.x * R;
  const int rows = min(R, N - row0);
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int G = K / 128;

  for (int r = 0; r < rows; ++r) {
    const float4* src = reinterpret_cast<const float4*>(W + static_cast<long long>(row0 + r) * K);
    float4* dst = reinterpret_cast<float4*>(w + static_cast<size_t>(r) * K);
    for (int v = tid; v < K / 4; v += kGptqThreads) dst[v] = __ldg(src + v);
  }
  // U[i, i] of the current column, loaded one column ahead by the deciding threads
  float d_next = (tid < rows) ? __ldg(U) : 1.f;
  __syncthreads();

  for (int i = 0; i < K; ++i) {
    if ((i & 127) == 0) {
      // group parameters: warp r reduces row r's 128 current values
      if (warp < rows) {
        const float* x = w + static_cast<size_t>(warp) * K + i;
        float lo = 0.f, hi = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float v = x[lane + 32 * k];
          lo = fminf(lo, v);
          hi = fmaxf(hi, v);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
          hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
        }
        if (lane == 0) {
          const float s32 = __fdiv_rn(__fsub_rn(hi, lo), 15.0f);
          __half s16 = __float2half_rn(s32);
          if ((__half_as_ushort(s16) & 0x7fffu) == 0u) s16 = __ushort_as_half(0x3c00u);  // zero -> 1.0
          const float s = __half2float(s16);
          const int z = __float2int_rn(__fdiv_rn(-lo, s));
          s_scale[warp] = s;
          s_zero[warp] = static_cast<float>(z);
          const long long gi = static_cast<long long>(row0 + warp) * G + (i >> 7);
          scales[gi] = s16;
          zeros[gi] = __int2half_rn(z);
        }
      }
      __syncthreads();
    }
    if (tid < rows) {
      const float x = w[static_cast<size_t>(tid) * K + i];
      const float s = s_scale[tid], zf = s_zero[tid];
      float q = __fadd_rn(rintf(__fdiv_rn(x, s)), zf);
      q = fminf(fmaxf(q, 0.f), 15.f);
      code[static_cast<size_t>(tid) * K + i] = static_cast<uint8_t>(q);
      const float w_hat = __fmul_rn(__fsub_rn(q, zf), s);
      s_err[tid] = __fdiv_rn(__fsub_rn(x, w_hat), d_next);
      if (i + 1 < K) d_next = __ldg(U + static_cast<long long>(i + 1) * K + (i + 1));
    }
    __syncthreads();
    const float* Ui = U + static_cast<long long>(i) * K;
    for (int j = i + 1 + tid; j < K; j += kGptqThreads) {
      const float u = __ldg(Ui + j);
      for (int r = 0; r < rows; ++r) {
        float* p = w + static_cast<size_t>(r) * K + j;
        *p = __fsub_rn(*p, __fmul_rn(s_err[r], u));
      }
    }
    __syncthreads();
  }

  // pack: word j of row r holds codes 8j .. 8j+7, low nibble first
  for (int r = 0; r < rows; ++r) {
    const uint8_t* c = code + static_cast<size_t>(r) * K;
    uint32_t* out = Wq + static_cast<long long>(row0 + r) * (K / 8);
    for (int j = tid; j < K / 8; j += kGptqThreads) {
      uint32_t word = 0u;
#pragma unroll
      for (int k = 0; k < 8; ++k) word |= static_cast<uint32_t>(c[8 * j + k]) << (4 * k);
      out[j] = word;
    }
  }
}

}  // namespace

int gptq_rows_per_cta(int64_t K) {
  const int64_t per_row = K * 5;   // fp32 value + one code byte per column
  int64_t r = kGptqSmem / per_row;
  if (r > kGptqMaxRows) r = kGptqMaxRows;
  return static_cast<int>(r);
}

cudaError_t launch_gptq_int4_g128(const float* W, int64_t N, int64_t K, const float* U, int32_t* Wq,
                                  uint16_t* scales, uint16_t* zeros, cudaStream_t stream) {
  const int R = gptq_rows_per_cta(K);
  if (R < 1) return cudaErrorInvalidValue;
  const size_t smem = static_cast<size_t>(R) * K * 5;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(k_gptq_int4_g128, cudaFuncAttributeMaxDynamicSharedMemorySize, kGptqSmem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  const long long grid = (N + R - 1) / R;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  k_gptq_int4_g128<<<static_cast<unsigned>(grid), kGptqThreads, smem, stream>>>(
      W, static_cast<int>(N), static_cast<int>(K), R, U, reinterpret_cast<uint32_t*>(Wq),
      reinterpret_cast<__half*>(scales), reinterpret_cast<__half*>(zeros));
  return cudaGetLastError();
}

}  // namespace wq
