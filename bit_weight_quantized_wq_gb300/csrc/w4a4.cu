// W4A4 in MXFP4 (第 6 课：量化源码走读, micro-scaling: weights and activations both in 4-bit
// E2M1 with one E8M0 scale per 32-element block; the activations quantized on the fly) on the
// FP8 tensor-core path of gemm_fp8.cu.
//
// Every MXFP4 value E2M1(c) * 2^e has at most two significant bits, so relative to a row
// reference 2^E it is exactly an E4M3 value E2M1(c) * 2^(e - E) whenever e - E lies in
// [-8, 6] (E4M3 spans 2^-9 .. 448; 6 * 2^6 = 384).  With E = (largest block exponent of the
// row) - 6, every block within 14 binades of the row's largest is re-encoded exactly; a block
// further below rounds to E4M3 (and to zero beyond 2^-13 of the row's largest block).  The
// row's 2^E becomes the per-row scale of the FP8 GEMM, whose epilogue applies 2^(Ex + Ew).
//   * weights: MXFP4-packed ([N, K/2] codes + [N, K/32] E8M0) -> E4M3 [N, K] + 2^E [N], once;
//   * activations: bf16 [M, K] -> MXFP4 by exactly the weight quantizer's rules (block amax,
//     E8M0 exponent from the IEEE fields, E2M1 by the grid's midpoints) -> E4M3 [M, K] + 2^E [M]
//     in one kernel, one CTA per token row.
#include "internal.h"
#include "mx_util.cuh"

namespace wq {
namespace w4 {

constexpr int kThreads = 256;
constexpr int kMaxBlocks = 4096;           // 32-element blocks per row (K <= 131072)
constexpr int kMinShift = -20;             // below 2^-13 of the row's largest block: E4M3 zero

__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}

// Value of an E2M1 code (sign bit 3), exact.
__device__ __forceinline__ float e2m1_value(uint32_t c) {
  const uint32_t m = c & 7u;
  const float mag = m < 2u ? 0.5f * static_cast<float>(m)
                           : ((m & 1u) ? 1.5f : 1.0f) * static_cast<float>(1u << ((m >> 1) - 1u));
  return (c & 8u) ? -mag : mag;
}

// 2^d as a float for d in [kMinShift, 6].
__device__ __forceinline__ float pow2_small(int d) {
  return __uint_as_float(static_cast<uint32_t>(d + 127) << 23);
}

// 2^e as a float for e in [-149, 127] (subnormal below -126).
__device__ __forceinline__ float pow2_any(int e) {
  return e >= -126 ? __uint_as_float(static_cast<uint32_t>(e + 127) << 23) : __uint_as_float(1u << (e + 149));
}

// E2M1 code pair -> fp16 pair (exact), fp16 pair times fp16 pair, fp16 pair -> E4M3 codes.
__device__ __forceinline__ uint32_t e2m1x2_f16x2(uint32_t byte) {
  uint32_t d;
  const unsigned short h = static_cast<unsigned short>(byte);
  asm("{\n\t.reg .b8 t, u;\n\tmov.b16 {t, u}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(d) : "h"(h));
  return d;
}
__device__ __forceinline__ uint32_t hmul2_bits(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t f16x2_e4m3x2(uint32_t h2) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(d) : "r"(h2));
  return d;
}

__device__ __forceinline__ int block_max_int(int v, int* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    v = lane < kThreads / 32 ? red[lane] : -1000;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (lane == 0) red[0] = v;
  }
  __syncthreads();
  return red[0];
}

// Eight E2M1 codes (one 32-bit word, element i in bits 4i..4i+3) of a block with exponent
// e, re-encoded against the row reference E: two words of E4M3 codes.
__device__ __forceinline__ uint2 reencode8(uint32_t word, int e, int E, bool zero_block) {
  int d = e - E;
  if (d < kMinShift) d = kMinShift;
  const float f = zero_block ? 0.f : pow2_small(d);
  uint32_t c[4];
#pragma unroll
  for (int q = 0; q < 4; ++q)
    c[q] = e4m3x2(e2m1_value((word >> (8 * q)) & 0xfu) * f, e2m1_value((word >> (8 * q + 4)) & 0xfu) * f);
  return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

// Weights: one CTA per row of the MXFP4-packed weight.
__global__ void __launch_bounds__(kThreads) k_mx_weights_to_e4m3(const uint32_t* __restrict__ Wq,
                                                                 const uint8_t* __restrict__ scales, int64_t K,
                                                                 uint8_t* __restrict__ W8, float* __restrict__ sw) {
  __shared__ int red[kThreads / 32];
  const int64_t n = blockIdx.x;
  const int64_t nb = K / 32;
  const uint8_t* srow = scales + n * nb;
  // a block's E8M0 byte is its exponent + 127 (0 for an all-zero block, whose codes are all
  // zero and re-encode to zero against any reference)
  int mx = -1000;
  for (int64_t b = threadIdx.x; b < nb; b += kThreads) mx = max(mx, static_cast<int>(srow[b]) - 127);
  const int E = block_max_int(mx, red) - 6;
  const uint32_t* wrow = Wq + n * (K / 8);
  uint8_t* orow = W8 + n * K;
  for (int64_t w = threadIdx.x; w < K / 8; w += kThreads) {
    *reinterpret_cast<uint2*>(orow + 8 * w) = reencode8(__ldg(wrow + w), static_cast<int>(srow[w / 4]) - 127, E, false);
  }
  if (threadIdx.x == 0) sw[n] = pow2_any(E);
}

// Activations: one CTA per token row, bf16 in.  Pass 1 finds every block's exponent (kept in
// shared memory) and the row's largest; pass 2 quantizes each block to E2M1 and re-encodes.
__global__ void __launch_bounds__(kThreads) k_quant_w4a4_act(const uint16_t* __restrict__ X, int64_t K,
                                                             uint8_t* __restrict__ X8, float* __restrict__ sx) {
  __shared__ int red[kThreads / 32];
  __shared__ int8_t be[kMaxBlocks];          // block exponent + 0 (zero block: -128)
  const int64_t m = blockIdx.x;
  const int64_t nb = K / 32;
  const uint16_t* xrow = X + m * K;
  pdl_launch_dependents();
  pdl_wait();                                // X may come from the previous kernel of the stream
  int mx = -1000;
  for (int64_t b = threadIdx.x; b < nb; b += kThreads) {
    const uint4* src = reinterpret_cast<const uint4*>(xrow + 32 * b);
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 v = __ldg(src + i);
      const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q)
        amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w4[q] << 16)), fabsf(__uint_as_float(w4[q] & 0xffff0000u))));
    }
    int e = -128;
    if (amax != 0.f) {
      const float r = __fdiv_rn(amax, 6.0f);
      e = r == 0.f ? -127 : max(-127, min(127, ceil_log2_pos(r)));
      mx = max(mx, e);
    }
    be[b] = static_cast<int8_t>(e);
  }
  const int emax = block_max_int(mx, red);   // (its barriers also publish be[])
  const int E = emax == -1000 ? 0 : emax - 6;
  uint8_t* orow = X8 + m * K;
  for (int64_t b = threadIdx.x; b < nb; b += kThreads) {
    const int e = be[b];
    const uint4* src = reinterpret_cast<const uint4*>(xrow + 32 * b);
    const float inv = exp2_int(-(e == -128 ? 0 : e));
    // 2^(e - E) as an fp16 pair (d >= kMinShift = -20: at least 2^-20, an exact fp16); an
    // E2M1 value times it has at most two significant bits and stays >= 2^-21, so the fp16
    // product is exact and its E4M3 rounding is that of the value itself
    int d = e - E;
    if (d < kMinShift) d = kMinShift;
    const uint32_t f1 = __half_as_ushort(__float2half_rn(pow2_small(d)));
    const uint32_t f2 = f1 | (f1 << 16);
#pragma unroll
    for (int i = 0; i < 4; ++i) {               // 8 elements per 16-byte load
      const uint4 v = __ldg(src + i);
      const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
      uint32_t c[4] = {0u, 0u, 0u, 0u};         // a zero block (e = -128) is all +0 codes
      if (e != -128) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float x0 = __uint_as_float(w4[q] << 16), x1 = __uint_as_float(w4[q] & 0xffff0000u);
          // E2M1 of x 2^-e: round to nearest, ties to the even code, saturating at +-6, sign
          // kept; then re-encoded against the row's 2^E
          const uint32_t codes = e2m1x2_rn(__fmul_rn(x1, inv), __fmul_rn(x0, inv));
          c[q] = f16x2_e4m3x2(hmul2_bits(e2m1x2_f16x2(codes), f2));
        }
      }
      *reinterpret_cast<uint2*>(orow + 32 * b + 8 * i) = make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
    }
  }
  if (threadIdx.x == 0) sx[m] = pow2_any(E);
}

}  // namespace w4

cudaError_t launch_mx_weights_to_e4m3(const int32_t* Wq, const uint8_t* scales, int64_t N, int64_t K, uint8_t* W8,
                                      float* sw, cudaStream_t stream) {
  if (N < 1 || K < 32 || K % 32 != 0 || N > 0x7fffffffLL) return cudaErrorInvalidValue;
  w4::k_mx_weights_to_e4m3<<<static_cast<unsigned>(N), w4::kThreads, 0, stream>>>(
      reinterpret_cast<const uint32_t*>(Wq), scales, K, W8, sw);
  return cudaGetLastError();
}

cudaError_t launch_quant_w4a4_act(const uint16_t* X, int64_t M, int64_t K, uint8_t* X8, float* sx,
                                  cudaStream_t stream) {
  if (M < 1 || K < 32 || K % 32 != 0 || K / 32 > w4::kMaxBlocks || M > 0x7fffffffLL) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(M));
  cfg.blockDim = dim3(w4::kThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, w4::k_quant_w4a4_act, X, K, X8, sx);
}

}  // namespace wq
