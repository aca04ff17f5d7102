// Quantize + pack kernels: asymmetric INT4 (group 128) and OCP MXFP4 (block 32).
//
// Both are one streaming pass over the float32 weights (4 B read, 0.53125 B written per
// weight), so they are HBM-bound: 128-bit loads, warp-shuffle reductions inside a group,
// packed stores.  The float32 operation sequence is fixed (IEEE round-to-nearest
// division/subtraction, no contraction) so that every code, scale and zero point is
// reproducible bit for bit.
#include "internal.h"
#include "mx_util.cuh"

namespace wq {

// ---------------------------------------------------------------------------------------
// INT4, group of 128 along K.  8 lanes per group, 16 consecutive floats per lane.
// 推理优化与量化算子深度技术调研 §1.2 / 第 1 章：推理加速全景 §4.1 with 2^4 - 1 = 15 levels.
// ---------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_quant_int4_g128(const float* __restrict__ W, int64_t groups,
                                                         int64_t groups_per_row,
                                                         uint32_t* __restrict__ Wq,
                                                         __half* __restrict__ scales,
                                                         __half* __restrict__ zeros) {
  const int64_t gid = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 3;  // group
  const uint32_t sub = threadIdx.x & 7u;                                                     // lane in group
  const bool active = gid < groups;
  const int64_t g = active ? gid : 0;

  float x[16];
  const float4* src = reinterpret_cast<const float4*>(W + g * 128 + sub * 16);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float4 v = active ? __ldcs(src + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    x[4 * i + 0] = v.x; x[4 * i + 1] = v.y; x[4 * i + 2] = v.z; x[4 * i + 3] = v.w;
  }
  // Range always contains 0 (so the zero point lands in [0, 15]).
  float lo = 0.f, hi = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) { lo = fminf(lo, x[i]); hi = fmaxf(hi, x[i]); }
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) {
    lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  }
  float s, zf;
  const __half s16 = int4_group_params(lo, hi, s, zf);

  // rint(x / s) with the IEEE quotient's rounding, from x times the correctly rounded 1/s:
  // that product is within 1.5 ulp of the quotient (|x / s| <= 16, ulp <= 2^-20), so both
  // round to the same integer unless the quotient is within 2^-17 of a rounding boundary
  // n + 1/2; there (rarely) the exact division decides.
  const float rs = __frcp_rn(s);
  uint32_t w0 = 0u, w1 = 0u;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float qa = __fmul_rn(x[i], rs);
    const float fr = qa - floorf(qa);
    const float qi = fabsf(fr - 0.5f) < 0x1p-17f ? rintf(__fdiv_rn(x[i], s)) : rintf(qa);
    float q = __fadd_rn(qi, zf);
    q = fminf(fmaxf(q, 0.f), 15.f);
    const uint32_t c = static_cast<uint32_t>(q);
    if (i < 8) w0 |= c << (4 * i);
    else w1 |= c << (4 * (i - 8));
  }
  if (active) {
    reinterpret_cast<uint2*>(Wq + g * 16)[sub] = make_uint2(w0, w1);
    if (sub == 0) {
      scales[g] = s16;
      zeros[g] = __float2half_rn(zf);
    }
  }
  (void)groups_per_row;
}

// ---------------------------------------------------------------------------------------
// MXFP4, block of 32 along K.  4 lanes per block, 8 consecutive floats per lane.
// ---------------------------------------------------------------------------------------

__global__ void __launch_bounds__(256) k_quant_mxfp4(const float* __restrict__ W, int64_t blocks,
                                                     uint32_t* __restrict__ Wq,
                                                     uint8_t* __restrict__ scales) {
  const int64_t bid = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 2;
  const uint32_t sub = threadIdx.x & 3u;
  const bool active = bid < blocks;
  const int64_t b = active ? bid : 0;

  float x[8];
  const float4* src = reinterpret_cast<const float4*>(W + b * 32 + sub * 8);
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    float4 v = active ? __ldcs(src + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    x[4 * i + 0] = v.x; x[4 * i + 1] = v.y; x[4 * i + 2] = v.z; x[4 * i + 3] = v.w;
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));

  const float r = __fdiv_rn(amax, 6.0f);
  int e = (r == 0.f) ? -127 : ceil_log2_pos(r);
  e = max(-127, min(127, e));
  const float inv = exp2_int(-e);

  // E2M1 by the hardware conversion (e2m1x2_rn): round to nearest, ties to the even code,
  // saturating at +-6, the sign kept (also on a zero); two values per instruction.
  uint32_t word = 0u;
  if (amax != 0.f) {
#pragma unroll
    for (int i = 0; i < 8; i += 2)
      word |= e2m1x2_rn(__fmul_rn(x[i + 1], inv), __fmul_rn(x[i], inv)) << (4 * i);
  }
  if (active) {
    Wq[b * 4 + sub] = word;
    if (sub == 0) scales[b] = (amax == 0.f) ? uint8_t(0) : static_cast<uint8_t>(e + 127);
  }
}

// ---------------------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------------------
cudaError_t launch_quant_int4_g128(const float* W, int64_t N, int64_t K, int32_t* Wq, uint16_t* scales,
                                   uint16_t* zeros, cudaStream_t stream) {
  const int64_t groups = N * (K / 128);
  const int64_t threads = groups * 8;
  const int block = 256;
  const int64_t grid = (threads + block - 1) / block;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  k_quant_int4_g128<<<static_cast<unsigned>(grid), block, 0, stream>>>(
      W, groups, K / 128, reinterpret_cast<uint32_t*>(Wq), reinterpret_cast<__half*>(scales),
      reinterpret_cast<__half*>(zeros));
  return cudaGetLastError();
}

cudaError_t launch_quant_mxfp4(const float* W, int64_t N, int64_t K, int32_t* Wq, uint8_t* scales,
                               cudaStream_t stream) {
  const int64_t blocks = N * (K / 32);
  const int64_t threads = blocks * 4;
  const int block = 256;
  const int64_t grid = (threads + block - 1) / block;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  k_quant_mxfp4<<<static_cast<unsigned>(grid), block, 0, stream>>>(W, blocks,
                                                                    reinterpret_cast<uint32_t*>(Wq), scales);
  return cudaGetLastError();
}

}  // namespace wq
