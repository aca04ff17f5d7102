// MXFP4 quantization helpers shared by the weight quantizer (quantize.cu) and the W4A4
// activation quantizer (w4a4.cu): the block's E8M0 exponent from the IEEE fields of
// amax / 6 and the E2M1 codes by round-to-nearest-even onto the grid.
#pragma once

#include "common.cuh"

namespace wq {

// ceil(log2 r) for a positive finite float, exact, from the IEEE fields.
__device__ __forceinline__ int ceil_log2_pos(float r) {
  const uint32_t b = __float_as_uint(r);
  const int ex = static_cast<int>((b >> 23) & 0xffu);
  const uint32_t man = b & 0x7fffffu;
  if (ex != 0) return (ex - 127) + (man != 0u ? 1 : 0);
  // subnormal: r = man * 2^-149
  const int p = 31 - __clz(static_cast<int>(man));       // highest set bit
  return (p - 149) + ((man & (man - 1u)) != 0u ? 1 : 0);
}

// 2^f for f in [-127, 127] as a float (2^-127 is subnormal).
__device__ __forceinline__ float exp2_int(int f) {
  return f >= -126 ? __uint_as_float(static_cast<uint32_t>(f + 127) << 23) : __uint_as_float(0x00400000u);
}

// Two floats to a byte of E2M1 codes (hi in bits 4-7, lo in bits 0-3), sign kept (also on a
// zero): the nearest of the grid {0, .5, 1, 1.5, 2, 3, 4, 6} in magnitude, a tie (0.25, 0.75,
// 1.25, 1.75, 2.5, 3.5, 5) to the even code, saturating at +-6 (cvt.rn.satfinite.e2m1x2.f32).
__device__ __forceinline__ uint32_t e2m1x2_rn(float hi, float lo) {
  uint16_t d;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u16.u8 %0, t;\n\t}"
      : "=h"(d)
      : "f"(hi), "f"(lo));
  return d;
}

}  // namespace wq
