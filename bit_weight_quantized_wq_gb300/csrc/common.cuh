// Shared device helpers for the sm_103a kernels: mbarriers, TMA, bounded waits, errors.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

namespace wq {

// ---------------------------------------------------------------------------------------
// Error word: every bounded wait that runs out ORs a code in here and its kernel returns.
// One word per translation unit that waits (see wq_read_error_flags in api.cu).
// ---------------------------------------------------------------------------------------
enum : uint32_t {
  kErrWaitFull = 1u << 0,     // consumer gave up waiting for a filled stage
  kErrWaitEmpty = 1u << 1,    // producer gave up waiting for a free stage
  kErrWaitAccum = 1u << 2,    // epilogue gave up waiting for the accumulator
  kErrWaitReduce = 1u << 3,   // split-K reduction gave up
  kErrDrain = 1u << 4,        // TMA drain at exit gave up
  kErrSelftestWait = 1u << 5, // the diagnostic wait of wq_selftest_wait_timeout ran out (expected)
  kErrNotPositiveDefinite = 1u << 6,  // GPTQ factor: a Cholesky pivot of H was not positive
};

// About two seconds of polling, measured on the global nanosecond timer.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Bytes to add to the dynamic shared-memory base to reach a 1024-byte boundary (the
// SWIZZLE_128B atom).  Applied as pointer arithmetic on the __shared__ array itself, so the
// compiler keeps the shared address space and emits shared-memory loads/stores (a round trip
// through an integer type would turn every access into a generic one).
__device__ __forceinline__ uint32_t smem_align_pad(const void* base) {
  return (1024u - (smem_u32(base) & 1023u)) & 1023u;
}

// ---------------------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the async proxy (TMA, tcgen05.commit).
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
               ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}

// Waits until the phase with the given parity has completed.  Returns false (after
// recording `code` in *err) if that takes longer than kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t* err, uint32_t code) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t spins = 0;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((++spins & 255u) == 0u) {
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        atomicOr(err, code);
        return false;
      }
    }
  }
}

// The same bounded wait with the limit given in nanoseconds.
__device__ __forceinline__ bool mbar_wait_for(uint64_t* bar, uint32_t parity, uint32_t* err, uint32_t code,
                                              uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > limit_ns) {
      atomicOr(err, code);
      return false;
    }
  }
}

// ---------------------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor), 2-D tiles, completion counted on an mbarrier
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const void* desc) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(desc)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* smem_dst, const void* desc, int32_t c0, int32_t c1,
                                            uint64_t* bar, uint64_t cache_hint) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;"
      ::"r"(smem_u32(smem_dst)), "l"(reinterpret_cast<uint64_t>(desc)), "r"(c0), "r"(c1),
        "r"(smem_u32(bar)), "l"(cache_hint)
      : "memory");
}

// Untiled bulk copy global -> shared: both addresses 16-byte aligned, `bytes` a multiple of 16;
// completion counted on an mbarrier (expect_tx armed by the caller).
__device__ __forceinline__ void bulk_load_1d(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_u32(smem_dst)), "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// Warm L2 with a 2-D tile (no shared-memory destination, no completion tracking).  L2 is the
// point of coherence, so a later write to the same lines by another kernel is never hidden.
__device__ __forceinline__ void tma_prefetch_l2_2d(const void* desc, int32_t c0, int32_t c1) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];"
               ::"l"(reinterpret_cast<uint64_t>(desc)), "r"(c0), "r"(c1)
               : "memory");
}

// Programmatic dependent launch.  launch_dependents lets the next kernel of the stream start
// its CTAs as SMs free up; wait blocks until every prerequisite grid has completed and its
// memory operations are visible (it returns at once for a kernel launched without the
// programmatic-serialization attribute).
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// L2 eviction-priority policies for the cache_hint operand.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---------------------------------------------------------------------------------------
// Named barriers for warp subsets
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

__device__ __forceinline__ bool elect_one() {
  uint32_t pred;
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b32 r;\n\t"
      "elect.sync r|p, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// Loads through L2 only (data written by other CTAs of the same kernel).
__device__ __forceinline__ float ld_cg_f32(const float* p) { return __ldcg(p); }

// Power-of-two exponent k that carries bf16 values into fp16 exactly: given mx, the largest
// |x| of a row (or tile) as a bf16 bit pattern without its sign, x * 2^-k is computed for every
// x of the row.  k = max(floor(log2 mx) - 14, -109) puts the largest value in [2^14, 2^15) when
// it can (no overflow: fp16's largest finite value is below 2^16) and scales small rows UP as
// well as large ones down.  Every bf16 value within 2^31 of the row's largest (normal fp16
// results keep all 8 significant bits), and every bf16 value at all when k = -109 (the scaled
// values are multiples of 2^-24, fp16's subnormal spacing), converts exactly.  Non-finite rows
// use k = 0.  Both 2^k and 2^-k are normal floats for k in [-109, 113].
__device__ __forceinline__ int bf16_to_f16_exponent(uint32_t mx) {
  if (mx >= 0x7f80u) return 0;
  const int ex = static_cast<int>(mx >> 7) - 127;   // floor(log2 mx); -127 for 0 and subnormals
  return max(ex - 14, -109);
}
// 2^k as a float for k in [-126, 127] (normal range only).
__device__ __forceinline__ float pow2_normal(int k) { return __uint_as_float(static_cast<uint32_t>(127 + k) << 23); }

// INT4 g128 group parameters from a group's range [lo, hi] (lo <= 0 <= hi), float32 with each
// operation rounded on its own (推理优化与量化算子深度技术调研 §1.2, 第 1 章：推理加速全景 §4.1):
//   s32 = (hi - lo) / 15;  s = fp16_rn(min(s32, 65504)), and 1 when that is 0;
//   z = min(rint(-lo / s), 15).
// The min on s32 saturates the stored scale at the largest finite fp16 value instead of
// letting it round to +inf (a group range above 15 * 65504); the min on z keeps the zero point
// a code (it exceeds 15 only when the stored scale is far below s32: an fp16-subnormal or a
// saturated scale).  Returns the stored scale, its float value and z as a float.
__device__ __forceinline__ __half int4_group_params(float lo, float hi, float& s, float& zf) {
  const float s32 = __fdiv_rn(__fsub_rn(hi, lo), 15.0f);
  __half s16 = __float2half_rn(fminf(s32, 65504.0f));
  if ((__half_as_ushort(s16) & 0x7fffu) == 0u) s16 = __ushort_as_half(0x3c00u);  // zero -> 1.0
  s = __half2float(s16);
  // through an integer: -lo is -0.0 for a group without negative values, and the stored zero
  // point must be +0 (an integer), not fp16 -0
  zf = static_cast<float>(static_cast<int>(fminf(rintf(__fdiv_rn(-lo, s)), 15.0f)));
  return s16;
}

// SiLU(g) = g * sigmoid(g) = g / (1 + e^-g), fp32, with the CUDA fast exponential and fast
// divide intrinsics (a few ulp: far inside the bf16 rounding of the result).  For g << 0 the
// denominator is huge or +inf and the quotient is 0, the function's limit.
__device__ __forceinline__ float silu_f32(float g) { return __fdividef(g, 1.f + __expf(-g)); }

// Output column of interleaved gate row n of the fused gate+up weight (row 16q + i, i < 8,
// holds gate row 8q + i; its up row is n + 8).
__device__ __forceinline__ int swiglu_col(int n) { return ((n >> 4) << 3) | (n & 7); }

}  // namespace wq
