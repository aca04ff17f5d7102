// W8A8 in FP8 E4M3 on the 5th-generation tensor cores (推理优化与量化算子深度技术调研 §1.4: FP8
// weights and activations with their FP32 scales kept beside the tensors; 第 6 课：量化源码走读 §4:
// W4A16 for small-batch decode, FP8 for large-batch prefill).
//
// Quantization, one CTA per row (weights: per output channel, offline; activations: per
// token, before every GEMM): s = amax / 448 in fp32 (a zero row gets 1), every element
// converted as fp32(x / s) -> E4M3 with round-to-nearest-even and saturation at +-448
// (cvt.rn.satfinite).  Codes and scales are bit-exact to the oracle.
//
// GEMM, swap-AB like the W4A16 prefill kernel:  D[n, m] = sum_k Wq[n, k] Xq[m, k]  (D = Y^T)
//   A = Wq tile [128 x 128 k], B = Xq tile [256 x 128 k]: both E4M3 straight from global
//   memory by TMA (128-byte swizzle, K-major) -- no dequantization, the tensor core reads
//   both operands from shared memory; MMA = tcgen05.mma.cta_group::1.kind::f8f6f4, M = 128,
//   N = 256, K = 32, issued by one thread; fp32 accumulation in tensor memory.
//   Persistent CTAs (one per SM) walk the tiles; tensor memory holds two 256-column
//   accumulators, so the epilogue of one tile (tcgen05.ld -> x s_w[n] s_x[m] -> bf16 ->
//   global) runs while the MMAs of the next accumulate into the other.
// Warp roles: warp 0 TMA producer, warp 1 TMEM allocator + MMA issuer, warps 2-5 epilogue
// (one warp per TMEM lane quarter).
#include "internal.h"
#include "tcgen05.cuh"

namespace wq {

__device__ uint32_t g_fp8_err;

uint32_t fp8_read_and_clear_error() {
  uint32_t v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, g_fp8_err, sizeof(v));
  cudaMemcpyToSymbol(g_fp8_err, &z, sizeof(z));
  return v;
}

namespace f8 {

// ------------------------------------------------------------------------------ quantize
constexpr int kQThreads = 256;
constexpr float kE4M3Max = 448.f;

// Two fp32 values -> two E4M3 codes, `lo` in the low byte (cvt puts its first source in the
// high byte).
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}

__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    v = lane < kQThreads / 32 ? red[lane] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (lane == 0) red[0] = v;
  }
  __syncthreads();
  return red[0];
}

// Eight values of a row (bf16 or fp32 input) as fp32.
template <bool BF16>
__device__ __forceinline__ void load8(const void* row, int64_t k, float (&x)[8]) {
  if constexpr (BF16) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(row) + k));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      x[2 * q] = __uint_as_float(w[q] << 16);
      x[2 * q + 1] = __uint_as_float(w[q] & 0xffff0000u);
    }
  } else {
    const float4 a = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(row) + k));
    const float4 b = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(row) + k + 4));
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  }
}

// One CTA per row: the row's absolute maximum, its scale, then every code.  The input may
// come from the previous kernel of the stream (activations): read after the dependency wait.
template <bool BF16>
__global__ void __launch_bounds__(kQThreads) k_quant_fp8_rows(const void* in, int64_t K, uint8_t* Q, float* scales) {
  __shared__ float red[kQThreads / 32];
  const int64_t r = blockIdx.x;
  const void* row = BF16 ? static_cast<const void*>(static_cast<const uint16_t*>(in) + r * K)
                         : static_cast<const void*>(static_cast<const float*>(in) + r * K);
  pdl_launch_dependents();
  pdl_wait();
  float mx = 0.f;
  for (int64_t k = 8 * static_cast<int64_t>(threadIdx.x); k < K; k += 8 * kQThreads) {
    float x[8];
    load8<BF16>(row, k, x);
#pragma unroll
    for (int q = 0; q < 8; ++q) mx = fmaxf(mx, fabsf(x[q]));
  }
  const float amax = block_max(mx, red);
  float s = __fdiv_rn(amax, kE4M3Max);
  if (s == 0.f) s = 1.f;
  uint8_t* qrow = Q + r * K;
  for (int64_t k = 8 * static_cast<int64_t>(threadIdx.x); k < K; k += 8 * kQThreads) {
    float x[8];
    load8<BF16>(row, k, x);
    uint32_t c[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) c[q] = e4m3x2(__fdiv_rn(x[2 * q], s), __fdiv_rn(x[2 * q + 1], s));
    *reinterpret_cast<uint2*>(qrow + k) = make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
  }
  if (threadIdx.x == 0) scales[r] = s;
}

// ------------------------------------------------------------------------------ GEMM
constexpr int BN = 128;            // weight rows per tile (MMA M)
constexpr int BM = 256;            // tokens per tile (MMA N)
constexpr int BK = 128;            // k per stage: one 128-byte swizzle row of E4M3
constexpr int kStages = 4;
constexpr int kWBytes = BN * BK;   // 16 KB
constexpr int kXBytes = BM * BK;   // 32 KB
constexpr int kAccBufs = 2;
constexpr int kTmemCols = 512;     // two BM-column fp32 accumulators
constexpr int kEpiWarps = 4;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kGroupM = 8;         // tile raster: 8 token tiles per group share the weights in L2

struct Smem {
  uint8_t w[kStages][kWBytes];     // 1024-aligned (SWIZZLE_128B atoms)
  uint8_t x[kStages][kXBytes];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t acc_full[kAccBufs];
  uint64_t acc_empty[kAccBufs];
  uint64_t mma_done;
  uint32_t tmem_base;
};

struct Params {
  const float* sx;   // [M] per-token scales
  const float* sw;   // [N] per-channel scales
  uint16_t* Y;       // [M, N] bf16
  int M, K, N;
  int tiles_n, tiles_m, tiles, k_stages;
};

// Instruction descriptor, kind::f8f6f4: fp32 accumulate, A and B E4M3 (format 0), both
// K-major, N = BM, M = BN.
constexpr uint32_t kIdesc = (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t(BM) >> 3) << 17) | ((uint32_t(BN) >> 4) << 24);

__device__ __forceinline__ void tile_coords(int t, int tiles_n, int tiles_m, int& tn, int& tm) {
  const int per_group = kGroupM * tiles_n;
  const int grp = t / per_group;
  const int first_m = grp * kGroupM;
  const int gsize = min(tiles_m - first_m, kGroupM);
  const int r = t % per_group;
  tm = first_m + r % gsize;
  tn = r / gsize;
}

__global__ void __launch_bounds__(kThreads, 1)
    k_gemm_fp8(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_x,
               const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw + smem_align_pad(smem_raw));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int b = 0; b < kAccBufs; ++b) {
      mbar_init(&sm.acc_full[b], 1);
      mbar_init(&sm.acc_empty[b], 32 * kEpiWarps);
    }
    mbar_init(&sm.mma_done, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  // The set-up overlaps the previous kernel (the activation quantizer); every read of global
  // memory and every write comes after the dependency wait (the MMA warp touches neither).
  pdl_launch_dependents();
  if (warp != 1) pdl_wait();

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmap_w);
      tma_prefetch_desc(&tmap_x);
      const uint64_t pol = l2_policy_evict_last();
      int it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < p.tiles && ok; t += gridDim.x) {
        int tn, tm;
        tile_coords(t, p.tiles_n, p.tiles_m, tn, tm);
        for (int kb = 0; kb < p.k_stages; ++kb, ++it) {
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1;
          if (!mbar_wait(&sm.empty[s], ph ^ 1, &g_fp8_err, kErrWaitEmpty)) { ok = false; break; }
          mbar_arrive_expect_tx(&sm.full[s], kWBytes + kXBytes);
          tma_load_2d(&sm.w[s][0], &tmap_w, kb * BK, tn * BN, &sm.full[s], pol);
          tma_load_2d(&sm.x[s][0], &tmap_x, kb * BK, tm * BM, &sm.full[s], pol);
        }
      }
      for (int j = it - kStages; j < it; ++j) {   // drain: the last fill of each slot landed
        if (j < 0) continue;
        mbar_wait(&sm.full[j % kStages], (j / kStages) & 1, &g_fp8_err, kErrDrain);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int it = 0, ti = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < p.tiles && ok; t += gridDim.x, ++ti) {
        const int b = ti % kAccBufs;
        const uint32_t aph = (ti / kAccBufs) & 1;
        // the epilogue is done with this accumulator (its previous tile)
        if (!mbar_wait(&sm.acc_empty[b], aph ^ 1, &g_fp8_err, kErrWaitEmpty)) break;
        tc_fence_after();
        const uint32_t d = tmem + static_cast<uint32_t>(b * BM);
        for (int kb = 0; kb < p.k_stages; ++kb, ++it) {
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1;
          if (!mbar_wait(&sm.full[s], ph, &g_fp8_err, kErrWaitFull)) { ok = false; break; }
          tc_fence_after();
          const uint64_t adesc = smem_desc_sw128(smem_u32(&sm.w[s][0]));
          const uint64_t bdesc = smem_desc_sw128(smem_u32(&sm.x[s][0]));
#pragma unroll
          for (int kk = 0; kk < BK / 32; ++kk)   // K = 32 per MMA: 32 bytes along the swizzled row
            tc_mma_ss_f8f6f4(d, adesc + static_cast<uint64_t>(2 * kk), bdesc + static_cast<uint64_t>(2 * kk), kIdesc,
                             (kb > 0 || kk > 0) ? 1u : 0u);
          tc_commit(&sm.empty[s]);
        }
        if (ok) tc_commit(&sm.acc_full[b]);
      }
      // every issued MMA has completed before tensor memory is released
      tc_commit(&sm.mma_done);
      mbar_wait(&sm.mma_done, 0, &g_fp8_err, kErrWaitAccum);
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;                          // TMEM lane quarter of this warp
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    int ti = 0;
    for (int t = blockIdx.x; t < p.tiles; t += gridDim.x, ++ti) {
      const int b = ti % kAccBufs;
      const uint32_t aph = (ti / kAccBufs) & 1;
      if (!mbar_wait(&sm.acc_full[b], aph, &g_fp8_err, kErrWaitAccum)) break;
      tc_fence_after();
      int tn, tm;
      tile_coords(t, p.tiles_n, p.tiles_m, tn, tm);
      const int n = tn * BN + 32 * q + lane;
      const int m0 = tm * BM;
      const bool row_ok = n < p.N;
      const float sw = row_ok ? __ldg(p.sw + n) : 0.f;
#pragma unroll 1
      for (int c = 0; c < BM; c += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + static_cast<uint32_t>(b * BM + c), v);
        tc_wait_ld();
        if (row_ok) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int m = m0 + c + j;
            if (m < p.M) {
              const float y = __uint_as_float(v[j]) * sw * __ldg(p.sx + m);
              p.Y[static_cast<long long>(m) * p.N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(y));
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&sm.acc_empty[b]);   // the MMA warp may accumulate the next tile here
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace f8

// ------------------------------------------------------------------------------ host side
cudaError_t launch_quant_fp8_rows(bool bf16_in, const void* in, int64_t R, int64_t K, uint8_t* Q, float* scales,
                                  cudaStream_t stream) {
  if (R < 1 || K < 16 || K % 16 != 0 || R > 0x7fffffffLL) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(R));
  cfg.blockDim = dim3(f8::kQThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (bf16_in) return cudaLaunchKernelEx(&cfg, f8::k_quant_fp8_rows<true>, in, K, Q, scales);
  return cudaLaunchKernelEx(&cfg, f8::k_quant_fp8_rows<false>, in, K, Q, scales);
}

cudaError_t launch_gemm_fp8(const uint8_t* Xq, const float* sx, int64_t M, int64_t K, int64_t N, const uint8_t* Wq,
                            const float* sw, uint16_t* Y, cudaStream_t stream) {
  using namespace f8;
  if (M < 1 || N < 1 || K < 16 || K % 16 != 0) return cudaErrorInvalidValue;
  Params p{};
  p.sx = sx;
  p.sw = sw;
  p.Y = Y;
  p.M = static_cast<int>(M);
  p.K = static_cast<int>(K);
  p.N = static_cast<int>(N);
  p.tiles_n = static_cast<int>((N + BN - 1) / BN);
  p.tiles_m = static_cast<int>((M + BM - 1) / BM);
  p.tiles = p.tiles_n * p.tiles_m;
  p.k_stages = static_cast<int>((K + BK - 1) / BK);
  CUtensorMap tw, tx;
  cudaError_t e = make_tmap_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, Wq, static_cast<uint64_t>(K), static_cast<uint64_t>(N),
                               static_cast<uint64_t>(K), BK, BN, CU_TENSOR_MAP_SWIZZLE_128B,
                               CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
  if (e != cudaSuccess) return e;
  e = make_tmap_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_UINT8, Xq, static_cast<uint64_t>(K), static_cast<uint64_t>(M),
                   static_cast<uint64_t>(K), BK, BM, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
  if (e != cudaSuccess) return e;
  static_assert(sizeof(Smem) + 1024 <= 227 * 1024, "FP8 GEMM shared memory over the per-CTA limit");
  const size_t smem = sizeof(Smem) + 1024;
  e = set_smem_attr_once(reinterpret_cast<const void*>(k_gemm_fp8), smem);
  if (e != cudaSuccess) return e;
  const long long sms = device_sm_count();
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(p.tiles < sms ? p.tiles : sms));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_gemm_fp8, tw, tx, p);
}

}  // namespace wq
