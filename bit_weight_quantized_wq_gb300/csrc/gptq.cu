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
// Rows are independent: one CTA owns R rows and keeps their current values on chip for the
// whole sweep -- the pages' lazy block update exists to avoid re-streaming W, which on-chip
// residency avoids altogether.  Two kernels:
//   K <= 16384  registers: thread t owns columns t + 512 k; the warp of the owner of column i
//               takes its decisions (lane r for row r, the owner's values broadcast by
//               shuffle), publishes e_i through shared memory (double-buffered, one barrier
//               per column) and every thread updates its own later columns with row i of U,
//               which a bulk async copy brought into shared memory two to four columns ahead.
//   larger K    shared memory: the rows' values live in shared memory; R threads decide, all
//               threads update, two barriers per column.
#include "internal.h"

namespace wq {

__device__ uint32_t g_gptq_err;

uint32_t gptq_read_and_clear_error() {
  uint32_t v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, g_gptq_err, sizeof(v));
  cudaMemcpyToSymbol(g_gptq_err, &z, sizeof(z));
  return v;
}

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
          float s, zf;
          const __half s16 = int4_group_params(lo, hi, s, zf);
          s_scale[warp] = s;
          s_zero[warp] = zf;
          const long long gi = static_cast<long long>(row0 + warp) * G + (i >> 7);
          scales[gi] = s16;
          zeros[gi] = __float2half_rn(zf);
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


template <int NJ>
__device__ __forceinline__ float pick(const float (&a)[NJ], int k) {
  float x = a[0];
#pragma unroll
  for (int m = 1; m < NJ; ++m)
    if (k == m) x = a[m];
  return x;
}

constexpr int kRegThreads = 512;
constexpr uint32_t kErrGptqWait = 1u;

// Register-resident sweep, R rows per CTA, columns t + 512 k (k < NJ) owned by thread t.  Row
// i of U reaches shared memory by a bulk copy issued D columns ahead (a ring of D rows).
template <int NJ, int R, int D>
__global__ void __launch_bounds__(kRegThreads, 1)
    k_gptq_int4_g128_reg(const float* __restrict__ W, int N, int K, const float* __restrict__ U,
                         uint32_t* __restrict__ Wq, __half* __restrict__ scales, __half* __restrict__ zeros) {
  constexpr int T = kRegThreads;
  extern __shared__ __align__(16) uint8_t smem[];
  float* urow = reinterpret_cast<float*>(smem);                                  // [D][K]
  uint8_t* code = smem + static_cast<size_t>(D) * K * sizeof(float);             // [R][K] codes
  __shared__ __align__(8) uint64_t full[D];
  __shared__ float s_err[2][R];
  __shared__ float s_scale[R], s_zero[R];
  __shared__ float s_lo[4][R], s_hi[4][R];
  const int row0 = blockIdx.x * R;
  const int rows = min(R, N - row0);
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int G = K / 128;

  // copy of row i of U from its 16-byte aligned column i & ~3 (covers the diagonal)
  auto issue = [&](int i) {
    const int c0 = i & ~3;
    float* dst = urow + static_cast<size_t>(i % D) * K + c0;
    const uint32_t bytes = static_cast<uint32_t>(K - c0) * 4u;
    mbar_arrive_expect_tx(&full[i % D], bytes);
    bulk_load_1d(dst, U + static_cast<long long>(i) * K + c0, bytes, &full[i % D]);
  };
  if (t == 0) {
    for (int q = 0; q < D; ++q) mbar_init(&full[q], 1);
    fence_barrier_init();
    for (int q = 0; q < D && q < K; ++q) issue(q);
  }

  float v[R][NJ];   // current values of the owned columns
#pragma unroll
  for (int k = 0; k < NJ; ++k) {
    const int j = t + T * k;
#pragma unroll
    for (int r = 0; r < R; ++r)
      v[r][k] = (r < rows && j < K) ? __ldg(W + static_cast<long long>(row0 + r) * K + j) : 0.f;
  }
  __syncthreads();

  int i = 0;
  for (; i < K; ++i) {
    const int ki = i / T;
    const int owner = i & (T - 1);
    const float* ui = urow + static_cast<size_t>(i % D) * K;
    bool bad = false;
    if ((i & 127) == 0) {
      // group parameters: the 4 warps owning columns i .. i + 127 reduce each row's range
      const int w0 = owner >> 5;
      if (warp >= w0 && warp < w0 + 4) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const float x = pick<NJ>(v[r], ki);
          float lo = fminf(0.f, x), hi = fmaxf(0.f, x);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
            hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
          }
          if (lane == 0) {
            s_lo[warp - w0][r] = lo;
            s_hi[warp - w0][r] = hi;
          }
        }
      }
      __syncthreads();
      if (warp == (owner >> 5) && lane < R) {
        // lane r of the owner's warp: row r's parameters (padding rows too: their values are
        // 0, so s = 1 and z = 0; only real rows are stored)
        const int r = lane;
        const float lo = fminf(fminf(s_lo[0][r], s_lo[1][r]), fminf(s_lo[2][r], s_lo[3][r]));
        const float hi = fmaxf(fmaxf(s_hi[0][r], s_hi[1][r]), fmaxf(s_hi[2][r], s_hi[3][r]));
        float sc, zf;
        const __half s16 = int4_group_params(lo, hi, sc, zf);
        s_scale[r] = sc;
        s_zero[r] = zf;
        if (r < rows) {
          const long long gi = static_cast<long long>(row0 + r) * G + (i >> 7);
          scales[gi] = s16;
          zeros[gi] = __float2half_rn(zf);
        }
      }
    }
    // row i of U has landed (every thread waits: all of them read it below)
    bad = !mbar_wait(&full[i % D], (i / D) & 1, &g_gptq_err, kErrGptqWait);
    if (warp == (owner >> 5)) {
      // The owner's warp decides column i: every lane picks its slot values in step, the
      // owner lane's R values are broadcast, and lane r takes row r's decision.
      const int ol = owner & 31;
      float xr = 0.f;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float x = __shfl_sync(0xffffffffu, pick<NJ>(v[r], ki), ol);
        if (lane == r) xr = x;
      }
      if (lane < R && !bad) {   // padding rows too (value 0, error 0)
        const float d = ui[i];   // U[i, i]
        const float sc = s_scale[lane], zf = s_zero[lane];
        float q = __fadd_rn(rintf(__fdiv_rn(xr, sc)), zf);
        q = fminf(fmaxf(q, 0.f), 15.f);
        code[static_cast<size_t>(lane) * K + i] = static_cast<uint8_t>(q);
        s_err[i & 1][lane] = __fdiv_rn(__fsub_rn(xr, __fmul_rn(__fsub_rn(q, zf), sc)), d);
      }
    }
    // one barrier per column; a timed-out wait anywhere stops every thread here together
    if (__syncthreads_or(bad)) break;
    // slot of row i - 1 is free: every thread finished reading it (column i - 1) before this
    // barrier, and nothing wrote it from the generic proxy, so the copy needs no proxy fence
    if (t == 0 && i >= 1 && i - 1 + D < K) issue(i - 1 + D);
    float e[R];
#pragma unroll
    for (int r = 0; r < R; ++r) e[r] = s_err[i & 1][r];
#pragma unroll
    for (int k = 0; k < NJ; ++k) {
      const int j = t + T * k;
      if (j > i && j < K) {
        const float u = ui[j];
#pragma unroll
        for (int r = 0; r < R; ++r) v[r][k] = __fsub_rn(v[r][k], __fmul_rn(e[r], u));
      }
    }
  }
  __syncthreads();
  if (i < K) {
    // stopped early at column i: rows i .. last were issued and may still be in flight; let
    // them land before the CTA exits
    if (t == 0) {
      const int last = (i == 0) ? min(K - 1, D - 1) : min(K - 1, i - 2 + D);
      for (int q = i; q <= last; ++q) mbar_wait(&full[q % D], (q / D) & 1, &g_gptq_err, kErrGptqWait);
    }
    __syncthreads();
    return;
  }
  for (int r = 0; r < rows; ++r) {
    const uint8_t* c = code + static_cast<size_t>(r) * K;
    uint32_t* out = Wq + static_cast<long long>(row0 + r) * (K / 8);
    for (int j = t; j < K / 8; j += T) {
      uint32_t word = 0u;
#pragma unroll
      for (int k = 0; k < 8; ++k) word |= static_cast<uint32_t>(c[8 * j + k]) << (4 * k);
      out[j] = word;
    }
  }
}

template <int NJ, int R, int D>
cudaError_t launch_reg(const float* W, int64_t N, int64_t K, const float* U, int32_t* Wq, uint16_t* scales,
                       uint16_t* zeros, cudaStream_t stream) {
  const size_t smem = static_cast<size_t>(D) * K * sizeof(float) + static_cast<size_t>(R) * K;
  const long long grid = (N + R - 1) / R;
  if (grid > 0x7fffffffLL || smem > static_cast<size_t>(kGptqSmem)) return cudaErrorInvalidValue;
  cudaError_t e = set_smem_attr_once(reinterpret_cast<const void*>(k_gptq_int4_g128_reg<NJ, R, D>), kGptqSmem);
  if (e != cudaSuccess) return e;
  k_gptq_int4_g128_reg<NJ, R, D><<<static_cast<unsigned>(grid), kRegThreads, smem, stream>>>(
      W, static_cast<int>(N), static_cast<int>(K), U, reinterpret_cast<uint32_t*>(Wq),
      reinterpret_cast<__half*>(scales), reinterpret_cast<__half*>(zeros));
  return cudaGetLastError();
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
  // R NJ values per thread within the 128 registers of a 512-thread CTA; the U ring (D rows)
  // and the codes (R rows) within shared memory
  if (K <= 512) return launch_reg<1, 8, 4>(W, N, K, U, Wq, scales, zeros, stream);
  if (K <= 1024) return launch_reg<2, 8, 4>(W, N, K, U, Wq, scales, zeros, stream);
  if (K <= 2048) return launch_reg<4, 8, 4>(W, N, K, U, Wq, scales, zeros, stream);
  if (K <= 4096) return launch_reg<8, 8, 4>(W, N, K, U, Wq, scales, zeros, stream);
  if (K <= 8192) return launch_reg<16, 5, 4>(W, N, K, U, Wq, scales, zeros, stream);
  if (K <= 16384) return launch_reg<32, 2, 2>(W, N, K, U, Wq, scales, zeros, stream);
  const int R = gptq_rows_per_cta(K);
  if (R < 1) return cudaErrorInvalidValue;
  const size_t smem = static_cast<size_t>(R) * K * 5;
  cudaError_t e = set_smem_attr_once(reinterpret_cast<const void*>(k_gptq_int4_g128), kGptqSmem);
  if (e != cudaSuccess) return e;
  const long long grid = (N + R - 1) / R;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  k_gptq_int4_g128<<<static_cast<unsigned>(grid), kGptqThreads, smem, stream>>>(
      W, static_cast<int>(N), static_cast<int>(K), R, U, reinterpret_cast<uint32_t*>(Wq),
      reinterpret_cast<__half*>(scales), reinterpret_cast<__half*>(zeros));
  return cudaGetLastError();
}

}  // namespace wq
