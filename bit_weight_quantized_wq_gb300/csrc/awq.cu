// AWQ: per-channel scaling of the salient input channels before INT4 g128 quantization
// (第 1 章：推理加速全景 §4.4; 推理优化与量化算子深度技术调研 §1.3; 量化与加速).
//
//   importance_j = mean_n |X[n, j]|                       (float64, samples in order)
//   salient      = the ceil(K / 100) most important channels (ties: lower index first)
//   s_j          = importance_j ^ (a / 20) on salient channels with importance > 0, else 1
//   a*           = argmin over a = 0 .. 20 of || X (Q(W diag(s)) diag(s)^-1 - W)^T ||_F^2
//   output       = Q(W diag(s*)) in the INT4 g128 format, and s* (activations are divided
//                  by s* at run time).
//
// Per candidate a: one pass quantizes W diag(s) group by group (the rules of the quantize
// kernel) and writes the weight error D = Q(W s) / s - W in fp32; an fp32 GEMM-shaped kernel
// forms E = X D^T tile by tile in K slices, a second pass adds the slices and squares, and the
// partial sums are added in a fixed order.  The candidates, the arg-min and the final packing run back to back
// on the stream with no host synchronisation.
#include "internal.h"

namespace wq {

namespace {

constexpr int kAwqGrid = 20;

__global__ void __launch_bounds__(256) k_awq_importance(const float* __restrict__ X, int n, int K,
                                                        double* __restrict__ imp) {
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= K) return;
  double acc = 0.0;
  for (int r = 0; r < n; ++r) acc += fabs(static_cast<double>(__ldg(X + static_cast<long long>(r) * K + j)));
  imp[j] = acc / static_cast<double>(n);
}

// rank of channel j = #{k : imp_k > imp_j, or imp_k == imp_j and k < j}; salient if rank < n_sal.
// Importances are non-negative, so their bit patterns order like the values.
__global__ void __launch_bounds__(256) k_awq_salient(const double* __restrict__ imp, int K, int n_sal,
                                                     uint8_t* __restrict__ mask) {
  __shared__ long long tile[256];
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  const long long mine = j < K ? __double_as_longlong(imp[j]) : 0;
  int rank = 0;
  for (int base = 0; base < K; base += 256) {
    const int k = base + threadIdx.x;
    tile[threadIdx.x] = k < K ? __double_as_longlong(imp[k]) : -1;
    __syncthreads();
    const int lim = min(256, K - base);
    for (int q = 0; q < lim; ++q) {
      const long long o = tile[q];
      rank += (o > mine || (o == mine && base + q < j)) ? 1 : 0;
    }
    __syncthreads();
  }
  if (j < K) mask[j] = rank < n_sal ? 1 : 0;
}

// s_j for candidate a (a_dev, when given, holds the candidate)
__global__ void __launch_bounds__(256) k_awq_scales(const double* __restrict__ imp, const uint8_t* __restrict__ mask,
                                                    int K, int a, const int* __restrict__ a_dev, float* __restrict__ s) {
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= K) return;
  const int aa = a_dev ? *a_dev : a;
  const double v = imp[j];
  s[j] = (mask[j] && v > 0.0) ? static_cast<float>(pow(v, static_cast<double>(aa) / static_cast<double>(kAwqGrid))) : 1.f;
}

// Quantizes W diag(s) (8 lanes per group of 128, 16 values per lane) by the INT4 g128 rules.
// D (when given) receives Q(W s) / s - W; Wq / scales / zeros (when given) the packed result.
__global__ void __launch_bounds__(256) k_awq_quant(const float* __restrict__ W, const float* __restrict__ s,
                                                   int64_t groups, int K, float* __restrict__ D,
                                                   uint32_t* __restrict__ Wq, __half* __restrict__ scales,
                                                   __half* __restrict__ zeros) {
  const int64_t gid = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 3;
  const uint32_t sub = threadIdx.x & 7u;
  const bool active = gid < groups;
  const int64_t g = active ? gid : 0;
  const int G = K / 128;
  const int k0 = static_cast<int>(g % G) * 128 + static_cast<int>(sub) * 16;

  float w[16], sv[16], x[16];
  const float4* src = reinterpret_cast<const float4*>(W + g * 128 + sub * 16);
  const float4* ss = reinterpret_cast<const float4*>(s + k0);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 v = active ? __ldg(src + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 u = __ldg(ss + i);
    w[4 * i + 0] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
    sv[4 * i + 0] = u.x; sv[4 * i + 1] = u.y; sv[4 * i + 2] = u.z; sv[4 * i + 3] = u.w;
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) x[i] = __fmul_rn(w[i], sv[i]);
  float lo = 0.f, hi = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) { lo = fminf(lo, x[i]); hi = fmaxf(hi, x[i]); }
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) {
    lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  }
  float sc, zf;
  const __half s16 = int4_group_params(lo, hi, sc, zf);

  uint32_t w0 = 0u, w1 = 0u;
  float d[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    float q = __fadd_rn(rintf(__fdiv_rn(x[i], sc)), zf);
    q = fminf(fmaxf(q, 0.f), 15.f);
    const uint32_t c = static_cast<uint32_t>(q);
    if (i < 8) w0 |= c << (4 * i);
    else w1 |= c << (4 * (i - 8));
    d[i] = __fsub_rn(__fdiv_rn(__fmul_rn(__fsub_rn(q, zf), sc), sv[i]), w[i]);
  }
  if (!active) return;
  if (D) {
    float4* dst = reinterpret_cast<float4*>(D + g * 128 + sub * 16);
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[i] = make_float4(d[4 * i], d[4 * i + 1], d[4 * i + 2], d[4 * i + 3]);
  }
  if (Wq) {
    reinterpret_cast<uint2*>(Wq + g * 16)[sub] = make_uint2(w0, w1);
    if (sub == 0) {
      scales[g] = s16;
      zeros[g] = __float2half_rn(zf);
    }
  }
}

// E = X D^T (X [n, K], D [N, K], both K-contiguous) in 64 x 64 tiles, 4 x 4 per thread, fp32,
// split along K into gridDim.z slices (more CTAs than SMs, so loads overlap compute): slice z
// writes its partial product to Epart[z][m][i].
constexpr int kTM = 64, kTN = 64, kTK = 32;

__global__ void __launch_bounds__(256) k_awq_err(const float* __restrict__ X, const float* __restrict__ D, int n,
                                                 int N, int K, float* __restrict__ Epart) {
  __shared__ float xs[kTK][kTM + 4];
  __shared__ float ds[kTK][kTN + 4];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int m0 = blockIdx.y * kTM, n0 = blockIdx.x * kTN;
  const int kslice = K / gridDim.z;
  const int kbeg = blockIdx.z * kslice, kend = kbeg + kslice;
  float acc[4][4] = {};
  for (int k0 = kbeg; k0 < kend; k0 += kTK) {
    // 64 x 32 floats of each operand, 8 per thread: element e = threadIdx.x + 256 q
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int e = threadIdx.x + 256 * q;
      const int r = e / kTK, c = e % kTK;
      const int xm = m0 + r, dn = n0 + r;
      xs[c][r] = xm < n ? __ldg(X + static_cast<long long>(xm) * K + k0 + c) : 0.f;
      ds[c][r] = dn < N ? __ldg(D + static_cast<long long>(dn) * K + k0 + c) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kTK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) { a[u] = xs[kk][ty * 4 + u]; b[u] = ds[kk][tx * 4 + u]; }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(a[u], b[v], acc[u][v]);
    }
    __syncthreads();
  }
  float* out = Epart + static_cast<long long>(blockIdx.z) * n * N;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int m = m0 + ty * 4 + u;
    if (m >= n) continue;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int i = n0 + tx * 4 + v;
      if (i < N) out[static_cast<long long>(m) * N + i] = acc[u][v];
    }
  }
}

// Sum of squares of E = sum over slices of Epart (slices added in order): each CTA takes a
// contiguous chunk of the n N elements and writes its fp64 sum to partial[blockIdx.x].
__global__ void __launch_bounds__(256) k_awq_sq(const float* __restrict__ Epart, int slices, long long count,
                                                double* __restrict__ partial) {
  __shared__ double red[256];
  const long long chunk = (count + gridDim.x - 1) / gridDim.x;
  const long long beg = static_cast<long long>(blockIdx.x) * chunk;
  const long long end = min(count, beg + chunk);
  // each thread's few elements in fp32 (fp64 throughput is low), then fp64 across threads
  float sq32 = 0.f;
  for (long long e = beg + threadIdx.x; e < end; e += blockDim.x) {
    float v = Epart[e];
    for (int z = 1; z < slices; ++z) v += Epart[static_cast<long long>(z) * count + e];
    sq32 = fmaf(v, v, sq32);
  }
  red[threadIdx.x] = static_cast<double>(sq32);
  __syncthreads();
  for (int o = 128; o > 0; o >>= 1) {
    if (threadIdx.x < o) red[threadIdx.x] += red[threadIdx.x + o];
    __syncthreads();
  }
  if (threadIdx.x == 0) partial[blockIdx.x] = red[0];
}

constexpr int kSqCtas = 256;

int awq_kslices(int64_t K) { return K >= 512 ? 4 : (K >= 256 ? 2 : 1); }

// One warp: lane l adds partials l, l + 32, ... in order, then a fixed shuffle tree.
__global__ void __launch_bounds__(32) k_awq_sum(const double* __restrict__ partial, int count, double* __restrict__ out) {
  double acc = 0.0;
  for (int i = threadIdx.x; i < count; i += 32) acc += partial[i];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (threadIdx.x == 0) *out = acc;
}

// the smallest a among the minimal losses
__global__ void k_awq_pick(const double* __restrict__ losses, int count, int* __restrict__ a_best,
                           int32_t* __restrict__ a_out) {
  int best = 0;
  for (int a = 1; a < count; ++a)
    if (losses[a] < losses[best]) best = a;
  *a_best = best;
  if (a_out) *a_out = best;
}

size_t align256(size_t b) { return (b + 255) / 256 * 256; }

}  // namespace

size_t awq_workspace_bytes(int64_t N, int64_t K, int64_t n) {
  return align256(K * sizeof(double)) + align256(K) + align256(K * sizeof(float)) +
         align256(static_cast<size_t>(N) * K * sizeof(float)) +
         align256(static_cast<size_t>(awq_kslices(K)) * n * N * sizeof(float)) + align256(kSqCtas * sizeof(double)) +
         align256((kAwqGrid + 1) * sizeof(double)) + align256(sizeof(int));
}

cudaError_t launch_awq_int4_g128(const float* W, int64_t N, int64_t K, const float* X, int64_t n, int32_t* Wq,
                                 uint16_t* scales, uint16_t* zeros, float* s_out, int32_t* a_out, double* losses_out,
                                 void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (ws_bytes < awq_workspace_bytes(N, K, n)) return cudaErrorInvalidValue;
  uint8_t* p = static_cast<uint8_t*>(ws);
  double* imp = reinterpret_cast<double*>(p);
  p += align256(K * sizeof(double));
  uint8_t* mask = p;
  p += align256(K);
  float* s = reinterpret_cast<float*>(p);
  p += align256(K * sizeof(float));
  float* D = reinterpret_cast<float*>(p);
  p += align256(static_cast<size_t>(N) * K * sizeof(float));
  const int slices = awq_kslices(K);
  float* Epart = reinterpret_cast<float*>(p);
  p += align256(static_cast<size_t>(slices) * n * N * sizeof(float));
  double* partial = reinterpret_cast<double*>(p);
  p += align256(kSqCtas * sizeof(double));
  const dim3 egrid(static_cast<unsigned>((N + kTN - 1) / kTN), static_cast<unsigned>((n + kTM - 1) / kTM),
                   static_cast<unsigned>(slices));
  double* losses = reinterpret_cast<double*>(p);
  p += align256((kAwqGrid + 1) * sizeof(double));
  int* a_best = reinterpret_cast<int*>(p);

  const unsigned kb = static_cast<unsigned>((K + 255) / 256);
  const int64_t groups = N * (K / 128);
  const int64_t qgrid = (groups * 8 + 255) / 256;
  if (qgrid > 0x7fffffffLL) return cudaErrorInvalidValue;
  const int n_sal = static_cast<int>((K + 99) / 100);

  k_awq_importance<<<kb, 256, 0, stream>>>(X, static_cast<int>(n), static_cast<int>(K), imp);
  k_awq_salient<<<kb, 256, 0, stream>>>(imp, static_cast<int>(K), n_sal, mask);
  for (int a = 0; a <= kAwqGrid; ++a) {
    k_awq_scales<<<kb, 256, 0, stream>>>(imp, mask, static_cast<int>(K), a, nullptr, s);
    k_awq_quant<<<static_cast<unsigned>(qgrid), 256, 0, stream>>>(W, s, groups, static_cast<int>(K), D, nullptr,
                                                                   nullptr, nullptr);
    k_awq_err<<<egrid, 256, 0, stream>>>(X, D, static_cast<int>(n), static_cast<int>(N), static_cast<int>(K), Epart);
    k_awq_sq<<<kSqCtas, 256, 0, stream>>>(Epart, slices, n * N, partial);
    k_awq_sum<<<1, 32, 0, stream>>>(partial, kSqCtas, losses + a);
  }
  k_awq_pick<<<1, 1, 0, stream>>>(losses, kAwqGrid + 1, a_best, a_out);
  k_awq_scales<<<kb, 256, 0, stream>>>(imp, mask, static_cast<int>(K), 0, a_best, s_out);
  k_awq_quant<<<static_cast<unsigned>(qgrid), 256, 0, stream>>>(W, s_out, groups, static_cast<int>(K), nullptr,
                                                                 reinterpret_cast<uint32_t*>(Wq),
                                                                 reinterpret_cast<__half*>(scales),
                                                                 reinterpret_cast<__half*>(zeros));
  if (losses_out) {
    cudaError_t e = cudaMemcpyAsync(losses_out, losses, (kAwqGrid + 1) * sizeof(double), cudaMemcpyDeviceToDevice,
                                    stream);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

}  // namespace wq
