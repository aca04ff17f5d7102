// GPTQ's inverse-Hessian factor from calibration activations, on the device in float64
// (第 1 章：推理加速全景 §4.2: H = 2 X^T X + lambda I over the calibration set, H^-1 through its
// Cholesky factor; 推理优化与量化算子深度技术调研 §1.3).
//
// The sweep needs the upper factor U of H^-1 = U^T U.  With J the index reversal,
//   J H J = L' L'^T  (lower Cholesky factor L')   =>   H = R R^T,  R = J L' J  (upper),
//   H^-1 = R^-T R^-1 = U^T U  with  U = R^-1 = J L'^-1 J,
// which is the unique upper factor with a positive diagonal, i.e. the same U as
// cholesky(H^-1)^T, from one Cholesky factorisation and one triangular inverse.
//
// Steps (all float64, row-major K x K, K a multiple of 64):
//   1. A = J (2 X^T X) J, lower 64 x 64 tiles only (tiled GEMM over the n samples);
//   2. lambda = 0.01 mean(diag), A += lambda I;
//   3. blocked right-looking Cholesky, 64 columns at a time: the diagonal block factored and
//      inverted in one CTA, the panel times that inverse transposed, the trailing lower
//      triangle updated by a tiled GEMM;
//   4. blocked triangular inverse, block row by block row:
//      Linv[i, 0:i] = -inv(L[i,i]) (L[i, 0:i] Linv[0:i, 0:i]);
//   5. U[i][j] = float(Linv[K-1-i][K-1-j]) for j >= i, 0 below the diagonal.
// Every sum runs in a fixed order, so the result is reproducible run to run.
#include "internal.h"

namespace wq {

__device__ uint32_t g_gptq_factor_err;

uint32_t gptq_factor_read_and_clear_error() {
  uint32_t v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, g_gptq_factor_err, sizeof(v));
  cudaMemcpyToSymbol(g_gptq_factor_err, &z, sizeof(z));
  return v;
}

namespace fac {

constexpr int BS = 64;            // block (tile) size
constexpr int kThreads = 256;     // 16 x 16 threads, 4 x 4 outputs each
constexpr int KC = 16;            // inner-dimension chunk held in shared memory

// C (M x N) = alpha op(A) op(B) + beta C over the inner range [k_lo, k_hi) (or, with
// b_lower, [max(k_lo, the tile's first column), k_hi): B lower triangular, its entries above
// the diagonal zero and skipped).  op(A) = A (M x Kd, lda) or A^T (A stored Kd x M); op(B) = B
// (Kd x N) or B^T (B stored N x Kd).  lower_only: tiles entirely above the diagonal of a
// square C are skipped.  beta == 0 overwrites C.
template <bool TA, bool TB>
__global__ void __launch_bounds__(kThreads) k_gemm_f64(int M, int N, int k_lo, int k_hi, double alpha,
                                                       const double* __restrict__ A, long long lda,
                                                       const double* __restrict__ B, long long ldb, double beta,
                                                       double* __restrict__ C, long long ldc, int lower_only,
                                                       int b_lower) {
  const int i0 = blockIdx.y * BS, j0 = blockIdx.x * BS;
  if (lower_only && j0 > i0 + BS - 1) return;
  __shared__ double sa[KC][BS + 1];   // op(A)[i0 + r][k] at sa[k][r]
  __shared__ double sb[KC][BS + 1];   // op(B)[k][j0 + c] at sb[k][c]
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  double acc[4][4];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) acc[a][b] = 0.0;
  const int kstart = b_lower ? max(k_lo, j0) : k_lo;
  for (int kc = kstart; kc < k_hi; kc += KC) {
    for (int e = threadIdx.x; e < KC * BS; e += kThreads) {
      const int kk = e / BS, r = e % BS;
      const int k = kc + kk;
      double va = 0.0, vb = 0.0;
      if (k < k_hi) {
        const int ia = i0 + r, jb = j0 + r;
        if (ia < M) va = TA ? A[static_cast<long long>(k) * lda + ia] : A[static_cast<long long>(ia) * lda + k];
        if (jb < N) vb = TB ? B[static_cast<long long>(jb) * ldb + k] : B[static_cast<long long>(k) * ldb + jb];
      }
      sa[kk][r] = va;
      sb[kk][r] = vb;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < KC; ++kk) {
      double a4[4], b4[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        a4[q] = sa[kk][ty + 16 * q];
        b4[q] = sb[kk][tx + 16 * q];
      }
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] = fma(a4[a], b4[b], acc[a][b]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int i = i0 + ty + 16 * a, j = j0 + tx + 16 * b;
      if (i < M && j < N) {
        double* c = C + static_cast<long long>(i) * ldc + j;
        *c = (beta == 0.0) ? alpha * acc[a][b] : fma(alpha, acc[a][b], beta * *c);
      }
    }
}

// A = J (2 X^T X) J on the lower tiles: A[i][j] = 2 sum_s X[s][K-1-i] X[s][K-1-j], the samples
// added in order.  X float32 [n, K].
__global__ void __launch_bounds__(kThreads) k_hessian_rev(const float* __restrict__ X, int n, int K,
                                                          double* __restrict__ A) {
  const int i0 = blockIdx.y * BS, j0 = blockIdx.x * BS;
  if (j0 > i0) return;
  __shared__ double sa[KC][BS + 1];
  __shared__ double sb[KC][BS + 1];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  double acc[4][4];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) acc[a][b] = 0.0;
  for (int sc = 0; sc < n; sc += KC) {
    for (int e = threadIdx.x; e < KC * BS; e += kThreads) {
      const int ss = e / BS, r = e % BS;
      const int s = sc + ss;
      double va = 0.0, vb = 0.0;
      if (s < n) {
        va = static_cast<double>(X[static_cast<long long>(s) * K + (K - 1 - (i0 + r))]);
        vb = static_cast<double>(X[static_cast<long long>(s) * K + (K - 1 - (j0 + r))]);
      }
      sa[ss][r] = va;
      sb[ss][r] = vb;
    }
    __syncthreads();
#pragma unroll
    for (int ss = 0; ss < KC; ++ss) {
      double a4[4], b4[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        a4[q] = sa[ss][ty + 16 * q];
        b4[q] = sb[ss][tx + 16 * q];
      }
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] = fma(a4[a], b4[b], acc[a][b]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int i = i0 + ty + 16 * a, j = j0 + tx + 16 * b;
      A[static_cast<long long>(i) * K + j] = 2.0 * acc[a][b];
    }
}

// lambda = damp * mean(diag(A)) added to the diagonal.  One CTA; the diagonal is summed in a
// fixed tree order.
__global__ void __launch_bounds__(kThreads) k_damp(double* __restrict__ A, int K, double damp) {
  __shared__ double red[kThreads];
  double s = 0.0;
  for (int i = threadIdx.x; i < K; i += kThreads) s += A[static_cast<long long>(i) * K + i];
  red[threadIdx.x] = s;
  __syncthreads();
  for (int w = kThreads / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  const double lam = damp * (red[0] / K);
  __syncthreads();
  for (int i = threadIdx.x; i < K; i += kThreads) A[static_cast<long long>(i) * K + i] += lam;
}

// Diagonal block kb of the Cholesky factorisation: A[kb:kb+64, kb:kb+64] (lower triangle,
// already updated by the earlier blocks) is factored in place, L L^T, and its inverse written
// to Dinv [64 x 64] (lower, zeros above).  One CTA.  A pivot that is not positive (H not
// positive definite) records bit 1 << 6 in the error word and continues with NaN.
__global__ void __launch_bounds__(kThreads) k_potrf_block(double* __restrict__ A, long long lda, int kb,
                                                          double* __restrict__ Dinv) {
  __shared__ double L[BS][BS + 1];
  __shared__ double I[BS][BS + 1];
  double* blk = A + static_cast<long long>(kb) * lda + kb;
  for (int e = threadIdx.x; e < BS * BS; e += kThreads) {
    const int r = e / BS, c = e % BS;
    L[r][c] = (c <= r) ? blk[static_cast<long long>(r) * lda + c] : 0.0;
  }
  __syncthreads();
  // unblocked right-looking Cholesky on the 64 x 64 block
  for (int j = 0; j < BS; ++j) {
    const double d = L[j][j];
    __syncthreads();
    if (threadIdx.x == 0) {
      if (!(d > 0.0)) atomicOr(&g_gptq_factor_err, kErrNotPositiveDefinite);
      L[j][j] = sqrt(d);
    }
    __syncthreads();
    const double dj = L[j][j];
    for (int r = j + 1 + threadIdx.x; r < BS; r += kThreads) L[r][j] = L[r][j] / dj;
    __syncthreads();
    for (int e = threadIdx.x; e < (BS - j - 1) * (BS - j - 1); e += kThreads) {
      const int r = j + 1 + e / (BS - j - 1), c = j + 1 + e % (BS - j - 1);
      if (c <= r) L[r][c] = fma(-L[r][j], L[c][j], L[r][c]);
    }
    __syncthreads();
  }
  // inverse of the lower factor by forward substitution, one column of the identity per
  // thread: column c of Linv solves L x = e_c
  if (threadIdx.x < BS) {
    const int c = threadIdx.x;
    for (int r = 0; r < BS; ++r) {
      double s = (r == c) ? 1.0 : 0.0;
      for (int k = c; k < r; ++k) s = fma(-L[r][k], I[k][c], s);
      I[r][c] = (r < c) ? 0.0 : s / L[r][r];
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < BS * BS; e += kThreads) {
    const int r = e / BS, c = e % BS;
    if (c <= r) blk[static_cast<long long>(r) * lda + c] = L[r][c];
    Dinv[e] = I[r][c];
  }
}

// dst (rows x 64, ldd) = src (rows x 64, lds)
__global__ void k_copy_cols64(const double* __restrict__ src, long long lds, double* __restrict__ dst,
                              long long ldd, int rows) {
  const long long e = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (e >= static_cast<long long>(rows) * BS) return;
  const long long r = e / BS, c = e % BS;
  dst[r * ldd + c] = src[r * lds + c];
}

// U[i][j] = float(Linv[K-1-i][K-1-j]) for j >= i, 0 below the diagonal.
__global__ void k_u_from_linv(const double* __restrict__ Linv, int K, float* __restrict__ U) {
  const long long e = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (e >= static_cast<long long>(K) * K) return;
  const int i = static_cast<int>(e / K), j = static_cast<int>(e % K);
  U[e] = (j >= i) ? static_cast<float>(Linv[static_cast<long long>(K - 1 - i) * K + (K - 1 - j)]) : 0.0f;
}

template <bool TA, bool TB>
cudaError_t gemm(int M, int N, int k_lo, int k_hi, double alpha, const double* A, long long lda, const double* B,
                 long long ldb, double beta, double* C, long long ldc, bool lower_only, bool b_lower, cudaStream_t s) {
  const dim3 grid((N + BS - 1) / BS, (M + BS - 1) / BS);
  k_gemm_f64<TA, TB><<<grid, kThreads, 0, s>>>(M, N, k_lo, k_hi, alpha, A, lda, B, ldb, beta, C, ldc,
                                              lower_only ? 1 : 0, b_lower ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace fac

size_t gptq_factor_workspace_bytes(int64_t K) {
  // A (then L) and Linv: K x K float64 each; the panel: K x 64; the diagonal blocks' inverses:
  // K x 64; the rows of the inverse in progress: 64 x K
  const size_t kk = static_cast<size_t>(K) * static_cast<size_t>(K) * sizeof(double);
  const size_t k64 = static_cast<size_t>(K) * fac::BS * sizeof(double);
  return 2 * kk + 3 * k64;
}

cudaError_t launch_gptq_factor(const float* X, int64_t n, int64_t K64, float* U, void* ws, cudaStream_t s) {
  using namespace fac;
  const int K = static_cast<int>(K64);
  const size_t kk = static_cast<size_t>(K) * static_cast<size_t>(K);
  double* A = reinterpret_cast<double*>(ws);
  double* Linv = A + kk;
  double* P = Linv + kk;                               // panel [K x 64]
  double* Dinv = P + static_cast<size_t>(K) * BS;      // diagonal inverses [K/64][64 x 64]
  double* T = Dinv + static_cast<size_t>(K) * BS;      // rows of the inverse in progress [64 x K]
  const int nb = K / BS;
  const dim3 tiles(nb, nb);
  cudaError_t e = cudaMemsetAsync(Linv, 0, kk * sizeof(double), s);
  if (e != cudaSuccess) return e;
  k_hessian_rev<<<tiles, kThreads, 0, s>>>(X, static_cast<int>(n), K, A);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  k_damp<<<1, kThreads, 0, s>>>(A, K, 0.01);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // Cholesky, block column by block column
  for (int b = 0; b < nb; ++b) {
    const int kb = b * BS, rest = K - kb - BS;
    k_potrf_block<<<1, kThreads, 0, s>>>(A, K, kb, Dinv + static_cast<size_t>(b) * BS * BS);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (rest == 0) break;
    double* panel = A + static_cast<size_t>(kb + BS) * K + kb;
    // P = panel Dinv^T  (the panel of L), then back into A
    e = gemm<false, true>(rest, BS, 0, BS, 1.0, panel, K, Dinv + static_cast<size_t>(b) * BS * BS, BS, 0.0, P, BS,
                          false, false, s);
    if (e != cudaSuccess) return e;
    const long long cells = static_cast<long long>(rest) * BS;
    k_copy_cols64<<<static_cast<unsigned>((cells + 255) / 256), 256, 0, s>>>(P, BS, panel, K, rest);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // trailing lower triangle: A22 -= P P^T
    double* a22 = A + static_cast<size_t>(kb + BS) * K + (kb + BS);
    e = gemm<false, true>(rest, rest, 0, BS, -1.0, P, BS, P, BS, 1.0, a22, K, true, false, s);
    if (e != cudaSuccess) return e;
  }
  // triangular inverse, block row by block row
  for (int b = 0; b < nb; ++b) {
    const int ib = b * BS;
    const double* di = Dinv + static_cast<size_t>(b) * BS * BS;
    // Linv[ib:ib+64, ib:ib+64] = inv(L[ib, ib]) (the blocks to its right stay zero and are
    // never read: the products below skip the zero upper triangle of Linv)
    k_copy_cols64<<<(BS * BS + 255) / 256, 256, 0, s>>>(di, BS, Linv + static_cast<size_t>(ib) * K + ib, K, BS);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (ib == 0) continue;
    // T = L[ib, 0:ib] Linv[0:ib, 0:ib]   (Linv lower: the inner range starts at each tile's column)
    e = gemm<false, false>(BS, ib, 0, ib, 1.0, A + static_cast<size_t>(ib) * K, K, Linv, K, 0.0, T, K, false, true, s);
    if (e != cudaSuccess) return e;
    // Linv[ib, 0:ib] = -inv(L[ib, ib]) T
    e = gemm<false, false>(BS, ib, 0, BS, -1.0, di, BS, T, K, 0.0, Linv + static_cast<size_t>(ib) * K, K, false,
                           false, s);
    if (e != cudaSuccess) return e;
  }
  const long long cells = static_cast<long long>(K) * K;
  k_u_from_linv<<<static_cast<unsigned>((cells + 255) / 256), 256, 0, s>>>(Linv, K, U);
  return cudaGetLastError();
}

}  // namespace wq
