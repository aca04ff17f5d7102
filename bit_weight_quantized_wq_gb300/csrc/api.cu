// The C ABI (include/wq.h): argument validation, per-shape dispatch, TMA descriptor
// encoding, status strings and the device error word.
#include <atomic>
#include <mutex>

#include "../../include/wq.h"
#include "internal.h"

namespace wq {

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

}  // namespace

cudaError_t make_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t dim0,
                         uint64_t dim1, uint64_t stride1_bytes, uint32_t box0, uint32_t box1,
                         CUtensorMapSwizzle swizzle, CUtensorMapL2promotion promo) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {dim0, dim1};
  const cuuint64_t strides[1] = {stride1_bytes};
  const cuuint32_t box[2] = {box0, box1};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle, promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

CUcontext current_context() {
  using CtxGetCurrentFn = CUresult (*)(CUcontext*);
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  CUcontext c = nullptr;
  if (fn && fn(&c) != CUDA_SUCCESS) c = nullptr;
  return c;
}

int device_sm_count() {
  // per-device cache; atomics because several host threads may make their first call at once
  static std::atomic<int> cached[64];
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64) {
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (n <= 0) return 1;
  if (dev >= 0 && dev < 64) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

cudaError_t set_smem_attr_once(const void* kern, size_t smem_bytes) {
  // (kernel, device) pairs whose dynamic shared-memory limit is already raised; guarded by a
  // mutex because several host threads may make their first call at once
  static std::mutex mu;
  static const void* done_kern[256];
  static int done_dev[256];
  static int n_done = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(mu);
  for (int i = 0; i < n_done; ++i)
    if (done_kern[i] == kern && done_dev[i] == dev) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem_bytes));
  if (e != cudaSuccess) return e;
  if (n_done < 256) {
    done_kern[n_done] = kern;
    done_dev[n_done] = dev;
    ++n_done;
  }
  return cudaSuccess;
}

}  // namespace wq

namespace {

constexpr int kMaxOverrides = 256;
struct ThresholdOverride {
  int fmt;
  int64_t K, N, T;
};
std::mutex g_thr_mu;
ThresholdOverride g_thr[kMaxOverrides];
int g_thr_n = 0;
int64_t g_thr_default[2] = {32, 32};   // the K = N = 8192 sweep's crossover, both formats

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

wq_status check_device_cached() {
  // Compute capability 10.3 (GB300) only: the kernels use sm_103a-specific instructions.
  static std::atomic<int> ok_dev[64];  // 0 unknown, 1 ok, 2 bad (atomic: concurrent first calls)
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return WQ_ERR_CUDA;
  if (dev >= 0 && dev < 64) {
    const int k = ok_dev[dev].load(std::memory_order_relaxed);
    if (k) return k == 1 ? WQ_OK : WQ_ERR_UNSUPPORTED_ARCH;
  }
  int maj = 0, min = 0;
  if (cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&min, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return WQ_ERR_CUDA;
  const bool ok = (maj == 10 && min == 3);
  if (dev >= 0 && dev < 64) ok_dev[dev].store(ok ? 1 : 2, std::memory_order_relaxed);
  return ok ? WQ_OK : WQ_ERR_UNSUPPORTED_ARCH;
}

wq_status check_linear_args(wq_fmt fmt, const uint16_t* X, int64_t M, int64_t K, int64_t N, const int32_t* Wq,
                            const void* scales, const uint16_t* zeros, uint16_t* Y) {
  if (fmt != WQ_FMT_INT4_G128_ASYM && fmt != WQ_FMT_MXFP4) return WQ_ERR_ARG;
  if (!X || !Wq || !scales || !Y) return WQ_ERR_NULL;
  if (fmt == WQ_FMT_INT4_G128_ASYM && !zeros) return WQ_ERR_NULL;
  if (fmt == WQ_FMT_MXFP4 && zeros) return WQ_ERR_ARG;
  if (M < 1 || N < 1 || K < 1) return WQ_ERR_SHAPE;
  if (M > (1LL << 30) || N > (1LL << 30) || K > (1LL << 30)) return WQ_ERR_SHAPE;
  if (K % (fmt == WQ_FMT_INT4_G128_ASYM ? 128 : 32) != 0) return WQ_ERR_SHAPE;
  if (!aligned16(X) || !aligned16(Wq) || !aligned16(scales) || !aligned16(Y) || (zeros && !aligned16(zeros)))
    return WQ_ERR_ALIGN;
  return WQ_OK;
}

wq_status from_cuda(cudaError_t e) { return e == cudaSuccess ? WQ_OK : WQ_ERR_CUDA; }

size_t round_up256(size_t b) { return (b + 255) / 256 * 256; }

}  // namespace

extern "C" {

wq_status wq_quantize_int4_g128(const float* W, int64_t N, int64_t K, int32_t* Wq, uint16_t* scales,
                                uint16_t* zeros, void* stream) {
  if (!W || !Wq || !scales || !zeros) return WQ_ERR_NULL;
  if (N < 1 || K < 128 || K % 128 != 0 || N > (1LL << 31) || K > (1LL << 31)) return WQ_ERR_SHAPE;
  if (!aligned16(W) || !aligned16(Wq) || !aligned16(scales) || !aligned16(zeros)) return WQ_ERR_ALIGN;
  wq_status st = check_device_cached();
  if (st != WQ_OK) return st;
  return from_cuda(wq::launch_quant_int4_g128(W, N, K, Wq, scales, zeros, static_cast<cudaStream_t>(stream)));
}

wq_status wq_quantize_mxfp4(const float* W, int64_t N, int64_t K, int32_t* Wq, uint8_t* scales, void* stream) {
  if (!W || !Wq || !scales) return WQ_ERR_NULL;
  if (N < 1 || K < 32 || K % 32 != 0 || N > (1LL << 31) || K > (1LL << 31)) return WQ_ERR_SHAPE;
  if (!aligned16(W) || !aligned16(Wq) || !aligned16(scales)) return WQ_ERR_ALIGN;
  wq_status st = check_device_cached();
  if (st != WQ_OK) return st;
  return from_cuda(wq::launch_quant_mxfp4(W, N, K, Wq, scales, static_cast<cudaStream_t>(stream)));
}

wq_status wq_gptq_int4_g128(const float* W, int64_t N, int64_t K, const float* U, int32_t* Wq, uint16_t* scales,
                            uint16_t* zeros, void* stream) {
  if (!W || !U || !Wq || !scales || !zeros) return WQ_ERR_NULL;
  if (N < 1 || K < 128 || K % 128 != 0 || N > (1LL << 30) || wq::gptq_rows_per_cta(K) < 1) return WQ_ERR_SHAPE;
  if (!aligned16(W) || !aligned16(U) || !aligned16(Wq) || !aligned16(scales) || !aligned16(zeros)) return WQ_ERR_ALIGN;
  wq_status st = check_device_cached();
  if (st != WQ_OK) return st;
  return from_cuda(wq::launch_gptq_int4_g128(W, N, K, U, Wq, scales, zeros, static_cast<cudaStream_t>(stream)));
}

size_t wq_gptq_workspace_bytes(int64_t K) {
  if (K < 128 || K % 128 != 0 || K > 46208) return 0;
  return wq::gptq_factor_workspace_bytes(K) + static_cast<size_t>(K) * static_cast<size_t>(K) * sizeof(float);
}

wq_status wq_gptq_factor(const float* X, int64_t n, int64_t K, float* U, void* workspace, size_t ws_bytes,
                         void* stream) {
  if (!X || !U) return WQ_ERR_NULL;
  if (n < 1 || n > (1LL << 30) || K < 128 || K % 128 != 0 || K > 46208) return WQ_ERR_SHAPE;
  if (!aligned16(X) || !aligned16(U)) return WQ_ERR_ALIGN;
  if (!workspace || ws_bytes < wq::gptq_factor_workspace_bytes(K)) return WQ_ERR_WORKSPACE;
  if (!aligned16(workspace)) return WQ_ERR_ALIGN;
  wq_status st = check_device_cached();
  if (st != WQ_OK) return st;
  return from_cuda(wq::launch_gptq_factor(X, n, K, U, workspace, static_cast<cudaStream_t>(stream)));
}

wq_status wq_gptq_int4_g128_calib(const float* W, int64_t N, int64_t K, const float* X, int64_t n, int32_t* Wq,
                                  uint16_t* scales, uint16_t* zeros, void* workspace, size_t ws_bytes, void* stream) {
  if (!W || !X || !Wq || !scales || !zeros) return WQ_ERR_NULL;
  if (N < 1 || N > (1LL << 30) || n < 1 || n > (1LL << 30) || K < 128 || K % 128 != 0 || K > 46208 ||
      wq::gptq_rows_per_cta(K) < 1)
    return WQ_ERR_SHAPE;
  if (!aligned16(W) || !aligned16(X) || !aligned16(Wq) || !aligned16(scales) || !aligned16(zeros)) return WQ_ERR_ALIGN;
  if (!workspace || ws_bytes < wq_gptq_workspace_bytes(K)) return WQ_ERR_WORKSPACE;
  if (!aligned16(workspace)) return WQ_ERR_ALIGN;
  wq_status st = check_device_cached();
  if (st != WQ_OK) return st;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* U = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + wq::gptq_factor_workspace_bytes(K));
  st = from_cuda(wq::launch_gptq_factor(X, n, K, U, workspace, s));
  if (st != WQ_OK) return st;
  return from_cuda(wq::launch_gptq_int4_g128(W, N, K, U, Wq, scales, zeros, s));
}

size_t wq_awq_workspace_bytes(int64_t N, int64_t K, int64_t n) {
  if (N < 1 || n < 1 || K < 128 || K % 128 != 0 || N > (1LL << 30) || K > (1LL << 30) || n > (1LL << 30)) return 0;
  return wq::awq_workspace_bytes(N, K, n);
}

wq_status wq_awq_int4_g128(const float* W, int64_t N, int64_t K, const float* X, int64_t n, int32_t* Wq,
                           uint16_t* scales, uint16_t* zeros, float* s, int32_t* alpha_index, double* losses,
                           void* workspace, size_t ws_bytes, void* stream) {
  if (!W || !X || !Wq || !scales || !zeros || !s) return WQ_ERR_NULL;
  if (N < 1 || n < 1 || K < 128 || K % 128 != 0 || N > (1LL << 30) || K > (1LL << 30) || n > (1LL << 30))
    return WQ_ERR_SHAPE;
  if (N * K > (1LL << 40)) return WQ_ERR_SHAPE;
  if (!aligned16(W) || !aligned16(X) || !aligned16(Wq) || !aligned16(scales) || !aligned16(zeros) || !aligned16(s) ||
      (alpha_index && (reinterpret_cast<uintptr_t>(alpha_index) & 3u)) ||
      (losses && (reinterpret_cast<uintptr_t>(losses) & 7u)))
    return WQ_ERR_ALIGN;
  if (!workspace || ws_bytes < wq::awq_workspace_bytes(N, K, n)) return WQ_ERR_WORKSPACE;
  if (!aligned16(workspace)) return WQ_ERR_ALIGN;
  wq_status st = check_device_cached();
  if (st != WQ_OK) return st;
  return from_cuda(wq::launch_awq_int4_g128(W, N, K, X, n, Wq, scales, zeros, s, alpha_index, losses, workspace,
                                            ws_bytes, static_cast<cudaStream_t>(stream)));
}

int64_t wq_dispatch_threshold(wq_fmt fmt, int64_t K, int64_t N) {
  if (fmt != WQ_FMT_INT4_G128_ASYM && fmt != WQ_FMT_MXFP4) return -1;
  std::lock_guard<std::mutex> lk(g_thr_mu);
  for (int i = 0; i < g_thr_n; ++i)
    if (g_thr[i].fmt == fmt && g_thr[i].K == K && g_thr[i].N == N) return g_thr[i].T;
  return g_thr_default[fmt];
}

wq_status wq_set_dispatch_threshold(wq_fmt fmt, int64_t K, int64_t N, int64_t T) {
  if (fmt != WQ_FMT_INT4_G128_ASYM && fmt != WQ_FMT_MXFP4) return WQ_ERR_ARG;
  if (T < 0 || T > wq::kDecodeMaxM || K < 0 || N < 0) return WQ_ERR_SHAPE;
  std::lock_guard<std::mutex> lk(g_thr_mu);
  if (K == 0 && N == 0) {
    g_thr_default[fmt] = T;
    return WQ_OK;
  }
  for (int i = 0; i < g_thr_n; ++i)
    if (g_thr[i].fmt == fmt && g_thr[i].K == K && g_thr[i].N == N) {
      g_thr[i].T = T;
      return WQ_OK;
    }
  if (g_thr_n >= kMaxOverrides) return WQ_ERR_SHAPE;
  g_thr[g_thr_n++] = {static_cast<int>(fmt), K, N, T};
  return WQ_OK;
}

size_t wq_gemm_workspace_bytes(wq_fmt fmt, int64_t M, int64_t K, int64_t N) {
  if (fmt != WQ_FMT_INT4_G128_ASYM && fmt != WQ_FMT_MXFP4) return 0;
  if (M < 1 || N < 1 || K < 1) return 0;
  size_t a = M <= wq::kDecodeMaxM ? wq::gemv_workspace_bytes(fmt, M, K, N) : 0;
  size_t b = wq::gemm_tc_workspace_bytes(fmt, M, K, N);
  return a > b ? a : b;
}

wq_status wq_gemv_w4a16(wq_fmt fmt, const uint16_t* X, int64_t M, int64_t K, int64_t N, const int32_t* Wq,
                        const void* scales, const uint16_t* zeros, uint16_t* Y, void* workspace, size_t ws_bytes,
                        void* stream) {
  wq_status st = check_linear_args(fmt, X, M, K, N, Wq, scales, zeros, Y);
  if (st != WQ_OK) return st;
  if (M > wq::kDecodeMaxM) return WQ_ERR_SHAPE;
  if ((N + wq::kDecodeBand - 1) / wq::kDecodeBand > wq::kWsMaxCounters) return WQ_ERR_SHAPE;
  const size_t need = wq::gemv_workspace_bytes(fmt, M, K, N);
  if (need > 0 && (!workspace || ws_bytes < need)) return WQ_ERR_WORKSPACE;
  if (workspace && !aligned16(workspace)) return WQ_ERR_ALIGN;
  st = check_device_cached();
  if (st != WQ_OK) return st;
  return from_cuda(wq::launch_gemv(fmt, X, M, K, N, Wq, scales, zeros, Y, workspace, ws_bytes,
                                   static_cast<cudaStream_t>(stream)));
}

wq_status wq_gemv_w4a16_noalloc(wq_fmt fmt, const uint16_t* X, int64_t M, int64_t K, int64_t N,
                                const int32_t* Wq, const void* scales, const uint16_t* zeros, uint16_t* Y,
                                void* stream) {
  wq_status st = check_linear_args(fmt, X, M, K, N, Wq, scales, zeros, Y);
  if (st != WQ_OK) return st;
  if (M > 16) return WQ_ERR_SHAPE;   // the library's array holds 16-row partial sums
  if ((N + wq::kDecodeBand - 1) / wq::kDecodeBand > wq::kWsMaxCounters) return WQ_ERR_SHAPE;
  st = check_device_cached();
  if (st != WQ_OK) return st;
  // Shapes whose scratch would not fit the library's fixed array (possible only on a device
  // with more SMs than it was sized for) are refused before anything is enqueued.
  if (wq::gemv_workspace_bytes(fmt, M, K, N) > wq::gemv_noalloc_scratch_bytes()) return WQ_ERR_SHAPE;
  return from_cuda(wq::launch_gemv_noalloc(fmt, X, M, K, N, Wq, scales, zeros, Y, static_cast<cudaStream_t>(stream)));
}

wq_status wq_gemm_tc_w4a16(wq_fmt fmt, const uint16_t* X, int64_t M, int64_t K, int64_t N, const int32_t* Wq,
                           const void* scales, const uint16_t* zeros, uint16_t* Y, void* workspace,
                           size_t ws_bytes, void* stream) {
  wq_status st = check_linear_args(fmt, X, M, K, N, Wq, scales, zeros, Y);
  if (st != WQ_OK) return st;
  const size_t need = wq::gemm_tc_workspace_bytes(fmt, M, K, N);
  if (need > 0 && (!workspace || ws_bytes < need)) return WQ_ERR_WORKSPACE;
  if (workspace && !aligned16(workspace)) return WQ_ERR_ALIGN;
  st = check_device_cached();
  if (st != WQ_OK) return st;
  return from_cuda(wq::launch_gemm_tc(fmt, X, M, K, N, Wq, scales, zeros, Y, workspace, ws_bytes,
                                      static_cast<cudaStream_t>(stream)));
}

wq_status wq_gemm_w4a16(wq_fmt fmt, const uint16_t* X, int64_t M, int64_t K, int64_t N, const int32_t* Wq,
                        const void* scales, const uint16_t* zeros, uint16_t* Y, void* workspace, size_t ws_bytes,
                        void* stream) {
  wq_status st = check_linear_args(fmt, X, M, K, N, Wq, scales, zeros, Y);
  if (st != WQ_OK) return st;
  if (M <= wq_dispatch_threshold(fmt, K, N))
    return wq_gemv_w4a16(fmt, X, M, K, N, Wq, scales, zeros, Y, workspace, ws_bytes, stream);
  return wq_gemm_tc_w4a16(fmt, X, M, K, N, Wq, scales, zeros, Y, workspace, ws_bytes, stream);
}

wq_status wq_gemv_w4a16_swiglu(wq_fmt fmt, const uint16_t* X, int64_t M, int64_t K, int64_t F, const int32_t* Wq,
                               const void* scales, const uint16_t* zeros, uint16_t* Y, void* workspace,
                               size_t ws_bytes, void* stream) {
  if (F < 8 || F % 8 != 0 || F > (1LL << 29)) return WQ_ERR_SHAPE;
  const int64_t N = 2 * F;
  wq_status st = check_linear_args(fmt, X, M, K, N, Wq, scales, zeros, Y);
  if (st != WQ_OK) return st;
  if (M > wq::kDecodeMaxM) return WQ_ERR_SHAPE;
  if ((N + wq::kDecodeBand - 1) / wq::kDecodeBand > wq::kWsMaxCounters) return WQ_ERR_SHAPE;
  const size_t need = wq::gemv_workspace_bytes(fmt, M, K, N);
  if (need > 0 && (!workspace || ws_bytes < need)) return WQ_ERR_WORKSPACE;
  if (workspace && !aligned16(workspace)) return WQ_ERR_ALIGN;
  st = check_device_cached();
  if (st != WQ_OK) return st;
  return from_cuda(wq::launch_gemv(fmt, X, M, K, N, Wq, scales, zeros, Y, workspace, ws_bytes,
                                   static_cast<cudaStream_t>(stream), wq::kEpiSwiglu));
}

wq_status wq_gemm_tc_w4a16_swiglu(wq_fmt fmt, const uint16_t* X, int64_t M, int64_t K, int64_t F,
                                  const int32_t* Wq, const void* scales, const uint16_t* zeros, uint16_t* Y,
                                  void* workspace, size_t ws_bytes, void* stream) {
  if (F < 8 || F % 8 != 0 || F > (1LL << 29)) return WQ_ERR_SHAPE;
  const int64_t N = 2 * F;
  wq_status st = check_linear_args(fmt, X, M, K, N, Wq, scales, zeros, Y);
  if (st != WQ_OK) return st;
  const size_t need = wq::gemm_tc_workspace_bytes(fmt, M, K, N);
  if (need > 0 && (!workspace || ws_bytes < need)) return WQ_ERR_WORKSPACE;
  if (workspace && !aligned16(workspace)) return WQ_ERR_ALIGN;
  st = check_device_cached();
  if (st != WQ_OK) return st;
  return from_cuda(wq::launch_gemm_tc(fmt, X, M, K, N, Wq, scales, zeros, Y, workspace, ws_bytes,
                                      static_cast<cudaStream_t>(stream), wq::kEpiSwiglu));
}

wq_status wq_gemm_w4a16_swiglu(wq_fmt fmt, const uint16_t* X, int64_t M, int64_t K, int64_t F, const int32_t* Wq,
                               const void* scales, const uint16_t* zeros, uint16_t* Y, void* workspace,
                               size_t ws_bytes, void* stream) {
  if (F < 8 || F % 8 != 0 || F > (1LL << 29)) return WQ_ERR_SHAPE;
  wq_status st = check_linear_args(fmt, X, M, K, 2 * F, Wq, scales, zeros, Y);
  if (st != WQ_OK) return st;
  if (M <= wq_dispatch_threshold(fmt, K, 2 * F))
    return wq_gemv_w4a16_swiglu(fmt, X, M, K, F, Wq, scales, zeros, Y, workspace, ws_bytes, stream);
  return wq_gemm_tc_w4a16_swiglu(fmt, X, M, K, F, Wq, scales, zeros, Y, workspace, ws_bytes, stream);
}

wq_status wq_gemm_w4a16_qkv(wq_fmt fmt, const uint16_t* X, int64_t M, int64_t K, int64_t Nq, int64_t Nkv,
                            const int32_t* Wq, const void* scales, const uint16_t* zeros, uint16_t* Yq, uint16_t* Yk,
                            uint16_t* Yv, void* workspace, size_t ws_bytes, void* stream) {
  if (Nq < 1 || Nkv < 1 || Nq > (1LL << 29) || Nkv > (1LL << 28)) return WQ_ERR_SHAPE;
  const int64_t N = Nq + 2 * Nkv;
  wq_status st = check_linear_args(fmt, X, M, K, N, Wq, scales, zeros, Yq);
  if (st != WQ_OK) return st;
  if (!Yk || !Yv) return WQ_ERR_NULL;
  if (!aligned16(Yk) || !aligned16(Yv)) return WQ_ERR_ALIGN;
  wq::OutSplit split{};
  split.y[0] = Yq;
  split.y[1] = Yk;
  split.y[2] = Yv;
  split.ld[0] = Nq;
  split.ld[1] = Nkv;
  split.ld[2] = Nkv;
  split.n1 = static_cast<int>(Nq);
  split.n2 = static_cast<int>(Nq + Nkv);
  const bool decode = M <= wq_dispatch_threshold(fmt, K, N);
  if (decode && (N + wq::kDecodeBand - 1) / wq::kDecodeBand > wq::kWsMaxCounters) return WQ_ERR_SHAPE;
  const size_t need = decode ? wq::gemv_workspace_bytes(fmt, M, K, N) : wq::gemm_tc_workspace_bytes(fmt, M, K, N);
  if (need > 0 && (!workspace || ws_bytes < need)) return WQ_ERR_WORKSPACE;
  if (workspace && !aligned16(workspace)) return WQ_ERR_ALIGN;
  st = check_device_cached();
  if (st != WQ_OK) return st;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (decode)
    return from_cuda(wq::launch_gemv(fmt, X, M, K, N, Wq, scales, zeros, Yq, workspace, ws_bytes, s, wq::kEpiSplit3,
                                     &split));
  return from_cuda(wq::launch_gemm_tc(fmt, X, M, K, N, Wq, scales, zeros, Yq, workspace, ws_bytes, s, wq::kEpiSplit3,
                                      &split));
}

wq_status wq_interleave_gate_up(const void* src, void* dst, int64_t F, int64_t row_bytes, void* stream) {
  if (!src || !dst) return WQ_ERR_NULL;
  if (F < 8 || F % 8 != 0 || row_bytes < 1 || F > (1LL << 30) || row_bytes > (1LL << 40) / F) return WQ_ERR_SHAPE;
  const uintptr_t s0 = reinterpret_cast<uintptr_t>(src), d0 = reinterpret_cast<uintptr_t>(dst);
  const uintptr_t bytes = static_cast<uintptr_t>(2 * F) * static_cast<uintptr_t>(row_bytes);
  if (s0 < d0 + bytes && d0 < s0 + bytes) return WQ_ERR_ARG;
  wq_status st = check_device_cached();
  if (st != WQ_OK) return st;
  return from_cuda(wq::launch_interleave_gate_up(src, dst, F, row_bytes, static_cast<cudaStream_t>(stream)));
}

const char* wq_status_str(wq_status s) {
  switch (s) {
    case WQ_OK: return "WQ_OK";
    case WQ_ERR_NULL: return "WQ_ERR_NULL: a required pointer is NULL";
    case WQ_ERR_SHAPE: return "WQ_ERR_SHAPE: size out of range or not a required multiple";
    case WQ_ERR_ALIGN: return "WQ_ERR_ALIGN: pointer not 16-byte aligned";
    case WQ_ERR_WORKSPACE: return "WQ_ERR_WORKSPACE: workspace missing or too small";
    case WQ_ERR_UNSUPPORTED_ARCH: return "WQ_ERR_UNSUPPORTED_ARCH: device is not compute capability 10.3";
    case WQ_ERR_CUDA: return "WQ_ERR_CUDA: CUDA call failed";
    case WQ_ERR_ARG: return "WQ_ERR_ARG: argument out of range";
  }
  return "unknown wq_status";
}

// ------------------------------------------------------------------ FP8 E4M3 W8A8
wq_status wq_quantize_fp8_weights(const float* W, int64_t N, int64_t K, uint8_t* Wq, float* scales, void* stream) {
  if (!W || !Wq || !scales) return WQ_ERR_NULL;
  if (N < 1 || K < 16 || K % 16 != 0 || N > (1LL << 30) || K > (1LL << 30)) return WQ_ERR_SHAPE;
  if (!aligned16(W) || !aligned16(Wq) || (reinterpret_cast<uintptr_t>(scales) & 3u)) return WQ_ERR_ALIGN;
  wq_status st = check_device_cached();
  if (st != WQ_OK) return st;
  return from_cuda(wq::launch_quant_fp8_rows(false, W, N, K, Wq, scales, static_cast<cudaStream_t>(stream)));
}

wq_status wq_quantize_fp8_activations(const uint16_t* X, int64_t M, int64_t K, uint8_t* Xq, float* scales,
                                      void* stream) {
  if (!X || !Xq || !scales) return WQ_ERR_NULL;
  if (M < 1 || K < 16 || K % 16 != 0 || M > (1LL << 30) || K > (1LL << 30)) return WQ_ERR_SHAPE;
  if (!aligned16(X) || !aligned16(Xq) || (reinterpret_cast<uintptr_t>(scales) & 3u)) return WQ_ERR_ALIGN;
  wq_status st = check_device_cached();
  if (st != WQ_OK) return st;
  return from_cuda(wq::launch_quant_fp8_rows(true, X, M, K, Xq, scales, static_cast<cudaStream_t>(stream)));
}

static wq_status check_fp8_gemm(int64_t M, int64_t K, int64_t N, const void* Wq, const float* s_w, uint16_t* Y) {
  if (!Wq || !s_w || !Y) return WQ_ERR_NULL;
  if (M < 1 || N < 1 || K < 16 || K % 16 != 0 || M > (1LL << 30) || N > (1LL << 30) || K > (1LL << 30))
    return WQ_ERR_SHAPE;
  if (!aligned16(Wq) || !aligned16(Y) || (reinterpret_cast<uintptr_t>(s_w) & 3u)) return WQ_ERR_ALIGN;
  return WQ_OK;
}

wq_status wq_gemm_fp8(const uint8_t* Xq, const float* s_x, int64_t M, int64_t K, int64_t N, const uint8_t* Wq,
                      const float* s_w, uint16_t* Y, void* stream) {
  if (!Xq || !s_x) return WQ_ERR_NULL;
  wq_status st = check_fp8_gemm(M, K, N, Wq, s_w, Y);
  if (st != WQ_OK) return st;
  if (!aligned16(Xq) || (reinterpret_cast<uintptr_t>(s_x) & 3u)) return WQ_ERR_ALIGN;
  st = check_device_cached();
  if (st != WQ_OK) return st;
  return from_cuda(wq::launch_gemm_fp8(Xq, s_x, M, K, N, Wq, s_w, Y, static_cast<cudaStream_t>(stream)));
}

size_t wq_gemm_w8a8_fp8_workspace_bytes(int64_t M, int64_t K) {
  if (M < 1 || K < 1) return 0;
  return round_up256(static_cast<size_t>(M) * static_cast<size_t>(K)) + round_up256(static_cast<size_t>(M) * 4);
}

wq_status wq_gemm_w8a8_fp8(const uint16_t* X, int64_t M, int64_t K, int64_t N, const uint8_t* Wq, const float* s_w,
                           uint16_t* Y, void* workspace, size_t ws_bytes, void* stream) {
  if (!X) return WQ_ERR_NULL;
  wq_status st = check_fp8_gemm(M, K, N, Wq, s_w, Y);
  if (st != WQ_OK) return st;
  if (!aligned16(X)) return WQ_ERR_ALIGN;
  if (!workspace || ws_bytes < wq_gemm_w8a8_fp8_workspace_bytes(M, K)) return WQ_ERR_WORKSPACE;
  if (!aligned16(workspace)) return WQ_ERR_ALIGN;
  st = check_device_cached();
  if (st != WQ_OK) return st;
  uint8_t* Xq = static_cast<uint8_t*>(workspace);
  float* s_x = reinterpret_cast<float*>(Xq + round_up256(static_cast<size_t>(M) * static_cast<size_t>(K)));
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = wq::launch_quant_fp8_rows(true, X, M, K, Xq, s_x, s);
  if (e != cudaSuccess) return WQ_ERR_CUDA;
  return from_cuda(wq::launch_gemm_fp8(Xq, s_x, M, K, N, Wq, s_w, Y, s));
}

// ------------------------------------------------------------------ W4A4 MXFP4
wq_status wq_mxfp4_weights_to_e4m3(const int32_t* Wq, const uint8_t* scales, int64_t N, int64_t K, uint8_t* Wq8,
                                   float* s_w, void* stream) {
  if (!Wq || !scales || !Wq8 || !s_w) return WQ_ERR_NULL;
  if (N < 1 || K < 32 || K % 32 != 0 || N > (1LL << 30) || K > (1LL << 30)) return WQ_ERR_SHAPE;
  if (!aligned16(Wq) || !aligned16(Wq8) || (reinterpret_cast<uintptr_t>(s_w) & 3u)) return WQ_ERR_ALIGN;
  wq_status st = check_device_cached();
  if (st != WQ_OK) return st;
  return from_cuda(wq::launch_mx_weights_to_e4m3(Wq, scales, N, K, Wq8, s_w, static_cast<cudaStream_t>(stream)));
}

wq_status wq_quantize_w4a4_activations(const uint16_t* X, int64_t M, int64_t K, uint8_t* Xq8, float* s_x,
                                       void* stream) {
  if (!X || !Xq8 || !s_x) return WQ_ERR_NULL;
  if (M < 1 || K < 32 || K % 32 != 0 || K > 131072 || M > (1LL << 30)) return WQ_ERR_SHAPE;
  if (!aligned16(X) || !aligned16(Xq8) || (reinterpret_cast<uintptr_t>(s_x) & 3u)) return WQ_ERR_ALIGN;
  wq_status st = check_device_cached();
  if (st != WQ_OK) return st;
  return from_cuda(wq::launch_quant_w4a4_act(X, M, K, Xq8, s_x, static_cast<cudaStream_t>(stream)));
}

wq_status wq_gemm_w4a4_mxfp4(const uint16_t* X, int64_t M, int64_t K, int64_t N, const uint8_t* Wq8, const float* s_w,
                             uint16_t* Y, void* workspace, size_t ws_bytes, void* stream) {
  if (!X) return WQ_ERR_NULL;
  wq_status st = check_fp8_gemm(M, K, N, Wq8, s_w, Y);
  if (st != WQ_OK) return st;
  if (K % 32 != 0 || K > 131072) return WQ_ERR_SHAPE;
  if (!aligned16(X)) return WQ_ERR_ALIGN;
  if (!workspace || ws_bytes < wq_gemm_w8a8_fp8_workspace_bytes(M, K)) return WQ_ERR_WORKSPACE;
  if (!aligned16(workspace)) return WQ_ERR_ALIGN;
  st = check_device_cached();
  if (st != WQ_OK) return st;
  uint8_t* Xq8 = static_cast<uint8_t*>(workspace);
  float* s_x = reinterpret_cast<float*>(Xq8 + round_up256(static_cast<size_t>(M) * static_cast<size_t>(K)));
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = wq::launch_quant_w4a4_act(X, M, K, Xq8, s_x, s);
  if (e != cudaSuccess) return WQ_ERR_CUDA;
  return from_cuda(wq::launch_gemm_fp8(Xq8, s_x, M, K, N, Wq8, s_w, Y, s));
}

wq_status wq_read_error_flags(uint32_t* out) {
  if (!out) return WQ_ERR_NULL;
  if (cudaDeviceSynchronize() != cudaSuccess) return WQ_ERR_CUDA;
  *out = wq::gemv_read_and_clear_error() | wq::gemm_tc_read_and_clear_error() |
         wq::gptq_read_and_clear_error() | wq::gptq_factor_read_and_clear_error() |
         wq::selftest_read_and_clear_error() | wq::fp8_read_and_clear_error();
  return cudaGetLastError() == cudaSuccess ? WQ_OK : WQ_ERR_CUDA;
}

wq_status wq_selftest_wait_timeout(uint32_t limit_us, uint32_t* timed_out, void* stream) {
  if (!timed_out) return WQ_ERR_NULL;
  if (limit_us < 1 || limit_us > 2000000) return WQ_ERR_ARG;
  wq_status st = check_device_cached();
  if (st != WQ_OK) return st;
  return from_cuda(wq::run_selftest_wait(static_cast<uint64_t>(limit_us) * 1000ull, timed_out,
                                         static_cast<cudaStream_t>(stream)));
}

wq_status wq_check_device(void) { return check_device_cached(); }

}  // extern "C"
