/*
 * wq.h -- C ABI of the GB300 (sm_103a) weight-only 4-bit quantized linear layer.
 *
 * Library: libwq.so (built from bit_weight_quantized_wq_gb300/csrc/).
 *
 * Two weight formats, both 0.53125 bytes per weight:
 *   WQ_FMT_INT4_G128_ASYM  asymmetric INT4, group of 128 along K, eight codes per int32
 *                          (low nibble first), one fp16 scale and one fp16 zero point per
 *                          (row, group).
 *   WQ_FMT_MXFP4           OCP MXFP4: E2M1 codes two per byte (element 2j in the low
 *                          nibble of byte j), one E8M0 scale byte per 32 elements along K.
 *
 * Conventions shared by every entry point
 *   - Row-major everywhere.  W is [N, K] (N output features, K input features), X is [M, K],
 *     Y is [M, N].  Wq is [N, K/8] int32 (equivalently [N, K/2] bytes).
 *   - fp16 and bf16 values cross the boundary as uint16_t bit patterns.
 *   - Every pointer is a DEVICE pointer on the current CUDA device, owned by the caller, and
 *     must be 16-byte aligned.  The library never allocates or frees device memory, never
 *     synchronizes, and enqueues work only on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) -- except wq_read_error_flags, which synchronizes the device to read
 *     the error word (and zeroes the library's own scratch array after a timed-out wait).
 *   - Argument errors are detected on the host before anything is enqueued and returned as
 *     a wq_status; nothing is launched then.  Launch failures return WQ_ERR_CUDA.  Device-side
 *     faults surface, as usual in CUDA, at the caller's next synchronization.
 *   - Every wait inside a kernel is bounded; a wait that runs out records a code readable
 *     with wq_read_error_flags() and the kernel returns early (its output is then invalid).
 *   - Non-finite weights give unspecified (but memory-safe) results.
 */
#ifndef WQ_H_
#define WQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  WQ_OK = 0,
  WQ_ERR_NULL = 1,             /* a required pointer is NULL                         */
  WQ_ERR_SHAPE = 2,            /* a size is out of range or not a multiple required  */
  WQ_ERR_ALIGN = 3,            /* a pointer is not 16-byte aligned                   */
  WQ_ERR_WORKSPACE = 4,        /* workspace missing or smaller than required         */
  WQ_ERR_UNSUPPORTED_ARCH = 5, /* current device is not compute capability 10.3      */
  WQ_ERR_CUDA = 6,             /* a CUDA runtime/driver call failed                  */
  WQ_ERR_ARG = 7               /* an enum argument is out of range                   */
} wq_status;

typedef enum { WQ_FMT_INT4_G128_ASYM = 0, WQ_FMT_MXFP4 = 1 } wq_fmt;

/*
 * Asymmetric INT4 quantize + pack, group size 128 along K.
 * Defined by: 推理优化与量化算子深度技术调研 §1.2 (asymmetric scale = (max-min)/(2^b-1),
 * zero_point = round(-min/scale), q = clamp(round(x/scale)+zp, 0, 2^b-1)) and
 * 第 1 章：推理加速全景 §4.1 (the b-bit form), with b = 4; packing per
 * 第 6 课：量化源码走读 (源码分层架构与生命周期: 8 INT4 codes in one int32 plus scale and zero
 * point tensors).  Per (row n, group g), float32 arithmetic:
 *   lo = min(min x, 0), hi = max(max x, 0); s32 = (hi - lo) / 15;
 *   s = fp16_rn(min(s32, 65504)), and s = 1 if that is 0; z = min(rint(-lo / s), 15);
 *   q = clamp(rint(x / s) + z, 0, 15).
 *   (The min on s32 saturates the scale of a group whose range exceeds 15 * 65504 at the
 *   largest finite fp16 value instead of +inf; its values beyond the range clip.  The min on
 *   z keeps the zero point a code when the stored scale is far below s32, which happens only
 *   for such groups and for fp16-subnormal scales, |x| below about 1e-6.)
 *   W       [N, K]    float32 input.
 *   Wq      [N, K/8]  int32 output; code k = 8j+i in bits 4i..4i+3 of word j.
 *   scales  [N, K/128] fp16 bits output.
 *   zeros   [N, K/128] fp16 bits output (small non-negative integers).
 * Errors: WQ_ERR_SHAPE unless N >= 1 and K >= 128, K % 128 == 0.
 */
wq_status wq_quantize_int4_g128(const float* W, int64_t N, int64_t K, int32_t* Wq,
                                uint16_t* scales, uint16_t* zeros, void* stream);

/*
 * OCP MXFP4 quantize + pack, one E8M0 scale per 32 elements along K.
 * Defined by: 大模型量化推理引擎全景大复盘 (里程碑六 / 方程 3: 32 four-bit elements share one
 * E8M0 scale; the simulator's scale 2^ceil(log2(amax/6)) on float32).  Per (row n, block b):
 *   amax = max|x|; r = amax / 6 (float32); e = ceil(log2 r) exactly, clamped to [-127, 127]
 *   (e = -127 when r == 0); v = x * 2^-e; magnitude code = nearest of
 *   {0, .5, 1, 1.5, 2, 3, 4, 6}, ties to the even code, saturating at 6; code = sign(x)<<3 |
 *   magnitude (sign bit of x kept, so -0 -> 8); an all-zero block has scale byte 0, codes 0.
 *   W       [N, K]    float32 input.
 *   Wq      [N, K/8]  int32 output == [N, K/2] bytes, element 2j in the low nibble of byte j.
 *   scales  [N, K/32] uint8 output, E8M0 byte e + 127.
 * Errors: WQ_ERR_SHAPE unless N >= 1 and K >= 32, K % 32 == 0.
 */
wq_status wq_quantize_mxfp4(const float* W, int64_t N, int64_t K, int32_t* Wq,
                            uint8_t* scales, void* stream);

/*
 * GPTQ quantize + pack into the WQ_FMT_INT4_G128_ASYM format: the columns of W are quantized
 * in order, each column's quantization error compensated on the columns not yet quantized
 * through the inverse Hessian of the layer's calibration objective.
 * Defined by: 第 1 章：推理加速全景 §4.2 (objective sum_j (W_j - Q(W_j))^T H (W_j - Q(W_j)) with
 * H = 2 X^T X + lambda I; quantize column i, e_i = W[i] - W_q[i], W[j] -= (e_i / H^-1[i,i])
 * H^-1[i,j] for j > i; H^-1 through its Cholesky factor) and 推理优化与量化算子深度技术调研 §1.3.
 * With U the upper Cholesky factor of H^-1 (H^-1 = U^T U) the ratio H^-1[i,j] / H^-1[i,i] of
 * the update is U[i,j] / U[i,i], so for every row, in float32 with each operation rounded on
 * its own:
 *   at i % 128 == 0: s, z of group i/128 from the row's CURRENT values of its 128 columns, by
 *                    the rules of wq_quantize_int4_g128;
 *   q_i = clamp(rint(w_i / s) + z, 0, 15);  e_i = (w_i - (q_i - z) s) / U[i,i];
 *   w_j = w_j - e_i * U[i,j]  for j > i.
 * With U diagonal (no correlation between input channels) this is wq_quantize_int4_g128.
 *   W       [N, K] float32 input (not modified).
 *   U       [K, K] float32, row-major: the upper Cholesky factor of H^-1 for the layer's
 *           calibration activations (the caller computes H and the factor; only the upper
 *           triangle including the positive diagonal is read).
 *   Wq, scales, zeros   outputs, as wq_quantize_int4_g128.
 * Work: N K^2 / 2 multiply-subtracts; rows are independent.
 * Errors: WQ_ERR_NULL; WQ_ERR_SHAPE unless N >= 1, K >= 128, K % 128 == 0 and K <= 46208
 *         (a row's values and codes must fit one CTA's shared memory); WQ_ERR_ALIGN;
 *         WQ_ERR_UNSUPPORTED_ARCH; WQ_ERR_CUDA.
 */
wq_status wq_gptq_int4_g128(const float* W, int64_t N, int64_t K, const float* U, int32_t* Wq,
                            uint16_t* scales, uint16_t* zeros, void* stream);

/*
 * GPTQ's inverse-Hessian factor from calibration activations, computed on the device:
 *   H = 2 X^T X + lambda I,  lambda = 0.01 * mean(diag(2 X^T X)),  U upper triangular with
 *   H^-1 = U^T U and a positive diagonal -- the factor wq_gptq_int4_g128 takes.
 * Defined by: 第 1 章：推理加速全景 §4.2 (H = 2 X^T X + lambda I over the calibration set; H^-1
 * through its Cholesky factor) and 推理优化与量化算子深度技术调研 §1.3 (a few hundred calibration
 * samples, 128 typically).  The pages give no value for lambda; 1 % of the mean diagonal is
 * used.  Computed in float64: a Cholesky factorisation of H with its row and column order
 * reversed, J H J = L L^T, and U = J L^-1 J (the unique upper factor of H^-1), rounded to
 * float32 once at the end.  Every sum runs in a fixed order (reproducible run to run).
 *   X       [n, K] float32 calibration activations (n >= 1).
 *   U       [K, K] float32 output, row-major, zero below the diagonal.
 *   workspace / ws_bytes: device scratch of at least wq_gptq_workspace_bytes(K) bytes (about
 *           16 K^2 bytes: float64 H and its inverse factor); no initialisation needed.
 * A non-positive Cholesky pivot (H not positive definite, e.g. X all zero) records bit 1 << 6
 * in the error word (wq_read_error_flags) and leaves NaN in U.
 * Work: about K^3 float64 multiply-adds (the factorisation and the triangular inverse) plus
 * n K^2 for H.
 * Errors: WQ_ERR_NULL; WQ_ERR_SHAPE unless n >= 1, K >= 128, K % 128 == 0, K <= 46208;
 *         WQ_ERR_ALIGN; WQ_ERR_WORKSPACE; WQ_ERR_UNSUPPORTED_ARCH; WQ_ERR_CUDA.
 */
size_t wq_gptq_workspace_bytes(int64_t K);
wq_status wq_gptq_factor(const float* X, int64_t n, int64_t K, float* U, void* workspace, size_t ws_bytes,
                         void* stream);

/*
 * GPTQ end to end from calibration activations: wq_gptq_factor into the workspace, then the
 * wq_gptq_int4_g128 sweep with that factor.  Arguments, outputs and errors as those two calls;
 * workspace / ws_bytes at least wq_gptq_workspace_bytes(K) (which includes room for U).
 */
wq_status wq_gptq_int4_g128_calib(const float* W, int64_t N, int64_t K, const float* X, int64_t n, int32_t* Wq,
                                  uint16_t* scales, uint16_t* zeros, void* workspace, size_t ws_bytes,
                                  void* stream);

/*
 * AWQ: scales the salient input channels of W before INT4 g128 quantization, the scale's
 * exponent chosen by a grid search on calibration activations.
 * Defined by: 第 1 章：推理加速全景 §4.4 (importance_j = mean |X_j| over the calibration set;
 * the top 1 % channels are salient; s_j = importance_j ^ alpha, alpha by grid search in [0, 1];
 * quantize W' = W diag(s)), 推理优化与量化算子深度技术调研 §1.3 (W'' = W * s, x'' = x / s, s minimising
 * || Q(W * s) * (x / s) - W x ||) and 量化与加速 (only the top 1 % channels are scaled).
 * Computed:
 *   importance_j = (sum over the n samples, in order, of |X[n, j]|) / n in float64;
 *   salient = the ceil(K / 100) channels of largest importance (equal: lower index first);
 *   for a = 0 .. 20: s_j = float32(importance_j ^ (a / 20)) on salient channels with
 *     importance > 0, else 1; L(a) = || X (Q(W diag(s)) diag(s)^-1 - W)^T ||_F^2 (fp32 products,
 *     fp64 sums of squares);  a* = the smallest a with minimal L(a);
 *   Wq, scales, zeros = wq_quantize_int4_g128 of float32(W_ij * s*_j).
 * At run time the layer's activations must be divided by s* (x / s*, usually folded into the
 * operation that produces x).
 *   W       [N, K] float32.       X  [n, K] float32 calibration activations (n >= 1).
 *   Wq, scales, zeros   outputs, as wq_quantize_int4_g128.
 *   s       [K] float32 output: s*.
 *   alpha_index   int32 output (may be NULL): a*.      losses  [21] double output (may be NULL).
 *   workspace / ws_bytes: at least wq_awq_workspace_bytes(N, K, n) bytes of device memory
 *           (includes an N x K fp32 scratch matrix); no initialisation needed.
 * Errors: WQ_ERR_NULL; WQ_ERR_SHAPE unless N >= 1, n >= 1, K >= 128, K % 128 == 0;
 *         WQ_ERR_ALIGN (losses: 8 bytes; the others 16); WQ_ERR_WORKSPACE;
 *         WQ_ERR_UNSUPPORTED_ARCH; WQ_ERR_CUDA.
 */
size_t wq_awq_workspace_bytes(int64_t N, int64_t K, int64_t n);
wq_status wq_awq_int4_g128(const float* W, int64_t N, int64_t K, const float* X, int64_t n, int32_t* Wq,
                           uint16_t* scales, uint16_t* zeros, float* s, int32_t* alpha_index, double* losses,
                           void* workspace, size_t ws_bytes, void* stream);

/*
 * Bytes of workspace wq_gemm_w4a16 / wq_gemv_w4a16 / wq_gemm_tc_w4a16 need for this shape.
 * Every layout starts with the same header: 64 KiB of split-K counters (the tensor-core
 * kernel's, when it splits the tiles of a last, partial wave along K), then 10 MiB for the
 * decode kernel's split-K exchange (the partial sums of CTAs sharing a band, where 0 means
 * "not posted yet"); the decode kernel uses only the part of it its shape needs, the
 * tensor-core kernel's other scratch comes after it.  The size depends on the device's SM
 * count, so query it on the device that runs the call.  Zero the workspace once before its
 * first use; every call that completes leaves the header at zero again, so one workspace can
 * serve calls of any shape and either kernel (after a call that reported a timed-out wait,
 * zero it again).  One workspace must not be used by two calls that can run at the same
 * time.  Returns 0 for invalid arguments, and 0 when the shape needs no workspace.
 */
size_t wq_gemm_workspace_bytes(wq_fmt fmt, int64_t M, int64_t K, int64_t N);

/*
 * Y = X * dequant(Wq)^T, bf16 activations, fp32 accumulation, bf16 output.
 * Defined by: 推理优化与量化算子深度技术调研 §1.2 (dequantization fused into the GEMM,
 * x_deq = (q - zp) * scale, before the multiply) and 第 6 课：量化源码走读 (W4A16 layer; the
 * "apply" step chooses a bandwidth kernel for small batch and a compute kernel for large
 * batch).  Dispatches on M: M <= T(fmt, K, N) runs the decode GEMV (T <= 64), otherwise the
 * tcgen05 tensor-core GEMM.
 *   X       [M, K] bf16 bits.
 *   Wq      [N, K/8] int32 (format fmt).
 *   scales  INT4: [N, K/128] fp16 bits; MXFP4: [N, K/32] uint8.
 *   zeros   INT4: [N, K/128] fp16 bits; MXFP4: must be NULL.
 *   Y       [M, N] bf16 bits output.
 *   workspace / ws_bytes: device scratch of at least wq_gemm_workspace_bytes(fmt, M, K, N)
 *           bytes (see there); may be NULL when that is 0.
 * Errors: WQ_ERR_SHAPE unless M >= 1, N >= 1, K % 128 == 0 (INT4) or K % 32 == 0 (MXFP4);
 *         WQ_ERR_NULL, WQ_ERR_ALIGN, WQ_ERR_WORKSPACE, WQ_ERR_ARG, WQ_ERR_UNSUPPORTED_ARCH,
 *         WQ_ERR_CUDA.
 */
wq_status wq_gemm_w4a16(wq_fmt fmt, const uint16_t* X, int64_t M, int64_t K, int64_t N,
                        const int32_t* Wq, const void* scales, const uint16_t* zeros,
                        uint16_t* Y, void* workspace, size_t ws_bytes, void* stream);

/*
 * The decode kernel alone (same arguments and errors as wq_gemm_w4a16; requires M <= 64
 * and N <= 2097152; M > 32 runs as consecutive 32-row launches).
 * Streams the packed weights with TMA, unpacks in registers and applies the group scale in
 * fp32 after exact integer-valued tensor-core products; the zero point enters as (q - z),
 * the cross term of 第 6 课：量化源码走读 §3.
 */
wq_status wq_gemv_w4a16(wq_fmt fmt, const uint16_t* X, int64_t M, int64_t K, int64_t N,
                        const int32_t* Wq, const void* scales, const uint16_t* zeros,
                        uint16_t* Y, void* workspace, size_t ws_bytes, void* stream);

/*
 * The decode kernel without a workspace argument, for callers that cannot allocate device
 * memory when they run the layer -- for example code running inside a host framework that
 * owns every device allocation and gives extensions none, or a latency-critical loop where
 * the synchronisation a cudaMalloc implies is not acceptable.  The pages have no counterpart:
 * this is a deployment convenience of this library, not part of the method.
 * Same arguments, results and errors as wq_gemv_w4a16 minus workspace/ws_bytes; allocates
 * nothing (no cudaMalloc/cudaFree, no allocating library call).  Its scratch (the split-K
 * exchange area, in the workspace layout) is one library-owned device array of 64 KiB +
 * 5 MiB, held by
 * every GPU that loads the library until the process exits; it covers M <= 16 and
 * N <= 2097152 (one CTA per SM, at most 160), and a shape it cannot hold (M > 16) is refused
 * with WQ_ERR_SHAPE before anything is enqueued.
 * The first call on each device looks up the array's device address (cudaGetSymbolAddress,
 * with that device current); make that first call before any stream capture.  The address is
 * looked up again when the device's current context has changed since (cudaDeviceReset
 * unloads the module, and the array may come back elsewhere); after a reset, make one call
 * outside any capture again before capturing.  The array starts zeroed and each call that
 * completes leaves it so (the call enqueues the kernel alone); after a call that reported a
 * timed-out wait, wq_read_error_flags zeroes it again.  All calls on a device share the one
 * array: calls that can overlap on the GPU (other streams, other threads) race and corrupt
 * each other's results -- serialise them.
 */
wq_status wq_gemv_w4a16_noalloc(wq_fmt fmt, const uint16_t* X, int64_t M, int64_t K, int64_t N,
                                const int32_t* Wq, const void* scales, const uint16_t* zeros,
                                uint16_t* Y, void* stream);

/*
 * The tensor-core (tcgen05, TMEM accumulator) kernel alone, for any M >= 1 (same arguments
 * and errors as wq_gemm_w4a16).  INT4: the dequantized weights (q - z) * s enter the tensor
 * core as fp16, so they must lie inside the fp16 range (|w| <= 65504; beyond it the outputs
 * are unspecified); activations of any finite bf16 magnitude are carried into fp16 exactly by
 * a power-of-two scale per row.
 */
wq_status wq_gemm_tc_w4a16(wq_fmt fmt, const uint16_t* X, int64_t M, int64_t K, int64_t N,
                           const int32_t* Wq, const void* scales, const uint16_t* zeros,
                           uint16_t* Y, void* workspace, size_t ws_bytes, void* stream);

/*
 * The fused gate+up projection of a SwiGLU FFN with its activation in the epilogue:
 *   Y[M, F] = SiLU(X * dequant(W_gate)^T) * (X * dequant(W_up)^T),   SiLU(g) = g / (1 + e^-g).
 * Defined by: 推理优化与量化算子深度技术调研 §4.6 (GEMM + activation fusion: W_gate and W_up
 * stacked into one GEMM, SiLU(gate) * up computed in registers, the intermediate never written
 * to memory).  The activation is applied to the fp32 accumulators; Y is rounded to bf16 once.
 * No bias (the SwiGLU projections of LLaMA-style models have none).
 *   X       [M, K] bf16 bits.
 *   F       output features (the FFN's intermediate size); F >= 8, F % 8 == 0.
 *   Wq, scales, zeros
 *           the packed weight of the stacked [W_gate; W_up] (2F rows, format fmt, same
 *           per-row layouts as wq_gemm_w4a16 with N = 2F), with its rows in the INTERLEAVED
 *           order of wq_interleave_gate_up (apply it to each of the three arrays).
 *   Y       [M, F] bf16 bits output.
 *   workspace / ws_bytes: at least wq_gemm_workspace_bytes(fmt, M, K, 2F) bytes.
 * Dispatch, errors and workspace rules as wq_gemm_w4a16 with N = 2F (threshold
 * T(fmt, K, 2F)); WQ_ERR_SHAPE also when F % 8 != 0.
 */
wq_status wq_gemm_w4a16_swiglu(wq_fmt fmt, const uint16_t* X, int64_t M, int64_t K, int64_t F,
                               const int32_t* Wq, const void* scales, const uint16_t* zeros,
                               uint16_t* Y, void* workspace, size_t ws_bytes, void* stream);

/* The decode kernel alone with the SwiGLU epilogue (M <= 64, 2F <= 2097152). */
wq_status wq_gemv_w4a16_swiglu(wq_fmt fmt, const uint16_t* X, int64_t M, int64_t K, int64_t F,
                               const int32_t* Wq, const void* scales, const uint16_t* zeros,
                               uint16_t* Y, void* workspace, size_t ws_bytes, void* stream);

/* The tensor-core kernel alone with the SwiGLU epilogue (any M >= 1). */
wq_status wq_gemm_tc_w4a16_swiglu(wq_fmt fmt, const uint16_t* X, int64_t M, int64_t K, int64_t F,
                                  const int32_t* Wq, const void* scales, const uint16_t* zeros,
                                  uint16_t* Y, void* workspace, size_t ws_bytes, void* stream);

/*
 * The fused QKV projection with its output split into Q, K and V:
 *   [Q | K | V] = X * dequant([W_Q; W_K; W_V])^T,  Q [M, Nq], K [M, Nkv], V [M, Nkv].
 * Defined by: 推理优化与量化算子深度技术调研 §4.2 (the fused QKV projection: one GEMM over the
 * stacked W_Q, W_K, W_V, then the result split into Q, K and V).  The split is done by the
 * kernels' epilogue, which writes each output column straight to its tensor, so the fused
 * [M, Nq + 2 Nkv] result is never written.  With grouped-query attention (H_q query heads and
 * H_kv key/value heads of d_head each) Nq = H_q d_head and Nkv = H_kv d_head.
 *   X       [M, K] bf16 bits.
 *   Wq, scales, zeros   the packed stacked weight of N = Nq + 2 Nkv rows (W_Q rows, then W_K,
 *           then W_V), format fmt, the layouts of wq_gemm_w4a16.
 *   Yq      [M, Nq], Yk [M, Nkv], Yv [M, Nkv] bf16 bits outputs, row-major, 16-byte aligned,
 *           three distinct buffers.
 *   workspace / ws_bytes: at least wq_gemm_workspace_bytes(fmt, M, K, Nq + 2 Nkv) bytes.
 * Arithmetic, dispatch (T(fmt, K, Nq + 2 Nkv)), errors and workspace rules as wq_gemm_w4a16;
 * WQ_ERR_SHAPE also unless Nq >= 1 and Nkv >= 1; WQ_ERR_NULL for a NULL output.
 */
wq_status wq_gemm_w4a16_qkv(wq_fmt fmt, const uint16_t* X, int64_t M, int64_t K, int64_t Nq, int64_t Nkv,
                            const int32_t* Wq, const void* scales, const uint16_t* zeros, uint16_t* Yq,
                            uint16_t* Yk, uint16_t* Yv, void* workspace, size_t ws_bytes, void* stream);

/*
 * Row re-layout of a stacked [gate; up] array (2F rows of row_bytes bytes each: the packed
 * codes, the scales or the zeros of the fused gate+up weight) into the order the SwiGLU
 * entry points read: gate and up rows alternate in blocks of 8,
 *   dst row 16q + 8h + i = src row h*F + 8q + i     (h = 0: gate, h = 1: up; i < 8).
 * A one-time offline transform, as the weight re-layout after loading of
 * 第 6 课：量化源码走读 §2.  Row-wise quantization commutes with it, so it may equally be
 * applied to the float weight before wq_quantize_*.
 *   src, dst  device pointers to 2F * row_bytes bytes; distinct, non-overlapping buffers.
 *             Here (only) any alignment is accepted; 16-byte aligned bases and
 *             row_bytes % 16 == 0 copy 16 bytes at a time.
 * Errors: WQ_ERR_NULL; WQ_ERR_SHAPE unless F >= 8, F % 8 == 0, row_bytes >= 1; WQ_ERR_ARG if
 *         the buffers overlap; WQ_ERR_UNSUPPORTED_ARCH; WQ_ERR_CUDA.
 */
wq_status wq_interleave_gate_up(const void* src, void* dst, int64_t F, int64_t row_bytes, void* stream);

/*
 * Dispatch threshold T(fmt, K, N): wq_gemm_w4a16 uses the decode kernel when M <= T.
 * wq_set_dispatch_threshold overrides it for one (fmt, K, N) (T in [0, 64]; K = N = 0 sets
 * the default for the format).  Returns WQ_ERR_ARG / WQ_ERR_SHAPE on bad input.  Host-side
 * state, process-wide, not thread-safe against concurrent calls.
 */
int64_t wq_dispatch_threshold(wq_fmt fmt, int64_t K, int64_t N);
wq_status wq_set_dispatch_threshold(wq_fmt fmt, int64_t K, int64_t N, int64_t T);

/* Human-readable name of a status. */
const char* wq_status_str(wq_status s);

/*
 * Reads (and clears) the device-side error word of the current device: 0 when no bounded
 * wait ran out since the last read.  Synchronizes the device.  When a decode kernel's split-K
 * wait ran out (bit 1 << 3), it also zeroes the scratch array of wq_gemv_w4a16_noalloc.
 */
wq_status wq_read_error_flags(uint32_t* out);

/*
 * Diagnostic of the bounded waits every kernel uses: launches one CTA that waits on an
 * mbarrier phase nothing completes, with a limit of limit_us microseconds (1 .. 2000000).
 * The wait runs out, records bit 1 << 5 in the error word (see wq_read_error_flags) and the
 * kernel returns; *timed_out (host) receives 1.  Synchronizes `stream`.  No fault, trap or
 * endless loop is involved, so the context stays usable.
 * Errors: WQ_ERR_NULL, WQ_ERR_ARG, WQ_ERR_UNSUPPORTED_ARCH, WQ_ERR_CUDA.
 */
wq_status wq_selftest_wait_timeout(uint32_t limit_us, uint32_t* timed_out, void* stream);

/*
 * W8A8 in FP8 E4M3 -- the large-batch prefill format of 第 6 课：量化源码走读 §4 (W4A16 for
 * small-batch decode, FP8 for large-batch prefill); the format of 推理优化与量化算子深度技术调研
 * §1.4 (E4M3 tensors stored as torch.float8_e4m3fn with their FP32 scales beside them) and
 * 量化与加速's format table (E4M3, +-448).
 *
 * Row quantization (both operands): per row r, s[r] = fp32(max_k |A[r, k]| / 448) (a zero
 * row gets 1), and code[r, k] = E4M3(fp32(A[r, k] / s[r])), round to nearest with ties to the
 * even code, saturating at +-448, the sign kept on a zero.  Codes and scales are bit-exact
 * run to run and against the library's CPU reference.
 *   wq_quantize_fp8_weights:     W [N, K] float32 -> Wq [N, K] uint8, scales [N] float32 (one
 *                                per output channel; offline).
 *   wq_quantize_fp8_activations: X [M, K] bf16 bits -> Xq [M, K] uint8, scales [M] float32
 *                                (one per token, computed from the token's own values).
 * Errors: WQ_ERR_NULL; WQ_ERR_SHAPE unless rows >= 1 and K % 16 == 0 (K >= 16);
 *         WQ_ERR_ALIGN (arrays 16-byte aligned, scales 4-byte); WQ_ERR_UNSUPPORTED_ARCH;
 *         WQ_ERR_CUDA.
 */
wq_status wq_quantize_fp8_weights(const float* W, int64_t N, int64_t K, uint8_t* Wq, float* scales, void* stream);
wq_status wq_quantize_fp8_activations(const uint16_t* X, int64_t M, int64_t K, uint8_t* Xq, float* scales,
                                      void* stream);

/*
 * Y[m, n] = bf16( s_x[m] * s_w[n] * sum_k E4M3(Xq[m, k]) * E4M3(Wq[n, k]) ): exact products,
 * fp32 accumulation on the tensor cores (tcgen05.mma kind::f8f6f4), the two scales applied
 * to the fp32 accumulator in the epilogue.
 *   Xq [M, K] uint8, s_x [M] float32 (wq_quantize_fp8_activations); Wq [N, K] uint8, s_w [N]
 *   float32 (wq_quantize_fp8_weights); Y [M, N] bf16 bits output.
 * Errors: WQ_ERR_NULL; WQ_ERR_SHAPE unless M, N >= 1 and K % 16 == 0 (K >= 16); WQ_ERR_ALIGN;
 *         WQ_ERR_UNSUPPORTED_ARCH; WQ_ERR_CUDA.
 */
wq_status wq_gemm_fp8(const uint8_t* Xq, const float* s_x, int64_t M, int64_t K, int64_t N, const uint8_t* Wq,
                      const float* s_w, uint16_t* Y, void* stream);

/*
 * The W8A8 layer from bf16 activations: quantizes X per token into the workspace
 * (wq_quantize_fp8_activations), then wq_gemm_fp8; both launches on `stream`.
 *   workspace / ws_bytes: at least wq_gemm_w8a8_fp8_workspace_bytes(M, K) bytes (M K bytes of
 *   codes and M scales), 16-byte aligned; its content on entry is irrelevant.
 * Errors as wq_gemm_fp8, plus WQ_ERR_WORKSPACE.
 */
size_t wq_gemm_w8a8_fp8_workspace_bytes(int64_t M, int64_t K);
wq_status wq_gemm_w8a8_fp8(const uint16_t* X, int64_t M, int64_t K, int64_t N, const uint8_t* Wq, const float* s_w,
                           uint16_t* Y, void* workspace, size_t ws_bytes, void* stream);

/*
 * W4A4 in MXFP4 -- 第 6 课：量化源码走读 (量化范式与精度矩阵: NVFP4/MXFP4 micro-scaling quantizes
 * weights and activations to 4 bits with one shared scale per small block, the activations on
 * the fly); the block format of 大模型量化推理引擎全景大复盘 (里程碑六 / 方程 3).  Executed on the
 * FP8 tensor-core path (wq_gemm_fp8): every MXFP4 value E2M1(c) 2^e is the E4M3 value
 * E2M1(c) 2^(e - E) times the row's power of two 2^E, exactly for every block within 14
 * binades of the row's largest block (E = that block's exponent - 6); a block further below
 * is rounded to E4M3 (zero beyond 2^-13 of the largest).
 *   wq_mxfp4_weights_to_e4m3:     MXFP4 weights as wq_quantize_mxfp4 writes them (Wq [N, K/8]
 *                                 int32, scales [N, K/32] E8M0) -> Wq8 [N, K] E4M3 codes and
 *                                 s_w [N] float32 powers of two (once per layer).
 *   wq_quantize_w4a4_activations: X [M, K] bf16 bits quantized per token row by exactly the
 *                                 rules of wq_quantize_mxfp4, then re-encoded the same way ->
 *                                 Xq8 [M, K], s_x [M].
 *   wq_gemm_w4a4_mxfp4:           the layer from bf16 activations: the activation quantizer into
 *                                 the workspace (wq_gemm_w8a8_fp8_workspace_bytes(M, K) bytes),
 *                                 then wq_gemm_fp8 with the powers of two as the row scales.
 * Errors: WQ_ERR_NULL; WQ_ERR_SHAPE unless K % 32 == 0 (activations: K <= 131072); WQ_ERR_ALIGN;
 *         WQ_ERR_WORKSPACE; WQ_ERR_UNSUPPORTED_ARCH; WQ_ERR_CUDA.
 */
wq_status wq_mxfp4_weights_to_e4m3(const int32_t* Wq, const uint8_t* scales, int64_t N, int64_t K, uint8_t* Wq8,
                                   float* s_w, void* stream);
wq_status wq_quantize_w4a4_activations(const uint16_t* X, int64_t M, int64_t K, uint8_t* Xq8, float* s_x,
                                       void* stream);
wq_status wq_gemm_w4a4_mxfp4(const uint16_t* X, int64_t M, int64_t K, int64_t N, const uint8_t* Wq8, const float* s_w,
                             uint16_t* Y, void* workspace, size_t ws_bytes, void* stream);

/* WQ_OK when the current device is a GB300-class part (compute capability 10.3). */
wq_status wq_check_device(void);

#ifdef __cplusplus
}
#endif

#endif /* WQ_H_ */
