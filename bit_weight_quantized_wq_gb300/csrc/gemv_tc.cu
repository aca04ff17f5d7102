// Decode kernel on the 5th-generation tensor cores (M <= 16): Y[M, N] = X[M, K] * dequant(Wq)^T.
//
// Bandwidth-bound (推理优化与量化算子深度技术调研 §1.3: the batch-1 W4A16 GEMV is limited by HBM
// bandwidth; 第 1 章：推理加速全景 §1.2-1.3: decode arithmetic intensity ~1 FLOP/B).  The goal
// is to stream the 0.53125 B/weight of packed weights + metadata once at full HBM bandwidth
// with as few instructions per weight as possible on the CUDA cores.
//
// Per CTA (one persistent CTA per SM), a stage is one 128-row band x one pair of 128-k
// groups.  Swap-AB with the weights as the MMA's M dimension:
//   D[n, m] = sum_k A[n, k] * X[m, k],   M_mma = 128 weight rows, N_mma = 16 activations.
//   A  -- dequant threads (one per weight row and group) unpack the stage's nibbles and write
//         them straight into tensor memory (tcgen05.st): no shared-memory round trip and no
//         register fragments.
//   B  -- the stage's raw activations arrive by TMA with its weights; prep warps rewrite them
//         into the 128-byte swizzled K-major layout the MMA reads (k order matching the
//         unpacked A, see below), shared memory to shared memory.
//   D  -- one fp32 accumulator per group in tensor memory; after the group's 8 MMAs the
//         fold thread of the row folds it into registers with the group's scale.
// Warps: 0 TMA (weights + metadata tiles), 1 TMEM allocator + MMA issuer, 2-5 prep,
// 6-13 unpack (warp w may touch TMEM lanes 32 (w % 4) .. +31; warps 6-9 take the stage's
// first group, 10-13 its second), 14-17 fold + output (one thread per row, both groups).
// Tensor memory holds 3 A buffers and 4 D buffers (512 columns), so the MMAs of a stage
// overlap the unpacking of the next three and the fold never stalls the unpack.
//
// Exactness, INT4: A holds 128 + q (bf16, exact; one lop3 for two weights), so per group
//     sum_k (q - z) s x = s * D  -  s (128 + z) * sum_k x,
// i.e. the zero-point cross term of 第 6 课：量化源码走读 §3 is compensated with the group sum
// of the activations.  The unpacked nibble pairs come out as (k, k+4); the prep warps store
// X in that same k order, so the contraction is unchanged.
// Exactness, MXFP4: A holds E2M1 * 2^(e_b - e_max) in fp16 (exact unless a block sits more
// than 24 binades below the largest block of its group, where it underflows; its share of
// the group is then below 2^-21 of the group's scale), e_max folded after the MMA.  X is
// converted to fp16 with a per-row power-of-two scale that keeps it in range.
// No operand is rounded to 16 bits otherwise; accumulation is fp32.
//
// Work split and the split-K reduction are as in the CUDA-core decode kernel: (128-row band,
// group pair) units split evenly over the CTAs in band-major order; a band shared by several
// CTAs is reduced through the workspace, deterministically, by the last CTA to finish it.
#include "internal.h"

namespace wq {

__device__ uint32_t g_gemv_tc_err;

uint32_t gemv_tc_read_and_clear_error() {
  uint32_t v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, g_gemv_tc_err, sizeof(v));
  cudaMemcpyToSymbol(g_gemv_tc_err, &z, sizeof(z));
  return v;
}

namespace dec {

constexpr int kBand = 128;                 // weight rows per band (MMA M)
constexpr int kN = 16;                     // MMA N: activations, padded
constexpr int kWStages = 4;                // weight ring (weights + metadata + raw activations)
constexpr int kXStages = 4;                // activation ring
constexpr int kWBytes = kBand * 128;       // 16 KB: 128 rows x 256 k of 4-bit codes, SW128
constexpr int kXBytes = kN * 256 * 2;      // 8 KB: 16 rows x 256 k, 16-bit, SW128 (4 k-blocks)
constexpr int kMetaBytes = kBand * 16 * 2; // raw metadata tiles: 16 B per row per tensor
constexpr int kXRawBytes = kN * 256 * 2;   // raw activation tile: 16 rows x 256 k bf16 (TMA, rows >= M zero)
constexpr int kPrepWarps = 4;
// Each prep warp owns whole slots of both rings, so it waits on every phase of their barriers
// in order (a parity wait two phases ahead would pass at once).
static_assert(kWStages % kPrepWarps == 0 && kXStages % kPrepWarps == 0, "prep warps must own whole slots");
constexpr int kFirstPrep = 2;
constexpr int kFirstDeq = kFirstPrep + kPrepWarps;  // 6
constexpr int kDeqWarps = 8;
constexpr int kFirstFold = kFirstDeq + kDeqWarps;   // 14
constexpr int kFoldWarps = 4;
constexpr int kThreads = 32 * (kFirstFold + kFoldWarps);  // 576
constexpr int kTmemCols = 512;
constexpr int kABufs = 3;     // A: buffer b at 128 b, group h at + 64 h (64 cols = 128 k of 16-bit)
constexpr int kDBufs = 4;     // D: buffer b at 384 + 32 b, group h at + 16 h
constexpr int kACol = 0;
constexpr int kDCol = kABufs * 128;

struct Params {
  const uint16_t* X;
  const void* scales;
  const uint16_t* zeros;
  uint16_t* Y;
  float* part;        // [P][2][MT][kBand] fp32 partials
  uint32_t* cnt;      // [bands] counters
  int M, K, N;
  int G, GP, KB;
  int bands;
  long long U;
  int P;
  int meta_tma;
};

struct Smem {
  uint8_t w[kWStages][kWBytes];          // 1024-aligned
  uint8_t x[kXStages][kXBytes];          // 1024-aligned
  uint8_t mraw[kWStages][kMetaBytes];
  uint8_t xraw[kWStages][kXRawBytes];
  float xs[8][2][kN];                    // INT4: group sums of X; MXFP4: row factor 2^k (h = 0)
  uint64_t w_full[kWStages], w_empty[kWStages];
  uint64_t x_full[kXStages], x_empty[kXStages];
  uint64_t a_full[kABufs], d_full[kDBufs], d_empty[kDBufs];
  uint64_t group_bar;
  uint32_t tmem_base;
  int reduce_flag;
};

__device__ __forceinline__ long long unit_start(long long U, int P, int c) { return (U * c) / P; }

struct Cursor {
  long long u, u0, u1, seg_start, seg_end;
  int band, j, GP, G;
  __device__ void set_seg() {
    const long long bs = static_cast<long long>(band) * GP;
    seg_start = bs > u0 ? bs : u0;
    seg_end = bs + GP < u1 ? bs + GP : u1;
  }
  __device__ void init(long long a, long long b, int gp, int g) {
    u = a; u0 = a; u1 = b; GP = gp; G = g;
    band = static_cast<int>(a / gp);
    j = static_cast<int>(a - static_cast<long long>(band) * gp);
    set_seg();
  }
  __device__ int ng() const { return (2 * j + 1 < G) ? 2 : 1; }
  __device__ bool seg_last() const { return u + 1 == seg_end; }
  __device__ void next() {
    ++u;
    if (++j == GP) { j = 0; ++band; set_seg(); }
  }
};

// ------------------------------------------------------------------------ tcgen05 / misc
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void tc_mma_ts(uint32_t d, uint32_t a, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a), "l"(bdesc), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row atoms 1024 B apart.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3ffffu) >> 4);
  d |= static_cast<uint64_t>(16 >> 4) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}
// kind::f16, fp32 accumulate, A/B K-major, M = 128, N = 16; ab_fmt 0 = f16, 1 = bf16.
__host__ __device__ constexpr uint32_t idesc(uint32_t ab_fmt) {
  return (1u << 4) | (ab_fmt << 7) | (ab_fmt << 10) | ((uint32_t(kN) >> 3) << 17) | ((uint32_t(kBand) >> 4) << 24);
}

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t d;
  const unsigned short h = static_cast<unsigned short>(byte);
  asm("{\n\t.reg .b8 t, u;\n\tmov.b16 {t, u}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(d) : "h"(h));
  return d;
}
__device__ __forceinline__ uint32_t hmul2_u(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Byte offset of 16-byte chunk q (0..31, 8 k each) of activation row m in a stage's X tile:
// k-block q / 8 (64 k, 2 KB: rows 0-7 then 8-15, 128 B per row), swizzled chunk (q % 8) ^ (m % 8).
__device__ __forceinline__ int x_chunk_off(int m, int q) {
  return (q >> 3) * 2048 + (m >> 3) * 1024 + (m & 7) * 128 + (((q & 7) ^ (m & 7)) << 4);
}

template <int FMT, int MT>
__global__ void __launch_bounds__(kThreads, 1)
    k_gemv_tc(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_s,
              const __grid_constant__ CUtensorMap tmap_z, const __grid_constant__ CUtensorMap tmap_x,
              const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw + smem_align_pad(smem_raw));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int cta = blockIdx.x;
  const long long u0 = unit_start(p.U, p.P, cta);
  const long long u1 = unit_start(p.U, p.P, cta + 1);
  const int nstages = static_cast<int>(u1 - u0);
  constexpr int kMetaTx = (FMT == kInt4G128) ? 2 * kBand * 16 : kBand * 16;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kWStages; ++s) {
      mbar_init(&sm.w_full[s], 1);
      mbar_init(&sm.w_empty[s], 32 * (kFoldWarps + 1));  // fold warps + the stage's prep warp
    }
    for (int s = 0; s < kXStages; ++s) {
      mbar_init(&sm.x_full[s], 32);
      mbar_init(&sm.x_empty[s], 1);
    }
    for (int b = 0; b < kABufs; ++b) mbar_init(&sm.a_full[b], 32 * kDeqWarps);
    for (int b = 0; b < kDBufs; ++b) {
      mbar_init(&sm.d_full[b], 1);
      mbar_init(&sm.d_empty[b], 32 * kFoldWarps);
    }
    mbar_init(&sm.group_bar, 32 * kFoldWarps);
    fence_barrier_init();
  }
  // Activation tiles: rows >= M stay zero for the whole kernel (the prep warps write rows < M).
  for (int i = threadIdx.x; i < kXStages * kXBytes / 16; i += kThreads)
    reinterpret_cast<uint4*>(&sm.x[0][0])[i] = make_uint4(0u, 0u, 0u, 0u);
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&sm.tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (warp == 0) {
    // -------------------------------------------------------------- TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmap_w);
      tma_prefetch_desc(&tmap_x);
      if (p.meta_tma) {
        tma_prefetch_desc(&tmap_s);
        if (FMT == kInt4G128) tma_prefetch_desc(&tmap_z);
      }
      const uint64_t pol_w = l2_policy_evict_first();
      const uint64_t pol_m = l2_policy_evict_last();
      Cursor st;
      st.init(u0, u1, p.GP, p.G);
      int i = 0;
      for (; i < nstages; ++i, st.next()) {
        const int s = i % kWStages;
        if (!mbar_wait(&sm.w_empty[s], ((i / kWStages) & 1) ^ 1, &g_gemv_tc_err, kErrWaitEmpty)) break;
        mbar_arrive_expect_tx(&sm.w_full[s], kWBytes + kXRawBytes + (p.meta_tma ? kMetaTx : 0));
        tma_load_2d(&sm.w[s][0], &tmap_w, st.j * 128, st.band * kBand, &sm.w_full[s], pol_w);
        tma_load_2d(&sm.xraw[s][0], &tmap_x, st.j * 256, 0, &sm.w_full[s], pol_m);
        if (p.meta_tma) {
          if constexpr (FMT == kInt4G128) {
            const int gx = (2 * st.j) & ~7;
            tma_load_2d(&sm.mraw[s][0], &tmap_s, gx, st.band * kBand, &sm.w_full[s], pol_m);
            tma_load_2d(&sm.mraw[s][kBand * 16], &tmap_z, gx, st.band * kBand, &sm.w_full[s], pol_m);
          } else {
            tma_load_2d(&sm.mraw[s][0], &tmap_s, (8 * st.j) & ~15, st.band * kBand, &sm.w_full[s], pol_m);
          }
        }
      }
      for (int jj = i - kWStages; jj < i; ++jj) {  // drain: the last fill of every slot landed
        if (jj < 0) continue;
        mbar_wait(&sm.w_full[jj % kWStages], (jj / kWStages) & 1, &g_gemv_tc_err, kErrDrain);
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t id = idesc(FMT == kInt4G128 ? 1u : 0u);
      Cursor st;
      st.init(u0, u1, p.GP, p.G);
      int issued = 0;
      for (int i = 0; i < nstages; ++i, st.next()) {
        const int ab = i % kABufs, db = i % kDBufs, sx = i % kXStages;
        if (!mbar_wait(&sm.a_full[ab], (i / kABufs) & 1, &g_gemv_tc_err, kErrWaitFull)) break;
        if (!mbar_wait(&sm.x_full[sx], (i / kXStages) & 1, &g_gemv_tc_err, kErrWaitFull)) break;
        if (i >= kDBufs && !mbar_wait(&sm.d_empty[db], ((i - kDBufs) / kDBufs) & 1, &g_gemv_tc_err, kErrWaitEmpty))
          break;
        tc_fence_after();
        const uint32_t xbase = smem_u32(&sm.x[sx][0]);
        for (int h = 0; h < st.ng(); ++h) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const int kb = 2 * h + (kk >> 2);                       // 64-k block of the stage
            const uint64_t bd = smem_desc_sw128(xbase + kb * 2048 + (kk & 3) * 32);
            tc_mma_ts(tmem + kDCol + 32 * db + 16 * h, tmem + kACol + 128 * ab + 64 * h + 8 * kk, bd, id,
                      kk > 0 ? 1u : 0u);
          }
        }
        tc_commit(&sm.d_full[db]);
        tc_commit(&sm.x_empty[sx]);
        issued = i + 1;
      }
      // Every issued MMA must finish before the tensor memory is released below.
      if (issued > 0) {
        const int last = issued - 1;
        mbar_wait(&sm.d_full[last % kDBufs], (last / kDBufs) & 1, &g_gemv_tc_err, kErrWaitAccum);
      }
    }
  } else if (warp < kFirstDeq) {
    // -------------------------------------------------------------- prep: activations
    const int pw = warp - kFirstPrep;
    Cursor st;
    st.init(u0, u1, p.GP, p.G);
    for (int q = 0; q < pw; ++q) st.next();
    for (int i = pw; i < nstages; i += kPrepWarps) {
      const int sx = i % kXStages;
      const int s = i % kWStages;
      // lane = 16-byte chunk q of the stage (8 k); group h = q / 16; rows m < M.  The raw tile
      // came with the stage's weights (TMA; rows >= M and k >= K are zero-filled).
      const int q = lane;
      const int h = q >> 4;
      if (!mbar_wait(&sm.w_full[s], (i / kWStages) & 1, &g_gemv_tc_err, kErrWaitFull)) break;
      uint4 r[MT];
#pragma unroll
      for (int m = 0; m < MT; ++m)
        r[m] = (m < p.M) ? *reinterpret_cast<const uint4*>(&sm.xraw[s][m * 512 + 16 * q]) : make_uint4(0u, 0u, 0u, 0u);
      mbar_arrive(&sm.w_empty[s]);  // the raw activations are in registers now
      if (!mbar_wait(&sm.x_empty[sx], ((i / kXStages) & 1) ^ 1, &g_gemv_tc_err, kErrWaitEmpty)) break;
      uint8_t* xt = &sm.x[sx][0];
      if constexpr (FMT == kInt4G128) {
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          if (m >= p.M) break;
          const uint4 x = r[m];
          uint4 o;  // k order (0,4) (1,5) (2,6) (3,7): the order of the unpacked nibble pairs
          o.x = prmt(x.x, x.z, 0x5410);
          o.y = prmt(x.x, x.z, 0x7632);
          o.z = prmt(x.y, x.w, 0x5410);
          o.w = prmt(x.y, x.w, 0x7632);
          *reinterpret_cast<uint4*>(xt + x_chunk_off(m, q)) = o;
          const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
          float sum = 0.f;
#pragma unroll
          for (int e = 0; e < 4; ++e) sum += __uint_as_float(w4[e] << 16) + __uint_as_float(w4[e] & 0xffff0000u);
#pragma unroll
          for (int o2 = 8; o2 > 0; o2 >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o2);
          if ((lane & 15) == 0) sm.xs[i & 7][h][m] = sum;
        }
      } else {
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          if (m >= p.M) break;
          const uint4 x = r[m];
          const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
          uint32_t mx = 0u;  // bf16 magnitudes order like integers
#pragma unroll
          for (int e = 0; e < 4; ++e) mx = max(mx, max(w4[e] & 0x7fffu, (w4[e] >> 16) & 0x7fffu));
#pragma unroll
          for (int o2 = 16; o2 > 0; o2 >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
          const int ex = static_cast<int>(mx >> 7) - 127;
          const int k = (mx >= 0x7f80u) ? 0 : max(0, ex - 14);   // |x| 2^-k < 2^15
          const float inv = __uint_as_float(static_cast<uint32_t>(127 - k) << 23);
          uint32_t o[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            __half2 hh = __floats2half2_rn(__uint_as_float(w4[e] << 16) * inv, __uint_as_float(w4[e] & 0xffff0000u) * inv);
            o[e] = *reinterpret_cast<uint32_t*>(&hh);
          }
          *reinterpret_cast<uint4*>(xt + x_chunk_off(m, q)) = make_uint4(o[0], o[1], o[2], o[3]);
          if (lane == 0) sm.xs[i & 7][0][m] = __uint_as_float(static_cast<uint32_t>(127 + k) << 23);
        }
      }
      fence_proxy_async_smem();  // generic writes -> visible to the tensor core
      mbar_arrive(&sm.x_full[sx]);
      for (int q2 = 0; q2 < kPrepWarps; ++q2) st.next();
    }
  } else if (warp < kFirstFold) {
    // -------------------------------------------------------------- unpack into tensor memory
    const int dw = warp - kFirstDeq;              // 0..7
    const int h = dw >> 2;                        // group of the stage this thread unpacks
    const int quarter = warp & 3;                 // TMEM lane quarter
    const int r = quarter * 32 + lane;            // weight row inside the band == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    Cursor st;
    st.init(u0, u1, p.GP, p.G);
    for (int i = 0; i < nstages; ++i, st.next()) {
      const int s = i % kWStages;
      const int ab = i % kABufs;
      if (!mbar_wait(&sm.w_full[s], (i / kWStages) & 1, &g_gemv_tc_err, kErrWaitFull)) break;
      const uint8_t* wrow = &sm.w[s][r * 128];
      uint4 wv[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) wv[c] = *reinterpret_cast<const uint4*>(wrow + (((4 * h + c) ^ (r & 7)) << 4));
      uint32_t a[2][32];
      if constexpr (FMT == kInt4G128) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t wd[4] = {wv[c].x, wv[c].y, wv[c].z, wv[c].w};
#pragma unroll
          for (int jw = 0; jw < 4; ++jw) {
            const int col = 16 * c + 4 * jw;  // 4 columns = 8 k per word, order (0,4)(1,5)(2,6)(3,7)
#pragma unroll
            for (int s2 = 0; s2 < 4; ++s2)
              a[col >> 5][(col & 31) + s2] = lop3_and_or(wd[jw] >> (4 * s2), 0x000f000fu, 0x43004300u);
          }
        }
      } else {
        // per-block offsets from the group's largest E8M0 scale, folded into the fp16 operand
        const int row = st.band * kBand + r;
        uint32_t e4 = 0u;
        if ((h < st.ng()) && (row < p.N)) {
          if (p.meta_tma) {
            e4 = reinterpret_cast<const uint32_t*>(&sm.mraw[s][0])[r * 4 + (((8 * st.j) & 15) >> 2) + h];
          } else {
            const uint8_t* E = reinterpret_cast<const uint8_t*>(p.scales) + static_cast<long long>(row) * p.KB;
            const int b0 = (2 * st.j + h) * 4;
#pragma unroll
            for (int q2 = 0; q2 < 4; ++q2)
              if (b0 + q2 < p.KB) e4 |= static_cast<uint32_t>(__ldg(E + b0 + q2)) << (8 * q2);
          }
        }
        int eb[4], emax = 0;
#pragma unroll
        for (int q2 = 0; q2 < 4; ++q2) {
          eb[q2] = static_cast<int>((e4 >> (8 * q2)) & 0xffu);
          emax = max(emax, eb[q2]);
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {           // chunk c == 32-block c of the group
          const int d = emax - eb[c];
          // 2^-d as fp16 (exact down to 2^-24; below that the block's weights vanish)
          const uint32_t f = d <= 14 ? (static_cast<uint32_t>(15 - d) << 10) : (d <= 24 ? (1u << (24 - d)) : 0u);
          const uint32_t f2 = f | (f << 16);
          const uint32_t wd[4] = {wv[c].x, wv[c].y, wv[c].z, wv[c].w};
#pragma unroll
          for (int jw = 0; jw < 4; ++jw) {
            const int col = 16 * c + 4 * jw;
#pragma unroll
            for (int bb = 0; bb < 4; ++bb) {
              uint32_t v = e2m1x2_to_f16x2((wd[jw] >> (8 * bb)) & 0xffu);
              if (d != 0) v = hmul2_u(v, f2);
              a[col >> 5][(col & 31) + bb] = v;
            }
          }
        }
      }
      // A buffer ab was last read by the MMAs of stage i - kABufs.
      if (i >= kABufs) {
        const int ip = i - kABufs;
        if (!mbar_wait(&sm.d_full[ip % kDBufs], (ip / kDBufs) & 1, &g_gemv_tc_err, kErrWaitAccum)) break;
        tc_fence_after();
      }
      tmem_st32(tmem + lane_base + kACol + 128 * ab + 64 * h, a[0]);
      tmem_st32(tmem + lane_base + kACol + 128 * ab + 64 * h + 32, a[1]);
      tc_wait_st();
      tc_fence_before();
      mbar_arrive(&sm.a_full[ab]);
    }
  } else {
    // -------------------------------------------------------------- fold + output
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;            // weight row inside the band == TMEM lane
    const int tid = threadIdx.x - 32 * kFirstFold;  // 0..127
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    float acc[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[m] = 0.f;
    uint32_t gphase = 0;
    Cursor st;
    st.init(u0, u1, p.GP, p.G);
    for (int i = 0; i < nstages; ++i, st.next()) {
      const int s = i % kWStages, db = i % kDBufs;
      if (!mbar_wait(&sm.d_full[db], (i / kDBufs) & 1, &g_gemv_tc_err, kErrWaitAccum)) break;
      tc_fence_after();
      uint32_t dv[2][16];
      tmem_ld16(tmem + lane_base + kDCol + 32 * db, dv[0]);
      tmem_ld16(tmem + lane_base + kDCol + 32 * db + 16, dv[1]);
      tc_wait_ld();
      tc_fence_before();
      mbar_arrive(&sm.d_empty[db]);
      // metadata of the stage (the weight slot is still held: this thread releases it below)
      if (!mbar_wait(&sm.w_full[s], (i / kWStages) & 1, &g_gemv_tc_err, kErrWaitFull)) break;
      const int row = st.band * kBand + r;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const bool live = (h < st.ng()) && (row < p.N);
        if (!live) continue;
        if constexpr (FMT == kInt4G128) {
          uint32_t sb, zb;
          if (p.meta_tma) {
            const int col = ((2 * st.j) & 7) + h;
            sb = reinterpret_cast<const uint16_t*>(&sm.mraw[s][0])[r * 8 + col];
            zb = reinterpret_cast<const uint16_t*>(&sm.mraw[s][kBand * 16])[r * 8 + col];
          } else {
            const long long idx = static_cast<long long>(row) * p.G + 2 * st.j + h;
            sb = __ldg(reinterpret_cast<const unsigned short*>(p.scales) + idx);
            zb = __ldg(p.zeros + idx);
          }
          const float sf = __half2float(__ushort_as_half(static_cast<unsigned short>(sb)));
          const float cf = -sf * (128.f + __half2float(__ushort_as_half(static_cast<unsigned short>(zb))));
#pragma unroll
          for (int m = 0; m < MT; ++m)
            acc[m] = fmaf(cf, sm.xs[i & 7][h][m], fmaf(sf, __uint_as_float(dv[h][m]), acc[m]));
        } else {
          uint32_t e4 = 0u;
          if (p.meta_tma) {
            e4 = reinterpret_cast<const uint32_t*>(&sm.mraw[s][0])[r * 4 + (((8 * st.j) & 15) >> 2) + h];
          } else {
            const uint8_t* E = reinterpret_cast<const uint8_t*>(p.scales) + static_cast<long long>(row) * p.KB;
            const int b0 = (2 * st.j + h) * 4;
#pragma unroll
            for (int q2 = 0; q2 < 4; ++q2)
              if (b0 + q2 < p.KB) e4 |= static_cast<uint32_t>(__ldg(E + b0 + q2)) << (8 * q2);
          }
          uint32_t emax = 0u;
#pragma unroll
          for (int q2 = 0; q2 < 4; ++q2) emax = max(emax, (e4 >> (8 * q2)) & 0xffu);
          const float F = emax ? __uint_as_float(emax << 23) : __uint_as_float(0x00400000u);
#pragma unroll
          for (int m = 0; m < MT; ++m) acc[m] = fmaf(F * sm.xs[i & 7][0][m], __uint_as_float(dv[h][m]), acc[m]);
        }
      }
      mbar_arrive(&sm.w_empty[s]);
      // ---- output at the end of a band segment
      if (st.seg_last()) {
        const int band = st.band;
        const bool full = (st.seg_start == static_cast<long long>(band) * p.GP) &&
                          (st.seg_end == static_cast<long long>(band + 1) * p.GP);
        const int n = band * kBand + r;
        if (full) {
          if (n < p.N)
            for (int m = 0; m < p.M; ++m)
              p.Y[static_cast<long long>(m) * p.N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[m]));
        } else {
          const int side = (u0 >= static_cast<long long>(band) * p.GP) ? 0 : 1;
          float* slotp = p.part + (static_cast<long long>(cta) * 2 + side) * MT * kBand;
#pragma unroll
          for (int m = 0; m < MT; ++m) __stcg(slotp + m * kBand + r, acc[m]);
          __threadfence();
          mbar_arrive(&sm.group_bar);
          if (!mbar_wait(&sm.group_bar, gphase, &g_gemv_tc_err, kErrWaitReduce)) break;
          gphase ^= 1u;
          if (tid == 0) {
            const uint32_t mine = static_cast<uint32_t>(st.seg_end - st.seg_start);
            const uint32_t old = atomicAdd(p.cnt + band, mine);
            sm.reduce_flag = (old + mine == static_cast<uint32_t>(p.GP)) ? 1 : 0;
          }
          mbar_arrive(&sm.group_bar);
          if (!mbar_wait(&sm.group_bar, gphase, &g_gemv_tc_err, kErrWaitReduce)) break;
          gphase ^= 1u;
          if (sm.reduce_flag) {
            __threadfence();
            const long long bs = static_cast<long long>(band) * p.GP, be = bs + p.GP;
            int c_lo = static_cast<int>((bs * p.P) / p.U);
            while (c_lo > 0 && unit_start(p.U, p.P, c_lo) > bs) --c_lo;
            while (unit_start(p.U, p.P, c_lo + 1) <= bs) ++c_lo;
            int c_hi = static_cast<int>(((be - 1) * p.P) / p.U);
            while (c_hi > c_lo && unit_start(p.U, p.P, c_hi) > be - 1) --c_hi;
            while (c_hi + 1 < p.P && unit_start(p.U, p.P, c_hi + 1) <= be - 1) ++c_hi;
            const int lo_side = unit_start(p.U, p.P, c_lo) < bs ? 1 : 0;
            for (int m = 0; m < p.M; ++m) {
              float sum = ld_cg_f32(p.part + (static_cast<long long>(c_lo) * 2 + lo_side) * MT * kBand + m * kBand + r);
              for (int c = c_lo + 1; c <= c_hi; ++c)
                sum += ld_cg_f32(p.part + static_cast<long long>(c) * 2 * MT * kBand + m * kBand + r);
              if (n < p.N) p.Y[static_cast<long long>(m) * p.N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(sum));
            }
            if (tid == 0) atomicExch(p.cnt + band, 0u);
          }
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[m] = 0.f;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

int num_ctas(long long U) {
  const long long sms = device_sm_count();
  return static_cast<int>(U < sms ? U : sms);
}

}  // namespace dec

size_t gemv_tc_workspace_bytes(int fmt, int64_t M, int64_t K, int64_t N) {
  if (M < 1 || M > 16 || N < 1 || K < 1) return 0;
  const int MT = M <= 8 ? 8 : 16;
  const long long G = (K + 127) / 128;
  const long long bands = (N + dec::kBand - 1) / dec::kBand;
  const int P = dec::num_ctas(bands * ((G + 1) / 2));
  (void)fmt;
  return kWsCounterBytes + static_cast<size_t>(P) * 2 * MT * dec::kBand * sizeof(float);
}

template <int FMT, int MT>
static cudaError_t launch_t(const CUtensorMap& tw, const CUtensorMap& ts, const CUtensorMap& tz, const CUtensorMap& tx,
                            const dec::Params& p, cudaStream_t stream) {
  const size_t smem = sizeof(dec::Smem) + 1024;
  auto kern = dec::k_gemv_tc<FMT, MT>;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  kern<<<p.P, dec::kThreads, smem, stream>>>(tw, ts, tz, tx, p);
  return cudaGetLastError();
}

cudaError_t launch_gemv_tc(int fmt, const uint16_t* X, int64_t M, int64_t K, int64_t N, const int32_t* Wq,
                           const void* scales, const uint16_t* zeros, uint16_t* Y, void* ws, size_t ws_bytes,
                           cudaStream_t stream) {
  dec::Params p{};
  p.X = X;
  p.scales = scales;
  p.zeros = zeros;
  p.Y = Y;
  p.M = static_cast<int>(M);
  p.K = static_cast<int>(K);
  p.N = static_cast<int>(N);
  p.G = static_cast<int>((K + 127) / 128);
  p.GP = (p.G + 1) / 2;
  p.KB = static_cast<int>(K / 32);
  p.bands = static_cast<int>((N + dec::kBand - 1) / dec::kBand);
  p.U = static_cast<long long>(p.bands) * p.GP;
  p.P = dec::num_ctas(p.U);
  if (p.bands > kWsMaxCounters) return cudaErrorInvalidValue;
  if (ws_bytes < gemv_tc_workspace_bytes(fmt, M, K, N)) return cudaErrorInvalidValue;
  p.cnt = reinterpret_cast<uint32_t*>(ws);
  p.part = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ws) + kWsCounterBytes);

  CUtensorMap tw, ts, tz, tx;
  cudaError_t e = make_tmap_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, Wq, static_cast<uint64_t>(K / 2),
                               static_cast<uint64_t>(N), static_cast<uint64_t>(K / 2), 128, dec::kBand,
                               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
  if (e != cudaSuccess) return e;
  // activations: 16 rows x 256 k per stage; rows >= M and columns >= K come back as zeros
  e = make_tmap_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, X, static_cast<uint64_t>(K), static_cast<uint64_t>(M),
                   static_cast<uint64_t>(K) * 2, 256, dec::kN, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
  if (e != cudaSuccess) return e;
  ts = tw;
  tz = tw;
  if (fmt == kInt4G128) {
    p.meta_tma = (p.G % 8 == 0) ? 1 : 0;
    if (p.meta_tma) {
      e = make_tmap_2d(&ts, CU_TENSOR_MAP_DATA_TYPE_UINT16, scales, static_cast<uint64_t>(p.G),
                       static_cast<uint64_t>(N), static_cast<uint64_t>(p.G) * 2, 8, dec::kBand,
                       CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE);
      if (e != cudaSuccess) return e;
      e = make_tmap_2d(&tz, CU_TENSOR_MAP_DATA_TYPE_UINT16, zeros, static_cast<uint64_t>(p.G),
                       static_cast<uint64_t>(N), static_cast<uint64_t>(p.G) * 2, 8, dec::kBand,
                       CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE);
      if (e != cudaSuccess) return e;
    }
  } else {
    p.meta_tma = (p.KB % 16 == 0) ? 1 : 0;
    if (p.meta_tma) {
      e = make_tmap_2d(&ts, CU_TENSOR_MAP_DATA_TYPE_UINT8, scales, static_cast<uint64_t>(p.KB),
                       static_cast<uint64_t>(N), static_cast<uint64_t>(p.KB), 16, dec::kBand,
                       CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE);
      if (e != cudaSuccess) return e;
    }
  }
  const bool small = M <= 8;
  if (fmt == kInt4G128)
    return small ? launch_t<kInt4G128, 8>(tw, ts, tz, tx, p, stream) : launch_t<kInt4G128, 16>(tw, ts, tz, tx, p, stream);
  return small ? launch_t<kMxfp4, 8>(tw, ts, tz, tx, p, stream) : launch_t<kMxfp4, 16>(tw, ts, tz, tx, p, stream);
}

}  // namespace wq
