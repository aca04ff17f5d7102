// Prefill kernel: Y[M, N] = X[M, K] * dequant(Wq)^T on the 5th-generation tensor cores.
//
// Compute-bound (第 1 章：推理加速全景 §1.3: prefill GEMMs run at 55-100 FLOP/B), so this is a
// dense contraction on tcgen05 with the dequantization fused in front of the tensor core
// (推理优化与量化算子深度技术调研 §1.2: "x_deq = (q - zp) * scale", done before the MMA).
//
// Swap-AB formulation, one 128 (weights) x 256 (activations) tile per CTA:
//   D[n, m] = sum_k What[n, k] * X[m, k]            (D = Y^T, fp32 in tensor memory)
//   A = What tile [128 x 64] -- dequantized by 128 threads (one per weight row = one TMEM
//       lane) and written straight into tensor memory with tcgen05.st: no shared-memory
//       round trip for the dequantized operand.
//   B = X tile [256 x 64]    -- TMA, 128-byte swizzle, K-major, read by the MMA from smem.
//   MMA = tcgen05.mma.cta_group::1.kind::f16, M=128, N=256, K=16, issued by one thread.
// Warp roles: warp 0 TMA producer, warp 1 TMEM allocator + MMA issuer, warps 2-13 dequant in
// three sets of four (one warp per TMEM lane quarter) that take stages in turn, so one set's
// tensor-memory stores overlap the others' unpacking; then the epilogue, each set a third of
// the tile's columns in interleaved 32-column chunks (tcgen05.ld -> scale -> bf16 -> global).
//
// Operand types.  MXFP4: w_hat = E2M1 * 2^e is exact in bf16, so the MMA runs in bf16 on X
// as given.  INT4: (q - z) * s needs up to 15 significant bits; rounding it to bf16 (8 bits)
// would put the layer outside 1e-2 (1 + |y|) of the float64 result at K = 4096..29568, so
// the MMA runs in fp16 (11 bits): a pre-pass converts X exactly to fp16, each row scaled by a
// power of two 2^-k_m that puts its largest |x| in [2^14, 2^15) (down for large rows, up for
// small ones), and the epilogue multiplies row m of Y by 2^k_m.
#include "internal.h"
#include "tcgen05.cuh"

namespace wq {

__device__ uint32_t g_gemm_err;

uint32_t gemm_tc_read_and_clear_error() {
  uint32_t v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, g_gemm_err, sizeof(v));
  cudaMemcpyToSymbol(g_gemm_err, &z, sizeof(z));
  return v;
}

namespace tc {

constexpr int BN = 128;          // weight rows per tile (MMA M)
constexpr int BK = 64;           // k per stage (one 128-byte swizzle row of 16-bit X)
constexpr int kWBytes = BN * BK / 2;        // 4 KB packed weights
constexpr int kDequantSets = 3;             // dequant warp sets, alternating stages
constexpr int kThreads = 64 + 128 * kDequantSets;   // producer + MMA warp + 4 dequant warps per set
constexpr int kTmemCols = 512;
constexpr int kAccCol = 0;                  // D: columns [0, BMT)
constexpr int kGroupM = 8;                  // tile raster: 8 activation tiles per group

// Activation rows per tile (MMA N) BMT: 256 for prefill, 128 or 64 when M is that small, so
// that a stage's activation tile (BMT x 64 k, TMA with SWIZZLE_128B) carries no zero rows.
// Smaller tiles leave room for more stages.
__host__ __device__ constexpr int stages_for(int bmt) { return bmt == 256 ? 6 : (bmt == 128 ? 8 : 10); }

template <int BMT>
struct Smem {
  static constexpr int kStages = stages_for(BMT);
  static constexpr int kXBytes = BMT * BK * 2;
  static constexpr int kACol = BMT;         // A stage s: columns [BMT + 32 s, +32)
  static_assert(kACol + 32 * kStages <= kTmemCols, "the A stages must fit the tensor-memory allocation");
  uint8_t x[kStages][kXBytes];    // 1024-aligned (SWIZZLE_128B atoms)
  uint8_t w[kStages][kWBytes];
  uint64_t full[kStages];
  uint64_t a_ready[kStages];
  uint64_t empty[kStages];
  uint64_t accum_full;
  uint32_t tmem_base;
  int last;              // split tile: this CTA finished last and writes the outputs
};

struct Params {
  const void* scales;
  const uint16_t* zeros;
  const float* xscale;   // INT4: 2^k_m per activation row (nullptr for MXFP4)
  uint16_t* Y;
  OutSplit split;        // EPI == kEpiSplit3: three output tensors by column range
  int M, K, N;
  int KB;                // MXFP4 scale bytes per row (K / 32)
  int G;                 // INT4 groups per row (K / 128)
  int tiles_n, tiles_m;
  int full_tiles;        // tiles [0, full_tiles) run whole; each later tile as `splits` K parts
  int splits;            // K parts per split tile (part q: stages [q KS / splits, (q + 1) KS / splits))
  int k_stages;          // ceil(K / BK)
  uint32_t* cnt;         // split tiles: one counter each (workspace header, left at zero)
  float* part;           // split tiles: [tile][part][BN][BMT] fp32 partial accumulators
};

// Instruction descriptor, kind::f16: fp32 accumulate, A/B K-major, A/B both fp16 or both bf16,
// MMA N = n (the activation rows of a tile, BMT), M = BN.
__host__ __device__ constexpr uint32_t idesc_f16(uint32_t ab_fmt /*0 f16, 1 bf16*/, uint32_t n) {
  return (1u << 4) | (ab_fmt << 7) | (ab_fmt << 10) | ((n >> 3) << 17) | ((uint32_t(BN) >> 4) << 24);
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t hsub2_u(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t hmul2_u(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t d;
  const unsigned short h = static_cast<unsigned short>(byte);
  asm("{\n\t.reg .b8 t, u;\n\tmov.b16 {t, u}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(d) : "h"(h));
  return d;
}
__device__ __forceinline__ float e8m0_to_f32(uint32_t byte) {
  return byte ? __uint_as_float(byte << 23) : __uint_as_float(0x00400000u);
}

// Barrier 1 among the dequant / epilogue warps (all warps but the producer and the MMA warp).
__device__ __forceinline__ void epi_bar() {
  asm volatile("barrier.sync 1, %0;" ::"n"(kThreads - 64) : "memory");
}
// The same barrier, returning whether every one of those threads passed `v`.
__device__ __forceinline__ bool epi_bar_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "barrier.red.and.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "n"(kThreads - 64)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Tile index -> (n tile, m tile), grouped so that a wave of CTAs shares activation tiles
// (kGroupM of them) and weight tiles in L2.
__device__ __forceinline__ void tile_coords(int t, int tiles_n, int tiles_m, int& tn, int& tm) {
  const int per_group = kGroupM * tiles_n;
  const int grp = t / per_group;
  const int first_m = grp * kGroupM;
  const int gsize = min(tiles_m - first_m, kGroupM);
  const int r = t % per_group;
  tm = first_m + r % gsize;
  tn = r / gsize;
}

template <int FMT, int EPI, int BMT>
__global__ void __launch_bounds__(kThreads, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_w,
              const Params p) {
  using S = Smem<BMT>;
  constexpr int kStages = S::kStages;
  constexpr int kXBytes = S::kXBytes;
  constexpr int kACol = S::kACol;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  S& sm = *reinterpret_cast<S*>(smem_raw + smem_align_pad(smem_raw));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Tiles past full_tiles run split along K on `splits` CTAs (the last, partial wave of a
  // prefill layer in two; every tile of a layer with too few tiles for the SMs in up to
  // eight), so that every SM has work.  Each part stores its fp32 accumulator; the last to
  // finish adds all parts in part order (deterministic) and writes Y.
  int t = blockIdx.x, part = -1;
  if (t >= p.full_tiles) {
    const int j = t - p.full_tiles;
    t = p.full_tiles + j / p.splits;
    part = j % p.splits;
  }
  int tn, tm;
  tile_coords(t, p.tiles_n, p.tiles_m, tn, tm);
  const int n0 = tn * BN, m0 = tm * BMT;
  const int kb = part < 0 ? 0 : (part * p.k_stages) / p.splits;                      // first stage
  const int KS = (part < 0 ? p.k_stages : ((part + 1) * p.k_stages) / p.splits) - kb;   // stages

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.a_ready[s], 128);
      mbar_init(&sm.empty[s], 1);
    }
    mbar_init(&sm.accum_full, 1);
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
  // Programmatic dependent launch: the set-up above overlaps the previous kernel's tail; every
  // read of global memory comes after the wait (the MMA warp reads none).
  pdl_launch_dependents();
  if (warp != 1) pdl_wait();

  if (warp == 0) {
    // -------------------------------------------------------------- TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmap_x);
      tma_prefetch_desc(&tmap_w);
      const uint64_t pol_x = l2_policy_evict_last();
      const uint64_t pol_w = l2_policy_evict_last();
      int i = 0;
      for (; i < KS; ++i) {
        const int s = i % kStages;
        const uint32_t ph = (i / kStages) & 1;
        if (!mbar_wait(&sm.empty[s], ph ^ 1, &g_gemm_err, kErrWaitEmpty)) break;
        mbar_arrive_expect_tx(&sm.full[s], kXBytes + kWBytes);
        tma_load_2d(&sm.x[s][0], &tmap_x, (kb + i) * BK, m0, &sm.full[s], pol_x);
        tma_load_2d(&sm.w[s][0], &tmap_w, (kb + i) * (BK / 2), n0, &sm.full[s], pol_w);
      }
      for (int j = i - kStages; j < i; ++j) {  // drain: the last fill of each slot landed
        if (j < 0) continue;
        mbar_wait(&sm.full[j % kStages], (j / kStages) & 1, &g_gemm_err, kErrDrain);
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(FMT == kInt4G128 ? 0u : 1u, static_cast<uint32_t>(BMT));
      bool ok = true;
      for (int i = 0; i < KS; ++i) {
        const int s = i % kStages;
        const uint32_t ph = (i / kStages) & 1;
        if (!mbar_wait(&sm.full[s], ph, &g_gemm_err, kErrWaitFull) ||
            !mbar_wait(&sm.a_ready[s], ph, &g_gemm_err, kErrWaitFull)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t bdesc = smem_desc_sw128(smem_u32(&sm.x[s][0]));
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          tc_mma_ts(tmem + kAccCol, tmem + kACol + 32 * s + 8 * kk, bdesc + static_cast<uint64_t>(2 * kk), idesc,
                    (i > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(&sm.empty[s]);
      }
      // Always commit: the epilogue (normal path) and the TMEM release below (any path)
      // must not run before every issued MMA has completed.
      tc_commit(&sm.accum_full);
      mbar_wait(&sm.accum_full, 0, &g_gemm_err, kErrWaitAccum);
      (void)ok;
    }
  } else {
    // -------------------------------------------------------------- dequant, then epilogue
    const int q = warp & 3;                 // TMEM lane quarter this warp may access
    const int set = (warp - 2) >> 2;        // stages set, set + kDequantSets, ... are this set's
    const int r = q * 32 + lane;            // weight row inside the tile == TMEM lane
    const int n = n0 + r;
    const bool row_ok = n < p.N;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    bool ok = true;
    for (int i = set; i < KS; i += kDequantSets) {
      const int s = i % kStages;
      const uint32_t ph = (i / kStages) & 1;
      uint32_t a[32];
      // metadata of this stage (loaded before the waits)
      uint32_t s2 = 0, zz = 0;          // INT4: f16x2 scale, f16x2 (1024 + z)
      uint32_t e2 = 0;                  // MXFP4: two E8M0 bytes
      const int k0 = (kb + i) * BK;
      if constexpr (FMT == kInt4G128) {
        const int g = k0 / 128;
        uint16_t sb = 0, zb = 0;
        if (row_ok) {
          sb = reinterpret_cast<const uint16_t*>(p.scales)[static_cast<long long>(n) * p.G + g];
          zb = p.zeros[static_cast<long long>(n) * p.G + g];
        }
        s2 = static_cast<uint32_t>(sb) | (static_cast<uint32_t>(sb) << 16);
        const __half zh = __float2half_rn(1024.f + __half2float(__ushort_as_half(zb)));
        const uint32_t zu = __half_as_ushort(zh);
        zz = zu | (zu << 16);
      } else {
        const int b = k0 / 32;
        if (row_ok) {
          const uint8_t* E = reinterpret_cast<const uint8_t*>(p.scales) + static_cast<long long>(n) * p.KB;
          const uint32_t lo = (b < p.KB) ? E[b] : 0u;
          const uint32_t hi = (b + 1 < p.KB) ? E[b + 1] : 0u;
          e2 = lo | (hi << 8);
        }
      }
      if (!mbar_wait(&sm.full[s], ph, &g_gemm_err, kErrWaitFull)) { ok = false; break; }
      const uint4* wrow = reinterpret_cast<const uint4*>(&sm.w[s][r * (BK / 2)]);
      const uint4 v0 = wrow[0], v1 = wrow[1];
      const uint32_t wv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
      if constexpr (FMT == kInt4G128) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t w = wv[j], w4 = wv[j] >> 4;
          // natural k order: (n0,n1) (n2,n3) (n4,n5) (n6,n7) as fp16 1024 + q
          const uint32_t p0 = lop3_and_or(prmt(w, w4, 0x4400), 0x000f000fu, 0x64006400u);
          const uint32_t p1 = lop3_and_or(prmt(w, w4, 0x5511), 0x000f000fu, 0x64006400u);
          const uint32_t p2 = lop3_and_or(prmt(w, w4, 0x6622), 0x000f000fu, 0x64006400u);
          const uint32_t p3 = lop3_and_or(prmt(w, w4, 0x7733), 0x000f000fu, 0x64006400u);
          a[4 * j + 0] = hmul2_u(hsub2_u(p0, zz), s2);
          a[4 * j + 1] = hmul2_u(hsub2_u(p1, zz), s2);
          a[4 * j + 2] = hmul2_u(hsub2_u(p2, zz), s2);
          a[4 * j + 3] = hmul2_u(hsub2_u(p3, zz), s2);
        }
      } else {
        const float f0 = e8m0_to_f32(e2 & 0xffu), f1 = e8m0_to_f32(e2 >> 8);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float f = j < 4 ? f0 : f1;
#pragma unroll
          for (int bb = 0; bb < 4; ++bb) {
            const uint32_t h2 = e2m1x2_to_f16x2((wv[j] >> (8 * bb)) & 0xffu);
            const float lo = __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xffffu))) * f;
            const float hi = __half2float(__ushort_as_half(static_cast<unsigned short>(h2 >> 16))) * f;
            __nv_bfloat162 bv = __floats2bfloat162_rn(lo, hi);
            a[4 * j + bb] = *reinterpret_cast<uint32_t*>(&bv);
          }
        }
      }
      // The A slot is free once the MMAs of its previous use completed.
      if (!mbar_wait(&sm.empty[s], ph ^ 1, &g_gemm_err, kErrWaitEmpty)) { ok = false; break; }
      tc_fence_after();
      tmem_st32(tmem + lane_base + kACol + 32 * s, a);
      tc_wait_st();
      tc_fence_before();
      mbar_arrive(&sm.a_ready[s]);
    }
    // ------------------------------------------------------------ epilogue
    // The dequant threads agree first that none of them timed out, so the barriers below are
    // reached by all of them or by none.
    const bool ready = ok && mbar_wait(&sm.accum_full, 0, &g_gemm_err, kErrWaitAccum);
    if (epi_bar_and(ready)) {
      tc_fence_after();
      bool write_y = true;
      const float* parts = nullptr;   // split tile, last CTA: this row's partial sums, part 0
      if (part >= 0) {
        // this part's accumulator to its slot; then one GPU-scope counter update per CTA
        // (release: after the barrier, covers every thread's stores) tells the last CTA to
        // finish the tile
        const long long slot = static_cast<long long>(t - p.full_tiles) * p.splits;
        float* mine = p.part + (slot + part) * (BN * BMT) + static_cast<long long>(r) * BMT;
#pragma unroll 1
        for (int c = 32 * set; c < BMT; c += 32 * kDequantSets) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_base + kAccCol + c, v);
          tc_wait_ld();
          float4* dst = reinterpret_cast<float4*>(mine + c);
#pragma unroll
          for (int u = 0; u < 8; ++u)
            __stcg(dst + u, make_float4(__uint_as_float(v[4 * u]), __uint_as_float(v[4 * u + 1]),
                                        __uint_as_float(v[4 * u + 2]), __uint_as_float(v[4 * u + 3])));
        }
        epi_bar();
        if (threadIdx.x == 64) {
          uint32_t* c = p.cnt + (t - p.full_tiles);
          const uint32_t old = atom_add_acq_rel_gpu(c, 1u);
          sm.last = old == static_cast<uint32_t>(p.splits - 1) ? 1 : 0;
          if (sm.last) atomicExch(c, 0u);   // ready for the next call
        }
        epi_bar();
        // The counter update's acquire (thread 64) and the barrier after it order the other
        // parts' stores before this CTA's loads of them; no further fence is needed.
        write_y = sm.last != 0;
        if (write_y) parts = p.part + slot * (BN * BMT) + static_cast<long long>(r) * BMT;
      }
#pragma unroll 1
      for (int c = 32 * set; c < BMT && write_y; c += 32 * kDequantSets) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + kAccCol + c, v);
        tc_wait_ld();
        if (parts) {
          if (p.splits == 2) {
            // two parts: this CTA's accumulator plus the other's, a two-term fp32 sum that is
            // the same whichever part finished last
            const float4* src = reinterpret_cast<const float4*>(parts + static_cast<long long>(1 - part) * (BN * BMT) + c);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const float4 o = __ldcg(src + u);
              v[4 * u + 0] = __float_as_uint(__uint_as_float(v[4 * u + 0]) + o.x);
              v[4 * u + 1] = __float_as_uint(__uint_as_float(v[4 * u + 1]) + o.y);
              v[4 * u + 2] = __float_as_uint(__uint_as_float(v[4 * u + 2]) + o.z);
              v[4 * u + 3] = __float_as_uint(__uint_as_float(v[4 * u + 3]) + o.w);
            }
          } else {
            // more parts: all of them from the workspace, added in part order (the same bits
            // whichever part finished last); each part's loads are issued before any addition
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              float4 o[8];
#pragma unroll
              for (int q = 0; q < 8; ++q)
                if (q < p.splits)
                  o[q] = __ldcg(reinterpret_cast<const float4*>(parts + static_cast<long long>(q) * (BN * BMT) + c) + u);
              float4 a = o[0];
#pragma unroll
              for (int q = 1; q < 8; ++q)
                if (q < p.splits) {
                  a.x += o[q].x;
                  a.y += o[q].y;
                  a.z += o[q].z;
                  a.w += o[q].w;
                }
              v[4 * u + 0] = __float_as_uint(a.x);
              v[4 * u + 1] = __float_as_uint(a.y);
              v[4 * u + 2] = __float_as_uint(a.z);
              v[4 * u + 3] = __float_as_uint(a.w);
            }
          }
        }
        if constexpr (EPI == kEpiSwiglu) {
          // Gate row n (lane bit 3 clear) and its up row n + 8 sit in lanes l and l ^ 8 of
          // this warp.  Per pair of accumulator columns (j, j + 1) one shuffle gives the gate
          // lane the up value of column j and the up lane the gate value of column j + 1, so
          // every lane evaluates SiLU(g) * u once per two columns.
          const bool gate = (lane & 8) == 0;
          const unsigned am = __activemask();   // the whole warp, unless a wait above timed out
          const int F = p.N >> 1;
          const long long col = swiglu_col(n & ~8);
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const int ma = m0 + c + j, mb = ma + 1;
            float y0 = __uint_as_float(v[j]), y1 = __uint_as_float(v[j + 1]);
            if constexpr (FMT == kInt4G128) {
              y0 *= __ldg(p.xscale + (ma < p.M ? ma : 0));
              y1 *= __ldg(p.xscale + (mb < p.M ? mb : 0));
            }
            const float recv = __shfl_xor_sync(am, gate ? y1 : y0, 8);
            const float g = gate ? y0 : recv, u = gate ? recv : y1;
            const int m = gate ? ma : mb;
            if (row_ok && m < p.M)
              p.Y[static_cast<long long>(m) * F + col] = __bfloat16_as_ushort(__float2bfloat16_rn(silu_f32(g) * u));
          }
        } else if (row_ok) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int m = m0 + c + j;
            if (m < p.M) {
              float y = __uint_as_float(v[j]);
              if constexpr (FMT == kInt4G128) y *= __ldg(p.xscale + m);
              const uint16_t yb = __bfloat16_as_ushort(__float2bfloat16_rn(y));
              if constexpr (EPI == kEpiSplit3) store_split3(p.split, m, n, yb);
              else p.Y[static_cast<long long>(m) * p.N + n] = yb;
            }
          }
        }
      }
    }
    tc_fence_before();
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// X (bf16) -> fp16 with a per-row power-of-two scale 2^-k (bf16_to_f16_exponent: |x| 2^-k <
// 2^15, small rows scaled up so that their values stay out of fp16's subnormal range); writes
// xs[m] = 2^k.  One CTA per row; the row is read twice (max, then convert), the second time
// from L2.
__global__ void __launch_bounds__(256) k_x_to_f16(const uint16_t* __restrict__ X, int K, uint16_t* __restrict__ Xh,
                                                  float* __restrict__ xs) {
  pdl_launch_dependents();
  pdl_wait();   // X may come from the previous kernel of the stream
  const int m = blockIdx.x;
  const uint4* row = reinterpret_cast<const uint4*>(X + static_cast<long long>(m) * K);
  uint4* out = reinterpret_cast<uint4*>(Xh + static_cast<long long>(m) * K);
  const int nv = K / 8;
  uint32_t mx = 0u;
  for (int v = threadIdx.x; v < nv; v += blockDim.x) {
    const uint4 r = __ldg(row + v);
    const uint32_t w4[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) mx = max(mx, max(w4[q] & 0x7fffu, (w4[q] >> 16) & 0x7fffu));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  __shared__ uint32_t red[8];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
  __syncthreads();
  mx = 0u;
#pragma unroll
  for (int w = 0; w < 8; ++w) mx = max(mx, red[w]);
  const int k = bf16_to_f16_exponent(mx);
  const float inv = pow2_normal(-k);
  for (int v = threadIdx.x; v < nv; v += blockDim.x) {
    const uint4 r = __ldg(row + v);
    const uint32_t w4[4] = {r.x, r.y, r.z, r.w};
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      __half2 h = __floats2half2_rn(__uint_as_float(w4[q] << 16) * inv, __uint_as_float(w4[q] & 0xffff0000u) * inv);
      o[q] = *reinterpret_cast<uint32_t*>(&h);
    }
    out[v] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (threadIdx.x == 0) xs[m] = pow2_normal(k);
}

}  // namespace tc

namespace {

// The launch plan: the activation tile (MMA N) the rows of M need, and which tiles run split
// along K on how many CTAs.  A layer with too few tiles for half the SMs (decode-sized to
// mid-sized M) splits every tile, up to 8 ways with at least 8 stages each; otherwise the
// tiles of a last, partial wave that fits in half the SMs split in two.
struct TcPlan {
  int bmt, tiles_n, tiles_m, k_stages, splits;
  long long tiles, nsplit;
};

TcPlan plan_tc(int64_t M, int64_t K, int64_t N) {
  using namespace tc;
  TcPlan pl{};
  pl.bmt = M <= 64 ? 64 : (M <= 128 ? 128 : 256);
  pl.tiles_n = static_cast<int>((N + BN - 1) / BN);
  pl.tiles_m = static_cast<int>((M + pl.bmt - 1) / pl.bmt);
  pl.k_stages = static_cast<int>((K + BK - 1) / BK);
  pl.tiles = static_cast<long long>(pl.tiles_n) * pl.tiles_m;
  const long long sms = device_sm_count();
  pl.splits = 1;
  pl.nsplit = 0;
  if (2 * pl.tiles <= sms) {
    long long s = sms / pl.tiles;
    if (s > pl.k_stages / 8) s = pl.k_stages / 8;
    if (s > 8) s = 8;
    if (s >= 2) {
      pl.splits = static_cast<int>(s);
      pl.nsplit = pl.tiles;
      return pl;
    }
  }
  const long long rem = pl.tiles % sms;
  if (rem > 0 && 2 * rem <= sms && pl.k_stages >= 2) {
    pl.splits = 2;
    pl.nsplit = rem;
  }
  return pl;
}

size_t round256(size_t b) { return (b + 255) / 256 * 256; }

template <int FMT, int BMT>
void (*pick_kernel(int epi))(CUtensorMap, CUtensorMap, tc::Params) {
  return epi == kEpiSwiglu ? tc::k_gemm_tc<FMT, kEpiSwiglu, BMT>
                           : (epi == kEpiSplit3 ? tc::k_gemm_tc<FMT, kEpiSplit3, BMT> : tc::k_gemm_tc<FMT, kEpiNone, BMT>);
}

template <int BMT>
cudaError_t launch_tc_t(int fmt, int epi, const CUtensorMap& tx, const CUtensorMap& tw, const tc::Params& p,
                        unsigned grid, cudaStream_t stream) {
  static_assert(sizeof(tc::Smem<BMT>) + 1024 <= 227 * 1024, "tensor-core kernel shared memory over the per-CTA limit");
  const size_t smem = sizeof(tc::Smem<BMT>) + 1024;
  void (*kern)(CUtensorMap, CUtensorMap, tc::Params) =
      fmt == kInt4G128 ? pick_kernel<kInt4G128, BMT>(epi) : pick_kernel<kMxfp4, BMT>(epi);
  cudaError_t e = set_smem_attr_once(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  // Programmatic stream serialization: the CTAs may start (barrier set-up, tensor-memory
  // allocation) while the previous kernel of the stream is still running; every read of
  // global memory comes after griddepcontrol.wait.
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(tc::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tx, tw, p);
}

}  // namespace

size_t gemm_tc_workspace_bytes(int fmt, int64_t M, int64_t K, int64_t N) {
  using namespace tc;
  const TcPlan pl = plan_tc(M, K, N);
  const size_t part = static_cast<size_t>(pl.nsplit) * pl.splits * BN * pl.bmt * sizeof(float);
  if (fmt != kInt4G128) return part ? kWsHeaderBytes + part : 0;
  const size_t xh = round256(static_cast<size_t>(M) * K * 2);
  return kWsHeaderBytes + xh + round256(static_cast<size_t>(M) * 4) + part;
}

cudaError_t launch_gemm_tc(int fmt, const uint16_t* X, int64_t M, int64_t K, int64_t N, const int32_t* Wq,
                           const void* scales, const uint16_t* zeros, uint16_t* Y, void* ws, size_t ws_bytes,
                           cudaStream_t stream, int epi, const OutSplit* split) {
  using namespace tc;
  if (epi == kEpiSwiglu && N % 16 != 0) return cudaErrorInvalidValue;
  if (epi == kEpiSplit3 && !split) return cudaErrorInvalidValue;
  if (ws_bytes < gemm_tc_workspace_bytes(fmt, M, K, N)) return cudaErrorInvalidValue;
  const TcPlan pl = plan_tc(M, K, N);
  Params p{};
  p.scales = scales;
  p.zeros = zeros;
  p.Y = Y;
  if (split) p.split = *split;
  p.M = static_cast<int>(M);
  p.K = static_cast<int>(K);
  p.N = static_cast<int>(N);
  p.KB = static_cast<int>(K / 32);
  p.G = static_cast<int>(K / 128);
  p.tiles_n = pl.tiles_n;
  p.tiles_m = pl.tiles_m;
  p.k_stages = pl.k_stages;
  p.full_tiles = static_cast<int>(pl.tiles - pl.nsplit);
  p.splits = pl.splits;
  p.cnt = reinterpret_cast<uint32_t*>(ws);
  p.part = nullptr;
  if (pl.nsplit) {
    size_t off = kWsHeaderBytes;
    if (fmt == kInt4G128) off += round256(static_cast<size_t>(M) * K * 2) + round256(static_cast<size_t>(M) * 4);
    p.part = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ws) + off);
  }
  const void* xsrc = X;
  if (fmt == kInt4G128) {
    uint8_t* base = reinterpret_cast<uint8_t*>(ws) + kWsHeaderBytes;  // never touch the header
    uint16_t* Xh = reinterpret_cast<uint16_t*>(base);
    float* xs = reinterpret_cast<float*>(base + ((static_cast<size_t>(M) * K * 2 + 255) / 256) * 256);
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(M));
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, k_x_to_f16, X, static_cast<int>(K), Xh, xs);
    if (e != cudaSuccess) return e;
    xsrc = Xh;
    p.xscale = xs;
  }
  CUtensorMap tx, tw;
  cudaError_t e = make_tmap_2d(&tx, fmt == kInt4G128 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                               xsrc, static_cast<uint64_t>(K), static_cast<uint64_t>(M), static_cast<uint64_t>(K) * 2,
                               BK, static_cast<uint32_t>(pl.bmt), CU_TENSOR_MAP_SWIZZLE_128B,
                               CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
  if (e != cudaSuccess) return e;
  e = make_tmap_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, Wq, static_cast<uint64_t>(K / 2), static_cast<uint64_t>(N),
                   static_cast<uint64_t>(K / 2), BK / 2, BN, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
  if (e != cudaSuccess) return e;
  const unsigned grid = static_cast<unsigned>(p.full_tiles + pl.nsplit * pl.splits);
  if (pl.bmt == 64) return launch_tc_t<64>(fmt, epi, tx, tw, p, grid, stream);
  if (pl.bmt == 128) return launch_tc_t<128>(fmt, epi, tx, tw, p, grid, stream);
  return launch_tc_t<256>(fmt, epi, tx, tw, p, grid, stream);
}

}  // namespace wq
