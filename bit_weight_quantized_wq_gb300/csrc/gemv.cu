// Decode kernel (M <= 16): Y[M, N] = X[M, K] * dequant(Wq)^T.
//
// Bandwidth-bound (推理优化与量化算子深度技术调研 §1.3: at batch 1 the W4A16 GEMV is limited by
// HBM bandwidth; 第 1 章：推理加速全景 §1.2-1.3: decode arithmetic intensity ~1 FLOP/B), so the
// design goal is to stream the 0.53125 B/weight of packed weights + metadata once, at full
// HBM bandwidth, with the arithmetic hidden underneath.
//
// Structure (one persistent CTA per SM, warp-specialised, 20 warps):
//   warp 0      TMA producer: 256-row x 128-byte tiles of the packed weights (two 128-k
//               groups of INT4 / 256 k of MXFP4), SWIZZLE_128B, into a 4- or 5-stage smem
//               ring, with the matching scale / zero-point (INT4) or E8M0 (MXFP4) tiles.
//   warps 1-3   prep (stage i by prep warp i % 3), on a separate 6-stage ring: the
//               activations of the stage's k-range (from L2; they are small and shared by
//               every CTA) in the exact order of the mma.sync B fragments, with their
//               per-group sums (INT4) or converted to fp16 with a per-row power-of-two scale
//               that keeps every value in fp16 range (MXFP4).  The activations do not depend
//               on the weights, so this runs ahead of the weight stream.
//   warps 4-19  consumers: 16 weight rows each; per-row metadata straight from its tile,
//               nibbles unpacked in registers, tensor-core mma.sync with fp32 accumulation,
//               group scale applied in fp32 afterwards.
//
// Exactness: the tensor-core operands are exact small integers (INT4: 128 + q in bf16) or
// exact E2M1 values (MXFP4, fp16); every product is exact and the per-group (INT4) or
// per-32 (MXFP4) scale is applied to the fp32 partial sum.  No operand is rounded to 16
// bits, which keeps the layer within 1e-2 (1 + |y|) of the float64 oracle at every K (a
// bf16-rounded dequantised weight would not).  INT4 per group and output:
//   sum_k (q - z) s x = s * sum_k (128 + q) x  -  s (128 + z) * sum_k x,
// i.e. the zero-point cross term of 第 6 课：量化源码走读 §3 is compensated with the group sum of
// the activations instead of subtracting z from every weight.
//
// Work split: the (256-row band, 256-k group pair) units -- one per pipeline stage -- are
// split evenly over the CTAs in band-major order.  A band covered by one CTA is written directly as bf16; a band shared
// by several CTAs is reduced through the workspace (fp32 partials + one counter per band,
// deterministic order: the last CTA to finish sums the partials in CTA order, writes bf16
// and resets the counter).
#include <mutex>

#include "decode_util.cuh"
#include "internal.h"

namespace wq {

__device__ uint32_t g_gemv_err;

uint32_t gemv_read_and_clear_error() {
  uint32_t v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, g_gemv_err, sizeof(v));
  cudaMemcpyToSymbol(g_gemv_err, &z, sizeof(z));
  return v;
}

namespace gemv {

using namespace dec;

constexpr int kConsumerWarps = 16;
constexpr int kRowsPerWarp = 16;                     // one m16 row tile per consumer warp
constexpr int kBand = kRowsPerWarp * kConsumerWarps;  // 256 weight rows per CTA tile
constexpr int kTileBytes = kBand * 128;              // 32 KB of packed weights per stage
constexpr int kPrepWarps = 3;                        // stage i is prepared by prep warp i % 3
constexpr int kXStages = 2 * kPrepWarps;             // activation-fragment ring depth
// Each prep warp owns whole ring slots (kXStages % kPrepWarps == 0), so it waits on every phase
// of its slots' barriers in order; a parity wait two phases ahead would pass at once.
static_assert(kXStages % kPrepWarps == 0, "prep warps must own whole ring slots");
constexpr int kFirstConsumer = 1 + kPrepWarps;       // warp index of the first consumer
constexpr int kThreads = 32 * (kFirstConsumer + kConsumerWarps);  // 640
constexpr int kGroupK = 128;                         // k per group (INT4 group; 4 MXFP4 blocks)
constexpr int kSmemLimit = 227 * 1024;               // dynamic shared memory per CTA
constexpr int kSmemReserve = 1024 + 512;             // alignment pad + barriers and flags

// Raw metadata tile(s) per weight stage: INT4 scales + zeros boxes of 8 groups x 256 rows
// (fp16); MXFP4 one box of 16 E8M0 bytes x 256 rows.
__host__ __device__ constexpr int meta_raw_bytes(int fmt) { return fmt == kInt4G128 ? 2 * kBand * 16 : kBand * 16; }
// One activation stage: B fragments + per-row group sums + per-row power-of-two factors.
__host__ __device__ constexpr int x_stage_bytes(int mt) { return (mt / 8) * 2 * 4 * 32 * 16 + 2 * mt * 4 + mt * 4; }
// Weight stages: as many as fit beside the activation ring (4 or 5).
__host__ __device__ constexpr int w_stages(int fmt, int mt) {
  return (kSmemLimit - kSmemReserve - kXStages * x_stage_bytes(mt)) / (kTileBytes + meta_raw_bytes(fmt)) > 6
             ? 6
             : (kSmemLimit - kSmemReserve - kXStages * x_stage_bytes(mt)) / (kTileBytes + meta_raw_bytes(fmt));
}

struct Params {
  const uint16_t* X;
  const void* scales;
  const uint16_t* zeros;
  uint16_t* Y;
  OutSplit split;     // EPI == kEpiSplit3: three output tensors by column range
  float* part;        // [P][2][MT][kBand] fp32 partials
  uint32_t* cnt;      // [bands] counters
  int M, K, N;
  int G;              // 128-k groups per row (ceil(K / 128))
  int GP;             // group pairs per row (ceil(G / 2)) -- one pair per stage
  int KB;             // MXFP4: scale bytes per row (K / 32)
  int bands;
  long long U;        // bands * GP units (one unit = one stage)
  int P;              // CTAs
  int meta_tma;       // 1: metadata tiles arrive by TMA with the weights; 0: consumers gather them
};

// The CTAs that share a band: [c_lo, c_hi].  CTA c_lo holds the band's first unit; every
// later contributor starts inside the band (partial slot 0); c_lo uses slot 1 when its range
// started in an earlier band (lo_side).
struct BandContrib { int c_lo, c_hi, lo_side; };


__device__ __forceinline__ long long unit_start(long long U, int P, int c) { return (U * c) / P; }

template <int FMT, int MT>
struct Smem {
  static constexpr int NT = MT / 8;
  static constexpr int WS = w_stages(FMT, MT);
  uint8_t w[WS][kTileBytes];                 // SWIZZLE_128B weight tiles (1024-aligned)
  uint8_t mraw[WS][meta_raw_bytes(FMT)];     // raw metadata tiles (TMA), 16 B per row per tensor
  // B fragments [nt][group][vec][lane].  A stage's raw activations (MT rows x 256 k bf16, row m
  // at byte 512 m -- the same size) land here by TMA and are converted in place.
  uint4 x[kXStages][NT][2][4][32];
  float xsum[kXStages][2][MT];               // INT4: sum of the group's activations per row m
  float xf[kXStages][MT];                    // MXFP4: power-of-two factor per activation row
  uint64_t full_w[WS];
  uint64_t empty_w[WS];
  uint64_t raw_x[kXStages];                  // the stage's raw activation rows landed (TMA)
  uint64_t full_x[kXStages];
  uint64_t empty_x[kXStages];
  uint64_t prep_done;                        // every prep thread arrives once it has no tail left
  // Split-K reductions this CTA must perform (a CTA has at most two partial bands): slot k
  // holds band + 1 once posted (release), 0 before; slots are claimed in order via req_alloc.
  int req_band[2];
  int req_alloc;
  // contributors of the CTA's first and last band (the only ones it can share), computed at
  // start-up off the critical path
  int ci_band[2];
  BandContrib ci[2];
};

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// Counter update that publishes (release) this CTA's partial sums and, for the last
// contributor, makes every other contributor's partial sums visible (acquire), at GPU scope.
__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ float4 ld_cg_f32x4(const float* p) { return __ldcg(reinterpret_cast<const float4*>(p)); }

__device__ __forceinline__ void st_release_cta(int* p, int v) {
  asm volatile("st.release.cta.shared.b32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire_cta(const int* p) {
  int v;
  asm volatile("ld.acquire.cta.shared.b32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
  return v;
}

// Contributors to a band: the CTAs whose unit range meets it, [c_lo, c_hi] (see BandContrib).

__device__ BandContrib band_contributors(const Params& p, int band) {
  const long long bs = static_cast<long long>(band) * p.GP, be = bs + p.GP;
  int c_lo = static_cast<int>((bs * p.P) / p.U);
  while (c_lo > 0 && unit_start(p.U, p.P, c_lo) > bs) --c_lo;
  while (unit_start(p.U, p.P, c_lo + 1) <= bs) ++c_lo;
  int c_hi = static_cast<int>(((be - 1) * p.P) / p.U);
  while (c_hi > c_lo && unit_start(p.U, p.P, c_hi) > be - 1) --c_hi;
  while (c_hi + 1 < p.P && unit_start(p.U, p.P, c_hi + 1) <= be - 1) ++c_hi;
  return BandContrib{c_lo, c_hi, unit_start(p.U, p.P, c_lo) < bs ? 1 : 0};
}

// One share of the deterministic split-K reduction of a band: the partial sums of every
// contributing CTA, added in CTA order, for the float4 slots idx = first, first + step, ...
// of the M x kBand outputs; bf16 results to Y.
template <int MT, int EPI>
__device__ __forceinline__ void reduce_band_share(const Params& p, int band, BandContrib bc, int first, int step) {
  const long long cstride = 2LL * MT * kBand;   // floats between two CTAs' partial slots
  [[maybe_unused]] const unsigned am = __activemask();   // the whole warp unless a wait timed out
  for (int idx = first; idx < p.M * (kBand / 4); idx += step) {
    int m, r4;
    if constexpr (EPI == kEpiSwiglu) {
      // slots idx and idx ^ 1 (lanes l and l ^ 1 of one warp): gate rows 16q + 4h .. + 3 and
      // the up rows 8 below them
      const int pr = idx >> 1, k = pr % (kBand / 8);
      m = pr / (kBand / 8);
      r4 = 16 * (k >> 1) + 4 * (k & 1) + 8 * (idx & 1);
    } else {
      m = idx / (kBand / 4);
      r4 = 4 * (idx % (kBand / 4));
    }
    const float* base = p.part + static_cast<long long>(m) * kBand + r4;
    float4 acc4 = ld_cg_f32x4(base + (static_cast<long long>(bc.c_lo) * 2 + bc.lo_side) * MT * kBand);
    for (int c = bc.c_lo + 1; c <= bc.c_hi; c += 8) {
      float4 v[8];   // up to eight contributors' loads in flight, summed in CTA order
#pragma unroll
      for (int q = 0; q < 8; ++q)
        v[q] = (c + q <= bc.c_hi) ? ld_cg_f32x4(base + static_cast<long long>(c + q) * cstride)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (c + q <= bc.c_hi) {
          acc4.x += v[q].x; acc4.y += v[q].y; acc4.z += v[q].z; acc4.w += v[q].w;
        }
    }
    const float o4[4] = {acc4.x, acc4.y, acc4.z, acc4.w};
    if constexpr (EPI == kEpiSwiglu) {
      // p.M * kBand / 4 is a multiple of 64 and every warp's idx range is 32-aligned: whole
      // warps run each iteration, so the shuffles below are converged
      float u4[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) u4[q] = __shfl_xor_sync(am, o4[q], 1);
      if ((idx & 1) == 0) {
        const int F = p.N >> 1;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int n = band * kBand + r4 + q;
          if (n < p.N)
            p.Y[static_cast<long long>(m) * F + swiglu_col(n)] =
                __bfloat16_as_ushort(__float2bfloat16_rn(silu_f32(o4[q]) * u4[q]));
        }
      }
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int n = band * kBand + r4 + q;
        if (n < p.N) {
          const uint16_t y = __bfloat16_as_ushort(__float2bfloat16_rn(o4[q]));
          if constexpr (EPI == kEpiSplit3) store_split3(p.split, m, n, y);
          else p.Y[static_cast<long long>(m) * p.N + n] = y;
        }
      }
    }
  }
}

// Stage i of a CTA = unit u0 + i = (band, group pair j).  Ranges are split at pair
// boundaries, so a stage never straddles a band.  The cursor divides once at start-up and
// then steps incrementally (64-bit division is a long software sequence on the GPU).
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
  __device__ bool seg_last() const { return u + 1 == seg_end; }    // last stage of this band here
  __device__ void next() {
    ++u;
    if (++j == GP) { j = 0; ++band; set_seg(); }
  }
};

template <int FMT, int MT, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    k_gemv(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_s,
           const __grid_constant__ CUtensorMap tmap_z, const __grid_constant__ CUtensorMap tmap_x,
           const Params p) {
  using S = Smem<FMT, MT>;
  constexpr int NT = MT / 8;
  constexpr int WS = S::WS;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  S& sm = *reinterpret_cast<S*>(smem_raw + smem_align_pad(smem_raw));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int cta = blockIdx.x;
  const long long u0 = unit_start(p.U, p.P, cta);
  const long long u1 = unit_start(p.U, p.P, cta + 1);
  const int nstages = static_cast<int>(u1 - u0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < WS; ++s) {
      mbar_init(&sm.full_w[s], 1);
      mbar_init(&sm.empty_w[s], 32 * kConsumerWarps);
    }
    for (int s = 0; s < kXStages; ++s) {
      mbar_init(&sm.raw_x[s], 1);
      mbar_init(&sm.full_x[s], 32);
      mbar_init(&sm.empty_x[s], 32 * kConsumerWarps);
    }
    mbar_init(&sm.prep_done, 32 * kPrepWarps);
    sm.req_band[0] = 0;
    sm.req_band[1] = 0;
    sm.req_alloc = 0;
    fence_barrier_init();
  }
  __syncthreads();

  // Metadata tile geometry (TMA path).
  //   INT4:  scales and zeros [N, G] fp16, box 8 groups x 256 rows at x = (2j) & ~7.
  //   MXFP4: E8M0 [N, K/32] bytes, box 16 bytes x 256 rows at x = (8j) & ~15.
  constexpr int kMetaBytes = meta_raw_bytes(FMT);

  // The next kernel of the stream may start its CTAs as this grid's CTAs exit.
  pdl_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
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
      {
        // While the previous kernel of the stream finishes: pull the first stages' weights
        // into L2.  Every read that lands in shared memory comes after the wait below.
        Cursor pf = st;
        for (int q = 0; q < WS && q < nstages; ++q, pf.next()) {
          tma_prefetch_l2_2d(&tmap_w, pf.j * 128, pf.band * kBand);
          if (p.meta_tma && (q == 0 || (FMT == kInt4G128 ? (pf.j & 3) == 0 : (pf.j & 1) == 0))) {
            if constexpr (FMT == kInt4G128) {
              tma_prefetch_l2_2d(&tmap_s, (2 * pf.j) & ~7, pf.band * kBand);
              tma_prefetch_l2_2d(&tmap_z, (2 * pf.j) & ~7, pf.band * kBand);
            } else {
              tma_prefetch_l2_2d(&tmap_s, (8 * pf.j) & ~15, pf.band * kBand);
            }
          }
        }
      }
      pdl_wait();
      int i = 0;
      for (; i < nstages; ++i, st.next()) {
        const int slot = i % WS;
        const uint32_t ph = (i / WS) & 1;
        if (!mbar_wait(&sm.empty_w[slot], ph ^ 1, &g_gemv_err, kErrWaitEmpty)) break;
        mbar_arrive_expect_tx(&sm.full_w[slot], kTileBytes + (p.meta_tma ? kMetaBytes : 0));
        tma_load_2d(&sm.w[slot][0], &tmap_w, st.j * 128, st.band * kBand, &sm.full_w[slot], pol_w);
        // the stage's activations into its fragment slot (free once stage i - kXStages is
        // consumed; never the binding wait: that ring is deeper than the weight ring)
        const int xs = i % kXStages;
        if (!mbar_wait(&sm.empty_x[xs], ((i / kXStages) & 1) ^ 1, &g_gemv_err, kErrWaitEmpty)) break;
        mbar_arrive_expect_tx(&sm.raw_x[xs], MT * 512);
        tma_load_2d(&sm.x[xs][0][0][0][0], &tmap_x, st.j * 256, 0, &sm.raw_x[xs], pol_m);
        if (p.meta_tma) {
          if constexpr (FMT == kInt4G128) {
            const int gx = (2 * st.j) & ~7;
            tma_load_2d(&sm.mraw[slot][0], &tmap_s, gx, st.band * kBand, &sm.full_w[slot], pol_m);
            tma_load_2d(&sm.mraw[slot][kBand * 16], &tmap_z, gx, st.band * kBand, &sm.full_w[slot], pol_m);
          } else {
            tma_load_2d(&sm.mraw[slot][0], &tmap_s, (8 * st.j) & ~15, st.band * kBand, &sm.full_w[slot], pol_m);
          }
        }
      }
      for (int jj = i - WS; jj < i; ++jj) {  // drain: the last fill of every slot landed
        if (jj < 0) continue;
        mbar_wait(&sm.full_w[jj % WS], (jj / WS) & 1, &g_gemv_err, kErrDrain);
      }
      for (int jj = i - kXStages; jj < i; ++jj) {
        if (jj < 0) continue;
        mbar_wait(&sm.raw_x[jj % kXStages], (jj / kXStages) & 1, &g_gemv_err, kErrDrain);
      }
    }
  } else if (warp < kFirstConsumer) {
    // ------------------------------------------------------------------ prep
    // Activations only.  The producer drops each stage's raw rows into the stage's fragment
    // slot by TMA (rows >= M and columns >= K zero-filled); prep warp i % 3 converts them in
    // place, off the weight ring's critical path and without global-memory latency.
    // Lane L owns the 16-byte chunk L (8 activations at k = 256 j + 8 L) of each row:
    //   INT4:  L = 16 h + 4 t + v  (group h, fragment lane t, vector v: k = 128 h + 32 t + 8 v)
    //   MXFP4: L = 16 h + 4 blk + t (group h, block blk, fragment lane t: k = 128 h + 32 blk + 8 t)
    const int pw = warp - 1;
    const int h = lane >> 4;
    const int ft = (FMT == kInt4G128) ? ((lane >> 2) & 3) : (lane & 3);   // fragment lane t
    const int fv = (FMT == kInt4G128) ? (lane & 3) : ((lane >> 2) & 3);   // vector / block
    Cursor st;
    st.init(u0, u1, p.GP, p.G);
    for (int q = 0; q < pw; ++q) st.next();
    // Split-K tails.  A band shared by several CTAs ends, in each of them, with fp32 partial
    // sums that the consumers store before releasing the stage's activation slot.  The prep
    // warp that next acquires that slot (the same warp: kXStages % kPrepWarps == 0) publishes
    // the contribution with one GPU-scope acq_rel counter update.  The last contributor posts
    // a reduction request; the 16 consumer warps sum every contributor's partials in CTA
    // order (deterministic) and write the bf16 outputs.  Nobody waits on another CTA.
    // Pending tails of this warp's last two stages (i - 3 and i - 6): band (-1: none), units.
    int tb0 = -1, tu0 = 0, tb1 = -1, tu1 = 0;
    auto split_tail = [&](int band, int units) {
      if (lane == 0) {
        const uint32_t old = atom_add_acq_rel_gpu(p.cnt + band, static_cast<uint32_t>(units));
        if (old + static_cast<uint32_t>(units) == static_cast<uint32_t>(p.GP)) {
          // last contributor: the consumers sum the band (acquire above, release below)
          atomicExch(p.cnt + band, 0u);   // ready for the next launch
          const int k = atomicAdd(&sm.req_alloc, 1);
          st_release_cta(&sm.req_band[k], band + 1);
        }
      }
      __syncwarp();
    };
    // (on the last prep warp: its first stage is the CTA's third, so short layers never wait for it)
    if (pw == kPrepWarps - 1 && lane == 0 && nstages > 0) {
#pragma unroll 1
      for (int q = 0; q < 2; ++q) {
        const int band = static_cast<int>((q == 0 ? u0 : u1 - 1) / p.GP);
        sm.ci_band[q] = band;
        sm.ci[q] = band_contributors(p, band);
      }
    }
    pdl_wait();   // the split-K counters may come from the previous kernel
    // Stages i >= nstages are not prepared; their slot waits only deliver the last tails.
    for (int i = pw; i < nstages + kXStages; i += kPrepWarps) {
      const int slot = i % kXStages;
      const uint32_t ph = (i / kXStages) & 1;
      const bool hs = ((i / kPrepWarps) & 1) != 0;
      const int pend_band = hs ? tb1 : tb0;          // tail of stage i - kXStages, -1 if none
      const int pend_units = hs ? tu1 : tu0;
      if (i >= nstages && pend_band < 0) continue;  // nothing left to publish
      if (!mbar_wait(&sm.empty_x[slot], ph ^ 1, &g_gemv_err, kErrWaitEmpty)) break;
      // the consumers are done with stage i - kXStages (same slot) and stored its partials
      if (pend_band >= 0) split_tail(pend_band, pend_units);
      int nb = -1, nu = 0;
      if (i < nstages && st.seg_last()) {
        const int band = st.band;
        const bool full = (st.seg_start == static_cast<long long>(band) * p.GP) &&
                          (st.seg_end == static_cast<long long>(band + 1) * p.GP);
        if (!full) { nb = band; nu = static_cast<int>(st.seg_end - st.seg_start); }
      }
      if (hs) { tb1 = nb; tu1 = nu; } else { tb0 = nb; tu0 = nu; }
      if (i >= nstages) continue;
      for (int q = 0; q < kPrepWarps; ++q) st.next();
      if (!mbar_wait(&sm.raw_x[slot], ph, &g_gemv_err, kErrWaitFull)) break;
      uint4* xs4 = &sm.x[slot][0][0][0][0];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        // 8 rows (one n-tile) in registers, then written back permuted: a row's fragment
        // positions hold other rows' raw chunks, so every read of the tile precedes every write.
        const int mlive = p.M - 8 * nt;   // rows of this tile below M
        uint4 cur[8];
#pragma unroll
        for (int r = 0; r < 8; ++r)
          cur[r] = (r < mlive) ? xs4[(8 * nt + r) * 32 + lane] : make_uint4(0u, 0u, 0u, 0u);
        __syncwarp();
        // MXFP4: one power-of-two scale 2^-k per stage and activation row carries every operand
        // into fp16 exactly (bf16_to_f16_exponent: the row's largest in [2^14, 2^15), small
        // rows scaled up); only values more than 2^31 below their row's largest lose bits, as
        // fp16 subnormals.  max |x| per row: bf16 magnitudes order like integers; two rows'
        // maxima share a word for the warp reduction.
        float inv[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) inv[r] = 1.f;
        if constexpr (FMT != kInt4G128) {
          uint32_t mxp[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t m2[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const uint4 x = cur[2 * q + u];
              const uint32_t v = __vmaxu2(__vmaxu2(x.x & 0x7fff7fffu, x.y & 0x7fff7fffu),
                                          __vmaxu2(x.z & 0x7fff7fffu, x.w & 0x7fff7fffu));
              m2[u] = max(v & 0xffffu, v >> 16);
            }
            mxp[q] = m2[0] | (m2[1] << 16);
          }
#pragma unroll
          for (int sh = 1; sh < 32; sh <<= 1)
#pragma unroll
            for (int q = 0; q < 4; ++q) mxp[q] = __vmaxu2(mxp[q], __shfl_xor_sync(0xffffffffu, mxp[q], sh));
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            const int kk = bf16_to_f16_exponent((mxp[r >> 1] >> (16 * (r & 1))) & 0xffffu);
            inv[r] = pow2_normal(-kk);
            if (lane == r) sm.xf[slot][8 * nt + r] = pow2_normal(kk);
          }
        }
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          uint4* dst = &sm.x[slot][nt][h][fv][4 * r + ft];
          if (r >= mlive) {   // zero-filled row: zero fragments (INT4: zero sums below)
            *dst = make_uint4(0u, 0u, 0u, 0u);
            continue;
          }
          const uint4 x = cur[r];
          const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
          if constexpr (FMT == kInt4G128) {
            // (x0,x4) (x1,x5) (x2,x6) (x3,x7): the k order of the unpacked nibble pairs.
            uint4 o;
            o.x = prmt(x.x, x.z, 0x5410);
            o.y = prmt(x.x, x.z, 0x7632);
            o.z = prmt(x.y, x.w, 0x5410);
            o.w = prmt(x.y, x.w, 0x7632);
            *dst = o;
          } else {
            uint32_t o[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              __half2 hh = __floats2half2_rn(__uint_as_float(w4[q] << 16) * inv[r],
                                             __uint_as_float(w4[q] & 0xffff0000u) * inv[r]);
              o[q] = *reinterpret_cast<uint32_t*>(&hh);
            }
            *dst = make_uint4(o[0], o[1], o[2], o[3]);
          }
        }
        if constexpr (FMT == kInt4G128) {
          // Per-group activation sums of the tile's 8 rows on the tensor core: an all-ones A
          // times the just-written B fragments gives every column sum (exact products, fp32
          // accumulation).  Lane (g = 0, t) receives rows 2t, 2t + 1 of the tile.
          __syncwarp();
          // (four independent accumulator chains per group: the MMA latency bounds this step)
          constexpr uint32_t kOnes = 0x3f803f80u;   // bf16 (1, 1)
#pragma unroll
          for (int hg = 0; hg < 2; ++hg) {
            float d[4][4];
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const uint4 b = sm.x[slot][nt][hg][v][lane];
#pragma unroll
              for (int e = 0; e < 4; ++e) d[v][e] = 0.f;
              mma_bf16(d[v], kOnes, kOnes, kOnes, kOnes, b.x, b.y);
              mma_bf16(d[v], kOnes, kOnes, kOnes, kOnes, b.z, b.w);
            }
            const float s0 = (d[0][0] + d[1][0]) + (d[2][0] + d[3][0]);
            const float s1 = (d[0][1] + d[1][1]) + (d[2][1] + d[3][1]);
            if (lane < 4) *reinterpret_cast<float2*>(&sm.xsum[slot][hg][8 * nt + 2 * lane]) = make_float2(s0, s1);
          }
        }
      }
      // the slot is refilled by TMA (async proxy) once consumed: order these generic writes first
      fence_proxy_async_smem();
      mbar_arrive(&sm.full_x[slot]);
    }
    mbar_arrive(&sm.prep_done);
  } else {
    // ------------------------------------------------------------------ consumers
    const int cw = warp - kFirstConsumer;
    const int g = lane >> 2;
    const int t = lane & 3;
    const int r0 = cw * kRowsPerWarp + frag_row(g);      // rows (inside the band) of this lane
    const int r1 = cw * kRowsPerWarp + frag_row(g + 8);

    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;

    Cursor st;
    st.init(u0, u1, p.GP, p.G);
    for (int i = 0; i < nstages; ++i, st.next()) {
      const int ws = i % WS;
      const uint32_t wph = (i / WS) & 1;
      const int xs = i % kXStages;
      const uint32_t xph = (i / kXStages) & 1;

      // Per-row metadata of the stage's two groups, rows r0 / r1 of this lane:
      //   INT4: sc[h][rr] = {s, c = -s (128 + z)}     MXFP4: eb[rr] = E8M0 bytes of the 8 blocks
      // Without metadata tiles they are gathered from global memory before the waits.
      uint32_t sraw[2] = {0u, 0u}, zraw[2] = {0u, 0u};   // INT4: fp16 pairs (group 2j, 2j+1)
      uint32_t eb[2][2] = {{0u, 0u}, {0u, 0u}};          // MXFP4: [row][group] 4 E8M0 bytes
      if (!p.meta_tma) {
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
          const int row = st.band * kBand + (rr ? r1 : r0);
          if (row >= p.N) continue;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if constexpr (FMT == kInt4G128) {
              if (2 * st.j + h < p.G) {
                const long long idx = static_cast<long long>(row) * p.G + 2 * st.j + h;
                sraw[rr] |= static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(p.scales) + idx)) << (16 * h);
                zraw[rr] |= static_cast<uint32_t>(__ldg(p.zeros + idx)) << (16 * h);
              }
            } else {
              const uint8_t* E = reinterpret_cast<const uint8_t*>(p.scales) + static_cast<long long>(row) * p.KB;
              const int b0 = (2 * st.j + h) * 4;
#pragma unroll
              for (int q2 = 0; q2 < 4; ++q2)
                if (b0 + q2 < p.KB) eb[rr][h] |= static_cast<uint32_t>(__ldg(E + b0 + q2)) << (8 * q2);
            }
          }
        }
      }

      if (!mbar_wait(&sm.full_x[xs], xph, &g_gemv_err, kErrWaitFull)) break;
      if (!mbar_wait(&sm.full_w[ws], wph, &g_gemv_err, kErrWaitFull)) break;

      if (p.meta_tma) {
        if constexpr (FMT == kInt4G128) {
          const int cb = 2 * ((2 * st.j) & 7);   // byte offset of group 2j inside the 16-byte row
          sraw[0] = *reinterpret_cast<const uint32_t*>(&sm.mraw[ws][r0 * 16 + cb]);
          sraw[1] = *reinterpret_cast<const uint32_t*>(&sm.mraw[ws][r1 * 16 + cb]);
          zraw[0] = *reinterpret_cast<const uint32_t*>(&sm.mraw[ws][kBand * 16 + r0 * 16 + cb]);
          zraw[1] = *reinterpret_cast<const uint32_t*>(&sm.mraw[ws][kBand * 16 + r1 * 16 + cb]);
        } else {
          const int cw4 = ((8 * st.j) & 15) >> 2;  // word of group 2j inside the 16-byte row
          const uint2 e0 = *reinterpret_cast<const uint2*>(&sm.mraw[ws][r0 * 16 + 4 * cw4]);
          const uint2 e1 = *reinterpret_cast<const uint2*>(&sm.mraw[ws][r1 * 16 + 4 * cw4]);
          eb[0][0] = e0.x; eb[0][1] = e0.y;
          eb[1][0] = e1.x; eb[1][1] = e1.y;
        }
      }

      const uint8_t* wt = &sm.w[ws][0];
      if constexpr (FMT == kInt4G128) {
        // Both groups at once.  PAR words per step with their own accumulators keep four
        // independent MMA chains in flight per warp (groups x word parity x n-tiles).
        constexpr int PAR = (NT == 1) ? 2 : 1;
        uint32_t w0[2][4], w1[2][4];   // [group][word] rows r0 / r1
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int c = 4 * h + t;
          const uint4 a = *reinterpret_cast<const uint4*>(wt + r0 * 128 + ((c ^ (r0 & 7)) << 4));
          const uint4 b = *reinterpret_cast<const uint4*>(wt + r1 * 128 + ((c ^ (r1 & 7)) << 4));
          w0[h][0] = a.x; w0[h][1] = a.y; w0[h][2] = a.z; w0[h][3] = a.w;
          w1[h][0] = b.x; w1[h][1] = b.y; w1[h][2] = b.z; w1[h][3] = b.w;
        }
        float ga[2][PAR][NT][4];
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int q = 0; q < PAR; ++q)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int e = 0; e < 4; ++e) ga[h][q][nt][e] = 0.f;
#pragma unroll
        for (int jh = 0; jh < 4 / PAR; ++jh) {
          uint4 bx[2][PAR][NT];
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int q = 0; q < PAR; ++q)
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) bx[h][q][nt] = sm.x[xs][nt][h][jh * PAR + q][lane];
#pragma unroll
          for (int hh = 0; hh < 2; ++hh)
#pragma unroll
            for (int q = 0; q < PAR; ++q)
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const int jw = jh * PAR + q;
                // nibble pairs (s, s+4) as bf16 128 + q (exact); the zero point is folded below
                const uint32_t a0 = lop3_and_or(w0[h][jw] >> (8 * hh), 0x000f000fu, 0x43004300u);
                const uint32_t a1 = lop3_and_or(w1[h][jw] >> (8 * hh), 0x000f000fu, 0x43004300u);
                const uint32_t a2 = lop3_and_or(w0[h][jw] >> (8 * hh + 4), 0x000f000fu, 0x43004300u);
                const uint32_t a3 = lop3_and_or(w1[h][jw] >> (8 * hh + 4), 0x000f000fu, 0x43004300u);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                  const uint4 bv = bx[h][q][nt];
                  mma_bf16(ga[h][q][nt], a0, a1, a2, a3, hh ? bv.z : bv.x, hh ? bv.w : bv.y);
                }
              }
        }
        // y += s * sum_k (128 + q) x + c * sum_k x,  c = -s (128 + z)   (zero-point cross term)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float s0 = __half2float(__ushort_as_half(static_cast<unsigned short>(sraw[0] >> (16 * h))));
          const float s1 = __half2float(__ushort_as_half(static_cast<unsigned short>(sraw[1] >> (16 * h))));
          const float c0 = -s0 * (128.f + __half2float(__ushort_as_half(static_cast<unsigned short>(zraw[0] >> (16 * h)))));
          const float c1 = -s1 * (128.f + __half2float(__ushort_as_half(static_cast<unsigned short>(zraw[1] >> (16 * h)))));
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const float2 xs2 = *reinterpret_cast<const float2*>(&sm.xsum[xs][h][2 * t + 8 * nt]);
            float gs[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              gs[e] = ga[h][0][nt][e];
#pragma unroll
              for (int q = 1; q < PAR; ++q) gs[e] += ga[h][q][nt][e];
            }
            acc[nt][0] = fmaf(c0, xs2.x, fmaf(s0, gs[0], acc[nt][0]));
            acc[nt][1] = fmaf(c0, xs2.y, fmaf(s0, gs[1], acc[nt][1]));
            acc[nt][2] = fmaf(c1, xs2.x, fmaf(s1, gs[2], acc[nt][2]));
            acc[nt][3] = fmaf(c1, xs2.y, fmaf(s1, gs[3], acc[nt][3]));
          }
        }
      } else {
        // MXFP4: lane t holds 8 codes of each 32-block; two k16 steps per block.  The two
        // groups' blocks run side by side (independent accumulators).
        float sacc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) sacc[nt][e] = 0.f;
#pragma unroll
        for (int blk = 0; blk < 4; ++blk) {
          uint32_t wr0[2], wr1[2];
          uint4 bx[2][NT];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int c = 4 * h + blk;
            wr0[h] = *reinterpret_cast<const uint32_t*>(wt + r0 * 128 + ((c ^ (r0 & 7)) << 4) + 4 * t);
            wr1[h] = *reinterpret_cast<const uint32_t*>(wt + r1 * 128 + ((c ^ (r1 & 7)) << 4) + 4 * t);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) bx[h][nt] = sm.x[xs][nt][h][blk][lane];
          }
          float bacc[2][NT][4];
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int e = 0; e < 4; ++e) bacc[h][nt][e] = 0.f;
          uint32_t f0[2][4], f1[2][4];   // [group][byte] rows r0 / r1 as f16x2
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            e2m1x8_to_f16x2x4(wr0[h], f0[h]);
            e2m1x8_to_f16x2x4(wr1[h], f1[h]);
          }
#pragma unroll
          for (int hh = 0; hh < 2; ++hh)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint32_t a0 = f0[h][2 * hh], a2 = f0[h][2 * hh + 1];
              const uint32_t a1 = f1[h][2 * hh], a3 = f1[h][2 * hh + 1];
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) {
                const uint4 bv = bx[h][nt];
                mma_f16(bacc[h][nt], a0, a1, a2, a3, hh ? bv.z : bv.x, hh ? bv.w : bv.y);
              }
            }
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const float f0 = e8m0_to_f32((eb[0][h] >> (8 * blk)) & 0xffu);
            const float f1 = e8m0_to_f32((eb[1][h] >> (8 * blk)) & 0xffu);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              sacc[nt][0] = fmaf(f0, bacc[h][nt][0], sacc[nt][0]);
              sacc[nt][1] = fmaf(f0, bacc[h][nt][1], sacc[nt][1]);
              sacc[nt][2] = fmaf(f1, bacc[h][nt][2], sacc[nt][2]);
              sacc[nt][3] = fmaf(f1, bacc[h][nt][3], sacc[nt][3]);
            }
          }
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const float2 xf = *reinterpret_cast<const float2*>(&sm.xf[xs][2 * t + 8 * nt]);
          acc[nt][0] = fmaf(xf.x, sacc[nt][0], acc[nt][0]);
          acc[nt][1] = fmaf(xf.y, sacc[nt][1], acc[nt][1]);
          acc[nt][2] = fmaf(xf.x, sacc[nt][2], acc[nt][2]);
          acc[nt][3] = fmaf(xf.y, sacc[nt][3], acc[nt][3]);
        }
      }
      mbar_arrive(&sm.empty_w[ws]);   // weights consumed: the producer may refill the slot

      if (st.seg_last()) {
        const int band = st.band;
        const bool full = (st.seg_start == static_cast<long long>(band) * p.GP) &&
                          (st.seg_end == static_cast<long long>(band + 1) * p.GP);
        if (full) {
          if constexpr (EPI == kEpiSwiglu) {
            // r1 = r0 + 8: this lane holds gate (e = 0, 1) and up (e = 2, 3) of one output
            const int n = band * kBand + r0;
            const int F = p.N >> 1;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int m = 2 * t + e + 8 * nt;
                if (m < p.M && n < p.N)
                  p.Y[static_cast<long long>(m) * F + swiglu_col(n)] =
                      __bfloat16_as_ushort(__float2bfloat16_rn(silu_f32(acc[nt][e]) * acc[nt][e + 2]));
              }
          } else {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int m = 2 * t + (e & 1) + 8 * nt;
                const int n = band * kBand + ((e >> 1) ? r1 : r0);
                if (m < p.M && n < p.N) {
                  const uint16_t y = __bfloat16_as_ushort(__float2bfloat16_rn(acc[nt][e]));
                  if constexpr (EPI == kEpiSplit3) store_split3(p.split, m, n, y);
                  else p.Y[static_cast<long long>(m) * p.N + n] = y;
                }
              }
          }
        } else {
          // partial sums; the prep warp owning this activation slot publishes them
          const int side = (u0 >= static_cast<long long>(band) * p.GP) ? 0 : 1;
          float* slotp = p.part + (static_cast<long long>(cta) * 2 + side) * MT * kBand;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int m = 2 * t + (e & 1) + 8 * nt;
              __stcg(slotp + m * kBand + ((e >> 1) ? r1 : r0), acc[nt][e]);
            }
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
      }
      mbar_arrive(&sm.empty_x[xs]);   // release: orders the partial-sum stores before the tail
    }
    // Reductions posted by the prep warps (the last tails are published after the final
    // stage): wait until the prep warps are done, then take this warp's share, 1/16 of the
    // float4 slots of each band.
    if (mbar_wait(&sm.prep_done, 0, &g_gemv_err, kErrWaitReduce)) {
#pragma unroll 1
      for (int k = 0; k < 2; ++k) {
        const int b1 = ld_acquire_cta(&sm.req_band[k]);
        if (b1 == 0) break;
        const BandContrib bc = sm.ci[sm.ci_band[0] == b1 - 1 ? 0 : 1];
        reduce_band_share<MT, EPI>(p, b1 - 1, bc, cw * 32 + lane, 32 * kConsumerWarps);
      }
    }
  }
}

int num_ctas(long long U) {
  const long long sms = device_sm_count();
  return static_cast<int>(U < sms ? U : sms);
}

}  // namespace gemv

size_t gemv_mma_workspace_bytes(int fmt, int64_t M, int64_t K, int64_t N) {
  if (M < 1 || M > 16 || N < 1 || K < 1) return 0;
  const int MT = M <= 8 ? 8 : 16;
  const long long G = (K + gemv::kGroupK - 1) / gemv::kGroupK;
  const long long bands = (N + gemv::kBand - 1) / gemv::kBand;
  const int P = gemv::num_ctas(bands * ((G + 1) / 2));
  (void)fmt;
  return kWsCounterBytes + static_cast<size_t>(P) * 2 * MT * gemv::kBand * sizeof(float);
}

template <int FMT, int MT, int EPI>
static cudaError_t launch_gemv_t(const CUtensorMap& tw, const CUtensorMap& ts, const CUtensorMap& tz,
                                 const gemv::Params& p, cudaStream_t stream) {
  // activations: MT rows x 256 k per stage; rows >= M and columns >= K come back as zeros
  CUtensorMap tx;
  cudaError_t ex = make_tmap_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.X, static_cast<uint64_t>(p.K),
                                static_cast<uint64_t>(p.M), static_cast<uint64_t>(p.K) * 2, 256, MT,
                                CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
  if (ex != cudaSuccess) return ex;
  using S = gemv::Smem<FMT, MT>;
  static_assert(sizeof(S) + 1024 <= gemv::kSmemLimit, "decode kernel shared memory over the per-CTA limit");
  const size_t smem = sizeof(S) + 1024;
  auto kern = gemv::k_gemv<FMT, MT, EPI>;
  cudaError_t ea = set_smem_attr_once(reinterpret_cast<const void*>(kern), smem);
  if (ea != cudaSuccess) return ea;
  // Programmatic stream serialization: the CTAs may launch while the previous kernel of the
  // stream is still running; the kernel itself waits (griddepcontrol.wait) before it reads
  // anything that kernel may have written.
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(p.P));
  cfg.blockDim = dim3(gemv::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tw, ts, tz, tx, p);
}

cudaError_t launch_gemv_mma(int fmt, const uint16_t* X, int64_t M, int64_t K, int64_t N, const int32_t* Wq,
                            const void* scales, const uint16_t* zeros, uint16_t* Y, void* ws, size_t ws_bytes,
                            cudaStream_t stream, int epi, const OutSplit* split) {
  if (epi == kEpiSwiglu && N % 16 != 0) return cudaErrorInvalidValue;
  if (epi == kEpiSplit3 && !split) return cudaErrorInvalidValue;
  gemv::Params p{};
  p.X = X;
  p.scales = scales;
  p.zeros = zeros;
  p.Y = Y;
  if (split) p.split = *split;
  p.M = static_cast<int>(M);
  p.K = static_cast<int>(K);
  p.N = static_cast<int>(N);
  p.G = static_cast<int>((K + gemv::kGroupK - 1) / gemv::kGroupK);
  p.GP = (p.G + 1) / 2;
  p.KB = static_cast<int>(K / 32);
  p.bands = static_cast<int>((N + gemv::kBand - 1) / gemv::kBand);
  p.U = static_cast<long long>(p.bands) * p.GP;
  p.P = gemv::num_ctas(p.U);
  if (p.bands > kWsMaxCounters) return cudaErrorInvalidValue;
  if (ws_bytes < gemv_mma_workspace_bytes(fmt, M, K, N)) return cudaErrorInvalidValue;
  p.cnt = reinterpret_cast<uint32_t*>(ws);
  p.part = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ws) + kWsCounterBytes);

  CUtensorMap tw, ts, tz;
  cudaError_t e = make_tmap_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, Wq, static_cast<uint64_t>(K / 2),
                               static_cast<uint64_t>(N), static_cast<uint64_t>(K / 2), 128, gemv::kBand,
                               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
  if (e != cudaSuccess) return e;
  // Metadata tiles travel with the weights by TMA when the metadata row pitch is a multiple
  // of 16 bytes (INT4: K % 1024 == 0; MXFP4: K % 512 == 0); otherwise the consumers gather
  // them.  Unused descriptors are copies of the weight descriptor (never dereferenced).
  ts = tw;
  tz = tw;
  if (fmt == kInt4G128) {
    p.meta_tma = (p.G % 8 == 0) ? 1 : 0;
    if (p.meta_tma) {
      e = make_tmap_2d(&ts, CU_TENSOR_MAP_DATA_TYPE_UINT16, scales, static_cast<uint64_t>(p.G),
                       static_cast<uint64_t>(N), static_cast<uint64_t>(p.G) * 2, 8, gemv::kBand,
                       CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE);
      if (e != cudaSuccess) return e;
      e = make_tmap_2d(&tz, CU_TENSOR_MAP_DATA_TYPE_UINT16, zeros, static_cast<uint64_t>(p.G),
                       static_cast<uint64_t>(N), static_cast<uint64_t>(p.G) * 2, 8, gemv::kBand,
                       CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE);
      if (e != cudaSuccess) return e;
    }
  } else {
    p.meta_tma = (p.KB % 16 == 0) ? 1 : 0;
    if (p.meta_tma) {
      e = make_tmap_2d(&ts, CU_TENSOR_MAP_DATA_TYPE_UINT8, scales, static_cast<uint64_t>(p.KB),
                       static_cast<uint64_t>(N), static_cast<uint64_t>(p.KB), 16, gemv::kBand,
                       CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE);
      if (e != cudaSuccess) return e;
    }
  }
  const bool small = M <= 8;
#define WQ_BAND_LAUNCH(EPIV)                                                                                   \
  if (fmt == kInt4G128)                                                                                        \
    return small ? launch_gemv_t<kInt4G128, 8, EPIV>(tw, ts, tz, p, stream)                                   \
                 : launch_gemv_t<kInt4G128, 16, EPIV>(tw, ts, tz, p, stream);                                 \
  return small ? launch_gemv_t<kMxfp4, 8, EPIV>(tw, ts, tz, p, stream)                                        \
               : launch_gemv_t<kMxfp4, 16, EPIV>(tw, ts, tz, p, stream);
  if (epi == kEpiSwiglu) { WQ_BAND_LAUNCH(kEpiSwiglu) }
  if (epi == kEpiSplit3) { WQ_BAND_LAUNCH(kEpiSplit3) }
  WQ_BAND_LAUNCH(kEpiNone)
#undef WQ_BAND_LAUNCH
}

// The decode entry points run the mma.sync kernel above.  (A tcgen05 variant was measured
// slower: at N = 16 one 128 x 16 x 16 tcgen05.mma costs ~56 cycles, which caps a 256-row
// stage below the per-SM share of HBM bandwidth.)
size_t gemv_workspace_bytes(int fmt, int64_t M, int64_t K, int64_t N) { return gemv_mma_workspace_bytes(fmt, M, K, N); }

cudaError_t launch_gemv(int fmt, const uint16_t* X, int64_t M, int64_t K, int64_t N, const int32_t* Wq,
                        const void* scales, const uint16_t* zeros, uint16_t* Y, void* ws, size_t ws_bytes,
                        cudaStream_t stream, int epi, const OutSplit* split) {
  return launch_gemv_mma(fmt, X, M, K, N, Wq, scales, zeros, Y, ws, ws_bytes, stream, epi, split);
}

// ---------------------------------------------------------------------------------------
// The decode kernel for callers that cannot allocate device memory.
//
// The split-K scratch of the decode kernel (reduction counters and fp32 partial sums) lives
// here in one fixed, library-owned device array instead of a caller-provided workspace.  It
// is sized for every decode shape the kernel accepts (M <= 16, N <= 2097152) on a device with
// at most kNoAllocMaxCtas SMs: 64 KiB of counters + 8 MiB of partials.  Every GPU that loads
// the library keeps this array until the process exits.
// ---------------------------------------------------------------------------------------
constexpr int kNoAllocMaxCtas = 256;
constexpr size_t kNoAllocScratchBytes =
    kWsCounterBytes + static_cast<size_t>(kNoAllocMaxCtas) * 2 * 16 * gemv::kBand * sizeof(float);

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

size_t gemv_noalloc_scratch_bytes() { return kNoAllocScratchBytes; }

cudaError_t launch_gemv_noalloc(int fmt, const uint16_t* X, int64_t M, int64_t K, int64_t N, const int32_t* Wq,
                                const void* scales, const uint16_t* zeros, uint16_t* Y, cudaStream_t stream) {
  // Set-up, once per device (and again if the device's context was replaced, e.g. after a
  // cudaDeviceReset, which unloads the module and can move the array), with that device
  // current: the array's name is only a host-side handle, so the kernel gets the device
  // address from cudaGetSymbolAddress.
  static std::mutex mu;
  static void* addr[64] = {nullptr};
  static CUcontext addr_ctx[64] = {nullptr};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (!addr[dev] || current_context() != addr_ctx[dev]) {
      void* a = nullptr;
      e = cudaGetSymbolAddress(&a, g_noalloc_scratch);
      if (e != cudaSuccess) return e;
      addr[dev] = a;
      addr_ctx[dev] = current_context();   // current now: the lookup initialised it
    }
    scratch = addr[dev];
  }
  if (gemv_workspace_bytes(fmt, M, K, N) > kNoAllocScratchBytes) return cudaErrorInvalidValue;
  // The array keeps whatever the previous call left; the counters must start at zero.
  const size_t bands = static_cast<size_t>((N + gemv::kBand - 1) / gemv::kBand);
  e = cudaMemsetAsync(scratch, 0, bands * sizeof(uint32_t), stream);
  if (e != cudaSuccess) return e;
  return launch_gemv(fmt, X, M, K, N, Wq, scales, zeros, Y, scratch, kNoAllocScratchBytes, stream);
}

}  // namespace wq
