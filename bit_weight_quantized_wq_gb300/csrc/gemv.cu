// Decode kernel (M <= 16): Y[M, N] = X[M, K] * dequant(Wq)^T.
//
// Bandwidth-bound (推理优化与量化算子深度技术调研 §1.3: at batch 1 the W4A16 GEMV is limited by
// HBM bandwidth; 第 1 章：推理加速全景 §1.2-1.3: decode arithmetic intensity ~1 FLOP/B), so the
// design goal is to stream the 0.53125 B/weight of packed weights + metadata once, at full
// HBM bandwidth, with the arithmetic hidden underneath.
//
// Structure (one persistent CTA per SM, warp-specialised, 20 warps):
//   warp 0      TMA producer: 256-row x 128-byte tiles of the packed weights (two 128-k
//               groups of INT4 / 256 k of MXFP4), SWIZZLE_128B, into a 3-stage smem ring,
//               plus the matching scale / zero-point (INT4) or E8M0 (MXFP4) tiles.
//   warps 1-3   prep (stage i by prep warp i % 3): the activations of the stage's k-range in
//               the exact order of the mma.sync B fragments, with their per-group sums (INT4)
//               or converted to fp16 with a per-row power-of-two scale that keeps every value
//               in fp16 range (MXFP4); and the per-row metadata of the stage in the form the
//               consumers use.  The consumers touch only shared memory in their main loop.
//   warps 4-19  consumers: 16 weight rows each; unpack nibbles in registers, tensor-core
//               mma.sync with fp32 accumulation, group scale applied in fp32 afterwards.
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

constexpr int kConsumerWarps = 16;
constexpr int kRowsPerWarp = 16;                     // one m16 row tile per consumer warp
constexpr int kBand = kRowsPerWarp * kConsumerWarps;  // 256 weight rows per CTA tile
constexpr int kStages = 3;
constexpr int kTileBytes = kBand * 128;              // 32 KB of packed weights per stage
constexpr int kPrepWarps = kStages;                  // stage i is prepared by prep warp i % 3
// Each prep warp owns whole ring slots (kStages % kPrepWarps == 0), so it waits on every phase
// of its slots' barriers in order; a parity wait two phases ahead would pass at once.
static_assert(kStages % kPrepWarps == 0, "prep warps must own whole ring slots");
constexpr int kFirstConsumer = 1 + kPrepWarps;       // warp index of the first consumer
constexpr int kThreads = 32 * (kFirstConsumer + kConsumerWarps);  // 608
constexpr int kGroupK = 128;                         // k per group (INT4 group; 4 MXFP4 blocks)
constexpr int kMetaRawBytes = kBand * 16 * 2;        // raw metadata tile(s) per stage (8 KB max)

struct Params {
  const uint16_t* X;
  const void* scales;
  const uint16_t* zeros;
  uint16_t* Y;
  float* part;        // [P][2][MT][kBand] fp32 partials
  uint32_t* cnt;      // [bands] counters
  int M, K, N;
  int G;              // 128-k groups per row (ceil(K / 128))
  int GP;             // group pairs per row (ceil(G / 2)) -- one pair per stage
  int KB;             // MXFP4: scale bytes per row (K / 32)
  int bands;
  long long U;        // bands * GP units (one unit = one stage)
  int P;              // CTAs
  int meta_tma;       // 1: metadata tiles arrive by TMA with the weights; 0: prep warps gather them
};

// Fragment row f (0..15) of a 16-row tile -> row inside the tile.  Rows g and g+4 of a
// smem swizzle atom then land in disjoint bank groups, so the consumer's 128-bit loads
// are conflict-free.
__device__ __forceinline__ int frag_row(int f) { return (f & 8) | ((f >> 1) & 3) | ((f & 1) << 2); }

__device__ __forceinline__ long long unit_start(long long U, int P, int c) { return (U * c) / P; }

template <int FMT, int MT>
struct Smem {
  static constexpr int NT = MT / 8;
  uint8_t w[kStages][kTileBytes];            // SWIZZLE_128B weight tiles (1024-aligned)
  uint8_t mraw[kStages][kMetaRawBytes];      // raw metadata tiles (TMA), 16 B per row per tensor
  uint8_t xraw[kStages][MT * 512];           // raw activations of the stage (TMA): MT rows x 256 k bf16
  uint4 x[kStages][NT][2][4][32];            // B fragments [nt][group][vec][lane]
  float xsum[kStages][2][MT];                // INT4: sum of the group's activations per row m
  float xf[kStages][MT];                     // MXFP4: power-of-two factor per activation row
  // Per-row metadata of the stage's two groups, prepared by the prep warps:
  //   INT4:  {s, c = -s (128 + z)}     MXFP4: {four E8M0 bytes, unused}
  float2 meta[kStages][2][kBand];
  uint64_t full_w[kStages];
  uint64_t full_x[kStages];
  uint64_t empty[kStages];
  uint64_t group_bar;                        // consumer barrier (bounded wait), split-K path
  int reduce_flag;
};

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));  // (a & b) | c
  return d;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Two E2M1 codes (low nibble = first element) -> f16x2 (low half = first element), exact.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t d;
  const unsigned short h = static_cast<unsigned short>(byte);
  asm("{\n\t.reg .b8 t, u;\n\tmov.b16 {t, u}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(d) : "h"(h));
  return d;
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 2^(byte - 127) as a float for an E8M0 byte (byte 0 -> 2^-127, subnormal).
__device__ __forceinline__ float e8m0_to_f32(uint32_t byte) {
  return byte ? __uint_as_float(byte << 23) : __uint_as_float(0x00400000u);
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
  __device__ int ng() const { return (2 * j + 1 < G) ? 2 : 1; }   // groups of the pair inside K
  __device__ bool seg_last() const { return u + 1 == seg_end; }    // last stage of this band here
  __device__ void next() {
    ++u;
    if (++j == GP) { j = 0; ++band; set_seg(); }
  }
};

template <int FMT, int MT>
__global__ void __launch_bounds__(kThreads, 1)
    k_gemv(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_s,
           const __grid_constant__ CUtensorMap tmap_z, const __grid_constant__ CUtensorMap tmap_x,
           const Params p) {
  using S = Smem<FMT, MT>;
  constexpr int NT = MT / 8;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  S& sm = *reinterpret_cast<S*>(smem_raw + smem_align_pad(smem_raw));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int cta = blockIdx.x;
  const long long u0 = unit_start(p.U, p.P, cta);
  const long long u1 = unit_start(p.U, p.P, cta + 1);
  const int nstages = static_cast<int>(u1 - u0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full_w[s], 1);
      mbar_init(&sm.full_x[s], 32);
      mbar_init(&sm.empty[s], 32 * (kConsumerWarps + 1));  // consumers + the stage's prep warp
    }
    mbar_init(&sm.group_bar, 32 * kConsumerWarps);
    fence_barrier_init();
  }
  __syncthreads();

  // Metadata tile geometry (TMA path).
  //   INT4:  scales and zeros [N, G] fp16, box 8 groups x 256 rows at x = (2j) & ~7.
  //   MXFP4: E8M0 [N, K/32] bytes, box 16 bytes x 256 rows at x = (8j) & ~15.
  constexpr int kMetaBytes = (FMT == kInt4G128) ? 2 * kBand * 16 : kBand * 16;

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
      int i = 0;
      for (; i < nstages; ++i, st.next()) {
        const int slot = i % kStages;
        const uint32_t ph = (i / kStages) & 1;
        if (!mbar_wait(&sm.empty[slot], ph ^ 1, &g_gemv_err, kErrWaitEmpty)) break;
        const uint32_t bytes = kTileBytes + MT * 512 + (p.meta_tma ? kMetaBytes : 0);
        mbar_arrive_expect_tx(&sm.full_w[slot], bytes);
        tma_load_2d(&sm.w[slot][0], &tmap_w, st.j * 128, st.band * kBand, &sm.full_w[slot], pol_w);
        tma_load_2d(&sm.xraw[slot][0], &tmap_x, st.j * 256, 0, &sm.full_w[slot], pol_m);
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
      for (int jj = i - kStages; jj < i; ++jj) {  // drain: the last fill of every slot landed
        if (jj < 0) continue;
        mbar_wait(&sm.full_w[jj % kStages], (jj / kStages) & 1, &g_gemv_err, kErrDrain);
      }
    }
  } else if (warp < kFirstConsumer) {
    // ------------------------------------------------------------------ prep
    const int pw = warp - 1;
    const int t = lane & 3;
    Cursor st;
    st.init(u0, u1, p.GP, p.G);
    for (int q = 0; q < pw; ++q) st.next();
    for (int i = pw; i < nstages; i += kPrepWarps) {
      const int slot = i % kStages;
      const uint32_t ph = (i / kStages) & 1;
      // (1) activations of the stage: the raw tile came by TMA with the stage's weights (rows
      //     >= M and columns >= K zero-filled), so this is shared memory to shared memory.
      if (!mbar_wait(&sm.full_w[slot], ph, &g_gemv_err, kErrWaitFull)) break;
      const uint8_t* xr = &sm.xraw[slot][0];
      if constexpr (FMT == kInt4G128) {
        uint4 r[NT][2][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int m = (lane >> 2) + 8 * nt;
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int v = 0; v < 4; ++v)
              r[nt][h][v] = (m < p.M) ? *reinterpret_cast<const uint4*>(xr + m * 512 + 256 * h + 64 * t + 16 * v)
                                      : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int m = (lane >> 2) + 8 * nt;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float sum = 0.f;
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const uint4 x = r[nt][h][v];
              // (x0,x4) (x1,x5) (x2,x6) (x3,x7): the k order of the unpacked nibble pairs.
              uint4 o;
              o.x = prmt(x.x, x.z, 0x5410);
              o.y = prmt(x.x, x.z, 0x7632);
              o.z = prmt(x.y, x.w, 0x5410);
              o.w = prmt(x.y, x.w, 0x7632);
              sm.x[slot][nt][h][v][lane] = o;
              const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
              for (int q = 0; q < 4; ++q) sum += __uint_as_float(w4[q] << 16) + __uint_as_float(w4[q] & 0xffff0000u);
            }
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);
            if (t == 0) sm.xsum[slot][h][m] = sum;
          }
        }
      } else {
        uint4 raw[NT][2][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int m = (lane >> 2) + 8 * nt;
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int blk = 0; blk < 4; ++blk)
              raw[nt][h][blk] = (m < p.M) ? *reinterpret_cast<const uint4*>(xr + m * 512 + 256 * h + 64 * blk + 16 * t)
                                          : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int m = (lane >> 2) + 8 * nt;
          // fp16 operands; row scale 2^-k keeps |x| 2^-k < 2^15 (k >= 0).
          uint32_t mx = 0u;  // max |x| bit pattern (bf16 magnitudes order like integers)
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int blk = 0; blk < 4; ++blk) {
              const uint4 x = raw[nt][h][blk];
              const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
              for (int q = 0; q < 4; ++q) mx = max(mx, max(w4[q] & 0x7fffu, (w4[q] >> 16) & 0x7fffu));
            }
          mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
          mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
          const int ex = static_cast<int>(mx >> 7) - 127;        // floor(log2 max) for normals
          const int k = (mx >= 0x7f80u) ? 0 : max(0, ex - 14);   // inf/nan: no scaling
          const float inv = __uint_as_float(static_cast<uint32_t>(127 - k) << 23);
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int blk = 0; blk < 4; ++blk) {
              const uint4 x = raw[nt][h][blk];
              const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
              uint32_t o[4];
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                __half2 hh = __floats2half2_rn(__uint_as_float(w4[q] << 16) * inv,
                                               __uint_as_float(w4[q] & 0xffff0000u) * inv);
                o[q] = *reinterpret_cast<uint32_t*>(&hh);
              }
              sm.x[slot][nt][h][blk][lane] = make_uint4(o[0], o[1], o[2], o[3]);
            }
          if (t == 0) sm.xf[slot][m] = __uint_as_float(static_cast<uint32_t>(127 + k) << 23);
        }
      }
      // (2) per-row metadata of the stage: lane handles rows lane + 32 q
      bool ok = true;
      {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int r = lane + 32 * q;
          const int row = st.band * kBand + r;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const bool live = (row < p.N) && (h < st.ng());
            float2 m2 = make_float2(0.f, 0.f);
            if constexpr (FMT == kInt4G128) {
              uint32_t sb = 0u, zb = 0u;
              if (p.meta_tma) {
                const int col = ((2 * st.j) & 7) + h;
                sb = reinterpret_cast<const uint16_t*>(&sm.mraw[slot][0])[r * 8 + col];
                zb = reinterpret_cast<const uint16_t*>(&sm.mraw[slot][kBand * 16])[r * 8 + col];
              } else if (live) {
                const long long idx = static_cast<long long>(row) * p.G + 2 * st.j + h;
                sb = __ldg(reinterpret_cast<const unsigned short*>(p.scales) + idx);
                zb = __ldg(p.zeros + idx);
              }
              const float s = live ? __half2float(__ushort_as_half(static_cast<unsigned short>(sb))) : 0.f;
              const float z = live ? __half2float(__ushort_as_half(static_cast<unsigned short>(zb))) : 0.f;
              m2.x = s;
              m2.y = -s * (128.f + z);
            } else {
              uint32_t v = 0u;
              if (p.meta_tma) {
                v = reinterpret_cast<const uint32_t*>(&sm.mraw[slot][0])[r * 4 + (((8 * st.j) & 15) >> 2) + h];
              } else if (live) {
                const uint8_t* E = reinterpret_cast<const uint8_t*>(p.scales) + static_cast<long long>(row) * p.KB;
                const int b0 = (2 * st.j + h) * 4;
#pragma unroll
                for (int q2 = 0; q2 < 4; ++q2)
                  if (b0 + q2 < p.KB) v |= static_cast<uint32_t>(__ldg(E + b0 + q2)) << (8 * q2);
              }
              m2.x = __uint_as_float(live ? v : 0u);
            }
            sm.meta[slot][h][r] = m2;
          }
        }
      }
      mbar_arrive(&sm.full_x[slot]);
      mbar_arrive(&sm.empty[slot]);   // this warp is done reading the slot's raw tiles
      if (!ok) break;
      for (int q = 0; q < kPrepWarps; ++q) st.next();
    }
  } else {
    // ------------------------------------------------------------------ consumers
    const int cw = warp - kFirstConsumer;
    const int g = lane >> 2;
    const int t = lane & 3;
    const int tid = threadIdx.x - 32 * kFirstConsumer;  // 0..511
    const int r0 = cw * kRowsPerWarp + frag_row(g);      // rows (inside the band) of this lane
    const int r1 = cw * kRowsPerWarp + frag_row(g + 8);

    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;

    uint32_t gphase = 0;  // phase parity of group_bar
    Cursor st;
    st.init(u0, u1, p.GP, p.G);
    for (int i = 0; i < nstages; ++i, st.next()) {
      const int slot = i % kStages;
      const uint32_t ph = (i / kStages) & 1;
      if (!mbar_wait(&sm.full_w[slot], ph, &g_gemv_err, kErrWaitFull)) break;
      if (!mbar_wait(&sm.full_x[slot], ph, &g_gemv_err, kErrWaitFull)) break;

      const uint8_t* wt = &sm.w[slot][0];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (h >= st.ng()) break;
        const float2 m0 = sm.meta[slot][h][r0];
        const float2 m1 = sm.meta[slot][h][r1];
        uint4 bx[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int v = 0; v < 4; ++v) bx[nt][v] = sm.x[slot][nt][h][v][lane];

        if constexpr (FMT == kInt4G128) {
          const int c = 4 * h + t;
          const uint4 wv0 = *reinterpret_cast<const uint4*>(wt + r0 * 128 + ((c ^ (r0 & 7)) << 4));
          const uint4 wv1 = *reinterpret_cast<const uint4*>(wt + r1 * 128 + ((c ^ (r1 & 7)) << 4));
          const uint32_t w0[4] = {wv0.x, wv0.y, wv0.z, wv0.w};
          const uint32_t w1[4] = {wv1.x, wv1.y, wv1.z, wv1.w};
          float ga[2][NT][4];  // two independent accumulation chains (even / odd words)
#pragma unroll
          for (int ch = 0; ch < 2; ++ch)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int e = 0; e < 4; ++e) ga[ch][nt][e] = 0.f;
#pragma unroll
          for (int jw = 0; jw < 4; ++jw) {
            // nibble pairs (s, s+4) as bf16 128 + q (exact); the zero point is folded below
            uint32_t pa[4], pb[4];
#pragma unroll
            for (int s = 0; s < 4; ++s) {
              pa[s] = lop3_and_or(w0[jw] >> (4 * s), 0x000f000fu, 0x43004300u);
              pb[s] = lop3_and_or(w1[jw] >> (4 * s), 0x000f000fu, 0x43004300u);
            }
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) {
                const uint4 bv = bx[nt][jw];
                mma_bf16(ga[jw & 1][nt], pa[2 * hh], pb[2 * hh], pa[2 * hh + 1], pb[2 * hh + 1], hh ? bv.z : bv.x,
                         hh ? bv.w : bv.y);
              }
          }
          // y += s * sum_k (128 + q) x + c * sum_k x,  c = -s (128 + z)   (zero-point cross term)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const float2 xs = *reinterpret_cast<const float2*>(&sm.xsum[slot][h][2 * t + 8 * nt]);
            acc[nt][0] = fmaf(m0.y, xs.x, fmaf(m0.x, ga[0][nt][0] + ga[1][nt][0], acc[nt][0]));
            acc[nt][1] = fmaf(m0.y, xs.y, fmaf(m0.x, ga[0][nt][1] + ga[1][nt][1], acc[nt][1]));
            acc[nt][2] = fmaf(m1.y, xs.x, fmaf(m1.x, ga[0][nt][2] + ga[1][nt][2], acc[nt][2]));
            acc[nt][3] = fmaf(m1.y, xs.y, fmaf(m1.x, ga[0][nt][3] + ga[1][nt][3], acc[nt][3]));
          }
        } else {
          // MXFP4: lane t holds 8 codes of each 32-block; two k16 steps per block.
          const uint32_t e0 = __float_as_uint(m0.x), e1 = __float_as_uint(m1.x);
          float sacc[NT][4];
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) sacc[nt][e] = 0.f;
#pragma unroll
          for (int blk = 0; blk < 4; ++blk) {
            const int c = 4 * h + blk;
            const uint32_t wr0 = *reinterpret_cast<const uint32_t*>(wt + r0 * 128 + ((c ^ (r0 & 7)) << 4) + 4 * t);
            const uint32_t wr1 = *reinterpret_cast<const uint32_t*>(wt + r1 * 128 + ((c ^ (r1 & 7)) << 4) + 4 * t);
            float bacc[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int e = 0; e < 4; ++e) bacc[nt][e] = 0.f;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const uint32_t a0 = e2m1x2_to_f16x2((wr0 >> (16 * hh)) & 0xffu);
              const uint32_t a2 = e2m1x2_to_f16x2((wr0 >> (16 * hh + 8)) & 0xffu);
              const uint32_t a1 = e2m1x2_to_f16x2((wr1 >> (16 * hh)) & 0xffu);
              const uint32_t a3 = e2m1x2_to_f16x2((wr1 >> (16 * hh + 8)) & 0xffu);
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) {
                const uint4 bv = bx[nt][blk];
                mma_f16(bacc[nt], a0, a1, a2, a3, hh ? bv.z : bv.x, hh ? bv.w : bv.y);
              }
            }
            const float f0 = e8m0_to_f32((e0 >> (8 * blk)) & 0xffu);
            const float f1 = e8m0_to_f32((e1 >> (8 * blk)) & 0xffu);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              sacc[nt][0] = fmaf(f0, bacc[nt][0], sacc[nt][0]);
              sacc[nt][1] = fmaf(f0, bacc[nt][1], sacc[nt][1]);
              sacc[nt][2] = fmaf(f1, bacc[nt][2], sacc[nt][2]);
              sacc[nt][3] = fmaf(f1, bacc[nt][3], sacc[nt][3]);
            }
          }
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const float2 xf = *reinterpret_cast<const float2*>(&sm.xf[slot][2 * t + 8 * nt]);
            acc[nt][0] = fmaf(xf.x, sacc[nt][0], acc[nt][0]);
            acc[nt][1] = fmaf(xf.y, sacc[nt][1], acc[nt][1]);
            acc[nt][2] = fmaf(xf.x, sacc[nt][2], acc[nt][2]);
            acc[nt][3] = fmaf(xf.y, sacc[nt][3], acc[nt][3]);
          }
        }
      }
      __syncwarp();
      mbar_arrive(&sm.empty[slot]);

      if (st.seg_last()) {
        const int band = st.band;
        const bool full = (st.seg_start == static_cast<long long>(band) * p.GP) &&
                          (st.seg_end == static_cast<long long>(band + 1) * p.GP);
        if (full) {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int m = 2 * t + (e & 1) + 8 * nt;
              const int n = band * kBand + ((e >> 1) ? r1 : r0);
              if (m < p.M && n < p.N)
                p.Y[static_cast<long long>(m) * p.N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[nt][e]));
            }
        } else {
          const int side = (u0 >= static_cast<long long>(band) * p.GP) ? 0 : 1;
          float* slotp = p.part + (static_cast<long long>(cta) * 2 + side) * MT * kBand;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int m = 2 * t + (e & 1) + 8 * nt;
              __stcg(slotp + m * kBand + ((e >> 1) ? r1 : r0), acc[nt][e]);
            }
          __threadfence();
          mbar_arrive(&sm.group_bar);
          if (!mbar_wait(&sm.group_bar, gphase, &g_gemv_err, kErrWaitReduce)) break;
          gphase ^= 1u;
          if (tid == 0) {
            const uint32_t mine = static_cast<uint32_t>(st.seg_end - st.seg_start);
            const uint32_t old = atomicAdd(p.cnt + band, mine);
            sm.reduce_flag = (old + mine == static_cast<uint32_t>(p.GP)) ? 1 : 0;
          }
          mbar_arrive(&sm.group_bar);
          if (!mbar_wait(&sm.group_bar, gphase, &g_gemv_err, kErrWaitReduce)) break;
          gphase ^= 1u;
          if (sm.reduce_flag) {
            __threadfence();
            // Contributors: CTAs whose unit range meets this band, summed in CTA order.  CTA
            // c_lo holds the band's first unit; every later contributor starts inside the band
            // (partial slot 0), c_lo uses slot 1 when its range started in an earlier band.
            const long long bs = static_cast<long long>(band) * p.GP, be = bs + p.GP;
            int c_lo = static_cast<int>((bs * p.P) / p.U);
            while (c_lo > 0 && unit_start(p.U, p.P, c_lo) > bs) --c_lo;
            while (unit_start(p.U, p.P, c_lo + 1) <= bs) ++c_lo;
            int c_hi = static_cast<int>(((be - 1) * p.P) / p.U);
            while (c_hi > c_lo && unit_start(p.U, p.P, c_hi) > be - 1) --c_hi;
            while (c_hi + 1 < p.P && unit_start(p.U, p.P, c_hi + 1) <= be - 1) ++c_hi;
            const int lo_side = unit_start(p.U, p.P, c_lo) < bs ? 1 : 0;
            const int r = tid & (kBand - 1);
            const int n = band * kBand + r;
            for (int m = tid >> 8; m < p.M; m += 2) {
              float sum = ld_cg_f32(p.part + (static_cast<long long>(c_lo) * 2 + lo_side) * MT * kBand + m * kBand + r);
              for (int c = c_lo + 1; c <= c_hi; ++c)
                sum += ld_cg_f32(p.part + static_cast<long long>(c) * 2 * MT * kBand + m * kBand + r);
              if (n < p.N) p.Y[static_cast<long long>(m) * p.N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(sum));
            }
            if (tid == 0) atomicExch(p.cnt + band, 0u);
          }
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
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

template <int FMT, int MT>
static cudaError_t launch_gemv_t(const CUtensorMap& tw, const CUtensorMap& ts, const CUtensorMap& tz,
                                 const gemv::Params& p, cudaStream_t stream) {
  // activations: MT rows x 256 k per stage; rows >= M and columns >= K come back as zeros
  CUtensorMap tx;
  cudaError_t ex = make_tmap_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.X, static_cast<uint64_t>(p.K),
                                static_cast<uint64_t>(p.M), static_cast<uint64_t>(p.K) * 2, 256, MT,
                                CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
  if (ex != cudaSuccess) return ex;
  using S = gemv::Smem<FMT, MT>;
  const size_t smem = sizeof(S) + 1024;
  auto kern = gemv::k_gemv<FMT, MT>;
  static bool attr_set[64] = {false};  // once per device
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  kern<<<p.P, gemv::kThreads, smem, stream>>>(tw, ts, tz, tx, p);
  return cudaGetLastError();
}

cudaError_t launch_gemv_mma(int fmt, const uint16_t* X, int64_t M, int64_t K, int64_t N, const int32_t* Wq,
                            const void* scales, const uint16_t* zeros, uint16_t* Y, void* ws, size_t ws_bytes,
                            cudaStream_t stream) {
  gemv::Params p{};
  p.X = X;
  p.scales = scales;
  p.zeros = zeros;
  p.Y = Y;
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
  // of 16 bytes (INT4: K % 1024 == 0; MXFP4: K % 512 == 0); otherwise the prep warps gather
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
  if (fmt == kInt4G128)
    return small ? launch_gemv_t<kInt4G128, 8>(tw, ts, tz, p, stream) : launch_gemv_t<kInt4G128, 16>(tw, ts, tz, p, stream);
  return small ? launch_gemv_t<kMxfp4, 8>(tw, ts, tz, p, stream) : launch_gemv_t<kMxfp4, 16>(tw, ts, tz, p, stream);
}

// The decode entry points run the mma.sync kernel above.  The tcgen05 decode kernel
// (gemv_tc.cu) is kept for comparison: at N = 16 a tcgen05.mma costs ~56 cycles per
// 128 x 16 x 16 instruction, which caps it below HBM speed on this shape.
size_t gemv_workspace_bytes(int fmt, int64_t M, int64_t K, int64_t N) { return gemv_mma_workspace_bytes(fmt, M, K, N); }

cudaError_t launch_gemv(int fmt, const uint16_t* X, int64_t M, int64_t K, int64_t N, const int32_t* Wq,
                        const void* scales, const uint16_t* zeros, uint16_t* Y, void* ws, size_t ws_bytes,
                        cudaStream_t stream) {
  return launch_gemv_mma(fmt, X, M, K, N, Wq, scales, zeros, Y, ws, ws_bytes, stream);
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
  // Set-up, once per device with that device current: the array's name is only a host-side
  // handle, so the kernel gets the device address from cudaGetSymbolAddress.
  static std::mutex mu;
  static void* addr[64] = {nullptr};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (!addr[dev]) {
      void* a = nullptr;
      e = cudaGetSymbolAddress(&a, g_noalloc_scratch);
      if (e != cudaSuccess) return e;
      addr[dev] = a;
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
