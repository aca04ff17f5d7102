// Decode kernel (M <= 16): Y[M, N] = X[M, K] * dequant(Wq)^T.
//
// Bandwidth-bound (推理优化与量化算子深度技术调研 §1.3: at batch 1 the W4A16 GEMV is limited by
// HBM bandwidth; 第 1 章：推理加速全景 §1.2-1.3: decode arithmetic intensity ~1 FLOP/B), so the
// design goal is to stream the 0.53125 B/weight of packed weights + metadata once, at full
// HBM bandwidth, with the arithmetic hidden underneath.
//
// Structure (one persistent CTA per SM, warp-specialised):
//   warp 0      TMA producer: 256-row x 128-byte tiles of the packed weights (two 128-k
//               groups of INT4 / 256 k of MXFP4), SWIZZLE_128B, into a 4-stage smem ring.
//   warps 1-2   prep (stage i by prep warp i % 2): the activations of the stage's k-range in
//               the exact order of the mma.sync B fragments (MXFP4: converted to fp16 with a
//               per-row power-of-two scale that keeps every value in fp16 range), plus the
//               scales / zero points (INT4) or E8M0 bytes (MXFP4) of the stage's rows.  The
//               consumers then touch only shared memory in their main loop.
//   warps 3-10  consumers: 32 weight rows each; unpack nibbles in registers, tensor-core
//               mma.sync with fp32 accumulation, group scale applied in fp32 afterwards.
//
// Exactness: the tensor-core operands are exact small integers (INT4: q - z in bf16) or
// exact E2M1 values (MXFP4, fp16); every product is exact and the per-group (INT4) or
// per-32 (MXFP4) power-of-two/fp16 scale is applied to the fp32 partial sum.  No operand
// is rounded to 16 bits, which keeps the layer within 1e-2 (1 + |y|) of the float64 oracle
// at every K (a bf16-rounded dequantised weight would not).  The zero point enters through
// (q - z), the cross term 第 6 课：量化源码走读 §3 warns must not be dropped.
//
// Work split: the (256-row band, 128-k group) units are split evenly over the CTAs in
// band-major order.  A band covered by one CTA is written directly as bf16; a band shared
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

constexpr int kConsumerWarps = 8;
constexpr int kBand = 32 * kConsumerWarps;          // weight rows per CTA tile
constexpr int kStages = 4;
constexpr int kTileBytes = kBand * 128;              // 32 KB of packed weights per stage
constexpr int kPrepWarps = 2;                        // stage i is prepared by prep warp i % 2
constexpr int kFirstConsumer = 1 + kPrepWarps;       // warp index of the first consumer
constexpr int kThreads = 32 * (kFirstConsumer + kConsumerWarps);  // 352
constexpr int kGroupK = 128;                         // k per unit (one INT4 group)

struct Params {
  const uint16_t* X;
  const void* scales;
  const uint16_t* zeros;
  uint16_t* Y;
  float* part;        // [P][2][MT][kBand] fp32 partials
  uint32_t* cnt;      // [bands] counters
  int M, K, N;
  int G;              // units (128-k groups) per row
  int KB;             // MXFP4: scale bytes per row (K / 32)
  int bands;
  long long U;        // bands * G
  int P;              // CTAs
};

// Fragment row f (0..15) of a 16-row tile -> row inside the tile.  Rows g and g+4 of a
// smem swizzle atom then land in disjoint bank groups, so the consumer's 128-bit loads
// are conflict-free.
__device__ __forceinline__ int frag_row(int f) { return (f & 8) | ((f >> 1) & 3) | ((f & 1) << 2); }

__device__ __forceinline__ long long unit_start(long long U, int P, int c) {
  return (U * c) / P;
}

// Iterator over the stages of one CTA's unit range: 1 or 2 units per stage, never crossing
// a band boundary.
struct StageIter {
  long long u, u0, u1;
  int G;
  __device__ void init(long long a, long long b, int g) { u = a; u0 = a; u1 = b; G = g; }
  __device__ bool done() const { return u >= u1; }
  __device__ int band() const { return static_cast<int>(u / G); }
  __device__ int g0() const { return static_cast<int>(u % G); }
  __device__ long long seg_end() const {
    long long be = (u / G + 1) * static_cast<long long>(G);
    return be < u1 ? be : u1;
  }
  __device__ int ng() const {
    long long r = seg_end() - u;
    return r >= 2 ? 2 : 1;
  }
  __device__ bool last_in_seg() const { return u + ng() == seg_end(); }
  __device__ long long seg_start() const {
    long long bs = (u / G) * static_cast<long long>(G);
    return bs > u0 ? bs : u0;
  }
  __device__ void next() { u += ng(); }
};

template <int FMT, int MT>
struct Smem {
  static constexpr int NT = MT / 8;
  static constexpr int kXBytes = NT * 2 * 4 * 32 * 16;  // [nt][group][vec][lane] uint4
  uint8_t w[kStages][kTileBytes];
  uint4 x[kStages][NT][2][4][32];
  float xf[kStages][MT];          // MXFP4: power-of-two factor per activation row
  // Per-row metadata of the stage's two groups, staged by the prep warps:
  //   INT4:  {scale as float, bf16x2 (128 + z) bits}    MXFP4: {four E8M0 bytes, unused}
  float2 meta[kStages][2][kBand];
  uint64_t full_w[kStages];
  uint64_t full_x[kStages];
  uint64_t empty[kStages];
  uint64_t group_bar;             // consumer-warp barrier (bounded wait) for the split-K path
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

__device__ __forceinline__ uint32_t bsub2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
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

template <int FMT, int MT>
__global__ void __launch_bounds__(kThreads, 1)
    k_gemv(const __grid_constant__ CUtensorMap tmap_w, const Params p) {
  using S = Smem<FMT, MT>;
  constexpr int NT = MT / 8;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  S& sm = *reinterpret_cast<S*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int cta = blockIdx.x;
  const long long u0 = unit_start(p.U, p.P, cta);
  const long long u1 = unit_start(p.U, p.P, cta + 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full_w[s], 1);
      mbar_init(&sm.full_x[s], 32);
      mbar_init(&sm.empty[s], 32 * kConsumerWarps);
    }
    mbar_init(&sm.group_bar, 32 * kConsumerWarps);
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmap_w);
      const uint64_t pol = l2_policy_evict_first();
      StageIter it;
      it.init(u0, u1, p.G);
      int i = 0;
      bool ok = true;
      for (; !it.done(); it.next(), ++i) {
        const int slot = i % kStages;
        const uint32_t ph = (i / kStages) & 1;
        if (!mbar_wait(&sm.empty[slot], ph ^ 1, &g_gemv_err, kErrWaitEmpty)) { ok = false; break; }
        mbar_arrive_expect_tx(&sm.full_w[slot], kTileBytes);
        tma_load_2d(&sm.w[slot][0], &tmap_w, it.g0() * 64, it.band() * kBand, &sm.full_w[slot], pol);
      }
      // Drain: the last fill of every slot must have landed before the CTA may exit.
      const int issued = i;
      for (int j = issued - kStages; j < issued; ++j) {
        if (j < 0) continue;
        const int slot = j % kStages;
        const uint32_t ph = (j / kStages) & 1;
        mbar_wait(&sm.full_w[slot], ph, &g_gemv_err, kErrDrain);
      }
      (void)ok;
    }
  } else if (warp < kFirstConsumer) {
    // ------------------------------------------------------------------ prep
    const int pw = warp - 1;
    StageIter it;
    it.init(u0, u1, p.G);
    const int t = lane & 3;
    for (int i = 0; !it.done(); it.next(), ++i) {
      if (i % kPrepWarps != pw) continue;
      const int slot = i % kStages;
      const uint32_t ph = (i / kStages) & 1;
      if (!mbar_wait(&sm.empty[slot], ph ^ 1, &g_gemv_err, kErrWaitEmpty)) break;
      const int ng = it.ng();
      const int g0 = it.g0();
      const int band = it.band();
      // metadata of the stage's rows: lane handles rows lane + 32 q
      {
        uint32_t ma[8][2], mb[8][2];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int row = band * kBand + lane + 32 * q;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const bool live = (row < p.N) && (h < ng);
            if constexpr (FMT == kInt4G128) {
              const long long idx = static_cast<long long>(row) * p.G + g0 + h;
              ma[q][h] = live ? __ldg(reinterpret_cast<const unsigned short*>(p.scales) + idx) : 0u;
              mb[q][h] = live ? __ldg(reinterpret_cast<const unsigned short*>(p.zeros) + idx) : 0u;
            } else {
              const uint8_t* E = reinterpret_cast<const uint8_t*>(p.scales) + static_cast<long long>(row) * p.KB;
              const int b0 = (g0 + h) * 4;
              uint32_t v = 0u;
              if (live) {
                if ((p.KB & 3) == 0) {
                  v = __ldg(reinterpret_cast<const uint32_t*>(E + b0));
                } else {
#pragma unroll
                  for (int q2 = 0; q2 < 4; ++q2)
                    if (b0 + q2 < p.KB) v |= static_cast<uint32_t>(__ldg(E + b0 + q2)) << (8 * q2);
                }
              }
              ma[q][h] = v;
              mb[q][h] = 0u;
            }
          }
        }
#pragma unroll
        for (int q = 0; q < 8; ++q)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float2 m2;
            if constexpr (FMT == kInt4G128) {
              m2.x = __half2float(__ushort_as_half(static_cast<unsigned short>(ma[q][h])));
              const float z = __half2float(__ushort_as_half(static_cast<unsigned short>(mb[q][h])));
              const uint32_t zb = __bfloat16_as_ushort(__float2bfloat16_rn(128.f + z));
              m2.y = __uint_as_float(zb | (zb << 16));
            } else {
              m2.x = __uint_as_float(ma[q][h]);
              m2.y = 0.f;
            }
            sm.meta[slot][h][lane + 32 * q] = m2;
          }
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int m = (lane >> 2) + 8 * nt;
        if constexpr (FMT == kInt4G128) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int kbase = (g0 + h) * kGroupK + 32 * t;
            const bool live = (m < p.M) && (h < ng);
            const uint4* src = reinterpret_cast<const uint4*>(p.X + static_cast<long long>(m) * p.K + kbase);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint4 r = live ? __ldg(src + v) : make_uint4(0u, 0u, 0u, 0u);
              // (x0,x4) (x1,x5) (x2,x6) (x3,x7): the k order of the unpacked nibble pairs.
              uint4 o;
              o.x = prmt(r.x, r.z, 0x5410);
              o.y = prmt(r.x, r.z, 0x7632);
              o.z = prmt(r.y, r.w, 0x5410);
              o.w = prmt(r.y, r.w, 0x7632);
              sm.x[slot][nt][h][v][lane] = o;
            }
          }
        } else {
          // MXFP4: fp16 operands.  Row scale 2^-k so that |x| * 2^-k < 2^15 (k >= 0).
          uint4 raw[2][4];
          uint32_t mx = 0u;  // max |x| bit pattern (bf16 magnitudes order like integers)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int blk = 0; blk < 4; ++blk) {
              const int kbase = (g0 + h) * kGroupK + 32 * blk + 8 * t;
              const bool live = (m < p.M) && (h < ng) && (kbase < p.K);
              uint4 r = live ? __ldg(reinterpret_cast<const uint4*>(p.X + static_cast<long long>(m) * p.K + kbase))
                             : make_uint4(0u, 0u, 0u, 0u);
              raw[h][blk] = r;
              const uint32_t w4[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                mx = max(mx, w4[q] & 0x7fffu);
                mx = max(mx, (w4[q] >> 16) & 0x7fffu);
              }
            }
          }
          mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
          mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
          const int ex = static_cast<int>(mx >> 7) - 127;        // floor(log2 max) for normals
          int k = (mx >= 0x7f80u) ? 0 : max(0, ex - 14);         // inf/nan: no scaling
          const float inv = __uint_as_float(static_cast<uint32_t>(127 - k) << 23);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int blk = 0; blk < 4; ++blk) {
              const uint4 r = raw[h][blk];
              const uint32_t w4[4] = {r.x, r.y, r.z, r.w};
              uint32_t o[4];
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const float lo = __uint_as_float(w4[q] << 16) * inv;
                const float hi = __uint_as_float(w4[q] & 0xffff0000u) * inv;
                __half2 hh = __floats2half2_rn(lo, hi);
                o[q] = *reinterpret_cast<uint32_t*>(&hh);
              }
              sm.x[slot][nt][h][blk][lane] = make_uint4(o[0], o[1], o[2], o[3]);
            }
          }
          if (t == 0) sm.xf[slot][m] = __uint_as_float(static_cast<uint32_t>(127 + k) << 23);
        }
      }
      mbar_arrive(&sm.full_x[slot]);
    }
  } else {
    // ------------------------------------------------------------------ consumers
    const int cw = warp - kFirstConsumer;
    const int g = lane >> 2;
    const int t = lane & 3;
    const int tid = threadIdx.x - 32 * kFirstConsumer;  // 0..255
    // Rows (inside the band) of this lane: [row-tile][fragment half]
    int rrow[2][2];
#pragma unroll
    for (int rt = 0; rt < 2; ++rt)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) rrow[rt][hf] = cw * 32 + rt * 16 + frag_row(g + 8 * hf);

    float acc[2][NT][4];
#pragma unroll
    for (int rt = 0; rt < 2; ++rt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[rt][nt][e] = 0.f;

    StageIter it;
    it.init(u0, u1, p.G);
    bool aborted = false;
    uint32_t gphase = 0;  // phase parity of group_bar
    for (int i = 0; !it.done(); it.next(), ++i) {
      const int slot = i % kStages;
      const uint32_t ph = (i / kStages) & 1;
      const int band = it.band();
      const int g0 = it.g0();
      const int ng = it.ng();

      if (!mbar_wait(&sm.full_w[slot], ph, &g_gemv_err, kErrWaitFull)) { aborted = true; break; }
      if (!mbar_wait(&sm.full_x[slot], ph, &g_gemv_err, kErrWaitFull)) { aborted = true; break; }

      // Scales / zero points (INT4) or E8M0 bytes (MXFP4) of this lane's rows, from smem.
      float sc[2][2][2];          // [h][rt][hf]
      uint32_t zz[2][2][2];       // INT4: bf16x2 (128 + z)
      uint32_t e8[2][2][2];       // MXFP4: four E8M0 bytes of the group
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int rt = 0; rt < 2; ++rt)
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const float2 m2 = sm.meta[slot][h][rrow[rt][hf]];
            sc[h][rt][hf] = m2.x;
            zz[h][rt][hf] = __float_as_uint(m2.y);
            e8[h][rt][hf] = __float_as_uint(m2.x);
          }

      const uint8_t* wt = &sm.w[slot][0];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (h >= ng) break;
        uint4 bx[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int v = 0; v < 4; ++v) bx[nt][v] = sm.x[slot][nt][h][v][lane];

#pragma unroll
        for (int rt = 0; rt < 2; ++rt) {
          if constexpr (FMT == kInt4G128) {
            uint4 wv[2];
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
              const int r = rrow[rt][hf];
              const int c = 4 * h + t;
              wv[hf] = *reinterpret_cast<const uint4*>(wt + r * 128 + ((c ^ (r & 7)) << 4));
            }
            float gacc[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int e = 0; e < 4; ++e) gacc[nt][e] = 0.f;
            const uint32_t w0[4] = {wv[0].x, wv[0].y, wv[0].z, wv[0].w};
            const uint32_t w1[4] = {wv[1].x, wv[1].y, wv[1].z, wv[1].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              // nibble pairs (s, s+4) as bf16 128+q, then minus (128+z): exact (q - z)
              uint32_t pa[4], pb[4];
#pragma unroll
              for (int s = 0; s < 4; ++s) {
                pa[s] = bsub2(lop3_and_or(w0[j] >> (4 * s), 0x000f000fu, 0x43004300u), zz[h][rt][0]);
                pb[s] = bsub2(lop3_and_or(w1[j] >> (4 * s), 0x000f000fu, 0x43004300u), zz[h][rt][1]);
              }
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                  const uint4 bv = bx[nt][j];
                  mma_bf16(gacc[nt], pa[2 * hh], pb[2 * hh], pa[2 * hh + 1], pb[2 * hh + 1], hh ? bv.z : bv.x,
                           hh ? bv.w : bv.y);
                }
              }
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              acc[rt][nt][0] = fmaf(sc[h][rt][0], gacc[nt][0], acc[rt][nt][0]);
              acc[rt][nt][1] = fmaf(sc[h][rt][0], gacc[nt][1], acc[rt][nt][1]);
              acc[rt][nt][2] = fmaf(sc[h][rt][1], gacc[nt][2], acc[rt][nt][2]);
              acc[rt][nt][3] = fmaf(sc[h][rt][1], gacc[nt][3], acc[rt][nt][3]);
            }
          } else {
            // MXFP4: lane t holds 8 codes of each 32-block; two k16 steps per block.
            float sacc[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int e = 0; e < 4; ++e) sacc[nt][e] = 0.f;
#pragma unroll
            for (int blk = 0; blk < 4; ++blk) {
              uint32_t wr[2];
#pragma unroll
              for (int hf = 0; hf < 2; ++hf) {
                const int r = rrow[rt][hf];
                const int c = 4 * h + blk;
                wr[hf] = *reinterpret_cast<const uint32_t*>(wt + r * 128 + ((c ^ (r & 7)) << 4) + 4 * t);
              }
              float bacc[NT][4];
#pragma unroll
              for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) bacc[nt][e] = 0.f;
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                const uint32_t a0 = e2m1x2_to_f16x2((wr[0] >> (16 * hh)) & 0xffu);
                const uint32_t a2 = e2m1x2_to_f16x2((wr[0] >> (16 * hh + 8)) & 0xffu);
                const uint32_t a1 = e2m1x2_to_f16x2((wr[1] >> (16 * hh)) & 0xffu);
                const uint32_t a3 = e2m1x2_to_f16x2((wr[1] >> (16 * hh + 8)) & 0xffu);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                  const uint4 bv = bx[nt][blk];
                  const uint32_t b0r = hh ? bv.z : bv.x;
                  const uint32_t b1r = hh ? bv.w : bv.y;
                  mma_f16(bacc[nt], a0, a1, a2, a3, b0r, b1r);
                }
              }
              const float f0 = e8m0_to_f32((e8[h][rt][0] >> (8 * blk)) & 0xffu);
              const float f1 = e8m0_to_f32((e8[h][rt][1] >> (8 * blk)) & 0xffu);
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
              const float x0 = sm.xf[slot][2 * t + 8 * nt];
              const float x1 = sm.xf[slot][2 * t + 1 + 8 * nt];
              acc[rt][nt][0] = fmaf(x0, sacc[nt][0], acc[rt][nt][0]);
              acc[rt][nt][1] = fmaf(x1, sacc[nt][1], acc[rt][nt][1]);
              acc[rt][nt][2] = fmaf(x0, sacc[nt][2], acc[rt][nt][2]);
              acc[rt][nt][3] = fmaf(x1, sacc[nt][3], acc[rt][nt][3]);
            }
          }
        }
      }
      __syncwarp();
      mbar_arrive(&sm.empty[slot]);

      if (it.last_in_seg()) {
        const long long ss = it.seg_start();
        const long long se = it.seg_end();
        const bool full = (ss == static_cast<long long>(band) * p.G) && (se == static_cast<long long>(band + 1) * p.G);
        if (full) {
#pragma unroll
          for (int rt = 0; rt < 2; ++rt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int m = 2 * t + (e & 1) + 8 * nt;
                const int n = band * kBand + rrow[rt][e >> 1];
                if (m < p.M && n < p.N)
                  p.Y[static_cast<long long>(m) * p.N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[rt][nt][e]));
              }
        } else {
          const int side = (static_cast<int>(u0 / p.G) == band) ? 0 : 1;
          float* slotp = p.part + (static_cast<long long>(cta) * 2 + side) * MT * kBand;
#pragma unroll
          for (int rt = 0; rt < 2; ++rt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int m = 2 * t + (e & 1) + 8 * nt;
                __stcg(slotp + m * kBand + rrow[rt][e >> 1], acc[rt][nt][e]);
              }
          __threadfence();
          mbar_arrive(&sm.group_bar);
          if (!mbar_wait(&sm.group_bar, gphase, &g_gemv_err, kErrWaitReduce)) { aborted = true; break; }
          gphase ^= 1u;
          if (tid == 0) {
            const uint32_t mine = static_cast<uint32_t>(se - ss);
            const uint32_t old = atomicAdd(p.cnt + band, mine);
            sm.reduce_flag = (old + mine == static_cast<uint32_t>(p.G)) ? 1 : 0;
          }
          mbar_arrive(&sm.group_bar);
          if (!mbar_wait(&sm.group_bar, gphase, &g_gemv_err, kErrWaitReduce)) { aborted = true; break; }
          gphase ^= 1u;
          if (sm.reduce_flag) {
            __threadfence();
            // Contributors: CTAs whose unit range meets this band, in CTA order.
            const long long bs = static_cast<long long>(band) * p.G, be = bs + p.G;
            int c_lo = static_cast<int>((bs * p.P) / p.U);
            while (c_lo > 0 && unit_start(p.U, p.P, c_lo) > bs) --c_lo;
            while (unit_start(p.U, p.P, c_lo + 1) <= bs) ++c_lo;
            const int r = tid;  // one band row per consumer thread
            const int n = band * kBand + r;
            for (int m = 0; m < p.M; ++m) {
              float sum = 0.f;
              for (int c = c_lo; c < p.P && unit_start(p.U, p.P, c) < be; ++c) {
                const int cs = (static_cast<int>(unit_start(p.U, p.P, c) / p.G) == band) ? 0 : 1;
                sum += ld_cg_f32(p.part + (static_cast<long long>(c) * 2 + cs) * MT * kBand + m * kBand + r);
              }
              if (n < p.N) p.Y[static_cast<long long>(m) * p.N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(sum));
            }
            if (tid == 0) atomicExch(p.cnt + band, 0u);
          }
        }
#pragma unroll
        for (int rt = 0; rt < 2; ++rt)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[rt][nt][e] = 0.f;
      }
    }
    (void)aborted;
  }
}

int num_ctas(long long U) {
  const long long sms = device_sm_count();
  return static_cast<int>(U < sms ? U : sms);
}

}  // namespace gemv

size_t gemv_workspace_bytes(int fmt, int64_t M, int64_t K, int64_t N) {
  if (M < 1 || M > 16 || N < 1 || K < 1) return 0;
  const int MT = M <= 8 ? 8 : 16;
  const long long G = (K + gemv::kGroupK - 1) / gemv::kGroupK;
  const long long bands = (N + gemv::kBand - 1) / gemv::kBand;
  const int P = gemv::num_ctas(bands * G);
  (void)fmt;
  return kWsCounterBytes + static_cast<size_t>(P) * 2 * MT * gemv::kBand * sizeof(float);
}

template <int FMT, int MT>
static cudaError_t launch_gemv_t(const CUtensorMap& tmap, const gemv::Params& p, cudaStream_t stream) {
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
  kern<<<p.P, gemv::kThreads, smem, stream>>>(tmap, p);
  return cudaGetLastError();
}

cudaError_t launch_gemv(int fmt, const uint16_t* X, int64_t M, int64_t K, int64_t N, const int32_t* Wq,
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
  p.KB = static_cast<int>(K / 32);
  p.bands = static_cast<int>((N + gemv::kBand - 1) / gemv::kBand);
  p.U = static_cast<long long>(p.bands) * p.G;
  p.P = gemv::num_ctas(p.U);
  if (p.bands > kWsMaxCounters) return cudaErrorInvalidValue;
  if (ws_bytes < gemv_workspace_bytes(fmt, M, K, N)) return cudaErrorInvalidValue;
  p.cnt = reinterpret_cast<uint32_t*>(ws);
  p.part = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ws) + kWsCounterBytes);

  CUtensorMap tmap;
  cudaError_t e = make_tmap_2d(&tmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, Wq, static_cast<uint64_t>(K / 2),
                               static_cast<uint64_t>(N), static_cast<uint64_t>(K / 2), 128, gemv::kBand,
                               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
  if (e != cudaSuccess) return e;
  const bool small = M <= 8;
  if (fmt == kInt4G128)
    return small ? launch_gemv_t<kInt4G128, 8>(tmap, p, stream) : launch_gemv_t<kInt4G128, 16>(tmap, p, stream);
  return small ? launch_gemv_t<kMxfp4, 8>(tmap, p, stream) : launch_gemv_t<kMxfp4, 16>(tmap, p, stream);
}

// ---------------------------------------------------------------------------------------
// The decode kernel for callers that cannot allocate device memory.
//
// The split-K scratch of the decode kernel (reduction counters and fp32 partial sums) lives
// here in one fixed, library-owned device array instead of a caller-provided workspace.  It
// is sized for every decode shape the kernel accepts (M <= 16, N <= 4194304) on a device with
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
