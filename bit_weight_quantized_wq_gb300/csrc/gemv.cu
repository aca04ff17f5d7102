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
//               activations of the stage's k-range, loaded straight from global memory (L2;
//               they are small and shared by every CTA) and written in the exact order of
//               the mma.sync B fragments, with their per-group sums (INT4) or converted to
//               fp16 with a per-row power-of-two scale that keeps every value in fp16 range
//               (MXFP4).  The activations do not depend on the weights, so this runs ahead
//               of the weight stream.
//   warps 4-19  consumers: 16 weight rows each; per-row metadata straight from its tile,
//               nibbles unpacked in registers, tensor-core mma.sync with fp32 accumulation,
//               group scale applied in fp32 afterwards.
//
// Exactness: the tensor-core operands are exact: the weights as small integers or E2M1
// values, the activations as bf16 or as fp16 after a power-of-two scale per stage and row;
// every product is exact and the per-group (INT4) or per-32 (MXFP4) scale is applied to the
// fp32 partial sum.  No operand is rounded to 16 bits, which keeps the layer within
// 1e-2 (1 + |y|) of the float64 oracle at every K (a bf16-rounded dequantised weight would
// not).  INT4 per group and output, the zero-point cross term of 第 6 课：量化源码走读 §3
// compensated with group sums of the activations instead of subtracting z from every weight:
//   up to 8 activation rows, fp16 1024 + q (1024 + 16 q for the odd nibble of a byte, one
//   shift saved per word; those activations carry 1/16), x' = x 2^-e, B' the B operand:
//     sum_k (q - z) s x = 2^e s (sum_k A' B' - 1024 sum_k B' - z sum_k x')
//   16 rows, bf16 128 + q and the raw activations:
//     sum_k (q - z) s x = s sum_k (128 + q) x - s (128 + z) sum_k x
//
// Work split: the (256-row band, 256-k group pair) units -- one per pipeline stage -- are
// split evenly over the CTAs in band-major order (the host computes each CTA's range).  A
// band covered by one CTA is written directly as bf16.  For a band shared by several CTAs
// (only a range's first and last band can be), each CTA posts its fp32 partial sums when its
// part of the band is done, and the band is reduced after the loops:
//   8-row tiles: by the CTA holding its first unit alone (its range ends inside the band, so
//     it gets there last; the others exit after posting);
//   16- and 32-row tiles, whose partial tiles are large: by all of its CTAs, each adding up
//     an equal share of the band's outputs.
// Either way the posted sums of the band's CTAs are added in CTA order (deterministic), the
// results written as bf16 and the words put back to 0 for the next call.  A posted value
// carries its own "written" mark (a word that is never 0, below), so a CTA waits on the
// partial sums themselves: no counter, fence or second read.  Every CTA posts all its
// partial sums before it waits for any, so the wait always ends as long as the band's CTAs
// get an SM (one CTA per SM, at most one CTA per SM launched; the wait is bounded).
#include <mutex>

#include "decode_util.cuh"
#include "internal.h"

namespace wq {

__device__ uint32_t g_gemv_err;

static void noalloc_scratch_reset();

uint32_t gemv_read_and_clear_error() {
  uint32_t v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, g_gemv_err, sizeof(v));
  cudaMemcpyToSymbol(g_gemv_err, &z, sizeof(z));
  // A reduction that gave up may leave posted partial sums behind (a contributor that came
  // later than the wait): the library-owned exchange area of the no-workspace entry point is
  // zeroed again here, as a caller zeroes its own workspace after such an error.
  if (v & kErrWaitReduce) noalloc_scratch_reset();
  return v;
}

namespace gemv {

using namespace dec;

constexpr int kConsumerWarps = 16;
constexpr int kRowsPerWarp = 16;                     // one m16 row tile per consumer warp
constexpr int kBand = kRowsPerWarp * kConsumerWarps;  // 256 weight rows per CTA tile
constexpr int kTileBytes = kBand * 128;              // 32 KB of packed weights per stage
constexpr int kPrepWarps = 3;                        // stage i is prepared by prep warp i % 3
// Activation-fragment ring depth: two slots per prep warp, one for 32- and 64-row tiles
// (whose fragments fill 16 and 32 KB a stage).
__host__ __device__ constexpr int x_stages(int mt) { return mt >= 32 ? kPrepWarps : 2 * kPrepWarps; }
// Each prep warp owns whole ring slots (x_stages % kPrepWarps == 0), so it waits on every phase
// of its slots' barriers in order; a parity wait two phases ahead would pass at once.
static_assert(x_stages(8) % kPrepWarps == 0 && x_stages(64) % kPrepWarps == 0, "prep warps must own whole ring slots");
constexpr int kFirstConsumer = 1 + kPrepWarps;       // warp index of the first consumer
constexpr int kThreads = 32 * (kFirstConsumer + kConsumerWarps);  // 640
constexpr int kGroupK = 128;                         // k per group (INT4 group; 4 MXFP4 blocks)
constexpr int kSmemLimit = 227 * 1024;               // dynamic shared memory per CTA
constexpr int kSmemReserve = 1024 + 512;             // alignment pad + barriers and flags
constexpr int kMaxCtas = 160;                        // CTAs per launch (one per SM, at most)
static_assert(kMaxCtas <= 256, "CTA indices are stored in bytes");

// Raw metadata tile(s) per weight stage: INT4 scales + zeros boxes of 8 groups x 256 rows
// (fp16); MXFP4 one box of 16 E8M0 bytes x 256 rows.
__host__ __device__ constexpr int meta_raw_bytes(int fmt) { return fmt == kInt4G128 ? 2 * kBand * 16 : kBand * 16; }
// One activation stage: B fragments + per-row group sums + per-row power-of-two factors.
__host__ __device__ constexpr int x_stage_bytes(int mt) { return (mt / 8) * 2 * 4 * 32 * 16 + 4 * mt * 4 + mt * 4; }
// Weight stages: as many as fit beside the activation ring (4 or 5).
__host__ __device__ constexpr int w_stages(int fmt, int mt) {
  return (kSmemLimit - kSmemReserve - x_stages(mt) * x_stage_bytes(mt)) / (kTileBytes + meta_raw_bytes(fmt)) > 6
             ? 6
             : (kSmemLimit - kSmemReserve - x_stages(mt) * x_stage_bytes(mt)) / (kTileBytes + meta_raw_bytes(fmt));
}

struct Params {
  const uint16_t* X;
  const void* scales;
  const uint16_t* zeros;
  uint16_t* Y;
  OutSplit split;     // EPI == kEpiSplit3: three output tensors by column range
  uint32_t* part;     // [2P][MT][kBand] tagged fp32 partial sums (0: not posted): tile c holds CTA c's
                      // first band when its range starts inside it, tile P + c its last band when
                      // it holds that band's first unit
  int M, K, N;
  int G;              // 128-k groups per row (ceil(K / 128))
  int GP;             // group pairs per row (ceil(G / 2)) -- one pair per stage
  int KB;             // MXFP4: scale bytes per row (K / 32)
  int bands;
  int U;              // bands * GP units (one unit = one stage)
  int P;              // CTAs
  int meta_tma;       // 1: metadata tiles arrive by TMA with the weights; 0: consumers gather them
  int ustart[kMaxCtas + 1];   // CTA c owns units [ustart[c], ustart[c + 1])
  // The CTAs holding the first and the last unit of CTA c's first band, and the last unit of
  // its last band (the host's answer, so no CTA scans ustart after its loop).
  uint8_t fb_first[kMaxCtas], fb_last[kMaxCtas], lb_last[kMaxCtas];
};

template <int FMT, int MT>
struct Smem {
  static constexpr int NT = MT / 8;
  static constexpr int WS = w_stages(FMT, MT);
  uint8_t w[WS][kTileBytes];                 // SWIZZLE_128B weight tiles (1024-aligned)
  uint8_t mraw[WS][meta_raw_bytes(FMT)];     // raw metadata tiles (TMA), 16 B per row per tensor
  // B fragments [nt][group][vec][lane]
  static constexpr int XS = x_stages(MT);
  uint4 x[XS][NT][2][4][32];
  float xsum[XS][2][MT];                     // INT4: sum of the group's (scaled) activations per row m
  float xoff[XS][2][MT];                     // INT4: 1024 x the sum of the group's B operand per row m
  float xf[XS][MT];                          // power-of-two factor per activation row
  uint64_t full_w[WS];
  uint64_t empty_w[WS];
  uint64_t full_x[XS];
  uint64_t empty_x[XS];
};

// Split-K exchange.  A contributor posts each fp32 partial sum as its bits XOR kPartTag, a
// signalling-NaN pattern that no arithmetic result has (a NaN produced by an fp32 operation
// is the canonical 0x7fffffff, and the partial sums are all results of fp32 operations), so a
// posted word is never 0.  The exchange area is all zeros between calls; a reducing CTA polls
// a word until it is non-zero, which is then the value itself (one 32-bit access: no ordering
// between a flag and the data is needed), and writes the 0 back.
constexpr uint32_t kPartTag = 0x7fbadbadu;
__device__ __forceinline__ uint32_t tag_partial(float v) { return __float_as_uint(v) ^ kPartTag; }
__device__ __forceinline__ float untag_partial(uint32_t w) { return __uint_as_float(w ^ kPartTag); }
__device__ __forceinline__ void st_relaxed_gpu(uint32_t* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint4 ld_relaxed_gpu_v4(const uint32_t* p) {
  uint4 v;
  asm volatile("ld.relaxed.gpu.global.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_gpu_v4_zero(uint32_t* p) {
  asm volatile("st.relaxed.gpu.global.v4.u32 [%0], {%1,%1,%1,%1};" ::"l"(p), "r"(0u) : "memory");
}
__device__ __forceinline__ bool all_posted(const uint4& v) { return v.x != 0u && v.y != 0u && v.z != 0u && v.w != 0u; }

// Posted words in flight per reduction slot (a band's CTAs are read in chunks of this many, in
// CTA order).
constexpr int kChunk = 12;

// Reduction slot idx of a shared band: activation row m and the first of its four output
// rows r4 inside the band.
template <int EPI>
__device__ __forceinline__ void reduce_slot(int idx, int& m, int& r4) {
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
}

// Exchange tile of CTA c for a shared band: c + P where c holds the band's first unit (the
// band is the last of its range), c where its range starts inside the band.
__device__ __forceinline__ long long part_tile(int c, int c_first, int P) { return c == c_first ? c + P : c; }

// Reads of one slot's posted words of CTAs c .. min(c + kChunk - 1, c_last) (base: the slot's
// word in tile 0); the entries past c_last read as posted dummies.
__device__ __forceinline__ void load_chunk(uint4 (&v)[kChunk], const uint32_t* base, long long stride, int c,
                                           int c_first, int c_last, int P) {
#pragma unroll
  for (int q = 0; q < kChunk; ++q)
    v[q] = (c + q <= c_last) ? ld_relaxed_gpu_v4(base + part_tile(c + q, c_first, P) * stride)
                             : make_uint4(1u, 1u, 1u, 1u);
}

// The slots lo + tid, lo + tid + nthreads, ... below hi of a shared band's M x kBand / 4
// float4 slots: the posted partial sums of the band's CTAs c_first .. c_last added in CTA
// order (deterministic); every word is waited for until posted and then cleared; bf16
// results to the outputs.  With `fresh`, v holds on entry the reads of the first slot's first
// chunk, issued by the caller.  Each round of the wait re-reads every word of the chunk not
// posted yet, all reads in flight together.  The wait ends kWaitLimitNs after the call at the
// latest (error flag set; the lanes keep going so that every warp stays converged: lo and
// nthreads are multiples of 32).
template <int MT, int EPI>
__device__ __forceinline__ void reduce_slots(const Params& p, int band, int c_first, int c_last, int lo, int hi,
                                             int tid, int nthreads, uint4 (&v)[kChunk], bool fresh) {
  const uint64_t t0 = globaltimer_ns();
  constexpr long long kStride = static_cast<long long>(MT) * kBand;
  bool live = true;
  for (int idx = lo + tid; idx < hi; idx += nthreads) {
    int m, r4;
    reduce_slot<EPI>(idx, m, r4);
    float4 acc4 = make_float4(0.f, 0.f, 0.f, 0.f);
    bool started = false;
    uint32_t* base = p.part + static_cast<long long>(m) * kBand + r4;
    for (int c = c_first; c <= c_last; c += kChunk) {
      if (!fresh) load_chunk(v, base, kStride, c, c_first, c_last, p.P);
      fresh = false;
      while (live) {
        bool all = true;
#pragma unroll
        for (int q = 0; q < kChunk; ++q) all = all && all_posted(v[q]);
        if (all) break;
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
          atomicOr(&g_gemv_err, kErrWaitReduce);
          live = false;
        } else {
#pragma unroll
          for (int q = 0; q < kChunk; ++q)
            if (!all_posted(v[q])) v[q] = ld_relaxed_gpu_v4(base + part_tile(c + q, c_first, p.P) * kStride);
        }
      }
#pragma unroll
      for (int q = 0; q < kChunk; ++q)
        if (c + q <= c_last) {
          const float4 f = make_float4(untag_partial(v[q].x), untag_partial(v[q].y), untag_partial(v[q].z),
                                       untag_partial(v[q].w));
          if (!started) {
            acc4 = f;   // the first CTA's sums start the chain (not 0 + x: keeps a -0)
            started = true;
          } else {
            acc4.x += f.x; acc4.y += f.y; acc4.z += f.z; acc4.w += f.w;
          }
          st_relaxed_gpu_v4_zero(base + part_tile(c + q, c_first, p.P) * kStride);
        }
    }
    const float o4[4] = {acc4.x, acc4.y, acc4.z, acc4.w};
    if constexpr (EPI == kEpiSwiglu) {
      // p.M * kBand / 4 is a multiple of 64 and every warp's idx range is 32-aligned: whole
      // warps run each iteration, so the shuffles below are converged
      float u4[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) u4[q] = __shfl_xor_sync(0xffffffffu, o4[q], 1);
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

// The bf16 outputs of one consumer lane: rows r0 / r1 of the band, activation rows
// 2t + (e & 1) + 8 nt.  SwiGLU: r1 = r0 + 8 is the up row of the gate row r0 (the
// interleaved layout), one output column per pair.
template <int MT, int EPI>
__device__ __forceinline__ void store_outputs(const Params& p, int band, int r0, int r1, int t,
                                              const float (&acc)[MT / 8][4]) {
  constexpr int NT = MT / 8;
  if constexpr (EPI == kEpiSwiglu) {
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
}

// Stage i of a CTA = unit u0 + i = (band, group pair j).  Ranges are split at pair
// boundaries, so a stage never straddles a band.  The cursor divides once at start-up and
// then steps incrementally.
struct Cursor {
  int u, u0, u1, seg_start, seg_end;
  int band, j, GP;
  __device__ void set_seg() {
    const int bs = band * GP;
    seg_start = bs > u0 ? bs : u0;
    seg_end = bs + GP < u1 ? bs + GP : u1;
  }
  __device__ void init(int a, int b, int gp) {
    u = a; u0 = a; u1 = b; GP = gp;
    band = a / gp;
    j = a - band * gp;
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
           const __grid_constant__ CUtensorMap tmap_z, const __grid_constant__ Params p) {
  using S = Smem<FMT, MT>;
  constexpr int NT = MT / 8;
  constexpr int WS = S::WS;
  // INT4 operand form: fp16 (1024 + q | 1024 + 16 q, scaled activations) for 8-row activation
  // tiles, where it saves unpack instructions; bf16 (128 + q, raw activations) for 16-row
  // tiles, where each unpacked weight feeds two MMAs and the leaner activation prep wins.
  constexpr bool kF16 = (FMT == kInt4G128) && (MT == 8);
  // Split-K reduction of a shared band by all of its CTAs (16 and 32-row tiles, whose partial
  // tiles are large) or by the CTA holding its first unit alone (8-row tiles).
  constexpr bool kAllReduce = MT >= 16;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  S& sm = *reinterpret_cast<S*>(smem_raw + smem_align_pad(smem_raw));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int cta = blockIdx.x;
  const int u0 = p.ustart[cta];
  const int u1 = p.ustart[cta + 1];
  const int nstages = u1 - u0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < WS; ++s) {
      mbar_init(&sm.full_w[s], 1);
      mbar_init(&sm.empty_w[s], 32 * kConsumerWarps);
    }
    for (int s = 0; s < S::XS; ++s) {
      mbar_init(&sm.full_x[s], 32);
      mbar_init(&sm.empty_x[s], 32 * kConsumerWarps);
    }
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
      if (p.meta_tma) {
        tma_prefetch_desc(&tmap_s);
        if (FMT == kInt4G128) tma_prefetch_desc(&tmap_z);
      }
      const uint64_t pol_w = l2_policy_evict_first();
      const uint64_t pol_m = l2_policy_evict_last();
      Cursor st;
      st.init(u0, u1, p.GP);
      // While the previous kernel of the stream finishes: pull the first stage's weight tile
      // into L2 (a hint only; every read that lands in shared memory follows the wait).  One
      // tile: hints for more stages, or for the metadata tiles, hold up this thread's first
      // loads after the wait by more than they save.
      tma_prefetch_l2_2d(&tmap_w, st.j * 128, st.band * kBand);
      pdl_wait();
      int i = 0;
      for (; i < nstages; ++i, st.next()) {
        const int slot = i % WS;
        const uint32_t ph = (i / WS) & 1;
        if (i >= WS && !mbar_wait(&sm.empty_w[slot], ph ^ 1, &g_gemv_err, kErrWaitEmpty)) break;
        mbar_arrive_expect_tx(&sm.full_w[slot], kTileBytes + (p.meta_tma ? kMetaBytes : 0));
        tma_load_2d(&sm.w[slot][0], &tmap_w, st.j * 128, st.band * kBand, &sm.full_w[slot], pol_w);
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
    }
  } else if (warp < kFirstConsumer) {
    // ------------------------------------------------------------------ prep
    // Activations only, read from global memory (they were written by the previous kernel of
    // the stream: every read follows the dependency wait) and converted in registers.
    // Lane L owns the 16-byte chunk L (8 activations at k = 256 j + 8 L) of each row:
    //   INT4:  L = 16 h + 4 t + v  (group h, fragment lane t, vector v: k = 128 h + 32 t + 8 v)
    //   MXFP4: L = 16 h + 4 blk + t (group h, block blk, fragment lane t: k = 128 h + 32 blk + 8 t)
    const int pw = warp - 1;
    const int h = lane >> 4;
    const int ft = (FMT == kInt4G128) ? ((lane >> 2) & 3) : (lane & 3);   // fragment lane t
    const int fv = (FMT == kInt4G128) ? (lane & 3) : ((lane >> 2) & 3);   // vector / block
    Cursor st;
    st.init(u0, u1, p.GP);
    for (int q = 0; q < pw && q < nstages; ++q) st.next();
    // Activation rows M .. MT-1 of a tile are zeros in every stage: this warp's ring slots get
    // them (and a unit row factor, zero group sums) once, here, and each stage converts rows
    // below M only.
    for (int slot = pw; slot < S::XS; slot += kPrepWarps) {
      uint4* xs = &sm.x[slot][0][0][0][0];
      for (int q = lane; q < NT * 2 * 4 * 32; q += 32) xs[q] = make_uint4(0u, 0u, 0u, 0u);
      if (lane < MT) {
        sm.xf[slot][lane] = 1.f;
#pragma unroll
        for (int hg = 0; hg < 2; ++hg) {
          sm.xsum[slot][hg][lane] = 0.f;
          sm.xoff[slot][hg][lane] = 0.f;
        }
      }
    }
    __syncwarp();
    pdl_wait();
    for (int i = pw; i < nstages; i += kPrepWarps) {
      const int slot = i % S::XS;
      const uint32_t ph = (i / S::XS) & 1;
      if (!mbar_wait(&sm.empty_x[slot], ph ^ 1, &g_gemv_err, kErrWaitEmpty)) break;
      const int k0 = 256 * st.j + 8 * lane;   // this lane's 8 activations of each row
      const bool kin = k0 < p.K;
      // up to 16 rows are all in flight at once; larger tiles are loaded 8 rows at a time
      constexpr int CR = MT <= 16 ? MT : 8;
      uint4 cur[CR];
      auto load_rows = [&](int r0) {
#pragma unroll
        for (int r = 0; r < CR; ++r)
          cur[r] = (r0 + r < p.M && kin)
                       ? __ldcg(reinterpret_cast<const uint4*>(p.X + static_cast<long long>(r0 + r) * p.K + k0))
                       : make_uint4(0u, 0u, 0u, 0u);
      };
      load_rows(0);
      for (int q = 0; q < kPrepWarps && st.u < u1; ++q) st.next();
      constexpr int kPrepUnroll = MT > 16 ? 1 : NT;   // wide tiles: one 8-row tile at a time
#pragma unroll kPrepUnroll
      for (int nt = 0; nt < NT; ++nt) {
        if constexpr (MT > 16) {
          if (nt > 0) load_rows(8 * nt);
        }
        constexpr int kCurTile = MT <= 16 ? 8 : 0;   // row offset of tile nt inside cur
        // One power-of-two scale 2^-k per stage and activation row carries every operand into
        // fp16 exactly (bf16_to_f16_exponent: the row's largest in [2^14, 2^15), small rows
        // scaled up); only values more than 2^31 below their row's largest lose bits, as fp16
        // subnormals.  max |x| per row: bf16 magnitudes order like integers.
        const int nrow = p.M - 8 * nt;   // rows of this 8-row tile in use (warp-uniform)
        if (nrow <= 0) continue;          // an all-zero tile: its slot rows stay zero
        float inv[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) inv[r] = 1.f;
        if constexpr (FMT != kInt4G128 || kF16) {
          // this lane's max per row, then one warp-wide max reduction per row in use
          auto row_scale = [&](int r) {
            const uint4 x = cur[kCurTile * nt + r];
            const uint32_t v = __vmaxu2(__vmaxu2(x.x & 0x7fff7fffu, x.y & 0x7fff7fffu),
                                        __vmaxu2(x.z & 0x7fff7fffu, x.w & 0x7fff7fffu));
            const uint32_t mx = __reduce_max_sync(0xffffffffu, max(v & 0xffffu, v >> 16));
            const int kk = bf16_to_f16_exponent(mx);
            inv[r] = pow2_normal(-kk);
            if (lane == r) sm.xf[slot][8 * nt + r] = pow2_normal(kk);
          };
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            if (r >= nrow) break;
            row_scale(r);
          }
        }
        // One row of the tile into its B-fragment slots.
        auto put_row = [&](int r) {
          uint4* dst = &sm.x[slot][nt][h][fv][4 * r + ft];
          const uint4 x = cur[kCurTile * nt + r];
          const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
          if constexpr (FMT == kInt4G128 && !kF16) {
            // (x0,x4) (x1,x5) (x2,x6) (x3,x7): the k order of the unpacked nibble pairs.
            uint4 o;
            o.x = prmt(x.x, x.z, 0x5410);
            o.y = prmt(x.x, x.z, 0x7632);
            o.z = prmt(x.y, x.w, 0x5410);
            o.w = prmt(x.y, x.w, 0x7632);
            *dst = o;
          } else if constexpr (FMT == kInt4G128) {
            // the same k order; the odd nibbles come out of the weights as 16 q, so their
            // activations carry 1/16
            const float f0 = inv[r], f1 = inv[r] * 0.0625f;
            const uint32_t lo[4] = {w4[0] << 16, w4[0] & 0xffff0000u, w4[1] << 16, w4[1] & 0xffff0000u};
            const uint32_t hi[4] = {w4[2] << 16, w4[2] & 0xffff0000u, w4[3] << 16, w4[3] & 0xffff0000u};
            uint32_t o[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float f = (q & 1) ? f1 : f0;
              __half2 hh = __floats2half2_rn(__uint_as_float(lo[q]) * f, __uint_as_float(hi[q]) * f);
              o[q] = *reinterpret_cast<uint32_t*>(&hh);
            }
            *dst = make_uint4(o[0], o[1], o[2], o[3]);
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
        };
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          if (r >= nrow) break;
          put_row(r);
        }
        if constexpr (FMT == kInt4G128 && !kF16) {
          // Per-group activation sums of the tile's 8 rows on the tensor core: an all-ones A
          // times the just-written B fragments gives every column sum (exact products, fp32
          // accumulation).  Lane (g = 0, t) receives rows 2t, 2t + 1 of the tile.
          __syncwarp();
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
        } else if constexpr (FMT == kInt4G128) {
          // Per-group sums of the tile's 8 rows on the tensor core (exact products, fp32
          // accumulation): A = (1, 1 | 16, 16) times the B fragments just written gives the
          // sum of the scaled activations; A = all ones gives the sum of the B operand itself,
          // whose 1024-fold the weights' fp16 offset adds.  Lane (g = 0, t) receives rows
          // 2t, 2t + 1 of the tile.
          __syncwarp();
          constexpr uint32_t kOne = 0x3c003c00u;      // fp16 (1, 1)
          constexpr uint32_t kSixteen = 0x4c004c00u;  // fp16 (16, 16)
#pragma unroll
          for (int hg = 0; hg < 2; ++hg) {
            float d[4][4], e[4][4];
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const uint4 b = sm.x[slot][nt][hg][v][lane];
#pragma unroll
              for (int q = 0; q < 4; ++q) { d[v][q] = 0.f; e[v][q] = 0.f; }
              mma_f16(d[v], kOne, kOne, kSixteen, kSixteen, b.x, b.y);
              mma_f16(d[v], kOne, kOne, kSixteen, kSixteen, b.z, b.w);
              mma_f16(e[v], kOne, kOne, kOne, kOne, b.x, b.y);
              mma_f16(e[v], kOne, kOne, kOne, kOne, b.z, b.w);
            }
            const float s0 = (d[0][0] + d[1][0]) + (d[2][0] + d[3][0]);
            const float s1 = (d[0][1] + d[1][1]) + (d[2][1] + d[3][1]);
            const float o0 = 1024.f * ((e[0][0] + e[1][0]) + (e[2][0] + e[3][0]));
            const float o1 = 1024.f * ((e[0][1] + e[1][1]) + (e[2][1] + e[3][1]));
            if (lane < 4) {
              *reinterpret_cast<float2*>(&sm.xsum[slot][hg][8 * nt + 2 * lane]) = make_float2(s0, s1);
              *reinterpret_cast<float2*>(&sm.xoff[slot][hg][8 * nt + 2 * lane]) = make_float2(o0, o1);
            }
          }
        }
      }
      mbar_arrive(&sm.full_x[slot]);
    }
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
    st.init(u0, u1, p.GP);
    // 8-row tiles: the CTA holding a shared band's first unit reduces the whole band (its
    // range ends inside the band, so it gets there last; the band is the range's last).
    // Larger tiles: every CTA of the band reduces a share.
    const int last_band = (u1 - 1) / p.GP;
    const int red_band =
        (!kAllReduce && u0 <= last_band * p.GP && u1 < (last_band + 1) * p.GP) ? last_band : -1;
    pdl_wait();   // outputs and the exchange area may be in use by the previous kernel
    for (int i = 0; i < nstages; ++i, st.next()) {
      const int ws = i % WS;
      const uint32_t wph = (i / WS) & 1;
      const int xs = i % S::XS;
      const uint32_t xph = (i / S::XS) & 1;

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
      if constexpr (NT >= 4) {
        // 32 or 64 activation rows: the n-tiles in chunks of four, each chunk unpacking the
        // weights again, so that one chunk's accumulators per group stay in registers.
        constexpr int NC = (FMT == kInt4G128 || NT < 8) ? 4 : 2;
#pragma unroll
        for (int cb = 0; cb < NT; cb += NC) {
          float sacc[NC][4];   // MXFP4: the stage's scaled block sums of this chunk
#pragma unroll
          for (int nc = 0; nc < NC; ++nc)
#pragma unroll
            for (int e = 0; e < 4; ++e) sacc[nc][e] = 0.f;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            // this group's words (INT4) or blocks (MXFP4), rows r0 / r1, read again per chunk
            uint32_t w0[4], w1[4];
            if constexpr (FMT == kInt4G128) {
              const int c = 4 * h + t;
              const uint4 a = *reinterpret_cast<const uint4*>(wt + r0 * 128 + ((c ^ (r0 & 7)) << 4));
              const uint4 b = *reinterpret_cast<const uint4*>(wt + r1 * 128 + ((c ^ (r1 & 7)) << 4));
              w0[0] = a.x; w0[1] = a.y; w0[2] = a.z; w0[3] = a.w;
              w1[0] = b.x; w1[1] = b.y; w1[2] = b.z; w1[3] = b.w;
            } else {
#pragma unroll
              for (int blk = 0; blk < 4; ++blk) {
                const int cc = 4 * h + blk;
                w0[blk] = *reinterpret_cast<const uint32_t*>(wt + r0 * 128 + ((cc ^ (r0 & 7)) << 4) + 4 * t);
                w1[blk] = *reinterpret_cast<const uint32_t*>(wt + r1 * 128 + ((cc ^ (r1 & 7)) << 4) + 4 * t);
              }
            }
            float ga[NC][4];
#pragma unroll
            for (int nc = 0; nc < NC; ++nc)
#pragma unroll
              for (int e = 0; e < 4; ++e) ga[nc][e] = 0.f;
#pragma unroll
            for (int jw = 0; jw < 4; ++jw) {
              uint32_t a[2][4];   // [hh] the A fragments of the two k16 steps
              if constexpr (FMT == kInt4G128) {
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                  a[hh][0] = lop3_and_or(w0[jw] >> (8 * hh), 0x000f000fu, 0x43004300u);
                  a[hh][1] = lop3_and_or(w1[jw] >> (8 * hh), 0x000f000fu, 0x43004300u);
                  a[hh][2] = lop3_and_or(w0[jw] >> (8 * hh + 4), 0x000f000fu, 0x43004300u);
                  a[hh][3] = lop3_and_or(w1[jw] >> (8 * hh + 4), 0x000f000fu, 0x43004300u);
                }
              } else {
                uint32_t f0[4], f1[4];
                e2m1x8_to_f16x2x4(w0[jw], f0);
                e2m1x8_to_f16x2x4(w1[jw], f1);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                  a[hh][0] = f0[2 * hh]; a[hh][1] = f1[2 * hh];
                  a[hh][2] = f0[2 * hh + 1]; a[hh][3] = f1[2 * hh + 1];
                }
              }
              float bacc[NC][4];   // MXFP4: this block's sums
#pragma unroll
              for (int nc = 0; nc < NC; ++nc) {
                const uint4 bv = sm.x[xs][cb + nc][h][jw][lane];
                if constexpr (FMT == kInt4G128) {
                  mma_bf16(ga[nc], a[0][0], a[0][1], a[0][2], a[0][3], bv.x, bv.y);
                  mma_bf16(ga[nc], a[1][0], a[1][1], a[1][2], a[1][3], bv.z, bv.w);
                } else {
#pragma unroll
                  for (int e = 0; e < 4; ++e) bacc[nc][e] = 0.f;
                  mma_f16(bacc[nc], a[0][0], a[0][1], a[0][2], a[0][3], bv.x, bv.y);
                  mma_f16(bacc[nc], a[1][0], a[1][1], a[1][2], a[1][3], bv.z, bv.w);
                }
              }
              if constexpr (FMT != kInt4G128) {
                const float e0 = e8m0_to_f32((eb[0][h] >> (8 * jw)) & 0xffu);
                const float e1 = e8m0_to_f32((eb[1][h] >> (8 * jw)) & 0xffu);
#pragma unroll
                for (int nc = 0; nc < NC; ++nc) {
                  sacc[nc][0] = fmaf(e0, bacc[nc][0], sacc[nc][0]);
                  sacc[nc][1] = fmaf(e0, bacc[nc][1], sacc[nc][1]);
                  sacc[nc][2] = fmaf(e1, bacc[nc][2], sacc[nc][2]);
                  sacc[nc][3] = fmaf(e1, bacc[nc][3], sacc[nc][3]);
                }
              }
            }
            if constexpr (FMT == kInt4G128) {
              // y += s * sum_k (128 + q) x + c * sum_k x,  c = -s (128 + z)
              const float s0 = __half2float(__ushort_as_half(static_cast<unsigned short>(sraw[0] >> (16 * h))));
              const float s1 = __half2float(__ushort_as_half(static_cast<unsigned short>(sraw[1] >> (16 * h))));
              const float c0 = -s0 * (128.f + __half2float(__ushort_as_half(static_cast<unsigned short>(zraw[0] >> (16 * h)))));
              const float c1 = -s1 * (128.f + __half2float(__ushort_as_half(static_cast<unsigned short>(zraw[1] >> (16 * h)))));
#pragma unroll
              for (int nc = 0; nc < NC; ++nc) {
                const float2 xs2 = *reinterpret_cast<const float2*>(&sm.xsum[xs][h][2 * t + 8 * (cb + nc)]);
                acc[cb + nc][0] = fmaf(c0, xs2.x, fmaf(s0, ga[nc][0], acc[cb + nc][0]));
                acc[cb + nc][1] = fmaf(c0, xs2.y, fmaf(s0, ga[nc][1], acc[cb + nc][1]));
                acc[cb + nc][2] = fmaf(c1, xs2.x, fmaf(s1, ga[nc][2], acc[cb + nc][2]));
                acc[cb + nc][3] = fmaf(c1, xs2.y, fmaf(s1, ga[nc][3], acc[cb + nc][3]));
              }
            }
          }
          if constexpr (FMT != kInt4G128) {
#pragma unroll
            for (int nc = 0; nc < NC; ++nc) {
              const float2 xf = *reinterpret_cast<const float2*>(&sm.xf[xs][2 * t + 8 * (cb + nc)]);
              acc[cb + nc][0] = fmaf(xf.x, sacc[nc][0], acc[cb + nc][0]);
              acc[cb + nc][1] = fmaf(xf.y, sacc[nc][1], acc[cb + nc][1]);
              acc[cb + nc][2] = fmaf(xf.x, sacc[nc][2], acc[cb + nc][2]);
              acc[cb + nc][3] = fmaf(xf.y, sacc[nc][3], acc[cb + nc][3]);
            }
          }
        }
      } else if constexpr (FMT == kInt4G128) {
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
                // nibble pairs (s, s+4) as fp16 1024 + q and (s+1, s+5) as 1024 + 16 q (exact;
                // their activations carry 1/16); the offset and zero point are folded below
                uint32_t a0, a1, a2, a3;
                if constexpr (kF16) {
                  const uint32_t u0 = hh ? (w0[h][jw] >> 8) : w0[h][jw];
                  const uint32_t u1 = hh ? (w1[h][jw] >> 8) : w1[h][jw];
                  a0 = lop3_and_or(u0, 0x000f000fu, 0x64006400u);
                  a1 = lop3_and_or(u1, 0x000f000fu, 0x64006400u);
                  a2 = lop3_and_or(u0, 0x00f000f0u, 0x64006400u);
                  a3 = lop3_and_or(u1, 0x00f000f0u, 0x64006400u);
                } else {
                  // bf16 128 + q: every nibble shifted to bit 0 (a byte's high nibble would
                  // reach bf16's exponent)
                  a0 = lop3_and_or(w0[h][jw] >> (8 * hh), 0x000f000fu, 0x43004300u);
                  a1 = lop3_and_or(w1[h][jw] >> (8 * hh), 0x000f000fu, 0x43004300u);
                  a2 = lop3_and_or(w0[h][jw] >> (8 * hh + 4), 0x000f000fu, 0x43004300u);
                  a3 = lop3_and_or(w1[h][jw] >> (8 * hh + 4), 0x000f000fu, 0x43004300u);
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                  const uint4 bv = bx[h][q][nt];
                  if constexpr (kF16) mma_f16(ga[h][q][nt], a0, a1, a2, a3, hh ? bv.z : bv.x, hh ? bv.w : bv.y);
                  else mma_bf16(ga[h][q][nt], a0, a1, a2, a3, hh ? bv.z : bv.x, hh ? bv.w : bv.y);
                }
              }
        }
        if constexpr (kF16) {
          // With x' = x 2^-e (per stage and activation row) and B' the B operand:
          //   sum_k (q - z) s x = 2^e s (D - 1024 sum_k B' - z sum_k x'),  D = sum_k A' B'
          // (offset and zero-point cross terms of 第 6 课：量化源码走读 §3, from the group sums).
          float sacc[NT][4];
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) sacc[nt][e] = 0.f;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const float s0 = __half2float(__ushort_as_half(static_cast<unsigned short>(sraw[0] >> (16 * h))));
            const float s1 = __half2float(__ushort_as_half(static_cast<unsigned short>(sraw[1] >> (16 * h))));
            const float z0 = __half2float(__ushort_as_half(static_cast<unsigned short>(zraw[0] >> (16 * h))));
            const float z1 = __half2float(__ushort_as_half(static_cast<unsigned short>(zraw[1] >> (16 * h))));
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              const float2 xs2 = *reinterpret_cast<const float2*>(&sm.xsum[xs][h][2 * t + 8 * nt]);
              const float2 xo2 = *reinterpret_cast<const float2*>(&sm.xoff[xs][h][2 * t + 8 * nt]);
              float gs[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                gs[e] = ga[h][0][nt][e];
#pragma unroll
                for (int q = 1; q < PAR; ++q) gs[e] += ga[h][q][nt][e];
              }
              sacc[nt][0] = fmaf(s0, gs[0] - fmaf(z0, xs2.x, xo2.x), sacc[nt][0]);
              sacc[nt][1] = fmaf(s0, gs[1] - fmaf(z0, xs2.y, xo2.y), sacc[nt][1]);
              sacc[nt][2] = fmaf(s1, gs[2] - fmaf(z1, xs2.x, xo2.x), sacc[nt][2]);
              sacc[nt][3] = fmaf(s1, gs[3] - fmaf(z1, xs2.y, xo2.y), sacc[nt][3]);
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
        } else {
          // y += s * sum_k (128 + q) x + c * sum_k x,  c = -s (128 + z)   (zero-point cross
          // term of 第 6 课：量化源码走读 §3, from the group sum of the activations)
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

      // Band end.  A band this CTA covers whole is written as bf16; a band shared with other
      // CTAs (only the range's first or last can be) has its partial sums posted, in tile
      // cta + P when this CTA holds the band's first unit, else in tile cta, and is reduced
      // after the loop.
      if (st.seg_last()) {
        const int band = st.band;
        const int bs = band * p.GP;
        if (st.seg_start == bs && st.seg_end == bs + p.GP) {
          store_outputs<MT, EPI>(p, band, r0, r1, t, acc);
        } else {
          uint32_t* slotp = p.part + (st.seg_start == bs ? cta + p.P : cta) * static_cast<long long>(MT) * kBand;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int m = 2 * t + (e & 1) + 8 * nt;
              if (m < p.M) st_relaxed_gpu(slotp + m * kBand + ((e >> 1) ? r1 : r0), tag_partial(acc[nt][e]));
            }
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
      }
      mbar_arrive(&sm.empty_x[xs]);   // activations consumed
    }
    // ---------------------------------------------------------------- shared bands
    // Every CTA has posted all its partial sums before it waits for any other's.
    constexpr int kSlotsPerRow = kBand / 4;
    const int tid = cw * 32 + lane;
    uint4 v[kChunk];
    if constexpr (kAllReduce) {
      const int fb = u0 / p.GP;
#pragma unroll 1
      for (int b = fb; b <= last_band; b += (last_band > fb ? last_band - fb : 1)) {
        if (u0 <= b * p.GP && u1 >= (b + 1) * p.GP) continue;   // covered whole: written above
        // the band's CTAs: this CTA holds the last band's first unit when that band is not its first
        const int c_first = (b == fb) ? p.fb_first[cta] : cta;
        const int c_last = (b == fb) ? p.fb_last[cta] : p.lb_last[cta];
        // CTA i of the band's n takes the 32-slot chunks [i nch / n, (i + 1) nch / n)
        const int n = c_last - c_first + 1, i = cta - c_first, nch = p.M * kSlotsPerRow / 32;
        reduce_slots<MT, EPI>(p, b, c_first, c_last, 32 * ((i * nch) / n), 32 * (((i + 1) * nch) / n), tid,
                              32 * kConsumerWarps, v, false);
      }
    } else if (red_band >= 0) {
      // the band's CTAs: this one and cta + 1 .. c_hi.  Each reading thread waits only for the
      // words of its own slots (its rows come from one consumer warp of each CTA), so no
      // barrier gathers this CTA's warps; the first chunk's reads go out at once.
      const int c_hi = p.lb_last[cta];
      if (tid < p.M * kSlotsPerRow) {
        int m, r4;
        reduce_slot<EPI>(tid, m, r4);
        load_chunk(v, p.part + static_cast<long long>(m) * kBand + r4, static_cast<long long>(MT) * kBand, cta,
                   cta, c_hi, p.P);
      }
      reduce_slots<MT, EPI>(p, red_band, cta, c_hi, 0, p.M * kSlotsPerRow, tid, 32 * kConsumerWarps, v, true);
    }
  }
}

int num_ctas(long long U) {
  long long sms = device_sm_count();
  if (sms > kMaxCtas) sms = kMaxCtas;
  if (U <= sms) return static_cast<int>(U);
  // as few CTAs as keep the longest range at ceil(U / sms) stages: the same critical path,
  // fewer CTAs sharing each band
  const long long per = (U + sms - 1) / sms;
  return static_cast<int>((U + per - 1) / per);
}

}  // namespace gemv

// Activation rows per launch: tiles of 8, 16 or 32; larger M runs as 32-row slices.
static int tile_rows(int64_t M) { return M <= 8 ? 8 : M <= 16 ? 16 : 32; }

// The exchange area of the largest launch (two tiles for each of kMaxCtas CTAs, 32-row tiles)
// fits the header's.
static_assert(2 * static_cast<size_t>(gemv::kMaxCtas) * 32 * gemv::kBand * sizeof(uint32_t) <= kWsDecodeBytes,
              "decode exchange area over its share of the workspace header");

size_t gemv_mma_workspace_bytes(int fmt, int64_t M, int64_t K, int64_t N) {
  if (M < 1 || M > kDecodeMaxM || N < 1 || K < 1) return 0;
  const int MT = tile_rows(M);
  const long long G = (K + gemv::kGroupK - 1) / gemv::kGroupK;
  const long long bands = (N + gemv::kBand - 1) / gemv::kBand;
  const int P = gemv::num_ctas(bands * ((G + 1) / 2));
  (void)fmt;
  return kWsCounterBytes + 2 * static_cast<size_t>(P) * MT * gemv::kBand * sizeof(uint32_t);
}

template <int FMT, int MT, int EPI>
static cudaError_t launch_gemv_t(const CUtensorMap& tw, const CUtensorMap& ts, const CUtensorMap& tz,
                                 const gemv::Params& p, cudaStream_t stream) {
  using S = gemv::Smem<FMT, MT>;
  static_assert(sizeof(S) + 1024 <= gemv::kSmemLimit, "decode kernel shared memory over the per-CTA limit");
  const size_t smem = sizeof(S) + 1024;
  auto kern = gemv::k_gemv<FMT, MT, EPI>;
  cudaError_t ea = set_smem_attr_once(reinterpret_cast<const void*>(kern), smem);
  if (ea != cudaSuccess) return ea;
  // Programmatic stream serialization: the CTAs may launch while the previous kernel of the
  // stream is still running; the kernel itself waits (griddepcontrol.wait) before it reads
  // anything that kernel may have written or writes anything.
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
  return cudaLaunchKernelEx(&cfg, kern, tw, ts, tz, p);
}

static cudaError_t launch_gemv_slice(int fmt, const uint16_t* X, int64_t M, int64_t K, int64_t N,
                                     const int32_t* Wq, const void* scales, const uint16_t* zeros, uint16_t* Y,
                                     void* ws, size_t ws_bytes, cudaStream_t stream, int epi,
                                     const OutSplit* split);

cudaError_t launch_gemv_mma(int fmt, const uint16_t* X, int64_t M, int64_t K, int64_t N, const int32_t* Wq,
                            const void* scales, const uint16_t* zeros, uint16_t* Y, void* ws, size_t ws_bytes,
                            cudaStream_t stream, int epi, const OutSplit* split) {
  if (epi == kEpiSwiglu && N % 16 != 0) return cudaErrorInvalidValue;
  if (epi == kEpiSplit3 && !split) return cudaErrorInvalidValue;
  // M > 32: consecutive 32-row slices of X and of the outputs, one launch each, in order on
  // the stream (they share the workspace; each leaves its exchange area at zero).
  constexpr int64_t kSlice = 32;
  const int64_t ldy = epi == kEpiSwiglu ? N / 2 : N;
  for (int64_t m0 = 0; m0 < M; m0 += kSlice) {
    const int64_t ms = M - m0 < kSlice ? M - m0 : kSlice;
    OutSplit sp{};
    if (split) {
      sp = *split;
      for (int q = 0; q < 3; ++q) sp.y[q] = split->y[q] + m0 * split->ld[q];
    }
    const cudaError_t e = launch_gemv_slice(fmt, X + m0 * K, ms, K, N, Wq, scales, zeros, Y ? Y + m0 * ldy : Y,
                                            ws, ws_bytes, stream, epi, split ? &sp : nullptr);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

static cudaError_t launch_gemv_slice(int fmt, const uint16_t* X, int64_t M, int64_t K, int64_t N,
                                     const int32_t* Wq, const void* scales, const uint16_t* zeros, uint16_t* Y,
                                     void* ws, size_t ws_bytes, cudaStream_t stream, int epi,
                                     const OutSplit* split) {
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
  const long long U = static_cast<long long>(p.bands) * p.GP;
  if (p.bands > kWsMaxCounters || U > (1LL << 30)) return cudaErrorInvalidValue;
  p.U = static_cast<int>(U);
  p.P = gemv::num_ctas(U);
  for (int c = 0; c <= p.P; ++c) p.ustart[c] = static_cast<int>((U * c) / p.P);   // P <= U: none empty
  {
    // owner(x): the CTA holding unit x (ranges are increasing: walk forward from a lower bound)
    auto owner = [&](long long x, int from) {
      int c = from;
      while (c + 1 < p.P && p.ustart[c + 1] <= x) ++c;
      return c;
    };
    // all three are nondecreasing in c, and the last two are >= c: each walk resumes where it
    // stopped, O(P) in all
    int lo = 0, hf = 0, hl = 0;
    for (int c = 0; c < p.P; ++c) {
      const long long fb = p.ustart[c] / p.GP, lb = (p.ustart[c + 1] - 1) / p.GP;
      lo = owner(fb * p.GP, lo);
      hf = owner(fb * p.GP + p.GP - 1, hf > c ? hf : c);
      hl = owner(lb * p.GP + p.GP - 1, hl > c ? hl : c);
      p.fb_first[c] = static_cast<uint8_t>(lo);
      p.fb_last[c] = static_cast<uint8_t>(hf);
      p.lb_last[c] = static_cast<uint8_t>(hl);
    }
  }
  if (ws_bytes < gemv_mma_workspace_bytes(fmt, M, K, N)) return cudaErrorInvalidValue;
  p.part = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(ws) + kWsCounterBytes);

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
  const int mt = tile_rows(M);
#define WQ_BAND_LAUNCH_F(F, EPIV)                                                                              \
  switch (mt) {                                                                                                \
    case 8: return launch_gemv_t<F, 8, EPIV>(tw, ts, tz, p, stream);                                           \
    case 16: return launch_gemv_t<F, 16, EPIV>(tw, ts, tz, p, stream);                                         \
    default: return launch_gemv_t<F, 32, EPIV>(tw, ts, tz, p, stream);                                         \
  }
#define WQ_BAND_LAUNCH(EPIV)                                                                                   \
  if (fmt == kInt4G128) { WQ_BAND_LAUNCH_F(kInt4G128, EPIV) }                                                  \
  WQ_BAND_LAUNCH_F(kMxfp4, EPIV)
  if (epi == kEpiSwiglu) { WQ_BAND_LAUNCH(kEpiSwiglu) }
  if (epi == kEpiSplit3) { WQ_BAND_LAUNCH(kEpiSplit3) }
  WQ_BAND_LAUNCH(kEpiNone)
#undef WQ_BAND_LAUNCH
#undef WQ_BAND_LAUNCH_F
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
// The split-K exchange area of the decode kernel lives here in one fixed, library-owned
// device array instead of a caller-provided workspace, in the workspace layout (64 KiB header
// of tensor-core counters, unused here, then the exchange area).  It is sized for every
// decode shape the kernel accepts (M <= 16, N <= 2097152) on a device with at most
// gemv::kMaxCtas CTAs: 64 KiB + 5 MiB.  It starts zeroed (a __device__ array), and every
// call that completes leaves it at zero.  Every GPU that loads the library keeps this array
// until the process exits.
// ---------------------------------------------------------------------------------------
constexpr size_t kNoAllocScratchBytes =
    kWsCounterBytes + 2 * static_cast<size_t>(gemv::kMaxCtas) * 16 * gemv::kBand * sizeof(uint32_t);

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

static void noalloc_scratch_reset() {
  void* a = nullptr;
  if (cudaGetSymbolAddress(&a, g_noalloc_scratch) != cudaSuccess) return;
  if (cudaMemset(a, 0, kNoAllocScratchBytes) == cudaSuccess) cudaDeviceSynchronize();
}

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
  return launch_gemv(fmt, X, M, K, N, Wq, scales, zeros, Y, scratch, kNoAllocScratchBytes, stream);
}

}  // namespace wq
