// Trellis decode-and-multiply GEMV for 1..16 tokens, plus the whole-matrix
// decode entry and the bounded-wait self test.
//
// y_pre[m, n] = sum_k xh[m, k] * W_inner[k, n], with W_inner never
// materialised: each 16x16 tile is decoded in registers from its trellis words
// ("The escha W2 format, recovered and verified", sections "Bit layout" and
// "Codebook: cb=1") and fed to the tensor cores.
//
// Kernel layout (persistent, one CTA per SM):
//   warps 0..2  producers, one per consumer group: stream each stage's code
//               words (16 k-tile rows x 8 tile columns, one 2-D TMA copy) and
//               the matching activation fragments into the group's stages of
//               a shared-memory ring, completing on mbarriers.
//   warps 3..26 consumers, three groups of eight.  Each group owns one of the
//               launch's contiguous unit ranges (CTA b of C: ranges b, b + C,
//               b + 2C) and three ring stages (four when every job is 2-bit,
//               two with 9..16 tokens); in a
//               group, warp w owns output tile column w of the current
//               128-channel group.  Per unit it reads its tile's two words per
//               lane, decodes eight weights per lane, and issues m16n8k16 MMAs
//               with the weight tile as A (rows = output channels) and up to 8
//               tokens as B (E4M3-rounded weights: one weight per half and
//               one MMA per tile); a second token block handles 9..16 tokens.
// The three groups share one CTA rather than running as three CTAs per SM:
// separate CTAs on one SM drift apart (the warp scheduler favours the oldest
// CTA, whose ring runs ahead while the youngest one's work piles up at the end
// of the launch, when the SM is no longer busy).  A TMA copy costs the issuing
// thread a roughly fixed time however small it is, so each full stage is one
// 2-D copy of 8-16 KB.
#include "common.cuh"
#include "internal.h"
#include "tensor_map.h"
#include "trellis_decode.cuh"

#include <algorithm>

namespace escha {

namespace {

constexpr int kUPS = 16;    // units per pipeline stage
constexpr int kCW = 8;      // consumer warps per group = tiles per unit
constexpr int kGroups = 3;  // consumer groups = unit ranges per CTA
// Storage layouts a launch can serve, fixed at compile time (see below).
constexpr int kModeWhole = kGemvWhole;
constexpr int kModeColHalves = kGemvColHalves;
constexpr int kModeRowHalves = kGemvRowHalves;

// Per layout, measured: whole matrices and experts' column halves run best
// with one producer warp per consumer group and, with one token block, three
// ring stages per group (216 KB); experts stored by input halves (a 2-D copy
// per half-unit, a tensor map acquired per half) with one producer warp (a
// lane per group) and two stages per group.  Stage s serves group s % kGroups.
template <int MODE>
__host__ __device__ constexpr int producer_warps() {
  return MODE == kModeRowHalves ? 1 : kGroups;
}
// NARROW (one token block): every job of the launch is 2 bits wide, so a
// stage's code words take half the bytes and the ring has 12 stages (four per
// group) in less memory; measured 1.2 % faster on 2-bit layers.  (With two
// token blocks a 9-stage narrow ring measured no faster than six stages.)
template <int TB, int MODE, bool NARROW = false>
__host__ __device__ constexpr int stages_for() {
  return MODE == kModeRowHalves ? 6 : TB == 1 ? (NARROW && MODE == kModeWhole ? 12 : 9) : 6;
}
constexpr int kConsumers = kCW * kGroups * 32;
template <int MODE>
__host__ __device__ constexpr int threads_for() {
  return kConsumers + 32 * producer_warps<MODE>();
}
// A stage's code words: sized for 4 bits, or for 2 in a NARROW launch.
template <bool NARROW = false>
__host__ __device__ constexpr int code_stage_bytes() {
  return kUPS * kCW * (NARROW ? 64 : 128);
}
static_assert(stages_for<1, kModeWhole>() % kGroups == 0 &&
                  stages_for<2, kModeWhole>() % kGroups == 0 &&
                  stages_for<1, kModeWhole, true>() % kGroups == 0 &&
                  stages_for<1, kModeColHalves>() % kGroups == 0,
              "a stage must always serve the same group");

// Activation fragments of a stage: kUPS units x M tokens x 64 bytes (M <= 8 TB).
template <int TB>
__host__ __device__ constexpr int xf_stage_bytes() {
  return kUPS * TB * 512;
}
template <int TB, int MODE, bool NARROW = false>
__host__ __device__ constexpr int gemv_smem_bytes() {
  return stages_for<TB, MODE, NARROW>() * (code_stage_bytes<NARROW>() + xf_stage_bytes<TB>()) +
         2 * stages_for<TB, MODE, NARROW>() * 8;
}
static_assert(gemv_smem_bytes<1, kModeWhole, true>() <= 227 * 1024 &&
                  gemv_smem_bytes<1, kModeWhole>() <= 227 * 1024,
              "ring fits shared memory");

constexpr int kInlineJobs = 2;

struct GemvArgs {
  const GemvJob* jobs;             // job table in device memory, unless n_inline > 0
  GemvJob inline_jobs[kInlineJobs];  // host-scheduled launches carry their jobs here,
  int n_inline;                      // read from parameter space (no memory round trip)
  long long units;
  long long job_units;         // > 0: every job has this many units (direct job lookup)
  int grid;                    // unit ranges (kGroups per CTA)
  const long long* dev_units;  // when set, units and grid are read from device memory
  const int* dev_grid;         // (a schedule built on the device, e.g. by MoE routing)
  int M;
  int mpad;
  int* err;
  uint64_t limit_ns;
  int maps_from_device;  // tensor maps were written by a kernel: fence before first use
  uint32_t cb_mask;  // kMcgMask and kMcgXor, as run-time values (see mcg_pair)
  uint32_t cb_xor;
};

__host__ __device__ __forceinline__ long long cta_start(long long c, long long U, int G) {
  return (c * U) / G;
}
__host__ __device__ __forceinline__ int cta_of_unit(long long u, long long U, int G) {
  return static_cast<int>(((u + 1) * G - 1) / U);
}

struct Chunk {
  int g, kt, n;
  bool seg_end;
};

// Walks a CTA's unit range in pipeline-stage chunks that never cross a
// (job, group) boundary.  The current job's fields and the (group, k-tile)
// position are kept in registers and advanced incrementally (one division at
// start-up only).
struct ChunkIter {
  long long u, u1;
  int j;
  int g, kt;
  // cached job
  const uint8_t* code;
  const CUtensorMap* tmap;
  const uint4* xfrag;
  float* part;
  long long ub, ue;
  int bits, KT, NG, N;
  int e4m3;
  const CUtensorMap* row_maps;

  __device__ __forceinline__ void load(const GemvJob* jobs) {
    const GemvJob& J = jobs[j];
    code = J.code;
    tmap = J.tmap;
    xfrag = J.xfrag;
    part = J.part;
    ub = J.unit_begin;
    bits = J.bits;
    KT = J.KT;
    NG = J.NG;
    N = J.N;
    e4m3 = J.e4m3;
    row_maps = J.row_maps;
    ue = ub + (long long)KT * NG;
  }
  __device__ __forceinline__ void init(const GemvJob* jobs, long long begin, long long end,
                                       long long job_units) {
    u = begin;
    u1 = end;
    // Launches with many equal jobs (routed experts by halves: thousands)
    // find the first job by division; the scan below then does not move.
    j = (job_units > 0 && u < u1) ? static_cast<int>(u / job_units) : 0;
    load(jobs);
    if (u >= u1) {  // empty range: nothing to walk
      g = kt = 0;
      return;
    }
    while (u >= ue) {
      ++j;
      load(jobs);
    }
    const long long rel = u - ub;
    g = static_cast<int>(rel / KT);
    kt = static_cast<int>(rel - (long long)g * KT);
  }
  // The next segment: the units of the range in the current (job, group),
  // from the current position on.
  __device__ __forceinline__ bool next_segment(const GemvJob* jobs, Chunk& ch) {
    if (u >= u1) return false;
    while (u >= ue) {  // entered the next job: it starts at its group 0, k-tile 0
      ++j;
      load(jobs);
      g = 0;
      kt = 0;
    }
    const long long left = u1 - u;
    int n = KT - kt;
    if ((long long)n > left) n = static_cast<int>(left);
    ch.g = g;
    ch.kt = kt;
    ch.n = n;
    ch.seg_end = true;
    u += n;
    kt += n;
    if (kt == KT) {
      kt = 0;
      ++g;
    }
    return true;
  }
  // The next stage-sized chunk (the producer's walk; within a segment it
  // splits the units exactly as the consumers' run_segment does).
  // rpu: the launch's k-tile rows per unit (1 or 8).
  __device__ __forceinline__ bool next(const GemvJob* jobs, Chunk& ch, int rpu) {
    if (u >= u1) return false;
    while (u >= ue) {  // entered the next job: it starts at its group 0, k-tile 0
      ++j;
      load(jobs);
      g = 0;
      kt = 0;
    }
    const long long left = u1 - u;
    // A unit of a matrix stored by input halves is 8 k-tile rows (rpu = 8):
    // two of them fill a stage.
    const int cap = rpu > 1 ? kUPS / 8 : kUPS;
    int n = KT - kt;
    if (n > cap) n = cap;
    if ((long long)n > left) n = static_cast<int>(left);
    ch.g = g;
    ch.kt = kt;
    ch.n = n;
    ch.seg_end = (kt + n == KT) || ((long long)n == left);
    u += n;
    kt += n;
    if (kt == KT) {
      kt = 0;
      ++g;
    }
    return true;
  }
};

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// One unit of this warp's tile column: decode the lane's eight codebook words
// and contract them with the unit's activation fragments.  xq[tb] points at
// the lane's fragment of token block tb in this unit.
template <int BITS, int TB, bool E4M3>
__device__ __forceinline__ void consume_unit(const uint32_t* p0, const uint32_t* p1,
                                             const uint4* const (&xq)[TB], int sh7, uint32_t mask,
                                             uint32_t xr, float (&acc)[TB][4]) {
  if (E4M3) {
    // E4M3 weights as plain fp16 A fragments (one weight per half): one MMA
    // per tile against (x[2t], x[2t+1]) and (x[2t+8], x[2t+9]), taken from
    // the repeated-activation fragment words by one byte permute each
    uint32_t fa[4];
    decode8_e4m3_frag<BITS>(*p0, *p1, sh7, mask, xr, fa);
#pragma unroll
    for (int tb = 0; tb < TB; ++tb) {
      const uint4 xf = *xq[tb];
      mma16816(acc[tb], fa[0], fa[1], fa[2], fa[3], __byte_perm(xf.x, xf.z, 0x5410),
               __byte_perm(xf.y, xf.w, 0x5410));
    }
    return;
  }
  uint32_t h[8];
  decode8_pairs<BITS>(*p0, *p1, sh7, mask, xr, h);
#pragma unroll
  for (int tb = 0; tb < TB; ++tb) {
    const uint4 xf = *xq[tb];
    mma16816(acc[tb], h[0], h[4], h[2], h[6], xf.x, xf.y);
    mma16816(acc[tb], h[1], h[5], h[3], h[7], xf.z, xf.w);
  }
}

// A consumer group's view of its ring stages (stage s serves group s % kGroups).
struct GroupRing {
  const uint8_t* codes;  // stage code words, code_stage_bytes() each
  const uint8_t* xfs;    // stage activation fragments
  uint64_t* bars;        // [0, S): full barriers; [S, 2S): empty barriers
  int q;                 // group
  int slot;              // next stage index within the group's stages
  uint32_t phase;
};

// One segment: n consecutive units of one job and one 128-channel output
// group, streamed through the group's stages (kUPS k-tile rows per full
// stage); this warp owns tile column wt.  Everything that does not change
// from stage to stage (the lane's word offsets, its funnel shift, its
// activation-fragment offsets) is set up once per segment.  The stage holds
// fragments for the M real tokens only; a lane whose token (8 tb + g) is at or
// past M reads token M-1's fragment instead: MMA output column g depends on B
// column g alone, and those columns are never stored.  MC > 0: the token
// count is the compile-time MC (fragment addresses become immediate offsets).
// Returns false if a bounded wait ran out.
template <int BITS, int TB, bool E4M3, int MC, int STAGES, int RPU, int CSB>
__device__ __forceinline__ bool run_segment(GroupRing& rg, int n, int wt, int lane, int M_rt,
                                            const GemvArgs& a, float (&acc)[TB][4]) {
  const int M = MC > 0 ? MC : M_rt;
  constexpr int T = 32 * BITS;            // bytes per tile
  constexpr int kRowWords = kCW * T / 4;  // uint32 words per k-tile row of the stage
  constexpr int cap = kUPS / RPU;         // units per full stage
  const LaneWindow lw = lane_window<BITS>(lane);
  const int o0 = wt * (T / 4) + lw.i0;
  const int o1 = wt * (T / 4) + lw.i1;
  const int g = lane >> 2;
  const int xstride = 4 * M;  // uint4 per k-tile row
  int xo[TB];
#pragma unroll
  for (int tb = 0; tb < TB; ++tb) xo[tb] = 4 * min(8 * tb + g, M - 1) + (lane & 3);
  const uint32_t mask = a.cb_mask, xr = a.cb_xor;
  for (int left = n; left > 0;) {
    const int nu = left < cap ? left : cap;
    const int stage = rg.q + kGroups * rg.slot;
    // warp-uniform: the MMAs below need every lane
    if (!__all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&rg.bars[stage]), rg.phase, a.limit_ns)))
      return false;
    const uint32_t* cw = reinterpret_cast<const uint32_t*>(rg.codes + stage * CSB);
    const uint4* xs = reinterpret_cast<const uint4*>(rg.xfs + stage * xf_stage_bytes<TB>());
    const uint32_t* p0 = cw + o0;
    const uint32_t* p1 = cw + o1;
    const uint4* xq[TB];
#pragma unroll
    for (int tb = 0; tb < TB; ++tb) xq[tb] = xs + xo[tb];
    const int rows = nu * RPU;
    if (rows == kUPS) {
#pragma unroll
      for (int i = 0; i < kUPS; ++i) {
        consume_unit<BITS, TB, E4M3>(p0 + i * kRowWords, p1 + i * kRowWords, xq, lw.sh7, mask, xr,
                                     acc);
#pragma unroll
        for (int tb = 0; tb < TB; ++tb) xq[tb] += xstride;
      }
    } else {
      for (int i = 0; i < rows; ++i) {
        consume_unit<BITS, TB, E4M3>(p0 + i * kRowWords, p1 + i * kRowWords, xq, lw.sh7, mask, xr,
                                     acc);
#pragma unroll
        for (int tb = 0; tb < TB; ++tb) xq[tb] += xstride;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&rg.bars[STAGES + stage]));
    if (++rg.slot == STAGES / kGroups) {
      rg.slot = 0;
      rg.phase ^= 1u;
    }
    left -= nu;
  }
  return true;
}

// The segment's decode at its width and rounding (key = bits + 8 * e4m3).
// F16_ONLY: the launch holds no E4M3-rounded job, so only the three fp16
// decodes are compiled in; NARROW: only the 2-bit one.
template <int TB, int MC, int STAGES, int RPU, bool F16_ONLY, bool NARROW>
__device__ __forceinline__ bool segment_dispatch(int key, GroupRing& rg, int n, int wt, int lane,
                                                 int M, const GemvArgs& a, float (&acc)[TB][4]) {
  constexpr int CSB = code_stage_bytes<NARROW>();
  if (NARROW) return run_segment<2, TB, false, MC, STAGES, RPU, CSB>(rg, n, wt, lane, M, a, acc);
  if (F16_ONLY) {
    switch (key) {
      case 2: return run_segment<2, TB, false, MC, STAGES, RPU, CSB>(rg, n, wt, lane, M, a, acc);
      case 3: return run_segment<3, TB, false, MC, STAGES, RPU, CSB>(rg, n, wt, lane, M, a, acc);
      default: return run_segment<4, TB, false, MC, STAGES, RPU, CSB>(rg, n, wt, lane, M, a, acc);
    }
  }
  switch (key) {
    case 2: return run_segment<2, TB, false, MC, STAGES, RPU, CSB>(rg, n, wt, lane, M, a, acc);
    case 3: return run_segment<3, TB, false, MC, STAGES, RPU, CSB>(rg, n, wt, lane, M, a, acc);
    case 4: return run_segment<4, TB, false, MC, STAGES, RPU, CSB>(rg, n, wt, lane, M, a, acc);
    case 10: return run_segment<2, TB, true, MC, STAGES, RPU, CSB>(rg, n, wt, lane, M, a, acc);
    case 11: return run_segment<3, TB, true, MC, STAGES, RPU, CSB>(rg, n, wt, lane, M, a, acc);
    default: return run_segment<4, TB, true, MC, STAGES, RPU, CSB>(rg, n, wt, lane, M, a, acc);
  }
}

// Launch modes, fixed at compile time so that the dense path's code is not
// shaped by the other two: kModeWhole, matrices stored whole (2-D tensor-map
// stage copies); kModeColHalves, every job is one 128-channel column half
// whose stage rows are contiguous (one 1-D bulk copy); kModeRowHalves, every
// job is stored by input halves (one unit = 8 k-tile rows, one 2-D copy per
// unit through the half's tensor map).
template <int TB, int MODE, bool F16_ONLY, bool NARROW = false>
__global__ void __launch_bounds__(threads_for<MODE>(), 1)
    trellis_gemv_kernel(const __grid_constant__ GemvArgs a) {
  constexpr int RPU = MODE == kModeRowHalves ? 8 : 1;  // k-tile rows per unit
  const GemvJob* const jobs = a.n_inline > 0 ? a.inline_jobs : a.jobs;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* codes = smem;
  constexpr int kStages = stages_for<TB, MODE, NARROW>();
  constexpr int CSB = code_stage_bytes<NARROW>();
  constexpr int PW = producer_warps<MODE>();
  uint8_t* xfs = smem + kStages * CSB;
  uint64_t* bars = reinterpret_cast<uint64_t*>(xfs + kStages * xf_stage_bytes<TB>());
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  pdl_trigger();
  long long U = a.units;
  int G = a.grid;
  if (a.dev_units != nullptr) {
    // The schedule is written by the previous kernel (the routing plan).
    pdl_wait();
    U = *a.dev_units;
    G = *a.dev_grid;
  }
  // CTA b works unit ranges b, b + C, b + 2C (C = CTAs launched), one per group.
  const int C = static_cast<int>(gridDim.x);
  if (static_cast<int>(blockIdx.x) >= G) return;  // launched for the worst case; not needed

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&bars[s]), 1);              // full: producer + tx bytes
      mbar_init(smem_u32(&bars[kStages + s]), kCW);  // empty: one arrive per warp of its group
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp < PW) {
    // ------------------------------------------------------------ producers
    // Lane 0 of warp q walks range blockIdx.x + q*C and fills group q's
    // stages, independently of the other groups' producers.  A full stage is
    // one tensor copy, a partial one (end of a segment or of the range) one
    // copy per k-tile row.
    // one warp per group (lane 0), or one warp with a lane per group
    const int q = PW == 1 ? lane : warp;
    const int r = static_cast<int>(blockIdx.x) + q * C;
    const bool mine = (PW == 1 ? q < kGroups : lane == 0) && r < G;
    ChunkIter it;
    if (mine) it.init(jobs, cta_start(r, U, G), cta_start(r + 1, U, G), a.job_units);
    const uint64_t pol = policy_evict_first();
    int slot = 0;  // next stage index within the group's stages
    uint32_t phase = 0;
    int armed[kStages / kGroups];
#pragma unroll
    for (int s = 0; s < kStages / kGroups; ++s) armed[s] = -1;
    bool waited = false, ok = true;
    const CUtensorMap* fenced = nullptr;
    // halves of the current job whose tensor maps this thread has acquired
    // (each output group walks the same halves again)
    const CUtensorMap* half_job = nullptr;
    uint64_t half_fenced = 0;
    for (;;) {
      Chunk ch;
      const bool has = mine && ok && it.next(jobs, ch, RPU);
      if (!__any_sync(0xFFFFFFFFu, has)) break;
      if (!has) continue;
      const int stage = q + kGroups * slot;
      if (!mbar_wait(smem_u32(&bars[kStages + stage]), phase ^ 1u, a.limit_ns)) {
        set_error(a.err, kDevErrTimeout);
        ok = false;
        continue;
      }
      const uint32_t full = smem_u32(&bars[stage]);
      const int T = 32 * it.bits;
      const int rowb = kCW * T;
      const uint32_t cdst = smem_u32(codes + stage * CSB);
      const int rows = ch.n * RPU;  // k-tile rows of the stage
      const uint32_t xbytes = rows * a.M * 64;
      mbar_arrive_expect_tx(full, rows * rowb + xbytes);
      if (MODE == kModeRowHalves) {
        // stored by input halves: each unit is one half's 8 rows of group g,
        // one 2-D copy through that half's tensor map (written on the device)
        if (it.row_maps != half_job) {
          half_job = it.row_maps;
          half_fenced = 0;
        }
        for (int i = 0; i < ch.n; ++i) {
          const int h = ch.kt + i;
          const CUtensorMap* hm = it.row_maps + h;
          const uint64_t bit = h < 64 ? (1ull << h) : 0ull;
          if (!(half_fenced & bit)) {
            tensormap_acquire(hm);
            half_fenced |= bit;
          }
          tma_load_2d_hint(cdst + i * 8 * rowb, hm, ch.g * rowb / 4, 0, full, pol);
        }
      } else if (MODE == kModeColHalves) {
        // a single 128-channel group (a column half): the stage's rows are
        // contiguous, one bulk copy
        bulk_g2s_evict_first(cdst, it.code + (size_t)ch.kt * rowb, rows * rowb, full, pol);
      } else if (ch.n == kUPS) {
        if (a.maps_from_device && it.tmap != fenced) {
          tensormap_acquire(it.tmap);
          fenced = it.tmap;
        }
        tma_load_2d_hint(cdst, it.tmap, ch.g * rowb / 4, ch.kt, full, pol);
      } else {
        const size_t NT = (size_t)it.NG * kCW;
        for (int i = 0; i < ch.n; ++i) {
          const uint8_t* src = it.code + ((size_t)(ch.kt + i) * NT + (size_t)kCW * ch.g) * T;
          bulk_g2s_evict_first(cdst + i * rowb, src, rowb, full, pol);
        }
      }
      if (!waited) {
        // The code words above do not depend on the previous kernel; the
        // rotated activations do.
        pdl_wait();
        waited = true;
      }
      bulk_g2s(smem_u32(xfs + stage * xf_stage_bytes<TB>()),
               it.xfrag + (size_t)ch.kt * RPU * a.M * 4, xbytes, full);
      armed[slot] = static_cast<int>(phase);
      if (++slot == kStages / kGroups) {
        slot = 0;
        phase ^= 1u;
      }
    }
    // Every copy issued must land before the CTA's shared memory goes away
    // (on the normal path these waits return at once).
    if (mine)
#pragma unroll
      for (int s = 0; s < kStages / kGroups; ++s)
        if (armed[s] >= 0)
          mbar_wait(smem_u32(&bars[q + kGroups * s]), static_cast<uint32_t>(armed[s]), a.limit_ns);
    return;
  }

  // -------------------------------------------------------------- consumers
  const int q = (warp - PW) / kCW;       // group: unit range blockIdx.x + q*C
  const int wt = (warp - PW) - q * kCW;  // tile column within a unit
  const int r = static_cast<int>(blockIdx.x) + q * C;
  if (r >= G) return;
  ChunkIter it;
  it.init(jobs, cta_start(r, U, G), cta_start(r + 1, U, G), a.job_units);
  Chunk sg;
  float acc[TB][4];
#pragma unroll
  for (int tb = 0; tb < TB; ++tb)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[tb][i] = 0.f;
  GroupRing rg{codes, xfs, bars, q, 0, 0u};
  // The range walks its units as segments, one per (job, 128-channel group)
  // it touches; each ends with the group's partial sums for this range.
  while (it.next_segment(jobs, sg)) {
    const int key = it.bits + 8 * it.e4m3;
    // One token (the common decode case) and a full second token block are
    // specialised: the fragment offsets become immediates.
    bool ok;
    if (TB == 1 && a.M == 1)
      ok = segment_dispatch<TB, 1, kStages, RPU, F16_ONLY, NARROW>(key, rg, sg.n, wt, lane, 1, a,
                                                                   acc);
    else if (TB == 2 && MODE == kModeWhole && a.M == 16)
      ok = segment_dispatch<TB, 16, kStages, RPU, F16_ONLY, NARROW>(key, rg, sg.n, wt, lane, 16,
                                                                    a, acc);
    else
      ok = segment_dispatch<TB, 0, kStages, RPU, F16_ONLY, NARROW>(key, rg, sg.n, wt, lane, a.M,
                                                                   a, acc);
    if (!ok) {
      set_error(a.err, kDevErrTimeout);
      break;
    }
    const long long gb = it.ub + (long long)sg.g * it.KT;
    const int ps = r - cta_of_unit(gb, U, G);  // partial-sum slot
    const int n0 = 128 * sg.g + 16 * wt + (lane >> 2);
    const int t2 = 2 * (lane & 3);
#pragma unroll
    for (int tb = 0; tb < TB; ++tb) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int tok = 8 * tb + t2 + i;
        if (tok < a.M) {
          float* row = it.part + ((size_t)ps * a.mpad + tok) * it.N;
          row[n0] = acc[tb][i];
          row[n0 + 8] = acc[tb][2 + i];
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[tb][i] = 0.f;
    }
  }
}

// One warp per tile: writes W_inner[16i + r][16j + c] in fp16.
template <int BITS, bool E4M3>
__global__ void trellis_decode_kernel(const uint8_t* code, uint16_t* w, int KT, int NT) {
  constexpr int T = 32 * BITS;
  const long long tile = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (tile >= (long long)KT * NT) return;
  const int i = static_cast<int>(tile / NT);
  const int j = static_cast<int>(tile - (long long)i * NT);
  const LaneWindow lw = lane_window<BITS>(lane);
  const uint32_t* tw = reinterpret_cast<const uint32_t*>(code + tile * T);
  uint32_t h[8];
  decode8<BITS, E4M3>(tw[lw.i0], tw[lw.i1], lw.sh7, h);
  const size_t N = (size_t)NT * 16;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int r = sym_row(lane, q);
    const int cc = sym_col(lane, q);
    w[(size_t)(16 * i + r) * N + 16 * j + cc] = static_cast<uint16_t>(h[q] & 0xFFFFu);
  }
}

__global__ void wait_selftest_kernel(int* err, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // Nobody arrives: phase 0 never completes, so the bounded wait must give up.
    if (!mbar_wait(smem_u32(&bar), 0, limit_ns)) set_error(err, kDevErrTimeout);
  }
}

template <int TB, bool F16_ONLY, bool NARROW = false>
cudaError_t launch_gemv_tb(const GemvSchedule& s, int M, int* err, cudaStream_t st) {
  const auto kern = trellis_gemv_kernel<TB, kModeWhole, F16_ONLY, NARROW>;
  constexpr int smem = gemv_smem_bytes<TB, kModeWhole, NARROW>();
  cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  GemvArgs a;
  a.jobs = s.d_jobs;
  a.n_inline = 0;
  if (s.jobs.size() <= (size_t)kInlineJobs) {
    for (size_t j = 0; j < s.jobs.size(); ++j) a.inline_jobs[j] = s.jobs[j];
    a.n_inline = static_cast<int>(s.jobs.size());
  }
  a.units = s.units;
  a.job_units = 0;
  a.grid = s.grid;
  a.dev_units = nullptr;
  a.dev_grid = nullptr;
  a.M = M;
  a.mpad = kGemvMaxTokens;
  a.err = err;
  a.maps_from_device = s.maps_from_device ? 1 : 0;
  a.limit_ns = kWaitLimitNs;
  a.cb_mask = kMcgMask;
  a.cb_xor = kMcgXor;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(s.ctas);
  cfg.blockDim = dim3(threads_for<kModeWhole>());
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace

bool encode_gemv_code_map(CUtensorMap* map, const void* code, int bits, int KT, int NT) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return false;
  const cuuint64_t row_words = (cuuint64_t)NT * 8 * bits;  // a tile is 8*bits words
  const cuuint64_t dims[2] = {row_words, (cuuint64_t)KT};
  const cuuint64_t strides[1] = {row_words * 4};
  const cuuint32_t box[2] = {(cuuint32_t)(kCW * 8 * bits), (cuuint32_t)kUPS};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(code), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_gemv_half_map(CUtensorMap* map, const void* code, int bits, int NT) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return false;
  const cuuint64_t row_words = (cuuint64_t)NT * 8 * bits;
  const cuuint64_t dims[2] = {row_words, 8};
  const cuuint64_t strides[1] = {row_words * 4};
  const cuuint32_t box[2] = {(cuuint32_t)(kCW * 8 * bits), 8};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(code), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int gemv_ranges_per_sm() {
  int n = 0;
  if (cudaFuncSetAttribute(trellis_gemv_kernel<2, kModeWhole, false>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           gemv_smem_bytes<2, kModeWhole>()) != cudaSuccess)
    return kGroups;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, trellis_gemv_kernel<2, kModeWhole, false>,
                                                    threads_for<kModeWhole>(),
                                                    gemv_smem_bytes<2, kModeWhole>()) != cudaSuccess)
    return kGroups;
  return kGroups * std::max(1, n);
}

void plan_gemv(GemvSchedule& s, int num_sms, int ranges_per_sm) {
  long long u = 0;
  for (auto& j : s.jobs) {
    j.unit_begin = u;
    u += (long long)j.KT * j.NG;
  }
  s.units = u;
  long long g = std::min<long long>((long long)num_sms * ranges_per_sm,
                                    std::max<long long>(1, u / kMinUnitsPerCta));
  s.grid = static_cast<int>(std::max<long long>(1, g));
  s.ctas = std::min(s.grid, num_sms * std::max(1, ranges_per_sm / kGroups));
  int ms = 1;
  for (size_t j = 0; j < s.jobs.size(); ++j)
    for (int gg = 0; gg < s.jobs[j].NG; ++gg)
      ms = std::max(ms, gemv_slots_for_group(s, static_cast<int>(j), gg));
  s.max_slots = ms;
}

int gemv_slots_for_group(const GemvSchedule& s, int job, int g) {
  const GemvJob& J = s.jobs[job];
  const long long ub = J.unit_begin + (long long)g * J.KT;
  return cta_of_unit(ub + J.KT - 1, s.units, s.grid) - cta_of_unit(ub, s.units, s.grid) + 1;
}

cudaError_t launch_gemv(const GemvSchedule& s, int M, int* err, cudaStream_t st) {
  bool f16 = true, narrow = true;
  for (const GemvJob& j : s.jobs) {
    f16 = f16 && !j.e4m3;
    narrow = narrow && !j.e4m3 && j.bits == 2;
  }
  if (M <= 8) {
    if (narrow) return launch_gemv_tb<1, true, true>(s, M, err, st);
    return f16 ? launch_gemv_tb<1, true>(s, M, err, st) : launch_gemv_tb<1, false>(s, M, err, st);
  }
  return f16 ? launch_gemv_tb<2, true>(s, M, err, st) : launch_gemv_tb<2, false>(s, M, err, st);
}

cudaError_t launch_gemv_device_schedule(const GemvJob* d_jobs, const long long* d_units,
                                        const int* d_grid, int max_grid, int M, int mpad,
                                        int* err, cudaStream_t st, long long job_units,
                                        bool maps_from_device, int layout, bool e4m3) {
  auto kern = layout == kGemvColHalves
                  ? (e4m3 ? trellis_gemv_kernel<1, kModeColHalves, false>
                          : trellis_gemv_kernel<1, kModeColHalves, true>)
              : layout == kGemvRowHalves
                  ? (e4m3 ? trellis_gemv_kernel<1, kModeRowHalves, false>
                          : trellis_gemv_kernel<1, kModeRowHalves, true>)
                  : (e4m3 ? trellis_gemv_kernel<1, kModeWhole, false>
                          : trellis_gemv_kernel<1, kModeWhole, true>);
  const int smem = layout == kGemvColHalves   ? gemv_smem_bytes<1, kModeColHalves>()
                   : layout == kGemvRowHalves ? gemv_smem_bytes<1, kModeRowHalves>()
                                              : gemv_smem_bytes<1, kModeWhole>();
  const int threads = layout == kGemvColHalves   ? threads_for<kModeColHalves>()
                      : layout == kGemvRowHalves ? threads_for<kModeRowHalves>()
                                                 : threads_for<kModeWhole>();
  cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  GemvArgs a;
  a.jobs = d_jobs;
  a.n_inline = 0;
  a.units = 0;
  a.job_units = job_units;
  a.grid = max_grid;
  a.dev_units = d_units;
  a.dev_grid = d_grid;
  a.M = M;
  a.mpad = mpad;
  a.err = err;
  a.maps_from_device = maps_from_device ? 1 : 0;
  a.limit_ns = kWaitLimitNs;
  a.cb_mask = kMcgMask;
  a.cb_xor = kMcgXor;
  PdlLaunch pl((max_grid + kGroups - 1) / kGroups, threads, smem, st);
  return cudaLaunchKernelEx(&pl.cfg, kern, a);
}

cudaError_t launch_decode(const int16_t* code, int bits, bool e4m3, int K, int N, uint16_t* w,
                          cudaStream_t st) {
  const int KT = K / 16, NT = N / 16;
  const long long tiles = (long long)KT * NT;
  const int wpb = 8;
  const unsigned blocks = static_cast<unsigned>((tiles + wpb - 1) / wpb);
  const uint8_t* c = reinterpret_cast<const uint8_t*>(code);
  switch (bits + 8 * (e4m3 ? 1 : 0)) {
    case 2: trellis_decode_kernel<2, false><<<blocks, 32 * wpb, 0, st>>>(c, w, KT, NT); break;
    case 3: trellis_decode_kernel<3, false><<<blocks, 32 * wpb, 0, st>>>(c, w, KT, NT); break;
    case 4: trellis_decode_kernel<4, false><<<blocks, 32 * wpb, 0, st>>>(c, w, KT, NT); break;
    case 10: trellis_decode_kernel<2, true><<<blocks, 32 * wpb, 0, st>>>(c, w, KT, NT); break;
    case 11: trellis_decode_kernel<3, true><<<blocks, 32 * wpb, 0, st>>>(c, w, KT, NT); break;
    default: trellis_decode_kernel<4, true><<<blocks, 32 * wpb, 0, st>>>(c, w, KT, NT); break;
  }
  return cudaGetLastError();
}

cudaError_t launch_wait_selftest(int* err, uint64_t limit_ns, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(err, limit_ns);
  return cudaGetLastError();
}

}  // namespace escha
