// Trellis decode-and-multiply GEMV for 1..16 tokens, plus the whole-matrix
// decode entry and the bounded-wait self test.
//
// y_pre[m, n] = sum_k xh[m, k] * W_inner[k, n], with W_inner never
// materialised: each 16x16 tile is decoded in registers from its trellis words
// ("The escha W2 format, recovered and verified", sections "Bit layout" and
// "Codebook: cb=1") and fed to the tensor cores.
//
// Kernel layout (persistent, several CTAs per SM):
//   warp 8      producer: one thread streams each unit's row of 8 tiles
//               (8 x 32*bits bytes, contiguous in HBM) and the matching
//               activation fragments into a shared-memory ring with 1-D bulk
//               copies (TMA engine), completing on mbarriers.
//   warps 0..7  consumers: warp w owns output tile column w of the current
//               128-channel group.  Per unit it reads its tile's two words per
//               lane, decodes eight weights per lane, and issues m16n8k16 MMAs
//               with the weight tile as A (rows = output channels) and up to 8
//               tokens as B; a second token block handles 9..16 tokens.
// Each A register holds one weight's codebook word as its two fp16 halves
// (lo, hi) and B carries the activation in both halves, so the MMA forms
// lo*x + hi*x in fp32: the codebook's final addition happens inside the
// contraction instead of as a separate fp16 add (which costs more integer and
// FMA-pipe instructions than the rest of the decode step).  The sum is not
// rounded to fp16 first; that changes each weight by at most half an fp16 ulp
// (relative RMS 2.2e-4 over uniform states).  Each MMA contracts 8 real input
// channels and two MMAs cover a tile.

#include "common.cuh"
#include "internal.h"
#include "trellis_decode.cuh"

#include <algorithm>

namespace escha {

namespace {

constexpr int kUPS = 8;     // units per pipeline stage
constexpr int kStages = 4;  // ring depth
constexpr int kCW = 8;      // consumer warps = tiles per unit
constexpr int kThreads = (kCW + 1) * 32;
constexpr int kCodeStageBytes = kUPS * kCW * 128;  // sized for bits = 4

template <int TB>
__host__ __device__ constexpr int xf_stage_bytes() {
  return kUPS * TB * 512;
}
template <int TB>
__host__ __device__ constexpr int gemv_smem_bytes() {
  return kStages * (kCodeStageBytes + xf_stage_bytes<TB>()) + 2 * kStages * 8;
}

struct GemvArgs {
  const GemvJob* jobs;
  long long units;
  int grid;
  const long long* dev_units;  // when set, units and grid are read from device memory
  const int* dev_grid;         // (a schedule built on the device, e.g. by MoE routing)
  int M;
  int mpad;
  int* err;
  uint64_t limit_ns;
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
  const uint4* xfrag;
  float* part;
  long long ub, ue;
  int bits, KT, NG, N;

  __device__ __forceinline__ void load(const GemvJob* jobs) {
    const GemvJob& J = jobs[j];
    code = J.code;
    xfrag = J.xfrag;
    part = J.part;
    ub = J.unit_begin;
    bits = J.bits;
    KT = J.KT;
    NG = J.NG;
    N = J.N;
    ue = ub + (long long)KT * NG;
  }
  __device__ __forceinline__ void init(const GemvJob* jobs, long long begin, long long end) {
    u = begin;
    u1 = end;
    j = 0;
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
  __device__ __forceinline__ bool next(const GemvJob* jobs, Chunk& ch) {
    if (u >= u1) return false;
    while (u >= ue) {  // entered the next job: it starts at its group 0, k-tile 0
      ++j;
      load(jobs);
      g = 0;
      kt = 0;
    }
    const long long left = u1 - u;
    int n = KT - kt;
    if (n > kUPS) n = kUPS;
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

template <int BITS, int TB>
__device__ __forceinline__ void consume_unit(const uint32_t* p0, const uint32_t* p1, const uint4* xp,
                                             int sh7, uint32_t mask, uint32_t xr,
                                             float (&acc)[TB][4]) {
  uint32_t h[8];
  decode8_pairs<BITS>(*p0, *p1, sh7, mask, xr, h);
#pragma unroll
  for (int tb = 0; tb < TB; ++tb) {
    const uint4 xf = xp[tb * 32];
    mma16816(acc[tb], h[0], h[4], h[2], h[6], xf.x, xf.y);
    mma16816(acc[tb], h[1], h[5], h[3], h[7], xf.z, xf.w);
  }
}

// One stage: n units (k-tile rows of 8 tiles); this warp owns tile column w.
template <int BITS, int TB>
__device__ __forceinline__ void consume_chunk(const uint8_t* codes_s, const uint4* xf_s, int n,
                                              int w, int lane, uint32_t mask, uint32_t xr,
                                              float (&acc)[TB][4]) {
  constexpr int T = 32 * BITS;
  constexpr int kRowWords = kCW * T / 4;  // uint32 words per unit in the stage
  const LaneWindow lw = lane_window<BITS>(lane);
  const uint32_t* base = reinterpret_cast<const uint32_t*>(codes_s + w * T);
  const uint32_t* p0 = base + lw.i0;
  const uint32_t* p1 = base + lw.i1;
  const uint4* xp = xf_s + lane;
  if (n == kUPS) {
#pragma unroll
    for (int i = 0; i < kUPS; ++i)
      consume_unit<BITS, TB>(p0 + i * kRowWords, p1 + i * kRowWords, xp + i * TB * 32, lw.sh7,
                             mask, xr, acc);
  } else {
    for (int i = 0; i < n; ++i)
      consume_unit<BITS, TB>(p0 + i * kRowWords, p1 + i * kRowWords, xp + i * TB * 32, lw.sh7,
                             mask, xr, acc);
  }
}

template <int TB>
__global__ void __launch_bounds__(kThreads, 3) trellis_gemv_kernel(const GemvArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* codes = smem;
  uint8_t* xfs = smem + kStages * kCodeStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(xfs + kStages * xf_stage_bytes<TB>());
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  pdl_trigger();
  long long U = a.units;
  int G = a.grid;
  if (a.dev_units != nullptr) {
    U = *a.dev_units;
    G = *a.dev_grid;
  }
  if (static_cast<int>(blockIdx.x) >= G) return;  // launched for the worst case; not needed

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&bars[s]), 1);              // full: producer + tx bytes
      mbar_init(smem_u32(&bars[kStages + s]), kCW);  // empty: one arrive per consumer warp
    }
    fence_mbar_init();
  }
  __syncthreads();

  const int c = blockIdx.x;
  ChunkIter it;
  it.init(a.jobs, cta_start(c, U, G), cta_start(c + 1, U, G));
  Chunk ch;

  if (warp == kCW) {
    // ------------------------------------------------------------ producer
    if (lane != 0) return;
    const uint64_t pol = policy_evict_first();
    int stage = 0;
    uint32_t phase = 0;
    int armed[kStages];
    for (int s = 0; s < kStages; ++s) armed[s] = -1;
    bool ok = true;
    bool waited = false;
    while (it.next(a.jobs, ch)) {
      const uint32_t full = smem_u32(&bars[stage]);
      if (!mbar_wait(smem_u32(&bars[kStages + stage]), phase ^ 1u, a.limit_ns)) {
        set_error(a.err, kDevErrTimeout);
        ok = false;
        break;
      }
      const int T = 32 * it.bits;
      const int rowb = kCW * T;
      const size_t NT = (size_t)it.NG * kCW;
      const uint32_t bytes = ch.n * rowb + ch.n * TB * 512;
      mbar_arrive_expect_tx(full, bytes);
      const uint32_t cdst = smem_u32(codes + stage * kCodeStageBytes);
      for (int i = 0; i < ch.n; ++i) {
        const uint8_t* src = it.code + ((size_t)(ch.kt + i) * NT + (size_t)kCW * ch.g) * T;
        bulk_g2s_evict_first(cdst + i * rowb, src, rowb, full, pol);
      }
      if (!waited) {
        // The code words above do not depend on the previous kernel; the
        // rotated activations do.
        pdl_wait();
        waited = true;
      }
      bulk_g2s(smem_u32(xfs + stage * xf_stage_bytes<TB>()), it.xfrag + (size_t)ch.kt * TB * 32,
               ch.n * TB * 512, full);
      armed[stage] = static_cast<int>(phase);
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (!ok) {
      // Let every copy already issued land before the CTA's shared memory goes away.
      for (int s = 0; s < kStages; ++s)
        if (armed[s] >= 0) mbar_wait(smem_u32(&bars[s]), static_cast<uint32_t>(armed[s]), a.limit_ns);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  float acc[TB][4];
#pragma unroll
  for (int tb = 0; tb < TB; ++tb)
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[tb][q] = 0.f;
  int stage = 0;
  uint32_t phase = 0;
  while (it.next(a.jobs, ch)) {
    if (!mbar_wait(smem_u32(&bars[stage]), phase, a.limit_ns)) {
      set_error(a.err, kDevErrTimeout);
      break;
    }
    const uint8_t* cs = codes + stage * kCodeStageBytes;
    const uint4* xs = reinterpret_cast<const uint4*>(xfs + stage * xf_stage_bytes<TB>());
    switch (it.bits) {
      case 2: consume_chunk<2, TB>(cs, xs, ch.n, warp, lane, a.cb_mask, a.cb_xor, acc); break;
      case 3: consume_chunk<3, TB>(cs, xs, ch.n, warp, lane, a.cb_mask, a.cb_xor, acc); break;
      default: consume_chunk<4, TB>(cs, xs, ch.n, warp, lane, a.cb_mask, a.cb_xor, acc); break;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&bars[kStages + stage]));
    if (++stage == kStages) {
      stage = 0;
      phase ^= 1u;
    }
    if (ch.seg_end) {
      const long long gb = it.ub + (long long)ch.g * it.KT;
      const int slot = c - cta_of_unit(gb, U, G);
      const int n0 = 128 * ch.g + 16 * warp + (lane >> 2);
      const int t2 = 2 * (lane & 3);
#pragma unroll
      for (int tb = 0; tb < TB; ++tb) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int tok = 8 * tb + t2 + q;
          if (tok < a.M) {
            float* row = it.part + ((size_t)slot * a.mpad + tok) * it.N;
            row[n0] = acc[tb][q];
            row[n0 + 8] = acc[tb][2 + q];
          }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[tb][q] = 0.f;
      }
    }
  }
}

// One warp per tile: writes W_inner[16i + r][16j + c] in fp16.
template <int BITS>
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
  decode8<BITS>(tw[lw.i0], tw[lw.i1], lw.sh7, h);
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

template <int TB>
cudaError_t launch_gemv_tb(const GemvSchedule& s, int M, int* err, cudaStream_t st) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(trellis_gemv_kernel<TB>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         gemv_smem_bytes<TB>());
    if (e != cudaSuccess) return e;
    configured = true;
  }
  GemvArgs a;
  a.jobs = s.d_jobs;
  a.units = s.units;
  a.grid = s.grid;
  a.dev_units = nullptr;
  a.dev_grid = nullptr;
  a.M = M;
  a.mpad = kGemvMaxTokens;
  a.err = err;
  a.limit_ns = kWaitLimitNs;
  a.cb_mask = kMcgMask;
  a.cb_xor = kMcgXor;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(s.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = gemv_smem_bytes<TB>();
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, trellis_gemv_kernel<TB>, a);
}

}  // namespace

int gemv_ctas_per_sm() {
  int n = 0;
  if (cudaFuncSetAttribute(trellis_gemv_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           gemv_smem_bytes<2>()) != cudaSuccess)
    return 1;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, trellis_gemv_kernel<2>, kThreads,
                                                    gemv_smem_bytes<2>()) != cudaSuccess)
    return 1;
  return std::max(1, n);
}

void plan_gemv(GemvSchedule& s, int num_sms, int ctas_per_sm) {
  long long u = 0;
  for (auto& j : s.jobs) {
    j.unit_begin = u;
    u += (long long)j.KT * j.NG;
  }
  s.units = u;
  long long g = std::min<long long>((long long)num_sms * ctas_per_sm,
                                    std::max<long long>(1, u / kMinUnitsPerCta));
  s.grid = static_cast<int>(std::max<long long>(1, g));
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
  if (M <= 8) return launch_gemv_tb<1>(s, M, err, st);
  return launch_gemv_tb<2>(s, M, err, st);
}

cudaError_t launch_gemv_device_schedule(const GemvJob* d_jobs, const long long* d_units,
                                        const int* d_grid, int max_grid, int M, int mpad,
                                        int* err, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(trellis_gemv_kernel<1>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       gemv_smem_bytes<1>());
  if (e != cudaSuccess) return e;
  GemvArgs a;
  a.jobs = d_jobs;
  a.units = 0;
  a.grid = max_grid;
  a.dev_units = d_units;
  a.dev_grid = d_grid;
  a.M = M;
  a.mpad = mpad;
  a.err = err;
  a.limit_ns = kWaitLimitNs;
  a.cb_mask = kMcgMask;
  a.cb_xor = kMcgXor;
  trellis_gemv_kernel<1><<<max_grid, kThreads, gemv_smem_bytes<1>(), st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_decode(const int16_t* code, int bits, int K, int N, uint16_t* w,
                          cudaStream_t st) {
  const int KT = K / 16, NT = N / 16;
  const long long tiles = (long long)KT * NT;
  const int wpb = 8;
  const unsigned blocks = static_cast<unsigned>((tiles + wpb - 1) / wpb);
  const uint8_t* c = reinterpret_cast<const uint8_t*>(code);
  switch (bits) {
    case 2: trellis_decode_kernel<2><<<blocks, 32 * wpb, 0, st>>>(c, w, KT, NT); break;
    case 3: trellis_decode_kernel<3><<<blocks, 32 * wpb, 0, st>>>(c, w, KT, NT); break;
    default: trellis_decode_kernel<4><<<blocks, 32 * wpb, 0, st>>>(c, w, KT, NT); break;
  }
  return cudaGetLastError();
}

cudaError_t launch_wait_selftest(int* err, uint64_t limit_ns, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(err, limit_ns);
  return cudaGetLastError();
}

}  // namespace escha
