// Prefill GEMM for trellis-coded layers on the 5th-generation tensor cores:
//   y[M, N] = fp16( had128( xh[M, K] @ W_inner[K, N] ) * sv ),  xh = had128(x * su)
// (activation-side reconstruction, "Escha-W2 runs on Metal"; decode as in
// "The escha W2 format, recovered and verified", "Bit layout" / "Codebook").
//
// Tiles are 512 x 128 (rows x output channels): four M=128 accumulators in
// TMEM (all 512 columns) share one decoded 128 x 64 B block per K step, so each
// weight is decoded once per 512 rows.  The kernel is persistent: the grid's
// CTAs split the (tile, K-block) units evenly and contiguously (stream-K).  A
// CTA whose range covers a whole tile runs the fused epilogue.  Where a tile is
// shared between CTAs, each decoder warp of each CTA either writes its rows'
// fp32 partial sums and counts itself in (a counter per tile and warp), or, if
// it is the last to get there, sums every CTA's partials in CTA order into its
// accumulators and runs the epilogue.  No CTA waits for another, and the sum
// does not depend on which CTA finishes.
//
// Warp roles (19 warps):
//   warp 0      A producer: TMA tiled loads of the 512 x 64 activation block
//               (two 256-row boxes, 128B swizzle, rows past M zero-filled)
//               into a 2-stage ring; at fp16 each box is reloaded as soon as
//               the two accumulators that read it are done.
//   warp 1      code producer: 1-D bulk copies of the block's 4 x 8 code tiles
//               into a 4-stage ring.
//   warp 2      owns TMEM; the whole warp walks the MMA loop (its waits and
//               descriptor arithmetic stay warp-uniform) and one elected lane
//               issues each block's tcgen05.mma kind::f16 (4 accumulators x 4
//               K16 steps) and the commits that free the rings.  Forming each
//               block's descriptors once and issuing from a converged warp
//               measured 14 % faster than issuing from a lone lane.
//   warps 3-18  decoders: two tiles per warp per block, decoded in registers
//               and stored as fp16 pairs into the canonical K-major 128B-swizzled
//               B layout (3-stage ring); then, per tile, the epilogue: the
//               128-point Hadamard over each row (the last two stages across
//               the four 32-column chunks through TMEM, then each chunk in
//               registers), * sv, fp16 stores -- or the raw fp32 partial sums.
//               fp16: the next segment's first two blocks are decoded before
//               the epilogue, and each warp frees TMEM after its last read.
// Every mbarrier wait is bounded; a wait that runs out sets the error word and
// the CTA unwinds (TMEM is always released, in-flight copies are drained).
// The kernel is launched as a programmatic dependent of the input rotation:
// setup, code streaming and the first decodes overlap the rotation's tail;
// the activation loads and the epilogue (which reads the FP8 scales and
// writes y) wait for it first (griddepcontrol.wait).
//
// FP8 variant (EXLR8 format page: weights rounded to E4M3 are exact FP8, so
// prefill can multiply on FP8 tensor cores).  The activations arrive as
// per-token E4M3 codes q with fp32 scales d (xh ~ q * d); a block is 128 K
// elements (still 128 bytes per row, so the swizzle, descriptors and ring
// sizes are unchanged), the MMA is kind::f8f6f4 with E4M3 A and B (K = 32 per
// instruction), each decoder warp decodes four tiles per block into E4M3
// bytes, and the epilogue multiplies each row by its d.

#include <cuda.h>
#include <cuda_runtime.h>

#include "act_layout.cuh"
#include "common.cuh"
#include "internal.h"
#include "tensor_map.h"
#include "trellis_decode.cuh"

namespace escha {

namespace {

constexpr int kBM = 512;          // rows per tile (four M=128 accumulators)
constexpr int kBN = 128;          // output channels per tile (= one Hadamard block)
constexpr int kRowBytes = 128;    // bytes of one operand row per K block
constexpr int kAStages = 2;
constexpr int kBStages = 3;
constexpr int kCStages = 4;
constexpr int kDecWarps = 16;
constexpr int kFirstDec = 3;
constexpr int kThreadsG = (kFirstDec + kDecWarps) * 32;  // 608
constexpr int kTmemCols = 512;

constexpr int kABytes = kBM * kRowBytes;  // 64 KB
constexpr int kBBytes = kBN * kRowBytes;  // 16 KB
constexpr int kOffB = kAStages * kABytes;

// Per-operand-type geometry: fp16 blocks are 64 K elements (4 k-tiles), E4M3
// blocks 128 (8 k-tiles); either way 128 bytes per operand row.
template <bool FP8>
struct BlockGeom {
  static constexpr int kKE = FP8 ? 128 : 64;           // K elements per block
  static constexpr int kKT = kKE / 16;                 // k-tiles per block
  static constexpr int kTilesPerWarp = kKT * 8 / kDecWarps;
  static constexpr int kCBytes = kKT * 8 * 128;        // code stage, sized for 4 bits
  static constexpr int kOffC = kOffB + kBStages * kBBytes;
  static constexpr int kOffBar = kOffC + kCStages * kCBytes;
  static constexpr int kOffSv = kOffBar + 256;  // per decoder warp: the tile's 128 output scales
  // fp16: each decoder warp stages its output rows in a 1 KB slot of its own,
  // so the decoded-B ring stays free during an epilogue and the decoders fill
  // kLookahead blocks of the next segment before it.  FP8 (no room) stages
  // them in the ring, which is idle during its epilogues.
  static constexpr int kOffScr = kOffSv + kDecWarps * kBN * 4;
  static constexpr int kLookahead = FP8 ? 0 : 2;
  static constexpr int kSmemBytes = kOffScr + (FP8 ? 0 : kDecWarps * 1024) + 1024;  // + slack
};
static_assert(BlockGeom<true>::kSmemBytes <= 227 * 1024, "FP8 ring does not fit");
static_assert(BlockGeom<false>::kSmemBytes <= 227 * 1024, "fp16 ring does not fit");

// barrier indices
// An activation stage has one full barrier and one empty barrier per 256-row
// half (index 2 * stage + half): at fp16 the half that accumulators 0 and 1
// read is refilled as soon as their MMAs are done (17408 -> 5120: 283.5 ->
// 266.6 us), while the MMA warp still waits once per stage; the FP8 route
// frees the whole stage at once (splitting measured 1 % slower there).
constexpr int kBarAFull = 0, kBarAEmpty = 2, kBarCFull = 6, kBarCEmpty = 10, kBarBFull = 14,
              kBarBEmpty = 17, kBarAcc = 20, kBarTmemFree = 21, kBarDrain = 22, kBarEpi = 23,
              kNumBars = 24;
static_assert((kNumBars + 2) * 8 <= 256, "barriers and the TMEM slot fit their 256 bytes");

struct GemmArgs {
  const uint8_t* code;
  const float* sv;
  const float* d;        // FP8: per-row activation scales [M]; else null
  uint32_t mcg_mask;     // the codebook's mask and flip words, passed at run time so
  uint32_t mcg_xor;      // that each state's mask-and-flip is one three-input logic op
  uint16_t* y;
  float* ws;             // partial sums: [grid][2][kBM][kBN] fp32
  int* tile_cnt;         // [tiles][kDecWarps] arrival counters, zero at launch
  int M, N, K;
  int n_blocks;          // N / kBN
  int kb_per_tile;       // K / (K elements per block)
  long long units;       // tiles * kb_per_tile
  int grid;
  int parts_last;        // walk each CTA's whole tiles before its shared parts (SegIter)
  int* err;
  uint64_t limit_ns;
};

__host__ __device__ __forceinline__ long long range_start(long long c, long long U, int G) {
  return (c * U) / G;
}

__host__ __device__ __forceinline__ int owner(long long u, long long U, int G) {
  return static_cast<int>(((u + 1) * G - 1) / U);
}

// ---------------------------------------------------------------- PTX wrappers

__device__ __forceinline__ void tmem_alloc(uint32_t smem_slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_slot),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// True in one lane of a converged warp (the same lane each time while the
// warp stays converged).
__device__ __forceinline__ bool elect_one() {
  uint32_t e;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "elect.sync _|p, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(e));
  return e != 0;
}

// D[tmem] (+)= A[smem desc] * B[smem desc], fp16 inputs, fp32 accumulate
// (one thread issues it).
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A * B with E4M3 A and B (K = 32 per instruction), fp32 accumulate.
__device__ __forceinline__ void mma_e4m3(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05 operation issued so far by this thread completes.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

// Lane-wise fp16 sum of two fp16 pairs (round to nearest even).
__device__ __forceinline__ uint32_t hadd2_u32(uint32_t a, uint32_t b) {
  const __half2 s = __hadd2(*reinterpret_cast<const __half2*>(&a),
                            *reinterpret_cast<const __half2*>(&b));
  return *reinterpret_cast<const uint32_t*>(&s);
}

// fp16(lo + hi) of a codebook word, in both halves (round to nearest even).
__device__ __forceinline__ uint32_t hsum_dup(uint32_t w) {
  const __half2 h = *reinterpret_cast<const __half2*>(&w);
  const __half2 s = __hadd2(__low2half2(h), __high2half2(h));
  return *reinterpret_cast<const uint32_t*>(&s);
}

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Two fp16 values (low half first) to two E4M3 bytes (low byte first),
// nearest even, saturating.
__device__ __forceinline__ uint16_t e4m3x2_from_f16x2(uint32_t h2) {
  uint16_t e;
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(e) : "r"(h2));
  return e;
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = __uint_as_float(r[j]);
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const float (&v)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(
                   taddr),
               "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
               "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
               "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7]))
               : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major operand whose rows are 128 bytes
// (64 fp16), 128-byte swizzle, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t smem_desc_k128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);  // start address
  d |= (uint64_t)1 << 16;                    // leading byte offset (unused with this swizzle)
  d |= (uint64_t)(1024 >> 4) << 32;          // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;                    // descriptor version
  d |= (uint64_t)2 << 61;                    // 128-byte swizzle
  return d;
}

// Instruction descriptor: fp32 D, A and B both K-major, M = 128, N = 128.
// The A/B format fields read 0 for f16 under kind::f16 and for E4M3 under
// kind::f8f6f4, so both kinds use the same word.
constexpr uint32_t kIdesc = (1u << 4)              // D format: f32
                            | (0u << 7)            // A format: f16 / E4M3
                            | (0u << 10)           // B format: f16 / E4M3
                            | ((kBN >> 3) << 17)   // N / 8
                            | ((128 >> 4) << 24);  // M / 16

// Two fp32 additions / subtractions / products in one instruction (each
// lane rounded exactly as the scalar operation).
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// Butterfly (p, q) -> (p + q, p - q) on neighbouring pairs of values.
__device__ __forceinline__ void f2_butterfly(float& p0, float& p1, float& q0, float& q1) {
  const uint64_t p = f2_pack(p0, p1), q = f2_pack(q0, q1);
  f2_unpack(f2_add(p, q), p0, p1);
  f2_unpack(f2_sub(p, q), q0, q1);
}

// Walsh-Hadamard butterflies (natural order, unnormalised) over 32 values
// held in registers: index bit 0 as scalar operations, bits 1..4 two
// butterflies per instruction pair (the same roundings).
__device__ __forceinline__ void fwht32_regs(float (&v)[32]) {
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    const float p = v[i], q = v[i + 1];
    v[i] = p + q;
    v[i + 1] = p - q;
  }
#pragma unroll
  for (int h = 2; h < 32; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 32; i += 2)
      if ((i & h) == 0) f2_butterfly(v[i], v[i + 1], v[i + h], v[i + h + 1]);
  }
}

// Position in a ring of S stages: stage index and phase parity.
template <int S>
struct Ring {
  int stage = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void advance() {
    if (++stage == S) {
      stage = 0;
      phase ^= 1u;
    }
  }
};

// One tile segment of a CTA's range: tile index and K-block range [kb0, kb1).
struct Segment {
  int tile, kb0, kb1;
};

// A CTA's range [u, u1) is at most: the end part of one tile (if u is not at a
// tile start), whole tiles, and the start part of another (if u1 is not).
// The parts are shared with the neighbouring CTAs.  parts_last: the whole
// tiles are walked first and the two parts last, so that both CTAs of a
// shared tile reach it near the end of the launch and the partial sums are
// still in L2 when the last of them merges them; otherwise range order.
struct SegIter {
  int ta, ka, tb, kb;  // the range starts at K block ka of tile ta, ends before kb of tb
  int KB;
  int parts_last;
  int step;  // segments handed out so far
  __device__ __forceinline__ SegIter(long long u, long long u1, int kb_per_tile, int last_mode)
      : KB(kb_per_tile), parts_last(last_mode), step(u < u1 ? 0 : -1) {
    ta = static_cast<int>(u / KB);
    ka = static_cast<int>(u - (long long)ta * KB);
    tb = static_cast<int>(u1 / KB);
    kb = static_cast<int>(u1 - (long long)tb * KB);
  }
  __device__ __forceinline__ bool next(Segment& s) {
    if (step < 0) return false;  // empty range
    const int i = step++;
    if (ta == tb) {  // inside one tile
      if (i > 0) return false;
      s.tile = ta;
      s.kb0 = ka;
      s.kb1 = kb;
      return true;
    }
    const int first = ka > 0 ? 1 : 0, last = kb > 0 ? 1 : 0;
    const int w0 = ta + first;  // whole tiles [w0, tb)
    const int nwhole = tb - w0;
    const int n = first + nwhole + last;
    if (i >= n) return false;
    const int k = !parts_last ? i : i < nwhole ? i + first : (i == nwhole && first) ? 0 : n - 1;
    if (first && k == 0) {
      s.tile = ta;
      s.kb0 = ka;
      s.kb1 = KB;
    } else if (last && k == n - 1) {
      s.tile = tb;
      s.kb0 = 0;
      s.kb1 = kb;
    } else {
      s.tile = w0 + k - first;
      s.kb0 = 0;
      s.kb1 = KB;
    }
    return true;
  }
};

// ---------------------------------------------------------------- kernel

template <int BITS, bool E4M3, bool FP8>
__global__ void __launch_bounds__(kThreadsG, 1)
    trellis_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const GemmArgs a) {
  using G = BlockGeom<FP8>;
  static_assert(!FP8 || E4M3, "the FP8 MMA needs E4M3 weights");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + G::kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars + 1);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  constexpr int T = 32 * BITS;
  const int NT = a.N / 16;
  const int c = blockIdx.x;
  const long long u_begin = range_start(c, a.units, a.grid);
  const long long u_end = range_start(c + 1, a.units, a.grid);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kAStages; ++s) mbar_init(bar(kBarAFull + s), 1);
    for (int s = 0; s < 2 * kAStages; ++s) mbar_init(bar(kBarAEmpty + s), 1);
    for (int s = 0; s < kCStages; ++s) {
      mbar_init(bar(kBarCFull + s), 1);
      mbar_init(bar(kBarCEmpty + s), kDecWarps);
    }
    for (int s = 0; s < kBStages; ++s) {
      mbar_init(bar(kBarBFull + s), kDecWarps);
      mbar_init(bar(kBarBEmpty + s), 1);
    }
    mbar_init(bar(kBarAcc), 1);
    mbar_init(bar(kBarTmemFree), kDecWarps);
    mbar_init(bar(kBarDrain), 1);
    mbar_init(bar(kBarEpi), kDecWarps);
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  SegIter it(u_begin, u_end, a.kb_per_tile, a.parts_last);
  Segment seg;

  if (warp == 0) {
    // ---------------------------------------------------------- A producer
    if (lane == 0) {
      int armed[kAStages] = {-1, -1};
      bool ok = true;
      Ring<kAStages> ra;
      pdl_wait();  // the activations are the previous kernel's output
      // Every tile of a 512-row block reads the same activations: keep them in
      // L2 ahead of the code words and outputs, which are touched once.
      const uint64_t keep = policy_evict_last();
      while (ok && it.next(seg)) {
        const int m0 = (seg.tile / a.n_blocks) * kBM;
        for (int kb = seg.kb0; kb < seg.kb1; ++kb, ra.advance()) {
          const int s = ra.stage;
          const uint32_t ph = ra.phase;
          // fp16: each half has its own empty barrier; FP8: the second half's
          // barrier frees the whole stage (the first is not used)
          if (!mbar_wait(bar(kBarAEmpty + 2 * s + (FP8 ? 1 : 0)), ph ^ 1u, a.limit_ns)) {
            set_error(a.err, kDevErrTimeout);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar(kBarAFull + s), kABytes);
          armed[s] = static_cast<int>(ph);
          const uint32_t dst = base + s * kABytes;
          tma_load_2d_hint(dst, &tmap_a, kb * G::kKE, m0, bar(kBarAFull + s), keep);
          // On a timeout the second half is still loaded (the result is
          // flagged as wrong), so that the stage's full barrier completes and
          // the drain below can wait for every copy in flight.
          if (!FP8 && !mbar_wait(bar(kBarAEmpty + 2 * s + 1), ph ^ 1u, a.limit_ns)) {
            set_error(a.err, kDevErrTimeout);
            ok = false;
          }
          tma_load_2d_hint(dst + kABytes / 2, &tmap_a, kb * G::kKE, m0 + kBM / 2,
                           bar(kBarAFull + s), keep);
          if (!ok) break;
        }
      }
      if (!ok)
        for (int s = 0; s < kAStages; ++s)
          if (armed[s] >= 0)
            mbar_wait(bar(kBarAFull + s), static_cast<uint32_t>(armed[s]), a.limit_ns);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- code producer
    if (lane == 0) {
      int armed[kCStages] = {-1, -1, -1, -1};
      bool ok = true;
      Ring<kCStages> rc;
      const uint32_t row_bytes = 8 * T;
      const uint64_t once = policy_evict_first();
      while (ok && it.next(seg)) {
        const int nb = seg.tile % a.n_blocks;
        for (int kb = seg.kb0; kb < seg.kb1; ++kb, rc.advance()) {
          const int s = rc.stage;
          const uint32_t ph = rc.phase;
          if (!mbar_wait(bar(kBarCEmpty + s), ph ^ 1u, a.limit_ns)) {
            set_error(a.err, kDevErrTimeout);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar(kBarCFull + s), G::kKT * row_bytes);
          const uint32_t dst = base + G::kOffC + s * G::kCBytes;
          for (int r = 0; r < G::kKT; ++r) {
            const uint8_t* src = a.code + ((size_t)(G::kKT * kb + r) * NT + 8 * nb) * T;
            bulk_g2s_evict_first(dst + r * row_bytes, src, row_bytes, bar(kBarCFull + s), once);
          }
          armed[s] = static_cast<int>(ph);
        }
      }
      if (!ok)
        for (int s = 0; s < kCStages; ++s)
          if (armed[s] >= 0)
            mbar_wait(bar(kBarCFull + s), static_cast<uint32_t>(armed[s]), a.limit_ns);
    }
  } else if (warp == 2) {
    // ---------------------------------------------------------- MMA issuer
    // The whole warp walks the loop (waits and descriptor arithmetic are
    // warp-uniform); one elected lane issues each MMA and commit.  Every wait
    // result is made warp-uniform so that the warp never splits.
    {
      bool ok = true;
      Ring<kAStages> ra;
      Ring<kBStages> rb;
      int nseg = 0;
      while (ok && it.next(seg)) {
        if (nseg > 0 &&
            !__all_sync(0xFFFFFFFFu, mbar_wait(bar(kBarTmemFree), (nseg - 1) & 1, a.limit_ns))) {
          if (lane == 0) set_error(a.err, kDevErrTimeout);
          break;
        }
        tc_fence_after();
        for (int kb = seg.kb0; kb < seg.kb1; ++kb, ra.advance(), rb.advance()) {
          const int sa = ra.stage;
          const uint32_t pa = ra.phase;
          const int sb = rb.stage;
          const uint32_t pb = rb.phase;
          const bool got = mbar_wait(bar(kBarAFull + sa), pa, a.limit_ns) &&
                           mbar_wait(bar(kBarBFull + sb), pb, a.limit_ns);
          if (!__all_sync(0xFFFFFFFFu, got)) {
            if (lane == 0) set_error(a.err, kDevErrTimeout);
            ok = false;
            break;
          }
          tc_fence_after();
          // Descriptors of the stage's first A and B rows; an operand
          // further into the stage adds its byte offset / 16 to the start
          // address field (shared memory is below 256 KB, so no carry).
          const uint64_t ad0 = smem_desc_k128(base + sa * kABytes);
          const uint64_t bd0 = smem_desc_k128(base + kOffB + sb * kBBytes);
          const uint32_t cont = kb > seg.kb0 ? 1u : 0u;
          if (elect_one()) {
#pragma unroll
            for (int acc = 0; acc < 4; ++acc) {
#pragma unroll
              for (int kk = 0; kk < kRowBytes / 32; ++kk) {  // 32 bytes of K per MMA
                const uint64_t ad = ad0 + (uint64_t)((acc * (kABytes / 4) + kk * 32) >> 4);
                const uint64_t bd = bd0 + (uint64_t)((kk * 32) >> 4);
                const uint32_t accum = kk > 0 ? 1u : cont;
                if constexpr (FP8)
                  mma_e4m3(tmem_base + acc * kBN, ad, bd, kIdesc, accum);
                else
                  mma_f16(tmem_base + acc * kBN, ad, bd, kIdesc, accum);
              }
              // accumulators 0 and 1 read the stage's first 256 rows (fp16:
              // that half is freed here)
              if (!FP8 && acc == 1) mma_commit(bar(kBarAEmpty + 2 * sa));
            }
            mma_commit(bar(kBarAEmpty + 2 * sa + 1));
            mma_commit(bar(kBarBEmpty + sb));
          }
          __syncwarp();
        }
        if (!ok) break;
        if (elect_one()) mma_commit(bar(kBarAcc));  // this segment's accumulators are complete
        __syncwarp();
        ++nseg;
      }
      if (elect_one()) mma_commit(bar(kBarDrain));
      __syncwarp();
      mbar_wait(bar(kBarDrain), 0, a.limit_ns);  // nothing in flight before TMEM is released
    }
  } else {
    // ---------------------------------------------------------- decoders + epilogue
    const int dw = warp - kFirstDec;   // 0..15
    constexpr int NTW = G::kTilesPerWarp;  // n-tiles this warp decodes per block: 2 or 4
    const int kt_local = dw / (8 / NTW);   // k-tile row of the block this warp decodes
    const int nt_base = (dw % (8 / NTW)) * NTW;
    const int quad = warp & 3;         // TMEM lane quadrant this warp may access
    const int acc = dw >> 2;           // accumulator (128-row slice) it finishes
    const LaneWindow lw = lane_window<BITS>(lane);
    const int g = lane >> 2, t = lane & 3;
    const uint32_t mcg_mask = a.mcg_mask, mcg_xor = a.mcg_xor;
    bool ok = true;
    Ring<kCStages> rc;
    Ring<kBStages> rb;
    int nseg = 0;
    // Decode the next code stage into the next decoded-B stage.
    auto decode_block = [&]() -> bool {
        const int sc = rc.stage;
        const uint32_t pc = rc.phase;
        const int sb = rb.stage;
        const uint32_t pb = rb.phase;
        if (!mbar_wait(bar(kBarCFull + sc), pc, a.limit_ns) ||
            !mbar_wait(bar(kBarBEmpty + sb), pb ^ 1u, a.limit_ns)) {
          set_error(a.err, kDevErrTimeout);
          return false;
        }
        const uint8_t* codes = smem + G::kOffC + sc * G::kCBytes;
        uint8_t* bt = smem + kOffB + sb * kBBytes;
#pragma unroll
        for (int i = 0; i < NTW; ++i) {
          const int nt = nt_base + i;
          const uint32_t* tw = reinterpret_cast<const uint32_t*>(codes + (kt_local * 8 + nt) * T);
          uint32_t v[8];  // codebook words (fp16 lo, fp16 hi) of the lane's symbols
          decode8_pairs<BITS>(tw[lw.i0], tw[lw.i1], lw.sh7, mcg_mask, mcg_xor, v);
          // symbols 2p, 2p+1 (p = 2 nh + rh) are input channels k, k+1 of output
          // channel n = 16 nt + g + 8 nh, k = 16 kt_local + 8 rh + 2t.  fp16:
          // two byte permutes gather the pair's (lo, lo) and (hi, hi), one
          // addition forms both weights.  FP8, whose decoders keep the integer
          // pipe busier: one addition per weight with its operands' halves
          // broadcast, then one permute per pair (measured 3 % faster there,
          // 4 % slower at fp16).
          uint32_t pair[4];
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            if constexpr (FP8)
              pair[p] = __byte_perm(hsum_dup(v[2 * p]), hsum_dup(v[2 * p + 1]), 0x5410);
            else
              pair[p] = hadd2_u32(__byte_perm(v[2 * p], v[2 * p + 1], 0x5410),
                                  __byte_perm(v[2 * p], v[2 * p + 1], 0x7632));
          }
          if constexpr (FP8) {
            // Bytes k, k+1 of row n, one 16-bit store per pair: rh = 0 at
            // bytes 2t, 2t+1 and rh = 1 at 8 + 2t of the row's 16-byte chunk
            // kt_local (no exchange between lanes).
#pragma unroll
            for (int nh = 0; nh < 2; ++nh) {
              const int n = 16 * nt + g + 8 * nh;   // n & 7 == g: the row's swizzle phase
              uint8_t* row = bt + n * 128 + (kt_local ^ g) * 16 + 2 * t;
              *reinterpret_cast<uint16_t*>(row) = e4m3x2_from_f16x2(pair[2 * nh]);
              *reinterpret_cast<uint16_t*>(row + 8) = e4m3x2_from_f16x2(pair[2 * nh + 1]);
            }
          } else {
#pragma unroll
            for (int p = 0; p < 4; ++p) {
              const int rh = p & 1, nh = p >> 1;
              const int n = 16 * nt + g + 8 * nh;
              const int chunk = (2 * kt_local + rh) ^ g;
              *reinterpret_cast<uint32_t*>(bt + n * 128 + chunk * 16 + 4 * t) =
                  E4M3 ? round_e4m3x2(pair[p]) : pair[p];
            }
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(kBarBFull + sb));
          mbar_arrive(bar(kBarCEmpty + sc));
        }
        return true;
    };
    int pre = 0;  // K blocks of the current segment decoded ahead of its loop
    while (ok && it.next(seg)) {
      const int nb = seg.tile % a.n_blocks;
      const int m0 = (seg.tile / a.n_blocks) * kBM;
      for (int kb = seg.kb0 + pre; kb < seg.kb1; ++kb, rc.advance(), rb.advance()) {
        if (!decode_block()) {
          ok = false;
          break;
        }
      }
      if (!ok) break;
      // fp16: the next segment's first blocks are decoded while this one's
      // last MMAs run (their ring stages free up as those MMAs complete), so
      // that the MMA warp finds them ready once the epilogue frees TMEM.
      pre = 0;
      if (G::kLookahead > 0) {
        SegIter peek = it;
        Segment nx;
        if (peek.next(nx)) {
          const int la = min(G::kLookahead, nx.kb1 - nx.kb0);
          for (; pre < la; ++pre, rc.advance(), rb.advance()) {
            if (!decode_block()) {
              ok = false;
              break;
            }
          }
        }
      }
      if (!ok) break;

      // ---- epilogue of this segment: row acc*128 + quad*32 + lane of the tile
      if (nseg == 0) pdl_wait();  // the scales d come from the previous kernel
      // the tile's 128 output scales, staged in this warp's slot while the
      // segment's last MMAs run (read back below as broadcasts)
      float* svs = reinterpret_cast<float*>(smem + G::kOffSv) + dw * kBN;
      {
        float4 sv4 = __ldg(reinterpret_cast<const float4*>(a.sv + nb * kBN) + lane);
        sv4.x *= kHadScale;  // 1/sqrt(128) folded in, as the products below take it
        sv4.y *= kHadScale;
        sv4.z *= kHadScale;
        sv4.w *= kHadScale;
        reinterpret_cast<float4*>(svs)[lane] = sv4;
      }
      __syncwarp();
      if (!mbar_wait(bar(kBarAcc), nseg & 1, a.limit_ns)) {
        set_error(a.err, kDevErrTimeout);
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t tl = tmem_base + ((uint32_t)(quad * 32) << 16) + acc * kBN;
      const int row = acc * 128 + quad * 32 + lane;
      const int m = m0 + row;
      const long long t_first = (long long)seg.tile * a.kb_per_tile;
      const int c_first = owner(t_first, a.units, a.grid);
      const int c_last = owner(t_first + a.kb_per_tile - 1, a.units, a.grid);
      const int n0 = nb * kBN;
      bool finish = c_first == c_last;  // this CTA holds the whole tile
      if (!finish) {
        // A shared tile.  This warp's rows of it are finished by the last of the
        // tile's c_last - c_first + 1 CTAs to arrive here; the others leave their
        // partial sums (slot 0: a CTA's first tile, slot 1: a later one).
        int* cnt = a.tile_cnt + (size_t)seg.tile * kDecWarps + dw;
        const int others = c_last - c_first;
        int is_last = 0;
        if (lane == 0) is_last = ld_acquire_gpu(cnt) == others;
        is_last = __shfl_sync(0xFFFFFFFFu, is_last, 0);
        if (!is_last) {
          // partial sums as [slot][column / 4][row][4]: a warp's 32 rows of
          // four columns are 512 contiguous bytes
          const int which = (t_first <= u_begin) ? 0 : 1;
          float4* wslot = reinterpret_cast<float4*>(a.ws) + (size_t)(2 * c + which) * (kBN / 4) * kBM;
#pragma unroll 1
          for (int c16 = 0; c16 < kBN; c16 += 16) {
            float u[16];
            tmem_ld16(tl + c16, u);
            tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < 4; ++q)
              wslot[(size_t)(c16 / 4 + q) * kBM + row] =
                  make_float4(u[4 * q], u[4 * q + 1], u[4 * q + 2], u[4 * q + 3]);
          }
          __syncwarp();
          if (lane == 0) {
            __threadfence();  // the warp's partial sums before its count
            is_last = atomicAdd(cnt, 1) == others;
          }
          is_last = __shfl_sync(0xFFFFFFFFu, is_last, 0);
          if (G::kLookahead > 0 && !is_last) {
            // fp16: this warp is done with TMEM for the segment
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarTmemFree));
          }
        }
        if (is_last && lane == 0) __threadfence();  // every other partial is visible
        __syncwarp();
        finish = is_last != 0;
      }
      if (finish && c_first != c_last) {
        // the last arrival: accumulators <- the CTAs' partial sums added in CTA
        // order (this CTA's own from its accumulators), 16 columns at a time
        // with each other CTA's loads in flight together
#pragma unroll 1
        for (int c16 = 0; c16 < kBN; c16 += 16) {
          float w[16], sacc[16];
          tmem_ld16(tl + c16, w);
#pragma unroll
          for (int j = 0; j < 16; ++j) sacc[j] = 0.f;
          tmem_wait_ld();
          for (int cc = c_first; cc <= c_last; ++cc) {
            if (cc == c) {
#pragma unroll
              for (int j = 0; j < 16; ++j) sacc[j] += w[j];
            } else {
              const int wh = (t_first <= range_start(cc, a.units, a.grid)) ? 0 : 1;
              const float4* src = reinterpret_cast<const float4*>(a.ws) +
                                  (size_t)(2 * cc + wh) * (kBN / 4) * kBM + (size_t)(c16 / 4) * kBM +
                                  row;
              float4 p[4];
#pragma unroll
              for (int q = 0; q < 4; ++q) p[q] = src[(size_t)q * kBM];
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                sacc[4 * q] += p[q].x;
                sacc[4 * q + 1] += p[q].y;
                sacc[4 * q + 2] += p[q].z;
                sacc[4 * q + 3] += p[q].w;
              }
            }
          }
          tmem_st8(tl + c16, reinterpret_cast<const float(&)[8]>(sacc[0]));
          tmem_st8(tl + c16 + 8, reinterpret_cast<const float(&)[8]>(sacc[8]));
        }
        tmem_wait_st();
      }
      if (finish) {
        // FP8: the row's activation scale joins the output scale
        const float dm = FP8 ? (m < a.M ? __ldg(a.d + m) : 0.f) : 1.f;
        // index bits 5 and 6 across the four 32-column chunks, in TMEM
#pragma unroll 1
        for (int c8 = 0; c8 < 32; c8 += 8) {
          float x0[8], x1[8], x2[8], x3[8];
          tmem_ld8(tl + c8, x0);
          tmem_ld8(tl + c8 + 32, x1);
          tmem_ld8(tl + c8 + 64, x2);
          tmem_ld8(tl + c8 + 96, x3);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 8; j += 2) {
            f2_butterfly(x0[j], x0[j + 1], x1[j], x1[j + 1]);  // bit 5
            f2_butterfly(x2[j], x2[j + 1], x3[j], x3[j + 1]);
            f2_butterfly(x0[j], x0[j + 1], x2[j], x2[j + 1]);  // bit 6
            f2_butterfly(x1[j], x1[j + 1], x3[j], x3[j + 1]);
          }
          tmem_st8(tl + c8, x0);
          tmem_st8(tl + c8 + 32, x1);
          tmem_st8(tl + c8 + 64, x2);
          tmem_st8(tl + c8 + 96, x3);
        }
        tmem_wait_st();
        // Index bits 0..4 on each chunk in registers, * sv / sqrt(128), fp16:
        // each lane then holds 64 contiguous bytes of its row.  They go out
        // through a shared-memory slot of this warp and are read back so that
        // several lanes store each row's bytes together instead of 32 lanes
        // writing scattered 16-byte pieces.  fp16: the warp's own 1 KB slot,
        // 16 rows at a time (two lanes per row, 32 contiguous bytes each),
        // with TMEM freed as soon as the last chunk is read.  FP8: 2 KB of the
        // decoded-B ring (idle during the epilogue: every MMA of the segment
        // has completed, and no decoder writes it again before all have passed
        // the barrier below), 32 rows at a time (four lanes per row).
        constexpr bool kOwnSlot = G::kLookahead > 0;
        uint8_t* scr = kOwnSlot ? smem + G::kOffScr + dw * 1024 : smem + kOffB + dw * 2048;
        const int qj = lane & 3, qb = lane & ~3;
#pragma unroll 1
        for (int q = 0; q < 4; ++q) {
          float w[32];
          tmem_ld32(tl + 32 * q, w);
          tmem_wait_ld();
          if (kOwnSlot && q == 3) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarTmemFree));
          }
          fwht32_regs(w);
          const float* scv = svs + 32 * q;
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const uint64_t sc = FP8 ? f2_pack(scv[2 * e] * dm, scv[2 * e + 1] * dm)
                                    : f2_pack(scv[2 * e], scv[2 * e + 1]);
            float o0, o1;
            f2_unpack(f2_mul(f2_pack(w[2 * e], w[2 * e + 1]), sc), o0, o1);
            const __half2 h = __floats2half2_rn(o0, o1);
            pk[e] = *reinterpret_cast<const uint32_t*>(&h);
          }
          if (kOwnSlot) {
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
              // rows 16 hr .. 16 hr + 15: row lane & 15 written by lane
              // 16 hr + (lane & 15), 16-byte piece p at chunk p ^ ((row >> 1) & 3)
              if ((lane >> 4) == hr) {
                const int lr = lane & 15;
#pragma unroll
                for (int p = 0; p < 4; ++p)
                  *reinterpret_cast<uint4*>(scr + lr * 64 + 16 * (p ^ ((lr >> 1) & 3))) =
                      make_uint4(pk[4 * p], pk[4 * p + 1], pk[4 * p + 2], pk[4 * p + 3]);
              }
              __syncwarp();
              const int lr = lane >> 1, hf = lane & 1;
              const int mr = m0 + acc * 128 + quad * 32 + 16 * hr + lr;
#pragma unroll
              for (int jj = 0; jj < 2; ++jj) {
                const int p = 2 * jj + hf;  // lanes 2lr, 2lr+1: 32 contiguous bytes
                const uint4 v =
                    *reinterpret_cast<const uint4*>(scr + lr * 64 + 16 * (p ^ ((lr >> 1) & 3)));
                if (mr < a.M)
                  *reinterpret_cast<uint4*>(a.y + (size_t)mr * a.N + n0 + 32 * q + 8 * p) = v;
              }
              __syncwarp();
            }
          } else {
            // row `lane`, 16-byte piece p at chunk p ^ ((lane >> 1) & 3): conflict-free
#pragma unroll
            for (int p = 0; p < 4; ++p)
              *reinterpret_cast<uint4*>(scr + lane * 64 + 16 * (p ^ ((lane >> 1) & 3))) =
                  make_uint4(pk[4 * p], pk[4 * p + 1], pk[4 * p + 2], pk[4 * p + 3]);
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int r = qb + i;  // this warp's row written by the lane's quad
              const uint4 v =
                  *reinterpret_cast<const uint4*>(scr + r * 64 + 16 * (qj ^ ((r >> 1) & 3)));
              const int mr = m0 + acc * 128 + quad * 32 + r;
              if (mr < a.M)
                *reinterpret_cast<uint4*>(a.y + (size_t)mr * a.N + n0 + 32 * q + 8 * qj) = v;
            }
            __syncwarp();
          }
        }
      }
      if (G::kLookahead == 0) {
        // FP8: no decoder writes the decoded-B ring (used above as scratch)
        // before every decoder warp has finished this epilogue (a bounded
        // wait: a warp that gave up earlier never arrives); then TMEM is free
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarEpi));
        if (!mbar_wait(bar(kBarEpi), nseg & 1, a.limit_ns)) {
          set_error(a.err, kDevErrTimeout);
          ok = false;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarTmemFree));
      }
      ++nseg;
    }
  }

  __syncthreads();
  if (warp == 2) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <int BITS, bool E4M3, bool FP8>
cudaError_t launch_gemm_bits(const CUtensorMap& map, const GemmArgs& a, cudaStream_t st) {
  constexpr int smem = BlockGeom<FP8>::kSmemBytes;
  cudaError_t e =
      set_smem_limit(reinterpret_cast<const void*>(trellis_gemm_kernel<BITS, E4M3, FP8>), smem);
  if (e != cudaSuccess) return e;
  PdlLaunch dl(a.grid, kThreadsG, smem, st);
  return cudaLaunchKernelEx(&dl.cfg, trellis_gemm_kernel<BITS, E4M3, FP8>, map, a);
}

// Shared by both operand types: the activation tensor map (rows of K elements
// of `esize` bytes, 128-byte boxes, 128B swizzle), the stream-K split and the
// kernel launch.
cudaError_t launch_gemm(const void* act, bool fp8, const float* d, const int16_t* code, int bits,
                        bool e4m3, int M, int K, int N, const float* sv, uint16_t* y, float* ws,
                        int* tile_cnt, int num_sms, int* err, cudaStream_t st) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return cudaErrorNotSupported;
  const int esize = fp8 ? 1 : 2;
  const int ke = kRowBytes / esize;  // K elements per block
  CUtensorMap map;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
  const cuuint64_t strides[1] = {(cuuint64_t)K * esize};
  const cuuint32_t box[2] = {(cuuint32_t)ke, kBM / 2};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(&map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                   const_cast<void*>(act), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  GemmArgs a;
  a.code = reinterpret_cast<const uint8_t*>(code);
  a.sv = sv;
  a.d = fp8 ? d : nullptr;
  a.mcg_mask = kMcgMask;
  a.mcg_xor = kMcgXor;
  a.y = y;
  a.ws = ws;
  a.tile_cnt = tile_cnt;
  a.M = M;
  a.N = N;
  a.K = K;
  a.n_blocks = N / kBN;
  a.kb_per_tile = K / ke;
  const long long tiles = (long long)((M + kBM - 1) / kBM) * a.n_blocks;
  a.units = tiles * a.kb_per_tile;
  // at least 16 K-blocks per CTA, at most one CTA per SM
  long long g = a.units / 16;
  if (g < 1) g = 1;
  if (g > num_sms) g = num_sms;
  a.grid = static_cast<int>(g);
  // With two or more tiles per CTA, shared parts last: measured 2.9 % faster at
  // 5120 -> 17408 (M = 2048) with the DRAM traffic down to the algorithmic
  // bytes; with about one tile per CTA (17408 -> 5120) range order is 2 % faster.
  a.parts_last = tiles >= 2LL * g ? 1 : 0;
  a.err = err;
  a.limit_ns = kWaitLimitNs;

  cudaError_t e;
  if (fp8) {
    switch (bits) {
      case 2: e = launch_gemm_bits<2, true, true>(map, a, st); break;
      case 3: e = launch_gemm_bits<3, true, true>(map, a, st); break;
      default: e = launch_gemm_bits<4, true, true>(map, a, st); break;
    }
  } else {
    switch (bits) {
      case 2: e = e4m3 ? launch_gemm_bits<2, true, false>(map, a, st) : launch_gemm_bits<2, false, false>(map, a, st); break;
      case 3: e = e4m3 ? launch_gemm_bits<3, true, false>(map, a, st) : launch_gemm_bits<3, false, false>(map, a, st); break;
      default: e = e4m3 ? launch_gemm_bits<4, true, false>(map, a, st) : launch_gemm_bits<4, false, false>(map, a, st); break;
    }
  }
  return e;
}

}  // namespace

size_t gemm_workspace_floats(int num_sms) { return (size_t)num_sms * 2 * kBM * kBN; }

size_t gemm_counter_ints(int M, int N) {
  return (size_t)((M + kBM - 1) / kBM) * (N / kBN) * kDecWarps;
}

// xh: rotated activations fp16 [M, K] (16-byte aligned, K a multiple of 128);
// ws: gemm_workspace_floats(num_sms) fp32.
cudaError_t launch_trellis_gemm(const uint16_t* xh, const int16_t* code, int bits, bool e4m3,
                                int M, int K, int N, const float* sv, uint16_t* y, float* ws,
                                int* tile_cnt, int num_sms, int* err, cudaStream_t st) {
  return launch_gemm(xh, false, nullptr, code, bits, e4m3, M, K, N, sv, y, ws, tile_cnt, num_sms,
                     err, st);
}

// xq: E4M3 activation codes [M, K] (16-byte aligned, K a multiple of 128) with
// per-row scales d [M]; the weights are decoded with the E4M3 rounding.
cudaError_t launch_trellis_gemm_fp8(const uint8_t* xq, const float* d, const int16_t* code,
                                    int bits, int M, int K, int N, const float* sv, uint16_t* y,
                                    float* ws, int* tile_cnt, int num_sms, int* err,
                                    cudaStream_t st) {
  return launch_gemm(xq, true, d, code, bits, true, M, K, N, sv, y, ws, tile_cnt, num_sms, err,
                     st);
}

}  // namespace escha
