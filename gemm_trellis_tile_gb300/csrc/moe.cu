// Routed-expert layer at decode (EXLR8 page, "The sharing trick"; GLM-5.3
// expert shapes): y[m] = sum_k w[m,k] * down_e(silu(gate_e(x[m])) * up_e(x[m])).
//
// The hidden side of every expert is one shared rotation: gate and up read one
// rotated activation had(x * su_hidden), and down's outputs are summed before
// one shared output rotation had(.) * sv_hidden (exact by linearity).  The
// intermediate side is per expert.
//
// One call, five launches on the caller's stream, no host synchronisation:
//   1. moe_plan         block 0 reads the routing on the device: distinct
//                       experts in order of first appearance, tokens per
//                       expert, and the job tables / unit counts / grid sizes
//                       of launches 2 and 4; the other blocks rotate the
//                       token(s): xfrag_hidden = fp16(had128(x * su_hidden))
//   2. trellis GEMV     gate and up of every distinct expert (mixed widths)
//   3. moe_mid          per (expert, token): had(gate)*sv_g, had(up)*sv_u,
//                       silu(g)*u, then had(h * su_down) into that expert's
//                       down fragments (zeros for tokens not routed to it)
//   4. trellis GEMV     down of every distinct expert
//   5. moe_out          y = fp16(had(sum_k w_k * down partials) * sv_hidden)
// Distinct experts decode once however many tokens route to them: the GEMV's
// B operand carries all 8 token slots, so every token of an expert shares one
// decode of its tiles.

#include <cuda_runtime.h>

#include <algorithm>
#include <new>

#include "act_layout.cuh"
#include "api_internal.h"
#include "common.cuh"
#include "internal.h"

namespace escha {

namespace {

constexpr int kWarpsPerBlock = 8;

// Device-side routing state written by moe_plan_kernel.
// Partial-sum slots per group: device_grid() keeps a group within 5 CTAs.
constexpr int kMoeSlots = 6;
// Expert slots of a call: the distinct routed experts, then the shared expert.
constexpr int kMoeMaxSlots = kMoeMaxDistinct + 1;

struct MoeRoute {
  long long units1;  // gate+up GEMV
  long long units2;  // down GEMV
  int grid1, grid2;
  int n_distinct;
  int pad;
  int expert[kMoeMaxSlots];                 // expert id of slot d (E: the shared expert)
  unsigned mask[kMoeMaxSlots];              // bit m set: token m routes to d
  int route[kMoeMaxTokens * kMoeMaxTopk];   // distinct slot of (m, k), -1 if skipped
  int shared_slot;                          // slot of the shared expert, -1 if none
};

struct MoePlanArgs {
  const int32_t* ids;
  int M, topk, E;
  int hidden, inter;
  const uint8_t* const* gate_code;
  const uint8_t* const* up_code;
  const uint8_t* const* down_code;
  const CUtensorMap* code_maps;  // [3][E + 1]: gate, up, down (entry E: the shared expert)
  int shared;                    // the shared expert is set: every token uses it
  const int* bits;
  int e4m3;                      // codebook values rounded to E4M3
  const uint32_t* xfrag_hidden;
  uint32_t* xfrag_down;   // [kMoeMaxDistinct][inter/16][M][4][4]
  float* part1;           // [2*kMoeMaxDistinct][slots][8][inter]
  float* part2;           // [kMoeMaxDistinct][slots][8][hidden]
  size_t part1_stride, part2_stride, xdown_stride;  // elements per job / per distinct slot
  GemvJob* jobs1;         // [2*kMoeMaxDistinct]
  GemvJob* jobs2;         // [kMoeMaxDistinct]
  MoeRoute* route;
  int grid1_max, grid2_max;
  int* err;
};

__device__ __forceinline__ GemvJob make_job(const uint8_t* code, const CUtensorMap* tmap,
                                            const uint32_t* xfrag, float* part, long long ub,
                                            int bits, int KT, int NG, int N, int e4m3) {
  GemvJob j;
  j.e4m3 = e4m3;
  j.code = code;
  j.tmap = tmap;
  j.xfrag = reinterpret_cast<const uint4*>(xfrag);
  j.part = part;
  j.unit_begin = ub;
  j.bits = bits;
  j.KT = KT;
  j.NG = NG;
  j.N = N;
  return j;
}

// The input rotation done by the plan launch's blocks 1..: xfrag_hidden =
// fp16(had128(x * su_hidden)), one warp per (token, 128-channel block).
struct MoeRotIn {
  const uint16_t* x;
  const float* su;
  uint32_t* xfrag;
  int K, M;
};
constexpr int kPlanThreads = 256;

// Blocks past the first: wait for the previous kernel (the previous call may
// still read xfrag), then rotate.  Returns true for block 0 (the plan).
__device__ __forceinline__ bool plan_block_or_rotate(const MoeRotIn& rot) {
  if (blockIdx.x == 0) return true;
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int nb = rot.K / kHad;
  const long long task = (long long)(blockIdx.x - 1) * (kPlanThreads / 32) + (threadIdx.x >> 5);
  if (task < (long long)rot.M * nb) {
    const int m = static_cast<int>(task / nb);
    rotate_in_block(rot.x, rot.su, rot.xfrag, rot.K, rot.M, m, static_cast<int>(task - (long long)m * nb),
                    lane);
  }
  return false;
}

unsigned plan_blocks(int M, int K) {
  const long long tasks = (long long)M * (K / kHad);
  return static_cast<unsigned>(1 + (tasks + kPlanThreads / 32 - 1) / (kPlanThreads / 32));
}

// Grid size that gives every CTA at least a quarter of a group's k-tiles, so
// a group's units span at most five CTAs (five partial-sum slots).
__device__ __forceinline__ int device_grid(long long units, int KT, int grid_max) {
  long long g = units * 4 / KT;
  if (g < 1) g = 1;
  if (g > grid_max) g = grid_max;
  return static_cast<int>(g);
}

// The routing part of a plan (all threads of the block call it): distinct
// experts in order of first appearance, the tokens of each, the slot of each
// (token, k).  first_slot: shared [E].  Returns the number of distinct experts.
//
// The routing is worked out in shared memory while the previous kernel in the
// stream may still run (it reads only the ids, which no kernel of the call
// writes); then the block waits for that kernel to finish before it writes
// any state the previous call's kernels read (the route, job tables and maps).
// Without the wait, a plan launched right behind a contraction (a caller that
// runs only some stages) could rewrite its job table under it.
__device__ int plan_routing(const int32_t* ids, int M, int topk, int E, int* first_slot,
                            MoeRoute* r, int* err) {
  __shared__ int s_nd;
  __shared__ int s_expert[kMoeMaxDistinct];
  __shared__ unsigned s_mask[kMoeMaxDistinct];
  __shared__ int s_route[kMoeMaxTokens * kMoeMaxTopk];
  for (int e = threadIdx.x; e < E; e += blockDim.x) first_slot[e] = -1;
  __syncthreads();
  if (threadIdx.x == 0) {
    // Sequential on purpose: slots are numbered in order of first appearance.
    int nd = 0;
    for (int i = 0; i < M * topk; ++i) {
      const int e = ids[i];
      int d = -1;
      if (e >= 0 && e < E) {
        d = first_slot[e];
        if (d < 0) {
          d = nd++;
          first_slot[e] = d;
          s_expert[d] = e;
          s_mask[d] = 0u;
        }
        s_mask[d] |= 1u << (i / topk);
      } else {
        set_error(err, kDevErrBadRoute);
      }
      s_route[i] = d;
    }
    s_nd = nd;
  }
  __syncthreads();
  pdl_wait();
  const int nd = s_nd;
  for (int d = threadIdx.x; d < nd; d += blockDim.x) {
    r->expert[d] = s_expert[d];
    r->mask[d] = s_mask[d];
  }
  for (int i = threadIdx.x; i < M * topk; i += blockDim.x) r->route[i] = s_route[i];
  __syncthreads();
  return nd;
}

__global__ void moe_plan_kernel(const MoePlanArgs a, const MoeRotIn rot) {
  extern __shared__ int first_slot[];  // [E]: distinct slot of each expert, -1 if none yet
  pdl_trigger();  // the GEMV may launch; it waits for this kernel before reading the plan
  if (!plan_block_or_rotate(rot)) return;
  MoeRoute* r = a.route;
  const int nrouted = plan_routing(a.ids, a.M, a.topk, a.E, first_slot, r, a.err);
  // the shared expert takes the slot after the routed ones, for every token
  if (threadIdx.x == 0) {
    r->shared_slot = a.shared ? nrouted : -1;
    if (a.shared) {
      r->expert[nrouted] = a.E;
      r->mask[nrouted] = (a.M >= 32) ? 0xFFFFFFFFu : ((1u << a.M) - 1u);
    }
  }
  __syncthreads();
  const int nd = nrouted + (a.shared ? 1 : 0);
  const int Es = a.E + 1;  // entries per matrix in the tables
  const int KTg = a.hidden / 16, NGg = a.inter / 128;
  const int KTd = a.inter / 16, NGd = a.hidden / 128;
  const long long ug = (long long)KTg * NGg, ud = (long long)KTd * NGd;
  // Slots past nd keep well-formed shapes (never scheduled: the unit counts stop at nd).
  for (int d = threadIdx.x; d < kMoeMaxSlots; d += blockDim.x) {
    const int e = d < nd ? r->expert[d] : 0;
    const int b = a.bits[e];
    a.jobs1[2 * d] = make_job(a.gate_code[e], a.code_maps + e, a.xfrag_hidden,
                              a.part1 + (2 * d) * a.part1_stride, (2 * d) * ug, b, KTg, NGg,
                              a.inter, a.e4m3);
    a.jobs1[2 * d + 1] = make_job(a.up_code[e], a.code_maps + Es + e, a.xfrag_hidden,
                                  a.part1 + (2 * d + 1) * a.part1_stride, (2 * d + 1) * ug, b, KTg,
                                  NGg, a.inter, a.e4m3);
    a.jobs2[d] = make_job(a.down_code[e], a.code_maps + 2 * Es + e,
                          a.xfrag_down + d * a.xdown_stride, a.part2 + d * a.part2_stride, d * ud,
                          b, KTd, NGd, a.hidden, a.e4m3);
  }
  if (threadIdx.x == 0) {
    r->n_distinct = nd;
    r->units1 = 2LL * nd * ug;
    r->units2 = (long long)nd * ud;
    r->grid1 = device_grid(r->units1, KTg, a.grid1_max);
    r->grid2 = device_grid(r->units2, KTd, a.grid2_max);
  }
}

// ---------------------------------------------------------------- by halves
//
// EXLR8 page, manifest paragraph: each expert matrix is stored as halves of
// 128 intermediate channels, with a width per half for gate and up and one
// width per expert for down, and kernels take a pointer table ptr[e][h] that
// is re-read at every launch.  Gate and up halves are 128 output channels
// each: every (distinct expert, matrix, half) is one GEMV job of one
// 128-channel group whose code rows are contiguous.  Down halves are 128
// input channels (8 k-tile rows) each: a down job's unit is one half of one
// output group, loaded through that half's tensor map, which this kernel
// writes from a per-width template with the half's address.

struct MoeHalvesPlanArgs {
  const int32_t* ids;
  int M, topk, E, H;
  int hidden, inter;
  const uint8_t* const* gate_half;  // caller's tables [E][H]
  const uint8_t* const* up_half;
  const uint8_t* const* down_half;
  const int* gate_bits;             // [E][H]
  const int* up_bits;               // [E][H]
  const int* down_bits;             // [E]
  const CUtensorMap* tmpl;          // [3]: down-half maps for 2, 3, 4 bits
  CUtensorMap* half_maps;           // [E][H]
  unsigned long long* half_map_key; // [E][H]: pointer | bits of each map (0: not written)
  const uint8_t* stand_in;          // zero code used in place of a failing entry
  int e4m3;
  const uint32_t* xfrag_hidden;
  uint32_t* xfrag_down;
  float* part1;
  float* part2;
  size_t part1_stride, part2_stride, xdown_stride;
  GemvJob* jobs1;                   // [2*kMoeMaxDistinct*H]: (slot, gate|up, half)
  GemvJob* jobs2;                   // [kMoeMaxDistinct]
  MoeRoute* route;
  int grid1_max, grid2_max;
  int* err;
};

// A table entry is used only if its pointer is non-null and 16-byte aligned
// (the copy engine's rule) and its width is 2, 3 or 4; otherwise the handle's
// error flag is set and a zero code of the largest half takes its place.
__device__ __forceinline__ const uint8_t* checked_half(const uint8_t* p, const uint8_t* stand_in,
                                                       int* err) {
  if (p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) != 0) {
    set_error(err, kDevErrBadTable);
    return stand_in;
  }
  return p;
}
__device__ __forceinline__ int checked_bits(int b, int* err) {
  if (b < 2 || b > 4) {
    set_error(err, kDevErrBadTable);
    return 2;
  }
  return b;
}

__global__ void moe_plan_halves_kernel(const MoeHalvesPlanArgs a, const MoeRotIn rot) {
  extern __shared__ int first_slot[];  // [E]
  pdl_trigger();
  if (!plan_block_or_rotate(rot)) return;
  MoeRoute* r = a.route;
  const int nd = plan_routing(a.ids, a.M, a.topk, a.E, first_slot, r, a.err);
  if (threadIdx.x == 0) r->shared_slot = -1;  // no shared expert for experts stored by halves
  const int H = a.H;
  const int KTg = a.hidden / 16;     // gate/up: units per half job
  const int NGd = a.hidden / 128;    // down: output groups, H units (halves) each
  const long long ud = (long long)H * NGd;
  // gate and up: job q = (2d + matrix) * H + half
  for (int q = threadIdx.x; q < 2 * nd * H; q += blockDim.x) {
    const int h = q % H, dm = q / H;
    const int e = r->expert[dm >> 1];
    const bool up = (dm & 1) != 0;
    const uint8_t* p = checked_half((up ? a.up_half : a.gate_half)[(size_t)e * H + h], a.stand_in,
                                    a.err);
    const int b = checked_bits((up ? a.up_bits : a.gate_bits)[(size_t)e * H + h], a.err);
    // the half's partial sums start at its first output channel
    a.jobs1[q] = make_job(p, nullptr, a.xfrag_hidden, a.part1 + dm * a.part1_stride + 128 * h,
                          (long long)q * KTg, b, KTg, 1, a.inter, a.e4m3);
  }
  // down: the tensor map of every half of every distinct expert, kept per
  // (expert, half) and rewritten only when the table's pointer or the
  // expert's width differs from what the map was written for (the tables are
  // re-read every call, so a caller may swap halves between calls)
  for (int q = threadIdx.x; q < nd * H; q += blockDim.x) {
    const int d = q / H, h = q - d * H;
    const int e = r->expert[d];
    const int b = checked_bits(a.down_bits[e], a.err);
    const uint8_t* p = checked_half(a.down_half[(size_t)e * H + h], a.stand_in, a.err);
    const size_t slot = (size_t)e * H + h;
    const unsigned long long key = reinterpret_cast<unsigned long long>(p) | (unsigned)b;
    if (a.half_map_key[slot] == key) continue;
    const uint4* src = reinterpret_cast<const uint4*>(a.tmpl + (b - 2));
    uint4* dst = reinterpret_cast<uint4*>(a.half_maps + slot);
#pragma unroll
    for (int i = 0; i < 8; ++i) dst[i] = src[i];
    asm volatile("tensormap.replace.tile.global_address.global.b1024.b64 [%0], %1;" ::"l"(dst),
                 "l"(reinterpret_cast<uint64_t>(p))
                 : "memory");
    tensormap_release();
    a.half_map_key[slot] = key;
  }
  for (int d = threadIdx.x; d < nd; d += blockDim.x) {
    const int e = r->expert[d];
    const int b = checked_bits(a.down_bits[e], a.err);
    GemvJob j = make_job(nullptr, nullptr, a.xfrag_down + d * a.xdown_stride,
                         a.part2 + d * a.part2_stride, d * ud, b, H, NGd, a.hidden, a.e4m3);
    j.row_maps = a.half_maps + (size_t)e * H;
    a.jobs2[d] = j;
  }
  if (threadIdx.x == 0) {
    r->n_distinct = nd;
    r->units1 = 2LL * nd * H * KTg;
    r->units2 = (long long)nd * ud;
    r->grid1 = device_grid(r->units1, KTg, a.grid1_max);
    r->grid2 = device_grid(r->units2, H, a.grid2_max);
  }
}

struct MoeMidArgs {
  const MoeRoute* route;
  const GemvJob* jobs1;
  int jobs_per_matrix;   // 1, or H when stored by halves (job of half 0 describes the matrix)
  const float* sv_gate;  // [E][inter]
  const float* sv_up;
  const float* su_down;
  uint32_t* xfrag_down;
  size_t xdown_stride;
  int M, inter;
};

// One warp per (distinct slot d, token m < M, 128-channel group g); the grid
// covers the most distinct experts the call can route to (M * topk, at most
// kMoeMaxDistinct).
__global__ void moe_mid_kernel(const MoeMidArgs a) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const long long wid = (long long)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const int NG = a.inter / kHad;
  const int d = static_cast<int>(wid / (a.M * NG));
  const int rem = static_cast<int>(wid - (long long)d * a.M * NG);
  const int m = rem / NG;
  const int g = rem - m * NG;
  if (d >= kMoeMaxSlots) return;
  const MoeRoute* r = a.route;
  if (d >= r->n_distinct) return;
  const int e = r->expert[d];
  if (m >= a.M) return;
  const bool routed = (r->mask[d] >> m) & 1u;
  const int n0 = g * kHad + 4 * lane;
  float h[4] = {0.f, 0.f, 0.f, 0.f};
  if (routed) {
    const size_t off = (size_t)e * a.inter + n0;
    const float4 sg = load4_f32(a.sv_gate + off);
    const float4 su = load4_f32(a.sv_up + off);
    const float4 sd = load4_f32(a.su_down + off);
    const GemvJob& jg = a.jobs1[(2 * d) * a.jobs_per_matrix];
    const GemvJob& ju = a.jobs1[(2 * d + 1) * a.jobs_per_matrix];
    float gv[4], uv[4];
    sum_slots_pair<kMoeSlots>(jg.part, jg.unit_begin, ju.part, ju.unit_begin, jg.KT, jg.N,
                              r->units1, r->grid1, kMoeMaxTokens, m, g, lane, gv, uv);
    fwht128_warp(gv, lane);
    fwht128_warp(uv, lane);
    const float sgv[4] = {sg.x, sg.y, sg.z, sg.w};
    const float suv[4] = {su.x, su.y, su.z, su.w};
    const float sdv[4] = {sd.x, sd.y, sd.z, sd.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float gg = gv[q] * kHadScale * sgv[q];
      const float uu = uv[q] * kHadScale * suv[q];
      h[q] = silu(gg) * uu * sdv[q];
    }
    fwht128_warp(h, lane);
  }
  uint32_t* xf = a.xfrag_down + d * a.xdown_stride;
#pragma unroll
  for (int q = 0; q < 4; ++q) xfrag_store(xf, a.M, m, n0 + q, float_to_half_bits(h[q] * kHadScale));
}

struct MoeOutArgs {
  const MoeRoute* route;
  const GemvJob* jobs2;
  const float* expert_w;  // [M][topk]
  const float* sv_hidden;
  uint16_t* y;
  int M, topk, hidden;
};

// One block per (token m, 128-channel group g of the hidden side), one warp
// per expert slot of the token: warp k < topk sums routed expert k's partial
// slots, warp kMoeMaxTopk the shared expert's, all at once (each is a chain
// of dependent loads: route, job, partial sums); then warp 0 adds them in
// routing order (the shared expert last, weight 1), transforms and scales.
constexpr int kOutWarps = kMoeMaxTopk + 1;
__global__ void __launch_bounds__(32 * kOutWarps) moe_out_kernel(const MoeOutArgs a) {
  __shared__ float4 ps[kOutWarps][32];
  pdl_wait();
  const int lane = threadIdx.x & 31, k = threadIdx.x >> 5;
  const int NG = a.hidden / kHad;
  const int m = blockIdx.x / NG;
  const int g = blockIdx.x - m * NG;
  const MoeRoute* r = a.route;
  const int d = k < a.topk ? r->route[m * a.topk + k] : (k == kMoeMaxTopk ? r->shared_slot : -1);
  float p[4] = {0.f, 0.f, 0.f, 0.f};
  if (d >= 0) {
    const GemvJob& j = a.jobs2[d];
    sum_slots<kMoeSlots>(j.part, j.unit_begin, j.KT, j.N, r->units2, r->grid2, kMoeMaxTokens, m, g,
                         lane, p);
  }
  ps[k][lane] = make_float4(p[0], p[1], p[2], p[3]);
  __syncthreads();
  if (k != 0) return;
  const int n0 = g * kHad + 4 * lane;
  const float4 s = load4_f32(a.sv_hidden + n0);
  float v[4] = {0.f, 0.f, 0.f, 0.f};
  for (int kk = 0; kk < a.topk; ++kk) {
    if (r->route[m * a.topk + kk] < 0) continue;
    const float w = a.expert_w[m * a.topk + kk];
    const float4 q = ps[kk][lane];
    v[0] += w * q.x;
    v[1] += w * q.y;
    v[2] += w * q.z;
    v[3] += w * q.w;
  }
  if (r->shared_slot >= 0) {
    const float4 q = ps[kMoeMaxTopk][lane];
    v[0] += q.x;
    v[1] += q.y;
    v[2] += q.z;
    v[3] += q.w;
  }
  fwht128_warp(v, lane);
  v[0] *= kHadScale * s.x;
  v[1] *= kHadScale * s.y;
  v[2] *= kHadScale * s.z;
  v[3] *= kHadScale * s.w;
  store4_half(a.y + (size_t)m * a.hidden + n0, v);
}

unsigned blocks_for(long long warps) {
  return static_cast<unsigned>((warps + kWarpsPerBlock - 1) / kWarpsPerBlock);
}


template <typename T>
escha_status_t upload(T** dst, const T* host, size_t n) {
  escha_status_t s = dev_alloc(dst, n);
  if (s != ESCHA_OK) return s;
  return cudaMemcpy(*dst, host, n * sizeof(T), cudaMemcpyHostToDevice) == cudaSuccess
             ? ESCHA_OK
             : ESCHA_ERR_CUDA;
}

}  // namespace

// Folded side vectors and the per-call scratch, shared by both ways of
// storing the experts.  jobs1_count: gate/up jobs of the largest call.
static escha_status_t moe_init_common(escha_moe_s* h, const uint16_t* rin_hidden,
                               const float* s_in_hidden, const uint16_t* rout_gate,
                               const float* s_out_gate, const uint16_t* rout_up,
                               const float* s_out_up, const uint16_t* rin_down,
                               const float* s_in_down, const uint16_t* rout_hidden,
                               const float* s_out_hidden, size_t jobs1_count, cudaStream_t st) {
  escha_status_t s = ESCHA_OK;
  const int E = h->E, hidden = h->hidden, inter = h->inter;
  const size_t ei = (size_t)E * inter;
  const size_t ei1 = ei + inter;  // one more row: the shared expert
  if ((s = dev_alloc(&h->su_hidden, hidden)) != ESCHA_OK) return s;
  if ((s = dev_alloc(&h->sv_hidden, hidden)) != ESCHA_OK) return s;
  if ((s = dev_alloc(&h->sv_gate, ei1)) != ESCHA_OK) return s;
  if ((s = dev_alloc(&h->sv_up, ei1)) != ESCHA_OK) return s;
  if ((s = dev_alloc(&h->su_down, ei1)) != ESCHA_OK) return s;
  if (launch_fold_scales(rin_hidden, s_in_hidden, h->su_hidden, hidden, st) != cudaSuccess ||
      launch_fold_scales(rout_hidden, s_out_hidden, h->sv_hidden, hidden, st) != cudaSuccess ||
      launch_fold_scales(rout_gate, s_out_gate, h->sv_gate, static_cast<int>(ei), st) != cudaSuccess ||
      launch_fold_scales(rout_up, s_out_up, h->sv_up, static_cast<int>(ei), st) != cudaSuccess ||
      launch_fold_scales(rin_down, s_in_down, h->su_down, static_cast<int>(ei), st) != cudaSuccess)
    return ESCHA_ERR_CUDA;

  h->xdown_stride = (size_t)(inter / 16) * kMoeMaxTokens * 16;  // words per distinct slot
  h->part1_stride = (size_t)kMoeSlots * kMoeMaxTokens * inter;
  h->part2_stride = (size_t)kMoeSlots * kMoeMaxTokens * hidden;
  if ((s = dev_alloc(&h->xfrag_hidden, (size_t)(hidden / 16) * kMoeMaxTokens * 16)) != ESCHA_OK)
    return s;
  if ((s = dev_alloc(&h->xfrag_down, h->xdown_stride * kMoeMaxSlots)) != ESCHA_OK) return s;
  if ((s = dev_alloc(&h->part1, h->part1_stride * 2 * kMoeMaxSlots)) != ESCHA_OK) return s;
  if ((s = dev_alloc(&h->part2, h->part2_stride * kMoeMaxSlots)) != ESCHA_OK) return s;
  if ((s = dev_alloc(&h->jobs1, jobs1_count)) != ESCHA_OK) return s;
  if ((s = dev_alloc(&h->jobs2, kMoeMaxSlots)) != ESCHA_OK) return s;
  unsigned char* rt = nullptr;
  if ((s = dev_alloc(&rt, sizeof(MoeRoute))) != ESCHA_OK) return s;
  h->route = rt;
  if ((s = dev_alloc(&h->err, 1)) != ESCHA_OK) return s;
  if (cudaMemset(h->err, 0, sizeof(int)) != cudaSuccess) return ESCHA_ERR_CUDA;
  if (cudaMemset(h->route, 0, sizeof(MoeRoute)) != cudaSuccess) return ESCHA_ERR_CUDA;
  h->grid_max = h->num_sms * gemv_ranges_per_sm();
  if (cudaStreamSynchronize(st) != cudaSuccess) return ESCHA_ERR_CUDA;
  return ESCHA_OK;
}

escha_status_t moe_init(escha_moe_s* h, int E, int hidden, int inter,
                        const int16_t* const* gate_code, const int16_t* const* up_code,
                        const int16_t* const* down_code, const int32_t* bits,
                        const uint16_t* rin_hidden, const float* s_in_hidden,
                        const uint16_t* rout_gate, const float* s_out_gate,
                        const uint16_t* rout_up, const float* s_out_up,
                        const uint16_t* rin_down, const float* s_in_down,
                        const uint16_t* rout_hidden, const float* s_out_hidden, cudaStream_t st) {
  escha_status_t s = device_info(&h->device, &h->num_sms);
  if (s != ESCHA_OK) return s;
  h->E = E;
  h->hidden = hidden;
  h->inter = inter;
  // Tables hold E + 1 entries: entry E is the shared expert
  // (escha_moe_set_shared_expert); until one is set it repeats expert 0 and
  // is never scheduled.
  const int Es = E + 1;
  std::vector<const uint8_t*> g(Es), u(Es), d(Es);
  std::vector<int> b(Es);
  for (int e = 0; e < Es; ++e) {
    const int src = e < E ? e : 0;
    g[e] = reinterpret_cast<const uint8_t*>(gate_code[src]);
    u[e] = reinterpret_cast<const uint8_t*>(up_code[src]);
    d[e] = reinterpret_cast<const uint8_t*>(down_code[src]);
    b[e] = bits[src];
  }
  if ((s = upload(&h->gate_code, g.data(), Es)) != ESCHA_OK) return s;
  if ((s = upload(&h->up_code, u.data(), Es)) != ESCHA_OK) return s;
  if ((s = upload(&h->down_code, d.data(), Es)) != ESCHA_OK) return s;
  if ((s = upload(&h->bits, b.data(), Es)) != ESCHA_OK) return s;
  {
    // Tensor maps of every expert's three code tensors, [gate | up | down][E + 1].
    std::vector<CUtensorMap> maps(3 * (size_t)Es);
    for (int e = 0; e < Es; ++e) {
      if (!encode_gemv_code_map(&maps[e], g[e], b[e], hidden / 16, inter / 16) ||
          !encode_gemv_code_map(&maps[Es + e], u[e], b[e], hidden / 16, inter / 16) ||
          !encode_gemv_code_map(&maps[2 * (size_t)Es + e], d[e], b[e], inter / 16, hidden / 16))
        return ESCHA_ERR_CUDA;
    }
    if ((s = upload(&h->code_maps, maps.data(), maps.size())) != ESCHA_OK) return s;
  }

  return moe_init_common(h, rin_hidden, s_in_hidden, rout_gate, s_out_gate, rout_up, s_out_up,
                         rin_down, s_in_down, rout_hidden, s_out_hidden, 2 * kMoeMaxSlots, st);
}

escha_status_t moe_init_halves(escha_moe_s* h, int E, int hidden, int inter,
                               const int16_t* const* gate_half, const int16_t* const* up_half,
                               const int16_t* const* down_half, const int32_t* gate_bits,
                               const int32_t* up_bits, const int32_t* down_bits,
                               const uint16_t* rin_hidden, const float* s_in_hidden,
                               const uint16_t* rout_gate, const float* s_out_gate,
                               const uint16_t* rout_up, const float* s_out_up,
                               const uint16_t* rin_down, const float* s_in_down,
                               const uint16_t* rout_hidden, const float* s_out_hidden,
                               cudaStream_t st) {
  escha_status_t s = device_info(&h->device, &h->num_sms);
  if (s != ESCHA_OK) return s;
  h->E = E;
  h->hidden = hidden;
  h->inter = inter;
  h->halves = 1;
  h->H = inter / 128;
  h->gate_half = reinterpret_cast<const uint8_t* const*>(gate_half);
  h->up_half = reinterpret_cast<const uint8_t* const*>(up_half);
  h->down_half = reinterpret_cast<const uint8_t* const*>(down_half);
  h->gate_bits = gate_bits;
  h->up_bits = up_bits;
  h->down_bits = down_bits;
  // Zero code as large as the largest half (4 bits), standing in for table
  // entries that fail the device-side checks.
  const size_t stand_bytes = (size_t)(hidden / 16) * 8 * 128;
  if ((s = dev_alloc(&h->stand_in, stand_bytes)) != ESCHA_OK) return s;
  if (cudaMemset(h->stand_in, 0, stand_bytes) != cudaSuccess) return ESCHA_ERR_CUDA;
  {
    CUtensorMap tm[3];
    for (int b = 2; b <= 4; ++b)
      if (!encode_gemv_half_map(&tm[b - 2], h->stand_in, b, hidden / 16)) return ESCHA_ERR_CUDA;
    if ((s = upload(&h->half_map_tmpl, tm, 3)) != ESCHA_OK) return s;
  }
  if ((s = dev_alloc(&h->half_maps, (size_t)E * h->H)) != ESCHA_OK) return s;
  if ((s = dev_alloc(&h->half_map_key, (size_t)E * h->H)) != ESCHA_OK) return s;
  if (cudaMemset(h->half_map_key, 0, (size_t)E * h->H * sizeof(unsigned long long)) != cudaSuccess)
    return ESCHA_ERR_CUDA;
  return moe_init_common(h, rin_hidden, s_in_hidden, rout_gate, s_out_gate, rout_up, s_out_up,
                         rin_down, s_in_down, rout_hidden, s_out_hidden,
                         (size_t)2 * kMoeMaxDistinct * h->H, st);
}

escha_status_t moe_set_shared_expert(escha_moe_s* h, const int16_t* gate_code,
                                     const int16_t* up_code, const int16_t* down_code, int bits,
                                     const uint16_t* rout_gate, const float* s_out_gate,
                                     const uint16_t* rout_up, const float* s_out_up,
                                     const uint16_t* rin_down, const float* s_in_down) {
  if (cudaDeviceSynchronize() != cudaSuccess) return ESCHA_ERR_CUDA;  // no call in flight
  if (!gate_code) {
    h->shared_on = 0;
    return ESCHA_OK;
  }
  const int E = h->E, Es = E + 1, hidden = h->hidden, inter = h->inter;
  const uint8_t* g = reinterpret_cast<const uint8_t*>(gate_code);
  const uint8_t* u = reinterpret_cast<const uint8_t*>(up_code);
  const uint8_t* d = reinterpret_cast<const uint8_t*>(down_code);
  CUtensorMap maps[3];
  if (!encode_gemv_code_map(&maps[0], g, bits, hidden / 16, inter / 16) ||
      !encode_gemv_code_map(&maps[1], u, bits, hidden / 16, inter / 16) ||
      !encode_gemv_code_map(&maps[2], d, bits, inter / 16, hidden / 16))
    return ESCHA_ERR_CUDA;
  bool ok = cudaMemcpy(h->gate_code + E, &g, sizeof(g), cudaMemcpyHostToDevice) == cudaSuccess &&
            cudaMemcpy(h->up_code + E, &u, sizeof(u), cudaMemcpyHostToDevice) == cudaSuccess &&
            cudaMemcpy(h->down_code + E, &d, sizeof(d), cudaMemcpyHostToDevice) == cudaSuccess &&
            cudaMemcpy(h->bits + E, &bits, sizeof(int), cudaMemcpyHostToDevice) == cudaSuccess;
  for (int p = 0; ok && p < 3; ++p)
    ok = cudaMemcpy(h->code_maps + (size_t)p * Es + E, &maps[p], sizeof(CUtensorMap),
                    cudaMemcpyHostToDevice) == cudaSuccess;
  const size_t off = (size_t)E * inter;
  ok = ok && launch_fold_scales(rout_gate, s_out_gate, h->sv_gate + off, inter, 0) == cudaSuccess &&
       launch_fold_scales(rout_up, s_out_up, h->sv_up + off, inter, 0) == cudaSuccess &&
       launch_fold_scales(rin_down, s_in_down, h->su_down + off, inter, 0) == cudaSuccess &&
       cudaDeviceSynchronize() == cudaSuccess;
  if (!ok) return ESCHA_ERR_CUDA;
  h->shared_on = 1;
  return ESCHA_OK;
}

void moe_free(escha_moe_s* h) {
  cudaFree(h->half_maps);
  cudaFree(h->half_map_key);
  cudaFree(h->half_map_tmpl);
  cudaFree(h->stand_in);
  cudaFree(h->code_maps);
  cudaFree(h->gate_code);
  cudaFree(h->up_code);
  cudaFree(h->down_code);
  cudaFree(h->bits);
  cudaFree(h->su_hidden);
  cudaFree(h->sv_hidden);
  cudaFree(h->sv_gate);
  cudaFree(h->sv_up);
  cudaFree(h->su_down);
  cudaFree(h->xfrag_hidden);
  cudaFree(h->xfrag_down);
  cudaFree(h->part1);
  cudaFree(h->part2);
  cudaFree(h->jobs1);
  cudaFree(h->jobs2);
  cudaFree(h->route);
  cudaFree(h->err);
}

escha_status_t moe_gemv_stage(escha_moe_s* h, int stage, const uint16_t* x, const int32_t* ids,
                              const float* w, uint16_t* y, int M, int topk, cudaStream_t st) {
  MoeRoute* route = reinterpret_cast<MoeRoute*>(h->route);
  cudaError_t e = cudaSuccess;
  switch (stage) {
    case 0: {
      // routing plan (block 0) and the shared input rotation (the other blocks)
      const MoeRotIn rot{x, h->su_hidden, h->xfrag_hidden, h->hidden, M};
      const unsigned nblk = plan_blocks(M, h->hidden);
      if (h->halves) {
        MoeHalvesPlanArgs pa;
        pa.ids = ids;
        pa.M = M;
        pa.topk = topk;
        pa.E = h->E;
        pa.H = h->H;
        pa.hidden = h->hidden;
        pa.inter = h->inter;
        pa.gate_half = h->gate_half;
        pa.up_half = h->up_half;
        pa.down_half = h->down_half;
        pa.gate_bits = h->gate_bits;
        pa.up_bits = h->up_bits;
        pa.down_bits = h->down_bits;
        pa.tmpl = h->half_map_tmpl;
        pa.half_maps = h->half_maps;
        pa.half_map_key = h->half_map_key;
        pa.stand_in = h->stand_in;
        pa.e4m3 = h->rounding == ESCHA_ROUND_E4M3 ? 1 : 0;
        pa.xfrag_hidden = h->xfrag_hidden;
        pa.xfrag_down = h->xfrag_down;
        pa.part1 = h->part1;
        pa.part2 = h->part2;
        pa.part1_stride = h->part1_stride;
        pa.part2_stride = h->part2_stride;
        pa.xdown_stride = h->xdown_stride;
        pa.jobs1 = h->jobs1;
        pa.jobs2 = h->jobs2;
        pa.route = route;
        pa.grid1_max = h->grid_max;
        pa.grid2_max = h->grid_max;
        pa.err = h->err;
        PdlLaunch pl(nblk, kPlanThreads, h->E * sizeof(int), st);
        e = cudaLaunchKernelEx(&pl.cfg, moe_plan_halves_kernel, pa, rot);
        break;
      }
      MoePlanArgs pa;
      pa.ids = ids;
      pa.M = M;
      pa.topk = topk;
      pa.E = h->E;
      pa.hidden = h->hidden;
      pa.inter = h->inter;
      pa.gate_code = h->gate_code;
      pa.up_code = h->up_code;
      pa.down_code = h->down_code;
      pa.code_maps = h->code_maps;
      pa.shared = h->shared_on;
      pa.e4m3 = h->rounding == ESCHA_ROUND_E4M3 ? 1 : 0;
      pa.bits = h->bits;
      pa.xfrag_hidden = h->xfrag_hidden;
      pa.xfrag_down = h->xfrag_down;
      pa.part1 = h->part1;
      pa.part2 = h->part2;
      pa.part1_stride = h->part1_stride;
      pa.part2_stride = h->part2_stride;
      pa.xdown_stride = h->xdown_stride;
      pa.jobs1 = h->jobs1;
      pa.jobs2 = h->jobs2;
      pa.route = route;
      pa.grid1_max = h->grid_max;
      pa.grid2_max = h->grid_max;
      pa.err = h->err;
      PdlLaunch pl(nblk, kPlanThreads, h->E * sizeof(int), st);
      e = cudaLaunchKernelEx(&pl.cfg, moe_plan_kernel, pa, rot);
      break;
    }
    case 1:
      h->prof.begin(st);
      // every job has the same number of units: one matrix, or one half of one
      e = launch_gemv_device_schedule(h->jobs1, &route->units1, &route->grid1, h->grid_max, M,
                                      kMoeMaxTokens, h->err, st,
                                      h->halves ? (long long)(h->hidden / 16)
                                                : (long long)(h->hidden / 16) * (h->inter / 128),
                                      false, h->halves ? kGemvColHalves : kGemvWhole,
                                      h->rounding == ESCHA_ROUND_E4M3);
      h->prof.end(st);
      break;
    case 2: {
      MoeMidArgs ma;
      ma.route = route;
      ma.jobs1 = h->jobs1;
      ma.jobs_per_matrix = h->halves ? h->H : 1;
      ma.sv_gate = h->sv_gate;
      ma.sv_up = h->sv_up;
      ma.su_down = h->su_down;
      ma.xfrag_down = h->xfrag_down;
      ma.xdown_stride = h->xdown_stride;
      ma.M = M;
      ma.inter = h->inter;
      const long long mid_warps =
          (long long)(std::min(kMoeMaxDistinct, M * topk) + (h->shared_on ? 1 : 0)) * M *
          (h->inter / kHad);
      PdlLaunch pl(blocks_for(mid_warps), 32 * kWarpsPerBlock, 0, st);
      e = cudaLaunchKernelEx(&pl.cfg, moe_mid_kernel, ma);
      break;
    }
    case 3:
      h->prof.begin(st);
      e = launch_gemv_device_schedule(h->jobs2, &route->units2, &route->grid2, h->grid_max, M,
                                      kMoeMaxTokens, h->err, st,
                                      h->halves ? (long long)h->H * (h->hidden / 128)
                                                : (long long)(h->inter / 16) * (h->hidden / 128),
                                      h->halves != 0, h->halves ? kGemvRowHalves : kGemvWhole,
                                      h->rounding == ESCHA_ROUND_E4M3);
      h->prof.end(st);
      break;
    case 4: {
      MoeOutArgs oa;
      oa.route = route;
      oa.jobs2 = h->jobs2;
      oa.expert_w = w;
      oa.sv_hidden = h->sv_hidden;
      oa.y = y;
      oa.M = M;
      oa.topk = topk;
      oa.hidden = h->hidden;
      PdlLaunch pl(static_cast<unsigned>(M * (h->hidden / kHad)), 32 * kOutWarps, 0, st);
      e = cudaLaunchKernelEx(&pl.cfg, moe_out_kernel, oa);
      break;
    }
    default:
      return ESCHA_ERR_INVALID_ARG;
  }
  return from_cuda(e);
}

escha_status_t moe_gemv(escha_moe_s* h, const uint16_t* x, const int32_t* ids, const float* w,
                        uint16_t* y, int M, int topk, cudaStream_t st) {
  for (int s = 0; s < ESCHA_MOE_STAGES; ++s) {
    const escha_status_t r = moe_gemv_stage(h, s, x, ids, w, y, M, topk, st);
    if (r != ESCHA_OK) return r;
  }
  return ESCHA_OK;
}

}  // namespace escha
