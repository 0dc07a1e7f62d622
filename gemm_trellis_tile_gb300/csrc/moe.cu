// Routed-expert layer at decode (EXLR8 page, "The sharing trick"; GLM-5.3
// expert shapes): y[m] = sum_k w[m,k] * down_e(silu(gate_e(x[m])) * up_e(x[m])).
//
// The hidden side of every expert is one shared rotation: gate and up read one
// rotated activation had(x * su_hidden), and down's outputs are summed before
// one shared output rotation had(.) * sv_hidden (exact by linearity).  The
// intermediate side is per expert.
//
// One call, six launches on the caller's stream, no host synchronisation:
//   1. rotate_in        xfrag_hidden = fp16(had128(x * su_hidden))
//   2. moe_plan         reads the routing on the device: distinct experts in
//                       order of first appearance, tokens per expert, and the
//                       job tables / unit counts / grid sizes of launches 3, 5
//   3. trellis GEMV     gate and up of every distinct expert (mixed widths)
//   4. moe_mid          per (expert, token): had(gate)*sv_g, had(up)*sv_u,
//                       silu(g)*u, then had(h * su_down) into that expert's
//                       down fragments (zeros for tokens not routed to it)
//   5. trellis GEMV     down of every distinct expert
//   6. moe_out          y = fp16(had(sum_k w_k * down partials) * sv_hidden)
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

struct MoeRoute {
  long long units1;  // gate+up GEMV
  long long units2;  // down GEMV
  int grid1, grid2;
  int n_distinct;
  int pad;
  int expert[kMoeMaxDistinct];              // expert id of distinct slot d
  unsigned mask[kMoeMaxDistinct];           // bit m set: token m routes to d
  int route[kMoeMaxTokens * kMoeMaxTopk];   // distinct slot of (m, k), -1 if skipped
};

struct MoePlanArgs {
  const int32_t* ids;
  int M, topk, E;
  int hidden, inter;
  const uint8_t* const* gate_code;
  const uint8_t* const* up_code;
  const uint8_t* const* down_code;
  const CUtensorMap* code_maps;  // [3][E]: gate, up, down
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

// Grid size that gives every CTA at least a quarter of a group's k-tiles, so
// a group's units span at most five CTAs (five partial-sum slots).
__device__ __forceinline__ int device_grid(long long units, int KT, int grid_max) {
  long long g = units * 4 / KT;
  if (g < 1) g = 1;
  if (g > grid_max) g = grid_max;
  return static_cast<int>(g);
}

__global__ void moe_plan_kernel(const MoePlanArgs a) {
  extern __shared__ int first_slot[];  // [E]: distinct slot of each expert, -1 if none yet
  __shared__ int s_nd;
  pdl_trigger();  // the GEMV may launch; it waits for this kernel before reading the plan
  for (int e = threadIdx.x; e < a.E; e += blockDim.x) first_slot[e] = -1;
  __syncthreads();
  MoeRoute* r = a.route;
  if (threadIdx.x == 0) {
    // Sequential on purpose: slots are numbered in order of first appearance.
    int nd = 0;
    for (int i = 0; i < a.M * a.topk; ++i) {
      const int e = a.ids[i];
      int d = -1;
      if (e >= 0 && e < a.E) {
        d = first_slot[e];
        if (d < 0) {
          d = nd++;
          first_slot[e] = d;
          r->expert[d] = e;
          r->mask[d] = 0u;
        }
        r->mask[d] |= 1u << (i / a.topk);
      } else {
        set_error(a.err, kDevErrBadRoute);
      }
      r->route[i] = d;
    }
    s_nd = nd;
  }
  __syncthreads();
  const int nd = s_nd;
  const int KTg = a.hidden / 16, NGg = a.inter / 128;
  const int KTd = a.inter / 16, NGd = a.hidden / 128;
  const long long ug = (long long)KTg * NGg, ud = (long long)KTd * NGd;
  // Slots past nd keep well-formed shapes (never scheduled: the unit counts stop at nd).
  for (int d = threadIdx.x; d < kMoeMaxDistinct; d += blockDim.x) {
    const int e = d < nd ? r->expert[d] : 0;
    const int b = a.bits[e];
    a.jobs1[2 * d] = make_job(a.gate_code[e], a.code_maps + e, a.xfrag_hidden,
                              a.part1 + (2 * d) * a.part1_stride, (2 * d) * ug, b, KTg, NGg,
                              a.inter, a.e4m3);
    a.jobs1[2 * d + 1] = make_job(a.up_code[e], a.code_maps + a.E + e, a.xfrag_hidden,
                                  a.part1 + (2 * d + 1) * a.part1_stride, (2 * d + 1) * ug, b, KTg,
                                  NGg, a.inter, a.e4m3);
    a.jobs2[d] = make_job(a.down_code[e], a.code_maps + 2 * a.E + e,
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
  // Finish only after the input rotation (launched before this kernel, which
  // does not read it) so that completing this kernel implies both.
  pdl_wait();
}

struct MoeMidArgs {
  const MoeRoute* route;
  const GemvJob* jobs1;
  const float* sv_gate;  // [E][inter]
  const float* sv_up;
  const float* su_down;
  uint32_t* xfrag_down;
  size_t xdown_stride;
  int M, inter;
};

// One warp per (distinct slot d, token slot m in 0..7, 128-channel group g).
__global__ void moe_mid_kernel(const MoeMidArgs a) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const long long wid = (long long)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const int NG = a.inter / kHad;
  const int d = static_cast<int>(wid / (8 * NG));
  const int rem = static_cast<int>(wid - (long long)d * 8 * NG);
  const int m = rem / NG;
  const int g = rem - m * NG;
  if (d >= kMoeMaxDistinct) return;
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
    const GemvJob& jg = a.jobs1[2 * d];
    const GemvJob& ju = a.jobs1[2 * d + 1];
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

// One warp per (token m, 128-channel group g of the hidden side).
__global__ void moe_out_kernel(const MoeOutArgs a) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const long long wid = (long long)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const int NG = a.hidden / kHad;
  if (wid >= (long long)a.M * NG) return;
  const int m = static_cast<int>(wid / NG);
  const int g = static_cast<int>(wid - (long long)m * NG);
  const MoeRoute* r = a.route;
  const int n0 = g * kHad + 4 * lane;
  const float4 s = load4_f32(a.sv_hidden + n0);
  // Routes, weights and job fields of all routed experts first (independent
  // loads), then their partial sums two experts at a time; the experts are
  // still added in routing order.
  int dk[kMoeMaxTopk];
  float wk[kMoeMaxTopk];
#pragma unroll
  for (int k = 0; k < kMoeMaxTopk; ++k) {
    dk[k] = k < a.topk ? r->route[m * a.topk + k] : -1;
    wk[k] = k < a.topk ? a.expert_w[m * a.topk + k] : 0.f;
  }
  float v[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int k = 0; k < kMoeMaxTopk; k += 2) {
    const int d0 = dk[k], d1 = dk[k + 1];
    float p0[4] = {0.f, 0.f, 0.f, 0.f}, p1[4] = {0.f, 0.f, 0.f, 0.f};
    if (d0 >= 0 && d1 >= 0) {
      const GemvJob& j0 = a.jobs2[d0];
      const GemvJob& j1 = a.jobs2[d1];
      sum_slots_pair<kMoeSlots>(j0.part, j0.unit_begin, j1.part, j1.unit_begin, j0.KT, j0.N,
                                r->units2, r->grid2, kMoeMaxTokens, m, g, lane, p0, p1);
    } else if (d0 >= 0 || d1 >= 0) {
      const GemvJob& j = a.jobs2[d0 >= 0 ? d0 : d1];
      sum_slots<kMoeSlots>(j.part, j.unit_begin, j.KT, j.N, r->units2, r->grid2, kMoeMaxTokens, m,
                           g, lane, d0 >= 0 ? p0 : p1);
    }
    if (d0 >= 0) {
#pragma unroll
      for (int q = 0; q < 4; ++q) v[q] += wk[k] * p0[q];
    }
    if (d1 >= 0) {
#pragma unroll
      for (int q = 0; q < 4; ++q) v[q] += wk[k + 1] * p1[q];
    }
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
  std::vector<const uint8_t*> g(E), u(E), d(E);
  std::vector<int> b(E);
  for (int e = 0; e < E; ++e) {
    g[e] = reinterpret_cast<const uint8_t*>(gate_code[e]);
    u[e] = reinterpret_cast<const uint8_t*>(up_code[e]);
    d[e] = reinterpret_cast<const uint8_t*>(down_code[e]);
    b[e] = bits[e];
  }
  if ((s = upload(&h->gate_code, g.data(), E)) != ESCHA_OK) return s;
  if ((s = upload(&h->up_code, u.data(), E)) != ESCHA_OK) return s;
  if ((s = upload(&h->down_code, d.data(), E)) != ESCHA_OK) return s;
  if ((s = upload(&h->bits, b.data(), E)) != ESCHA_OK) return s;
  {
    // Tensor maps of every expert's three code tensors, [gate | up | down][E].
    std::vector<CUtensorMap> maps(3 * (size_t)E);
    for (int e = 0; e < E; ++e) {
      if (!encode_gemv_code_map(&maps[e], g[e], b[e], hidden / 16, inter / 16) ||
          !encode_gemv_code_map(&maps[E + e], u[e], b[e], hidden / 16, inter / 16) ||
          !encode_gemv_code_map(&maps[2 * (size_t)E + e], d[e], b[e], inter / 16, hidden / 16))
        return ESCHA_ERR_CUDA;
    }
    if ((s = upload(&h->code_maps, maps.data(), maps.size())) != ESCHA_OK) return s;
  }

  const size_t ei = (size_t)E * inter;
  if ((s = dev_alloc(&h->su_hidden, hidden)) != ESCHA_OK) return s;
  if ((s = dev_alloc(&h->sv_hidden, hidden)) != ESCHA_OK) return s;
  if ((s = dev_alloc(&h->sv_gate, ei)) != ESCHA_OK) return s;
  if ((s = dev_alloc(&h->sv_up, ei)) != ESCHA_OK) return s;
  if ((s = dev_alloc(&h->su_down, ei)) != ESCHA_OK) return s;
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
  if ((s = dev_alloc(&h->xfrag_down, h->xdown_stride * kMoeMaxDistinct)) != ESCHA_OK) return s;
  if ((s = dev_alloc(&h->part1, h->part1_stride * 2 * kMoeMaxDistinct)) != ESCHA_OK) return s;
  if ((s = dev_alloc(&h->part2, h->part2_stride * kMoeMaxDistinct)) != ESCHA_OK) return s;
  if ((s = dev_alloc(&h->jobs1, 2 * kMoeMaxDistinct)) != ESCHA_OK) return s;
  if ((s = dev_alloc(&h->jobs2, kMoeMaxDistinct)) != ESCHA_OK) return s;
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

void moe_free(escha_moe_s* h) {
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
      RotInJob rj{x, h->su_hidden, h->xfrag_hidden, h->hidden};
      e = launch_rotate_in_xfrag(&rj, 1, M, st);
      break;
    }
    case 1: {
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
      PdlLaunch pl(1, 128, h->E * sizeof(int), st);
      e = cudaLaunchKernelEx(&pl.cfg, moe_plan_kernel, pa);
      break;
    }
    case 2:
      h->prof.begin(st);
      e = launch_gemv_device_schedule(h->jobs1, &route->units1, &route->grid1, h->grid_max, M,
                                      kMoeMaxTokens, h->err, st);
      h->prof.end(st);
      break;
    case 3: {
      MoeMidArgs ma;
      ma.route = route;
      ma.jobs1 = h->jobs1;
      ma.sv_gate = h->sv_gate;
      ma.sv_up = h->sv_up;
      ma.su_down = h->su_down;
      ma.xfrag_down = h->xfrag_down;
      ma.xdown_stride = h->xdown_stride;
      ma.M = M;
      ma.inter = h->inter;
      const long long mid_warps = (long long)kMoeMaxDistinct * 8 * (h->inter / kHad);
      PdlLaunch pl(blocks_for(mid_warps), 32 * kWarpsPerBlock, 0, st);
      e = cudaLaunchKernelEx(&pl.cfg, moe_mid_kernel, ma);
      break;
    }
    case 4:
      h->prof.begin(st);
      e = launch_gemv_device_schedule(h->jobs2, &route->units2, &route->grid2, h->grid_max, M,
                                      kMoeMaxTokens, h->err, st);
      h->prof.end(st);
      break;
    case 5: {
      MoeOutArgs oa;
      oa.route = route;
      oa.jobs2 = h->jobs2;
      oa.expert_w = w;
      oa.sv_hidden = h->sv_hidden;
      oa.y = y;
      oa.M = M;
      oa.topk = topk;
      oa.hidden = h->hidden;
      const long long out_warps = (long long)M * (h->hidden / kHad);
      PdlLaunch pl(blocks_for(out_warps), 32 * kWarpsPerBlock, 0, st);
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
