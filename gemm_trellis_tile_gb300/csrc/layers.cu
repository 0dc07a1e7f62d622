// Host orchestration of the dense trellis layer and the gated MLP at decode.
//
// Dense layer, 1..16 tokens (three launches on the caller's stream):
//   1. rotate_in:  xfrag = fp16(had128(x * su)) in the GEMV's fragment order
//   2. trellis GEMV: fp32 partial sums of xh @ W_inner (decode in registers)
//   3. rotate_out: y = fp16(had128(sum of partials) * sv)
// Gated MLP (five launches): both input rotations in one launch, gate and up
// contracted in one GEMV launch, one fused middle kernel (output rotations,
// silu(g)*u, the down layer's input rotation), the down GEMV, and the output
// rotation.

#include <cuda_runtime.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <utility>

#include "api_internal.h"

namespace escha {

cudaError_t set_smem_limit(const void* func, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  // The largest limit set so far per (kernel, device): a launch with less
  // dynamic shared memory than the limit is fine, so the limit only rises
  // (kernels whose shared memory depends on the layer see several sizes).
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> limit;
  std::lock_guard<std::mutex> lock(mu);
  int& cur = limit[std::make_pair(func, dev)];
  if (bytes <= cur) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) cur = bytes;
  return e;
}

template <typename T>
escha_status_t dev_alloc(T** p, size_t count) {
  *p = nullptr;
  if (count == 0) return ESCHA_OK;
  cudaError_t e = cudaMalloc(reinterpret_cast<void**>(p), count * sizeof(T));
  if (e != cudaSuccess) {
    cudaGetLastError();
    *p = nullptr;
    return e == cudaErrorMemoryAllocation ? ESCHA_ERR_OOM : ESCHA_ERR_CUDA;
  }
  return ESCHA_OK;
}
template escha_status_t dev_alloc<int>(int**, size_t);
template escha_status_t dev_alloc<float>(float**, size_t);
template escha_status_t dev_alloc<uint32_t>(uint32_t**, size_t);
template escha_status_t dev_alloc<uint16_t>(uint16_t**, size_t);
template escha_status_t dev_alloc<GemvJob>(GemvJob**, size_t);
template escha_status_t dev_alloc<const uint8_t*>(const uint8_t***, size_t);
template escha_status_t dev_alloc<unsigned char>(unsigned char**, size_t);
template escha_status_t dev_alloc<CUtensorMap>(CUtensorMap**, size_t);
template escha_status_t dev_alloc<unsigned long long>(unsigned long long**, size_t);

namespace {

GemvJob make_job(const escha_linear_s* h, const uint32_t* xfrag, float* part) {
  GemvJob j;
  j.code = reinterpret_cast<const uint8_t*>(h->code);
  j.tmap = h->tmap;
  j.xfrag = reinterpret_cast<const uint4*>(xfrag);
  j.part = part;
  j.unit_begin = 0;
  j.bits = h->bits;
  j.KT = h->K / 16;
  j.NG = h->N / 128;
  j.N = h->N;
  j.e4m3 = h->rounding == ESCHA_ROUND_E4M3 ? 1 : 0;
  return j;
}

size_t xfrag_words(int K) { return (size_t)(K / 16) * kGemvMaxTokens * 16; }

PartRef part_ref(const GemvSchedule& s, int job) {
  PartRef r;
  r.part = s.jobs[job].part;
  r.unit_begin = s.jobs[job].unit_begin;
  r.KT = s.jobs[job].KT;
  r.N = s.jobs[job].N;
  return r;
}

}  // namespace

escha_status_t linear_init(escha_linear_s* h, const int16_t* code, int bits, int K, int N,
                           const uint16_t* rin, const uint16_t* rout, const float* s_in,
                           const float* s_out, cudaStream_t st) {
  escha_status_t s = device_info(&h->device, &h->num_sms);
  if (s != ESCHA_OK) return s;
  h->K = K;
  h->N = N;
  h->bits = bits;
  h->code = code;
  if ((s = dev_alloc(&h->su, K)) != ESCHA_OK) return s;
  if ((s = dev_alloc(&h->sv, N)) != ESCHA_OK) return s;
  if ((s = dev_alloc(&h->xfrag, xfrag_words(K))) != ESCHA_OK) return s;
  if ((s = dev_alloc(&h->err, 1)) != ESCHA_OK) return s;
  if (cudaMemset(h->err, 0, sizeof(int)) != cudaSuccess) return ESCHA_ERR_CUDA;
  {
    CUtensorMap map;
    if (!encode_gemv_code_map(&map, code, bits, K / 16, N / 16)) return ESCHA_ERR_CUDA;
    unsigned char* d = nullptr;
    if ((s = dev_alloc(&d, sizeof(CUtensorMap))) != ESCHA_OK) return s;
    h->tmap = reinterpret_cast<CUtensorMap*>(d);
    if (cudaMemcpy(h->tmap, &map, sizeof(map), cudaMemcpyHostToDevice) != cudaSuccess)
      return ESCHA_ERR_CUDA;
  }

  if (launch_fold_scales(rin, s_in, h->su, K, st) != cudaSuccess) return ESCHA_ERR_CUDA;
  if (launch_fold_scales(rout, s_out, h->sv, N, st) != cudaSuccess) return ESCHA_ERR_CUDA;

  h->sched.jobs.assign(1, make_job(h, h->xfrag, nullptr));
  plan_gemv(h->sched, h->num_sms, gemv_ranges_per_sm());
  if ((s = dev_alloc(&h->part, (size_t)h->sched.max_slots * kGemvMaxTokens * N)) != ESCHA_OK)
    return s;
  h->sched.jobs[0].part = h->part;
  if ((s = upload_jobs(h->sched)) != ESCHA_OK) return s;
  if (cudaStreamSynchronize(st) != cudaSuccess) return ESCHA_ERR_CUDA;
  return ESCHA_OK;
}

void linear_free(escha_linear_s* h) {
  cudaFree(h->tmap);
  cudaFree(h->su);
  cudaFree(h->sv);
  cudaFree(h->xfrag);
  cudaFree(h->part);
  cudaFree(h->err);
  cudaFree(h->sched.d_jobs);
  cudaFree(h->xh);
  cudaFree(h->xd);
  cudaFree(h->gemm_ws);
  cudaFree(h->gemm_cnt);
  h->gemm_ws = nullptr;
  h->gemm_cnt = nullptr;
  h->gemm_cnt_ints = 0;
  h->xd = nullptr;
  h->su = h->sv = nullptr;
  h->xfrag = nullptr;
  h->tmap = nullptr;
  h->part = nullptr;
  h->err = nullptr;
  h->sched.d_jobs = nullptr;
  h->xh = nullptr;
}

escha_status_t linear_gemv_stage(escha_linear_s* h, int stage, const uint16_t* x, uint16_t* y,
                                 int M, cudaStream_t st) {
  cudaError_t e = cudaSuccess;
  switch (stage) {
    case 0: {
      RotInJob rj{x, h->su, h->xfrag, h->K};
      e = launch_rotate_in_xfrag(&rj, 1, M, st);
      break;
    }
    case 1:
      h->prof.begin(st);
      e = launch_gemv(h->sched, M, h->err, st);
      h->prof.end(st);
      break;
    case 2:
      e = launch_rotate_out(part_ref(h->sched, 0), h->sched.units, h->sched.grid, h->sv, y, M,
                            kGemvMaxTokens, st);
      break;
    default:
      return ESCHA_ERR_INVALID_ARG;
  }
  return from_cuda(e);
}

escha_status_t linear_gemv(escha_linear_s* h, const uint16_t* x, uint16_t* y, int M,
                           cudaStream_t st) {
  for (int s = 0; s < ESCHA_LINEAR_STAGES; ++s) {
    const escha_status_t r = linear_gemv_stage(h, s, x, y, M, st);
    if (r != ESCHA_OK) return r;
  }
  return ESCHA_OK;
}

escha_status_t linear_set_rounding(escha_linear_s* h, int rounding) {
  if (cudaDeviceSynchronize() != cudaSuccess) return ESCHA_ERR_CUDA;  // no call in flight
  h->rounding = rounding;
  h->sched.jobs[0].e4m3 = rounding == ESCHA_ROUND_E4M3 ? 1 : 0;
  return upload_jobs(h->sched);
}

// Arrival counters for M-row prefill calls; a larger array replaces the old
// one after the device has finished with it.
escha_status_t reserve_counters(escha_linear_s* h, int M) {
  const size_t need = gemm_counter_ints(M, h->N);
  if (need <= h->gemm_cnt_ints) return ESCHA_OK;
  if (h->gemm_cnt) {
    if (cudaDeviceSynchronize() != cudaSuccess) return ESCHA_ERR_CUDA;
    cudaFree(h->gemm_cnt);
    h->gemm_cnt = nullptr;
    h->gemm_cnt_ints = 0;
  }
  escha_status_t s = dev_alloc(&h->gemm_cnt, need);
  if (s != ESCHA_OK) return s;
  h->gemm_cnt_ints = need;
  return ESCHA_OK;
}

escha_status_t linear_reserve(escha_linear_s* h, int rows) {
  if (rows <= h->xh_rows) return ESCHA_OK;
  if (h->xh) {
    if (cudaDeviceSynchronize() != cudaSuccess) return ESCHA_ERR_CUDA;
    cudaFree(h->xh);
    cudaFree(h->xd);
    h->xh = nullptr;
    h->xd = nullptr;
    h->xh_rows = 0;
  }
  escha_status_t s = dev_alloc(&h->xh, (size_t)rows * h->K);
  if (s != ESCHA_OK) return s;
  if ((s = dev_alloc(&h->xd, (size_t)rows)) != ESCHA_OK) return s;
  h->xh_rows = rows;
  if (!h->gemm_ws && (s = dev_alloc(&h->gemm_ws, gemm_workspace_floats(h->num_sms))) != ESCHA_OK)
    return s;
  return reserve_counters(h, rows);
}

// The prefill GEMM's split-tile workspace for M rows: partial sums (fixed size)
// and arrival counters (grown on demand).  The counters must be zero when the
// GEMM starts: the activation kernel that precedes it clears them, or, with
// clear set (no such kernel), a clear on `st` here.
escha_status_t gemm_prepare(escha_linear_s* h, int M, cudaStream_t st, bool clear) {
  escha_status_t s;
  if (!h->gemm_ws && (s = dev_alloc(&h->gemm_ws, gemm_workspace_floats(h->num_sms))) != ESCHA_OK)
    return s;
  if ((s = reserve_counters(h, M)) != ESCHA_OK) return s;
  if (!clear) return ESCHA_OK;
  return from_cuda(
      cudaMemsetAsync(h->gemm_cnt, 0, gemm_counter_ints(M, h->N) * sizeof(int), st));
}

escha_status_t linear_gemm(escha_linear_s* h, const uint16_t* x, uint16_t* y, int M,
                           cudaStream_t st) {
  escha_status_t s = linear_reserve(h, M);
  if (s != ESCHA_OK) return s;
  if ((s = gemm_prepare(h, M, st, false)) != ESCHA_OK) return s;
  cudaError_t e = launch_rotate_in_plain(x, h->su, h->xh, M, h->K, h->gemm_cnt,
                                         static_cast<int>(gemm_counter_ints(M, h->N)), st);
  if (e != cudaSuccess) return from_cuda(e);
  h->prof.begin(st);
  e = launch_trellis_gemm(h->xh, h->code, h->bits, h->rounding == ESCHA_ROUND_E4M3, M, h->K,
                          h->N, h->sv, y, h->gemm_ws, h->gemm_cnt,
                          h->num_sms, h->err, st);
  h->prof.end(st);
  return from_cuda(e);
}

// FP8 prefill (E4M3-rounded layers only): per-token E4M3 activations from the
// input rotation, then the kind::f8f6f4 GEMM; the codes reuse the rotated-
// activation workspace (K bytes of its 2K per row).
escha_status_t linear_gemm_fp8(escha_linear_s* h, const uint16_t* x, uint16_t* y, int M,
                               cudaStream_t st) {
  if (h->rounding != ESCHA_ROUND_E4M3) return ESCHA_ERR_UNSUPPORTED;
  if (quantize_e4m3_smem_bytes(h->K) > kMaxQuantSmem) return ESCHA_ERR_UNSUPPORTED;
  escha_status_t s = linear_reserve(h, M);
  if (s != ESCHA_OK) return s;
  if ((s = gemm_prepare(h, M, st, false)) != ESCHA_OK) return s;
  uint8_t* xq = reinterpret_cast<uint8_t*>(h->xh);
  cudaError_t e = launch_quantize_e4m3_rows(x, h->su, xq, h->xd, M, h->K, h->gemm_cnt,
                                            static_cast<int>(gemm_counter_ints(M, h->N)), st);
  if (e != cudaSuccess) return from_cuda(e);
  h->prof.begin(st);
  e = launch_trellis_gemm_fp8(xq, h->xd, h->code, h->bits, M, h->K, h->N, h->sv, y, h->gemm_ws,
                              h->gemm_cnt, h->num_sms, h->err, st);
  h->prof.end(st);
  return from_cuda(e);
}

escha_status_t linear_gemm_fp8_codes(escha_linear_s* h, const uint8_t* q, const float* d,
                                     uint16_t* y, int M, cudaStream_t st) {
  if (h->rounding != ESCHA_ROUND_E4M3) return ESCHA_ERR_UNSUPPORTED;
  escha_status_t s = gemm_prepare(h, M, st, true);
  if (s != ESCHA_OK) return s;
  h->prof.begin(st);
  cudaError_t e = launch_trellis_gemm_fp8(q, d, h->code, h->bits, M, h->K, h->N, h->sv, y,
                                          h->gemm_ws, h->gemm_cnt, h->num_sms, h->err, st);
  h->prof.end(st);
  return from_cuda(e);
}

escha_status_t mlp_init(escha_mlp_s* m, escha_linear_s* gate, escha_linear_s* up,
                        escha_linear_s* down) {
  m->gate = gate;
  m->up = up;
  m->down = down;
  escha_status_t s;
  if ((s = dev_alloc(&m->xfrag_gate, xfrag_words(gate->K))) != ESCHA_OK) return s;
  if ((s = dev_alloc(&m->xfrag_up, xfrag_words(up->K))) != ESCHA_OK) return s;
  if ((s = dev_alloc(&m->xfrag_down, xfrag_words(down->K))) != ESCHA_OK) return s;
  if ((s = dev_alloc(&m->err, 1)) != ESCHA_OK) return s;
  if (cudaMemset(m->err, 0, sizeof(int)) != cudaSuccess) return ESCHA_ERR_CUDA;

  const int cps = gemv_ranges_per_sm();
  m->s_gate_up.jobs = {make_job(gate, m->xfrag_gate, nullptr), make_job(up, m->xfrag_up, nullptr)};
  plan_gemv(m->s_gate_up, gate->num_sms, cps);
  m->s_down.jobs = {make_job(down, m->xfrag_down, nullptr)};
  plan_gemv(m->s_down, down->num_sms, cps);
  const size_t rows = (size_t)kGemvMaxTokens;
  if ((s = dev_alloc(&m->part_gate, m->s_gate_up.max_slots * rows * gate->N)) != ESCHA_OK) return s;
  if ((s = dev_alloc(&m->part_up, m->s_gate_up.max_slots * rows * up->N)) != ESCHA_OK) return s;
  if ((s = dev_alloc(&m->part_down, m->s_down.max_slots * rows * down->N)) != ESCHA_OK) return s;
  m->s_gate_up.jobs[0].part = m->part_gate;
  m->s_gate_up.jobs[1].part = m->part_up;
  m->s_down.jobs[0].part = m->part_down;
  if ((s = upload_jobs(m->s_gate_up)) != ESCHA_OK) return s;
  if ((s = upload_jobs(m->s_down)) != ESCHA_OK) return s;
  return ESCHA_OK;
}

void mlp_free(escha_mlp_s* m) {
  cudaFree(m->xfrag_gate);
  cudaFree(m->xfrag_up);
  cudaFree(m->xfrag_down);
  cudaFree(m->part_gate);
  cudaFree(m->part_up);
  cudaFree(m->part_down);
  cudaFree(m->err);
  cudaFree(m->norm_g_gate);
  cudaFree(m->norm_g_up);
  cudaFree(m->s_gate_up.d_jobs);
  cudaFree(m->s_down.d_jobs);
}

escha_status_t mlp_gemv_stage(escha_mlp_s* m, int stage, const uint16_t* x, uint16_t* y, int M,
                              cudaStream_t st) {
  cudaError_t e = cudaSuccess;
  switch (stage) {
    case 0: {
      if (m->norm_on) {
        e = launch_rotate_in_norm(x, m->norm_g_gate, m->norm_g_up, m->xfrag_gate, m->xfrag_up,
                                  m->gate->K, M, m->norm_eps, st);
        break;
      }
      RotInJob rj[2] = {{x, m->gate->su, m->xfrag_gate, m->gate->K},
                        {x, m->up->su, m->xfrag_up, m->up->K}};
      e = launch_rotate_in_xfrag(rj, 2, M, st);
      break;
    }
    case 1:
      m->prof.begin(st);
      e = launch_gemv(m->s_gate_up, M, m->err, st);
      m->prof.end(st);
      break;
    case 2:
      e = launch_mlp_mid(part_ref(m->s_gate_up, 0), part_ref(m->s_gate_up, 1), m->s_gate_up.units,
                         m->s_gate_up.grid, m->gate->sv, m->up->sv, m->down->su, m->xfrag_down, M,
                         st);
      break;
    case 3:
      m->prof.begin(st);
      e = launch_gemv(m->s_down, M, m->err, st);
      m->prof.end(st);
      break;
    case 4:
      e = launch_rotate_out(part_ref(m->s_down, 0), m->s_down.units, m->s_down.grid, m->down->sv,
                            y, M, kGemvMaxTokens, st);
      break;
    default:
      return ESCHA_ERR_INVALID_ARG;
  }
  return from_cuda(e);
}

escha_status_t mlp_set_input_norm(escha_mlp_s* m, const uint16_t* w, float eps,
                                  int stored_minus_one) {
  if (cudaDeviceSynchronize() != cudaSuccess) return ESCHA_ERR_CUDA;  // no call in flight
  if (!w) {
    m->norm_on = 0;
    return ESCHA_OK;
  }
  const int K = m->gate->K;
  escha_status_t s;
  if (!m->norm_g_gate && (s = dev_alloc(&m->norm_g_gate, K)) != ESCHA_OK) return s;
  if (!m->norm_g_up && (s = dev_alloc(&m->norm_g_up, K)) != ESCHA_OK) return s;
  const float off = stored_minus_one ? 1.0f : 0.0f;
  if (launch_fold_norm(w, off, m->gate->su, m->norm_g_gate, K, 0) != cudaSuccess ||
      launch_fold_norm(w, off, m->up->su, m->norm_g_up, K, 0) != cudaSuccess ||
      cudaDeviceSynchronize() != cudaSuccess)
    return ESCHA_ERR_CUDA;
  m->norm_eps = eps;
  m->norm_on = 1;
  return ESCHA_OK;
}

escha_status_t mlp_gemv(escha_mlp_s* m, const uint16_t* x, uint16_t* y, int M, cudaStream_t st) {
  for (int s = 0; s < ESCHA_MLP_STAGES; ++s) {
    const escha_status_t r = mlp_gemv_stage(m, s, x, y, M, st);
    if (r != ESCHA_OK) return r;
  }
  return ESCHA_OK;
}

Profiler* profiler_of(void* handle, int kind) {
  if (!handle) return nullptr;
  switch (kind) {
    case ESCHA_KIND_LINEAR: return &static_cast<escha_linear_s*>(handle)->prof;
    case ESCHA_KIND_MLP: return &static_cast<escha_mlp_s*>(handle)->prof;
    case ESCHA_KIND_MOE: return &static_cast<escha_moe_s*>(handle)->prof;
    default: return nullptr;
  }
}

}  // namespace escha
