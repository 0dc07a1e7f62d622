// C ABI of libescha (declared in include/escha.h): handle life cycle, argument
// validation, scheduling of the trellis kernels and status reporting.

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <cstdlib>
#include <new>
#include <utility>
#include <vector>

#include "api_internal.h"
#include "escha.h"
#include "internal.h"

using namespace escha;

namespace escha {

static thread_local char g_last_error[256] = "";

escha_status_t from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return ESCHA_OK;
  snprintf(g_last_error, sizeof(g_last_error), "%s: %s", cudaGetErrorName(e),
           cudaGetErrorString(e));
  if (e == cudaErrorMemoryAllocation) return ESCHA_ERR_OOM;
  return ESCHA_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---------------------------------------------------------------- profiler

// Inside stream capture a plain cudaEventRecord only orders captured work; an
// external record turns into an event node that fires on every graph replay.
static void record(cudaEvent_t ev, cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(ev, st, cudaEventRecordExternal);
  else
    cudaEventRecord(ev, st);
}

void Profiler::begin(cudaStream_t st) {
  if (!on) return;
  std::pair<cudaEvent_t, cudaEvent_t> ev{nullptr, nullptr};
  if (!pool.empty()) {
    ev = pool.back();
    pool.pop_back();
  } else {
    cudaEventCreate(&ev.first);
    cudaEventCreate(&ev.second);
  }
  record(ev.first, st);
  pending.push_back(ev);
}

void Profiler::end(cudaStream_t st) {
  if (!on || pending.empty()) return;
  record(pending.back().second, st);
}

escha_status_t Profiler::collect(double* ms_total, int* launches) {
  double total = 0.0;
  int n = 0;
  for (auto& ev : pending) {
    if (cudaEventSynchronize(ev.second) != cudaSuccess) return ESCHA_ERR_CUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, ev.first, ev.second) != cudaSuccess) return ESCHA_ERR_CUDA;
    total += ms;
    ++n;
    pool.push_back(ev);
  }
  pending.clear();
  if (ms_total) *ms_total = total;
  if (launches) *launches = n;
  return ESCHA_OK;
}

Profiler::~Profiler() {
  for (auto& ev : pending) pool.push_back(ev);
  for (auto& ev : pool) {
    cudaEventDestroy(ev.first);
    cudaEventDestroy(ev.second);
  }
}

// ---------------------------------------------------------------- device info

escha_status_t device_info(int* dev, int* sms) {
  if (cudaGetDevice(dev) != cudaSuccess) return ESCHA_ERR_CUDA;
  int major = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, *dev) != cudaSuccess)
    return ESCHA_ERR_CUDA;
  if (major != 10) return ESCHA_ERR_UNSUPPORTED;  // built for sm_103a only
  if (cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, *dev) != cudaSuccess)
    return ESCHA_ERR_CUDA;
  return ESCHA_OK;
}

// Read a small int32 array that may live on the host or on the device.
escha_status_t read_host_or_device(const int32_t* p, int n, int32_t* out, cudaStream_t st) {
  cudaPointerAttributes attr;
  cudaError_t e = cudaPointerGetAttributes(&attr, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    attr.type = cudaMemoryTypeUnregistered;
  }
  if (attr.type == cudaMemoryTypeDevice) {
    if (cudaMemcpyAsync(out, p, n * sizeof(int32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess)
      return ESCHA_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return ESCHA_ERR_CUDA;
  } else {
    std::memcpy(out, p, n * sizeof(int32_t));
  }
  return ESCHA_OK;
}

escha_status_t parse_config(const int32_t* cfg, int len, int* bits, int* in_f, int* out_f) {
  if (len == 6) {
    // [16, bits, cb, 1, in, out]
    if (cfg[0] != 16) return ESCHA_ERR_UNSUPPORTED;
    if (cfg[2] != 1 || cfg[3] != 1) return ESCHA_ERR_UNSUPPORTED;
    *bits = cfg[1];
    *in_f = cfg[4];
    *out_f = cfg[5];
  } else if (len == 9) {
    // [tile=16, K, bits, mcg_flag, num_experts, in, out, in_p, out_p]
    if (cfg[0] != 16 || cfg[3] != 1 || cfg[4] != 1) return ESCHA_ERR_UNSUPPORTED;
    *bits = cfg[2];
    if (cfg[1] != *bits && cfg[1] != 16 * *bits) return ESCHA_ERR_UNSUPPORTED;
    *in_f = cfg[5];
    *out_f = cfg[6];
    if (cfg[7] != *in_f || cfg[8] != *out_f) return ESCHA_ERR_UNSUPPORTED;
  } else {
    return ESCHA_ERR_INVALID_ARG;
  }
  if (*bits < 2 || *bits > 4) return ESCHA_ERR_UNSUPPORTED;
  if (*in_f <= 0 || *out_f <= 0) return ESCHA_ERR_INVALID_ARG;
  if (*in_f % 128 != 0 || *out_f % 128 != 0) return ESCHA_ERR_UNSUPPORTED;
  return ESCHA_OK;
}

escha_status_t upload_jobs(GemvSchedule& s) {
  escha_status_t st = dev_alloc(&s.d_jobs, s.jobs.size());
  if (st != ESCHA_OK) return st;
  if (cudaMemcpy(s.d_jobs, s.jobs.data(), s.jobs.size() * sizeof(GemvJob),
                 cudaMemcpyHostToDevice) != cudaSuccess)
    return ESCHA_ERR_CUDA;
  return ESCHA_OK;
}

// ESCHA_SYNC_DEBUG=1 in the environment (read once): every compute call
// synchronises its stream after launching and reports an asynchronous CUDA
// error at that call instead of a later one.
bool sync_debug() {
  static const bool on = [] {
    const char* v = std::getenv("ESCHA_SYNC_DEBUG");
    return v != nullptr && v[0] == '1';
  }();
  return on;
}

escha_status_t after_launch(escha_status_t s, cudaStream_t st) {
  if (s != ESCHA_OK || !sync_debug()) return s;
  if (cudaStreamSynchronize(st) != cudaSuccess) return ESCHA_ERR_CUDA;
  return from_cuda(cudaGetLastError());
}

escha_status_t read_and_clear_error(int* d_err, cudaStream_t st) {
  if (cudaStreamSynchronize(st) != cudaSuccess) return ESCHA_ERR_CUDA;
  if (cudaGetLastError() != cudaSuccess) return ESCHA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, d_err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return ESCHA_ERR_CUDA;
  if (v != 0 && cudaMemset(d_err, 0, sizeof(int)) != cudaSuccess) return ESCHA_ERR_CUDA;
  if (v == kDevErrTimeout) return ESCHA_ERR_TIMEOUT;
  if (v == kDevErrBadRoute || v == kDevErrBadTable) return ESCHA_ERR_INVALID_ARG;
  return v == 0 ? ESCHA_OK : ESCHA_ERR_CUDA;
}

}  // namespace escha

// ====================================================================== ABI

extern "C" {

const char* escha_status_string(escha_status_t s) {
  switch (s) {
    case ESCHA_OK: return "ok";
    case ESCHA_ERR_INVALID_ARG: return "invalid argument";
    case ESCHA_ERR_UNSUPPORTED: return "unsupported configuration";
    case ESCHA_ERR_CUDA: return "CUDA error";
    case ESCHA_ERR_OOM: return "out of device memory";
    case ESCHA_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

int escha_version(void) { return 100; }

const char* escha_last_error_string(void) { return g_last_error; }

escha_status_t escha_linear_create(escha_linear_t* out, const int16_t* code, const uint16_t* rin,
                                   const uint16_t* rout, const float* s_in, const float* s_out,
                                   const int32_t* config, int config_len, void* stream) {
  if (!out) return ESCHA_ERR_INVALID_ARG;
  *out = nullptr;
  if (!code || !rin || !rout || !config) return ESCHA_ERR_INVALID_ARG;
  if (!aligned16(code)) return ESCHA_ERR_INVALID_ARG;
  if (config_len != 6 && config_len != 9) return ESCHA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t cfg[9];
  escha_status_t s = read_host_or_device(config, config_len, cfg, st);
  if (s != ESCHA_OK) return s;
  int bits, in_f, out_f;
  s = parse_config(cfg, config_len, &bits, &in_f, &out_f);
  if (s != ESCHA_OK) return s;

  escha_linear_s* h = new (std::nothrow) escha_linear_s();
  if (!h) return ESCHA_ERR_OOM;
  s = linear_init(h, code, bits, in_f, out_f, rin, rout, s_in, s_out, st);
  if (s != ESCHA_OK) {
    linear_free(h);
    delete h;
    return s;
  }
  *out = h;
  return ESCHA_OK;
}

escha_status_t escha_linear_destroy(escha_linear_t h) {
  if (!h) return ESCHA_ERR_INVALID_ARG;
  cudaDeviceSynchronize();
  linear_free(h);
  delete h;
  return ESCHA_OK;
}

escha_status_t escha_linear_shape(escha_linear_t h, int* in_features, int* out_features,
                                  int* bits) {
  if (!h) return ESCHA_ERR_INVALID_ARG;
  if (in_features) *in_features = h->K;
  if (out_features) *out_features = h->N;
  if (bits) *bits = h->bits;
  return ESCHA_OK;
}

escha_status_t escha_linear_decode(escha_linear_t h, uint16_t* w_inner, void* stream) {
  if (!h || !w_inner) return ESCHA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(w_inner) & 1u) != 0) return ESCHA_ERR_INVALID_ARG;
  return from_cuda(launch_decode(h->code, h->bits, h->rounding == ESCHA_ROUND_E4M3, h->K, h->N,
                                 w_inner, static_cast<cudaStream_t>(stream)));
}

escha_status_t escha_linear_set_rounding(escha_linear_t h, int rounding) {
  if (!h) return ESCHA_ERR_INVALID_ARG;
  if (rounding != ESCHA_ROUND_FP16 && rounding != ESCHA_ROUND_E4M3) return ESCHA_ERR_INVALID_ARG;
  return linear_set_rounding(h, rounding);
}

escha_status_t escha_moe_set_rounding(escha_moe_t m, int rounding) {
  if (!m) return ESCHA_ERR_INVALID_ARG;
  if (rounding != ESCHA_ROUND_FP16 && rounding != ESCHA_ROUND_E4M3) return ESCHA_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return ESCHA_ERR_CUDA;  // no call in flight
  m->rounding = rounding;  // read by the routing plan of every call
  return ESCHA_OK;
}

static bool gemv_args_ok(const void* h, const void* x, const void* y, int M) {
  return h && x && y && M >= 1 && M <= kGemvMaxTokens && aligned16(x) && aligned16(y);
}

escha_status_t escha_linear_gemv(escha_linear_t h, const uint16_t* x, uint16_t* y, int M,
                                 void* stream) {
  if (!gemv_args_ok(h, x, y, M)) return ESCHA_ERR_INVALID_ARG;
  return after_launch(linear_gemv(h, x, y, M, static_cast<cudaStream_t>(stream)),
                      static_cast<cudaStream_t>(stream));
}

escha_status_t escha_linear_gemv_stage(escha_linear_t h, int stage, const uint16_t* x,
                                       uint16_t* y, int M, void* stream) {
  if (!gemv_args_ok(h, x, y, M)) return ESCHA_ERR_INVALID_ARG;
  return after_launch(linear_gemv_stage(h, stage, x, y, M, static_cast<cudaStream_t>(stream)),
                      static_cast<cudaStream_t>(stream));
}

escha_status_t escha_linear_check(escha_linear_t h, void* stream) {
  if (!h) return ESCHA_ERR_INVALID_ARG;
  return read_and_clear_error(h->err, static_cast<cudaStream_t>(stream));
}

escha_status_t escha_mlp_set_input_norm(escha_mlp_t m, const uint16_t* norm_w, float eps,
                                        int stored_minus_one) {
  if (!m) return ESCHA_ERR_INVALID_ARG;
  if (norm_w && !(eps >= 0.0f && eps < 1.0f)) return ESCHA_ERR_INVALID_ARG;
  if (norm_w && (reinterpret_cast<uintptr_t>(norm_w) & 1u)) return ESCHA_ERR_INVALID_ARG;
  return mlp_set_input_norm(m, norm_w, eps, stored_minus_one);
}

escha_status_t escha_mlp_check(escha_mlp_t m, void* stream) {
  if (!m) return ESCHA_ERR_INVALID_ARG;
  return read_and_clear_error(m->err, static_cast<cudaStream_t>(stream));
}

escha_status_t escha_mlp_create(escha_mlp_t* out, escha_linear_t gate, escha_linear_t up,
                                escha_linear_t down) {
  if (!out) return ESCHA_ERR_INVALID_ARG;
  *out = nullptr;
  if (!gate || !up || !down) return ESCHA_ERR_INVALID_ARG;
  if (gate->K != up->K || gate->N != up->N || down->K != gate->N || down->N != gate->K)
    return ESCHA_ERR_INVALID_ARG;
  escha_mlp_s* m = new (std::nothrow) escha_mlp_s();
  if (!m) return ESCHA_ERR_OOM;
  escha_status_t s = mlp_init(m, gate, up, down);
  if (s != ESCHA_OK) {
    mlp_free(m);
    delete m;
    return s;
  }
  *out = m;
  return ESCHA_OK;
}

escha_status_t escha_mlp_destroy(escha_mlp_t m) {
  if (!m) return ESCHA_ERR_INVALID_ARG;
  cudaDeviceSynchronize();
  mlp_free(m);
  delete m;
  return ESCHA_OK;
}

escha_status_t escha_mlp_gemv(escha_mlp_t m, const uint16_t* x, uint16_t* y, int M,
                              void* stream) {
  if (!gemv_args_ok(m, x, y, M)) return ESCHA_ERR_INVALID_ARG;
  return after_launch(mlp_gemv(m, x, y, M, static_cast<cudaStream_t>(stream)),
                      static_cast<cudaStream_t>(stream));
}

escha_status_t escha_mlp_gemv_stage(escha_mlp_t m, int stage, const uint16_t* x, uint16_t* y,
                                    int M, void* stream) {
  if (!gemv_args_ok(m, x, y, M)) return ESCHA_ERR_INVALID_ARG;
  return after_launch(mlp_gemv_stage(m, stage, x, y, M, static_cast<cudaStream_t>(stream)),
                      static_cast<cudaStream_t>(stream));
}

escha_status_t escha_profile_enable(void* handle, int kind, int on) {
  Profiler* p = profiler_of(handle, kind);
  if (!p) return ESCHA_ERR_INVALID_ARG;
  p->on = (on != 0);
  return ESCHA_OK;
}

escha_status_t escha_profile_collect(void* handle, int kind, double* ms_total, int* launches) {
  Profiler* p = profiler_of(handle, kind);
  if (!p) return ESCHA_ERR_INVALID_ARG;
  return p->collect(ms_total, launches);
}

escha_status_t escha_trellis_encode(const float* w, int in_features, int out_features, int bits,
                                    int rounding, int16_t* code, float* sq_err, void* stream) {
  if (!w || !code) return ESCHA_ERR_INVALID_ARG;
  if (in_features <= 0 || out_features <= 0) return ESCHA_ERR_INVALID_ARG;
  if (in_features % 16 != 0 || out_features % 16 != 0) return ESCHA_ERR_UNSUPPORTED;
  if (bits < 2 || bits > 4) return ESCHA_ERR_UNSUPPORTED;
  if (rounding != ESCHA_ROUND_FP16 && rounding != ESCHA_ROUND_E4M3) return ESCHA_ERR_INVALID_ARG;
  int dev, sms;
  escha_status_t s = device_info(&dev, &sms);
  if (s != ESCHA_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const long long tiles = (long long)(in_features / 16) * (out_features / 16);
  const int ctas = static_cast<int>(tiles < sms ? tiles : sms);
  void* scratch = nullptr;
  cudaError_t e = cudaMallocAsync(&scratch, encode_scratch_bytes(bits, ctas), st);
  if (e != cudaSuccess) return from_cuda(e);
  e = launch_trellis_encode(w, in_features, out_features, bits, rounding == ESCHA_ROUND_E4M3,
                            code, sq_err, static_cast<uint8_t*>(scratch), ctas, st);
  const cudaError_t ef = cudaFreeAsync(scratch, st);
  if (e != cudaSuccess) return from_cuda(e);
  return from_cuda(ef);
}

escha_status_t escha_selftest_wait_timeout(int limit_us, void* stream) {
  if (limit_us < 1 || limit_us > 1000000) return ESCHA_ERR_INVALID_ARG;
  int dev, sms;
  escha_status_t s = device_info(&dev, &sms);
  if (s != ESCHA_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* err = nullptr;
  s = dev_alloc(&err, 1);
  if (s != ESCHA_OK) return s;
  if (cudaMemset(err, 0, sizeof(int)) != cudaSuccess) {
    cudaFree(err);
    return ESCHA_ERR_CUDA;
  }
  cudaError_t e = launch_wait_selftest(err, static_cast<uint64_t>(limit_us) * 1000ull, st);
  if (e != cudaSuccess) {
    cudaFree(err);
    return from_cuda(e);
  }
  s = read_and_clear_error(err, st);
  cudaFree(err);
  return s;
}

escha_status_t escha_linear_gemm(escha_linear_t h, const uint16_t* x, uint16_t* y, int M,
                                 void* stream) {
  if (!h || !x || !y) return ESCHA_ERR_INVALID_ARG;
  if (M < 1) return ESCHA_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y)) return ESCHA_ERR_INVALID_ARG;
  return after_launch(linear_gemm(h, x, y, M, static_cast<cudaStream_t>(stream)),
                      static_cast<cudaStream_t>(stream));
}

escha_status_t escha_linear_gemm_fp8(escha_linear_t h, const uint16_t* x, uint16_t* y, int M,
                                     void* stream) {
  if (!h || !x || !y) return ESCHA_ERR_INVALID_ARG;
  if (M < 1) return ESCHA_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y)) return ESCHA_ERR_INVALID_ARG;
  return after_launch(linear_gemm_fp8(h, x, y, M, static_cast<cudaStream_t>(stream)),
                      static_cast<cudaStream_t>(stream));
}

escha_status_t escha_linear_gemm_fp8_codes(escha_linear_t h, const uint8_t* q, const float* d,
                                           uint16_t* y, int M, void* stream) {
  if (!h || !q || !d || !y) return ESCHA_ERR_INVALID_ARG;
  if (M < 1) return ESCHA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(y) || (reinterpret_cast<uintptr_t>(d) & 3u))
    return ESCHA_ERR_INVALID_ARG;
  return after_launch(linear_gemm_fp8_codes(h, q, d, y, M, static_cast<cudaStream_t>(stream)),
                      static_cast<cudaStream_t>(stream));
}

escha_status_t escha_quantize_e4m3_rows(const uint16_t* xh, uint8_t* q, float* d, int M, int K,
                                        void* stream) {
  if (!xh || !q || !d || M < 1 || K < 128 || K % 128 != 0) return ESCHA_ERR_INVALID_ARG;
  if (escha::quantize_e4m3_smem_bytes(K) > escha::kMaxQuantSmem) return ESCHA_ERR_INVALID_ARG;
  if (!aligned16(xh) || !aligned16(q) || !aligned16(d)) return ESCHA_ERR_INVALID_ARG;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  return after_launch(escha::from_cuda(escha::launch_quantize_e4m3_rows(xh, nullptr, q, d, M, K, nullptr, 0, st)),
                      st);
}

escha_status_t escha_linear_reserve(escha_linear_t h, int max_m) {
  if (!h || max_m < 1) return ESCHA_ERR_INVALID_ARG;
  return linear_reserve(h, max_m);
}
escha_status_t escha_moe_create(escha_moe_t* out, int num_experts, int hidden, int inter,
                                const int16_t* const* gate_code, const int16_t* const* up_code,
                                const int16_t* const* down_code, const int32_t* bits,
                                const uint16_t* rin_hidden, const float* s_in_hidden,
                                const uint16_t* rout_gate, const float* s_out_gate,
                                const uint16_t* rout_up, const float* s_out_up,
                                const uint16_t* rin_down, const float* s_in_down,
                                const uint16_t* rout_hidden, const float* s_out_hidden,
                                void* stream) {
  if (!out) return ESCHA_ERR_INVALID_ARG;
  *out = nullptr;
  if (num_experts < 1 || hidden <= 0 || inter <= 0) return ESCHA_ERR_INVALID_ARG;
  if (num_experts > kMoeMaxExperts) return ESCHA_ERR_UNSUPPORTED;
  if (hidden % 128 != 0 || inter % 128 != 0) return ESCHA_ERR_UNSUPPORTED;
  if (!gate_code || !up_code || !down_code || !bits || !rin_hidden || !rout_gate || !rout_up ||
      !rin_down || !rout_hidden)
    return ESCHA_ERR_INVALID_ARG;
  for (int e = 0; e < num_experts; ++e) {
    if (!gate_code[e] || !up_code[e] || !down_code[e]) return ESCHA_ERR_INVALID_ARG;
    if (!aligned16(gate_code[e]) || !aligned16(up_code[e]) || !aligned16(down_code[e]))
      return ESCHA_ERR_INVALID_ARG;
    if (bits[e] < 2 || bits[e] > 4) return ESCHA_ERR_UNSUPPORTED;
  }
  escha_moe_s* h = new (std::nothrow) escha_moe_s();
  if (!h) return ESCHA_ERR_OOM;
  escha_status_t s = moe_init(h, num_experts, hidden, inter, gate_code, up_code, down_code, bits,
                              rin_hidden, s_in_hidden, rout_gate, s_out_gate, rout_up, s_out_up,
                              rin_down, s_in_down, rout_hidden, s_out_hidden,
                              static_cast<cudaStream_t>(stream));
  if (s != ESCHA_OK) {
    moe_free(h);
    delete h;
    return s;
  }
  *out = h;
  return ESCHA_OK;
}

escha_status_t escha_moe_create_halves(escha_moe_t* out, int num_experts, int hidden, int inter,
                                       const int16_t* const* gate_half,
                                       const int16_t* const* up_half,
                                       const int16_t* const* down_half, const int32_t* gate_bits,
                                       const int32_t* up_bits, const int32_t* down_bits,
                                       const uint16_t* rin_hidden, const float* s_in_hidden,
                                       const uint16_t* rout_gate, const float* s_out_gate,
                                       const uint16_t* rout_up, const float* s_out_up,
                                       const uint16_t* rin_down, const float* s_in_down,
                                       const uint16_t* rout_hidden, const float* s_out_hidden,
                                       void* stream) {
  if (!out) return ESCHA_ERR_INVALID_ARG;
  *out = nullptr;
  if (num_experts < 1 || hidden <= 0 || inter <= 0) return ESCHA_ERR_INVALID_ARG;
  if (num_experts > kMoeMaxExperts) return ESCHA_ERR_UNSUPPORTED;
  if (hidden % 128 != 0 || inter % 128 != 0) return ESCHA_ERR_UNSUPPORTED;
  if (!gate_half || !up_half || !down_half || !gate_bits || !up_bits || !down_bits ||
      !rin_hidden || !rout_gate || !rout_up || !rin_down || !rout_hidden)
    return ESCHA_ERR_INVALID_ARG;
  const uintptr_t pa = reinterpret_cast<uintptr_t>(gate_half) | reinterpret_cast<uintptr_t>(up_half) |
                       reinterpret_cast<uintptr_t>(down_half);
  const uintptr_t ba = reinterpret_cast<uintptr_t>(gate_bits) | reinterpret_cast<uintptr_t>(up_bits) |
                       reinterpret_cast<uintptr_t>(down_bits);
  if ((pa & 7u) != 0 || (ba & 3u) != 0) return ESCHA_ERR_INVALID_ARG;
  escha_moe_s* h = new (std::nothrow) escha_moe_s();
  if (!h) return ESCHA_ERR_OOM;
  escha_status_t s = moe_init_halves(h, num_experts, hidden, inter, gate_half, up_half, down_half,
                                     gate_bits, up_bits, down_bits, rin_hidden, s_in_hidden,
                                     rout_gate, s_out_gate, rout_up, s_out_up, rin_down, s_in_down,
                                     rout_hidden, s_out_hidden, static_cast<cudaStream_t>(stream));
  if (s != ESCHA_OK) {
    moe_free(h);
    delete h;
    return s;
  }
  *out = h;
  return ESCHA_OK;
}

escha_status_t escha_moe_set_shared_expert(escha_moe_t m, const int16_t* gate_code,
                                           const int16_t* up_code, const int16_t* down_code,
                                           int bits, const uint16_t* rout_gate,
                                           const float* s_out_gate, const uint16_t* rout_up,
                                           const float* s_out_up, const uint16_t* rin_down,
                                           const float* s_in_down) {
  if (!m) return ESCHA_ERR_INVALID_ARG;
  if (m->halves) return ESCHA_ERR_UNSUPPORTED;
  if (gate_code) {
    if (!up_code || !down_code || !rout_gate || !rout_up || !rin_down)
      return ESCHA_ERR_INVALID_ARG;
    if (!aligned16(gate_code) || !aligned16(up_code) || !aligned16(down_code))
      return ESCHA_ERR_INVALID_ARG;
    if (bits < 2 || bits > 4) return ESCHA_ERR_UNSUPPORTED;
  }
  return moe_set_shared_expert(m, gate_code, up_code, down_code, bits, rout_gate, s_out_gate,
                               rout_up, s_out_up, rin_down, s_in_down);
}

escha_status_t escha_moe_destroy(escha_moe_t m) {
  if (!m) return ESCHA_ERR_INVALID_ARG;
  cudaDeviceSynchronize();
  moe_free(m);
  delete m;
  return ESCHA_OK;
}

static bool moe_args_ok(const void* m, const void* x, const void* ids, const void* w,
                        const void* y, int M, int topk) {
  return m && x && ids && w && y && M >= 1 && M <= kMoeMaxTokens && topk >= 1 &&
         topk <= kMoeMaxTopk && aligned16(x) && aligned16(y);
}

escha_status_t escha_linear_moe_gemv(escha_moe_t m, const uint16_t* x, const int32_t* expert_ids,
                                     const float* expert_w, uint16_t* y, int M, int topk,
                                     void* stream) {
  if (!moe_args_ok(m, x, expert_ids, expert_w, y, M, topk)) return ESCHA_ERR_INVALID_ARG;
  return after_launch(
      moe_gemv(m, x, expert_ids, expert_w, y, M, topk, static_cast<cudaStream_t>(stream)),
      static_cast<cudaStream_t>(stream));
}

escha_status_t escha_linear_moe_gemv_stage(escha_moe_t m, int stage, const uint16_t* x,
                                           const int32_t* expert_ids, const float* expert_w,
                                           uint16_t* y, int M, int topk, void* stream) {
  if (!moe_args_ok(m, x, expert_ids, expert_w, y, M, topk)) return ESCHA_ERR_INVALID_ARG;
  return moe_gemv_stage(m, stage, x, expert_ids, expert_w, y, M, topk,
                        static_cast<cudaStream_t>(stream));
}

escha_status_t escha_moe_check(escha_moe_t m, void* stream) {
  if (!m) return ESCHA_ERR_INVALID_ARG;
  return read_and_clear_error(m->err, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
