// Handle structures behind the opaque C ABI types, and the host routines the
// ABI entry points call.
#pragma once

#include <cuda_runtime.h>

#include <utility>
#include <vector>

#include "escha.h"
#include "internal.h"

namespace escha {

struct Profiler {
  bool on = false;
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> pending;
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> pool;
  void begin(cudaStream_t st);
  void end(cudaStream_t st);
  escha_status_t collect(double* ms_total, int* launches);
  ~Profiler();
};

escha_status_t from_cuda(cudaError_t e);
bool aligned16(const void* p);
escha_status_t device_info(int* dev, int* sms);
escha_status_t upload_jobs(GemvSchedule& s);
escha_status_t read_and_clear_error(int* d_err, cudaStream_t st);
template <typename T>
escha_status_t dev_alloc(T** p, size_t count);

}  // namespace escha

struct escha_linear_s {
  int device = 0;
  int num_sms = 0;
  int K = 0, N = 0, bits = 0;
  const int16_t* code = nullptr;
  float* su = nullptr;        // rin * s_in, fp32 [K]
  float* sv = nullptr;        // rout * s_out, fp32 [N]
  uint32_t* xfrag = nullptr;  // rotated activations in fragment order, [K/16][2][32][4]
  float* part = nullptr;      // GEMV partial sums, [max_slots][16][N]
  int* err = nullptr;         // device error word
  escha::GemvSchedule sched;  // one job: this matrix
  uint16_t* xh = nullptr;     // prefill workspace: rotated activations [xh_rows, K]
  int xh_rows = 0;
  escha::Profiler prof;
};

struct escha_mlp_s {
  escha_linear_t gate = nullptr, up = nullptr, down = nullptr;
  uint32_t* xfrag_gate = nullptr;
  uint32_t* xfrag_up = nullptr;
  uint32_t* xfrag_down = nullptr;
  float* part_gate = nullptr;
  float* part_up = nullptr;
  float* part_down = nullptr;
  int* err = nullptr;
  escha::GemvSchedule s_gate_up;  // jobs: gate, up
  escha::GemvSchedule s_down;     // job: down
  escha::Profiler prof;
};

namespace escha {

escha_status_t linear_init(escha_linear_s* h, const int16_t* code, int bits, int K, int N,
                           const uint16_t* rin, const uint16_t* rout, const float* s_in,
                           const float* s_out, cudaStream_t st);
void linear_free(escha_linear_s* h);
escha_status_t linear_gemv(escha_linear_s* h, const uint16_t* x, uint16_t* y, int M,
                           cudaStream_t st);
escha_status_t mlp_init(escha_mlp_s* m, escha_linear_s* gate, escha_linear_s* up,
                        escha_linear_s* down);
void mlp_free(escha_mlp_s* m);
escha_status_t mlp_gemv(escha_mlp_s* m, const uint16_t* x, uint16_t* y, int M, cudaStream_t st);
Profiler* profiler_of(void* handle, int kind);

}  // namespace escha
