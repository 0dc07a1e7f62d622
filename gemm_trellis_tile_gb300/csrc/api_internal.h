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
escha_status_t after_launch(escha_status_t s, cudaStream_t st);
bool sync_debug();
template <typename T>
escha_status_t dev_alloc(T** p, size_t count);

}  // namespace escha

struct escha_linear_s {
  int device = 0;
  int rounding = 0;           // ESCHA_ROUND_FP16 or ESCHA_ROUND_E4M3
  int num_sms = 0;
  int K = 0, N = 0, bits = 0;
  const int16_t* code = nullptr;
  float* su = nullptr;        // rin * s_in, fp32 [K]
  float* sv = nullptr;        // rout * s_out, fp32 [N]
  CUtensorMap* tmap = nullptr;  // device copy of the GEMV's tensor map of `code`
  uint32_t* xfrag = nullptr;    // rotated activations in fragment order, [K/16][16][4][4]
  float* part = nullptr;      // GEMV partial sums, [max_slots][16][N]
  int* err = nullptr;         // device error word
  escha::GemvSchedule sched;  // one job: this matrix
  uint16_t* xh = nullptr;     // prefill workspace: rotated activations [xh_rows, K]
                              // (FP8 prefill: their E4M3 codes, K bytes a row)
  float* xd = nullptr;        // FP8 prefill: per-row activation scales [xh_rows]
  int xh_rows = 0;
  float* gemm_ws = nullptr;   // prefill partial sums of tiles shared between CTAs
  int* gemm_cnt = nullptr;    // prefill arrival counters of shared tiles, cleared per call
  size_t gemm_cnt_ints = 0;
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
  // input RMSNorm (escha_mlp_set_input_norm): (w + offset) * su of gate and up
  int norm_on = 0;
  float norm_eps = 0.f;
  float* norm_g_gate = nullptr;
  float* norm_g_up = nullptr;
  int* err = nullptr;
  escha::GemvSchedule s_gate_up;  // jobs: gate, up
  escha::GemvSchedule s_down;     // job: down
  escha::Profiler prof;
};

struct escha_moe_s {
  int device = 0;
  int rounding = 0;           // ESCHA_ROUND_FP16 or ESCHA_ROUND_E4M3
  int num_sms = 0;
  int E = 0, hidden = 0, inter = 0;
  const uint8_t** gate_code = nullptr;  // device [E] tables of borrowed code pointers
  const uint8_t** up_code = nullptr;
  const uint8_t** down_code = nullptr;
  CUtensorMap* code_maps = nullptr;     // device [3][E]: gate, up, down tensor maps per expert
  int* bits = nullptr;                  // device [E]
  float* su_hidden = nullptr;           // shared input side of gate/up [hidden]
  float* sv_hidden = nullptr;           // shared output side of down [hidden]
  float* sv_gate = nullptr;             // per expert [E][inter]
  float* sv_up = nullptr;
  float* su_down = nullptr;
  uint32_t* xfrag_hidden = nullptr;     // rotated token(s), fragment order
  uint32_t* xfrag_down = nullptr;       // per distinct expert slot
  float* part1 = nullptr;               // gate/up partial sums per job
  float* part2 = nullptr;               // down partial sums per distinct expert
  escha::GemvJob* jobs1 = nullptr;      // written on the device each call
  escha::GemvJob* jobs2 = nullptr;
  // Stored by halves (escha_moe_create_halves): H = inter / 128 halves per
  // matrix; the caller's device tables are borrowed and re-read every call.
  int halves = 0;
  int H = 0;
  int shared_on = 0;  // a shared expert is set (entry E of the whole-matrix tables)
  const uint8_t* const* gate_half = nullptr;  // [E][H] code of each gate half
  const uint8_t* const* up_half = nullptr;    // [E][H]
  const uint8_t* const* down_half = nullptr;  // [E][H] (halves along down's input)
  const int* gate_bits = nullptr;             // [E][H]
  const int* up_bits = nullptr;               // [E][H]
  const int* down_bits = nullptr;             // [E]
  CUtensorMap* half_maps = nullptr;     // [E][H] down-half maps, rewritten when a half's entry changes
  unsigned long long* half_map_key = nullptr;  // [E][H] pointer | bits each map was written for (0: none)
  CUtensorMap* half_map_tmpl = nullptr; // [3] down-half map templates for 2/3/4 bits
  uint8_t* stand_in = nullptr;          // zero code replacing table entries that fail checks
  unsigned char* route = nullptr;       // device routing state
  int* err = nullptr;
  size_t xdown_stride = 0, part1_stride = 0, part2_stride = 0;
  int grid_max = 0;
  escha::Profiler prof;
};

namespace escha {

escha_status_t moe_init(escha_moe_s* h, int E, int hidden, int inter,
                        const int16_t* const* gate_code, const int16_t* const* up_code,
                        const int16_t* const* down_code, const int32_t* bits,
                        const uint16_t* rin_hidden, const float* s_in_hidden,
                        const uint16_t* rout_gate, const float* s_out_gate,
                        const uint16_t* rout_up, const float* s_out_up,
                        const uint16_t* rin_down, const float* s_in_down,
                        const uint16_t* rout_hidden, const float* s_out_hidden, cudaStream_t st);
escha_status_t moe_init_halves(escha_moe_s* h, int E, int hidden, int inter,
                               const int16_t* const* gate_half, const int16_t* const* up_half,
                               const int16_t* const* down_half, const int32_t* gate_bits,
                               const int32_t* up_bits, const int32_t* down_bits,
                               const uint16_t* rin_hidden, const float* s_in_hidden,
                               const uint16_t* rout_gate, const float* s_out_gate,
                               const uint16_t* rout_up, const float* s_out_up,
                               const uint16_t* rin_down, const float* s_in_down,
                               const uint16_t* rout_hidden, const float* s_out_hidden,
                               cudaStream_t st);
void moe_free(escha_moe_s* h);
escha_status_t moe_set_shared_expert(escha_moe_s* h, const int16_t* gate_code,
                                     const int16_t* up_code, const int16_t* down_code, int bits,
                                     const uint16_t* rout_gate, const float* s_out_gate,
                                     const uint16_t* rout_up, const float* s_out_up,
                                     const uint16_t* rin_down, const float* s_in_down);
escha_status_t moe_gemv_stage(escha_moe_s* h, int stage, const uint16_t* x, const int32_t* ids,
                              const float* w, uint16_t* y, int M, int topk, cudaStream_t st);
escha_status_t moe_gemv(escha_moe_s* h, const uint16_t* x, const int32_t* ids, const float* w,
                        uint16_t* y, int M, int topk, cudaStream_t st);

escha_status_t linear_init(escha_linear_s* h, const int16_t* code, int bits, int K, int N,
                           const uint16_t* rin, const uint16_t* rout, const float* s_in,
                           const float* s_out, cudaStream_t st);
void linear_free(escha_linear_s* h);
escha_status_t linear_set_rounding(escha_linear_s* h, int rounding);
escha_status_t linear_gemv_stage(escha_linear_s* h, int stage, const uint16_t* x, uint16_t* y,
                                 int M, cudaStream_t st);
escha_status_t linear_gemv(escha_linear_s* h, const uint16_t* x, uint16_t* y, int M,
                           cudaStream_t st);
escha_status_t linear_reserve(escha_linear_s* h, int rows);
escha_status_t linear_gemm_fp8(escha_linear_s* h, const uint16_t* x, uint16_t* y, int M,
                               cudaStream_t st);
escha_status_t linear_gemm_fp8_codes(escha_linear_s* h, const uint8_t* q, const float* d,
                                     uint16_t* y, int M, cudaStream_t st);
escha_status_t linear_gemm(escha_linear_s* h, const uint16_t* x, uint16_t* y, int M,
                           cudaStream_t st);
escha_status_t mlp_init(escha_mlp_s* m, escha_linear_s* gate, escha_linear_s* up,
                        escha_linear_s* down);
void mlp_free(escha_mlp_s* m);
escha_status_t mlp_set_input_norm(escha_mlp_s* m, const uint16_t* w, float eps,
                                  int stored_minus_one);
escha_status_t mlp_gemv_stage(escha_mlp_s* m, int stage, const uint16_t* x, uint16_t* y, int M,
                              cudaStream_t st);
escha_status_t mlp_gemv(escha_mlp_s* m, const uint16_t* x, uint16_t* y, int M, cudaStream_t st);
Profiler* profiler_of(void* handle, int kind);

}  // namespace escha
