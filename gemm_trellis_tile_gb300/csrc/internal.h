// Host-side internals of libescha shared between translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

namespace escha {

// Device error codes written to a handle's error word.
constexpr int kDevErrTimeout = 1;
constexpr int kDevErrBadRoute = 2;
constexpr int kDevErrBadTable = 3;  // a code pointer or width in a caller's device table

// ---------------------------------------------------------------- GEMV schedule
//
// A launch of the trellis GEMV kernel contracts one or more matrices ("jobs").
// Job j's work is cut into units: unit (g, kt) = k-tile row kt of output group
// g (128 output channels = 8 tiles of 16).  Units are numbered job-major, then
// group-major, then k.  The launch's units are split into `grid` contiguous,
// near-equal ranges (range r owns [r*U/G, (r+1)*U/G)); persistent CTA b of C
// works ranges b, b + C and b + 2C, one per consumer warp group.  Where a range covers a
// group only partly, it writes its fp32 partial sums to slot (r - first range
// of that group); the output kernel sums the slots.
struct GemvJob {
  const uint8_t* code;       // tiles, [KT][NT][32*bits bytes]
  const CUtensorMap* tmap;   // `code` as a 2-D tensor (encode_gemv_code_map), in device memory
  const uint4* xfrag;        // rotated activations in fragment order, [KT][M][4] x uint4
  float* part;           // partial sums, [slots][mpad][N]
  long long unit_begin;  // first unit of this job within the launch
  int bits;
  int KT;                // in / 16
  int NG;                // out / 128
  int N;                 // out
  int e4m3;              // codebook values rounded to FP8 E4M3 (EXLR8 variant)
  // Matrices stored by halves along the input side (an expert's down matrix):
  // half h is loaded through row_maps[h] (tensor maps written on the device,
  // one 8-row box per copy); such launches count one unit per half (8 k-tile
  // rows) of one group, and KT counts halves.  Null otherwise.  (A matrix
  // stored by halves along the output side is one job per half, with `part`
  // pointing at the half's first output channel.)
  const CUtensorMap* row_maps = nullptr;
};

struct GemvSchedule {
  std::vector<GemvJob> jobs;
  GemvJob* d_jobs = nullptr;
  long long units = 0;
  int grid = 0;   // unit ranges
  int ctas = 0;   // CTAs launched (each works up to three ranges)
  int max_slots = 0;
  bool maps_from_device = false;  // the jobs' tensor maps are written by a kernel
};

constexpr int kGemvMaxTokens = 16;

// Routed-expert limits: tokens per call, experts per token, distinct experts
// per call (kMoeMaxTokens * kMoeMaxTopk), experts per layer.
constexpr int kMoeMaxTokens = 8;
constexpr int kMoeMaxTopk = 8;
constexpr int kMoeMaxDistinct = kMoeMaxTokens * kMoeMaxTopk;
constexpr int kMoeMaxExperts = 4096;
constexpr int kMinUnitsPerCta = 8;

// Make sure a kernel may take `bytes` of dynamic shared memory on the current
// device: the limit is raised when `bytes` exceeds every earlier request for
// that kernel and device, never lowered; thread-safe.
cudaError_t set_smem_limit(const void* func, int bytes);

int gemv_ranges_per_sm();
// Fill unit_begin, units, grid and max_slots for the given jobs.
void plan_gemv(GemvSchedule& s, int num_sms, int ranges_per_sm);
int gemv_slots_for_group(const GemvSchedule& s, int job, int g);

cudaError_t launch_gemv(const GemvSchedule& s, int M, int* err, cudaStream_t st);
// The 2-D tensor map through which the GEMV loads a stage's rows of code
// words: `code` [KT][NT][32*bits bytes] seen as uint32 rows of NT*8*bits
// words, one box = 8 tile columns x 16 k-tile rows.  Host only; false if the
// driver cannot encode it.
bool encode_gemv_code_map(CUtensorMap* map, const void* code, int bits, int KT, int NT);
// Map of one half of a matrix stored by input halves: `code` [8][NT][32*bits
// bytes] as uint32 rows of NT*8*bits words, one box = 8 tile columns x the
// half's 8 k-tile rows.  Host only.
bool encode_gemv_half_map(CUtensorMap* map, const void* code, int bits, int NT);

// Up to 8 tokens, with the job table, unit count and grid size written on the
// device (max_grid ranges are launched for; CTAs whose ranges start past the
// device grid exit).
// job_units > 0: every job of the launch has that many units (the kernel finds
// a range's first job by division instead of a scan).  maps_from_device: the
// jobs' tensor maps were written by a kernel.  layout: how every job of the
// launch is stored -- kGemvWhole (whole matrices, tensor maps in `tmap`),
// kGemvColHalves (each job one 128-channel column half: NG = 1, contiguous
// rows, no tensor map), kGemvRowHalves (input halves through row_maps; one
// unit = 8 k-tile rows).  e4m3: some job may be E4M3-rounded; false promises
// that none is and launches the kernel built with the fp16 decodes only.
constexpr int kGemvWhole = 0;
constexpr int kGemvColHalves = 1;
constexpr int kGemvRowHalves = 2;
cudaError_t launch_gemv_device_schedule(const GemvJob* d_jobs, const long long* d_units,
                                        const int* d_grid, int max_grid, int M, int mpad,
                                        int* err, cudaStream_t st, long long job_units = 0,
                                        bool maps_from_device = false, int layout = kGemvWhole,
                                        bool e4m3 = true);
// Prefill GEMM on tcgen05: y = fp16(had128(xh @ W_inner) * sv) for any M >= 1;
// xh is fp16 [M, K], 16-byte aligned; ws holds gemm_workspace_floats(num_sms)
// fp32 for tiles shared between CTAs; tile_cnt holds gemm_counter_ints(M, N)
// ints that are zero when the kernel starts (the caller clears them first).
size_t gemm_workspace_floats(int num_sms);
size_t gemm_counter_ints(int M, int N);
cudaError_t launch_trellis_gemm(const uint16_t* xh, const int16_t* code, int bits, bool e4m3,
                                int M, int K, int N, const float* sv, uint16_t* y, float* ws,
                                int* tile_cnt, int num_sms, int* err, cudaStream_t st);
// FP8 prefill: xq E4M3 codes [M, K] with per-row scales d (xh ~ xq * d); the
// weights are decoded with the E4M3 rounding and multiplied on kind::f8f6f4.
cudaError_t launch_trellis_gemm_fp8(const uint8_t* xq, const float* d, const int16_t* code,
                                    int bits, int M, int K, int N, const float* sv, uint16_t* y,
                                    float* ws, int* tile_cnt, int num_sms, int* err,
                                    cudaStream_t st);
// Per-token E4M3 quantisation: q [M, K], d [M] from xh = fp16(had128(x * su))
// (su != null) or from x itself (su == null).  K a multiple of 128; the block
// keeps the row in quantize_e4m3_smem_bytes(K) of shared memory.
size_t quantize_e4m3_smem_bytes(int K);
constexpr size_t kMaxQuantSmem = 128 * 1024;  // K <= 65536
// cnt/ncnt: the prefill GEMM's arrival counters, zeroed by the kernel (null/0: none).
cudaError_t launch_quantize_e4m3_rows(const uint16_t* x, const float* su, uint8_t* q, float* d,
                                      int M, int K, int* cnt, int ncnt, cudaStream_t st);
cudaError_t launch_decode(const int16_t* code, int bits, bool e4m3, int K, int N, uint16_t* w,
                          cudaStream_t st);
cudaError_t launch_wait_selftest(int* err, uint64_t limit_ns, cudaStream_t st);

// Viterbi trellis encoder: code [in/16][out/16][16*bits] (int16) of W_inner
// w [in, out] (fp32, row-major); sq_err [in/16 * out/16] (may be null) gets
// each tile's squared error.  scratch: encode_scratch_bytes(bits, ctas).
size_t encode_scratch_bytes(int bits, int ctas);
cudaError_t launch_trellis_encode(const float* w, int in_features, int out_features, int bits,
                                  bool e4m3, int16_t* code, float* sq_err, uint8_t* scratch,
                                  int ctas, cudaStream_t st);

// Launch configuration with programmatic stream serialisation: the kernel
// may start before its predecessor in the stream finishes and must call
// griddepcontrol.wait (pdl_wait) before it touches the predecessor's output.
struct PdlLaunch {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  PdlLaunch(unsigned blocks, unsigned threads, size_t smem, cudaStream_t st) {
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
};

// ---------------------------------------------------------------- rotations

struct RotInJob {
  const uint16_t* x;  // [M, K] fp16
  const float* su;    // [K]
  uint32_t* xfrag;    // [K/16][M][4][4]
  int K;
};

// Slot bookkeeping the output kernels need to sum a group's partial sums.
struct PartRef {
  const float* part;
  long long unit_begin;
  int KT;
  int N;
};

cudaError_t launch_fold_scales(const uint16_t* r, const float* s, float* out, int n,
                               cudaStream_t st);
cudaError_t launch_rotate_in_xfrag(const RotInJob* jobs, int njobs, int M, cudaStream_t st);
// Gated-MLP input rotations with the input RMSNorm: per token m,
// n = x / sqrt(mean(x^2) + eps); xfrag_gate = had128(n * g_gate), likewise up.
cudaError_t launch_rotate_in_norm(const uint16_t* x, const float* g_gate, const float* g_up,
                                  uint32_t* xfrag_gate, uint32_t* xfrag_up, int K, int M, float eps,
                                  cudaStream_t st);
cudaError_t launch_fold_norm(const uint16_t* w, float offset, const float* su, float* g, int n,
                             cudaStream_t st);
// cnt/ncnt: the prefill GEMM's arrival counters, zeroed by the kernel.
cudaError_t launch_rotate_in_plain(const uint16_t* x, const float* su, uint16_t* xh, int M,
                                   int K, int* cnt, int ncnt, cudaStream_t st);
cudaError_t launch_rotate_out(const PartRef& pr, long long units, int grid, const float* sv,
                              uint16_t* y, int M, int mpad, cudaStream_t st);
cudaError_t launch_mlp_mid(const PartRef& gate, const PartRef& up, long long units, int grid,
                           const float* sv_gate, const float* sv_up, const float* su_down,
                           uint32_t* xfrag_down, int M, cudaStream_t st);

}  // namespace escha
