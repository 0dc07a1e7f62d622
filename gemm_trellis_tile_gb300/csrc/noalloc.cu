// Allocation-free dense trellis layer at decode: escha_linear_gemv_noalloc.
//
// Some callers must not allocate device memory at all: runtimes that reserve
// every byte of device memory up front for their own pool, and code that runs
// where a cudaMalloc would synchronise the device or is forbidden.  For them
// this entry point computes the same layer as escha_linear_gemv (the same
// rotation, trellis GEMV and output kernels, the same launch configuration)
// without a handle, keeping all of its scratch -- folded scales, rotated
// activations in fragment order, fp32 partial sums, the job descriptor and the
// error word -- in one fixed file-scope device array.
//
// The array is ESCHA_NOALLOC_SCRATCH_BYTES (16 MiB) and is held on every GPU
// that loads the library until the process exits.  Its address is obtained
// once per device, on the first call made with that device current, with
// cudaGetSymbolAddress.  Every call reuses the array and leaves its contents
// behind; everything a call reads is rewritten by that call first.  Two calls
// whose work overlaps on the GPU (other streams, other host threads) race on
// the array.
//
// With no handle there is no error flag for the caller to read later, so a
// bounded wait of the GEMV that runs out marks the call's own output instead:
// a last small kernel sees the scratch error word set and fills y with fp16
// NaN.  With ESCHA_SYNC_DEBUG=1 the call also synchronises and returns
// ESCHA_ERR_TIMEOUT.

#include <cuda_runtime.h>

#include <mutex>

#include "api_internal.h"
#include "common.cuh"
#include "escha.h"
#include "internal.h"

using namespace escha;

namespace {

constexpr size_t kScratchBytes = ESCHA_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool ready = false;
  unsigned char* scratch = nullptr;  // device address of g_noalloc_scratch
  int num_sms = 0;
  int ranges_per_sm = 1;
  GemvSchedule sched;                // one job; its vector keeps capacity 1
};

DeviceState g_state[kMaxDevices];
std::mutex g_mutex;

// Writes the job table and the code tensor map into the scratch array (a
// kernel, not a copy from host memory, so the call stays capturable).
__global__ void put_job_kernel(GemvJob job, GemvJob* dst, const __grid_constant__ CUtensorMap map,
                               CUtensorMap* map_dst) {
  *dst = job;
  *map_dst = map;
  tensormap_release();
}

// Runs last: if a bounded wait of this call ran out (error word set), every
// element of y becomes fp16 NaN, so the failure reaches the caller's data.
__global__ void mark_failed_output_kernel(const int* err, uint16_t* y, size_t count) {
  if (*reinterpret_cast<const volatile int*>(err) == 0) return;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < count;
       i += (size_t)gridDim.x * blockDim.x)
    y[i] = 0x7E00u;
}

size_t round256(size_t b) { return (b + 255) & ~size_t(255); }

// First call on a device: look up the array's device address with that device
// current.  In host code the array's name only stands in for the symbol.
escha_status_t setup_device(int dev, DeviceState& s) {
  int d = 0, sms = 0;
  escha_status_t st = device_info(&d, &sms);
  if (st != ESCHA_OK) return st;
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess || p == nullptr) {
    cudaGetLastError();
    return ESCHA_ERR_CUDA;
  }
  s.scratch = static_cast<unsigned char*>(p);
  s.num_sms = sms;
  s.ranges_per_sm = gemv_ranges_per_sm();
  s.sched.jobs.reserve(1);
  s.ready = true;
  (void)dev;
  return ESCHA_OK;
}

}  // namespace

extern "C" escha_status_t escha_linear_gemv_noalloc(const int16_t* code, const uint16_t* rin,
                                                    const uint16_t* rout, const float* s_in,
                                                    const float* s_out, int in_features,
                                                    int out_features, int bits,
                                                    const uint16_t* x, uint16_t* y, int M,
                                                    void* stream) {
  if (!code || !rin || !rout || !x || !y) return ESCHA_ERR_INVALID_ARG;
  if (!aligned16(code) || !aligned16(x) || !aligned16(y)) return ESCHA_ERR_INVALID_ARG;
  if (M < 1 || M > kGemvMaxTokens) return ESCHA_ERR_INVALID_ARG;
  if (in_features <= 0 || out_features <= 0) return ESCHA_ERR_INVALID_ARG;
  if (bits < 2 || bits > 4) return ESCHA_ERR_UNSUPPORTED;
  if (in_features % 128 != 0 || out_features % 128 != 0) return ESCHA_ERR_UNSUPPORTED;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ESCHA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return ESCHA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& s = g_state[dev];
  if (!s.ready) {
    escha_status_t st = setup_device(dev, s);
    if (st != ESCHA_OK) return st;
  }

  const int K = in_features, N = out_features;
  GemvJob job;
  job.code = reinterpret_cast<const uint8_t*>(code);
  job.tmap = nullptr;
  job.xfrag = nullptr;
  job.e4m3 = 0;
  job.part = nullptr;
  job.unit_begin = 0;
  job.bits = bits;
  job.KT = K / 16;
  job.NG = N / 128;
  job.N = N;
  s.sched.jobs.assign(1, job);
  plan_gemv(s.sched, s.num_sms, s.ranges_per_sm);

  // Scratch layout, each piece on a 256-byte boundary.
  const size_t off_job = 0;
  const size_t off_err = 256;
  const size_t off_map = 512;
  const size_t off_su = 768;
  const size_t off_sv = off_su + round256((size_t)K * sizeof(float));
  const size_t off_xf = off_sv + round256((size_t)N * sizeof(float));
  const size_t off_part = off_xf + round256((size_t)(K / 16) * 2 * 32 * 4 * sizeof(uint32_t));
  const size_t end =
      off_part + (size_t)s.sched.max_slots * kGemvMaxTokens * (size_t)N * sizeof(float);
  if (end > kScratchBytes) return ESCHA_ERR_UNSUPPORTED;  // layer too large for the fixed scratch

  unsigned char* base = s.scratch;
  int* err = reinterpret_cast<int*>(base + off_err);
  float* su = reinterpret_cast<float*>(base + off_su);
  float* sv = reinterpret_cast<float*>(base + off_sv);
  uint32_t* xfrag = reinterpret_cast<uint32_t*>(base + off_xf);
  float* part = reinterpret_cast<float*>(base + off_part);
  CUtensorMap* d_map = reinterpret_cast<CUtensorMap*>(base + off_map);
  CUtensorMap map;
  if (!encode_gemv_code_map(&map, code, bits, K / 16, N / 16)) return ESCHA_ERR_CUDA;
  s.sched.jobs[0].tmap = d_map;
  s.sched.maps_from_device = true;
  s.sched.jobs[0].xfrag = reinterpret_cast<const uint4*>(xfrag);
  s.sched.jobs[0].part = part;
  s.sched.d_jobs = reinterpret_cast<GemvJob*>(base + off_job);

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(err, 0, sizeof(int), st);
  if (e != cudaSuccess) return from_cuda(e);
  put_job_kernel<<<1, 1, 0, st>>>(s.sched.jobs[0], s.sched.d_jobs, map, d_map);
  if ((e = cudaGetLastError()) != cudaSuccess) return from_cuda(e);
  if ((e = launch_fold_scales(rin, s_in, su, K, st)) != cudaSuccess) return from_cuda(e);
  if ((e = launch_fold_scales(rout, s_out, sv, N, st)) != cudaSuccess) return from_cuda(e);
  RotInJob rj{x, su, xfrag, K};
  if ((e = launch_rotate_in_xfrag(&rj, 1, M, st)) != cudaSuccess) return from_cuda(e);
  if ((e = launch_gemv(s.sched, M, err, st)) != cudaSuccess) return from_cuda(e);
  PartRef pr;
  pr.part = part;
  pr.unit_begin = s.sched.jobs[0].unit_begin;
  pr.KT = s.sched.jobs[0].KT;
  pr.N = N;
  e = launch_rotate_out(pr, s.sched.units, s.sched.grid, sv, y, M, kGemvMaxTokens, st);
  if (e != cudaSuccess) return from_cuda(e);
  mark_failed_output_kernel<<<1, 256, 0, st>>>(err, y, (size_t)M * N);
  if ((e = cudaGetLastError()) != cudaSuccess) return from_cuda(e);
  escha_status_t status = after_launch(ESCHA_OK, st);
  if (status == ESCHA_OK && sync_debug()) status = read_and_clear_error(err, st);
  return status;
}
