// Activation-side transforms of a trellis layer: the input rotation
// xh = had128(x * su) and the output rotation y = had128(y_pre) * sv.
// "Escha-W2 runs on Metal" (activation-side reconstruction): the scales sit
// outside the Hadamard, so both transforms are cheap elementwise+butterfly
// passes on activations; the Hadamard never touches the weights.
//
// Every kernel here maps one warp to one 128-channel block of one token: lane
// l holds elements 4l..4l+3, two butterfly stages run in registers and five
// across lanes (fwht128_warp), all in fp32, rounded to fp16 once at the end.

#include "act_layout.cuh"
#include "common.cuh"
#include "internal.h"

namespace escha {

namespace {

constexpr int kWarpsPerBlock = 8;

// Sum a group's partial-sum slots for token m, channels 128g + 4l .. +3.
__device__ __forceinline__ void sum_part_slots(const PartRef& pr, long long U, int G, int mpad,
                                               int m, int g, int lane, float (&v)[4]) {
  sum_slots(pr.part, pr.unit_begin, pr.KT, pr.N, U, G, mpad, m, g, lane, v);
}

__global__ void fold_scales_kernel(const uint16_t* r, const float* s, float* out, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) out[i] = half_bits_to_float(r[i]) * (s ? s[i] : 1.0f);
}

struct RotInArgs {
  RotInJob jobs[2];
  int njobs;
  int M;
};

// xfrag = fp16(had128(x * su)) for tokens 0..M-1.
__global__ void rotate_in_xfrag_kernel(const RotInArgs a) {
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  long long wid = (long long)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const int mp = a.M;
  int j = 0;
  for (; j < a.njobs; ++j) {
    const long long n = (long long)mp * (a.jobs[j].K / kHad);
    if (wid < n) break;
    wid -= n;
  }
  if (j >= a.njobs) return;
  const RotInJob J = j == 0 ? a.jobs[0] : a.jobs[1];
  const int nb = J.K / kHad;
  const int m = static_cast<int>(wid / nb);
  const int kb = static_cast<int>(wid - (long long)m * nb);
  rotate_in_block(J.x, J.su, J.xfrag, J.K, a.M, m, kb, lane);
}

// Input RMSNorm fused into the gate/up input rotations of a gated MLP: one
// block per token; n = x / sqrt(mean(x^2) + eps), then
// xfrag_gate = fp16(had128(n * g_gate)), xfrag_up = fp16(had128(n * g_up)),
// where g = (stored norm weight + offset) * su was folded when the norm was set.
constexpr int kNormThreads = 1024;
constexpr int kNormCached = 2;  // 128-blocks per warp kept in registers between the passes
__global__ void __launch_bounds__(kNormThreads)
    rotate_in_norm_kernel(const uint16_t* x, const float* g_gate, const float* g_up,
                          uint32_t* xfrag_gate, uint32_t* xfrag_up, int K, int M, float eps) {
  __shared__ float part[kNormThreads / 32];
  constexpr int W = kNormThreads / 32;
  pdl_trigger();  // the GEMV may start streaming code; it waits for this kernel's output
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int m = blockIdx.x;
  const int nb = K / kHad;
  const uint16_t* xr = x + (size_t)m * K;
  float cache[kNormCached][4];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < kNormCached; ++i) {
    const int b = warp + i * W;
    if (b < nb) {
      load4_half(xr + b * kHad + 4 * lane, cache[i]);
#pragma unroll
      for (int q = 0; q < 4; ++q) ss += cache[i][q] * cache[i][q];
    }
  }
  for (int b = warp + kNormCached * W; b < nb; b += W) {
    float v[4];
    load4_half(xr + b * kHad + 4 * lane, v);
    ss += v[0] * v[0] + v[1] * v[1] + v[2] * v[2] + v[3] * v[3];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
  if (lane == 0) part[warp] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < W; ++w) tot += part[w];
  const float r = rsqrtf(tot / static_cast<float>(K) + eps);
  for (int i = 0, b = warp; b < nb; ++i, b += W) {
    const int k0 = b * kHad + 4 * lane;
    float v[4];
    if (i < kNormCached) {
#pragma unroll
      for (int q = 0; q < 4; ++q) v[q] = i == 0 ? cache[0][q] : cache[1][q];
    } else {
      load4_half(xr + k0, v);
    }
    const float4 sg = *reinterpret_cast<const float4*>(g_gate + k0);
    const float4 su = *reinterpret_cast<const float4*>(g_up + k0);
    float a[4] = {v[0] * r * sg.x, v[1] * r * sg.y, v[2] * r * sg.z, v[3] * r * sg.w};
    float c[4] = {v[0] * r * su.x, v[1] * r * su.y, v[2] * r * su.z, v[3] * r * su.w};
    fwht128_warp(a, lane);
    fwht128_warp(c, lane);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      xfrag_store(xfrag_gate, M, m, k0 + q, float_to_half_bits(a[q] * kHadScale));
      xfrag_store(xfrag_up, M, m, k0 + q, float_to_half_bits(c[q] * kHadScale));
    }
  }
}

// g[k] = (w[k] + offset) * su[k]: a stored norm weight folded into an input scale.
__global__ void fold_norm_kernel(const uint16_t* w, float offset, const float* su, float* g,
                                 int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) g[i] = (half_bits_to_float(w[i]) + offset) * su[i];
}

// Loads (16 bytes per lane: a pair of 128-blocks per warp) the E4M3 quantiser
// keeps in flight per warp before it transforms any.
constexpr int kRotBatch = 4;

// Zero the prefill GEMM's shared-tile arrival counters.  The kernels that
// produce the GEMM's activations do it: the GEMM reads the counters only after
// waiting for its predecessor (griddepcontrol.wait), and these kernels are
// launched in plain stream order after the previous GEMM, so no separate clear
// is needed between calls.
__device__ __forceinline__ void clear_counters(int* cnt, int n) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
    cnt[i] = 0;
}

constexpr int kPlainPairs = 4;  // pairs of 128-blocks per warp in rotate_in_plain

// xh = fp16(had128(x * su)), row-major [M, K] (the prefill GEMM's A operand).
// One warp per token and 2 * kPlainPairs consecutive 128-blocks: each lane
// loads 16 bytes of each pair (half-warp h holds block 2i + h), all loads in
// flight before the transforms; 16-byte stores.
__global__ void rotate_in_plain_kernel(const uint16_t* x, const float* su, uint16_t* xh, int M,
                                       int K, int* cnt, int ncnt) {
  pdl_trigger();  // the GEMM may set up; it waits for this kernel before loading xh
  clear_counters(cnt, ncnt);
  const int lane = threadIdx.x & 31;
  const long long wid = (long long)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const int nb = K / kHad;
  constexpr int kPer = 2 * kPlainPairs;
  const int ng = (nb + kPer - 1) / kPer;
  if (wid >= (long long)M * ng) return;
  const int m = static_cast<int>(wid / ng);
  const int b0 = static_cast<int>(wid - (long long)m * ng) * kPer + (lane >> 4);
  const int e = 8 * (lane & 15);
  const uint16_t* xr = x + (size_t)m * K;
  uint4 raw[kPlainPairs];
#pragma unroll
  for (int i = 0; i < kPlainPairs; ++i) {
    const int b = b0 + 2 * i;
    raw[i] = b < nb ? *reinterpret_cast<const uint4*>(xr + b * kHad + e) : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int i = 0; i < kPlainPairs; ++i) {
    const int b = b0 + 2 * i;
    const bool valid = b < nb;
    const int k0 = b * kHad + e;
    float v[8];
    const uint32_t w[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[2 * j] = half_bits_to_float(w[j] & 0xFFFF);
      v[2 * j + 1] = half_bits_to_float(w[j] >> 16);
    }
    if (valid) {
      const float4 s0 = *reinterpret_cast<const float4*>(su + k0);
      const float4 s1 = *reinterpret_cast<const float4*>(su + k0 + 4);
      v[0] *= s0.x;
      v[1] *= s0.y;
      v[2] *= s0.z;
      v[3] *= s0.w;
      v[4] *= s1.x;
      v[5] *= s1.y;
      v[6] *= s1.z;
      v[7] *= s1.w;
    }
    fwht128_halfwarp(v, lane);  // every lane, valid or not
    if (valid) {
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        o[j] = float_to_half_bits(v[2 * j] * kHadScale) |
               (uint32_t(float_to_half_bits(v[2 * j + 1] * kHadScale)) << 16);
      *reinterpret_cast<uint4*>(xh + (size_t)m * K + k0) = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

// Per-token E4M3 activations for the FP8 prefill (EXLR8 format page: weights
// that are exact E4M3 values let prefill multiply on FP8 tensor cores; the
// page leaves the activation side open, and this kernel scales each token by
// its largest magnitude).  One block per token:
//   xh   = fp16(had128(x * su))           (ROTATE; else x is xh already)
//   amax = max |xh|,  inv = 448 / amax,  d = amax / 448   (IEEE-rounded fp32)
//   q    = E4M3(xh * inv), nearest even, saturating  (the product rounded to fp32 first)
// A row of zeros gives q = 0 and d = 0.  The row's xh waits in shared memory
// (2K bytes) between the two passes.
// Threads per block: eight warps for long rows, four for short ones (each
// measured faster in its range).
constexpr int kQuantThreadsLong = 256;
constexpr int kQuantThreadsShort = 128;
constexpr int kQuantLongK = 8192;
constexpr int kQuantWarpsMax = kQuantThreadsLong / 32;
constexpr float kE4M3Max = 448.0f;

// Two fp32 values to two E4M3 bytes: `lo` in the low byte.
__device__ __forceinline__ uint32_t e4m3x2_from_f32(float lo, float hi) {
  uint16_t e;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(e) : "f"(hi), "f"(lo));
  return e;
}

// One block of THREADS per token (as many blocks per SM as threads and the
// row's 2K bytes of shared memory allow).  Warp w of W takes the pairs of
// 128-blocks w, w + W, ...: each lane loads 16 bytes of a pair (half-warp h
// holds block 2p + h) and their scales, up to kRotBatch pairs in flight, then
// the half-warp transforms.
template <bool ROTATE, int THREADS>
__global__ void __launch_bounds__(THREADS)
    quantize_e4m3_rows_kernel(const uint16_t* x, const float* su, uint8_t* q, float* d, int K,
                              int* cnt, int ncnt) {
  extern __shared__ __align__(16) uint16_t xrow[];
  constexpr int kQuantWarps = THREADS / 32;
  __shared__ float part[kQuantWarpsMax];
  pdl_trigger();  // the GEMM may set up; it waits for this kernel before loading q or d
  clear_counters(cnt, ncnt);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int m = blockIdx.x;
  const uint16_t* xr = x + (size_t)m * K;
  const int nb = K / kHad;
  const int np = (nb + 1) / 2;  // pairs of blocks (the last may hold one)
  const int e = 8 * (lane & 15);
  float amax = 0.f;
  for (int p0 = warp; p0 < np; p0 += kQuantWarps * kRotBatch) {
    // the batch's activations and scales all in flight before the first transform
    uint4 batch[kRotBatch];
    float4 sc[kRotBatch][2];
#pragma unroll
    for (int i = 0; i < kRotBatch; ++i) {
      const int b = 2 * (p0 + kQuantWarps * i) + (lane >> 4);
      const bool in = b < nb && p0 + kQuantWarps * i < np;
      batch[i] = in ? *reinterpret_cast<const uint4*>(xr + b * kHad + e) : make_uint4(0, 0, 0, 0);
      if (ROTATE) {
        sc[i][0] = in ? *reinterpret_cast<const float4*>(su + b * kHad + e) : make_float4(0.f, 0.f, 0.f, 0.f);
        sc[i][1] = in ? *reinterpret_cast<const float4*>(su + b * kHad + e + 4)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int i = 0; i < kRotBatch; ++i) {
      const int p = p0 + kQuantWarps * i;
      if (p >= np) break;  // uniform across the warp
      const int b = 2 * p + (lane >> 4);
      const bool valid = b < nb;
      const int k0 = b * kHad + e;
      uint4 raw = batch[i];
      if (ROTATE) {
        float v[8];
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          v[2 * j] = half_bits_to_float(w[j] & 0xFFFF);
          v[2 * j + 1] = half_bits_to_float(w[j] >> 16);
        }
        if (valid) {
          const float4 s0 = sc[i][0];
          const float4 s1 = sc[i][1];
          v[0] *= s0.x;
          v[1] *= s0.y;
          v[2] *= s0.z;
          v[3] *= s0.w;
          v[4] *= s1.x;
          v[5] *= s1.y;
          v[6] *= s1.z;
          v[7] *= s1.w;
        }
        fwht128_halfwarp(v, lane);  // every lane of the warp
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          o[j] = float_to_half_bits(v[2 * j] * kHadScale) |
                 (uint32_t(float_to_half_bits(v[2 * j + 1] * kHadScale)) << 16);
        raw = make_uint4(o[0], o[1], o[2], o[3]);
      }
      if (valid) {
        *reinterpret_cast<uint4*>(xrow + k0) = raw;
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          amax = fmaxf(amax, fabsf(half_bits_to_float(w[j] & 0xFFFF)));
          amax = fmaxf(amax, fabsf(half_bits_to_float(w[j] >> 16)));
        }
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
  if (lane == 0) part[warp] = amax;
  __syncthreads();
  amax = 0.f;
#pragma unroll
  for (int w = 0; w < kQuantWarps; ++w) amax = fmaxf(amax, part[w]);
  const float inv = amax > 0.f ? __fdiv_rn(kE4M3Max, amax) : 0.f;
  if (threadIdx.x == 0) d[m] = amax > 0.f ? __fdiv_rn(amax, kE4M3Max) : 0.f;
  uint8_t* qr = q + (size_t)m * K;
  for (int k = 16 * threadIdx.x; k < K; k += 16 * THREADS) {
    const uint4 a = *reinterpret_cast<const uint4*>(xrow + k);
    const uint4 b = *reinterpret_cast<const uint4*>(xrow + k + 8);
    const uint32_t h[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t out[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t w0 = h[2 * i], w1 = h[2 * i + 1];
      const uint32_t lo = e4m3x2_from_f32(__fmul_rn(half_bits_to_float(w0 & 0xFFFF), inv),
                                          __fmul_rn(half_bits_to_float(w0 >> 16), inv));
      const uint32_t hi = e4m3x2_from_f32(__fmul_rn(half_bits_to_float(w1 & 0xFFFF), inv),
                                          __fmul_rn(half_bits_to_float(w1 >> 16), inv));
      out[i] = lo | (hi << 16);
    }
    *reinterpret_cast<uint4*>(qr + k) = make_uint4(out[0], out[1], out[2], out[3]);
  }
}

// y = fp16(had128(sum of partial slots) * sv).
__global__ void rotate_out_kernel(const PartRef pr, long long U, int G, const float* sv,
                                  uint16_t* y, int M, int mpad) {
  const int lane = threadIdx.x & 31;
  const long long wid = (long long)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const int NG = pr.N / kHad;
  const int m = static_cast<int>(wid / NG);
  const int g = static_cast<int>(wid - (long long)m * NG);
  const int n0 = g * kHad + 4 * lane;
  const bool active = wid < (long long)M * NG;
  // The scales were written at creation: load them while the GEMV finishes.
  const float4 s = active ? *reinterpret_cast<const float4*>(sv + n0) : make_float4(0.f, 0.f, 0.f, 0.f);
  pdl_wait();
  if (!active) return;
  float v[4];
  sum_part_slots(pr, U, G, mpad, m, g, lane, v);
  fwht128_warp(v, lane);
  v[0] *= kHadScale * s.x;
  v[1] *= kHadScale * s.y;
  v[2] *= kHadScale * s.z;
  v[3] *= kHadScale * s.w;
  store4_half(y + (size_t)m * pr.N + n0, v);
}

// Gated-MLP middle: g = had(gate_pre)*sv_g, u = had(up_pre)*sv_u, h = silu(g)*u,
// then the down layer's input rotation had(h * su_down) into its fragments.
__global__ void mlp_mid_kernel(const PartRef gate, const PartRef up, long long U, int G,
                               const float* sv_gate, const float* sv_up, const float* su_down,
                               uint32_t* xfrag_down, int M) {
  const int lane = threadIdx.x & 31;
  const long long wid = (long long)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const int NG = gate.N / kHad;
  const int m = static_cast<int>(wid / NG);
  const int g = static_cast<int>(wid - (long long)m * NG);
  const int n0 = g * kHad + 4 * lane;
  const bool active = wid < (long long)M * NG;
  // The scales were written at creation: load them while the GEMV finishes.
  float4 sg = make_float4(0.f, 0.f, 0.f, 0.f), su = sg, sd = sg;
  if (active) {
    sg = *reinterpret_cast<const float4*>(sv_gate + n0);
    su = *reinterpret_cast<const float4*>(sv_up + n0);
    sd = *reinterpret_cast<const float4*>(su_down + n0);
  }
  pdl_wait();
  pdl_trigger();
  if (!active) return;
  float h[4];
  {
    float gv[4], uv[4];
    sum_slots_pair(gate.part, gate.unit_begin, up.part, up.unit_begin, gate.KT, gate.N, U, G,
                   kGemvMaxTokens, m, g, lane, gv, uv);
    fwht128_warp(gv, lane);
    fwht128_warp(uv, lane);
    const float sgv[4] = {sg.x, sg.y, sg.z, sg.w};
    const float suv[4] = {su.x, su.y, su.z, su.w};
    const float sdv[4] = {sd.x, sd.y, sd.z, sd.w};
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const float gg = gv[r] * kHadScale * sgv[r];
      const float uu = uv[r] * kHadScale * suv[r];
      h[r] = silu(gg) * uu * sdv[r];
    }
    fwht128_warp(h, lane);
  }
#pragma unroll
  for (int r = 0; r < 4; ++r)
    xfrag_store(xfrag_down, M, m, n0 + r, float_to_half_bits(h[r] * kHadScale));
}

unsigned blocks_for(long long warps) {
  return static_cast<unsigned>((warps + kWarpsPerBlock - 1) / kWarpsPerBlock);
}

}  // namespace

cudaError_t launch_fold_scales(const uint16_t* r, const float* s, float* out, int n,
                               cudaStream_t st) {
  fold_scales_kernel<<<(n + 255) / 256, 256, 0, st>>>(r, s, out, n);
  return cudaGetLastError();
}

cudaError_t launch_rotate_in_xfrag(const RotInJob* jobs, int njobs, int M, cudaStream_t st) {
  RotInArgs a;
  long long warps = 0;
  for (int j = 0; j < njobs; ++j) {
    a.jobs[j] = jobs[j];
    warps += (long long)M * (jobs[j].K / kHad);
  }
  a.njobs = njobs;
  a.M = M;
  rotate_in_xfrag_kernel<<<blocks_for(warps), 32 * kWarpsPerBlock, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_rotate_in_norm(const uint16_t* x, const float* g_gate, const float* g_up,
                                  uint32_t* xfrag_gate, uint32_t* xfrag_up, int K, int M, float eps,
                                  cudaStream_t st) {
  rotate_in_norm_kernel<<<M, kNormThreads, 0, st>>>(x, g_gate, g_up, xfrag_gate, xfrag_up, K, M,
                                                    eps);
  return cudaGetLastError();
}

cudaError_t launch_fold_norm(const uint16_t* w, float offset, const float* su, float* g, int n,
                             cudaStream_t st) {
  fold_norm_kernel<<<(n + 255) / 256, 256, 0, st>>>(w, offset, su, g, n);
  return cudaGetLastError();
}

cudaError_t launch_rotate_in_plain(const uint16_t* x, const float* su, uint16_t* xh, int M,
                                   int K, int* cnt, int ncnt, cudaStream_t st) {
  const long long warps = (long long)M * ((K / kHad + 2 * kPlainPairs - 1) / (2 * kPlainPairs));
  rotate_in_plain_kernel<<<blocks_for(warps), 32 * kWarpsPerBlock, 0, st>>>(x, su, xh, M, K, cnt,
                                                                           ncnt);
  return cudaGetLastError();
}

size_t quantize_e4m3_smem_bytes(int K) { return (size_t)K * 2; }

cudaError_t launch_quantize_e4m3_rows(const uint16_t* x, const float* su, uint8_t* q, float* d,
                                      int M, int K, int* cnt, int ncnt, cudaStream_t st) {
  const size_t smem = quantize_e4m3_smem_bytes(K);
  const bool lng = K >= kQuantLongK;
  const void* fn =
      su ? (lng ? reinterpret_cast<const void*>(quantize_e4m3_rows_kernel<true, kQuantThreadsLong>)
                : reinterpret_cast<const void*>(quantize_e4m3_rows_kernel<true, kQuantThreadsShort>))
         : (lng ? reinterpret_cast<const void*>(quantize_e4m3_rows_kernel<false, kQuantThreadsLong>)
                : reinterpret_cast<const void*>(quantize_e4m3_rows_kernel<false, kQuantThreadsShort>));
  cudaError_t e = set_smem_limit(fn, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int threads = lng ? kQuantThreadsLong : kQuantThreadsShort;
  void* args[] = {const_cast<uint16_t**>(&x), const_cast<float**>(&su), &q, &d, &K, &cnt, &ncnt};
  e = cudaLaunchKernel(fn, dim3(M), dim3(threads), args, smem, st);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_rotate_out(const PartRef& pr, long long units, int grid, const float* sv,
                              uint16_t* y, int M, int mpad, cudaStream_t st) {
  const long long warps = (long long)M * (pr.N / kHad);
  PdlLaunch dl(blocks_for(warps), 32 * kWarpsPerBlock, 0, st);
  return cudaLaunchKernelEx(&dl.cfg, rotate_out_kernel, pr, units, grid, sv, y, M, mpad);
}

cudaError_t launch_mlp_mid(const PartRef& gate, const PartRef& up, long long units, int grid,
                           const float* sv_gate, const float* sv_up, const float* su_down,
                           uint32_t* xfrag_down, int M, cudaStream_t st) {
  const long long warps = (long long)M * (gate.N / kHad);
  PdlLaunch dl(blocks_for(warps), 32 * kWarpsPerBlock, 0, st);
  return cudaLaunchKernelEx(&dl.cfg, mlp_mid_kernel, gate, up, units, grid, sv_gate, sv_up,
                            su_down, xfrag_down, M);
}

}  // namespace escha
