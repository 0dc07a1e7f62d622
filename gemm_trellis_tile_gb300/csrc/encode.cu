// Trellis encoder: the Viterbi search that picks each tile's code.
//
// EXLR8 format page, the Viterbi search: each 16x16 tile is coded as a whole,
// by the trellis path whose decoded values (the mcg codebook's value of each
// step's state) have the least squared error against the tile; the E4M3
// variant rounds every codebook value inside the search.  The stream is
// circular (tail-biting; "Escha-W2 runs on Metal": code i is the 16-bit window
// at offset i*K, wrapping around).
//
// State s of symbol i is its 16-bit window; the next state is
// ((s << K) | new K bits) & 0xFFFF, so the predecessors of state s are the
// 2^K states (s >> K) | (t << (16 - K)).  Writing u for the low 16 - K bits
// of a state, all states of group u = {u | t << (16 - K)} have the same
// successors.  Between steps the search keeps, per group, only the least cost
// of its states (m[u]) and the t that reaches it:
//   m_i[u] = min_t ( (v_i - c(u | t << (16-K)))^2 + m_{i-1}[(u | t << (16-K)) >> K] ).
// The tail-biting constraint is met with two passes: pass 1 lets every start
// state in; pass 2 fixes the 16 - K bits the last window shares with the first
// (taken from pass 1's best end state) and allows only start and end states
// that agree with them.
//
// Arithmetic is fp32 with the difference, square and sum each rounded (no
// fused multiply-add) and ties broken towards the lowest t and the lowest end
// state, so the search takes the same decisions as the CPU oracle's.
//
// One CTA of 1024 threads per tile (persistent over tiles); m lives in shared
// memory (two buffers of 2^(16-K) floats), the per-step choices of t in a
// global scratch area (256 x 2^(16-K) bytes per CTA).

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"
#include "trellis_decode.cuh"

namespace escha {

namespace {

constexpr int kEncThreads = 1024;
#define ENC_INF __int_as_float(0x7f800000)

// Codebook value of a state as fp16 (the fp16 value, or its E4M3 rounding;
// both are exact in fp16).
template <bool E4M3>
__device__ __forceinline__ __half codebook_h(uint32_t s) {
  uint32_t d = mcg_decode_dup(s);
  if (E4M3) d = round_e4m3x2(d);
  return __ushort_as_half(static_cast<unsigned short>(d & 0xFFFFu));
}

// A thread's states: groups u = tid + k * kEncThreads (k < KPT) of the states
// u | t << (16 - K) (t < 2^K) -- 64 states, the same at every step.  Their
// codebook values stay in registers for the whole search, value k * 2^K + t
// in half (k * 2^K + t) & 1 of cb[(k * 2^K + t) / 2].
constexpr int kCbPairs = (1 << 16) / kEncThreads / 2;

template <int K, bool E4M3>
__device__ __forceinline__ void load_codebook(__half2 (&cb)[kCbPairs]) {
  constexpr int TT = 1 << K;
  const uint32_t tid = threadIdx.x;
#pragma unroll
  for (int q = 0; q < kCbPairs; ++q) {
    const int i0 = 2 * q, i1 = 2 * q + 1;
    const uint32_t s0 = (tid + (i0 / TT) * kEncThreads) | (uint32_t(i0 % TT) << (16 - K));
    const uint32_t s1 = (tid + (i1 / TT) * kEncThreads) | (uint32_t(i1 % TT) << (16 - K));
    cb[q] = __halves2half2(codebook_h<E4M3>(s0), codebook_h<E4M3>(s1));
  }
}

__device__ __forceinline__ float cb_value(const __half2 (&cb)[kCbPairs], int idx) {
  return (idx & 1) ? __high2float(cb[idx >> 1]) : __low2float(cb[idx >> 1]);
}

// One forward pass.  Pass 1 (o < 0): any start state.  Pass 2: start states
// with (s >> K) == o, end states with (s & mask) == o.  Leaves the choices of t
// in `back` ([256][nu] bytes) and returns the best end state (all threads).
// The predecessor (u | t << (16-K)) >> K of group u = tid + k * kEncThreads is
// (tid >> K) + k * (kEncThreads >> K) + t * 2^(16-2K): a fixed offset from
// the thread's base for every (k, t).
template <int K, bool E4M3>
__device__ int viterbi_pass(const __half2 (&cb)[kCbPairs], const float* vals, float* m0,
                            float* m1, uint8_t* back, int o, float* red_v, int* red_s,
                            float* total) {
  constexpr int kNu = 1 << (16 - K);
  constexpr uint32_t kMask = kNu - 1;
  constexpr int KPT = kNu / kEncThreads;  // groups per thread
  constexpr int TT = 1 << K;
  const int tid = threadIdx.x;
  const int pbase = tid >> K;
  // step 0: group minima of the first symbol's costs
  {
    const float v = vals[0];
#pragma unroll
    for (int k = 0; k < KPT; ++k) {
      const uint32_t u = static_cast<uint32_t>(tid + k * kEncThreads);
      float best = ENC_INF;
      int bt = 0;
#pragma unroll
      for (int t = 0; t < TT; ++t) {
        const uint32_t s = u | (static_cast<uint32_t>(t) << (16 - K));
        const float d = __fsub_rn(v, cb_value(cb, k * TT + t));
        float cost = __fmul_rn(d, d);
        if (o >= 0 && static_cast<int>(s >> K) != o) cost = ENC_INF;
        if (t == 0 || cost < best) {
          best = cost;
          bt = t;
        }
      }
      m0[u] = best;
      back[1 * kNu + u] = static_cast<uint8_t>(bt);
    }
  }
  __syncthreads();
  float* mp = m0;
  float* mc = m1;
  for (int i = 1; i < 255; ++i) {
    const float v = vals[i];
    const float* mpb = mp + pbase;
    uint8_t* bk = back + (size_t)(i + 1) * kNu;
#pragma unroll
    for (int k = 0; k < KPT; ++k) {
      const int u = tid + k * kEncThreads;
      float best = ENC_INF;
      int bt = 0;
#pragma unroll
      for (int t = 0; t < TT; ++t) {
        const float d = __fsub_rn(v, cb_value(cb, k * TT + t));
        const float cost =
            __fadd_rn(__fmul_rn(d, d), mpb[k * (kEncThreads >> K) + t * (1 << (16 - 2 * K))]);
        if (t == 0 || cost < best) {
          best = cost;
          bt = t;
        }
      }
      mc[u] = best;
      bk[u] = static_cast<uint8_t>(bt);
    }
    __syncthreads();
    float* tmp = mp;
    mp = mc;
    mc = tmp;
  }
  // last symbol: full costs, least one (lowest state on ties)
  float best = ENC_INF;
  int bs = 0x7fffffff;
  {
    const float v = vals[255];
    const float* mpb = mp + pbase;
#pragma unroll
    for (int k = 0; k < KPT; ++k) {
#pragma unroll
      for (int t = 0; t < TT; ++t) {
        const int s = (tid + k * kEncThreads) | (t << (16 - K));
        if (o >= 0 && static_cast<int>(static_cast<uint32_t>(s) & kMask) != o) continue;
        const float d = __fsub_rn(v, cb_value(cb, k * TT + t));
        const float cost =
            __fadd_rn(__fmul_rn(d, d), mpb[k * (kEncThreads >> K) + t * (1 << (16 - 2 * K))]);
        if (cost < best || (cost == best && s < bs)) {
          best = cost;
          bs = s;
        }
      }
    }
  }
  // block reduction: least cost, then least state
  const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float ov = __shfl_down_sync(0xFFFFFFFFu, best, off);
    const int os = __shfl_down_sync(0xFFFFFFFFu, bs, off);
    if (ov < best || (ov == best && os < bs)) {
      best = ov;
      bs = os;
    }
  }
  if (lane == 0) {
    red_v[warp] = best;
    red_s[warp] = bs;
  }
  __syncthreads();
  if (warp == 0) {
    best = red_v[lane];
    bs = red_s[lane];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_down_sync(0xFFFFFFFFu, best, off);
      const int os = __shfl_down_sync(0xFFFFFFFFu, bs, off);
      if (ov < best || (ov == best && os < bs)) {
        best = ov;
        bs = os;
      }
    }
    if (lane == 0) {
      red_s[0] = bs;
      *total = best;
    }
  }
  __syncthreads();
  const int end_state = red_s[0];
  __syncthreads();
  return end_state;
}

template <int K, bool E4M3>
__global__ void __launch_bounds__(kEncThreads, 1)
    trellis_encode_kernel(const float* w, int in_features, int out_features, int16_t* code,
                          float* sq_err, uint8_t* back_all) {
  constexpr int kNu = 1 << (16 - K);
  constexpr int kWords = 16 * K;  // int16 words per tile
  extern __shared__ __align__(16) float esm[];
  float* m0 = esm;
  float* m1 = esm + kNu;
  float* vals = esm + 2 * kNu;                             // [256]
  float* red_v = vals + 256;                               // [32]
  int* red_s = reinterpret_cast<int*>(red_v + 32);         // [32]
  uint32_t* states = reinterpret_cast<uint32_t*>(red_s + 32);  // [256]
  float* total = reinterpret_cast<float*>(states + 256);   // [1]
  uint8_t* back = back_all + (size_t)blockIdx.x * 256 * kNu;
  const int tid = threadIdx.x;
  const int KT = in_features / 16, NT = out_features / 16;
  const long long tiles = (long long)KT * NT;
  __half2 cb[kCbPairs];
  load_codebook<K, E4M3>(cb);
  for (long long tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
    const int ti = static_cast<int>(tile / NT);
    const int tj = static_cast<int>(tile - (long long)ti * NT);
    // symbol 8L + j sits at tile row sym_row(L, j), column sym_col(L, j)
    if (tid < 256) {
      const int lane = tid >> 3, j = tid & 7;
      const int r = sym_row(lane, j), c = sym_col(lane, j);
      vals[tid] = w[(size_t)(16 * ti + r) * out_features + 16 * tj + c];
    }
    __syncthreads();
    const int end1 = viterbi_pass<K, E4M3>(cb, vals, m0, m1, back, -1, red_v, red_s, total);
    const int o = end1 & (kNu - 1);
    const int end2 = viterbi_pass<K, E4M3>(cb, vals, m0, m1, back, o, red_v, red_s, total);
    if (tid == 0) {
      // trace the path back from the end state
      uint32_t s = static_cast<uint32_t>(end2) & 0xFFFFu;
      states[255] = s;
      for (int i = 255; i > 0; --i) {
        const uint32_t u = s >> K;
        s = u | (static_cast<uint32_t>(back[i * kNu + u]) << (16 - K));
        states[i - 1] = s;
      }
      if (sq_err) sq_err[tile] = *total;
    }
    __syncthreads();
    // stream bit K*i + t is bit K-1-t of state i; words MSB first, each uint32
    // split into two little-endian int16 words
    if (tid < kWords / 2) {
      uint32_t word = 0;
      for (int b = 0; b < 32; ++b) {
        const int pos = 32 * tid + b;
        const int i = pos / K, t = pos - (pos / K) * K;
        word |= ((states[i] >> (K - 1 - t)) & 1u) << (31 - b);
      }
      int16_t* dst = code + (size_t)tile * kWords + 2 * tid;
      dst[0] = static_cast<int16_t>(word & 0xFFFFu);
      dst[1] = static_cast<int16_t>(word >> 16);
    }
    __syncthreads();
  }
}

template <int K>
constexpr size_t enc_smem_bytes() {
  return (size_t)(2 * (1 << (16 - K)) + 256 + 32 + 32 + 256 + 4) * sizeof(float);
}

template <int K, bool E4M3>
cudaError_t launch_encode_k(const float* w, int in_f, int out_f, int16_t* code, float* sq_err,
                            uint8_t* back, int ctas, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(trellis_encode_kernel<K, E4M3>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(enc_smem_bytes<K>()));
  if (e != cudaSuccess) return e;
  trellis_encode_kernel<K, E4M3><<<ctas, kEncThreads, enc_smem_bytes<K>(), st>>>(
      w, in_f, out_f, code, sq_err, back);
  return cudaGetLastError();
}

}  // namespace

size_t encode_scratch_bytes(int bits, int ctas) {
  return (size_t)ctas * 256 * ((size_t)1 << (16 - bits));
}

cudaError_t launch_trellis_encode(const float* w, int in_features, int out_features, int bits,
                                  bool e4m3, int16_t* code, float* sq_err, uint8_t* scratch,
                                  int ctas, cudaStream_t st) {
  switch (bits + 8 * (e4m3 ? 1 : 0)) {
    case 2: return launch_encode_k<2, false>(w, in_features, out_features, code, sq_err, scratch, ctas, st);
    case 3: return launch_encode_k<3, false>(w, in_features, out_features, code, sq_err, scratch, ctas, st);
    case 4: return launch_encode_k<4, false>(w, in_features, out_features, code, sq_err, scratch, ctas, st);
    case 10: return launch_encode_k<2, true>(w, in_features, out_features, code, sq_err, scratch, ctas, st);
    case 11: return launch_encode_k<3, true>(w, in_features, out_features, code, sq_err, scratch, ctas, st);
    default: return launch_encode_k<4, true>(w, in_features, out_features, code, sq_err, scratch, ctas, st);
  }
}

}  // namespace escha
