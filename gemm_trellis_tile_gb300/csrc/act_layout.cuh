// Activation-side helpers shared by the rotation, MLP and MoE kernels: the
// GEMV's fragment layout for rotated activations, fp16 vector loads/stores,
// and the sum over a 128-channel group's partial-sum slots.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace escha {

// CTA that owns unit u when U units are split into G near-equal contiguous
// ranges (CTA c owns [c*U/G, (c+1)*U/G)).
__host__ __device__ __forceinline__ int owner_cta(long long u, long long U, int G) {
  return static_cast<int>(((u + 1) * G - 1) / U);
}

// Store one rotated activation (fp16 bits) of token m (of M) at its place in
// the GEMV's B-fragment layout [K/16][M][4][4 words]: per k-tile and token,
// lane t's four words (x[2t], x[2t]), (x[2t+8], x[2t+8]), (x[2t+1], x[2t+1]),
// (x[2t+9], x[2t+9]) -- each activation in both halves, against the (lo, hi)
// halves of a codebook word in the weight operand.  Only the M real tokens
// are stored; the GEMV gives lanes of absent tokens zeros.
__device__ __forceinline__ void xfrag_store(uint32_t* xf, int M, int m, int k, uint16_t hb) {
  const int kt = k >> 4, kk = k & 15;
  const int t = (kk & 7) >> 1, odd = kk & 1, hi8 = kk >> 3;
  const int reg = 2 * odd + hi8;
  xf[(((size_t)kt * M + m) * 4 + t) * 4 + reg] = uint32_t(hb) | (uint32_t(hb) << 16);
}

__device__ __forceinline__ void load4_half(const uint16_t* p, float (&v)[4]) {
  const uint2 raw = *reinterpret_cast<const uint2*>(p);
  v[0] = half_bits_to_float(raw.x & 0xFFFF);
  v[1] = half_bits_to_float(raw.x >> 16);
  v[2] = half_bits_to_float(raw.y & 0xFFFF);
  v[3] = half_bits_to_float(raw.y >> 16);
}

__device__ __forceinline__ void store4_half(uint16_t* p, const float (&v)[4]) {
  uint2 raw;
  raw.x = float_to_half_bits(v[0]) | (uint32_t(float_to_half_bits(v[1])) << 16);
  raw.y = float_to_half_bits(v[2]) | (uint32_t(float_to_half_bits(v[3])) << 16);
  *reinterpret_cast<uint2*>(p) = raw;
}

__device__ __forceinline__ float4 load4_f32(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}

// Sum a group's partial-sum slots for token m, channels 128g + 4*lane .. +3.
// The group's KT units start at unit `ub`; slot s belongs to the s-th CTA
// that covers them.  All slot loads (up to 16 at a time) are issued before the
// first addition so their L2 latencies overlap; the slots are added in order.
// kBatch: loads in flight (more registers; a caller with few slots picks less).
template <int kBatch = 16>
__device__ __forceinline__ void sum_slots(const float* part, long long ub, int KT, int N,
                                          long long U, int G, int mpad, int m, int g, int lane,
                                          float (&v)[4]) {
  const long long gb = ub + (long long)g * KT;
  const int ns = owner_cta(gb + KT - 1, U, G) - owner_cta(gb, U, G) + 1;
  const float* p = part + (size_t)m * N + 128 * g + 4 * lane;
  const size_t step = (size_t)mpad * N;
  v[0] = v[1] = v[2] = v[3] = 0.f;
  for (int s0 = 0; s0 < ns; s0 += kBatch) {
    float4 q[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i)
      if (s0 + i < ns) q[i] = load4_f32(p + (size_t)(s0 + i) * step);
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      if (s0 + i < ns) {
        v[0] += q[i].x;
        v[1] += q[i].y;
        v[2] += q[i].z;
        v[3] += q[i].w;
      }
    }
  }
}

// Two groups' sums at once (the gate and up matrices of a gated MLP): both
// sets of slot loads are in flight together.
template <int kBatch = 8>
__device__ __forceinline__ void sum_slots_pair(const float* part_a, long long ub_a, const float* part_b,
                                               long long ub_b, int KT, int N, long long U, int G,
                                               int mpad, int m, int g, int lane, float (&va)[4],
                                               float (&vb)[4]) {
  const long long ga = ub_a + (long long)g * KT, gbb = ub_b + (long long)g * KT;
  const int na = owner_cta(ga + KT - 1, U, G) - owner_cta(ga, U, G) + 1;
  const int nb = owner_cta(gbb + KT - 1, U, G) - owner_cta(gbb, U, G) + 1;
  const float* pa = part_a + (size_t)m * N + 128 * g + 4 * lane;
  const float* pb = part_b + (size_t)m * N + 128 * g + 4 * lane;
  const size_t step = (size_t)mpad * N;
  va[0] = va[1] = va[2] = va[3] = 0.f;
  vb[0] = vb[1] = vb[2] = vb[3] = 0.f;
  const int n = na > nb ? na : nb;
  for (int s0 = 0; s0 < n; s0 += kBatch) {
    float4 qa[kBatch], qb[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      if (s0 + i < na) qa[i] = load4_f32(pa + (size_t)(s0 + i) * step);
      if (s0 + i < nb) qb[i] = load4_f32(pb + (size_t)(s0 + i) * step);
    }
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      if (s0 + i < na) {
        va[0] += qa[i].x;
        va[1] += qa[i].y;
        va[2] += qa[i].z;
        va[3] += qa[i].w;
      }
      if (s0 + i < nb) {
        vb[0] += qb[i].x;
        vb[1] += qb[i].y;
        vb[2] += qb[i].z;
        vb[3] += qb[i].w;
      }
    }
  }
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

// One warp's share of an input rotation: token m, 128-channel block kb of
// xh = fp16(had128(x * su)), stored in the GEMV's fragment layout (M tokens).
__device__ __forceinline__ void rotate_in_block(const uint16_t* x, const float* su,
                                               uint32_t* xfrag, int K, int M, int m, int kb,
                                               int lane) {
  const int k0 = kb * kHad + 4 * lane;
  float v[4];
  load4_half(x + (size_t)m * K + k0, v);
  const float4 s = *reinterpret_cast<const float4*>(su + k0);
  v[0] *= s.x;
  v[1] *= s.y;
  v[2] *= s.z;
  v[3] *= s.w;
  fwht128_warp(v, lane);
#pragma unroll
  for (int r = 0; r < 4; ++r) xfrag_store(xfrag, M, m, k0 + r, float_to_half_bits(v[r] * kHadScale));
}

}  // namespace escha
