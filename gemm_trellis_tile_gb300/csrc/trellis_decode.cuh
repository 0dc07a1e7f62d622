// Trellis tile decode in registers.
//
// A 16x16 tile of `BITS`-bit weights is 8*BITS little-endian uint32 words.
// Read MSB first, word after word, they form a circular stream of 256*BITS
// bits; state s is the 16-bit window ending at stream bit BITS*(s+1)-1
// ("The escha W2 format, recovered and verified", section "Bit layout"; the
// Metal page calls it the window at offset i*K, tail-biting).
//
// Lane L of a warp decodes symbols 8L..8L+7.  All eight windows lie inside one
// 64-bit pair of consecutive words (i0, i1), where i1 holds the last bit of
// symbol 8L+7.  After one funnel shift by sh7 the windows sit at the fixed
// offsets BITS*(7-j), so the per-symbol work is a constant-offset extraction.
//
// Each state goes through the cb=1 MCG codebook (section "Codebook: cb=1"):
//   v = state * 0xCBAC1FED; v = (v & 0x8FFF8FFF) ^ 0x3B603B60;
//   w = fp16(v.lo) + fp16(v.hi)   -- one fp16 addition, round to nearest even.
// In the EXLR8 variant (EXLR8 format page) w is then rounded to FP8 E4M3,
// nearest even, saturating at 448.
//
// Placement: lane L = 4g + t, symbol j of the lane sits at tile row (input
// channel) r = 2t + (j&1) + 8((j>>1)&1) and column (output channel)
// c = g + 8(j>>2): the m16n8k16 B-fragment order (Metal page, closed-form
// inverse of the tensor-core permutation).  Seen as W^T (rows = output
// channel), the same eight values are the lane's m16n8k16 A fragment:
//   a0 <- j=0,1   a1 <- j=4,5   a2 <- j=2,3   a3 <- j=6,7.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace escha {

constexpr uint32_t kMcgMult = 0xCBAC1FEDu;
constexpr uint32_t kMcgMask = 0x8FFF8FFFu;
constexpr uint32_t kMcgXor = 0x3B603B60u;

struct LaneWindow {
  int i0;    // word holding the start of the lane's bit span
  int i1;    // word holding the last bit of symbol 8L+7
  int sh7;   // right shift of (w[i0]:w[i1]) that puts symbol 7's window at bit 0
};

template <int BITS>
__device__ __forceinline__ LaneWindow lane_window(int lane) {
  const int nwords = 8 * BITS;
  const int e7 = BITS * (8 * lane + 8) - 1;  // stream bit ending symbol 8L+7
  LaneWindow lw;
  lw.i1 = e7 >> 5;
  lw.i0 = (lw.i1 + nwords - 1) % nwords;     // circular: tail-biting
  lw.sh7 = 31 - (e7 & 31);
  return lw;
}

// Codebook value of one state, replicated into both fp16 halves: one HADD2
// with both operands broadcast from the word, (lo,lo) + (hi,hi).
__device__ __forceinline__ uint32_t mcg_decode_dup(uint32_t state) {
  uint32_t v = state * kMcgMult;
  v = (v & kMcgMask) ^ kMcgXor;
  const __half2 h = *reinterpret_cast<const __half2*>(&v);
  const __half2 s = __hadd2(__low2half2(h), __high2half2(h));
  return *reinterpret_cast<const uint32_t*>(&s);
}

// E4M3 rounding of a pair of fp16 values (nearest even, saturating to the
// largest finite E4M3 value), returned as the two fp16 values it rounds to
// (every E4M3 value is exact in fp16).  One hardware conversion each way.
__device__ __forceinline__ uint32_t round_e4m3x2(uint32_t w2) {
  uint16_t e;
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(e) : "r"(w2));
  uint32_t d;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"(e));
  return d;
}

// The codebook word of one state before its final addition: fp16 lo in the
// low half, fp16 hi in the high half.  A tensor-core contraction against an
// operand that carries the same activation in both halves forms lo*x + hi*x
// in fp32, i.e. the codebook sum without its fp16 rounding (the rounding
// changes a weight by at most half an fp16 ulp of lo + hi).
//
// `mask` and `xr` are kMcgMask and kMcgXor, passed in at run time: given two
// literal constants the compiler spends two integer instructions on the
// mask-and-flip, given one in a register it uses a single three-input logic op.
__device__ __forceinline__ uint32_t mcg_pair(uint32_t state, uint32_t mask, uint32_t xr) {
  return ((state * kMcgMult) & mask) ^ xr;
}

// 16-bit field starting at byte `b` (0..2) of x, zero-extended (one PRMT).
__device__ __forceinline__ uint32_t field16_at_byte(uint32_t x, int b) {
  return __byte_perm(x, 0u, b == 0 ? 0x4410 : (b == 1 ? 0x4421 : 0x4432));
}

// The lane's eight 16-bit states.  (lo, hi) is the lane's 64-bit span shifted
// so that symbol 7's window starts at bit 0; symbol j's window starts at bit
// s = BITS*(7-j) <= 28.  A window with s <= 16 is moved up to the next byte
// boundary of lo by a left shift (s + k = 8*ceil(s/8), and the window still
// ends by bit 32), the others likewise in m = bits 16..47 of the span; one
// byte permute then extracts it zero-extended.  The left shifts are constant
// multiplies, which the compiler can issue on the multiply pipe, leaving the
// integer ALU pipe (the decode's bottleneck) one permute per state.
template <int BITS>
__device__ __forceinline__ void lane_states(uint32_t lo, uint32_t hi, uint32_t (&st)[8]) {
  const uint32_t m = __funnelshift_r(lo, hi, 16);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int s = BITS * (7 - j);
    const uint32_t src = s <= 16 ? lo : m;
    const int sr = s <= 16 ? s : s - 16;
    const int b = (sr + 7) / 8;
    const int k = 8 * b - sr;
    st[j] = field16_at_byte(src * (1u << k), b);
  }
}

// Decode the lane's eight symbols from its word pair.  out[j] holds symbol
// 8L+j's value in both fp16 halves (E4M3: the codebook value rounded to E4M3).
template <int BITS, bool E4M3 = false>
__device__ __forceinline__ void decode8(uint32_t w0, uint32_t w1, int sh7, uint32_t (&out)[8]) {
  const uint32_t lo = __funnelshift_r(w1, w0, sh7);
  const uint32_t hi = w0 >> sh7;
  uint32_t st[8];
  lane_states<BITS>(lo, hi, st);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    out[j] = mcg_decode_dup(st[j]);
    if (E4M3) out[j] = round_e4m3x2(out[j]);
  }
}

// E4M3 variant for the GEMV in the m16n8k16 A-fragment layout: the lane's
// eight weights as four registers of two weights each (a0 <- symbols 0,1,
// a1 <- 4,5, a2 <- 2,3, a3 <- 6,7: two input channels of one output channel),
// each the codebook's fp16 sum rounded to E4M3 (and held exactly in fp16).
// Per pair of states: one HADD2 each with its operands' halves broadcast
// ((lo, lo) + (hi, hi), no separate permute), one byte permute joins the two
// sums, one conversion pair rounds both to E4M3.
template <int BITS>
__device__ __forceinline__ void decode8_e4m3_frag(uint32_t w0, uint32_t w1, int sh7, uint32_t mask,
                                                  uint32_t xr, uint32_t (&a)[4]) {
  const uint32_t lo = __funnelshift_r(w1, w0, sh7);
  const uint32_t hi = w0 >> sh7;
  uint32_t st[8];
  lane_states<BITS>(lo, hi, st);
  uint32_t v[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = mcg_pair(st[j], mask, xr);
  constexpr int first[4] = {0, 4, 2, 6};  // a0..a3
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int j = first[r];
    const __half2 h0 = *reinterpret_cast<const __half2*>(&v[j]);
    const __half2 h1 = *reinterpret_cast<const __half2*>(&v[j + 1]);
    const __half2 s0 = __hadd2(__low2half2(h0), __high2half2(h0));
    const __half2 s1 = __hadd2(__low2half2(h1), __high2half2(h1));
    a[r] = round_e4m3x2(__byte_perm(*reinterpret_cast<const uint32_t*>(&s0),
                                    *reinterpret_cast<const uint32_t*>(&s1), 0x5410));
  }
}

// The lane's eight codebook words as (lo, hi) fp16 pairs (see mcg_pair).
template <int BITS>
__device__ __forceinline__ void decode8_pairs(uint32_t w0, uint32_t w1, int sh7, uint32_t mask,
                                              uint32_t xr, uint32_t (&out)[8]) {
  const uint32_t lo = __funnelshift_r(w1, w0, sh7);
  const uint32_t hi = w0 >> sh7;
  uint32_t st[8];
  lane_states<BITS>(lo, hi, st);
#pragma unroll
  for (int j = 0; j < 8; ++j) out[j] = mcg_pair(st[j], mask, xr);
}

// Tile coordinates of lane symbol j (row = input channel, col = output channel).
__device__ __forceinline__ int sym_row(int lane, int j) {
  return 2 * (lane & 3) + (j & 1) + 8 * ((j >> 1) & 1);
}
__device__ __forceinline__ int sym_col(int lane, int j) { return (lane >> 2) + 8 * (j >> 2); }

}  // namespace escha
