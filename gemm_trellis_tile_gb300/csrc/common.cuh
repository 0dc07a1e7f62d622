// Device-side helpers shared by the libescha kernels: mbarrier waits with a
// time limit, 1-D bulk copies (TMA engine), the in-register Hadamard-128
// butterflies and fp16 bit helpers.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace escha {

constexpr int kHad = 128;                          // Hadamard block size
constexpr float kHadScale = 0.08838834764831845f;  // 1/sqrt(128)

// Default limit of a bounded device wait (nanoseconds).
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void set_error(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- dependent launch

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialisation may start before its predecessor in the stream finishes.
// pdl_wait() blocks until the predecessor grid has completed and its writes
// are visible (a no-op when the kernel was launched normally);
// pdl_trigger() lets the successor grid be scheduled early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Named barrier among `nthreads` threads (a multiple of 32, whole warps).
// Id 0 is the one __syncthreads() uses.
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------- tensor maps

// A tensor map in global memory that was written through ordinary stores
// (or copied from the host) becomes visible to the TMA unit after this fence.
__device__ __forceinline__ void tensormap_acquire(const void* map) {
  asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(map) : "memory");
}
// Writer side of the same hand-over (after storing a tensor map).
__device__ __forceinline__ void tensormap_release() {
  asm volatile("fence.proxy.tensormap::generic.release.gpu;" ::: "memory");
}

// 2-D tiled TMA load of box (x, y) of `map` into shared memory, completing on
// an mbarrier, with an L2 cache policy.
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const void* map, int x, int y,
                                                 uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Same, but the thread may stay suspended inside the instruction for up to
// `hint_ns` until the phase completes (fewer polling instructions while a
// stage is in flight).
__device__ __forceinline__ bool mbar_try_wait_hint(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1; it < (1u << 30); ++it) {
    if (mbar_try_wait_hint(bar, parity, 100000u)) return true;
    if ((it & 7u) == 0 && globaltimer_ns() - t0 > limit_ns) return false;
  }
  return false;
}

// ---------------------------------------------------------------- bulk copy

// 1-D bulk copy global -> shared, completing on an mbarrier (TMA engine).
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Same, with an L2 eviction-priority hint (streamed once: evict first).
__device__ __forceinline__ void bulk_g2s_evict_first(uint32_t dst, const void* src, uint32_t bytes,
                                                     uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], "
      "[%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---------------------------------------------------------------- Hadamard

// Fast Walsh-Hadamard transform of one 128-block held by a warp, four
// consecutive elements per lane (element 4*lane + r in v[r]); natural
// (Sylvester) order, unnormalised.  Two butterfly stages in registers, five
// across lanes.  A cross-lane stage forms v + o in the lower lane and o - v in
// the upper one as fma(+-1, v, o): the product by +-1 is exact, so this is the
// same single rounding as the addition, in one instruction.
__device__ __forceinline__ void fwht128_warp(float (&v)[4], int lane) {
  const float a0 = v[0] + v[1], a1 = v[0] - v[1];
  const float a2 = v[2] + v[3], a3 = v[2] - v[3];
  v[0] = a0 + a2;
  v[2] = a0 - a2;
  v[1] = a1 + a3;
  v[3] = a1 - a3;
#pragma unroll
  for (int s = 0; s < 5; ++s) {
    const int m = 1 << s;
    const float sgn = (lane & m) ? -1.0f : 1.0f;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const float o = __shfl_xor_sync(0xffffffffu, v[r], m);
      v[r] = fmaf(sgn, v[r], o);
    }
  }
}

// The same transform with eight consecutive elements per lane: a 128-block
// per half-warp (element 8*(lane & 15) + r in v[r]).  Three butterfly stages
// in registers, four across the half-warp's lanes, in the same order of index
// bits and with the same operations as fwht128_warp, so the results are
// bit-identical.  Every lane of the warp must take part.
__device__ __forceinline__ void fwht128_halfwarp(float (&v)[8], int lane) {
#pragma unroll
  for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if ((i & h) == 0) {
        const float p = v[i], q = v[i + h];
        v[i] = p + q;
        v[i + h] = p - q;
      }
    }
  }
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const int m = 1 << s;
    const float sgn = (lane & m) ? -1.0f : 1.0f;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const float o = __shfl_xor_sync(0xffffffffu, v[r], m);
      v[r] = fmaf(sgn, v[r], o);
    }
  }
}

__device__ __forceinline__ float half_bits_to_float(uint16_t b) {
  return __half2float(__ushort_as_half(b));
}

__device__ __forceinline__ uint16_t float_to_half_bits(float f) {
  return __half_as_ushort(__float2half_rn(f));
}

}  // namespace escha
