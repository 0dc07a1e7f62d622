// Prefill GEMM for trellis-coded layers on the 5th-generation tensor cores:
//   y[M, N] = fp16( had128( xh[M, K] @ W_inner[K, N] ) * sv ),  xh = had128(x * su)
// (activation-side reconstruction, "Escha-W2 runs on Metal"; decode as in
// "The escha W2 format, recovered and verified", "Bit layout" / "Codebook").
//
// One CTA computes a 256 x 128 output tile (two M=128 accumulators in TMEM
// sharing one decoded B tile, so each weight is decoded once per 256 rows).
// The K loop runs in blocks of 64 (one 128-byte swizzle row of fp16) through
// a 4-stage shared-memory ring:
//   warp 0     producer: TMA tiled load of the A block (256 x 64, 128B
//              swizzle, rows past M zero-filled) and 1-D bulk copies of the
//              4 x 8 code tiles of the block, on one mbarrier.
//   warp 1     owns TMEM (256 columns) and, from one lane, issues the
//              tcgen05.mma kind::f16 instructions (2 accumulators x 4 K-steps)
//              once a stage's A has landed and its B is decoded; a
//              tcgen05.commit frees the stage.
//   warps 2-17 decoders: each decodes 2 tiles per block in registers and
//              stores fp16 pairs straight into the canonical K-major
//              128B-swizzled B layout; then the epilogue: TMEM -> registers ->
//              shared stash, 128-point Hadamard across each row's 128 output
//              channels (one warp per row), * sv, coalesced fp16 stores.
// Every mbarrier wait is bounded; a wait that runs out sets the error word and
// the CTA unwinds without hanging (TMEM is always released).

#include <cuda.h>
#include <cuda_runtime.h>

#include "act_layout.cuh"
#include "common.cuh"
#include "internal.h"
#include "trellis_decode.cuh"

namespace escha {

namespace {

constexpr int kBM = 256;          // rows per CTA (two M=128 MMAs)
constexpr int kBN = 128;          // output channels per CTA (= one Hadamard block)
constexpr int kBK = 64;           // K per pipeline stage (128 bytes of fp16)
constexpr int kStagesG = 4;
constexpr int kThreadsG = 576;    // 18 warps
constexpr int kDecWarps = 16;
constexpr int kTmemCols = 256;

constexpr int kABytes = kBM * kBK * 2;           // 32 KB
constexpr int kBBytes = kBN * kBK * 2;           // 16 KB
constexpr int kCodeBytes = 4 * 8 * 128;          // 4 k-tiles x 8 n-tiles, sized for 4 bits
constexpr int kStageBytes = kABytes + kBBytes + kCodeBytes;
constexpr int kStashStride = kBN + 1;            // floats per stashed row (bank-conflict free)
constexpr int kSmemBytes = kStagesG * kStageBytes + 1024 /*barriers*/ + 1024 /*alignment*/;
static_assert(kBM * kStashStride * 4 <= kStagesG * kStageBytes, "stash must fit the ring");

struct GemmArgs {
  const uint8_t* code;
  const float* sv;
  uint16_t* y;
  int M, N, K;
  int* err;
  uint64_t limit_ns;
};

// ---------------------------------------------------------------- PTX wrappers

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t smem_slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_slot),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc], fp16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05 operation issued so far by this thread completes.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void named_barrier(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Shared-memory matrix descriptor: K-major operand whose rows are 128 bytes
// (64 fp16), 128-byte swizzle, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t smem_desc_k128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);  // start address
  d |= (uint64_t)1 << 16;                    // leading byte offset (unused with this swizzle)
  d |= (uint64_t)(1024 >> 4) << 32;          // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;                    // descriptor version
  d |= (uint64_t)2 << 61;                    // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: fp16 A and B (both K-major), fp32 D,
// M = 128, N = 128.
constexpr uint32_t kIdesc = (1u << 4)            // D format: f32
                            | (0u << 7)          // A format: f16
                            | (0u << 10)         // B format: f16
                            | ((kBN >> 3) << 17) // N / 8
                            | ((128 >> 4) << 24);  // M / 16

// ---------------------------------------------------------------- kernel

template <int BITS>
__global__ void __launch_bounds__(kThreadsG, 1)
    trellis_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  // ring: per stage [A 32 KB][B 16 KB][codes 4 KB]; then barriers
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStagesG * kStageBytes);
  // bars[0..3] load_full, [4..7] b_full, [8..11] empty, [12] acc_full, [13] mma_done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 16);
  auto stage_a = [&](int s) { return base + s * kStageBytes; };
  auto stage_b = [&](int s) { return base + s * kStageBytes + kABytes; };
  auto stage_code = [&](int s) { return smem + s * kStageBytes + kABytes + kBBytes; };
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_block = blockIdx.x;
  const int m0 = blockIdx.y * kBM;
  const int n0 = n_block * kBN;
  const int num_kb = a.K / kBK;
  constexpr int T = 32 * BITS;
  const int NT = a.N / 16;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesG; ++s) {
      mbar_init(bar(s), 1);              // load_full: producer arrive + tx bytes
      mbar_init(bar(4 + s), kDecWarps);  // b_full: one arrive per decoder warp
      mbar_init(bar(8 + s), 1);          // empty: tcgen05.commit
    }
    mbar_init(bar(12), 1);  // acc_full
    mbar_init(bar(13), 1);  // mma_done (unwinding)
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      int armed[kStagesG];
      for (int s = 0; s < kStagesG; ++s) armed[s] = -1;
      bool ok = true;
      for (int kb = 0; kb < num_kb; ++kb) {
        const int s = kb % kStagesG;
        const uint32_t ph = (kb / kStagesG) & 1;
        if (!mbar_wait(bar(8 + s), ph ^ 1u, a.limit_ns)) {
          set_error(a.err, kDevErrTimeout);
          ok = false;
          break;
        }
        const uint32_t row_bytes = 8 * T;
        mbar_arrive_expect_tx(bar(s), kABytes + 4 * row_bytes);
        tma_load_2d(stage_a(s), &tmap_a, kb * kBK, m0, bar(s));
        const uint32_t cdst = smem_u32(stage_code(s));
        for (int r = 0; r < 4; ++r) {
          const uint8_t* src = a.code + ((size_t)(4 * kb + r) * NT + 8 * n_block) * T;
          bulk_g2s(cdst + r * row_bytes, src, row_bytes, bar(s));
        }
        armed[s] = static_cast<int>(ph);
      }
      if (!ok) {
        for (int s = 0; s < kStagesG; ++s)
          if (armed[s] >= 0) mbar_wait(bar(s), static_cast<uint32_t>(armed[s]), a.limit_ns);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      for (int kb = 0; kb < num_kb; ++kb) {
        const int s = kb % kStagesG;
        const uint32_t ph = (kb / kStagesG) & 1;
        if (!mbar_wait(bar(s), ph, a.limit_ns) || !mbar_wait(bar(4 + s), ph, a.limit_ns)) {
          set_error(a.err, kDevErrTimeout);
          break;
        }
        tc_fence_after();
        const uint32_t sa = stage_a(s), sb = stage_b(s);
#pragma unroll
        for (int acc = 0; acc < 2; ++acc) {
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint64_t ad = smem_desc_k128(sa + acc * (kABytes / 2) + kk * 32);
            const uint64_t bd = smem_desc_k128(sb + kk * 32);
            mma_f16(tmem_base + acc * kBN, ad, bd, kIdesc, (kb > 0 || kk > 0) ? 1u : 0u);
          }
        }
        mma_commit(bar(8 + s));  // stage s may be refilled once these MMAs are done
      }
      mma_commit(bar(12));  // accumulators complete
      mma_commit(bar(13));
      mbar_wait(bar(13), 0, a.limit_ns);  // nothing left in flight before TMEM is released
    }
  } else {
    // ---------------------------------------------------------- decoders
    const int dw = warp - 2;          // 0..15
    const int kt_local = dw >> 2;     // k-tile row within the block
    const int nt_base = (dw & 3) * 2; // 2 n-tiles per warp
    const LaneWindow lw = lane_window<BITS>(lane);
    const int g = lane >> 2, t = lane & 3;
    bool ok = true;
    for (int kb = 0; kb < num_kb && ok; ++kb) {
      const int s = kb % kStagesG;
      const uint32_t ph = (kb / kStagesG) & 1;
      // B[s] must be free (previous MMAs on it done) and the codes must have landed.
      if (!mbar_wait(bar(8 + s), ph ^ 1u, a.limit_ns) || !mbar_wait(bar(s), ph, a.limit_ns)) {
        set_error(a.err, kDevErrTimeout);
        ok = false;
        break;
      }
      const uint8_t* codes = stage_code(s);
      uint8_t* bt = smem + (stage_b(s) - base);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int nt = nt_base + i;
        const uint32_t* tw = reinterpret_cast<const uint32_t*>(codes + (kt_local * 8 + nt) * T);
        uint32_t h[8];
        decode8<BITS>(tw[lw.i0], tw[lw.i1], lw.sh7, h);
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const int rh = p & 1, nh = p >> 1;
          const int n = 16 * nt + g + 8 * nh;
          const int chunk = (2 * kt_local + rh) ^ g;
          const uint32_t pair = __byte_perm(h[2 * p], h[2 * p + 1], 0x5410);
          *reinterpret_cast<uint32_t*>(bt + n * 128 + chunk * 16 + 4 * t) = pair;
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(4 + s));
    }

    // ---------------------------------------------------------- epilogue
    // Pass 1: each (accumulator, TMEM lane quadrant, 64-column half) is one warp.
    const int quad = warp & 3;        // TMEM lane quadrant this warp may access
    const int acc = (dw >> 2) & 1;
    const int half = dw >> 3;
    __syncwarp();
    const bool have = ok && mbar_wait(bar(12), 0, a.limit_ns);
    if (!have && ok) set_error(a.err, kDevErrTimeout);
    tc_fence_after();
    float* stash = reinterpret_cast<float*>(smem);
    if (have) {
      const int row = acc * 128 + quad * 32 + lane;
#pragma unroll
      for (int c = 64 * half; c < 64 * half + 64; c += 32) {
        uint32_t r[32];
        tmem_ld32(tmem_base + ((uint32_t)(quad * 32) << 16) + acc * kBN + c, r);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) stash[row * kStashStride + c + j] = __uint_as_float(r[j]);
      }
    }
    tc_fence_before();
    named_barrier(1, kDecWarps * 32);
    // Pass 2: one warp per row, element lane + 32*q in v[q].
    if (have) {
      float svv[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) svv[q] = a.sv[n0 + lane + 32 * q] * kHadScale;
      for (int rr = 0; rr < kBM / kDecWarps; ++rr) {
        const int row = dw * (kBM / kDecWarps) + rr;
        const int m = m0 + row;
        if (m >= a.M) break;
        float v[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) v[q] = stash[row * kStashStride + lane + 32 * q];
        fwht128_warp_strided(v, lane);
        uint16_t* yr = a.y + (size_t)m * a.N + n0 + lane;
#pragma unroll
        for (int q = 0; q < 4; ++q) yr[32 * q] = float_to_half_bits(v[q] * svv[q]);
      }
    }
  }

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

template <int BITS>
cudaError_t launch_gemm_bits(const CUtensorMap& map, const GemmArgs& a, cudaStream_t st) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(trellis_gemm_kernel<BITS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  dim3 grid(a.N / kBN, (a.M + kBM - 1) / kBM);
  trellis_gemm_kernel<BITS><<<grid, kThreadsG, kSmemBytes, st>>>(map, a);
  return cudaGetLastError();
}

}  // namespace

// xh: rotated activations fp16 [M, K] (16-byte aligned, K a multiple of 128).
cudaError_t launch_trellis_gemm(const uint16_t* xh, const int16_t* code, int bits, int M, int K,
                                int N, const float* sv, uint16_t* y, int* err, cudaStream_t st) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  CUtensorMap map;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
  const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  const cuuint32_t box[2] = {kBK, kBM};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<uint16_t*>(xh), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  GemmArgs a;
  a.code = reinterpret_cast<const uint8_t*>(code);
  a.sv = sv;
  a.y = y;
  a.M = M;
  a.N = N;
  a.K = K;
  a.err = err;
  a.limit_ns = kWaitLimitNs;
  switch (bits) {
    case 2: return launch_gemm_bits<2>(map, a, st);
    case 3: return launch_gemm_bits<3>(map, a, st);
    default: return launch_gemm_bits<4>(map, a, st);
  }
}

}  // namespace escha
