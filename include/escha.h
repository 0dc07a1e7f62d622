/*
 * escha.h -- C ABI of libescha: trellis-coded (EXL3-style, cb=1) linear layers on
 * one sm_103a GPU.
 *
 * What is computed.  A layer stores W_inner [in, out] as 16x16 tiles, each tile a
 * tail-biting stream of 256 16-bit trellis states packed at `bits` bits per weight
 * (2, 3 or 4).  Each state decodes through the cb=1 MCG codebook
 *     v = state * 0xCBAC1FED;  v = (v & 0x8FFF8FFF) ^ 0x3B603B60;
 *     w = fp16(v.lo) + fp16(v.hi)            (one fp16 addition)
 * and lands in the tile at its tensor-core position.  The layer is applied on the
 * activation side:
 *     su = rin * s_in;  sv = rout * s_out
 *     y  = had128( had128(x * su) @ W_inner ) * sv
 * where had128 is the normalised Sylvester Hadamard H_128/sqrt(128) applied to
 * each consecutive block of 128 channels.
 * Sources: "The escha W2 format, recovered and verified" (sections "Tensor
 * mapping", "Reconstruction", "Codebook: cb=1 (MCG), verified", "Bit layout");
 * "Escha-W2 runs on Metal" (activation-side reconstruction, three-instruction
 * codebook, tile packing and the closed-form permutation inverse); the EXLR8
 * format page (shared per-layer rotation for routed experts, tile packing).
 *
 * Conventions for every call.
 *   - Tensor arguments are DEVICE pointers unless stated otherwise, row-major and
 *     contiguous, 16-byte aligned.  fp16 tensors are passed as uint16_t bit
 *     patterns (IEEE binary16).
 *   - Borrowing: code words and the caller's x / y buffers are borrowed, never
 *     copied; the caller keeps code alive for the handle's lifetime.  rin, rout,
 *     s_in, s_out are read once at create time (folded into su, sv).  The handle
 *     owns its folded scales and scratch memory.
 *   - Streams: `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Every compute call is asynchronous on that stream; create and
 *     destroy synchronise.
 *   - Errors: every call returns an escha_status_t; nothing is thrown across the
 *     ABI.  Argument errors are detected on the host before any launch.
 *     Asynchronous CUDA errors surface as ESCHA_ERR_CUDA on a later call.  A
 *     device-side wait that exceeds its time limit sets the handle's error flag;
 *     escha_linear_check() reports it as ESCHA_ERR_TIMEOUT.
 *   - Shapes: in and out must be multiples of 128; bits in {2,3,4}; cb == 1;
 *     tile == 16.  Anything else is ESCHA_ERR_UNSUPPORTED.
 *   - No CPU fallback exists: without a usable sm_103a device every compute call
 *     fails with ESCHA_ERR_CUDA.
 *   - Debugging: with ESCHA_SYNC_DEBUG=1 in the environment (read at the first
 *     call) every gemv/gemm/moe call and stage synchronises its stream after
 *     launching and reports an asynchronous CUDA error at that call.
 */
#ifndef ESCHA_H
#define ESCHA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ESCHA_OK = 0,
  ESCHA_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size, bad handle */
  ESCHA_ERR_UNSUPPORTED = 2,  /* well-formed but outside what is implemented */
  ESCHA_ERR_CUDA = 3,         /* a CUDA runtime call failed */
  ESCHA_ERR_OOM = 4,          /* device allocation failed */
  ESCHA_ERR_TIMEOUT = 5       /* a bounded device-side wait ran out */
} escha_status_t;

typedef struct escha_linear_s* escha_linear_t;
typedef struct escha_mlp_s* escha_mlp_t;
typedef struct escha_moe_s* escha_moe_t;

/* Human-readable name of a status code (static string, never NULL). */
const char* escha_status_string(escha_status_t status);

/* Name and description of the last CUDA error this thread saw inside the
 * library ("" if none); the string stays valid until the thread's next call. */
const char* escha_last_error_string(void);

/* Library version as major*10000 + minor*100 + patch. */
int escha_version(void);

/*
 * Create a dense trellis-coded linear layer.
 *   code    int16 [in/16, out/16, 16*bits]: tile (i, j) holds
 *           W_inner[16i:16i+16, 16j:16j+16] ("Tensor mapping": escha_code / EXL3
 *           trellis; K-tile index major).
 *   rin     fp16 [in]  per-input-channel scale (EXL3 suh).
 *   rout    fp16 [out] per-output-channel scale (EXL3 svh).
 *   s_in    fp32 [in], s_out fp32 [out]: escha's extra scales (may be NULL = 1.0).
 *   config  int32 [config_len], host OR device pointer, either layout:
 *           [6] = [16, bits, cb, 1, in, out]          ("Tensor mapping")
 *           [9] = [16, K, bits, mcg, E, in, out, in_p, out_p]  (Metal page tensor
 *                 table; E must be 1, K must equal bits or 16*bits, mcg 1,
 *                 in_p == in, out_p == out).
 * The handle borrows `code`; scales are folded into owned fp32 su/sv.
 */
escha_status_t escha_linear_create(escha_linear_t* out, const int16_t* code,
                                   const uint16_t* rin, const uint16_t* rout,
                                   const float* s_in, const float* s_out,
                                   const int32_t* config, int config_len, void* stream);

escha_status_t escha_linear_destroy(escha_linear_t h);

/* Shape of a handle (any output pointer may be NULL). */
escha_status_t escha_linear_shape(escha_linear_t h, int* in_features, int* out_features, int* bits);

/*
 * Decode the whole W_inner into fp16 [in, out] (test and inspection entry).
 * Uses the same device decode routine as the GEMV and GEMM kernels.
 * Source: "Bit layout" (stream, windows, lane L holds symbols 8L..8L+7) and the
 * tile packing paragraph of the Metal page (closed-form permutation inverse).
 */
escha_status_t escha_linear_decode(escha_linear_t h, uint16_t* w_inner, void* stream);

/*
 * Decode-time layer: y[M, out] = had(had(x * su) @ W_inner) * sv for 1 <= M <= 16.
 *   x  fp16 [M, in];  y  fp16 [M, out] (may not alias x).
 * Fused decode-and-multiply: the codes stream from HBM once; weights are decoded
 * in registers and never written anywhere.  Source: Metal page, activation-side
 * reconstruction (xh = had(x*su); y_pre = xh @ W; y = had(y_pre)*sv).
 */
escha_status_t escha_linear_gemv(escha_linear_t h, const uint16_t* x, uint16_t* y, int M,
                                 void* stream);

/*
 * Prefill layer for any M >= 1: the same function as escha_linear_gemv, computed
 * with tiles decoded into shared memory feeding tcgen05 fp16 MMAs (fp32 TMEM
 * accumulators) and the output rotation fused into the epilogue.
 * The handle keeps a workspace for the rotated activations; it grows on demand
 * (a call with a larger M than any before allocates).  escha_linear_reserve()
 * sizes it up front.  Tiles that the kernel's even split shares between CTAs
 * are finished by the last CTA to reach them, summing the CTAs' partial sums
 * in CTA order, so repeated calls give the same bits; each call clears the
 * handle's arrival counters for this with a cudaMemsetAsync on `stream`
 * (capturable in a CUDA graph).  Calls that share a handle must be ordered.
 */
escha_status_t escha_linear_gemm(escha_linear_t h, const uint16_t* x, uint16_t* y, int M,
                                 void* stream);
escha_status_t escha_linear_reserve(escha_linear_t h, int max_m);

/*
 * FP8 prefill, for handles with ESCHA_ROUND_E4M3 (else ESCHA_ERR_UNSUPPORTED).
 * The EXLR8 format page notes that weights rounded to E4M3 are exact FP8
 * values, so prefill can multiply them on FP8 tensor cores; it leaves the
 * activation side open.  Here each token's rotated activations
 * xh = fp16(had(x * su)) are quantised per token as escha_quantize_e4m3_rows
 * describes (codes q, scale d), and
 *     y = fp16( had( d * (q @ W_inner) ) * sv )
 * with tcgen05 kind::f8f6f4 MMAs (E4M3 x E4M3, fp32 TMEM accumulators).  The
 * result differs from escha_linear_gemm's by the activation rounding (up to
 * 2^-4 relative per activation).  x fp16 [M, in], y fp16 [M, out], M >= 1,
 * in <= 65536 (else ESCHA_ERR_UNSUPPORTED); 16-byte aligned.  Uses the same
 * workspace as escha_linear_gemm (codes in place of the rotated activations).
 */
escha_status_t escha_linear_gemm_fp8(escha_linear_t h, const uint16_t* x, uint16_t* y, int M,
                                     void* stream);

/*
 * The FP8 prefill's contraction on activations the caller has quantised:
 *     y = fp16( had( d * (q @ W_inner) ) * sv )
 * q uint8 [M, in]: E4M3 bit patterns of the rotated activations (for example
 * from escha_quantize_e4m3_rows); d fp32 [M]: their per-row scales.  Device
 * pointers, q and y 16-byte aligned, d 4-byte aligned; M >= 1.  Same handle
 * requirement (ESCHA_ROUND_E4M3) and workspace as escha_linear_gemm_fp8.
 */
escha_status_t escha_linear_gemm_fp8_codes(escha_linear_t h, const uint8_t* q, const float* d,
                                           uint16_t* y, int M, void* stream);

/*
 * Per-token FP8 E4M3 quantisation of fp16 activations, the FP8 prefill's
 * activation step on its own (a reading of the EXLR8 format page, which leaves
 * it open).  For each row m of xh:
 *     amax = max_k |xh[m, k]|,  inv = 448 / amax,  d[m] = amax / 448
 *     q[m, k] = E4M3( xh[m, k] * inv )    nearest even, saturating at 448
 * with both quotients and the product rounded to fp32 (IEEE, nearest); a row
 * of zeros gives q = 0 and d = 0.  xh fp16 [M, K], q uint8 [M, K] (E4M3 bit
 * patterns), d fp32 [M]; all device pointers, 16-byte aligned, owned by the
 * caller.  K a multiple of 128 with 128 <= K <= 65536, M >= 1, else
 * ESCHA_ERR_INVALID_ARG.  Asynchronous on `stream`.
 */
escha_status_t escha_quantize_e4m3_rows(const uint16_t* xh, uint8_t* q, float* d, int M, int K,
                                        void* stream);

/*
 * Gated MLP at decode: y = down( silu(gate(x)) * up(x) ), each matrix a dense
 * trellis layer with its own rin/rout/s_in/s_out.  gate and up map in -> inter,
 * down maps inter -> in.  The three handles are borrowed.  1 <= M <= 16.
 * Source: model layout in the Qwen3.8-27B ANE notes, section 1 (MLP 5120->17408);
 * each matrix is the activation-side layer above.
 */
escha_status_t escha_mlp_create(escha_mlp_t* out, escha_linear_t gate, escha_linear_t up,
                                escha_linear_t down);
escha_status_t escha_mlp_destroy(escha_mlp_t m);
escha_status_t escha_mlp_gemv(escha_mlp_t m, const uint16_t* x, uint16_t* y, int M, void* stream);

/*
 * Input RMSNorm of a gated MLP ("Escha-W2 runs on Metal", model-loading
 * paragraph): after this call escha_mlp_gemv computes
 *     n = x / sqrt(mean(x^2) + eps) * w,   y = down( silu(gate(n)) * up(n) )
 * per token, the norm fused into the input rotations (one launch per call, as
 * before).  norm_w: DEVICE fp16 [in], the weight as stored; escha keeps
 * its RMSNorm weights minus one, so with stored_minus_one != 0 the weight
 * applied is norm_w + 1 (the gated norms inside a linear-attention block carry
 * no offset: pass 0).  norm_w is read during this call only (folded with the
 * gate and up input scales); eps in [0, 1).  norm_w = NULL removes the norm.
 * Synchronises the device.
 */
escha_status_t escha_mlp_set_input_norm(escha_mlp_t m, const uint16_t* norm_w, float eps,
                                        int stored_minus_one);

/*
 * Routed-expert layer (EXLR8 page, "The sharing trick" and the GLM-5.3 expert
 * shapes): E experts, each with gate/up [hidden -> inter] and down [inter ->
 * hidden] trellis matrices at its own width bits[e] in {2,3,4}.  The hidden side
 * is shared by all experts: gate/up use one su_hidden = rin_hidden * s_in_hidden
 * and down uses one sv_hidden = rout_hidden * s_out_hidden, so a token is rotated
 * once and one rotated activation serves every routed expert.  The intermediate
 * side is per expert.
 *   gate_code/up_code/down_code: HOST arrays [E] of DEVICE pointers to each
 *     expert's int16 code tensor ([hidden/16, inter/16, 16*b] and
 *     [inter/16, hidden/16, 16*b]).  Borrowed.
 *   bits: HOST int32 [E].
 *   rin_hidden fp16 [hidden], s_in_hidden fp32 [hidden] (NULL = 1.0)
 *   rout_gate, rout_up fp16 [E, inter]; s_out_gate, s_out_up fp32 [E, inter]
 *   rin_down fp16 [E, inter]; s_in_down fp32 [E, inter]
 *   rout_hidden fp16 [hidden]; s_out_hidden fp32 [hidden]
 */
escha_status_t escha_moe_create(escha_moe_t* out, int num_experts, int hidden, int inter,
                                const int16_t* const* gate_code, const int16_t* const* up_code,
                                const int16_t* const* down_code, const int32_t* bits,
                                const uint16_t* rin_hidden, const float* s_in_hidden,
                                const uint16_t* rout_gate, const float* s_out_gate,
                                const uint16_t* rout_up, const float* s_out_up,
                                const uint16_t* rin_down, const float* s_in_down,
                                const uint16_t* rout_hidden, const float* s_out_hidden,
                                void* stream);

/*
 * Routed-expert layer stored by halves (EXLR8 page, manifest paragraph): each
 * expert matrix is split into H = inter/128 halves of 128 intermediate
 * channels.  Gate and up are split along their output channels and each half
 * has its own width; down is split along its input channels and has one width
 * per expert.  The kernels read a device table of half pointers, ptr[e][h], in
 * place of one pointer per matrix, fetching it anew on every launch.  Everything else (shared
 * hidden-side rotation, side vectors, the call escha_linear_moe_gemv and its
 * stages, rounding, check) is as for escha_moe_create.
 *   gate_half, up_half  DEVICE arrays [E * H] of device pointers: entry
 *       e*H + h is the code of output channels 128h .. 128h+127 of expert e's
 *       gate (up) matrix, int16 [hidden/16, 8, 16*b] with b = gate_bits[e*H + h]
 *       (up_bits[e*H + h]) -- the tiles of those 128 columns in the layout of
 *       escha_moe_create's code tensors.
 *   down_half  DEVICE array [E * H] of device pointers: entry e*H + h is the
 *       code of input channels 128h .. 128h+127 of expert e's down matrix,
 *       int16 [8, hidden/16, 16*b] with b = down_bits[e].
 *   gate_bits, up_bits  DEVICE int32 [E * H]; down_bits DEVICE int32 [E].
 *   Side vectors: as for escha_moe_create.
 * The six tables are borrowed, not copied: each call's routing kernel reads
 * the entries of the experts it routes to, so the caller may point halves at
 * other code or change widths between calls (not while a call that uses them
 * is in flight on the GPU) without creating a new handle.  The tables must be
 * 8-byte (pointers) and 4-byte (widths) aligned.  An entry that is null, not
 * 16-byte aligned, or a width outside {2,3,4} is replaced by a zero code of
 * width 2 and sets the handle's error flag: escha_moe_check then reports
 * ESCHA_ERR_INVALID_ARG and that call's output is not meaningful.
 */
escha_status_t escha_moe_create_halves(escha_moe_t* out, int num_experts, int hidden, int inter,
                                       const int16_t* const* gate_half,
                                       const int16_t* const* up_half,
                                       const int16_t* const* down_half, const int32_t* gate_bits,
                                       const int32_t* up_bits, const int32_t* down_bits,
                                       const uint16_t* rin_hidden, const float* s_in_hidden,
                                       const uint16_t* rout_gate, const float* s_out_gate,
                                       const uint16_t* rout_up, const float* s_out_up,
                                       const uint16_t* rin_down, const float* s_in_down,
                                       const uint16_t* rout_hidden, const float* s_out_hidden,
                                       void* stream);
escha_status_t escha_moe_destroy(escha_moe_t m);

/*
 * Shared expert of a routed-expert layer (EXLR8 page, "The sharing trick": the
 * hidden-side rotation is shared by all routed experts and the shared
 * expert).  After this call escha_linear_moe_gemv adds, for every token, the
 * shared expert's down(silu(gate(x)) * up(x)) with weight 1 to the weighted
 * sum of its routed experts.  The shared expert has the routed experts'
 * shapes and uses the layer's hidden-side vectors; its intermediate side is
 * its own.  gate_code, up_code [hidden/16, inter/16, 16*bits], down_code
 * [inter/16, hidden/16, 16*bits]: DEVICE, borrowed; rout_gate, rout_up,
 * rin_down fp16 [inter]; s_out_gate, s_out_up, s_in_down fp32 [inter] (may be
 * NULL = 1.0), read during this call.  gate_code = NULL removes the shared
 * expert.  Handles from escha_moe_create only (ESCHA_ERR_UNSUPPORTED for
 * experts stored by halves).  Synchronises the device.
 */
escha_status_t escha_moe_set_shared_expert(escha_moe_t m, const int16_t* gate_code,
                                           const int16_t* up_code, const int16_t* down_code,
                                           int bits, const uint16_t* rout_gate,
                                           const float* s_out_gate, const uint16_t* rout_up,
                                           const float* s_out_up, const uint16_t* rin_down,
                                           const float* s_in_down);

/*
 * y[m] = sum_k expert_w[m,k] * down_e( silu(gate_e(x[m])) * up_e(x[m]) ),
 * e = expert_ids[m,k].  1 <= M <= 8, 1 <= topk <= 8; ids in [0, E) and distinct
 * within a token (duplicates are summed, out-of-range ids are skipped and set
 * the handle's error flag).
 *   x fp16 [M, hidden]; expert_ids int32 [M, topk]; expert_w fp32 [M, topk];
 *   y fp16 [M, hidden].  All device pointers; routing is read on the device.
 */
escha_status_t escha_linear_moe_gemv(escha_moe_t m, const uint16_t* x, const int32_t* expert_ids,
                                     const float* expert_w, uint16_t* y, int M, int topk,
                                     void* stream);

/*
 * One stage of a decode-time call, for timing and inspecting the stages one by
 * one.  Each takes the arguments of its full call (validated the same way)
 * plus `stage`; running stages 0 .. N-1 in order on one stream with the same
 * arguments is exactly the full call.  Intermediate results stay in the
 * handle's own device buffers, so the stages of one pass must not interleave
 * with another call on the same handle.
 *   linear (ESCHA_LINEAR_STAGES = 3): 0 input rotation xh = had(x * su);
 *     1 trellis decode-and-multiply into fp32 partial sums; 2 output rotation
 *     y = had(sum of partials) * sv.
 *   mlp (ESCHA_MLP_STAGES = 5): 0 input rotation (shared by gate and up);
 *     1 gate and up contraction (one launch); 2 output rotations of gate and
 *     up, silu(gate) * up, input rotation of down; 3 down contraction;
 *     4 output rotation of down.
 *   moe (ESCHA_MOE_STAGES = 5): 0 routing plan (reads expert_ids) and, in
 *     the same launch, the input rotation (shared hidden side); 1 gate and up
 *     contraction of the routed experts; 2 their output rotations,
 *     silu(gate) * up and the input rotation of down; 3 down contraction;
 *     4 output rotation, weighted sum over the routed experts (reads
 *     expert_w).
 * Stage numbers outside [0, N) return ESCHA_ERR_INVALID_ARG.
 */
#define ESCHA_LINEAR_STAGES 3
#define ESCHA_MLP_STAGES 5
#define ESCHA_MOE_STAGES 5
escha_status_t escha_linear_gemv_stage(escha_linear_t h, int stage, const uint16_t* x,
                                       uint16_t* y, int M, void* stream);
escha_status_t escha_mlp_gemv_stage(escha_mlp_t m, int stage, const uint16_t* x, uint16_t* y,
                                    int M, void* stream);
escha_status_t escha_linear_moe_gemv_stage(escha_moe_t m, int stage, const uint16_t* x,
                                           const int32_t* expert_ids, const float* expert_w,
                                           uint16_t* y, int M, int topk, void* stream);

/*
 * Codebook rounding of a handle's weights.  ESCHA_ROUND_FP16 (default): each
 * weight is the codebook's fp16 value.  ESCHA_ROUND_E4M3: the EXLR8 variant
 * (EXLR8 format page, the E4M3 rounding inside the Viterbi search): the fp16
 * value is rounded to the nearest FP8 E4M3 value, ties to even, magnitudes
 * past 448 clamped to 448.
 * Applies to every later decode, GEMV and GEMM of the handle (MoE: every
 * routed expert).  Synchronises the device.  A gated MLP takes each matrix's
 * rounding when it is created.  Other values: ESCHA_ERR_INVALID_ARG.
 */
#define ESCHA_ROUND_FP16 0
#define ESCHA_ROUND_E4M3 1
escha_status_t escha_linear_set_rounding(escha_linear_t h, int rounding);
escha_status_t escha_moe_set_rounding(escha_moe_t m, int rounding);

/*
 * Synchronise `stream` and report the handle's device error flag:
 * ESCHA_ERR_TIMEOUT if a bounded wait in one of its kernels ran out,
 * ESCHA_ERR_INVALID_ARG if routing ids were out of range, ESCHA_ERR_CUDA on an
 * asynchronous CUDA error, else ESCHA_OK.  The flag is cleared by the read.
 * A gated MLP has a flag of its own for its launches; its three layers keep
 * theirs (read them with escha_linear_check).
 */
escha_status_t escha_linear_check(escha_linear_t h, void* stream);
escha_status_t escha_mlp_check(escha_mlp_t m, void* stream);
escha_status_t escha_moe_check(escha_moe_t m, void* stream);

/*
 * Per-kernel timing of the trellis contraction launches (the dominant kernel).
 * When enabled on a handle, every trellis GEMV/GEMM launch made for it is
 * bracketed by CUDA events on the launching stream (inside stream capture the
 * events become graph nodes that fire on every replay).  collect() synchronises
 * those events and returns the summed milliseconds and the number of launches
 * since the previous collect(), then resets.  kind selects the handle type.
 */
escha_status_t escha_profile_enable(void* handle, int kind, int on);
escha_status_t escha_profile_collect(void* handle, int kind, double* ms_total, int* launches);
#define ESCHA_KIND_LINEAR 0
#define ESCHA_KIND_MLP 1
#define ESCHA_KIND_MOE 2

/*
 * Allocation-free dense layer at decode.  The source pages have no counterpart:
 * this entry point is for callers that must not allocate device memory, such as
 * runtimes that reserve all device memory for their own pool up front, or code
 * running where a cudaMalloc would synchronise the device or is not allowed.
 * It computes the same y[M, out] = had(had(x * su) @ W_inner) * sv as
 * escha_linear_gemv, with the same kernels, but takes the layer's tensors
 * directly (no handle, no create) and allocates nothing: its scratch (folded
 * scales, rotated activations, partial sums) lives in one fixed device array
 * of ESCHA_NOALLOC_SCRATCH_BYTES that every GPU loading the library holds
 * until the process exits.
 *   code, rin, rout, s_in, s_out: as for escha_linear_create (device pointers;
 *     s_in / s_out may be NULL = 1.0); in_features, out_features multiples of
 *     128; bits in {2,3,4}; x fp16 [M, in], y fp16 [M, out]; 1 <= M <= 16.
 * Returns ESCHA_ERR_UNSUPPORTED, before launching anything, when the layer
 * needs more scratch than the fixed array holds (folded scales 4*(in+out)
 * bytes, rotated activations 64*in bytes and fp32 partial sums 64*out bytes
 * per partial-sum slot, plus 512 bytes).  The first call on a device looks up
 * the array's device address; make that first call before any stream capture.
 * Every call reuses the same array: calls whose work overlaps on the GPU (on
 * other streams or from other host threads) race and must be ordered by the
 * caller.  The call is asynchronous on `stream` and returns argument and
 * launch errors.  There is no handle whose error flag could be read later, so
 * if a bounded device wait of the GEMV runs out, the call writes fp16 NaN to
 * every element of y; with ESCHA_SYNC_DEBUG=1 it also synchronises `stream`
 * and returns ESCHA_ERR_TIMEOUT (or ESCHA_ERR_CUDA for an asynchronous error).
 */
#define ESCHA_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
escha_status_t escha_linear_gemv_noalloc(const int16_t* code, const uint16_t* rin,
                                         const uint16_t* rout, const float* s_in,
                                         const float* s_out, int in_features, int out_features,
                                         int bits, const uint16_t* x, uint16_t* y, int M,
                                         void* stream);

/*
 * Trellis encoder: the code of W_inner [in, out] (fp32, device), written to
 * code int16 [in/16, out/16, 16*bits] in the layout escha_linear_create takes.
 * Each 16x16 tile is encoded on its own by a Viterbi search over the 2^16
 * trellis states that minimises the tile's squared error between W_inner and
 * the decoded weights (EXLR8 format page, "Viterbi search"; with rounding ==
 * ESCHA_ROUND_E4M3 the search uses the E4M3-rounded codebook values).  The
 * stream is circular, so the path must be tail-biting (the first window
 * continues the last; Metal page, windows at offset i*K): a first pass searches
 * with a free start, a second pass fixes the 16-bits bits that the last window
 * shares with the first (taken from the first pass's best end state) and
 * returns the best path that agrees with them.  Costs are fp32 with every
 * difference, square and sum rounded on its own; ties go to the lowest state.
 *   w       fp32 [in, out] row-major, device.
 *   code    int16 [in/16, out/16, 16*bits], device, written.
 *   sq_err  fp32 [in/16 * out/16], device, may be NULL: each tile's squared
 *           error (the path cost) in tile order.
 * in_features, out_features: positive multiples of 16; bits in {2,3,4};
 * rounding ESCHA_ROUND_FP16 or ESCHA_ROUND_E4M3.  The call allocates its
 * scratch (256 * 2^(16-bits) bytes per SM used) stream-ordered on `stream` and
 * frees it there; it is asynchronous like every compute call.
 */
escha_status_t escha_trellis_encode(const float* w, int in_features, int out_features, int bits,
                                    int rounding, int16_t* code, float* sq_err, void* stream);

/*
 * Self-test of the bounded device wait: launches one block that waits on an
 * mbarrier no one arrives at, with a limit of `limit_us` microseconds (1..1e6).
 * Returns ESCHA_ERR_TIMEOUT when the kernel gave up and reported it (the expected
 * outcome), ESCHA_OK if the wait unexpectedly completed.  The context stays usable.
 */
escha_status_t escha_selftest_wait_timeout(int limit_us, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* ESCHA_H */
