/*
 * moe4.h -- C ABI of libmoe4.so: the 4-bit MoE expert-layer numerics on B300 (sm_103a).
 *
 * The method (described in prose on the pages cited below) quantises the forward operands of the
 * expert layers to NVFP4, picking each block's scale by Four Over Six, multiplies them in a
 * block-scaled grouped expert GEMM, requantises the transposed forward operands to MXFP8 with
 * stochastic rounding for the backward GEMMs, and encodes expert outputs for the return path
 * with a Hadamard transform before quantisation.
 *
 * Pages:
 *   [DEBUT] "Inkling 2 Small's Native 4-Bit Training: Debut and Doubts" (agihunt.info),
 *           "Confirmed": NVFP4 forward of the expert layers with dedicated kernels, MXFP8
 *           backward with requantisation and stochastic rounding, Four Over Six, per-expert
 *           scales.
 *   [LHC]   "4-bit computation from the start of Inkling 2 Small's pretraining" (lhc.media):
 *           fewer-bits paragraph (4-bit values, one scale per sixteen, 4.5 bits/value);
 *           backward-pass paragraphs (dequantise, transpose at higher precision, requantise to
 *           MXFP8 with stochastic rounding); communication paragraph (NVFP4 dispatch, Hadamard
 *           transform before the return path is quantised); the paragraph on in-house kernels
 *           that fuse the transform and quantisation into the matrix multiplication.
 *   [4WEEK] "Thinking Machines: Nvidia FP4 Up to 6x Faster, Runs Gain 8%" (fourweekmba.com):
 *           model-card update (48 layers, 8 of 384 experts per token), "What Thinking Machines
 *           Changed" (NVFP4 expert forward with a dedicated kernel, MXFP8 backward).
 *
 * Conventions for every call:
 *   - Every pointer argument is a DEVICE pointer owned by the caller, unless a comment says
 *     "host".  No call allocates device memory (no cudaMalloc) or frees what it is given; the
 *     library's own device data is static and exists from the moment it is loaded: the status
 *     word of moe4_get_status and the 16 KiB scratch array of nvfp4_quantize_noalloc.
 *     Calls that need scratch take (ws, ws_bytes); moe4_workspace_size() gives the size.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).  Every call
 *     only enqueues work on it and returns; nothing is synchronised unless a comment says so.
 *   - bf16 values are passed as their uint16_t bit patterns; E2M1, E4M3 and E8M0 values as raw
 *     bytes.  Matrices are row-major with their contraction / blocking dimension contiguous.
 *   - NVFP4 tensor [R, C]: codes uint8 [R, C/2] (element 2j in the low nibble, 2j+1 in the high
 *     nibble), sf uint8 E4M3 [R, C/16] ("canonical" layout), and one float per-tensor decode
 *     scale g_dec (per matrix; per expert for weights).
 *   - MXFP8 tensor [R, C]: q uint8 E4M3 [R, C], e8 uint8 E8M0 [R, C/32] (canonical layout).
 *   - Return value: MOE4_OK, or a negative status.  After MOE4_ERR_ARG or MOE4_ERR_WORKSPACE
 *     nothing has been enqueued; after MOE4_ERR_CUDA part of the call's work may have been.
 *     Argument checks cover null pointers, sizes, divisibility and 16-byte alignment of every
 *     vector-accessed buffer.  NaN and infinite inputs are not checked and give unspecified
 *     codes.  Index arrays that live in device memory (group_offs, row_of, src_of) are read
 *     only by the kernels and are not checked: entries outside the ranges a call documents give
 *     undefined results, including reads out of bounds (moe4_permute_plan produces valid ones).
 */
#ifndef MOE4_H
#define MOE4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------------ status codes */
#define MOE4_OK               0
#define MOE4_ERR_ARG        (-1) /* null pointer, bad size, misaligned buffer, bad flag */
#define MOE4_ERR_UNSUPPORTED (-2) /* a valid request the library does not implement */
#define MOE4_ERR_CUDA       (-3) /* a CUDA call or kernel launch failed */
#define MOE4_ERR_TIMEOUT    (-4) /* a device-side wait gave up (reported by moe4_get_status) */
#define MOE4_ERR_WORKSPACE  (-5) /* ws is NULL or smaller than moe4_workspace_size() */

/* ------------------------------------------------------------------ flags */
#define MOE4_FOUR_OVER_SIX  0x00001u /* NVFP4: per block choose scale amax->6 or amax->4 */
#define MOE4_AMAX_GIVEN     0x00002u /* NVFP4: use amax_in instead of computing the amax */
#define MOE4_SR             0x00004u /* MXFP8: stochastic rounding (else nearest-even) */
#define MOE4_ROWWISE        0x00010u /* MXFP8 quantise: blocks along the rows' contiguous dim */
#define MOE4_COLWISE        0x00020u /* MXFP8 quantise: the transpose, blocks along rows */
#define MOE4_OUT_F32        0x00100u /* output binary32 */
#define MOE4_OUT_BF16       0x00200u /* output bf16 */
#define MOE4_GROUP_M        0x01000u /* grouped GEMM: groups are row ranges of A and D */
#define MOE4_GROUP_K        0x02000u /* grouped GEMM: groups are ranges of the contraction */
#define MOE4_ACCUMULATE     0x04000u /* grouped GEMM: D += result (binary32 output only) */
#define MOE4_SF_MMA_LAYOUT  0x10000u /* scale factors are in the tensor-core tile layout */
#define MOE4_MXFP8          0x20000u /* Hadamard codec: the 8.25-bit MXFP8 variant */
#define MOE4_SF_OUT_MMA     0x40000u /* MXFP8 producers: output scales in the tensor-core tile layout */
#define MOE4_PASS_QUANT     0x100000u /* weight path: run only its first pass (the NVFP4 quantiser) */
#define MOE4_PASS_REQUANT   0x200000u /* weight path: run only its second pass (the requantiser) */
#define MOE4_SHARE_SMS      0x400000u /* weight path: the quantiser keeps to part of each SM */

/* ------------------------------------------------------------------ library */
int moe4_version(void);                      /* e.g. 100 for 0.1.0 */
const char *moe4_status_string(int status);  /* static string, never NULL */

/* Operation ids for moe4_workspace_size(). */
#define MOE4_OP_NVFP4_QUANTIZE   1 /* a = nmat */
#define MOE4_OP_HADAMARD_QUANT   2 /* no arguments */
#define MOE4_OP_PERMUTE_PLAN     3 /* a = tokens, b = top_k, c = experts */
size_t moe4_workspace_size(int op, int64_t a, int64_t b, int64_t c);
/* Scratch for the grouped GEMMs when their scale factors come in the canonical layout:
 * kind 0 = NVFP4 (16-blocks), 1 = MXFP8 (32-blocks); a_rows x K for A, E x b_rows x K for B.
 * Kind 1 adds 16 KiB that grouped_gemm_mxfp8_wgrad_sgd uses for its tile schedule (an order of
 * the experts by group size); with less, that kernel runs its tiles in expert order. */
size_t moe4_workspace_size_gemm(int kind, int64_t a_rows, int64_t E, int64_t b_rows, int64_t K);

/* moe4_check_group_offsets: checks, on the host, group offsets the caller holds in HOST memory
 * (offs_host [E+1]) against the rules the grouped GEMMs assume of their device copy: offs[0] = 0,
 * non-decreasing, every entry a multiple of `align` (128 for the GEMMs), offs[E] = total.
 * Returns MOE4_OK or MOE4_ERR_ARG; reads nothing on the device and enqueues nothing.  The GEMMs
 * themselves do not read their offsets back to check them. */
int moe4_check_group_offsets(const int32_t *offs_host, int64_t E, int64_t total, int64_t align);

/* Synchronise `stream`, then read and clear the device status word that kernels set when a
 * bounded wait gives up.  Returns MOE4_OK or MOE4_ERR_TIMEOUT (or MOE4_ERR_CUDA). */
int moe4_get_status(void *stream);

/* moe4_selftest_wait: runs, on `stream`, one wait that nothing completes, through the same
 * bounded-wait path as the GEMM kernels: it gives up after limit_cycles SM clock cycles
 * (1 <= limit_cycles <= 2^32) and records the timeout, so that moe4_get_status then returns
 * MOE4_ERR_TIMEOUT once and the context stays usable.  A check of the failure path without a
 * fault; the pages have no counterpart. */
int moe4_selftest_wait(int64_t limit_cycles, void *stream);

/* moe4_tensor_peak_probe: the throughput ceiling of the tensor pipe for the GEMMs' instruction
 * mix.  Each of `ctas` CTAs (one per SM) keeps one operand stage in shared memory and issues
 * `iters` rounds of the grouped GEMMs' four block-scaled MMAs into one tensor-memory accumulator:
 * kind 0 = NVFP4 (mxf4nvf4, 128 x 256 x 256 per round, 2^24 FLOP), kind 1 = MXFP8 (mxf8f6f4,
 * 128 x 256 x 128 per round, 2^23 FLOP); kinds 2 and 3 are the same with each round's scale
 * factors copied into tensor memory again first (tcgen05.cp), as the GEMMs do per operand stage.
 * No operand traffic, so FLOPs / time is the pipe's own rate; time it with events on `stream`.  1 <= iters <= 2^20, 1 <= ctas <= 4096; sink [ctas]
 * uint32 (never written in practice; it keeps the result live).  A measurement aid; the pages
 * quote only datasheet peaks. */
int moe4_tensor_peak_probe(int kind, int64_t iters, int64_t ctas, uint32_t *sink, void *stream);

/* ------------------------------------------------------------------ NVFP4 [LHC fewer bits; DEBUT]
 * nvfp4_quantize: x bf16 [nmat, rows, ld] (the first `cols` of each row are used; ld >= cols,
 * ld % 8 == 0).  For each matrix m: amax_m = max|x| (or amax_in[m] with MOE4_AMAX_GIVEN);
 * g_enc = 2688/amax_m (1 if amax is 0, FLT_MAX on overflow), g_dec[m] = 1/g_enc; y = x * g_enc;
 * per 16-block along cols, candidate scales E4M3(blockamax/6) and, with MOE4_FOUR_OVER_SIX,
 * E4M3(blockamax/4); codes E2M1(y * (1/scale)) (nearest-even, saturating); the 4-candidate is
 * kept iff its pairwise-tree sum of squared errors in the y domain is strictly smaller.
 * Outputs: codes [nmat, rows, cols/2], sf [nmat, rows, cols/16] (canonical, or the tensor-core
 * tile layout of moe4_sf_to_mma_layout with MOE4_SF_MMA_LAYOUT, which needs rows % 128 == 0 and
 * cols % 64 == 0), g_dec [nmat].  cols % 16 == 0.
 * ws: moe4_workspace_size(MOE4_OP_NVFP4_QUANTIZE, nmat) bytes unless MOE4_AMAX_GIVEN.  Without
 * MOE4_AMAX_GIVEN nmat is at most 65535 (the amax pass runs one grid row per matrix); beyond
 * that MOE4_ERR_ARG, before anything is enqueued.
 * Bit-exact with the oracle: every binary32 step is one correctly rounded operation. */
int nvfp4_quantize(const uint16_t *x, int64_t nmat, int64_t rows, int64_t cols, int64_t ld,
                   uint8_t *codes, uint8_t *sf, float *g_dec, const float *amax_in,
                   uint32_t flags, void *ws, size_t ws_bytes, void *stream);

/* nvfp4_quantize_f32: the same quantiser reading binary32 x [nmat, rows, ld] (ld % 4 == 0): each
 * value is rounded to bf16 (nearest-even) as it is read, so the outputs equal those of
 * nvfp4_quantize on the bf16 copy of x, byte for byte, and amax_m is max |bf16(x)|.  For FP32
 * master weights whose bf16 copy is never stored (grouped_gemm_mxfp8_wgrad_sgd with
 * w_bf16 = NULL): 4 bytes read per value instead of 2 written and 2 read. */
int nvfp4_quantize_f32(const float *x, int64_t nmat, int64_t rows, int64_t cols, int64_t ld,
                       uint8_t *codes, uint8_t *sf, float *g_dec, const float *amax_in,
                       uint32_t flags, void *ws, size_t ws_bytes, void *stream);

/* nvfp4_quantize_noalloc: the same quantisation as nvfp4_quantize (amax computed here, flags
 * MOE4_FOUR_OVER_SIX and MOE4_SF_MMA_LAYOUT only), for callers that cannot allocate device
 * memory: a host runtime that plans all of its device memory when it starts and allows no
 * allocation afterwards, or code loaded into a process whose memory pool it cannot reach, has
 * no way to provide the `ws` buffer that nvfp4_quantize needs.  The pages describe no such
 * entry point; it is an interface convenience of this library.
 *   - Scratch: the per-matrix amax lives in a fixed array of 4096 uint32 (16 KiB) that every GPU
 *     which loads the library holds until the process exits.  nmat > 4096 returns MOE4_ERR_ARG.
 *   - Allocation: none.  The call makes no cudaMalloc or cudaFree and no allocating library call.
 *   - Every call looks up the array's device address in the current context
 *     (cudaGetSymbolAddress, which allocates nothing), so the call stays correct after the
 *     context has been torn down and created again (cudaDeviceReset moves the array).  The first
 *     call in a context also loads the library's device code there; make it before any stream
 *     capture.
 *   - Every call uses the same array and clears the part it needs first; calls whose work
 *     overlaps on the GPU (on different streams, or on different host threads) race on it. */
int nvfp4_quantize_noalloc(const uint16_t *x, int64_t nmat, int64_t rows, int64_t cols,
                           int64_t ld, uint8_t *codes, uint8_t *sf, float *g_dec, uint32_t flags,
                           void *stream);

/* nvfp4_dequantize: x_hat = (e2m1(q) * e4m3(sf)) * g_dec[m]; out [nmat, rows, cols] as bf16
 * (MOE4_OUT_BF16, nearest-even) or binary32 (MOE4_OUT_F32).  Canonical sf only. */
int nvfp4_dequantize(const uint8_t *codes, const uint8_t *sf, const float *g_dec, int64_t nmat,
                     int64_t rows, int64_t cols, void *out, uint32_t flags, void *stream);

/* ------------------------------------------------------------------ MXFP8 [LHC backward pass]
 * mxfp8_requant_transpose_sr: for each matrix m of NVFP4 [rows, cols]: dequantise to binary32,
 * transpose, and quantise each 32-block along the new contiguous dimension (rows) to MXFP8:
 * scale exponent e = smallest integer with blockamax <= 448 * 2^e, clamped to [-127, 127], stored
 * as e + 127; elements v = x_hat * 2^-e rounded to E4M3 stochastically (MOE4_SR) or to
 * nearest-even.  Stochastic rounding of the element with linear index idx in the output
 * [nmat, cols, rows] draws a 16-bit number r: half idx % 2 (0 = low) of word (idx / 2) % 4 of
 * Philox4x32-10(counter = (lo(idx/8), hi(idx/8), stream_id, 0), key = (lo(seed), hi(seed))), so one
 * call serves eight consecutive elements; the magnitude rounds up iff r < floor(frac * 2^16),
 * frac being its distance above the E4M3 value below, in units of the gap.  The probability of
 * rounding up is therefore frac less at most 2^-16: the expected result lies within 2^-16 of a
 * gap of the value, toward zero.  Outputs q_t [nmat, cols, rows], e8_t [nmat, cols, rows/32] (canonical).
 * rows % 32 == 0, cols % 32 == 0.  Input scales canonical, or in the tensor-core tile layout with
 * MOE4_SF_MMA_LAYOUT (rows % 128 == 0, cols % 64 == 0).  With MOE4_SF_OUT_MMA, e8_t is written in
 * the tensor-core tile layout of moe4_sf_to_mma_layout (as [nmat * cols, rows / 32]; rows % 128
 * == 0, cols % 128 == 0), ready for the MXFP8 GEMMs' MOE4_SF_MMA_LAYOUT.  nmat and cols / 64 at
 * most 65535 (one thread block per 128 x 64 tile on a three-dimensional grid); beyond that
 * MOE4_ERR_ARG. */
int mxfp8_requant_transpose_sr(const uint8_t *codes, const uint8_t *sf, const float *g_dec,
                               int64_t nmat, int64_t rows, int64_t cols, uint8_t *q_t,
                               uint8_t *e8_t, uint64_t seed, uint32_t stream_id, uint32_t flags,
                               void *stream);

/* nvfp4_quantize_f32_requant: the weight path of one training step over the binary32 master
 * weights x [nmat, rows, cols] (contiguous rows), in one call: nvfp4_quantize_f32 with MOE4_AMAX_GIVEN
 * (amax_in [nmat]; Four Over Six with MOE4_FOUR_OVER_SIX) writes codes [nmat, rows, cols/2], sf
 * (canonical, or the tile layout with MOE4_SF_MMA_LAYOUT) and g_dec [nmat] for the forward GEMM,
 * and mxfp8_requant_transpose_sr of that result (seed, stream_id, MOE4_SR, MOE4_SF_OUT_MMA as
 * there) writes q_t [nmat, cols, rows] and e8_t for the backward GEMM [LHC backward pass:
 * dequantise, transpose at higher precision, requantise to MXFP8 with stochastic rounding].  Every
 * output byte equals that of the two calls in sequence.  group_offs: device int32 [nmat + 1] or
 * NULL; a matrix m with group_offs[m + 1] == group_offs[m] (an expert that received no rows) is
 * skipped and its outputs are left as they are.  rows % 32 == 0 (% 128 with either tile-layout
 * flag), cols % 64 == 0 (% 128 with MOE4_SF_OUT_MMA); x, codes and q_t 16-byte aligned; nmat, and
 * cols / 64, at most 65535.
 * Split passes: MOE4_PASS_QUANT runs only the quantiser (q_t and e8_t are not touched),
 * MOE4_PASS_REQUANT only the requantiser, which reads the codes, sf and g_dec a MOE4_PASS_QUANT
 * call with the same arguments wrote (at most one of the two; neither = both passes in order).
 * mat_base (0 <= mat_base <= 2^40): the call's matrices are matrices mat_base .. mat_base + nmat - 1
 * of a larger stack, whose other arguments the caller has offset to that slice (x, amax_in, codes,
 * sf, g_dec, q_t, e8_t, group_offs); the stochastic rounding's random index of an element is its
 * index in the whole stack's q_t, so calls over slices write the bytes of one call over the stack.
 * 0 for a call over a whole stack.
 * MOE4_SHARE_SMS runs the quantiser on a small grid that holds part of each SM only, so that a
 * requantiser launched beside it on another stream (another matrix set's MOE4_PASS_REQUANT) runs
 * on the rest of every SM at the same time: the quantiser's memory waits and the requantiser's
 * arithmetic then overlap.  The outputs do not depend on these flags.  With rows == 0 the call
 * writes nothing (g_dec included) and returns MOE4_OK. */
int nvfp4_quantize_f32_requant(const float *x, int64_t nmat, int64_t rows, int64_t cols,
                               const float *amax_in, uint8_t *codes, uint8_t *sf, float *g_dec,
                               uint8_t *q_t, uint8_t *e8_t, uint64_t seed, uint32_t stream_id,
                               int64_t mat_base, const int32_t *group_offs, uint32_t flags, void *stream);

/* mxfp8_quantize: bf16 x [rows, cols] to MXFP8 with the same scale and rounding rules.
 * MOE4_ROWWISE: q [rows, cols], e8 [rows, cols/32] (cols % 32 == 0); random index = the
 * element's index in q.  MOE4_COLWISE: q [cols, rows], e8 [cols, rows/32] (rows % 32 == 0,
 * cols % 32 == 0); random index = the element's index in that transposed output.  Exactly one
 * of the two flags.  Nearest-even unless MOE4_SR. */
int mxfp8_quantize(const uint16_t *x, int64_t rows, int64_t cols, uint8_t *q, uint8_t *e8,
                   uint64_t seed, uint32_t stream_id, uint32_t flags, void *stream);

/* mxfp8_quantize_rowcol: both layouts of mxfp8_quantize from one read of x, nearest-even (the
 * backward's dY and dGU feed the rows-grouped dgrad row-wise and the contraction-grouped wgrad
 * transposed [DEBUT] confirmed list).  q_row [rows, cols], e8_row [rows, cols/32]; q_col
 * [cols, rows], e8_col [cols, rows/32]; the bytes equal those of the two single-layout calls.
 * rows % 32 == 0, cols % 32 == 0; x, q_row and q_col 16-byte aligned.  flags: 0, or
 * MOE4_SF_OUT_MMA to write both scale outputs in the tensor-core tile layout (rows % 128 == 0,
 * cols % 128 == 0). */
int mxfp8_quantize_rowcol(const uint16_t *x, int64_t rows, int64_t cols, uint8_t *q_row,
                          uint8_t *e8_row, uint8_t *q_col, uint8_t *e8_col, uint32_t flags,
                          void *stream);

/* ------------------------------------------------------------------ Hadamard codec [LHC comms]
 * hadamard_quant: x bf16 [rows, cols], cols % 128 == 0.  Each contiguous 128-chunk of a row is
 * rotated by the Sylvester-ordered Hadamard matrix (butterflies of span 1, 2, ..., 64, then
 * times RN(1/sqrt(128))) in binary32, and the rotated tensor is NVFP4-quantised as above (its
 * own amax; Four Over Six per flags).  ws: moe4_workspace_size(MOE4_OP_HADAMARD_QUANT), 4-byte
 * aligned; with MOE4_AMAX_GIVEN, ws instead holds that amax already (binary32, as
 * grouped_expert_gemm_nvfp4_hadamard_amax returns it) and the amax pass over x is skipped.
 * hadamard_dequant: NVFP4 dequantise, the same rotation (it is its own inverse), bf16 out.
 * With MOE4_MXFP8 (the only flag then), the 8.25-bit variant [LHC communication: the return path
 * falls from sixteen to 8.25 bits per value]: after the rotation each 32-block is quantised to
 * MXFP8 (E4M3 elements, E8M0 scale by the ceiling rule, nearest-even) in one pass; `codes` is
 * E4M3 [rows, cols], `sf` is E8M0 [rows, cols/32], g_dec and ws are not used (may be NULL).
 * hadamard_dequant with MOE4_MXFP8 reads that layout. */
int hadamard_quant(const uint16_t *x, int64_t rows, int64_t cols, uint8_t *codes, uint8_t *sf,
                   float *g_dec, uint32_t flags, void *ws, size_t ws_bytes, void *stream);
int hadamard_dequant(const uint8_t *codes, const uint8_t *sf, const float *g_dec, int64_t rows,
                     int64_t cols, uint16_t *out_bf16, uint32_t flags, void *stream);

/* ------------------------------------------------------------------ grouped GEMMs
 * grouped_expert_gemm_nvfp4 [DEBUT; 4WEEK: NVFP4 expert forward with a dedicated kernel]:
 * A: NVFP4 [rows_total, K] (a_codes, a_sf, a_g_dec[1]); B: E expert matrices NVFP4 [N, K]
 * (b_codes [E, N, K/2], b_sf, b_g_dec[E]).  group_offs: device int32 [E+1], non-decreasing,
 * offs[0] = 0, offs[E] = rows_total, every entry a multiple of 128.  For each expert e and row
 * i in [offs[e], offs[e+1]):  D[i, n] = a_g_dec * b_g_dec[e] * sum_k deq(A)[i,k] * deq(B_e)[n,k]
 * accumulated in binary32 by the tensor cores.  D [rows_total, N]: binary32 (MOE4_OUT_F32) or
 * bf16 (MOE4_OUT_BF16).  N % 256 == 0, K % 256 == 0.  Scale factors are canonical unless
 * MOE4_SF_MMA_LAYOUT; canonical ones are converted into ws
 * (moe4_workspace_size_gemm(0, rows_total, E, N, K) bytes). */
int grouped_expert_gemm_nvfp4(const uint8_t *a_codes, const uint8_t *a_sf, const float *a_g_dec,
                              const uint8_t *b_codes, const uint8_t *b_sf, const float *b_g_dec,
                              const int32_t *group_offs, int64_t E, int64_t rows_total, int64_t N,
                              int64_t K, void *d, uint32_t flags, void *ws, size_t ws_bytes,
                              void *stream);

/* grouped_expert_gemm_nvfp4_swiglu: the gate/up projection with the SwiGLU between the GEMMs in
 * its last stage.  B = W_gu, E matrices NVFP4 [2f, K] (gate rows 0 .. f-1, then up rows).  Writes
 * gu [rows_total, 2f] binary32, exactly grouped_expert_gemm_nvfp4's D with MOE4_OUT_F32, and
 * h [rows_total, f] bf16, h = RN_bf16(silu(g) * u) with g = gu[:, j], u = gu[:, f + j] and
 * silu(g) = g / (1 + exp(-g)), each step one binary32 rounding, exactly as moe4_swiglu_amax
 * computes it from gu; amax_out[0] = max |h| as moe4_swiglu_amax returns it.  Each tile of the
 * GEMM holds 128 gate columns and the same 128 up columns, so gu is not read back.  f % 128 == 0,
 * K % 256 == 0, rows_total % 128 == 0; gu, h 16-byte aligned; scales and ws as
 * grouped_expert_gemm_nvfp4 with N = 2f. */
int grouped_expert_gemm_nvfp4_swiglu(const uint8_t *a_codes, const uint8_t *a_sf, const float *a_g_dec,
                                     const uint8_t *b_codes, const uint8_t *b_sf, const float *b_g_dec,
                                     const int32_t *group_offs, int64_t E, int64_t rows_total, int64_t f,
                                     int64_t K, float *gu, uint16_t *h, float *amax_out, uint32_t flags,
                                     void *ws, size_t ws_bytes, void *stream);

/* grouped_expert_gemm_nvfp4_hadamard_amax: grouped_expert_gemm_nvfp4 with bf16 output d, which
 * also returns in amax_out[0] the largest magnitude of the Hadamard(128)-rotated d (each 128-column
 * chunk of a row rotated as hadamard_quant does it), computed in the GEMM's last stage from the
 * bf16 values it stores [LHC kernels paragraph: the transform and quantisation fused into the
 * final stage of the matrix multiplication].  It is exactly the amax hadamard_quant would compute
 * for d, so the return-path encoder can take it with MOE4_AMAX_GIVEN and read d once: the NVFP4
 * codec needs its per-tensor scale before the first block is quantised, so the quantisation
 * itself is a second pass.  d as for MOE4_OUT_BF16; amax_out 4-byte aligned, cleared first; flags
 * MOE4_SF_MMA_LAYOUT or 0; other rules as grouped_expert_gemm_nvfp4. */
int grouped_expert_gemm_nvfp4_hadamard_amax(const uint8_t *a_codes, const uint8_t *a_sf, const float *a_g_dec,
                                            const uint8_t *b_codes, const uint8_t *b_sf, const float *b_g_dec,
                                            const int32_t *group_offs, int64_t E, int64_t rows_total, int64_t N,
                                            int64_t K, uint16_t *d, float *amax_out, uint32_t flags, void *ws,
                                            size_t ws_bytes, void *stream);

/* grouped_expert_gemm_nvfp4_hadamard_mx: the expert GEMM above with the return-path codec fused
 * into its last stage [LHC kernels paragraph: the transform and the quantisation run in the final
 * stage of the matrix multiplication; communication paragraph: 8.25 bits per value].  The product
 * is rounded to bf16 as with MOE4_OUT_BF16, then each 128-column chunk of a row is rotated and
 * quantised exactly as hadamard_quant with MOE4_MXFP8 does: q [rows_total, N] E4M3 codes and
 * e8 [rows_total, N/32] E8M0 scales, byte for byte the result of those two calls in sequence,
 * without the bf16 tensor in memory.  Same argument rules as grouped_expert_gemm_nvfp4 (q 16-byte
 * aligned); flags: MOE4_SF_MMA_LAYOUT or 0. */
int grouped_expert_gemm_nvfp4_hadamard_mx(const uint8_t *a_codes, const uint8_t *a_sf, const float *a_g_dec,
                                          const uint8_t *b_codes, const uint8_t *b_sf, const float *b_g_dec,
                                          const int32_t *group_offs, int64_t E, int64_t rows_total, int64_t N,
                                          int64_t K, uint8_t *q, uint8_t *e8, uint32_t flags, void *ws,
                                          size_t ws_bytes, void *stream);

/* grouped_gemm_mxfp8 [DEBUT, 4WEEK: MXFP8 backward]: D = A * B^T per group, both operands MXFP8
 * with their contraction dimension contiguous.
 * MOE4_GROUP_M (dgrad): A [M, K] (q, e8), B [E, N, K]; rows offs[e]..offs[e+1] of A and D use
 *   B[e]; D [M, N]; offs[E] = M.
 * MOE4_GROUP_K (wgrad): A [M, Ktot], B [N, Ktot]; D [E, M, N] with
 *   D[e] = A[:, offs[e]:offs[e+1]] * B[:, offs[e]:offs[e+1]]^T; offs[E] = Ktot = K; an empty
 *   group writes zeros (or leaves D[e] untouched with MOE4_ACCUMULATE).
 * offs entries are multiples of 128; M % 128 == 0, N % 256 == 0, K % 128 == 0; M, E*N and K
 * below 2^31 (and E*M with MOE4_GROUP_K).  Output binary32 or bf16; MOE4_ACCUMULATE adds into a binary32 D.  Canonical scale factors are
 * converted into ws (moe4_workspace_size_gemm(1, ...)). */
int grouped_gemm_mxfp8(const uint8_t *a, const uint8_t *a_e8, const uint8_t *b,
                       const uint8_t *b_e8, const int32_t *group_offs, int64_t E, int64_t M,
                       int64_t N, int64_t K, void *d, uint32_t flags, void *ws, size_t ws_bytes,
                       void *stream);

/* grouped_gemm_mxfp8_swiglu_backward: the down projection's dgrad with the SwiGLU backward in its
 * last stage.  dH = grouped_gemm_mxfp8's rows-grouped product of A [M, K] and the experts' B [f, K]
 * (MOE4_GROUP_M, binary32), never written; instead dgu [M, 2f] bf16 receives
 * moe4_swiglu_backward(gu, dH): dg = (dh * u) * (s * (1 + g * (1 - s))), du = dh * (g * s),
 * s = 1 / (1 + exp(-g)), with g = gu[:, j], u = gu[:, f + j], each step one binary32 rounding,
 * exactly as that call computes them [LHC kernels paragraph: element-wise work fused into the
 * matrix multiplication's final stage].  gu [M, 2f] binary32 is read once.  f % 256 == 0,
 * K % 128 == 0 and > 0, M % 128 == 0; gu, dgu 16-byte aligned; scales and ws as
 * grouped_gemm_mxfp8 with N = f; flags: MOE4_SF_MMA_LAYOUT or 0. */
int grouped_gemm_mxfp8_swiglu_backward(const uint8_t *a, const uint8_t *a_e8, const uint8_t *b,
                                       const uint8_t *b_e8, const int32_t *group_offs, int64_t E, int64_t M,
                                       int64_t f, int64_t K, const float *gu, uint16_t *dgu, uint32_t flags,
                                       void *ws, size_t ws_bytes, void *stream);

/* grouped_gemm_mxfp8_wgrad_sgd: the contraction-grouped MXFP8 weight-gradient GEMM fused with
 * the FP32 master-weight update [LHC precisions: master weights in FP32; kernels paragraph:
 * fusing work into the final stage of the matrix multiplication].  For each expert e:
 * dW = A[:, offs[e]:offs[e+1]] * B[:, offs[e]:offs[e+1]]^T accumulated in binary32 (never
 * written to memory), then w32[e] <- w32[e] - lr * dW (one product, one difference, as
 * moe4_sgd_update), w_bf16[e] <- bf16(w32[e]) (nearest-even), and amax_out[e] = max |w_bf16[e]|
 * (binary32; exactly the amax the next nvfp4_quantize of w_bf16 would compute, so that call can
 * take MOE4_AMAX_GIVEN).  Bit-identical to grouped_gemm_mxfp8(MOE4_GROUP_K | MOE4_OUT_F32)
 * followed by moe4_sgd_update.  A [M, K], B [N, K], w32 / w_bf16 [E, M, N]; M % 128 == 0,
 * N % 256 == 0, K % 128 == 0; offs as for grouped_gemm_mxfp8 (offs[E] = K).  Experts with no rows
 * are skipped: under plain SGD their weights do not change, so their w32, w_bf16 and amax_out
 * entries are left as they are (amax_out[e] keeps the value an earlier call wrote).  w_bf16 may be
 * NULL: the bf16 copy is then not written and amax_out still gets max |bf16(w32[e])| (for
 * nvfp4_quantize_f32 of w32 with MOE4_AMAX_GIVEN).  flags: MOE4_SF_MMA_LAYOUT or 0 (canonical
 * scales are converted into ws, moe4_workspace_size_gemm(1, M, 1, N, K) bytes); with room in ws
 * after the staged scales for E + 1 int32 (E < 4096), the tiles run in a size-interleaved order
 * of the experts that have rows. */
int grouped_gemm_mxfp8_wgrad_sgd(const uint8_t *a, const uint8_t *a_e8, const uint8_t *b,
                                 const uint8_t *b_e8, const int32_t *group_offs, int64_t E,
                                 int64_t M, int64_t N, int64_t K, float *w32, uint16_t *w_bf16,
                                 float lr, float *amax_out, uint32_t flags, void *ws,
                                 size_t ws_bytes, void *stream);

/* moe4_sf_to_mma_layout: rearrange canonical scale factors sf [nmat, rows, nblk] into the
 * tensor-core tile layout: for each 128-row tile and each group of 4 consecutive blocks, 512
 * bytes where row r = 32*j + i of the tile puts its 4 bytes at offset 16*i + 4*j.  rows % 128
 * == 0, nblk % 4 == 0.  A pure permutation (bit-exact). */
int moe4_sf_to_mma_layout(const uint8_t *sf, int64_t nmat, int64_t rows, int64_t nblk,
                          uint8_t *out, void *stream);

/* ------------------------------------------------------------------ routing and dispatch
 * [4WEEK model card: 8 of 384 experts per token; LHC: inputs dispatched in NVFP4]
 * moe4_route_topk: logits f32 [T, E] -> idx int32 [T, k] (descending logit, ties to the lower
 * expert index) and w f32 [T, k] = softmax over the k chosen logits.  1 <= k <= 32, E <= 4096. */
int moe4_route_topk(const float *logits, int64_t T, int64_t E, int64_t k, int32_t *idx, float *w,
                    void *stream);

/* moe4_permute_plan: from idx [T, k] build offs int32 [E+1] (each expert's rows, stable in
 * (token, slot), zero-padded to a multiple of 128), row_of int32 [T, k] (dispatched row of each
 * (token, slot)) and src_of int32 [rows_cap] (source token of each dispatched row, -1 for
 * padding).  rows_cap >= T*k + 127*E, and T*k + 127*E <= 2^31 - 1 (row indices are int32).
 * ws: moe4_workspace_size(MOE4_OP_PERMUTE_PLAN, T, k, E). */
int moe4_permute_plan(const int32_t *idx, int64_t T, int64_t k, int64_t E, int32_t *offs,
                      int32_t *row_of, int32_t *src_of, int64_t rows_cap, void *ws,
                      size_t ws_bytes, void *stream);

/* moe4_permute_nvfp4: gather NVFP4 rows: out row r = input row src_of[r], or zeros (codes 0,
 * scale 0) when src_of[r] < 0; r < rows_total.  codes [T, cols/2], sf [T, cols/16] canonical;
 * cols % 32 == 0.  With MOE4_SF_MMA_LAYOUT the output scales are written in the tensor-core tile
 * layout (rows_total % 128 == 0, cols % 64 == 0).  With MOE4_MXFP8 (alone) the rows are MXFP8
 * instead: codes [T, cols] E4M3, sf [T, cols/32] E8M0, padding rows all-zero bytes — the
 * dispatch of the MXFP8 forward pass of the final layers [DEBUT] confirmed list, [4WEEK]. */
int moe4_permute_nvfp4(const uint8_t *codes, const uint8_t *sf, int64_t T, int64_t cols,
                       const int32_t *src_of, int64_t rows_total, uint8_t *out_codes,
                       uint8_t *out_sf, uint32_t flags, void *stream);

/* moe4_swiglu: gu f32 [rows, 2f] -> h bf16 [rows, f], h = g/(1+exp(-g)) * u with g the first f
 * columns and u the last f (binary32, then nearest-even to bf16).  f % 4 == 0. */
int moe4_swiglu(const float *gu, int64_t rows, int64_t f, uint16_t *h, void *stream);

/* moe4_swiglu_amax: moe4_swiglu, and amax_out[0] = max |h| over the bf16 results (binary32; 0 for
 * rows == 0), exactly the amax nvfp4_quantize would compute for h, so that call can take
 * MOE4_AMAX_GIVEN and skip its own pass over h.  amax_out 4-byte aligned; it is cleared first. */
int moe4_swiglu_amax(const float *gu, int64_t rows, int64_t f, uint16_t *h, float *amax_out, void *stream);

/* moe4_swiglu_backward: gu f32 [rows, 2f] (the forward's gate | up), dh f32 [rows, f] ->
 * dgu bf16 [rows, 2f]: dg = dh * u * s * (1 + g * (1 - s)), du = dh * g * s with
 * s = 1/(1+exp(-g)), binary32 then nearest-even to bf16.  f % 4 == 0. */
int moe4_swiglu_backward(const float *gu, const float *dh, int64_t rows, int64_t f, uint16_t *dgu,
                         void *stream);

/* moe4_swiglu_backward_mxfp8: the SwiGLU gradient fused with its MXFP8 quantisation, for the
 * backward GEMMs [LHC backward pass: MXFP8 operands; the weight gradient's SwiGLU step].  The
 * bf16 dgu of moe4_swiglu_backward (same arithmetic, same bits) is never written: its row-wise
 * MXFP8 q_row [rows, 2f], e8_row [rows, 2f/32] and its transposed MXFP8 q_col [2f, rows],
 * e8_col [2f, rows/32] are, byte for byte as mxfp8_quantize_rowcol of that dgu would give them
 * (nearest-even).  rows % 32 == 0, f % 32 == 0; gu, dh, q_row, q_col 16-byte aligned.  flags: 0,
 * or MOE4_SF_OUT_MMA (both scale outputs in the tile layout; rows % 128 == 0, f % 64 == 0). */
int moe4_swiglu_backward_mxfp8(const float *gu, const float *dh, int64_t rows, int64_t f, uint8_t *q_row,
                               uint8_t *e8_row, uint8_t *q_col, uint8_t *e8_col, uint32_t flags, void *stream);

/* moe4_combine_hadamard: the combine straight from the NVFP4-encoded return path [LHC
 * communication paragraph: the expert outputs come back Hadamard-rotated and quantised, and are
 * combined]: y[t] = sum over slots j in order of w[t,j] * yhat[row_of[t,j]], where yhat is what
 * hadamard_dequant decodes from (codes [rows, d/2], sf [rows, d/16] canonical, g_dec[0]) — the
 * bytes of hadamard_dequant followed by moe4_combine, without the decoded rows in memory (only the
 * rows a token maps to are decoded).  y bf16 [T, d]; 1 <= k <= 32; d % 128 == 0; T * d / 16 below
 * 2^32; codes and y 16-byte aligned. */
int moe4_combine_hadamard(const uint8_t *codes, const uint8_t *sf, const float *g_dec, const int32_t *row_of,
                          const float *w, int64_t T, int64_t k, int64_t d, uint16_t *y, void *stream);

/* moe4_combine_backward: the gradient of the combine with respect to the returned rows:
 * dyhat[row_of[t,j]] = bf16(w[t,j] * dy[t]) (one binary32 product per value), and zero rows for
 * padding (src_of < 0).  dy bf16 [T, d], dyhat bf16 [rows_total, d]; d % 8 == 0, k <= 32.  The
 * Hadamard return-path codec is passed straight through. */
int moe4_combine_backward(const uint16_t *dy, const int32_t *row_of, const float *w,
                          const int32_t *src_of, int64_t T, int64_t k, int64_t d,
                          int64_t rows_total, uint16_t *dyhat, void *stream);

/* moe4_combine_backward_mxfp8: the combine's gradient fused with its MXFP8 quantisation for the
 * backward GEMMs [LHC backward pass: MXFP8 operands]: the bf16 dyhat of moe4_combine_backward
 * (same arithmetic, same bits) is never written; its row-wise MXFP8 q_row [rows_total, d],
 * e8_row [rows_total, d/32] and transposed MXFP8 q_col [d, rows_total], e8_col [d, rows_total/32]
 * are, byte for byte as mxfp8_quantize_rowcol of that dyhat would give them (nearest-even).
 * d % 32 == 0, rows_total % 32 == 0; dy, q_row, q_col 16-byte aligned.  flags: 0, or
 * MOE4_SF_OUT_MMA (both scale outputs in the tile layout; rows_total % 128 == 0, d % 128 == 0). */
int moe4_combine_backward_mxfp8(const uint16_t *dy, const int32_t *row_of, const float *w, const int32_t *src_of,
                                int64_t T, int64_t k, int64_t d, int64_t rows_total, uint8_t *q_row,
                                uint8_t *e8_row, uint8_t *q_col, uint8_t *e8_col, uint32_t flags, void *stream);

/* moe4_combine: y bf16 [T, d], y[t] = sum over slots j in order of w[t,j] * yhat[row_of[t,j]]:
 * one binary32 product and one binary32 add per slot from 0, then nearest-even to bf16.
 * yhat bf16 [rows, d]; 1 <= k <= 32 (as moe4_route_topk); d % 8 == 0. */
int moe4_combine(const uint16_t *yhat, const int32_t *row_of, const float *w, int64_t T,
                 int64_t k, int64_t d, uint16_t *y, void *stream);

/* moe4_dispatch_backward: the gradient of the dispatch (the NVFP4 row gather is passed straight
 * through): dx[t] = sum over slots j in order of dxp[row_of[t,j]], one binary32 add per slot from
 * 0, then nearest-even to bf16 [LHC communication paragraph: tokens are sent to the processors of
 * their experts and the results combined; this is that send's adjoint].  dxp bf16 [rows, d], dx
 * bf16 [T, d]; 1 <= k <= 32; d % 8 == 0; dxp and dx 16-byte aligned. */
int moe4_dispatch_backward(const uint16_t *dxp, const int32_t *row_of, int64_t T, int64_t k, int64_t d,
                           uint16_t *dx, void *stream);

/* moe4_sgd_update: FP32 master weights [LHC: master weights in FP32] w32 <- w32 - lr * dw (one
 * product, one difference) and w_bf16 <- bf16(w32) (nearest-even); n % 4 == 0. */
int moe4_sgd_update(float *w32, const float *dw, int64_t n, float lr, uint16_t *w_bf16,
                    void *stream);

/* ------------------------------------------------------------------ conversions (for checks)
 * moe4_convert: the device's own conversions of binary32 in[n]: kind 0 = E2M1 code (one byte
 * per value, nearest-even, saturating, sign kept), 1 = E4M3 code (nearest-even, saturating),
 * 2 = bf16 bits (two bytes per value), 3 = E4M3 code by stochastic rounding of value i with the
 * 16-bit number of index i that moe4_sr_words(seed=0, stream_id=0) gives.  n % 4 == 0; in 16-byte
 * aligned, out 4-byte aligned (8-byte for kind 2). */
int moe4_convert(int kind, const float *in, int64_t n, void *out, void *stream);

/* moe4_sr_words: the 16-bit stochastic-rounding numbers of output indices idx_base ..
 * idx_base+n-1 (see mxfp8_requant_transpose_sr), uint16 out[n]; n % 8 == 0, idx_base % 8 == 0,
 * out 16-byte aligned. */
int moe4_sr_words(uint64_t seed, uint32_t stream_id, uint64_t idx_base, int64_t n, uint16_t *out,
                  void *stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE4_H */
