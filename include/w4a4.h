/*
 * w4a4.h -- C ABI of libw4a4.so: the prompt-processing (prefill) matmul of a
 * Hadamard-rotated Q4_0 model run as W4A4, on one NVIDIA GB300 (sm_103a).
 *
 * The method is the one described on the engine docs page "The lean option:
 * ROCmFP4, ROCmI4 and Hadamard Q4_0", section "Hadamard-rotated Q4_0: W4A4
 * prompt processing":
 *   - weights are plain Q4_0 (one fp16 scale per 32 values along K, 4-bit codes
 *     q standing for q - 8), made once from weights rotated per 32-element block
 *     along K by a normalised 32-point Walsh-Hadamard transform H32;
 *   - activations get the same per-block rotation at run time and are rounded
 *     to 4 bits per block (int4 codes, one scale per block);
 *   - each output is  Y[m][n] = sum_b d_w[n][b] * d_a[m][b] * P[m][n][b],
 *     P[m][n][b] = sum_{j<32} (q_w - 8) * q_a  (an exact integer, |P| <= 2048).
 * Section "MoE: W4A4 on the experts" applies the same product to the routed
 * expert matmuls (MUL_MAT_ID).  The engine's per-tensor rotation flag (engine
 * PR #262, "Pin ROCmFPX fc664ba: Hadamard rotation per tensor ...") is kept as
 * a per-operand tag: a rotated operand is never multiplied with an unrotated
 * one (the silently-wrong mixed case the PR's review warns about is refused).
 *
 * Conventions for every entry point:
 *   - Ownership: the caller allocates every buffer.  Pointers named "device"
 *     are CUDA device (or managed) memory of the current device; nothing is
 *     retained after the call returns.  The library allocates no memory and
 *     keeps no per-call global state.
 *   - Streams: all GPU work is enqueued on `stream` (a cudaStream_t; 0 is the
 *     legacy default stream) and is asynchronous with respect to the host;
 *     outputs are valid once the stream reaches that point.
 *   - Errors: arguments are checked before anything is launched; a failed
 *     check returns a status (never aborts, never throws) and records a message
 *     for w4a4_last_error() (thread-local).  A launch failure returns
 *     W4A4_ERR_CUDA with the CUDA error text.  Data errors found on the device
 *     (expert ids out of range) are reported through a device flag, see
 *     w4a4_gemm_id / w4a4_gemm_id_status.
 *   - Sizes: K is a positive multiple of 32 (the block size); B = K / 32.
 *     Row counts may be 0 (nothing is launched, W4A4_OK).
 *   - Alignment: every device pointer must be 16-byte aligned and every row
 *     stride must keep rows 16-byte aligned, else W4A4_ERR_ALIGNMENT.
 *   - Domain: inputs are finite; a nonzero block whose largest magnitude is
 *     below 2^-100 is outside the domain (its reciprocal scale overflows).
 */
#ifndef W4A4_H
#define W4A4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t, declared without the CUDA headers. */
typedef struct CUstream_st* w4a4_stream_t;

typedef enum {
  W4A4_OK = 0,
  W4A4_ERR_INVALID_ARG = 1,  /* bad size, null pointer, bad enum value          */
  W4A4_ERR_ALIGNMENT = 2,    /* pointer or row stride not 16-byte aligned        */
  W4A4_ERR_MISMATCH = 3,     /* operand tags disagree (rotated vs unrotated, K)  */
  W4A4_ERR_UNSUPPORTED = 4,  /* valid request this build does not handle         */
  W4A4_ERR_CUDA = 5,         /* a CUDA call or kernel launch failed              */
  W4A4_ERR_DEVICE_FLAG = 6,  /* the device reported bad data (see gemm_id)       */
  W4A4_ERR_WORKSPACE = 7,    /* workspace missing or smaller than required       */
  W4A4_ERR_TIMEOUT = 8       /* a bounded wait inside a kernel gave up           */
} w4a4_status;

/* Operand tags: a magic in the high half, flags in the low half. */
#define W4A4_TAG_Q4_0 0x51340000u    /* Q4_0 weights                          */
#define W4A4_TAG_ACT4 0x41340000u    /* int4 activations                      */
#define W4A4_TAG_ACT8 0x41380000u    /* int8 activations (the exact path)     */
#define W4A4_TAG_ACT16 0x41420000u   /* bf16 activations (rotate-only route)  */
#define W4A4_TAG_MAGIC_MASK 0xFFFF0000u
#define W4A4_TAG_ROTATED 0x00000001u /* values were rotated by H32 per block  */

/* Weight input element types for h32_q4_0_pack_weights. */
#define W4A4_DTYPE_BF16 0
#define W4A4_DTYPE_F32 1

/*
 * Q4_0 weights, structure of arrays (rows = output features N, or E*N for
 * stacked experts):
 *   codes : device, [rows][K/2] bytes.  Block b of row r is the 16 bytes at
 *           codes + r*K/2 + 16*b; byte i holds code q_i in its low nibble and
 *           q_{i+16} in its high nibble (the Q4_0 block order); code q stands
 *           for the integer q - 8.
 *   scales: device, [rows][K/32] IEEE fp16 (binary16 bits), the block scale d.
 *   sums  : device, [rows][K/32] int16, the block's code sum sum_j (q_j - 8).
 *           Derived data (no extra information): written by h32_q4_0_pack_weights
 *           and q4_0_import from the codes, read by the GEMMs.
 *   expanded: device, [round_up(rows, 8)][K] bytes, or NULL.  Optional derived
 *           data: byte k of row r is q_k - 8 as an fp8 e4m3 value times 2^9
 *           (sign and magnitude: q - 8 >= 0 -> q - 8, else 0x80 | (8 - q)), in
 *           element order; the pad rows are zero.  When the packers or the
 *           import get it they fill it; w4a4_gemm then loads the weights straight
 *           into the tensor-core operand layout instead of converting the codes
 *           in every tile.  Twice the codes' memory (w4a4_q4_0_expanded_bytes).
 */
typedef struct {
  uint8_t* codes;
  uint16_t* scales;
  int16_t* sums;
  int64_t rows;
  int64_t K;
  uint32_t tag; /* W4A4_TAG_Q4_0 | (W4A4_TAG_ROTATED if rotated) */
  uint8_t* expanded;
} w4a4_q4_0;

/*
 * int4 activations, structure of arrays:
 *   codes : device, [rows][K/2] bytes, same nibble order as Q4_0; each nibble is
 *           a 4-bit two's complement integer in -8..7.
 *   scales: device, [rows][K/32] fp32, the block scale d_a.
 *   expanded: device, [round_up(rows, 8)][K] bytes, or NULL.  Optional derived
 *           data: byte k of row r is the offset code a_k + 8 (0..15), which is
 *           also the fp8 e4m3 value (a_k + 8) * 2^-9, in element order.  When
 *           w4a4_rotate_quantize_act gets it, it fills rows 0..rows-1 (the pad
 *           rows are never read into a result and are left as they are);
 *           w4a4_gemm, given expanded weights as well, then loads both operands
 *           straight into the tensor-core layout and converts nothing.  Twice the
 *           codes' memory (w4a4_act4_expanded_bytes).  The other entry points
 *           ignore it.
 */
typedef struct {
  uint8_t* codes;
  float* scales;
  int64_t rows;
  int64_t K;
  uint32_t tag; /* W4A4_TAG_ACT4 | (W4A4_TAG_ROTATED if rotated) */
  uint8_t* expanded;
} w4a4_act4;

/*
 * int8 activations of the exact path, per 32-element block along K (section
 * "Hadamard-rotated Q4_0: W4A4 prompt processing": with W4A4 off, a rotated
 * file runs on the exact int8 path):
 *   codes : device, [rows][K] int8 in element order, each in -127..127.
 *   scales: device, [rows][K/32] fp32, the block scale d_a = amax / 127.
 */
typedef struct {
  int8_t* codes;
  float* scales;
  int64_t rows;
  int64_t K;
  uint32_t tag; /* W4A4_TAG_ACT8 | (W4A4_TAG_ROTATED if rotated) */
} w4a4_act8;

/*
 * Activations of the rotate-only route (section "Hadamard-rotated Q4_0: W4A4
 * prompt processing": the same rotated files also run with the activations
 * rotated and not rounded to 4 bits):
 *   values: device, [rows][K] bf16 (bit patterns) in element order: the rotated
 *           fp32 values rounded to nearest even.  No scales.
 */
typedef struct {
  uint16_t* values;
  int64_t rows;
  int64_t K;
  uint32_t tag; /* W4A4_TAG_ACT16 | (W4A4_TAG_ROTATED if rotated) */
} w4a4_act16;

/* Bytes needed for the two arrays of a Q4_0 / int4 operand (0 if K is invalid). */
size_t w4a4_q4_0_codes_bytes(int64_t rows, int64_t K);
size_t w4a4_q4_0_scales_bytes(int64_t rows, int64_t K);
size_t w4a4_q4_0_sums_bytes(int64_t rows, int64_t K);
size_t w4a4_q4_0_expanded_bytes(int64_t rows, int64_t K);
size_t w4a4_act4_codes_bytes(int64_t rows, int64_t K);
size_t w4a4_act4_scales_bytes(int64_t rows, int64_t K);
size_t w4a4_act4_expanded_bytes(int64_t rows, int64_t K);
size_t w4a4_act8_codes_bytes(int64_t rows, int64_t K);
size_t w4a4_act8_scales_bytes(int64_t rows, int64_t K);
size_t w4a4_act16_values_bytes(int64_t rows, int64_t K);

/*
 * h32_q4_0_pack_weights -- rotate weights per 32-block along K and quantise to
 * Q4_0 (engine docs "The lean option ...", section "Hadamard-rotated Q4_0: W4A4
 * prompt processing": the same rotation applied to the weights once, then plain
 * Q4_0; section "MoE: W4A4 on the experts": one scale per 32 values).
 *   w      : device, [N][ldw] elements of type w_dtype (row n holds W[n][0..K-1]).
 *   rotate : 1 = apply H32 (normalised) before quantising; 0 = plain Q4_0.
 *   out    : host struct; out->codes, out->scales and out->sums must point to
 *            caller buffers of w4a4_q4_0_codes_bytes / _scales_bytes /
 *            _sums_bytes; rows, K and tag are written by this call.
 * Per block: y = H32 w / sqrt(32) (fp32 butterfly, stages 1,2,4,8,16, then one
 * multiply by fl32(1/sqrt 32)); m = the y of largest magnitude (lowest index on
 * ties); d = m / -8; q = clamp(round_half_away(y * (1/d)) + 8, 0, 15) (q = 8
 * when d = 0); stored scale = fp16(d), round to nearest even.
 */
w4a4_status h32_q4_0_pack_weights(const void* w, int w_dtype, int64_t N, int64_t K, int64_t ldw,
                                  int rotate, w4a4_q4_0* out, w4a4_stream_t stream);

/*
 * h32_q4_0_pack_weights_imatrix -- as h32_q4_0_pack_weights, with the block
 * scales chosen against an importance vector (the converter's imatrix
 * quantisation, section "Hadamard-rotated Q4_0: W4A4 prompt processing": the
 * tensors are quantised with the imatrix given the change matching the
 * rotation).
 *   imatrix : device, K fp32 importances of the (unrotated) input channels, or
 *             NULL for uniform importance; 16-byte aligned.  Negative or
 *             non-finite entries count as 0, a block of zeros as uniform.
 *             With rotate = 1 the importance of the rotated channels is
 *             diag(Hn diag(imp) Hn^T) (Hn = H32/sqrt 32 per block): the block
 *             mean, flat across the block.
 *   Per block (values y, weights om): d minimises sum om (y - d c)^2 with each
 *   c the nearest integer to y/d in -8..7 (every interval where the nearest
 *   codes are fixed is tried); the stored fp16 scale is the best of fp16(m/-8),
 *   fp16(d) and its two fp16 neighbours by that weighted error, with the codes
 *   q = clamp(round_half_away(y * fl32(1/d16)) + 8, 0, 15).  Layout, tags and
 *   errors as h32_q4_0_pack_weights.  Runs once per model: about 10^5 fp32
 *   operations per block.
 */
w4a4_status h32_q4_0_pack_weights_imatrix(const void* w, int w_dtype, int64_t N, int64_t K, int64_t ldw, int rotate,
                                          const float* imatrix, w4a4_q4_0* out, w4a4_stream_t stream);

/*
 * q4_0_import -- take existing Q4_0 weights bit for bit (section "Hadamard-
 * rotated Q4_0: W4A4 prompt processing": the kernel reads plain Q4_0 weights
 * bit for bit).
 *   blocks : device, [N][K/32] canonical 18-byte Q4_0 blocks (little-endian fp16
 *            scale, then 16 code bytes), 2-byte aligned.
 *   rotated: 1 if the file's weights were rotated by H32 (the stamped files of
 *            the page), 0 for plain Q4_0.
 *   out    : as for h32_q4_0_pack_weights.
 */
w4a4_status q4_0_import(const void* blocks, int64_t N, int64_t K, int rotated, w4a4_q4_0* out,
                        w4a4_stream_t stream);

/*
 * w4a4_rotate_quantize_act -- rotate activations per 32-block along K and
 * round them to int4 per block (section "Hadamard-rotated Q4_0: W4A4 prompt
 * processing": only the activations are rounded to 4 bits, after the same
 * rotation).
 *   x      : device, fp32 [M][ldx] (row m holds X[m][0..K-1]).
 *   rotate : 1 = rotate (for rotated weights); 0 = quantise unrotated values.
 *   out    : host struct; out->codes / out->scales point to caller buffers of
 *            w4a4_act4_codes_bytes / _scales_bytes; rows, K, tag are written.
 *            out->expanded: NULL, or a 16-byte aligned buffer of
 *            w4a4_act4_expanded_bytes, which then also receives the offset
 *            codes a + 8 of rows 0..M-1 (see w4a4_act4).
 * Per block: y as for the weights; a = max |y|; d_a = a / 7 (fp32, stored);
 * q = clamp(round_half_away(y * (1/d_a)), -8, 7) (q = 0 when d_a = 0).
 */
w4a4_status w4a4_rotate_quantize_act(const float* x, int64_t M, int64_t K, int64_t ldx, int rotate,
                                     w4a4_act4* out, w4a4_stream_t stream);

/*
 * w4a4_gemm -- Y = the block-scaled W4A4 product (MUL_MAT), section
 * "Hadamard-rotated Q4_0: W4A4 prompt processing".
 *   w   : Q4_0 weights, rows = N.       a : int4 activations, rows = M.
 *   y   : device, fp32 [M][ldy], ldy >= N, 4-byte aligned (the one exception to
 *         the 16-byte rule); Y[m][n] = sum_b d_w d_a P (fp32).
 * w->K must equal a->K and both tags must agree on rotation, else
 * W4A4_ERR_MISMATCH.  The per-block integer partials are exact on the tensor
 * cores; the scale fold is fp32.  When a->expanded is set, the super-tile kernel
 * loads it instead of converting the activation codes, and reads w->expanded,
 * if set, instead of converting the weight codes (same result, bit for bit); an
 * expanded buffer must then hold the expanded form of the same codes.  Without
 * a->expanded, a kernel that converts both operands' codes runs.
 *   ws  : optional device workspace (NULL, or w4a4_gemm_workspace_bytes(M, N,
 *         K) bytes or more, 16-byte aligned, all zero before its first use).
 *         Its first MiB holds arrival counters that every call leaves at zero
 *         again (CUDA-graph replays included), so one workspace serves any
 *         sequence of shapes; after W4A4_ERR_TIMEOUT, zero it before reuse.  With it, shapes whose
 *         tiles would leave SMs idle in the last wave run a stream-K schedule:
 *         the K work of all tiles is split evenly over the SMs and a tile cut
 *         between CTAs is summed in a fixed order, so the result does not depend
 *         on timing.  Without it (or when the size query returns 0) each CTA
 *         takes whole tiles.  A smaller non-NULL ws is W4A4_ERR_WORKSPACE.
 *         Calls that share a workspace must not overlap on the GPU.
 */
w4a4_status w4a4_gemm(const w4a4_q4_0* w, const w4a4_act4* a, float* y, int64_t ldy, void* ws,
                      size_t ws_bytes, w4a4_stream_t stream);

/* Workspace bytes for w4a4_gemm at this shape on the current device; 0 when the
 * whole-tile schedule is used (no workspace needed). */
size_t w4a4_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K);

/*
 * w4a4_gemm_small_m -- w4a4_gemm for batches of 1 to 8 tokens (a drafter's
 * verification batch; the engine docs page above keeps a row-tiled Q4_0 kernel
 * for 8-column verification batches, each weight unpacked once for all columns).
 * A weight-streaming CUDA-core kernel; its output is bit for bit that of
 * w4a4_gemm without a workspace (the whole-tile schedule).  Arguments, layouts
 * and errors as w4a4_gemm; a->rows > 8 is W4A4_ERR_UNSUPPORTED.
 */
w4a4_status w4a4_gemm_small_m(const w4a4_q4_0* w, const w4a4_act4* a, float* y, int64_t ldy,
                              w4a4_stream_t stream);

/*
 * The exact path: rotated Q4_0 weights times int8 activations (section
 * "Hadamard-rotated Q4_0: W4A4 prompt processing" compares W4A4 with it, about
 * 400 against 509 tok/s on the pages' hardware).
 *
 * w4a8_rotate_quantize_act -- as w4a4_rotate_quantize_act, with 8-bit codes:
 *   per block, y as there; a = max |y|; d_a = a / 127 (fp32, stored);
 *   q = clamp(round_half_away(y * (1/d_a)), -127, 127) (q = 0 when d_a = 0).
 *   out->codes / out->scales are caller buffers of w4a4_act8_codes_bytes /
 *   _scales_bytes; rows, K and tag are written.
 *
 * w4a8_gemm -- Y[m][n] = sum_b d_w d_a P with P = sum_j (q_w - 8) q_a exact;
 *   arguments, layout, workspace and errors as w4a4_gemm (its workspace size
 *   from w4a8_gemm_workspace_bytes).  The integer products run as f16
 *   tensor-core MMAs, in which every int4 and int8 value and every 32-term
 *   block sum is exact.
 *
 * w4a8_gemm_partials -- the exact P[m][n][b] (int32 [M][N][K/32]), |P| <= 32512.
 */
w4a4_status w4a8_rotate_quantize_act(const float* x, int64_t M, int64_t K, int64_t ldx, int rotate,
                                     w4a4_act8* out, w4a4_stream_t stream);
w4a4_status w4a8_gemm(const w4a4_q4_0* w, const w4a4_act8* a, float* y, int64_t ldy, void* ws,
                      size_t ws_bytes, w4a4_stream_t stream);
w4a4_status w4a8_gemm_partials(const w4a4_q4_0* w, const w4a4_act8* a, int32_t* P, w4a4_stream_t stream);
size_t w4a8_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K);

/*
 * The rotate-only route (section "Hadamard-rotated Q4_0: W4A4 prompt
 * processing": on the backend without W4A4, the rotated files run with the
 * activations rotated as a matmul and not rounded to 4 bits).  This build
 * carries the rotated activations as bf16, the tensor cores' 16-bit type.
 *
 * w4a16_rotate_act -- per 32-element block of each row of x (fp32, device,
 *   [M][ldx]): y = fl32(FWHT32(x_blk) * c) as in w4a4_rotate_quantize_act
 *   (rotate = 1) or y = x_blk (rotate = 0), stored as bf16 (round to nearest
 *   even) in out->values, a caller buffer of w4a4_act16_values_bytes(M, K)
 *   bytes; rows, K and tag are written.  Errors as w4a4_rotate_quantize_act.
 *
 * w4a16_gemm -- Y[m][n] = sum_b d_w[n][b] * sum_j y[m][32b+j] * (q_w - 8):
 *   bf16 tensor-core MMAs (every q - 8 is exact in bf16) with fp32 block sums,
 *   folded by the fp16 weight scale in fp32.  Arguments, layout, workspace
 *   (size from w4a16_gemm_workspace_bytes) and errors as w4a4_gemm; the
 *   rotation tags of w and a must agree (W4A4_ERR_MISMATCH otherwise).
 */
w4a4_status w4a16_rotate_act(const float* x, int64_t M, int64_t K, int64_t ldx, int rotate, w4a4_act16* out,
                             w4a4_stream_t stream);
w4a4_status w4a16_gemm(const w4a4_q4_0* w, const w4a4_act16* a, float* y, int64_t ldy, void* ws, size_t ws_bytes,
                       w4a4_stream_t stream);
size_t w4a16_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K);

/*
 * w4a4_gemm_partials -- the exact per-block integer dot products
 * P[m][n][b] = sum_j (q_w - 8) q_a (int32, device [M][N][K/32]), computed by the
 * same tensor-core main loop as w4a4_gemm.  For verification.
 */
w4a4_status w4a4_gemm_partials(const w4a4_q4_0* w, const w4a4_act4* a, int32_t* P,
                               w4a4_stream_t stream);

/*
 * w4a4_gemm_id -- the expert-routed product (MUL_MAT_ID), section "MoE: W4A4 on
 * the experts": token t's slot s uses expert e = ids[t][s].
 *   experts : Q4_0 weights of all experts stacked along rows, rows = E * N;
 *             expert e owns rows e*N .. e*N+N-1.
 *   a       : int4 activations; rows = M (act_per_slot = 0: one row per token,
 *             the gate/up projections) or M * top_k (act_per_slot = 1: row
 *             t*top_k + s per token-slot, the down projection).
 *   ids     : device, int32 [M][top_k].
 *   y       : device, fp32 [M][top_k][N] (row t*top_k + s), contiguous,
 *             4-byte aligned.
 *   ws      : device workspace of at least w4a4_gemm_id_workspace_bytes(M,
 *             top_k, E, K) bytes (sized on the current device), 16-byte aligned;
 *             its contents on entry do not matter.  It holds the routing
 *             (counts, offsets, pair list), the routed activation rows gathered
 *             in expert order, a device error flag (its first word), and the
 *             slots of the GEMM's stream-K schedule: the (tile x K-stage) units
 *             of all routed tiles are cut into one equal range per SM, and a
 *             tile cut between CTAs is summed in CTA order (a fixed order: the
 *             result does not depend on timing).
 * An id outside [0, E) is not used: its output row is zeroed, the device flag in
 * ws is set, and w4a4_gemm_id_status() on the same ws returns
 * W4A4_ERR_DEVICE_FLAG.  Each call clears the flag first.
 */
w4a4_status w4a4_gemm_id(const w4a4_q4_0* experts, int E, int64_t N, const w4a4_act4* a,
                         const int32_t* ids, int64_t M, int top_k, int act_per_slot, float* y,
                         void* ws, size_t ws_bytes, w4a4_stream_t stream);

size_t w4a4_gemm_id_workspace_bytes(int64_t M, int top_k, int E, int64_t K);

/*
 * w4a4_gemm_id_status -- synchronise `stream`, then read the device flag that
 * the last w4a4_gemm_id on `ws` left: W4A4_OK, or W4A4_ERR_DEVICE_FLAG if some
 * id was out of range (or W4A4_ERR_CUDA).
 */
w4a4_status w4a4_gemm_id_status(const void* ws, w4a4_stream_t stream);

/*
 * w4a4_gemm_id_static -- w4a4_gemm_id without a caller workspace.  The pages
 * describe no such call: it is an interface convenience of this library.
 *
 * Some callers cannot hand device memory to an op at the call site.  One case
 * is an op plugged into a host engine whose callback passes only its tensors:
 * the engine owns every buffer, and no allocator is in reach.  Another is a
 * step loop that must not call cudaMalloc/cudaFree, which can synchronise the
 * device and whose cost varies from call to call.  For them this entry point
 * keeps the routing scratch in a fixed device array inside the library,
 * W4A4_GEMM_ID_STATIC_SCRATCH_BYTES bytes per device.  It makes no allocation
 * of its own, through CUDA or any other library.
 *
 * Arguments, layouts and results are those of w4a4_gemm_id without ws and
 * ws_bytes.  The output is the same as w4a4_gemm_id's on the same inputs.
 *   - Size limit: a problem with w4a4_gemm_id_workspace_bytes(M, top_k, E, K)
 *     greater than W4A4_GEMM_ID_STATIC_SCRATCH_BYTES is refused with
 *     W4A4_ERR_WORKSPACE before anything runs; use w4a4_gemm_id for it.  (The
 *     MoE workload of 1024 tokens, top-8, K 2048 on 152 SMs needs about 49 MiB,
 *     most of it the stream-K slots.)
 *   - Set-up: the first call on a device, with that device current, looks up
 *     the array's device address once (cudaGetSymbolAddress) and keeps it.
 *     Make that first call before any stream capture.
 *   - Starting state: nothing in the array needs to be zero on entry.  Each
 *     call's first kernel writes every count, offset, pair index and flag that
 *     the later kernels read.
 *   - Concurrency: one array serves all calls on a device.  Two calls whose
 *     kernels can overlap on the GPU race on it and give wrong results.  This
 *     includes calls on different streams, or from different host threads,
 *     without an ordering between them.  Calls ordered on one stream are safe.
 *   - Bad ids: an id outside [0, E) zeroes its output row as in w4a4_gemm_id.
 *     The flag that records it stays inside the library, so no status query
 *     reports it.  Callers that need the check use w4a4_gemm_id.
 */
#define W4A4_GEMM_ID_STATIC_SCRATCH_BYTES ((size_t)64 << 20)

w4a4_status w4a4_gemm_id_static(const w4a4_q4_0* experts, int E, int64_t N, const w4a4_act4* a,
                                const int32_t* ids, int64_t M, int top_k, int act_per_slot, float* y,
                                w4a4_stream_t stream);

/*
 * w4a4_check -- synchronise `stream`, then report whether any GEMM kernel run
 * since the last check gave up on one of its bounded internal waits (a pipeline
 * that stopped making progress for a second).  Such a kernel stops early, so
 * its output is incomplete: W4A4_ERR_TIMEOUT.  Clears the condition.  Returns
 * W4A4_ERR_CUDA for an error already pending on the stream.
 *
 * The library caches, per device, the addresses of its device-side state (this
 * error word, the static routing scratch of w4a4_gemm_id_static) and each
 * kernel's launch attributes.  cudaDeviceReset invalidates them: a process that
 * resets a device must not call the library on that device again.
 */
w4a4_status w4a4_check(w4a4_stream_t stream);

/*
 * w4a4_debug_set_wait_limit -- a test hook for the bounded waits.  Later launches
 * of the super-tile GEMM kernel (w4a4_gemm with the expanded activation operand,
 * and w4a4_gemm_id) give up on a pipeline wait after wait_ns nanoseconds instead
 * of one second, and their producer holds its first copy back for
 * producer_delay_ns.  With a delay longer than the limit every CTA gives up: the
 * kernel returns by itself, with its output incomplete, and w4a4_check reports
 * W4A4_ERR_TIMEOUT.  (0, 0) restores the defaults.  Not synchronised with other
 * host threads; for tests only.  The wind-down waits (copies in flight, MMAs in
 * flight before TMEM is released) keep their one-second bound.
 */
void w4a4_debug_set_wait_limit(uint64_t wait_ns, uint64_t producer_delay_ns);

/* The message of the last failed call on this thread ("" if none). */
const char* w4a4_last_error(void);
/* A fixed name for a status value. */
const char* w4a4_status_name(w4a4_status s);
/* ABI version of this library (major * 100 + minor).  2.00: w4a4_act4 gained the
 * `expanded` field (a layout change; callers built against 1.xx must rebuild). */
int w4a4_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* W4A4_H */
