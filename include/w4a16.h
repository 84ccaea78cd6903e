/*
 * w4a16.h - C ABI of the GB300 (sm_103a) weight-only INT4 round-to-nearest
 * library: quantize/pack of bf16 weights and the W4A16 GEMM.
 *
 * The operation.  "Kernel dispatch and Humming quantization in PhyAI",
 * section "Humming makes the separation useful": weights are post-training
 * quantized at load by round-to-nearest; attention and MLP projections are
 * stored as INT4 with group size 128 while activations stay BF16 (or FP16),
 * and the quantized layers execute through a kernel that understands the
 * packed layout (a plain BF16 GEMM cannot execute it).  The method
 * specification fixes the rest: symmetric codes in [-8, 7], one fp16 scale
 * per group of 128 consecutive K values equal to fp32 absmax / 7, round half
 * to even, and scale 1 for an all-zero group.
 *
 * Data layout (all row-major, all device memory, all owned by the caller):
 *   W       [N, K]     bf16   weight to quantize (K contiguous)
 *   packed  tiles      uint8  tiled storage of the codes: row n, byte j
 *                             of the row-major [N, K/2] code array (code of
 *                             k = 2j in the low nibble, k = 2j+1 in the high
 *                             nibble, two's complement) is stored at offset
 *                             ((n / 128) * (K / 128) + j / 64) * 8192
 *                             + (n % 128) * 64 + j % 64.  Each 128 x 128
 *                             tile is one contiguous 8 KiB block; rows past N
 *                             (to the next multiple of 128) hold zeros.  Size
 *                             w4a16_packed_bytes(N, K).  The layout belongs
 *                             to this library's GEMM ("Kernel dispatch and
 *                             Humming quantization in PhyAI", section
 *                             "Humming makes the separation useful": the
 *                             packed layout is executed only by its
 *                             matching kernel).
 *   scales  [K/128, N] fp16   scale of group g of row n at scales[g * N + n]
 *   A       [M, K]     bf16   activations
 *   bias    [N]        bf16   optional
 *   Y       [M, N]     bf16   Y = bf16(A . dequant(W)^T + bias), fp32
 *                             accumulation, bias added in fp32 before the one
 *                             final rounding ("Piper Kernels", section "NVFP4
 *                             construction": scales and bias are applied in
 *                             FP32 before the final output conversion)
 *
 * Calling conventions ("Piper Kernels", section "Validation contract"):
 *   - Arguments are checked from metadata only (sizes, alignment, group):
 *     no tensor contents are read, no synchronisation, no allocation, no
 *     extra launch.  Contents are caller preconditions: finite values and
 *     |w| small enough that absmax / 7 fits fp16.  Inputs and outputs must
 *     not alias.
 *   - w4a16_quantize and w4a16_gemm are asynchronous on `stream` (a
 *     cudaStream_t; NULL = the legacy default stream) and can be captured
 *     into a CUDA graph.  They launch on the current CUDA device.
 *   - Argument errors are returned before anything is launched.  A launch
 *     failure returns W4A16_ERR_CUDA.  A kernel whose internal wait ran
 *     out of time records W4A16_ERR_TIMEOUT in a device word that
 *     w4a16_get_device_error reports.
 *   - There is no CPU fallback: every call runs on the GPU or fails.
 *
 * Shape limits: group == 128; K % 128 == 0; K >= 128; N % 8 == 0; N >= 8;
 * M >= 1; all of M, N, K < 2^31 and M*N, N*K < 2^40.  Every pointer must be
 * 16-byte aligned.
 */
#ifndef W4A16_H_
#define W4A16_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  W4A16_OK = 0,
  W4A16_ERR_INVALID_ARG = 1,  /* null pointer, size out of range          */
  W4A16_ERR_UNSUPPORTED = 2,  /* group != 128, K % 128, N % 8, bad variant */
  W4A16_ERR_ALIGNMENT = 3,    /* a pointer is not 16-byte aligned          */
  W4A16_ERR_WORKSPACE = 4,    /* workspace missing or too small            */
  W4A16_ERR_NO_VARIANT = 5,   /* no GEMM variant is usable for the shape   */
  W4A16_ERR_CUDA = 6,         /* a CUDA runtime/driver call failed         */
  W4A16_ERR_TIMEOUT = 7       /* a device-side bounded wait expired        */
} w4a16_status;

/* Human-readable name of a status code.  Never NULL. */
const char* w4a16_status_string(int status);

/* Bytes of the tiled code storage of an [N, K] weight:
 * ceil(N / 128) * 128 * K / 2. */
size_t w4a16_packed_bytes(int64_t N, int64_t K);

/* Bytes of the scale array: (K / group) * N * 2.  0 if group != 128. */
size_t w4a16_scales_bytes(int64_t N, int64_t K, int group);

/* Bytes of the row-major packed codes of an [N, K] weight: N * K / 2 (byte
 * j of row n holds the codes of k = 2j, low nibble, and k = 2j + 1, high
 * nibble, two's complement). */
size_t w4a16_packed_rowmajor_bytes(int64_t N, int64_t K);

/*
 * Row-major packed codes -> the tiled storage the GEMM reads ("Kernel
 * dispatch and Humming quantization in PhyAI", section "Humming makes the
 * separation useful": a packed INT4 layout runs only through the kernel that
 * understands it; this is the conversion from the plain interchange form,
 * e.g. codes read from a checkpoint, to this library's layout).
 * packed_rowmajor: [N, K/2] bytes as above, w4a16_packed_rowmajor_bytes(N,
 * K) (read).  packed_out: w4a16_packed_bytes(N, K) bytes (written; rows past
 * N zero).  Byte (n, j) lands at the offset given in the layout table at the
 * top of this file; nothing is decoded, so the same call serves the FP4
 * formats' nibbles.  Shape limits: K % 128 == 0, N % 8 == 0, N, K >= 1 and
 * the limits of w4a16_quantize; both pointers 16-byte aligned and not
 * overlapping.  Errors: W4A16_ERR_INVALID_ARG (null pointer, N or K < 1),
 * W4A16_ERR_UNSUPPORTED (K % 128, N % 8, size limits), W4A16_ERR_ALIGNMENT,
 * W4A16_ERR_CUDA (launch).  Allocates nothing, one kernel launch on
 * `stream`, capture-safe.
 */
int w4a16_repack_rowmajor(const void* packed_rowmajor, int64_t N, int64_t K, void* packed_out,
                          void* stream);

/*
 * RTN quantize/pack ("Kernel dispatch and Humming quantization in PhyAI",
 * section "Humming makes the separation useful": round-to-nearest at load,
 * INT4, group 128).  For each row n and group g:
 *   amax = max |W[n, k]| (fp32);  s = fp16_rn(amax / 7.0f);  s = 1 if s == 0;
 *   q = clamp(rint_even(W[n, k] / s), -8, 7)   (IEEE fp32 division)
 * writes the codes to packed_out (tiled storage, padding rows zero) and s
 * to scales_out[g * N + n].  W: [N, K] bf16 (read);  packed_out:
 * w4a16_packed_bytes(N, K) bytes;  scales_out: (K/128)*N fp16 (both
 * written).  One kernel launch on `stream`.
 */
int w4a16_quantize(const void* W_bf16, int64_t N, int64_t K, int group, void* packed_out,
                   void* scales_out, void* stream);

/*
 * Stochastic-rounding quantize/pack ("Piper Kernels", section "Stochastic
 * quantization": one of the two adjacent codes, chosen with probability
 * proportional to the distance, so the expected code is the unrounded
 * ratio; section "ConvRot INT8": the deterministic scales are kept).  Same
 * arguments, scales, storage, alignment and errors as w4a16_quantize, plus
 * an unsigned 64-bit seed.  With r = W[n, k] / s (IEEE fp32 division):
 *   if -8 <= r <= 7:  q = floor(r) + (u < r - floor(r) ? 1 : 0)
 *   else:             q = clamp(rint_even(r), -8, 7)  (never perturbed)
 * u = (word >> 8) * 2^-24 from Philox4x32-10 (Salmon et al., "Parallel
 * random numbers: as easy as 1, 2, 3"): key (seed mod 2^32, seed div 2^32),
 * counter (e div 4 as two 32-bit words, 0, 0), word e mod 4, with e = n * K
 * + k the logical element offset.  The same seed gives the same codes on
 * every launch and launch geometry.  One kernel launch on `stream`.
 */
int w4a16_quantize_sr(const void* W_bf16, int64_t N, int64_t K, int group, uint64_t seed,
                      void* packed_out, void* scales_out, void* stream);

/*
 * Workspace the GEMM needs for this shape with the variant the library's
 * table selects (split-K partial sums and per-tile arrival counters).  May
 * be 0.  The workspace must be zero-filled before its first use
 * (w4a16_workspace_init does that); every successful call leaves it
 * reusable.  One workspace must not be used by two GEMMs that can run at
 * the same time.
 */
size_t w4a16_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K);

/* Upper bound of w4a16_gemm_workspace_bytes over every variant of the
 * catalogue for this shape. */
size_t w4a16_gemm_workspace_bytes_max(int64_t M, int64_t N, int64_t K);

/* Zero `bytes` of a workspace asynchronously on `stream` (cudaMemsetAsync). */
int w4a16_workspace_init(void* workspace, size_t bytes, void* stream);

/*
 * W4A16 GEMM: Y[M, N] = bf16( A[M, K] . dequant(packed, scales)^T + bias ),
 * dequant(q, s) = q * s, fp32 accumulation on the tcgen05 tensor cores.
 * bias_bf16_or_null may be NULL.  workspace may be NULL when
 * w4a16_gemm_workspace_bytes(M, N, K) is 0.  The variant comes from the
 * library's per-shape table (w4a16_select_variant).  1 launch on `stream`.
 */
int w4a16_gemm(const void* A_bf16, int64_t M, int64_t N, int64_t K, const void* packed,
               const void* scales, int group, const void* bias_bf16_or_null, void* Y_bf16,
               void* workspace, size_t workspace_bytes, void* stream);

/*
 * W4A16 GEMM with FP16 activations ("Kernel dispatch and Humming quantization
 * in PhyAI", section "Humming makes the separation useful": activations stay
 * BF16 or FP16).  Same operation, packed codes, scales, shape limits,
 * workspace and calling conventions as w4a16_gemm, with A [M, K], bias [N]
 * and Y [M, N] in fp16: Y = fp16( A . dequant(packed, scales)^T + bias ),
 * fp32 accumulation, bias added in fp32 before the one final rounding.  The
 * weight operand enters the tensor cores as fp16 (exact integer codes with
 * the group scale applied in fp32, or fp16_rn(q * s)).
 */
int w4a16_gemm_f16(const void* A_f16, int64_t M, int64_t N, int64_t K, const void* packed,
                   const void* scales, int group, const void* bias_f16_or_null, void* Y_f16,
                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * W4A16 GEMM with a SwiGLU epilogue, for the gate/up projection of an MLP.
 * The pages fuse SwiGLU into the input preparation of the next linear, from a
 * raw [up | gate] tensor ("Piper Kernels", section "ConvRot INT8"); here it is
 * fused into the GEMM that produces that tensor, which then writes half the
 * bytes.  The weight's N rows (N even) interleave the two halves in the same
 * order: row 2f is up row f, row 2f + 1 is gate row f (a weight stored as
 * halves is interleaved once before w4a16_quantize; quantization is per row,
 * so the packed codes and scales are the interleaved ones).  bias (optional)
 * is [N] in the same interleaved order.  With y = A . dequant(packed,
 * scales)^T + bias in fp32 (as w4a16_gemm, before its rounding):
 *   Y[m, f] = bf16( silu(y[m, 2f + 1]) * y[m, 2f] ),  silu(g) = g / (1 + e^-g),
 * computed in fp32 (expf), one rounding.  Y is [M, N/2] bf16.  Shape limits,
 * packed layout, alignment and workspace rules are w4a16_gemm's; workspace
 * bytes from w4a16_gemm_swiglu_workspace_bytes.  The variant is the SwiGLU
 * table's (w4a16_tune_swiglu), else the one w4a16_select_variant gives unless
 * that is a streaming variant for M <= 16 (simt_*, rb_*) or a cluster split-K
 * variant (*_csk), whose epilogues have no SwiGLU form: then the rule's best
 * tcgen05 variant that has one.  1 launch on `stream`.
 */
int w4a16_gemm_swiglu(const void* A_bf16, int64_t M, int64_t N, int64_t K, const void* packed,
                      const void* scales, int group, const void* bias_bf16_or_null, void* Y_bf16,
                      void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes w4a16_gemm_swiglu needs for this shape (may be 0). */
size_t w4a16_gemm_swiglu_workspace_bytes(int64_t M, int64_t N, int64_t K);

/* w4a16_gemm_swiglu with an explicit variant; W4A16_ERR_UNSUPPORTED for a
 * streaming (simt_*, rb_*) or cluster split-K (*_csk) variant or a bad id,
 * W4A16_ERR_NO_VARIANT if the
 * variant cannot run the shape.  Otherwise the same contract. */
int w4a16_gemm_swiglu_variant(int variant, const void* A_bf16, int64_t M, int64_t N, int64_t K,
                              const void* packed, const void* scales, int group,
                              const void* bias_bf16_or_null, void* Y_bf16, void* workspace,
                              size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------- variants
 * The GEMM catalogue holds several kernel configurations (activation-tile
 * width, scaling mode, schedule).  The table maps a shape to one of them; it
 * is filled by measurement (w4a16_tune), in the spirit of the memoized,
 * autotuned kernel choice of "Kernel dispatch and Humming quantization in
 * PhyAI", section "Keep selection work out of repeated inference".  A shape
 * with no entry uses a fixed rule; both only ever choose GPU variants.
 * Families: tc_* the tcgen05/TMEM GEMM (group or dequant mode, whole-tile,
 * stream-K or cluster split-K (*_csk) schedules); rb_m1, rb_m2, rb_m4, rb_m8,
 * rb_m16 the row-block warp-MMA kernel for M <= 1, 2, 4, 8, 16; simt_m*_sk the CUDA-core
 * stream-K workers for M <= 1, 2, 4, 8.  None of the streaming and cluster
 * split-K variants has a SwiGLU form; the CUDA-core workers and the cluster
 * split-K variants run single problems only, the row-block kernel also
 * grouped launches (in its persistent form). */

/* Number of variants in the catalogue; ids are 0 .. count-1. */
int w4a16_variant_count(void);

/* Short name of a variant ("tc_a64_grp_sk" ...), or NULL for a bad id. */
const char* w4a16_variant_name(int variant);

/* 1 if `variant` can run this shape, else 0. */
int w4a16_variant_eligible(int variant, int64_t M, int64_t N, int64_t K);

/* Workspace bytes `variant` needs for this shape. */
size_t w4a16_variant_workspace_bytes(int variant, int64_t M, int64_t N, int64_t K);

/* The variant w4a16_gemm uses for this shape (table entry, else the rule). */
int w4a16_select_variant(int64_t M, int64_t N, int64_t K);

/* The launch the library would make for `variant` on this shape, on a GPU
 * of num_sms SMs (0: the current device's, or 152 when there is none).
 * Host-only (no launch, no device memory).  out[5] (caller-owned):
 *   out[0] grid (CTAs), out[1] whole tiles run data-parallel, out[2]
 *   stream-K (tile, unit) pairs, out[3] cluster size (CTAs of one thread-
 *   block cluster sharing a tile's or a row block's K range; 0 or 1: none),
 *   out[4] warps per team of the row-block kernel (rb_*; 0 otherwise).
 * W4A16_ERR_INVALID_ARG for a null out or a negative num_sms,
 * W4A16_ERR_NO_VARIANT if the variant cannot run the shape. */
int w4a16_variant_schedule(int variant, int64_t M, int64_t N, int64_t K, int num_sms, int* out);

/* w4a16_gemm with an explicit variant (tests, tuning).  Same contract. */
int w4a16_gemm_variant(int variant, const void* A_bf16, int64_t M, int64_t N, int64_t K,
                       const void* packed, const void* scales, int group,
                       const void* bias_bf16_or_null, void* Y_bf16, void* workspace,
                       size_t workspace_bytes, void* stream);

/* w4a16_gemm_f16 with an explicit variant.  Same contract. */
int w4a16_gemm_variant_f16(int variant, const void* A_f16, int64_t M, int64_t N, int64_t K,
                           const void* packed, const void* scales, int group,
                           const void* bias_f16_or_null, void* Y_f16, void* workspace,
                           size_t workspace_bytes, void* stream);

/*
 * Time every eligible variant on synthetic device buffers of this shape
 * and store the fastest in the table.  Allocates, synchronises and
 * launches many kernels: call it at set-up, never inside graph capture.
 * If out_variant is not NULL it receives the chosen id.
 */
int w4a16_tune(int64_t M, int64_t N, int64_t K, void* stream, int* out_variant);

/* Put an entry in the table by hand (variant must be eligible). */
int w4a16_table_set(int64_t M, int64_t N, int64_t K, int variant);

/*
 * The other catalogues are chosen by measurement the same way, each with its
 * own entries in the table ("Kernel dispatch and Humming quantization in
 * PhyAI", section "Keep selection work out of repeated inference": every
 * prepared kernel choice is tuned and memoized, not redone per call):
 *   w4a16_tune_swiglu: the INT4 variants with the SwiGLU epilogue (its best
 *     variant can differ from the plain GEMM's); w4a16_gemm_swiglu uses it;
 *   w8a16_tune: the INT8 catalogue, used by w8a16_gemm;
 *   fp4a16_tune: the FP4 catalogue, timed with `format`'s scales; one entry
 *     per shape serves both FP4 formats in fp4a16_gemm.
 * Same contract as w4a16_tune: allocates, synchronises and launches many
 * kernels (never inside graph capture); the fastest id goes to *out_variant
 * (may be NULL).  W4A16_ERR_UNSUPPORTED for shapes the catalogue cannot run
 * (SwiGLU: odd N; FP4: N % 16, unknown format).  The *_table_set calls put
 * an entry by hand (W4A16_ERR_NO_VARIANT if the variant is not eligible).
 */
int w4a16_tune_swiglu(int64_t M, int64_t N, int64_t K, void* stream, int* out_variant);
int w8a16_tune(int64_t M, int64_t N, int64_t K, void* stream, int* out_variant);
int fp4a16_tune(int format, int64_t M, int64_t N, int64_t K, void* stream, int* out_variant);
int w4a16_swiglu_table_set(int64_t M, int64_t N, int64_t K, int variant);
int w8a16_table_set(int64_t M, int64_t N, int64_t K, int variant);
int fp4a16_table_set(int64_t M, int64_t N, int64_t K, int variant);

/* Forget every table entry (all catalogues). */
void w4a16_table_clear(void);

/* Write / read the table (all catalogues) as text: lines "M N K variant"
 * for the INT4 GEMM and "swiglu|int8|fp4 M N K variant" for the others; '#'
 * starts a comment line.  W4A16_VARIANT_TABLE names a file loaded at the
 * first selection. */
int w4a16_table_save(const char* path);
int w4a16_table_load(const char* path);

/* ----------------------------------------------------------------- groups
 * Independent problems in one launch: "Kernel dispatch and Humming
 * quantization in PhyAI", section "Humming makes the separation useful",
 * quantizes the attention and MLP projections of a block (qkv, o, gate_up,
 * down); with few tokens each of those GEMMs is too small to fill the GPU
 * and pays a full launch, so the library can run a set of them together.
 * Each problem runs on its own share of the CTAs (in proportion to its
 * work); the problems must be independent: no output of one may be an input
 * or output of another. */
#define W4A16_MAX_GROUP 8

/* Epilogue of one problem of a grouped GEMM. */
#define W4A16_EPILOGUE_NONE 0    /* Y = A . dequant(W)^T + bias                 */
#define W4A16_EPILOGUE_SWIGLU 1  /* w4a16_gemm_swiglu's: the weight's rows
                                  * interleave up and gate (row 2f up f, row 2f+1
                                  * gate f); Y is [M, N/2] = silu(gate) * up in
                                  * fp32, one rounding to bf16; N even, bf16
                                  * activations only                           */

typedef struct {
  const void* A;             /* [M, K] activations (bf16; fp16 when act_f16) */
  const void* packed;        /* tiled codes of the [N, K] weight            */
  const void* scales;        /* [K/128, N] fp16                             */
  const void* bias_or_null;  /* [N], activation type, or NULL               */
  void* Y;                   /* [M, N] (or [M, N/2] for SwiGLU), act. type  */
  int64_t M, N, K;
  int epilogue;              /* W4A16_EPILOGUE_NONE (0) or _SWIGLU          */
} w4a16_gemm_problem;

typedef struct {
  const void* W_bf16;        /* [N, K] bf16 */
  int64_t N, K;
  void* packed_out;          /* w4a16_packed_bytes(N, K) bytes */
  void* scales_out;          /* (K/128) * N fp16 */
} w4a16_quantize_problem;

/* w4a16_quantize for `count` (1 .. W4A16_MAX_GROUP) weights in one launch.
 * Same per-problem contract as w4a16_quantize; argument errors of any
 * problem are returned before anything is launched. */
int w4a16_quantize_grouped(const w4a16_quantize_problem* problems, int count, int group,
                           void* stream);

/*
 * Times every candidate plan of a grouped GEMM of these shapes (each variant
 * with its per-problem schedules) as CUDA graphs of back-to-back launches on
 * synthetic operands of the same shapes, and memoizes the fastest: later
 * grouped launches of these shapes with variant -1 use it ("Kernel dispatch
 * and Humming quantization in PhyAI", section "Keep selection work out of
 * repeated inference").  Only the shapes of `problems` are read; the
 * library allocates its own operands (not capture-safe; synchronizes
 * `stream`).  *out_variant (may be NULL) receives the chosen variant.
 */
int w4a16_tune_grouped(const w4a16_gemm_problem* problems, int count, int act_f16, void* stream,
                       int* out_variant);

/* Sets the memoized plan of grouped launches of these shapes (variant -1) to
 * `variant` with its per-problem schedules, as w4a16_tune_grouped would when
 * it chose that variant (for replaying a tuned choice without timing).  Only
 * the shapes of `problems` are read. */
int w4a16_set_grouped_variant(const w4a16_gemm_problem* problems, int count, int variant);

/* Workspace the grouped GEMM needs for these problems (variant = -1: the one
 * the library chooses; else that catalogue entry).  0 if none is needed or
 * the arguments are invalid.  Same zero-once rule as w4a16_gemm. */
size_t w4a16_gemm_grouped_workspace_bytes(const w4a16_gemm_problem* problems, int count,
                                          int variant);

/* `count` (1 .. W4A16_MAX_GROUP) independent W4A16 GEMMs in one launch:
 * problem i computes Y_i = A_i . dequant(W_i)^T + bias_i as w4a16_gemm (or
 * w4a16_gemm_f16 when act_f16 != 0), or, with epilogue
 * W4A16_EPILOGUE_SWIGLU, Y_i = silu(gate) * up as w4a16_gemm_swiglu (bf16
 * only: W4A16_ERR_UNSUPPORTED with act_f16, an odd N or another epilogue
 * value), so an MLP block's gate/up projection runs in the same launch as
 * its other projections.  One variant serves the whole group (variant = -1:
 * chosen by the library; at M <= 16 without epilogues the plan may take the
 * row-block kernel, each problem on its own sub-grid).  Argument errors of
 * any problem are returned before anything is launched. */
int w4a16_gemm_grouped(const w4a16_gemm_problem* problems, int count, int group, int act_f16,
                       int variant, void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------ diagnostics */

/*
 * Synchronise `stream`, then return and clear the device error word of the
 * current device: W4A16_OK, or W4A16_ERR_TIMEOUT if a kernel's bounded wait
 * expired since the last call (that kernel's output is then undefined and a
 * workspace it used must be re-initialised).
 *
 * The library looks up device addresses of its own static device storage
 * (this error word, the scratch of w4a16_gemm_noalloc) once per device and
 * keeps them for the life of the process.  cudaDeviceReset destroys the
 * device's primary context and with it those addresses: after a reset, do
 * not call this library on that device again in the same process.
 */
int w4a16_get_device_error(void* stream);

/* Set the time a kernel-internal wait may take before it gives up and
 * records W4A16_ERR_TIMEOUT (default 2 s).  Applies to later launches. */
void w4a16_set_wait_timeout_ns(uint64_t ns);

/*
 * Declare the GEMM weights static (enable != 0) or not (0, the default), for
 * GEMM launches from now on (every w4a16_gemm* and w8a16/fp4a16 GEMM call of
 * the process, and the tuners' timings).  Static means: no kernel that can
 * run just before a GEMM launch on the same stream writes that GEMM's packed
 * codes or scales; that holds for weights quantized at load ("Kernel
 * dispatch and Humming quantization in PhyAI", section "Humming makes the
 * separation useful": post-training quantization at load), and fails for a
 * quantize launched on the stream right before the GEMM that reads its
 * output.  With static weights a GEMM launched behind another kernel
 * (programmatic dependent launch) starts copying the codes and scales of its
 * first pipeline stages before that kernel has finished; activations, bias,
 * workspace and output are still touched only after it finished.  With the
 * declaration broken the GEMM may read stale weights.  Not synchronised with
 * launches in flight: change it only between launches.
 */
void w4a16_set_weights_static(int enable);

/* The current declaration of w4a16_set_weights_static (0 or 1). */
int w4a16_weights_static(void);

/*
 * Failure-detection self test: launch one small kernel whose thread waits on
 * an mbarrier that nothing ever arrives at, with a limit of `timeout_ns`;
 * the wait runs out, the kernel records W4A16_ERR_TIMEOUT and returns.
 * Nothing faults or hangs.  Read the result with w4a16_get_device_error.
 */
int w4a16_selftest_wait_timeout(uint64_t timeout_ns, void* stream);

/*
 * Self test of the quantizer's division.  The quantize kernels compute
 * fl32(w / s) as a reciprocal product plus one remainder correction
 * (Markstein's theorem gives the correctly rounded quotient when 1 / s is
 * correctly rounded); this launch checks that code against the IEEE division
 * on the device, value by value:
 *   mode 0: every normal finite fp16 scale s and every finite bf16 w with
 *           |w| <= 7.5 s (the INT4 modes' whole domain);
 *   mode 1: the same scales, |w| <= 127.5 s (INT8);
 *   mode 2: fp32 divisors of the NVFP4 form fl32(e4m3 * g) for the 126
 *           nonzero E4M3 codes and 512 fixed tensor scales g in [2^-40,
 *           2^41), |w| <= 8 d, E2M1 codes.  No kernel uses the corrected
 *           quotient for such divisors (the NVFP4 quantize divides with
 *           IEEE division): this mode shows why, it finds codes that differ.
 * counts: device uint64[4], 8-byte aligned, caller-owned; the call zeroes it
 * on `stream`, then counts[0] = pairs checked, counts[1] = pairs whose
 * stored code differs (rint of the quotient, ties to even, for INT4 and
 * INT8; the E2M1 code in mode 2): the bit-exactness claim, counts[2] =
 * quotients that differ where |w| >= 2^-100 (the remainder is then a normal
 * float, computed exactly), counts[3] = quotients that differ anywhere (for
 * smaller |w| the remainder can underflow; with a normal fp16 scale those
 * quotients are below 2^-86 and round to code 0 either way).  +0 and -0
 * count as equal.
 * Errors: W4A16_ERR_INVALID_ARG (null), W4A16_ERR_UNSUPPORTED (mode),
 * W4A16_ERR_ALIGNMENT, W4A16_ERR_CUDA.
 */
int w4a16_selftest_quotient(int mode, unsigned long long* counts, void* stream);

/* Number of kernel launches this library has made in this process. */
uint64_t w4a16_launch_count(void);

/* Text of the last CUDA failure that made a call of this thread return
 * W4A16_ERR_CUDA ("" if none).  The library clears the CUDA runtime's
 * per-thread last error when it reports such a failure. */
const char* w4a16_last_error_detail(void);

/*
 * W4A16 GEMM without a caller-provided workspace.  The paper has no
 * counterpart: this is an addition for callers that cannot allocate device
 * memory themselves, e.g. code whose device memory is owned by another
 * allocator (a framework's caching pool or a fixed arena, where an extra
 * cudaMalloc would bypass its accounting), real-time control loops that
 * forbid allocation after start-up (cudaMalloc can synchronise the device and
 * has unbounded latency), or C callers with no workspace management.
 * Same operation and argument contract as w4a16_gemm.  The split-K scratch
 * is a 16 MiB array in static device storage of this library; every GPU that
 * loads the library holds it until the process exits.  A shape whose variant
 * needs more scratch than that returns W4A16_ERR_WORKSPACE (the reason is in
 * w4a16_last_error_detail) before anything is launched.  The first call on a
 * device looks up the array's device address (cudaGetSymbolAddress); make
 * that first call before any stream capture on that device.  Each call
 * clears the scratch's arrival counters with a cudaMemsetAsync on `stream`,
 * then launches the GEMM; it calls no cudaMalloc, cudaFree or other
 * allocating routine.  All calls on one device share that device's array, so
 * calls that can overlap on the GPU (for example on two streams) race: the
 * caller must serialise them.
 */
int w4a16_gemm_noalloc(const void* A_bf16, int64_t M, int64_t N, int64_t K, const void* packed,
                       const void* scales, int group, const void* bias_bf16_or_null, void* Y_bf16,
                       void* stream);

/* ------------------------------------------------------------------------
 * INT8 weight-only scheme (W8A16).  "Kernel dispatch and Humming
 * quantization in PhyAI", section "Choose precision by layer and hardware":
 * INT8 is one of the Humming weight schemes, with BF16 activations.  The
 * method is the INT4 one with 8-bit codes; scales, groups, alignment,
 * workspace rules and error codes are those of the INT4 calls.
 * ---------------------------------------------------------------------- */

/* Bytes of the tiled INT8 code storage: (N rounded up to 128) * K. */
size_t w8a16_packed_bytes(int64_t N, int64_t K);

/*
 * RTN INT8 quantize/pack.  For each row n and group g of 128 along K:
 *   amax = max |W[n, k]| (fp32);  s = fp16_rn(amax / 127.0f);  s = 1 if s == 0;
 *   q = clamp(rint_even(W[n, k] / s), -128, 127)   (IEEE fp32 division)
 * Codes as two's-complement bytes in tiles of 128 rows x 128 K values
 * (16 KiB, row-major inside), tile (n/128, g) at ((n/128) * K/128 + g) *
 * 16384, padding rows zero; s to scales_out[g * N + n].  W: [N, K] bf16
 * (read); packed_out: w8a16_packed_bytes(N, K) bytes; scales_out: (K/128)*N
 * fp16 (both written).  One kernel launch on `stream`.
 */
int w8a16_quantize(const void* W_bf16, int64_t N, int64_t K, int group, void* packed_out,
                   void* scales_out, void* stream);

/* Workspace the W8A16 GEMM needs for this shape (0: none). */
size_t w8a16_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K);

/*
 * Y[M, N] = bf16( A[M, K] . dequant8(W)[N, K]^T + bias[N] ), dequant8(W)[n, k]
 * = q[n, k] * s[k/128, n], accumulated in fp32, bias added in fp32; packed and
 * scales as written by w8a16_quantize; otherwise as w4a16_gemm.  The variant
 * is chosen by the library's cost model over the INT8 catalogue.
 */
int w8a16_gemm(const void* A_bf16, int64_t M, int64_t N, int64_t K, const void* packed,
               const void* scales, int group, const void* bias_bf16_or_null, void* Y_bf16,
               void* workspace, size_t workspace_bytes, void* stream);

/* The INT8 catalogue: count, names, eligibility, workspace, the rule's
 * choice (-1: none) and a forced-variant GEMM (W4A16_ERR_NO_VARIANT when the
 * variant cannot run the shape). */
int w8a16_variant_count(void);
const char* w8a16_variant_name(int variant);
int w8a16_variant_eligible(int variant, int64_t M, int64_t N, int64_t K);
size_t w8a16_variant_workspace_bytes(int variant, int64_t M, int64_t N, int64_t K);
int w8a16_select_variant(int64_t M, int64_t N, int64_t K);
int w8a16_gemm_variant(int variant, const void* A_bf16, int64_t M, int64_t N, int64_t K,
                       const void* packed, const void* scales, int group,
                       const void* bias_bf16_or_null, void* Y_bf16, void* workspace,
                       size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * FP4 weight-only schemes (MXFP4, NVFP4) with BF16 activations.  "Kernel
 * dispatch and Humming quantization in PhyAI", section "Choose precision by
 * layer and hardware": MXFP4 and NVFP4 are Humming weight schemes.  "Piper
 * Kernels", section "NVFP4 construction": NVFP4 weights use blocks of 16
 * values and a global per-tensor scale, applied with the bias in FP32 before
 * the final output conversion.
 *
 * Elements are FP4 E2M1 (sign, 2 exponent bits with bias 1, 1 mantissa bit:
 * magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6), rounded to nearest with ties to
 * the even mantissa and saturated at +-6; a value that rounds to 0 is +0.
 *   MXFP4 (OCP MX v1.0): per row and block of 32 values along K, the E8M0
 *     scale code E = floor(log2 amax) - 2 + 127 (clamped to [0, 254]; 127
 *     for an all-zero block); codes e2m1(W / 2^(E - 127)).
 *   NVFP4: g = fl32(amax(W) / 2688) (1 for an all-zero tensor); per row and
 *     block of 16, the E4M3 scale code sb = e4m3_rn_sat(fl32(fl32(amax_b /
 *     6) / g)); codes e2m1(fl32(W / fl32(sb * g))) (0 where that step is 0).
 * Codes are nibbles in the INT4 tiled layout (w4a16_quantize: byte j of a
 * row holds k = 2j low, 2j + 1 high; 128 x 128 tiles of 8 KiB); the scale
 * codes are bytes, scales_out[b * N + n] for block b of row n.  N must be a
 * multiple of 16 and K of 128.
 * ---------------------------------------------------------------------- */
#define FP4A16_MXFP4 1
#define FP4A16_NVFP4 2

/* Bytes of the packed codes (as w4a16_packed_bytes) and of the scale codes:
 * (K/32) * N (MXFP4) or (K/16) * N (NVFP4); 0 for an unknown format. */
size_t fp4a16_packed_bytes(int64_t N, int64_t K);
size_t fp4a16_scales_bytes(int format, int64_t N, int64_t K);

/*
 * FP4 quantize/pack of W: [N, K] bf16 (read).  packed_out:
 * fp4a16_packed_bytes(N, K) bytes; scales_out: fp4a16_scales_bytes bytes
 * (both written).  NVFP4 also writes tensor_scale_out[0] = g and
 * tensor_scale_out[1] = amax(W) (device fp32[2], 8-byte aligned; ignored for
 * MXFP4, may be null there).  Work on `stream`: MXFP4 one kernel; NVFP4 a
 * memset of tensor_scale_out, an absmax kernel and the quantize kernel.
 * Errors: W4A16_ERR_UNSUPPORTED (format, K % 128, N % 16),
 * W4A16_ERR_INVALID_ARG (null pointers), W4A16_ERR_ALIGNMENT.
 */
int fp4a16_quantize(int format, const void* W_bf16, int64_t N, int64_t K, void* packed_out,
                    void* scales_out, float* tensor_scale_out, void* stream);

/* Workspace the FP4 GEMM needs for this shape (0: none). */
size_t fp4a16_gemm_workspace_bytes(int format, int64_t M, int64_t N, int64_t K);

/*
 * Y[M, N] = bf16( g * (A[M, K] . D[N, K]^T) + bias[N] ), D[n, k] =
 * e2m1(code) * block scale (MXFP4: 2^(E - 127); NVFP4: the E4M3 value), the
 * products rounded to bf16 (exact for MXFP4 block exponents E in [2, 248]
 * and every NVFP4 scale), accumulated in fp32; g = tensor_scale[0] (NVFP4,
 * device fp32) or 1 (MXFP4: tensor_scale is ignored); the bias is added in
 * fp32.  packed, scales, tensor_scale as written by fp4a16_quantize; A, Y,
 * bias, workspace and errors as w4a16_gemm.  The variant is chosen by the
 * library's cost model over the FP4 catalogue.
 */
int fp4a16_gemm(int format, const void* A_bf16, int64_t M, int64_t N, int64_t K,
                const void* packed, const void* scales, const float* tensor_scale,
                const void* bias_bf16_or_null, void* Y_bf16, void* workspace,
                size_t workspace_bytes, void* stream);

/* The FP4 catalogue (one for both formats): count, names, eligibility,
 * workspace, the rule's choice (-1: none) and a forced-variant GEMM
 * (W4A16_ERR_NO_VARIANT when the variant cannot run the shape). */
int fp4a16_variant_count(void);
const char* fp4a16_variant_name(int variant);
int fp4a16_variant_eligible(int variant, int64_t M, int64_t N, int64_t K);
size_t fp4a16_variant_workspace_bytes(int variant, int64_t M, int64_t N, int64_t K);
int fp4a16_select_variant(int64_t M, int64_t N, int64_t K);
int fp4a16_gemm_variant(int variant, int format, const void* A_bf16, int64_t M, int64_t N,
                        int64_t K, const void* packed, const void* scales,
                        const float* tensor_scale, const void* bias_bf16_or_null, void* Y_bf16,
                        void* workspace, size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* W4A16_H_ */
