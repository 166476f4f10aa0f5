/*
 * nvfp4.h -- C ABI of the GB300 (sm_103a) NVFP4 block-scaled quantisation
 * library: bf16 -> NVFP4 encoding and the scale-learning STE backward.
 *
 * Conventions shared by every entry point
 * ----------------------------------------
 *  - Every pointer argument except `stream` is a DEVICE pointer owned by the
 *    caller. The library allocates nothing and never synchronises: all work is
 *    enqueued on `stream` (a cudaStream_t; NULL = the legacy default stream)
 *    and the call returns as soon as it is enqueued.
 *  - Tensors are row-major and C-contiguous. bf16 data is passed as `void*`
 *    holding IEEE bfloat16 bit patterns.
 *  - Alignment: every tensor pointer (x, codes, scales, choice, dequant,
 *    gradients) must be 16-byte aligned; fp32 scalars and scale arrays
 *    4-byte aligned.
 *  - Argument errors are returned synchronously BEFORE anything is enqueued.
 *  - Data errors (NaN/Inf inputs, unusable scales or amax values) are found
 *    by the kernels and OR-ed into `*status` (a device int32, may be NULL) as
 *    NVFP4_DEV_* bits. The caller clears it; it accumulates over calls. When a
 *    bit is set the outputs of that call are unspecified.
 *  - Empty inputs (a zero dimension) return NVFP4_OK and enqueue nothing.
 *  - NVFP4_ERR_CUDA means a launch failed; earlier work on the stream is not
 *    affected by the call.
 *
 * Number formats (End-to-End 4-Bit Training, "Low-precision formats on
 * Blackwell"; UE5M3 blog, math derivation):
 *  - element: E2M1, magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}, bit 3 = sign;
 *  - block scale: E4M3 (bias 7, max 448) or unsigned UE5M3 (bias 15, max
 *    122880, all 256 codes finite), one per 16 values;
 *  - outer scale: FP32 decode scale g = gamax / (6 * M) per slice, with
 *    M = scale_max (448, or 256 under Four-Over-Six: "Four Over Six",
 *    implementation details), g = 1 when gamax = 0.
 *  A value is reconstructed as e2m1(code) * scale(block) * g.
 */
#ifndef NVFP4_H
#define NVFP4_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define NVFP4_API __attribute__((visibility("default")))
#else
#define NVFP4_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  NVFP4_OK = 0,
  NVFP4_ERR_NULL = 1,  /* a required pointer is NULL                          */
  NVFP4_ERR_SHAPE = 2, /* negative size, a size or element count above 2^60 - 1,
                          or a blocked dim not a multiple of 16 */
  NVFP4_ERR_ALIGN = 3, /* a pointer is not aligned as required                 */
  NVFP4_ERR_ENUM = 4,  /* a configuration field is out of range                */
  NVFP4_ERR_CUDA = 6   /* a CUDA launch failed                                 */
} nvfp4_status;

/* Bits of the device status word. */
#define NVFP4_DEV_NONFINITE_INPUT 1 /* an input element is NaN or Inf        */
#define NVFP4_DEV_BAD_SCALE 2       /* s_pre not in [FLT_MIN, FLT_MAX] or a   */
                                    /* non-finite s_post                       */
#define NVFP4_DEV_BAD_AMAX 4        /* a global amax is NaN, Inf or negative  */

/* nvfp4_config.blocks */
#define NVFP4_BLOCKS_ROW 1  /* 1x16 blocks along the last dimension            */
#define NVFP4_BLOCKS_COL 2  /* 16x1 blocks along rows: the row encoding of X^T */
#define NVFP4_BLOCKS_BOTH 3 /* both encodings from one read of X               */
#define NVFP4_BLOCKS_TILE16 4 /* one scale per 16x16 tile (see nvfp4_quantize)   */
/* nvfp4_config.scale_fmt */
#define NVFP4_SCALE_E4M3 0
#define NVFP4_SCALE_UE5M3 1
/* nvfp4_config.four_over_six_rule ("Four Over Six": the three selection rules
 * evaluated; MSE is the adopted one). Sums use the fixed in-block order. */
#define NVFP4_FOS_MSE 0 /* sum of squared errors                              */
#define NVFP4_FOS_MAE 1 /* sum of absolute errors                             */
#define NVFP4_FOS_MAX 2 /* largest absolute error                             */
/* nvfp4_config.rounding */
#define NVFP4_ROUND_RNE 0 /* E2M1 round to nearest, ties to the even code    */
#define NVFP4_ROUND_SR 1  /* stochastic rounding, Philox4x32-10 bits         */

typedef struct {
  int32_t blocks;        /* NVFP4_BLOCKS_*                                     */
  int32_t scale_fmt;     /* NVFP4_SCALE_*                                      */
  int32_t rounding;      /* NVFP4_ROUND_*                                      */
  int32_t four_over_six; /* 0 or 1: per block keep the lower-error of max->6   */
                         /* and max->4 (sum of squared errors; ties keep 6)    */
  float scale_max;       /* M of the outer scale; 0 = 256 with 4/6, else 448   */
  uint32_t seed;         /* stochastic rounding key word 0                     */
  uint32_t step;         /* stochastic rounding key word 1 (training step)     */
  int32_t four_over_six_rule; /* NVFP4_FOS_*: the error the 4/6 choice compares */
} nvfp4_config;

/* Outputs of one encoding (row or column). Shapes for an input [S][R][C]:
 *   row encoding: codes [S][R][C/2], scales [S][R][C/16], dequant [S][R][C]
 *   col encoding: codes [S][C][R/2], scales [S][C][R/16], dequant [S][C][R]
 *   choice: [S][W] 32-bit words, W = ceil(R*C/16/32); bit b%32 of word b/32
 *           of slice s is block b of that slice (blocks in output order);
 *           1 = the block was encoded with its max scaled to 4.
 * codes: two E2M1 codes per byte, the even element in the low nibble.
 * scales: one scale byte per block, no swizzle. */
typedef struct {
  uint8_t* codes;   /* required                                              */
  uint8_t* scales;  /* required                                              */
  uint32_t* choice; /* required when four_over_six = 1, ignored otherwise    */
  void* dequant;    /* bf16 of code * scale * g (each product rounded to     */
                    /* fp32, then to bf16); NULL = not written               */
} nvfp4_out;

/* Global amax (End-to-End 4-Bit Training, "Low-precision formats on
 * Blackwell": the FP32 outer scale is set per tensor; UE5M3 blog: current
 * tensor scaling recomputes it every step, periodic scaling every T steps).
 * x: bf16 [slices][rows][cols]; amax: fp32 [slices], overwritten with the
 * largest |x| of each slice. A caller doing periodic scaling calls this on
 * refresh steps only and passes the same buffer to nvfp4_quantize in between.
 * Errors: NULL x/amax, negative sizes, misaligned x. */
NVFP4_API nvfp4_status nvfp4_amax(const void* x, int64_t slices, int64_t rows, int64_t cols,
                        float* amax, int32_t* status, void* stream);

/* Bytes of device workspace nvfp4_amax_ws needs for `slices` slices: two
 * 32-bit words per slice (0 for slices <= 0). */
NVFP4_API size_t nvfp4_amax_ws_bytes(int64_t slices);

/* The global amax of nvfp4_amax (same passages, same result) in ONE kernel
 * launch: nvfp4_amax zeroes amax[] with a kernel of its own before the
 * reduction's atomic max; here every CTA folds its maximum into a workspace
 * word and takes a ticket, and the CTA holding a slice's last ticket writes
 * amax[s] and returns the slice's two words to zero. No CTA waits for another.
 * x: bf16 [slices][rows][cols]; amax: fp32 [slices], overwritten.
 * workspace: device memory owned by the caller, >= nvfp4_amax_ws_bytes(slices)
 * bytes (ws_bytes), 4-byte aligned, ALL ZERO before its first use (e.g. one
 * cudaMemsetAsync when it is allocated); every call leaves it zero again. A
 * workspace serves one call at a time: calls that may run at the same time
 * (other streams) need their own workspaces.
 * Errors: those of nvfp4_amax; NVFP4_ERR_NULL for a NULL workspace,
 * NVFP4_ERR_SHAPE for ws_bytes below nvfp4_amax_ws_bytes(slices),
 * NVFP4_ERR_ALIGN for a misaligned workspace. */
NVFP4_API nvfp4_status nvfp4_amax_ws(const void* x, int64_t slices, int64_t rows, int64_t cols,
                                     float* amax, void* workspace, size_t ws_bytes,
                                     int32_t* status, void* stream);

/* The one-launch global amax for callers that cannot allocate device memory.
 * The pages have no counterpart: this entry point exists for callers that may
 * not call cudaMalloc or cudaFree, or hold no spare buffer to lend: an
 * operator hook inside another framework that hands out no workspace, a
 * serving or real-time loop that fixes all of its memory at start-up, code
 * that must not let an allocation synchronise the device. It computes what
 * nvfp4_amax_ws computes, bit for bit, taking its scratch (two 32-bit words
 * per slice) from a fixed array in the library's own device image instead of
 * a caller's workspace; it allocates nothing.
 * x: bf16 [slices][rows][cols]; amax: fp32 [slices], overwritten.
 * - At most NVFP4_AMAX_NOALLOC_MAX_SLICES (4096) slices; more returns
 *   NVFP4_ERR_SHAPE. The array (32 KiB) is held by every GPU that loads the
 *   library until the process exits.
 * - The first call on a device looks up the array's device address (with that
 *   device current) and keeps it; make that first call before any stream
 *   capture.
 * - Each call clears the words it uses (a small zeroing kernel) and then runs
 *   the amax kernel: two launches on `stream`.
 * - Every call shares the one array per device: calls that overlap on the GPU
 *   (on different streams, or from different host threads without ordering)
 *   race on it and may return wrong maxima. Order them (one stream, or events).
 * Errors: those of nvfp4_amax, plus NVFP4_ERR_SHAPE above the slice limit and
 * NVFP4_ERR_CUDA when the array's address cannot be looked up. */
#define NVFP4_AMAX_NOALLOC_MAX_SLICES 4096
NVFP4_API nvfp4_status nvfp4_amax_noalloc(const void* x, int64_t slices, int64_t rows,
                                          int64_t cols, float* amax, int32_t* status,
                                          void* stream);

/* NVFP4 quantisation of x: bf16 [slices][rows][cols] (End-to-End 4-Bit
 * Training, "Low-precision formats on Blackwell" and "Block-scaled backward
 * passes"; UE5M3 blog, math derivation and stochastic rounding; "Four Over
 * Six", method). Per block of 16: block amax, block-scale code
 * Q(amax * (1 / (k * g))) for k = 6 (and k = 4 under 4/6), element codes
 * E2M1(x * (1 / (scale * g))) by RNE or stochastic rounding, 4/6 selection,
 * packing, optional dequant.
 * global_amax: fp32 [slices], current (from nvfp4_amax) or stale (periodic).
 * row: outputs of the row encoding, required iff blocks has the ROW bit.
 * col: outputs of the column encoding, required iff blocks has the COL bit.
 * Stochastic rounding: the 16 random bits of the element at flat index idx of
 * an encoding's output layout come from Philox4x32-10 with key (seed, step),
 * counter (idx/8 low word, idx/8 high word, 0 for rows / 1 for columns, 0),
 * 16-bit half idx%2 of word (idx%8)/2; the value rounds up iff
 * bits/65536 < (|y| - lo) / (hi - lo).
 * blocks = NVFP4_BLOCKS_TILE16 (End-to-End 4-Bit Training, "Block-scaled
 * backward passes": one scale per 16x16 tile from its largest value, the same
 * when the tensor is transposed): rows % 16 == 0 and cols % 16 == 0; each
 * tile's scale is the block scale (target 6) of the tile's amax and every
 * 1x16 row block of the tile is encoded with it; `row` (required) receives
 * the row-encoding layout, every row block of a tile carrying the tile's
 * scale byte; `col` (optional) receives exactly its transpose (codes, scales,
 * dequant: the stochastic draws are the row layout's, so the two are bit for
 * bit transposes); both or neither write dequant; four_over_six must be 0
 * (NVFP4_ERR_ENUM); M defaults to 448; choice is ignored.
 * Errors: NULL required pointers, ROW with cols % 16, COL with rows % 16,
 * enum fields out of range, scale_max < 0, misaligned buffers. */
NVFP4_API nvfp4_status nvfp4_quantize(const nvfp4_config* cfg, const void* x, int64_t slices,
                            int64_t rows, int64_t cols, const float* global_amax,
                            const nvfp4_out* row, const nvfp4_out* col, int32_t* status,
                            void* stream);

/* NVFP4 quantisation with per-token outer scales (End-to-End 4-Bit Training,
 * "Recipe details": activations are quantised with one FP32 outer scale per
 * token, weights with one per expert). x: bf16 [rows][cols], cols % 16 == 0.
 * Each row r gets g_r = amax_r / (6 M) from its own amax, computed in the same
 * kernel, so x is read from HBM once. The outputs are byte for byte those of
 * nvfp4_amax + nvfp4_quantize with slices = rows and rows = 1: codes
 * [rows][cols/2], scales [rows][cols/16], dequant [rows][cols], 4/6 bitmap
 * [rows][ceil(cols/512)] words; row_amax (fp32 [rows]) receives every amax_r.
 * cfg->blocks must be NVFP4_BLOCKS_ROW. Errors: as nvfp4_quantize, plus NULL
 * row_amax. */
NVFP4_API nvfp4_status nvfp4_quantize_per_token(const nvfp4_config* cfg, const void* x,
                                                int64_t rows, int64_t cols, float* row_amax,
                                                const nvfp4_out* out, int32_t* status,
                                                void* stream);

/* Fake quantisation for scale learning (Scale Learning blog, "How Scale
 * Learning Works", first and dual-scale equations):
 *   xq = bf16(s_post * clamp(round(x * (1 / s_pre)), -6, 6))
 * with round the E2M1 RNE rounding. x, xq: bf16 [rows][cols], cols % 16 == 0;
 * s_pre, s_post: fp32 [rows][cols/16] per-block scales; s_post = NULL for a
 * single (tied) scale. Errors: NULL pointers, cols % 16, misalignment. */
NVFP4_API nvfp4_status nvfp4_fakequant_fwd(const void* x, int64_t rows, int64_t cols,
                                 const float* s_pre, const float* s_post, void* xq,
                                 int32_t* status, void* stream);

/* STE backward of nvfp4_fakequant_fwd (Scale Learning blog, "How Scale
 * Learning Works": derivative of x~ w.r.t. s, s_post and s_pre, with the
 * derivative of round taken as 1). gq = dL/dx~ (bf16 [rows][cols]).
 * With r = x * (1/s_pre), q = clamp(round(r)), in = (-6 <= r <= 6):
 *   gx      = bf16(in ? gq * a : 0), a = s_post * (1/s_pre) (dual), 1 (tied)
 *   dual:   gs_post = sum gq * q,   gs_pre = -a * sum gq * (in ? r : 0)
 *   tied:   gs_pre  = sum gq * (in ? q - r : q)      (gs_post must be NULL)
 * Block sums are fp32 in a fixed order: per half of 8, even and odd positions
 * accumulate separately with fma from +0; half = even + odd; block = half0 +
 * half1. gx may be NULL (scale-only learning). gs_pre is required; gs_post is
 * required for dual scales. Outputs: fp32 [rows][cols/16].
 * Errors: NULL pointers, cols % 16, misalignment, gs_post without s_post. */
NVFP4_API nvfp4_status nvfp4_scale_grad_bwd(const void* x, const void* gq, int64_t rows, int64_t cols,
                                  const float* s_pre, const float* s_post, void* gx,
                                  float* gs_pre, float* gs_post, int32_t* status,
                                  void* stream);

/* ---- scale learning with FP8 block scales --------------------------------
 * Scale Learning blog, "How Scale Learning Works" (the per-block scale is
 * itself quantised to FP8 and passed through with a straight-through
 * estimator; the learned post-scale is baked into the exported checkpoint)
 * and "Using Scale Learning" (MSE scale setting with an FP8 scale sweep).
 * Shared definitions: global_amax is a device fp32 [1] holding the tensor's
 * global amax; g = global_amax / (6 * 448) (1 when it is 0), rg = 1/g clamped
 * to FLT_MAX; Q8(s) = dec(E4M3_RNE(s * rg)) * g for s >= 0. x: bf16
 * [rows][cols], cols % 16 == 0; per-block arrays [rows][cols/16]. */

/* As nvfp4_fakequant_fwd, evaluated at Q8(s_pre) and Q8(s_post) (Q8(s_pre)
 * alone when s_post is NULL). NVFP4_DEV_BAD_SCALE also when s_post is
 * negative or Q8(s_pre) is below FLT_MIN; NVFP4_DEV_BAD_AMAX for a NaN, Inf or
 * negative global amax. */
NVFP4_API nvfp4_status nvfp4_fakequant_fwd_fp8scale(const void* x, int64_t rows, int64_t cols,
                                                    const float* s_pre, const float* s_post,
                                                    const float* global_amax, void* xq,
                                                    int32_t* status, void* stream);

/* As nvfp4_scale_grad_bwd, evaluated at the FP8-rounded scales; the scale
 * gradients are returned as the gradients of the unrounded scales (the
 * derivative of Q8 taken as 1). Same errors as the fp32 form plus those of
 * nvfp4_fakequant_fwd_fp8scale. */
NVFP4_API nvfp4_status nvfp4_scale_grad_bwd_fp8scale(const void* x, const void* gq, int64_t rows,
                                                     int64_t cols, const float* s_pre,
                                                     const float* s_post,
                                                     const float* global_amax, void* gx,
                                                     float* gs_pre, float* gs_post,
                                                     int32_t* status, void* stream);

/* MSE scale setting: per 1x16 block, every E4M3 scale s_c = dec(c) * g for
 * c = 1..126 is tried; the block is fake-quantised at s_c (q =
 * clamp(round(x * (1/s_c))), 1/s_c clamped to FLT_MAX) and the error
 * e = fma(-q, s_c, x) summed in the fixed block order of
 * nvfp4_scale_grad_bwd; the smallest sum wins, ties keep the smaller code.
 * (The kernel skips the codes that provably cannot win; the result is that
 * of trying every code.)
 * Outputs (either may be NULL, not both): scale_codes u8 [rows][cols/16], the
 * winning code; s fp32 [rows][cols/16], its scale dec(code) * g (an initial
 * s_pre = s_post for scale learning). Errors: NULL x / global_amax / both
 * outputs, cols % 16, misalignment. */
NVFP4_API nvfp4_status nvfp4_scale_init_mse(const void* x, int64_t rows, int64_t cols,
                                            const float* global_amax, uint8_t* scale_codes,
                                            float* s, int32_t* status, void* stream);

/* Export of learned scales to an NVFP4 row encoding: out->codes [rows][cols/2]
 * are the codes of nvfp4_fakequant_fwd_fp8scale (rounding x * (1/Q8(s_pre))),
 * out->scales [rows][cols/16] the E4M3 bytes of s_post (of s_pre when s_post
 * is NULL) in units of g, so that de-quantising with the same global amax
 * (M = 448, E4M3 scales) gives that forward's output. out->choice is ignored;
 * out->dequant must be NULL (NVFP4_ERR_ENUM). Errors and status bits as
 * nvfp4_fakequant_fwd_fp8scale. */
NVFP4_API nvfp4_status nvfp4_export_scales(const void* x, int64_t rows, int64_t cols,
                                           const float* s_pre, const float* s_post,
                                           const float* global_amax, const nvfp4_out* out,
                                           int32_t* status, void* stream);

/* nvfp4_requant_transpose target */
#define NVFP4_TARGET_MXFP8 0 /* E4M3 values, one E8M0 power-of-two scale per 32 */
#define NVFP4_TARGET_NVFP4 1 /* the NVFP4 row encoding of the transposed tensor  */

/* Backward-operand re-quantisation (End-to-End 4-Bit Training,
 * "Re-quantization with stochastic rounding" and its quantised-linear-layer
 * figure): de-quantise the forward row encoding of X [slices][rows][cols],
 * transpose it, and quantise it again along the other axis, so that the
 * backward GEMM sees X^T blocked along its own contraction dimension.
 * Input: codes [S][R][C/2] and scales [S][R][C/16] exactly as nvfp4_quantize's
 * row encoding wrote them, with src its config (scale_fmt, four_over_six and
 * scale_max fix the decoding; other fields are ignored) and global_amax
 * (fp32 [S]) the amax it was given. De-quantised value: the fp32 product
 * e2m1(code) * (dec(scale) * g), never rounded to bf16.
 * target NVFP4_TARGET_MXFP8 (rows % 32 == 0): per 32 consecutive values of a
 * column, shared exponent e = the smallest integer with amax <= 448 * 2^e
 * (clamped to [-127, 127]); out->scales [S][C][R/32] receives e + 127 (E8M0);
 * out->codes [S][C][R] one signed E4M3 byte per value, the code of v * 2^-e
 * (RNE, or stochastic rounding onto the E4M3 grid), never saturating.
 * target NVFP4_TARGET_NVFP4 (rows % 16 == 0): out is the row encoding of the
 * fp32 matrix X^T with the outer scale g = global_amax / (6 M_dst) and the
 * block-scale format, 4/6 mode and rule of dst: codes [S][C][R/2], scales
 * [S][C][R/16], choice [S][ceil(R*C/512)] words (required iff
 * dst->four_over_six).
 * dst supplies rounding, seed and step (both targets) and scale_fmt,
 * four_over_six, four_over_six_rule and scale_max (NVFP4 target); dst->blocks
 * is ignored. Stochastic rounding draws its bits as nvfp4_quantize does, with
 * direction 2 in the counter and idx the flat index of the output layout.
 * out->dequant must be NULL. A de-quantised value that is not finite (a
 * scale times g overflowing fp32) sets NVFP4_DEV_NONFINITE_INPUT; a bad
 * global amax sets NVFP4_DEV_BAD_AMAX.
 * Errors: NULL required pointers, non-NULL out->dequant (NVFP4_ERR_ENUM),
 * cols % 16, rows % 32 (MXFP8) or % 16 (NVFP4), enum fields out of range,
 * misaligned buffers (codes, scales and outputs 16-byte aligned). */
NVFP4_API nvfp4_status nvfp4_requant_transpose(const nvfp4_config* src, const nvfp4_config* dst,
                                               int32_t target, const uint8_t* codes,
                                               const uint8_t* scales, int64_t slices,
                                               int64_t rows, int64_t cols,
                                               const float* global_amax, const nvfp4_out* out,
                                               int32_t* status, void* stream);

/* MXFP8 quantisation of a bf16 tensor x [slices][rows][cols] (End-to-End
 * 4-Bit Training, the quantised-linear-layer figure: the bf16 output gradient
 * is quantised to MXFP8 with stochastic rounding for the DGRAD GEMM and,
 * transposed, for the WGRAD GEMM). Per 32 consecutive values: shared
 * exponent e = the smallest integer with amax <= 448 * 2^e (clamped to
 * [-127, 127]; 448 = E4M3's largest value), scale byte e + 127 (E8M0);
 * element byte = the signed E4M3 code of v * 2^-e (one fp32 rounding), by
 * RNE or by stochastic rounding onto the E4M3 grid; never saturating, as
 * |v * 2^-e| <= 448.
 * cfg: blocks NVFP4_BLOCKS_ROW / COL / BOTH (both from one read of x),
 * rounding, seed, step; the other fields are ignored.
 *   row encoding (blocks along cols, cols % 32 == 0): row->codes
 *     [S][R][C] bytes, row->scales [S][R][C/32];
 *   col encoding (the row encoding of X^T, rows % 32 == 0): col->codes
 *     [S][C][R], col->scales [S][C][R/32].
 * choice is ignored; dequant must be NULL (NVFP4_ERR_ENUM). Stochastic
 * rounding: the 16 random bits of the element at flat index idx of its
 * output layout are those nvfp4_quantize uses, with direction 0 (rows) or 1
 * (columns) in the counter. A block holding NaN or Inf sets
 * NVFP4_DEV_NONFINITE_INPUT; its bytes are then unspecified.
 * Errors: NULL cfg / x / a required output, blocks or rounding out of range,
 * negative sizes, cols % 32 (rows wanted) or rows % 32 (columns wanted), x
 * or an output buffer not 16-byte aligned, status not 4-byte aligned. */
NVFP4_API nvfp4_status nvfp4_mx_quantize(const nvfp4_config* cfg, const void* x, int64_t slices,
                                         int64_t rows, int64_t cols, const nvfp4_out* row,
                                         const nvfp4_out* col, int32_t* status, void* stream);

/* ---- diagnostics: the device codecs element by element -------------------
 * For exhaustive checks of the conversions the kernels use. op:
 *   0: out[i] = E2M1 RNE code of in[i]
 *   1: out[i] = E4M3 code of in[i] >= 0        (block-scale encoder)
 *   2: out[i] = UE5M3 code of in[i] >= 0       (block-scale encoder)
 *   3: out[i] = E2M1 stochastic code of in[i] with random bits aux[i] & 0xFFFF
 *   4: out[i] = signed E4M3 RNE code of in[i]   (MXFP8 element encoder)
 *   5: out[i] = signed E4M3 stochastic code of in[i] with bits aux[i] & 0xFFFF
 *   6: out[i] = E8M0 byte (e + 127) of the MX shared exponent for amax in[i]
 *   7: as 5, by the unsaturated form the kernels use (defined for
 *      |in[i]| <= 448)
 * Ops 0 and 3 convert groups of 8 consecutive inputs exactly as the kernels do.
 * in, aux (ops 3, 5): device arrays of n elements; out: device uint8 [n].
 * This entry point has no counterpart on the pages; it exists for testing. */
NVFP4_API nvfp4_status nvfp4_codec_probe(int32_t op, const float* in, const uint32_t* aux, int64_t n,
                               uint8_t* out, void* stream);

/* The 16 random bits the stochastic rounder draws for elements idx0 ..
 * idx0 + n - 1 of an encoding (direction 0 = rows, 1 = columns, 2 =
 * re-quantisation), written to
 * out (device uint32 [n]). Diagnostics; no counterpart on the pages. */
NVFP4_API nvfp4_status nvfp4_sr_bits(uint32_t seed, uint32_t step, uint32_t direction, uint64_t idx0,
                           int64_t n, uint32_t* out, void* stream);

/* Short text for a status code. */
NVFP4_API const char* nvfp4_status_string(nvfp4_status s);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_H */
