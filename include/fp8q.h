/*
 * fp8q.h -- C ABI of libfp8q: FP8 scaled quantization and the scaled FP8 GEMM
 * that consumes it, for NVIDIA GB300 (sm_103a).
 *
 * The path (sources are the pages this library follows):
 *   amax -> scale -> quantize / cast-transpose -> scaled FP8 GEMM,
 * with four scaling recipes:
 *   - per-tensor current scaling: scale from this tensor's max |x|
 *     ("Colossal-AI FP8" page, "current scaling"; "FP8 quantized-training
 *     guide" page, section "tensor-level scaling" / "instant scaling scheme");
 *   - per-tensor delayed scaling: scale from a history of past amaxes, updated
 *     next to the GEMM (Colossal-AI FP8 page, "delayed scaling"; guide,
 *     "delayed scaling scheme");
 *   - blockwise scaling: one scale per 1x128 tile (activations, gradients) or
 *     per 128x128 tile (weights), E4M3 (guide, section "block-level scaling");
 *   - MXFP8: one E8M0 power-of-two scale per 1x32 block (guide, section
 *     "MXFP8 scaling").
 * Formats: E4M3 (1-4-3, max 448, no infinity) and E5M2 (1-5-2, max 57344)
 * (guide, section "format choice E4M3 and E5M2").  GEMM inputs are FP8, the
 * accumulation FP32, the output BF16 (fprop / dgrad) or FP32 (wgrad) (the
 * search-result page's mixed-precision dataflow paragraph).
 *
 * Conventions shared by every call:
 *   - Ownership: the caller allocates and owns every buffer.  The library holds
 *     no allocation.  Pointers marked "device" are device pointers.
 *   - Asynchrony: every call is enqueued on `stream` and returns without
 *     waiting (except fp8_get_device_status).  No call synchronizes the host.
 *   - Layouts: matrices are dense row-major.  A "[R, C] bf16" input has R rows
 *     of C bfloat16 values.  The column-wise copy of an [R, C] input is the
 *     [C, R] matrix of its transpose, quantized with the recipe's blocks along
 *     its own rows.
 *   - Alignment: matrix pointers must be 16-byte aligned; FP32 scale arrays
 *     4-byte aligned; GEMM-ready MX scale arrays 16-byte aligned.
 *   - Errors: arguments are checked on the host before anything is enqueued;
 *     a rejected call enqueues nothing and returns FP8_ERR_INVALID_ARG,
 *     FP8_ERR_SHAPE, FP8_ERR_ALIGNMENT or FP8_ERR_UNSUPPORTED.  A CUDA launch
 *     error returns FP8_ERR_CUDA.  Kernels never trap: a device-side failure
 *     (a wait that ran out of time, a state argument out of range, and in the
 *     debug library an access outside its buffer) sets a device error word,
 *     read and cleared by fp8_get_device_status.
 */
#ifndef FP8Q_H
#define FP8Q_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FP8_OK = 0,
  FP8_ERR_INVALID_ARG = 1, /* null pointer, bad enum, negative size */
  FP8_ERR_SHAPE = 2,       /* a size the recipe or kernel cannot tile */
  FP8_ERR_ALIGNMENT = 3,   /* a pointer not aligned as required */
  FP8_ERR_UNSUPPORTED = 4, /* an operand / recipe pairing not provided */
  FP8_ERR_CUDA = 5,        /* a CUDA runtime error */
  FP8_ERR_TIMEOUT = 6,     /* a device wait ran out of time (see fp8_get_device_status) */
  FP8_ERR_DEVICE_STATE = 7, /* a device-resident state argument was out of range */
  FP8_ERR_INDEX = 8         /* (debug library only) a kernel access fell outside its buffer and was skipped */
} fp8_status;

typedef enum { FP8_E4M3 = 0, FP8_E5M2 = 1 } fp8_format;

typedef enum {
  FP8_TENSOR = 0,        /* one FP32 scale for the whole tensor (current or delayed) */
  FP8_BLOCK_1x128 = 1,   /* one FP32 scale per 128 consecutive elements of a row */
  FP8_BLOCK_128x128 = 2, /* one FP32 scale per 128x128 tile */
  FP8_MX_1x32 = 3,       /* one E8M0 byte per 32 consecutive elements of a row, row-major */
  FP8_MX_1x32_TILED = 4, /* the same exponents in the GEMM-ready tiled layout (below) */
  /* MXFP8 with the floor-rule exponent, the documented alternate of the default ceil
   * rule: e = floor(log2 amax) - emax (emax 8 for E4M3, 15 for E5M2), so a block's
   * largest elements may saturate to +-FMAX.  Same layouts as FP8_MX_1x32 and
   * FP8_MX_1x32_TILED; everything that reads E8M0 scales (GEMM, dequantize) takes them
   * like the default MX recipes. */
  FP8_MX_1x32_FLOOR = 5,
  FP8_MX_1x32_FLOOR_TILED = 6
} fp8_recipe;

typedef enum { FP8_OUT_BF16 = 0, FP8_OUT_FP32 = 1 } fp8_out_dtype;

/*
 * fp8_amax -- per-tensor amax.  Colossal-AI FP8 page, "current scaling" (the
 * scale is computed from the maximum of the current tensor).
 *   x     device, [rows, cols] bf16 (any shape; rows * cols may be 0)
 *   amax  device, 1 float: receives max |x| over all elements, NaN ignored
 *         (0 for an empty tensor).  Exact, independent of reduction order.
 */
fp8_status fp8_amax(const void* x, int64_t rows, int64_t cols, float* amax, cudaStream_t stream);

/*
 * fp8_amax_f32 -- fp8_amax of a binary32 tensor (e.g. the FP32 master copy of a
 * weight that is quantized with current scaling; search-result page, the
 * mixed-precision dataflow paragraph: FP8 weights come from the higher-precision
 * copy).  x is device, [rows, cols] float, 16-byte aligned; otherwise as fp8_amax.
 */
fp8_status fp8_amax_f32(const float* x, int64_t rows, int64_t cols, float* amax, cudaStream_t stream);

/*
 * fp8_compute_scale -- per-tensor current-scaling scale.  Colossal-AI FP8
 * page, "current scaling"; guide, "instant scaling scheme".
 *   amax       device, 1 float (input)
 *   scale      device, 1 float: FMAX / amax as one binary32 division
 *              (FMAX = 448 for E4M3, 57344 for E5M2); 1 when amax is 0 or not
 *              finite; FLT_MAX when the quotient overflows
 *   scale_inv  device, 1 float: 1 / scale (binary32 division), the
 *              dequantization multiplier the GEMM takes
 */
fp8_status fp8_compute_scale(const float* amax, fp8_format fmt, float* scale, float* scale_inv,
                             cudaStream_t stream);

/*
 * amax_history_update -- one delayed-scaling step.  Colossal-AI FP8 page,
 * "delayed scaling" (the scale comes from a past time window); guide, "delayed
 * scaling scheme" (a buffer holding the maxima of several past steps).
 *   hist       device, len floats: the history ring (caller initialises to 0)
 *   len        history length, >= 1 (16 in the reference configuration)
 *   pos        device, 1 int32: next write slot, in [0, len) (initialise to 0)
 *   amax       device, 1 float: this step's amax (e.g. the amax_out of the cast)
 *   scale,     device, 1 float each: the scale the NEXT step quantizes with and
 *   scale_inv  its reciprocal (initialise to 1 and 1).
 * Effect: hist[pos] = amax; pos = (pos + 1) mod len; m = max(hist);
 * if 0 < m < inf: scale = FMAX / m (overflow -> FLT_MAX), scale_inv = 1 / scale;
 * otherwise scale and scale_inv are left unchanged.  A pos outside [0, len)
 * leaves everything unchanged and sets the device error word
 * (FP8_ERR_DEVICE_STATE from fp8_get_device_status).
 * The state is these four caller-owned buffers: saving and restoring them
 * resumes the sequence bit-identically.
 */
fp8_status amax_history_update(float* hist, int32_t len, int32_t* pos, const float* amax, fp8_format fmt,
                               float* scale, float* scale_inv, cudaStream_t stream);

/*
 * fp8_cast_transpose -- quantize a bf16 matrix into a row-wise and/or a
 * column-wise FP8 copy plus their scales.  Guide, sections "tensor-level
 * scaling", "block-level scaling" and "MXFP8 scaling"; the column-wise copy
 * serves the backward GEMMs, which consume the operands along the other axis
 * (the search-result page's dataflow paragraph).
 *   x      device, [rows, cols] bf16
 *   scale  FP8_TENSOR only: device, 1 float, the scale to multiply by (from
 *          fp8_compute_scale, or the delayed-scaling state).  NULL otherwise.
 *   amax_out  optional device float: receives max |x| of this input (NaN
 *          ignored).  Delayed scaling casts with the previous scale and records
 *          this step's amax here.
 *   q_row  device, [rows, cols] u8 FP8 codes, or NULL to skip the row-wise copy
 *   s_row  its dequantization multipliers:
 *            FP8_TENSOR:        1 float (1 / scale), may be NULL
 *            FP8_BLOCK_1x128:   float [rows, cols/128]
 *            FP8_BLOCK_128x128: float [rows/128, cols/128]
 *            FP8_MX_1x32:       u8 E8M0 [rows, cols/32] (exponent e stored as e + 127)
 *            FP8_MX_1x32_TILED: u8 E8M0, (rows/128) * (cols/128) atoms of 512 B;
 *                               exponent (r, b) at ((r/128)*(cols/128) + b/4)*512
 *                               + (r%32)*16 + ((r%128)/32)*4 + b%4
 *   q_col  device, [cols, rows] u8: the column-wise copy (the transpose,
 *          quantized with blocks along its rows), or NULL to skip it
 *   s_col  its multipliers, as s_row with rows and cols exchanged
 *          (FP8_BLOCK_128x128: the transpose of s_row)
 * Element rule: q = saturating round-to-nearest-even FP8 of (float(x) * s), one
 * binary32 product, with s = FMAX / amax of the block (FP32 recipes; same edge
 * rules as fp8_compute_scale) or s = 2^-e (MX: e the smallest integer with
 * amax <= FMAX * 2^e, clamped to [-127, 127]; 0 for an all-zero block).
 * Shapes: FP8_TENSOR takes any shape.  Blocked dimensions must be multiples of
 * the block (128 for the 1x128 copy's rows, 128 for both dims of 128x128, 32
 * for MX, 128 for both dims of MX_TILED); otherwise FP8_ERR_SHAPE.
 */
fp8_status fp8_cast_transpose(const void* x, int64_t rows, int64_t cols, fp8_recipe recipe, fp8_format fmt,
                              const float* scale, float* amax_out, uint8_t* q_row, void* s_row, uint8_t* q_col,
                              void* s_col, cudaStream_t stream);

/*
 * fp8_cast_transpose_f32 -- fp8_cast_transpose of a binary32 matrix: the FP32
 * master copy of a weight quantized directly, without a bf16 copy in between
 * (search-result page, mixed-precision dataflow paragraph: the FP8 weights come
 * from the higher-precision copy).  Every argument, output, layout, shape rule and
 * error as fp8_cast_transpose, except
 *   x  device, [rows, cols] float (binary32), 16-byte aligned
 * Element rule: q = saturating round-to-nearest-even FP8 of (x * s), one binary32
 * product of the binary32 input; block amaxes (and amax_out) are taken over the
 * binary32 values, NaN ignored.
 */
fp8_status fp8_cast_transpose_f32(const float* x, int64_t rows, int64_t cols, fp8_recipe recipe, fp8_format fmt,
                                  const float* scale, float* amax_out, uint8_t* q_row, void* s_row, uint8_t* q_col,
                                  void* s_col, cudaStream_t stream);

/*
 * fp8_cast_transpose_multi -- several fp8_cast_transpose calls in one launch (e.g.
 * the activation and the weight of a layer, each with its own recipe): the tiles
 * of all jobs are spread over one persistent grid, so the fixed cost of a launch
 * (the first loads, the last stores) is paid once.  Same results as calling
 * fp8_cast_transpose on each job in order.  Guide, "tensor-level scaling",
 * "block-level scaling", "MXFP8 scaling" (as fp8_cast_transpose).
 *   jobs    host array of n_jobs descriptions; each field as the argument of the
 *           same name of fp8_cast_transpose
 *   n_jobs  0..4 (FP8_ERR_INVALID_ARG beyond)
 * Every job is checked (as fp8_cast_transpose checks its arguments) before any
 * device work; the first failing job's status is returned.  Two jobs whose
 * recipes are (BLOCK_1x128, BLOCK_128x128), two MX_1x32 recipes (any layout or
 * exponent rule) or (TENSOR, TENSOR), in that order, run in a kernel compiled for
 * that pairing; any other mix in the general one.  The results do not depend on
 * which.
 */
typedef struct fp8_cast_job {
  const void* x;
  int64_t rows, cols;
  fp8_recipe recipe;
  fp8_format fmt;
  const float* scale;
  float* amax_out;
  uint8_t* q_row;
  void* s_row;
  uint8_t* q_col;
  void* s_col;
} fp8_cast_job;
fp8_status fp8_cast_transpose_multi(const fp8_cast_job* jobs, int32_t n_jobs, cudaStream_t stream);

/*
 * fp8_quantize -- the row-wise copy only: fp8_cast_transpose with q_col = NULL.
 */
fp8_status fp8_quantize(const void* x, int64_t rows, int64_t cols, fp8_recipe recipe, fp8_format fmt,
                        const float* scale, float* amax_out, uint8_t* q, void* s, cudaStream_t stream);

/*
 * fp8_dequantize -- FP8 -> BF16 (e.g. FP8 weights to BF16; search-result page,
 * the FP8-to-BF16 weight conversion; guide, "block-level scaling" and "MXFP8
 * scaling" for the multipliers).
 *   q       device, [rows, cols] u8 FP8 codes (format fmt), row-major: a
 *           row-wise copy, or a column-wise copy passed as its own [rows, cols]
 *   recipe  how q was quantized; s holds the multipliers (scale_inv) exactly as
 *           fp8_cast_transpose wrote them for that copy:
 *           TENSOR float[1]; BLOCK_1x128 float[rows, cols/128];
 *           BLOCK_128x128 float[rows/128, cols/128]; MX_1x32 u8 E8M0
 *           [rows, cols/32]; MX_1x32_TILED the GEMM-ready atoms
 *   y       device, [rows, cols] bf16: the exact product decode(q) * multiplier
 *           rounded once to bfloat16 (nearest, ties to even; gradual underflow;
 *           overflow to inf).  E8M0 byte 0xFF (its NaN) gives NaN.
 * q and y 16-byte aligned (FP8_ERR_ALIGNMENT).  Shapes: TENSOR any; 1x128
 * cols % 128; 128x128 and MX_1x32_TILED rows and cols % 128; MX_1x32 cols % 32
 * (FP8_ERR_SHAPE).  rows or cols == 0 is a no-op.
 */
fp8_status fp8_dequantize(const uint8_t* q, int64_t rows, int64_t cols, fp8_recipe recipe, fp8_format fmt,
                          const void* s, void* y, cudaStream_t stream);

/*
 * fp8_allreduce_sum -- FP8 gradient all-reduce with a shared scale (FP8-LM news
 * article, "automatic scaling": the gradient's scaling factor keeps its values
 * inside FP8's range through the all-reduce), for k data-parallel ranks whose
 * gradients are held on this device as the rows of g.  The ranks agree on the
 * global amax A (the all-reduce MAX), all use the per-tensor scale
 * s = FMAX / A (fp8_compute_scale's rule), and the reduction sums the decoded
 * FP8 payloads in rank order in binary32, then multiplies once by 1 / s.
 *   g          device, [k, n] bf16 row-major (rank r's gradient in row r)
 *   amax       device float[1], overwritten with A
 *   q          device, [k, n] u8: rank r's payload encode_sat(g[r] * s) (fmt)
 *   scale_inv  device float[1]: 1 / s
 *   out        device, [n] fp32: the reduced gradient
 * k >= 1; n % 8 == 0 (FP8_ERR_SHAPE); g and out 16-byte aligned, q 8-byte
 * aligned (FP8_ERR_ALIGNMENT).  n == 0 is a no-op.  For E4M3 and k <= 64 the
 * sum is exact, so out does not depend on the rank order.
 */
fp8_status fp8_allreduce_sum(const void* g, int32_t k, int64_t n, fp8_format fmt, float* amax, uint8_t* q,
                             float* scale_inv, float* out, cudaStream_t stream);

/*
 * fp8_allreduce_sum_noalloc -- fp8_allreduce_sum without its amax argument: the
 * per-rank and global amaxes live in scratch the library owns, so a caller that
 * cannot provide device memory beyond the buffers it reduces (a gradient-reduction
 * hook in a runtime without a device allocator of its own, or a process whose
 * device memory a caching allocator has reserved in full) needs none.  The pages
 * have no counterpart; results are bit-identical to fp8_allreduce_sum's (the
 * maximum is exact and order-free).
 *   g, k, n, fmt, q, scale_inv, out   as fp8_allreduce_sum
 * Scratch: a file-scope device array of 1025 floats (4 KB) per device, one amax
 * per rank and the global one, so k <= 1024 (FP8_ERR_SHAPE beyond).  Nothing in
 * it has to start at zero: each call clears the slots it uses first.  All calls on
 * a device share it: calls whose executions overlap (other streams, other host
 * threads) race and must be ordered by the caller.  The first call on a device
 * looks up the scratch address (cudaGetSymbolAddress, with that device current)
 * and keeps it; make that first call before any stream capture.  A first call
 * made while `stream` is being captured does nothing and returns
 * FP8_ERR_INVALID_ARG.
 */
fp8_status fp8_allreduce_sum_noalloc(const void* g, int32_t k, int64_t n, fp8_format fmt, uint8_t* q, float* scale_inv,
                                     float* out, cudaStream_t stream);

/*
 * fp8_scaled_gemm -- C = deq(A) . deq(B)^T with FP32 accumulation.
 * Search-result page, dataflow paragraph (FP8 inputs, FP32 accumulation, BF16
 * output; wgrad output FP32); guide, "code changes" (the three GEMMs of a layer
 * take quantized inputs); guide, "block-level scaling" and "MXFP8 scaling" for
 * the scale pairings.
 *   A   device, [M, K] u8 FP8 (format fa), K contiguous
 *   B   device, [N, K] u8 FP8 (format fb), K contiguous
 *   sA, sB  the multipliers written by fp8_cast_transpose for A and B
 *   C   device, [M, N] row-major, bf16 (FP8_OUT_BF16, round to nearest) or fp32
 * Pairings (ra, rb): (TENSOR, TENSOR); (BLOCK_1x128, BLOCK_128x128);
 * (BLOCK_1x128, BLOCK_1x128); (MX_1x32_TILED, MX_1x32_TILED).  Others return
 * FP8_ERR_UNSUPPORTED.  M, N, K must be multiples of 128 (FP8_ERR_SHAPE);
 * M or N == 0 is a no-op, K == 0 writes zeros.
 * Workspace: with (TENSOR, TENSOR) or (MX, MX) and M % 256 == 0, a GEMM whose tiles
 * do not fill a whole number of waves of CTA pairs may cut tiles along K (two or three
 * full waves, or one when K >= 8192: every pair takes an equal share of the last tiles'
 * K blocks; otherwise,
 * when the last wave leaves at least half of the pairs idle, with one wave or with
 * K >= 8192, that wave's tiles are cut into K ranges) and sums the parts of a tile in a
 * fixed order; it uses a workspace the library allocates on
 * the first such call on `stream` (SMs / 2 slots of 256 KB and their counters, kept
 * for the process's lifetime; up to 16 streams a device).  A call on a stream that is
 * being captured and has none yet runs unsplit.  Results are deterministic either way
 * but differ in the last bits between the split and unsplit runs of one shape.
 */
fp8_status fp8_scaled_gemm(const uint8_t* A, fp8_format fa, fp8_recipe ra, const void* sA, const uint8_t* B,
                           fp8_format fb, fp8_recipe rb, const void* sB, int64_t M, int64_t N, int64_t K, void* C,
                           fp8_out_dtype out, cudaStream_t stream);

/*
 * fp8_scaled_gemm_amax -- fp8_scaled_gemm with the next layer's per-tensor
 * quantization fused into its epilogue.  Colossal-AI FP8 article, "delayed
 * scaling": the scale comes from a window of past maxima and its update is
 * fused with the GEMM; guide, "delayed scaling scheme".  With y the value the
 * plain GEMM stores in C (rounded to bf16 for FP8_OUT_BF16, the FP32 value
 * for FP8_OUT_FP32):
 *   C           device, nullable: as fp8_scaled_gemm
 *   c_amax      device float[1], nullable: overwritten with max |y| (NaN
 *               ignored) -- the value the scale history records
 *   c_scale     device float[1]: the per-tensor scale of C's FP8 copy (a
 *               delayed-scaling state's scale); required with C_q
 *   fc, C_q     device [M, N] u8 row-major, nullable: encode_sat(y * c_scale),
 *               round-to-nearest-even, the bytes fp8_quantize(TENSOR) writes
 *               for C with that scale
 *   c_scale_inv device float[1], nullable (only with C_q): 1 / c_scale
 * At least one of c_amax and C_q (FP8_ERR_INVALID_ARG); C and C_q 16-byte
 * aligned.  Shapes, pairings and errors as fp8_scaled_gemm; M, N or K == 0
 * give amax 0 and all-zero codes.
 */
fp8_status fp8_scaled_gemm_amax(const uint8_t* A, fp8_format fa, fp8_recipe ra, const void* sA, const uint8_t* B,
                                fp8_format fb, fp8_recipe rb, const void* sB, int64_t M, int64_t N, int64_t K, void* C,
                                fp8_out_dtype out, float* c_amax, const float* c_scale, fp8_format fc, uint8_t* C_q,
                                float* c_scale_inv, cudaStream_t stream);

/*
 * fp8_get_device_status -- synchronize `stream`, then read and clear the
 * device error word of the current device.  Returns FP8_OK, FP8_ERR_TIMEOUT
 * (some kernel gave up a wait), FP8_ERR_DEVICE_STATE, FP8_ERR_INDEX (debug
 * library: a kernel skipped an access outside its buffer), or FP8_ERR_CUDA.
 */
fp8_status fp8_get_device_status(cudaStream_t stream);

/*
 * fp8_debug_wait_timeout -- enqueue a one-CTA kernel that waits on a barrier
 * nothing will complete, with the same bounded wait every kernel uses; it
 * gives up after about one second and reports FP8_ERR_TIMEOUT through
 * fp8_get_device_status.  Exists to test the failure path without a fault.
 */
fp8_status fp8_debug_wait_timeout(cudaStream_t stream);

/*
 * fp8_debug_index_check -- enqueue a one-thread kernel that checks `index` against
 * `extent` as the kernels check their plain global accesses, touching no memory.  The
 * debug library (built with FP8Q_DEBUG_INDEX) reports an index outside [0, extent) as
 * FP8_ERR_INDEX through fp8_get_device_status; the release library checks nothing.
 * Exists to test that reporting path without a fault.
 */
fp8_status fp8_debug_index_check(int64_t index, int64_t extent, cudaStream_t stream);

/*
 * fp8_debug_gemm_plan -- how fp8_scaled_gemm (fused != 0: fp8_scaled_gemm_amax with an
 * FP8 copy of C) would divide an M x N x K product with these recipes and output type on
 * a device with `num_sms` SMs of which `resident_pairs` 2-CTA clusters fit at once (0: no
 * limit): host logic only, no device call.  Writes plan[0..7] = {CTA pairs (0/1), kernel
 * variant (0 per-tensor, 1 blockwise one CTA 128-deep stages, 3 MXFP8, 4 blockwise per-row
 * B one CTA, 5 blockwise 256-deep stages, 6 blockwise per-row B pairs, 7 blockwise 256 x
 * 160 pair tiles), tile width, tile count, stream-K (0/1), K ranges of the last wave (1:
 * uncut), first tile shared or cut, CTAs or pairs launched}.  A stream-K or K-range plan
 * also needs the per-stream workspace; a real call without one runs whole tiles.  Errors
 * as fp8_scaled_gemm's argument checks; `plan` (8 int64, host memory) is the caller's.
 * Exists to test the dispatch rules without a GPU.
 */
fp8_status fp8_debug_gemm_plan(fp8_recipe ra, fp8_recipe rb, fp8_out_dtype out, int64_t M, int64_t N, int64_t K,
                               int32_t fused, int32_t num_sms, int32_t resident_pairs, int64_t* plan);

/* Human-readable name of a status code (static storage). */
const char* fp8_status_string(fp8_status status);

#ifdef __cplusplus
}
#endif

#endif /* FP8Q_H */
