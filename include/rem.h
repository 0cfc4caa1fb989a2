/*
 * rem.h -- row-exact few-row quantized mat-vec on GB300 (sm_103a), C ABI.
 *
 * The operation is the one mlx-native 0.18.0 src/ops/row_exact_matvec.rs
 * defines (module doc "Row-exact few-row mat-vec"):
 *
 *     y[b, j, :] = W[b] . x[b, j, :]      for b < batch, j < m, 1 <= m <= 8
 *
 * with F32 input rows x, F32 output y and weights W stored row-major as F16
 * or as Q8_0 / Q4_K / Q6_K / Q5_0 blocks (RowExactWeight).  Batch b reads the
 * weight rows b*n .. b*n+n-1, i.e. bytes from b*n*row_bytes(k)
 * (RowExactMatvecShape, "Batched / grouped products").
 *
 * Row exactness (module doc "Row exactness"): output row j is bitwise
 * identical whether it is computed alone (m = 1) or as one row of any
 * m <= 8, on every run, as long as the split factor and the engine are the
 * same.  Both are derived from (wtype, batch*n, k) alone (rem_split_factor,
 * rem_engine_of); rows_per_cta and the lane layout only pack rows and never
 * change bits.
 *
 * Memory and ownership.  Every pointer passed to a compute call is a CUDA
 * device pointer (or managed memory) owned by the caller; the library never
 * allocates, frees, synchronises or copies to the host on these calls.
 * `stream` is a cudaStream_t (NULL = the legacy default stream); the work is
 * enqueued asynchronously on it and the call returns before it runs.  It
 * keeps stream order: it sees every earlier write of the stream and later
 * work sees its output (the kernel may start early and prefetch weights into
 * L2, but reads x and W into the SM and writes y only once the previous
 * kernel of the stream has completed).
 *
 * Errors.  Every call validates its arguments before it launches anything;
 * on an error nothing is written and a message prefixed "rem_matvec:" (or the
 * call's name) is available from rem_last_error() on the calling thread.
 * A kernel never waits without bound: a wait that runs out (the schedule's
 * wait_ns, 10 s by default) makes the launch write NaN for the outputs it
 * could not finish and records the event in a per-device status word that
 * rem_device_status() reads.  The library reads no environment variables.
 *
 * Engines.  Two kernels compute the product, and the engine is part of the
 * arithmetic, like the split factor: rows are bitwise comparable between
 * calls with the same engine and split.  By default the engine follows from
 * (wtype, batch*n, k) alone (rem_engine_of).
 *   REM_ENGINE_SIMT  lanes over rows on the FP32 pipe: every weight type
 *   REM_ENGINE_TC    the tensor cores (tcgen05) for Q8_0, Q5_0 and Q6_K: per
 *                    block, the exact codes times each input split into two
 *                    bfloat16 parts, summed in binary32, then scaled by the
 *                    block scale in binary32; up to 32 input rows per pass
 *                    over the weights (Q6_K: 16)
 */
#ifndef REM_H
#define REM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Weight storage (RowExactWeight); the integer values are part of the ABI. */
typedef enum {
    REM_F16 = 0,   /* row-major [batch*n, k] IEEE binary16, little-endian     */
    REM_Q8_0 = 1,  /* [batch*n, k/32] blocks of 34 B: d f16 | int8 qs[32]      */
    REM_Q4_K = 2,  /* [batch*n, k/256] blocks of 144 B: d, dmin f16 | 12 B
                      6-bit scales/mins | 128 B nibbles                        */
    REM_Q6_K = 3,  /* [batch*n, k/256] blocks of 210 B: 128 B low nibbles |
                      64 B high 2-bit | int8 scales[16] | d f16                */
    REM_Q5_0 = 4,  /* [batch*n, k/32] blocks of 22 B: d f16 | u32 high bits |
                      16 B nibbles                                             */
    /* dense weights under the same row contract (the row-independent gemv of
       nuvec-core 0.6.0 src/gpu.rs, gemv_rows over F32 / F16 / BF16 matrices) */
    REM_F32 = 5,   /* row-major [batch*n, k] IEEE binary32, little-endian     */
    REM_BF16 = 6,  /* row-major [batch*n, k] bfloat16 (upper half of binary32) */
    /* affine group quantization (the Affine mode of nuvec-core 0.6.0
       src/gpu.rs, with (group_size, bits) and pack_factor): codes
       [batch*n, k*bits/32] uint32 words holding one little-endian bit
       stream per row, code i at stream bits [bits*i, bits*i + bits), lowest
       first; scales and biases [batch*n, k/group] binary16 in their own
       arrays; w = scale*q + bias.  Only through rem_matvec_affine /
       rem_dequantize_affine.                                             */
    REM_A4_G32 = 7, REM_A4_G64 = 8, REM_A4_G128 = 9,    /* 4-bit codes */
    REM_A8_G32 = 10, REM_A8_G64 = 11, REM_A8_G128 = 12, /* 8-bit codes */
    REM_A3_G32 = 13, REM_A3_G64 = 14, REM_A3_G128 = 15, /* 3-bit codes, 8 per 3-byte packing unit */
    REM_A5_G32 = 16, REM_A5_G64 = 17, REM_A5_G128 = 18, /* 5-bit codes, 8 per 5-byte packing unit */
    REM_A6_G32 = 19, REM_A6_G64 = 20, REM_A6_G128 = 21  /* 6-bit codes, 4 per 3-byte packing unit */
} rem_wtype;

/* Status codes. */
typedef enum {
    REM_OK = 0,
    REM_EINVAL = -1,   /* an argument broke a validation rule; nothing launched */
    REM_ELAUNCH = -2,  /* the schedule needs more threads per block than every
                          kernel of the weight type can launch on this device */
    REM_ECUDA = -3     /* a CUDA call failed (device, attribute or launch)     */
} rem_status;

/* Engines (see "Engines" above). */
#define REM_ENGINE_AUTO (-1)
#define REM_ENGINE_SIMT 0
#define REM_ENGINE_TC 1

/* Test hook of rem_schedule.test_flags: the kernel issues no copy for its
   first pipeline stage (TMA staging only), so that stage's waits run out
   after wait_ns and the launch reports through rem_device_status. */
#define REM_TEST_SKIP_FIRST_STAGE 1u

/*
 * Schedule of rem_matvec_sched.  Zero / -1 fields take the default.
 *   split         K ranges per weight row (0 = rem_split_factor); changes bits
 *   rows_per_cta  0, 32, 64 or 128 (SIMT engine; numerically inert; the
 *                 tensor-core engine always takes 128 rows per thread block)
 *   layout        -1, or the SIMT engine's lane layout 0..3: one weight row per
 *                 lane, two rows per lane, two lane groups of two rows each
 *                 sharing the input rows, two lane groups of four rows each
 *                 (2 needs m >= 2; 3 exists for F16 / BF16 at m = 6 and 8 only;
 *                 Q6_K has layout 0 only; a layout without a kernel for the
 *                 call is REM_ELAUNCH).  Numerically inert.
 *   engine        REM_ENGINE_AUTO, REM_ENGINE_SIMT or REM_ENGINE_TC; changes bits
 *   wait_ns       bound of every in-kernel wait in nanoseconds (0 = 10 s)
 *   test_flags    0, or REM_TEST_SKIP_FIRST_STAGE (tests only)
 */
typedef struct {
    uint32_t split;
    uint32_t rows_per_cta;
    int32_t layout;
    int32_t engine;
    uint64_t wait_ns;
    uint32_t test_flags;
} rem_schedule;

#define REM_MAX_ROWS 8     /* ROW_EXACT_MATVEC_MAX_ROWS */
#define REM_MAX_SPLIT 16   /* largest split factor the argument rules accept */
#define REM_MAX_CLUSTER_SPLIT 8  /* largest split the kernels launch (cluster size); above: REM_ELAUNCH */

/*
 * rem_matvec -- y[b, j, :] = W[b] . x[b, j, :] with the default schedule
 * (dispatch_row_exact_matvec).
 *
 *   W       device pointer to batch*n weight rows of rem_row_bytes(wtype, k)
 *           bytes each, row-major, batch-major.  Alignment: F16 8 B, Q8_0 2 B,
 *           Q4_K 16 B, Q6_K 2 B, Q5_0 2 B, F32 4 B, BF16 8 B.
 *   wtype   a rem_wtype value.
 *   n, k    output columns per batch (= weight rows per batch) and inner
 *           dimension; k must be a multiple of 4 (F16, F32, BF16), 32 (Q8_0,
 *           Q5_0) or 256 (Q4_K, Q6_K).
 *   batch   independent products, >= 1.
 *   x       device F32 input, 16-byte aligned.
 *   m       input rows, 1..8.
 *   x_batch_stride, y_batch_stride   elements between batches.
 *   y       device F32 output, 4-byte aligned.
 *
 * Row strides are not arguments here.  They are inferred:
 *   batch == 1                        x_row_stride = k,       y_row_stride = n
 *   batch > 1, x_batch_stride < m*k   x_row_stride = batch*k, y_row_stride = batch*n
 *                                     (token-major grouped projection,
 *                                      RowExactMatvecShape::grouped_token_major)
 *   otherwise (batch-major)           x_row_stride = k,       y_row_stride = n
 * Use rem_matvec_ex to state them.
 *
 * Returns REM_OK, or REM_EINVAL / REM_ELAUNCH / REM_ECUDA (see rem_status).
 */
int rem_matvec(const void* W, int wtype, uint32_t n, uint32_t k, uint32_t batch,
               const float* x, uint32_t m, uint32_t x_batch_stride,
               float* y, uint32_t y_batch_stride, void* stream);

/*
 * rem_matvec_ex -- the full form (dispatch_row_exact_matvec_scheduled with
 * an explicit RowExactMatvecShape and RowExactMatvecSchedule).
 *
 *   x_row_stride, x_batch_stride   elements, multiples of 4
 *   y_row_stride, y_batch_stride   elements; the m*batch output rows of n
 *                                  elements must not overlap
 *   split         K ranges per weight row, 1..REM_MAX_SPLIT, or 0 for
 *                 rem_split_factor(wtype, batch*n, k).  Rows are bitwise
 *                 comparable only between calls with the same split.
 *   rows_per_cta  0 (automatic) or 32, 64 or 128: weight rows one thread
 *                 block handles.  Numerically inert.
 *
 * A split whose thread block would exceed the kernels' launch limit returns
 * REM_ELAUNCH instead of launching (the page refuses such a launch rather
 * than let Metal drop it; CUDA would fail it).
 */
int rem_matvec_ex(const void* W, int wtype, uint32_t n, uint32_t k, uint32_t batch,
                  const float* x, uint32_t m, uint32_t x_row_stride, uint32_t x_batch_stride,
                  float* y, uint32_t y_row_stride, uint32_t y_batch_stride,
                  uint32_t split, uint32_t rows_per_cta, void* stream);

/*
 * rem_matvec_axpby -- y[b, j, :] = alpha * (W[b] . x[b, j, :]) + beta * c[b, j, :],
 * the fused epilogue of the gemv with an addend (nuvec-core 0.6.0
 * src/gpu.rs, the gemv "axpby" variant: alpha, beta and the addend's strides
 * along the output).  Each output is fma(alpha, acc, beta * c) with beta * c
 * rounded first; with beta == 0 c is not read and y = alpha * acc (so
 * alpha = 1, beta = 0 is bitwise rem_matvec_ex with split 0).  The epilogue
 * acts on every output after the fixed reduction, so rows stay exact.
 *
 *   x, y, strides   as rem_matvec_ex (automatic split and packing)
 *   c               F32 addend, element (b, j, i) at
 *                   b*c_batch_stride + j*c_row_stride + i; c_row_stride = 0
 *                   broadcasts one bias vector over the m rows,
 *                   c_batch_stride = 0 over the batch.  c may be y itself
 *                   with the same strides (y = alpha*W.x + beta*y); any other
 *                   overlap of c and y is refused.  Ignored when beta == 0.
 */
int rem_matvec_axpby(const void* W, int wtype, uint32_t n, uint32_t k, uint32_t batch,
                     const float* x, uint32_t m, uint32_t x_row_stride, uint32_t x_batch_stride,
                     float* y, uint32_t y_row_stride, uint32_t y_batch_stride,
                     float alpha, float beta, const float* c, uint32_t c_row_stride,
                     uint32_t c_batch_stride, void* stream);

/*
 * rem_matvec_affine -- y[b, j, :] = W[b] . x[b, j, :] for affine group-quantized
 * W (next step 2 of the few-row path: the Affine quantized matmul of nuvec-core
 * 0.6.0 src/gpu.rs).  The page fixes the (group_size, bits) parameters and the
 * packing factor (pack_factor: 8 codes per packing unit for 3 and 5 bits, 4
 * for 6 bits, 32/bits for 4 and 8 bits, so every unit is whole bytes); the
 * element formula and layout are the plain reading of that mode:
 *   codes    batch*n rows of k*bits/32 uint32 words, little-endian; a row's
 *            codes are one bit stream (byte j = stream bits 8j .. 8j+7) and
 *            code i sits at stream bits [bits*i, bits*i + bits), lowest bit
 *            first (for 4 and 8 bits: bits [bits*(i % (32/bits)), +bits) of
 *            word i / (32/bits)); 4-byte aligned (16-byte aligned rows use
 *            TMA staging)
 *   scales, biases   batch*n rows of k/group binary16 values, 2-byte aligned
 *   w[r, i] = fl(fl(scale[r, i/group] * q) + bias[r, i/group])
 * wtype is one of REM_A4_G32 .. REM_A6_G128; k must be a multiple of the
 * group size.  Other arguments as rem_matvec_ex (split 0 = automatic).  Row
 * exactness holds as for the other formats.
 */
int rem_matvec_affine(const void* codes, const uint16_t* scales, const uint16_t* biases, int wtype,
                      uint32_t n, uint32_t k, uint32_t batch, const float* x, uint32_t m,
                      uint32_t x_row_stride, uint32_t x_batch_stride, float* y,
                      uint32_t y_row_stride, uint32_t y_batch_stride, uint32_t split, void* stream);

/*
 * rem_dequantize_affine -- exact F32 weights out[r, :] of `rows` affine rows
 * (test hook, as rem_dequantize): w = fl(fl(scale*q) + bias).
 */
int rem_dequantize_affine(const void* codes, const uint16_t* scales, const uint16_t* biases, int wtype,
                          uint32_t rows, uint32_t k, float* out, void* stream);

/*
 * rem_matvec_many -- the same product for any number of input rows m >= 1,
 * the first of the next steps past the few-row limit (ROW_EXACT_MATVEC_MAX_ROWS
 * in row_exact_matvec.rs caps one dispatch at 8 rows; the matrix-vector regime
 * extends further, cf. qmv_batch_limit in nuvec-core 0.6.0 src/gpu.rs).  The
 * m input rows run in groups, one launch per group, each reading W once:
 * groups of up to 32 rows on the tensor-core engine (16 for Q6_K), of up to
 * REM_MAX_ROWS on the SIMT engine.  Rows are independent, so row j is bitwise the
 * row an m = 1 call with the same split and engine produces.
 *
 *   Arguments as rem_matvec_ex (strides in elements, split 0 = automatic from
 *   (wtype, batch*n, k)) without rows_per_cta.  The output rules apply to all
 *   m rows; every group is validated before the first launch, so an argument
 *   error writes nothing.  A CUDA error in a later group leaves the earlier
 *   groups written.
 */
int rem_matvec_many(const void* W, int wtype, uint32_t n, uint32_t k, uint32_t batch,
                    const float* x, uint32_t m, uint32_t x_row_stride, uint32_t x_batch_stride,
                    float* y, uint32_t y_row_stride, uint32_t y_batch_stride,
                    uint32_t split, void* stream);

/*
 * rem_matvec_sched -- the product for any m >= 1 with an explicit schedule
 * (NULL = all defaults).  Arguments as rem_matvec_many; the input rows run in
 * launches of up to 8 rows (SIMT engine) or 32 rows (tensor-core engine;
 * 16 for Q6_K),
 * each reading W once, all checked before the first launch.
 * Returns REM_EINVAL for a schedule field out of range, for the tensor-core
 * engine on a format it does not take, and for the argument errors of
 * rem_matvec_ex.
 */
int rem_matvec_sched(const void* W, int wtype, uint32_t n, uint32_t k, uint32_t batch,
                     const float* x, uint32_t m, uint32_t x_row_stride, uint32_t x_batch_stride,
                     float* y, uint32_t y_row_stride, uint32_t y_batch_stride,
                     const rem_schedule* sched, void* stream);

/*
 * rem_set_thread_schedule -- schedule defaults for every later call of the
 * calling thread (NULL: back to the library's defaults).  The fields mean
 * what they mean in rem_schedule; an explicit split or rows_per_cta argument
 * and the set fields of rem_matvec_sched's schedule take precedence.  Meant
 * for tests and tuning (pinning a lane layout or an engine); it changes no
 * other thread.  REM_EINVAL for a field out of range.  Host only.
 */
int rem_set_thread_schedule(const rem_schedule* sched);

/*
 * rem_engine_of -- the engine the default schedule uses for `rows`
 * (= batch*n) weight rows of k elements: REM_ENGINE_TC for Q6_K (whose
 * sub-block decode is the costliest on the FP32 pipe), REM_ENGINE_SIMT
 * otherwise (Q8_0 and Q5_0 take the tensor-core engine only when a schedule
 * asks for it); -1 for an unknown wtype or rows == 0 or k == 0.  Host only;
 * makes no CUDA call.
 */
int rem_engine_of(int wtype, uint32_t rows, uint32_t k);

/*
 * rem_device_status -- REM_OK, or REM_ECUDA (with a message) if a kernel of
 * this library on the current device gave up on a bounded wait since the
 * status was last cleared; `clear` != 0 clears it.  Synchronous (it reads a
 * word of device memory); not for the hot path.
 */
int rem_device_status(int clear);

/*
 * rem_row_bytes -- bytes of one weight row of k elements
 * (RowExactWeight::row_bytes): F16 2k, Q8_0 k/32*34, Q4_K k/256*144,
 * Q6_K k/256*210, Q5_0 k/32*22; F32 4k, BF16 2k.  Returns 0 for an unknown
 * wtype.  Host only.
 */
uint64_t rem_row_bytes(int wtype, uint32_t k);

/*
 * rem_split_factor -- the split factor rem_matvec uses for a weight of
 * `rows` (= batch*n) rows of k elements (the analogue of
 * row_exact_reduction_nsg followed by the device cap of
 * RowExactMatvecSchedule::for_device).  It depends on (wtype, rows, k) only:
 * a power of two so that rows/32 * split reaches about 2048, at most the
 * number of chunks of a row (72 F16 or BF16 values, 36 F32 values, 4 Q8_0
 * blocks, 8 Q5_0 blocks, one Q4_K / Q6_K super-block) and at most REM_MAX_CLUSTER_SPLIT (8): the
 * split ranges of a row run as the thread blocks of one cluster, and 8 is
 * the portable cluster size (the page's device cap on threads per
 * threadgroup becomes this cap).  Returns 0 for an unknown wtype or
 * rows == 0 or k == 0.  Host only; makes no CUDA call.
 */
uint32_t rem_split_factor(int wtype, uint32_t rows, uint32_t k);

/*
 * rem_dequantize -- exact F32 weights out[r, :] of `rows` weight rows
 * (test hook for bit-exact decode checks).  Element values:
 *   F16  the binary16 value;   Q8_0  d*q;   Q5_0  d*(q-16);
 *   Q4_K (d*sc)*q - dmin*mn;   Q6_K  (d*sc)*(q-32)
 * each product and the difference separately rounded to nearest even.
 * W as for rem_matvec; out is a device F32 buffer of rows*k elements,
 * 4-byte aligned.  Async on `stream`.
 */
int rem_dequantize(const void* W, int wtype, uint32_t rows, uint32_t k, float* out, void* stream);

/*
 * rem_quantize -- quantize F32 rows src[r, :] (device, rows*k elements,
 * 4-byte aligned) into `rows` weight rows at W (device, alignment as for
 * rem_matvec).  Round-to-nearest quantizers with fp16 scales: Q8_0
 * d = amax/127; Q5_0 d = vmax/-16; Q4_K 6-bit sub-block scales and mins;
 * Q6_K int8 sub-block scales; F16 rounds to nearest even.  Codes are
 * roundf of x over the stored scale.  Async on `stream`.
 */
int rem_quantize(const float* src, int wtype, uint32_t rows, uint32_t k, void* W, void* stream);

/* Thread-local message of the last failing call on this thread ("" if none). */
const char* rem_last_error(void);

/* Thread-local one-line description of the last launch on this thread
   (engine, split, layout, stages, grid, ...; "" before the first). */
const char* rem_last_plan(void);

/* ABI version of this header (incremented on incompatible changes; 2: the
   schedule struct replaces the environment pin of the lane layout). */
int rem_version(void);

#ifdef __cplusplus
}
#endif

#endif /* REM_H */
