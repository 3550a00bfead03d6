/*
 * mxfp4.h -- C ABI of the GB300 (sm_103a) H16/H32 + MXFP4 linear-layer GEMM library
 * (libmxfp4.so).
 *
 * What it computes (cited by web-page title and section):
 *   "Pretraining Large Language Models with MXFP4 on Native FP4 Hardware"
 *     - A.1 "MXFP4 and micro-scaling": a block of 32 values shares one power-of-two
 *       scale 2^E and each element is rounded to the nearest FP4 (E2M1) value:
 *       x_B ~ 2^E * Q_FP4(x_B / 2^E).
 *     - A.2 "Hadamard transform architecture": a deterministic, tiled (block-
 *       diagonal) 16x16 Hadamard rotation is applied before every MXFP4 GEMM.
 *     - C.1-C.3: the rotation is applied along each GEMM's contraction dimension, so
 *       it cancels: Y = (XH)(WH)^T = XW^T, dX = (dY H)(W^T H)^T = dY W,
 *       dW = (dY^T H)(X^T H)^T = dY^T X.
 *     - D "1D and 2D quantisation strategies": 1x32 row-wise, 32x1 column-wise
 *       (needs a transpose) and 32x32 2D block scales.
 *   "Decomposing MXFP4 quantization error for LLM reinforcement learning"
 *     - E8M0 scales (powers of two only) and the E2M1 grid
 *       {0, +-0.5, +-1, +-1.5, +-2, +-3, +-4, +-6}; the ceiling scale (never below
 *       amax/6); W4A4 QDQ numerics = same grid, same E8M0 scale, FP32 accumulation.
 *
 * Conventions shared by every entry point
 *   - Ownership: the caller owns every buffer (inputs, quantised tensors, outputs,
 *     workspace).  The library allocates no memory; its only global state is one
 *     device status word per device (see mxfp4_device_status).
 *   - Asynchrony: every compute call validates its arguments on the host, then
 *     enqueues kernels on `stream` and returns without synchronising.  Pointers
 *     marked "device" must be device-accessible memory of the current device.
 *   - Validation: invalid arguments return an error status WITHOUT launching
 *     anything.  A thread-local message describing the last error is available
 *     from mxfp4_last_error().
 *   - Numbers: inputs are finite bf16 with |x| < 2^123.  Non-finite inputs give
 *     unspecified codes but never a fault or hang.
 *   - Packed FP4: element 2j in the low nibble of byte j, element 2j+1 in the high
 *     nibble; code bit 3 = sign, bits 0-2 index {0, .5, 1, 1.5, 2, 3, 4, 6}.
 *   - E8M0: byte b means 2^(b-127); this library produces 0 <= b <= 253.
 */
#ifndef MXFP4_H
#define MXFP4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* mxfp4_stream_t;

typedef enum {
    MXFP4_OK = 0,
    MXFP4_ERR_INVALID_ARG = 1,       /* null pointer, bad enum, negative size          */
    MXFP4_ERR_UNSUPPORTED_SHAPE = 2, /* a quantised dim not a multiple of 32, ...     */
    MXFP4_ERR_MISALIGNED = 3,        /* pointer not 16-byte aligned, ld % 8 != 0      */
    MXFP4_ERR_WORKSPACE = 4,         /* workspace null or smaller than required        */
    MXFP4_ERR_CUDA = 5,              /* a CUDA runtime/driver call or launch failed    */
    MXFP4_ERR_TIMEOUT = 6,           /* a bounded device-side wait expired             */
    MXFP4_ERR_UNSUPPORTED_DEVICE = 7 /* the current device is not sm_103 (GB300)       */
} mxfp4_status;

typedef enum { MXFP4_HAD_NONE = 0, MXFP4_HAD_16 = 16, MXFP4_HAD_32 = 32 } mxfp4_hadamard;

/* FLOOR_OCP: e = floor(log2 amax) - 2 (OCP MX rule).  CEIL: smallest e with
 * 6 * 2^e >= amax.  Both clamped to the E8M0 range; amax == 0 gives e = -127. */
typedef enum { MXFP4_SCALE_FLOOR_OCP = 0, MXFP4_SCALE_CEIL = 1 } mxfp4_scale_mode;

/* Layout bitmask for mxfp4_rotate_quantize. */
enum { MXFP4_LAYOUT_ROW = 1, MXFP4_LAYOUT_COLT = 2, MXFP4_LAYOUT_2D = 4 };

typedef enum { MXFP4_OUT_F32 = 0, MXFP4_OUT_BF16 = 1 } mxfp4_out_dtype;

/* Scale-factor storage.
 *   PLAIN: row-major [rows][cols/32] bytes (2D layout: [rows/32][cols/32]).
 *   MMA:   the tile order the tensor cores read.  rows are padded to a multiple of
 *          128 and the 32-element blocks per row (kb = cols/32) to a multiple of 8;
 *          padding bytes are written as 0.  The byte for (row r, block k) is at
 *            ((r/128) * (kb_pad/4) + k/4) * 512 + (r%32) * 16 + ((r/32)%4) * 4 + k%4.
 *          Only MMA-layout tensors can feed mxfp4_gemm. */
typedef enum { MXFP4_SF_PLAIN = 0, MXFP4_SF_MMA = 1 } mxfp4_sf_layout;

/* A quantised matrix of `rows` x `cols` logical elements, quantised in blocks of 32
 * along `cols` (the contraction dimension of the GEMM that consumes it).  For the
 * column-transposed copy of an [R, C] input the stored matrix is [C, R].
 *   codes:  device, rows * cols / 2 bytes, row-major (row pitch cols/2 bytes),
 *           16-byte aligned.
 *   scales: device, mxfp4_scales_bytes(rows, cols, layout, sf_layout) bytes,
 *           16-byte aligned.
 * mxfp4_rotate_quantize fills rows, cols, layout, had and mode; the caller sets
 * codes, scales and sf_layout. */
typedef struct {
    void* codes;
    uint8_t* scales;
    int64_t rows;
    int64_t cols;
    int32_t layout;    /* one MXFP4_LAYOUT_* value */
    int32_t sf_layout; /* mxfp4_sf_layout */
    int32_t had;       /* mxfp4_hadamard used when it was produced */
    int32_t mode;      /* mxfp4_scale_mode used when it was produced */
} mxfp4_tensor;

typedef struct {
    int32_t had;        /* mxfp4_hadamard */
    int32_t mode;       /* mxfp4_scale_mode */
    int32_t out_dtype;  /* mxfp4_out_dtype of the GEMM output */
    int32_t accumulate; /* 1: C += result (fp32 output only); 0: C = result */
} mxfp4_config;

enum { MXFP4_OP_FPROP = 0, MXFP4_OP_DGRAD = 1, MXFP4_OP_WGRAD = 2, MXFP4_OP_BACKWARD = 3 };

/* Bytes of packed codes for a rows x cols quantised matrix. */
size_t mxfp4_codes_bytes(int64_t rows, int64_t cols);
/* Bytes of scale factors for a rows x cols quantised matrix in the given layout
 * (MXFP4_LAYOUT_*) and scale-factor storage (mxfp4_sf_layout); 0 if invalid. */
size_t mxfp4_scales_bytes(int64_t rows, int64_t cols, int layout, int sf_layout);
/* codes bytes rounded up to 256 plus scales bytes rounded up to 256: the size of
 * one quantised tensor when both live in one buffer (codes first). */
size_t mxfp4_quantized_bytes(int64_t rows, int64_t cols, int layout, int sf_layout);

/* Fused rotate + quantise ("Pretraining ... Native FP4 Hardware", A.1, A.2, D).
 * x: device bf16 [rows, cols], leading dimension ld >= cols elements (ld % 8 == 0,
 *    x 16-byte aligned).  Read once.
 * had, mode: rotation (applied along the quantised dimension of each output, in
 *    contiguous blocks starting at index 0) and scale rule.
 * layouts: bitmask of MXFP4_LAYOUT_*; ROW and COLT may be combined (one pass emits
 *    both), 2D is produced on its own.
 *    ROW:  row_out  = [rows, cols], rotated/quantised along cols (needs cols % 32 == 0)
 *    COLT: colT_out = [cols, rows], column j of x rotated/quantised along rows
 *          (needs rows % 32 == 0 and cols % 32 == 0)
 *    2D:   twoD_out = [rows, cols], rotated along cols, one scale per 32x32 tile
 *          (needs rows % 32 == 0, cols % 32 == 0; PLAIN scales only)
 * Outputs not requested may be NULL.
 * The rotation is evaluated in fp32 in the Sylvester order (stage strides 1, 2, 4,
 * 8 (, 16), every add rounded) and multiplied by fl32(1/sqrt(n)); rounding to E2M1
 * is to nearest, ties to even, saturating at +-6, sign of zero kept. */
mxfp4_status mxfp4_rotate_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld, int had, int mode,
                                   unsigned layouts, mxfp4_tensor* row_out, mxfp4_tensor* colT_out,
                                   mxfp4_tensor* twoD_out, mxfp4_stream_t stream);

/* Two matrices with the same number of columns -- a GEMM's two operands, which share
 * the contraction dimension (Fprop's X [M, K] and W [N, K]) -- rotated and quantised
 * in ONE launch, each exactly as mxfp4_rotate_quantize would (same had, mode and
 * layouts for both; ROW, COLT or both, no 2D).  One launch spares the smaller matrix
 * its own ramp-up and partly filled last wave.
 * a: device bf16 [a_rows, cols] (leading dimension a_ld); b: [b_rows, cols] (b_ld);
 * both under the rules of mxfp4_rotate_quantize.  Outputs as there: a_row / b_row for
 * ROW, a_colT ([cols, a_rows]) / b_colT for COLT; outputs not requested may be NULL.
 * Validation of both matrices and all outputs precedes the launch. */
mxfp4_status mxfp4_rotate_quantize_pair(const void* a, int64_t a_rows, int64_t a_ld, const void* b, int64_t b_rows,
                                        int64_t b_ld, int64_t cols, int had, int mode, unsigned layouts,
                                        mxfp4_tensor* a_row, mxfp4_tensor* a_colT, mxfp4_tensor* b_row,
                                        mxfp4_tensor* b_colT, mxfp4_stream_t stream);

/* Block-scaled MXFP4 GEMM C = A . B^T with FP32 accumulation on the tcgen05 tensor
 * cores (QDQ numerics: "Decomposing MXFP4 quantization error", experiments).
 * A: [M, K] quantised along K, B: [N, K] quantised along K, both MXFP4_SF_MMA,
 *    same K (cols).
 * Provenance (MXFP4_ERR_INVALID_ARG otherwise): A and B carry the same `had` and
 *    `mode` -- the rotations cancel only when both sides of the contraction were
 *    rotated by the same H (C.1-C.3) -- and each is a ROW or COLT copy, with a COLT
 *    A only beside a COLT B.  The linear layer's pairs are (ROW, ROW) in Fprop,
 *    (ROW, COLT) in Dgrad and (COLT, COLT) in Wgrad.
 * C: device, [M, N] row-major with leading dimension ldc >= N (ldc % 8 == 0,
 *    16-byte aligned), fp32 or bf16 per out_dtype.  accumulate = 1 adds to C
 *    (fp32 only).
 * ws/ws_bytes: unused by this kernel (pass NULL/0); reserved for split-K. */
mxfp4_status mxfp4_gemm(const mxfp4_tensor* A, const mxfp4_tensor* B, void* C, int64_t ldc, int out_dtype,
                        int accumulate, void* ws, size_t ws_bytes, mxfp4_stream_t stream);

/* One problem of mxfp4_gemm_group: C = A . B^T with the rules of mxfp4_gemm. */
typedef struct {
    const mxfp4_tensor* A;
    const mxfp4_tensor* B;
    void* C;
    int64_t ldc;
    int32_t out_dtype;  /* mxfp4_out_dtype */
    int32_t accumulate; /* 1: C += A . B^T (fp32 output only) */
} mxfp4_gemm_desc;

/* 1 to 8 independent GEMMs in ONE persistent launch of the CTA-pair kernel: their
 * 256 x 256 output tiles form one schedule, so the problems share the launch's fixed
 * costs (set-up, pipeline fill, last-tile drain) and fill one another's partly used
 * last waves.  The linear layer's backward is such a pair (Dgrad and Wgrad, "Pretraining
 * ... Native FP4 Hardware" C.2-C.3; both read only quantised copies made beforehand), and
 * so are projections that read the same input (q, k, v of attention).
 * Every problem follows mxfp4_gemm's rules and is checked before anything is launched;
 * no two outputs may share a byte (MXFP4_ERR_INVALID_ARG).  Each output equals what
 * mxfp4_gemm computes for that problem with the CTA-pair kernel (M > 128 and N > 128),
 * bit for bit; narrower problems also run on the pair kernel here.  A group of one is
 * exactly mxfp4_gemm. */
mxfp4_status mxfp4_gemm_group(const mxfp4_gemm_desc* descs, int count, mxfp4_stream_t stream);

/* Error-decomposition measurement ("Decomposing MXFP4 quantization error for LLM
 * reinforcement learning", core insight and property 1).  x: device bf16 [rows, cols]
 * (ld elements, cols % 32 == 0), rotated along cols with `had` and quantised row-wise
 * with scale rule `mode`, as mxfp4_rotate_quantize does.  Per 32-block, with s_b the
 * E8M0 scale and s* = amax/6 the ideal scale, Q = s_b*grid(x/s_b), Q* = s*·grid(x/s*):
 *   e_scale = Q - Q*, e_DZ = Q* - x where |x| < amax/24 (the deadzone), e_grid = Q* - x
 *   elsewhere.
 * out: device, 7 doubles (8-byte aligned), overwritten with the tensor-wide sums
 *   [sum e^2, sum e_scale^2, sum e_DZ^2, sum e_grid^2, sum e_scale*e_grid,
 *    deadzone count, element count].
 * Under the ceiling scale, sum e^2 = scale2 + dz2 + grid2 + 2*scale_grid (property 1).
 * fp64 sums are accumulated atomically, so the last bits depend on the order. */
mxfp4_status mxfp4_error_decomposition(const void* x, int64_t rows, int64_t cols, int64_t ld, int had, int mode,
                                       double* out, mxfp4_stream_t stream);

/* Tensor-core peak probe (measurement helper, synchronous): every SM issues `iters`
 * back-to-back M=128 N=256 tcgen05.mma instructions on operands resident in shared
 * memory, and *tflops receives the dense rate.  kind 0: kind::mxf4 (E2M1, UE8M0 per
 * 32, the GEMM's instruction); 1: kind::mxf4nvf4 with the same 2X UE8M0 scaling;
 * 2: kind::f16 with bf16 operands (calibration); 3: kind::mxf4nvf4 scale_vec::4X with
 * UE4M3 scales per 16 (the NVFP4 form, for comparison only); 4: kind::mxf4 issued by CTA
 * pairs (.cta_group::2, M = 256 per pair).  Allocates no global memory. */
mxfp4_status mxfp4_mma_peak_probe(int kind, int64_t iters, double* tflops);

/* Quantiser fixes of "Decomposing MXFP4 quantization error for LLM reinforcement
 * learning" (sections MBS and OF), row layout only: x [rows, cols] bf16 (ld elements per
 * row, 16-byte aligned, ld % 8 == 0) is rotated along cols exactly as by
 * mxfp4_rotate_quantize (had, mode as there).  Output descriptors are filled in like
 * row_out of mxfp4_rotate_quantize (codes, scales, sf_layout set by the caller; the
 * library writes rows, cols, layout, had, mode).  Asynchronous on `stream`.
 *
 * Outlier fallback (OF): q1 = Q(v) and q2 = Q(v - dq(q1)), the residual being exact in
 * fp32.  The residual weight alpha = 2^alpha_log2 (alpha_log2 in [-8, 0]; the pages use
 * 0.5) is carried by q2's E8M0 bytes: stored byte = max(byte + alpha_log2, 0), so the
 * OF value is dq(q1) + dq(q2) and both tensors feed mxfp4_gemm unchanged (a GEMM over
 * an OF operand is two accumulating GEMMs).  cols % 32 == 0. */
mxfp4_status mxfp4_rotate_quantize_of(const void* x, int64_t rows, int64_t cols, int64_t ld, int had, int mode,
                                      int alpha_log2, mxfp4_tensor* q1, mxfp4_tensor* q2, mxfp4_stream_t stream);

/* Macro-block scaling (MBS): per 128 consecutive rotated values of a row one byte k,
 * the largest value with (1 + k/256) * f <= T for the macro-block amax A = f * 2^E
 * (T = 1.5 if f <= 1.5, else 3; A zero or subnormal gives k = 0).  The values are
 * prescaled to fl32((1 + k/256) v) and quantised to q; the reconstruction is
 * dq(q) / (1 + k/256).  mbs: device bytes [rows, cols/128], row-major, written by the
 * call.  The post-scale varies along the contraction: mxfp4_gemm_mbs applies it per
 * macro block (mxfp4_gemm does not).  cols % 128 == 0. */
mxfp4_status mxfp4_rotate_quantize_mbs(const void* x, int64_t rows, int64_t cols, int64_t ld, int had, int mode,
                                       mxfp4_tensor* q, uint8_t* mbs, mxfp4_stream_t stream);

/* GEMM over macro-block-scaled operands ("Decomposing MXFP4 quantization error ...",
 * MBS: x_hat = Q((1 + m) x) / (1 + m)): C = x_hat_A . x_hat_B^T, i.e. for each macro
 * block kb of 128 elements along K the MXFP4 partial product P_kb (fp32 on the tensor
 * cores) is scaled by f_A[m][kb] f_B[n][kb], f = 256 / (256 + byte) computed in fp32,
 * and the scaled partials are summed in fp32.  The page says the postscale fuses into
 * the GEMM epilogue; it can as one factor only when it is constant along K, and here it
 * changes every 128 elements of K, so each partial is scaled as it leaves the tensor
 * cores instead.
 * A, B, C, ldc, out_dtype, accumulate: as for mxfp4_gemm (A and B from
 * mxfp4_rotate_quantize_mbs or any row-quantised copy).  mbs_a: device bytes
 * [M, K/128] row-major (the `mbs` output of mxfp4_rotate_quantize_mbs), or NULL for
 * a plain MXFP4 A (factor 1); mbs_b likewise [N, K/128].  K % 128 == 0 and
 * K <= 16384 (MXFP4_ERR_UNSUPPORTED_SHAPE otherwise).  Runs 128 x 128 single-CTA
 * tiles; within the GEMM tolerance of the oracle's fp64 product of the reconstructions. */
mxfp4_status mxfp4_gemm_mbs(const mxfp4_tensor* A, const uint8_t* mbs_a, const mxfp4_tensor* B, const uint8_t* mbs_b,
                            void* C, int64_t ldc, int out_dtype, int accumulate, mxfp4_stream_t stream);

/* Randomised quantiser baselines of "Pretraining Large Language Models with MXFP4 on
 * Native FP4 Hardware" (A.2: random sign flips before the Hadamard; the
 * stochastic-rounding runs of the ablation).  The random numbers are inputs, owned by
 * the caller, device memory, 16-byte aligned; NULL disables an option:
 *   col_signs: bitmask of ceil(cols/8) bytes (bit i of byte i/8 = column i): column i is
 *              negated before the rotation along cols (row copy).  A GEMM's two
 *              operands must use the same mask over their shared contraction.
 *   row_signs: bitmask over rows, for the rotation along rows (transposed copy).
 *   sr_row:    uint16 [rows, cols] row-major, uniform integers: stochastic rounding of
 *              the row copy.  A magnitude a in [lo, lo + step) of the E2M1 grid rounds
 *              up iff r < ((a - lo) / step) * 65536; a >= 6 saturates; the sign is
 *              kept.  The E8M0 scales are those of `mode`.
 *   sr_colT:   uint16 [cols, rows] for the transposed copy.
 * Stochastic rounding is on for a call when any requested layout has its array, and
 * then every requested layout needs one. */
typedef struct {
    const uint8_t* col_signs;
    const uint8_t* row_signs;
    const uint16_t* sr_row;
    const uint16_t* sr_colT;
} mxfp4_quant_opts;

/* mxfp4_rotate_quantize with the options above (layouts ROW, COLT or both; the 2D
 * layout returns MXFP4_ERR_UNSUPPORTED_SHAPE when an option is set).  opts == NULL or
 * all-NULL gives exactly mxfp4_rotate_quantize. */
mxfp4_status mxfp4_rotate_quantize_ex(const void* x, int64_t rows, int64_t cols, int64_t ld, int had, int mode,
                                      unsigned layouts, const mxfp4_quant_opts* opts, mxfp4_tensor* row_out,
                                      mxfp4_tensor* colT_out, mxfp4_tensor* twoD_out, mxfp4_stream_t stream);

/* The randomised baselines with their random numbers drawn in the kernel from
 * Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as easy as
 * 1, 2, 3", SC'11), a counter-based generator: nothing random is read from memory, and
 * every number is a fixed function of (seed, counter), so a run can be replayed.
 *   col_signs: 1 negates column j (row copy) when bit j of the sign vector of seed
 *     col_sign_seed is set -- bit j % 32 of output word (j % 128) / 32 of
 *     Philox(counter (j / 128, 0, 0, 0), key (seed low 32 bits, seed high 32 bits)).
 *     The sign vector belongs to a dimension: a GEMM's two operands must use the same
 *     seed for their shared contraction (X's and W's columns: K; W's rows and dY's
 *     columns: N; X's and dY's rows: M) so that the rotation still cancels.
 *   row_signs: the same over the rows (transposed copy), seed row_sign_seed.
 *   stochastic_rounding: the rule of mxfp4_quant_opts with the 16-bit integer of
 *     (line l, position i) of the stored copy (row copy: l = row, i = column; transposed
 *     copy: l = column, i = row) taken as half i % 8 (word (i % 8) / 2, low half
 *     first) of Philox(counter (i / 8, l, copy, 0), key (sr_seed low, sr_seed high)),
 *     copy = 0 for the row copy and 1 for the transposed copy.
 * With the same numbers, the result equals mxfp4_rotate_quantize_ex given those numbers
 * as arrays.  reserved must be 0. */
typedef struct {
    uint64_t col_sign_seed;
    uint64_t row_sign_seed;
    uint64_t sr_seed;
    int32_t col_signs;
    int32_t row_signs;
    int32_t stochastic_rounding;
    int32_t reserved;
} mxfp4_philox_opts;

/* mxfp4_rotate_quantize (ROW, COLT or both) with in-kernel Philox random signs and/or
 * stochastic rounding as set in opts (every option 0: exactly mxfp4_rotate_quantize). */
mxfp4_status mxfp4_rotate_quantize_philox(const void* x, int64_t rows, int64_t cols, int64_t ld, int had, int mode,
                                          unsigned layouts, const mxfp4_philox_opts* opts, mxfp4_tensor* row_out,
                                          mxfp4_tensor* colT_out, mxfp4_stream_t stream);

/* Workspace bytes needed by mxfp4_linear_{fprop,dgrad,wgrad} (op = MXFP4_OP_*). */
size_t mxfp4_workspace_bytes(int op, int64_t M, int64_t N, int64_t K, const mxfp4_config* cfg);

/* Fprop Y = X W^T ("Pretraining ... Native FP4 Hardware", C.1).
 * x: device bf16 [M, K] (ld K), w: device bf16 [N, K] (ld K), y: device [M, N] (ld N)
 * in cfg->out_dtype.  Both operands are rotated and quantised along K (row layout)
 * into the workspace (256-byte aligned, mxfp4_workspace_bytes bytes), then multiplied.
 * save_xT (optional, NULL to skip): receives X^T quantised along M, [K, M], the Wgrad
 *    operand (needs M % 32 == 0); produced in the same pass that reads X.
 * save_wT (optional): receives W^T quantised along N, [K, N], the Dgrad operand
 *    (needs N % 32 == 0); produced in the same pass that reads W.
 * Saved tensors must be MXFP4_SF_MMA.  K % 32 == 0, N % 8 == 0 (y's leading dimension).
 * X and W are quantised in one launch (as by mxfp4_rotate_quantize_pair) when both
 * transposed copies, or neither, are requested.
 * Every argument of both quantiser passes and of the GEMM is checked before the first
 * launch: a rejected call leaves the workspace, the saved copies and y untouched. */
mxfp4_status mxfp4_linear_fprop(const void* x, const void* w, int64_t M, int64_t N, int64_t K,
                                const mxfp4_config* cfg, void* y, mxfp4_tensor* save_xT, mxfp4_tensor* save_wT,
                                void* ws, size_t ws_bytes, mxfp4_stream_t stream);

/* Dgrad dX = dY W ("Pretraining ... Native FP4 Hardware", C.2).
 * dy: device bf16 [M, N] (ld N); wT: W^T quantised along N ([K, N], from
 * mxfp4_linear_fprop's save_wT); dx: device [M, K] (ld K).  dY is rotated and
 * quantised along N (row layout) into the workspace.
 * save_dyT (optional): receives dY^T quantised along M, [N, M], the Wgrad operand
 *    (needs M % 32 == 0).  N % 32 == 0, K % 8 == 0 (dx's leading dimension).
 * wT must be a COLT copy made under cfg's had and mode (MXFP4_ERR_INVALID_ARG
 * otherwise): W's row copy has the same shape when W is square, and a copy under
 * another rotation would not cancel.  Everything is checked before the first launch. */
mxfp4_status mxfp4_linear_dgrad(const void* dy, const mxfp4_tensor* wT, int64_t M, int64_t N, int64_t K,
                                const mxfp4_config* cfg, void* dx, mxfp4_tensor* save_dyT, void* ws,
                                size_t ws_bytes, mxfp4_stream_t stream);

/* Wgrad dW = dY^T X ("Pretraining ... Native FP4 Hardware", C.3), contraction over
 * the M tokens.  dyT: [N, M], xT: [K, M] (both quantised along M, MMA scales);
 * dw: device [N, K] (ld K) in cfg->out_dtype; cfg->accumulate adds to dw.
 * dyT and xT must both be COLT copies made under cfg's had and mode
 * (MXFP4_ERR_INVALID_ARG otherwise). */
mxfp4_status mxfp4_linear_wgrad(const mxfp4_tensor* dyT, const mxfp4_tensor* xT, const mxfp4_config* cfg,
                                void* dw, void* ws, size_t ws_bytes, mxfp4_stream_t stream);

/* The whole backward of a linear layer ("Pretraining ... Native FP4 Hardware", C.2 and
 * C.3): dY [M, N] bf16 (ld N) is rotated and quantised once, along N (row copy, the
 * Dgrad operand) and along M (transposed copy, the Wgrad operand), into the workspace
 * (mxfp4_workspace_bytes(MXFP4_OP_BACKWARD, ...)); then Dgrad dX = dY W and Wgrad
 * dW = dY^T X run as ONE grouped launch (mxfp4_gemm_group).
 * wT: [K, N] and xT: [K, M], the COLT copies saved by mxfp4_linear_fprop, made under
 * cfg's had and mode.  dx: device [M, K] (ld K) in cfg->out_dtype, overwritten.
 * dw: device fp32 [N, K] (ld K), overwritten, or added to when cfg->accumulate
 * (gradient accumulation).  M % 32 == 0, N % 32 == 0.  Everything is checked before
 * the first launch.  Outputs equal mxfp4_linear_dgrad + mxfp4_linear_wgrad bit for bit
 * where those run on the CTA-pair kernel (M, N, K > 128). */
mxfp4_status mxfp4_linear_backward(const void* dy, const mxfp4_tensor* wT, const mxfp4_tensor* xT, int64_t M,
                                   int64_t N, int64_t K, const mxfp4_config* cfg, void* dx, void* dw, void* ws,
                                   size_t ws_bytes, mxfp4_stream_t stream);

/* Fprop without caller-provided scratch.  The pages have no counterpart: this entry
 * exists for callers that cannot allocate device memory -- a plugin inside a host
 * framework whose allocator owns all device memory and passes it only input and
 * output pointers, or a latency-critical loop that must not call cudaMalloc or
 * cudaFree (they can synchronise the device).
 * Same arguments, results and validation as mxfp4_linear_fprop, minus ws/ws_bytes:
 * the quantised X and W live in a fixed 64 MiB scratch area inside the library
 * (mxfp4_noalloc_scratch_bytes()), which every GPU running this library holds until
 * the process exits.  Shapes whose mxfp4_workspace_bytes(MXFP4_OP_FPROP, ...) exceed
 * it are rejected with MXFP4_ERR_WORKSPACE before anything is launched.
 * The 64 MiB is reserved by the CUDA driver when the library's device code is loaded
 * on a device: at library load under eager module loading, or -- under the default
 * lazy loading -- on this entry point's first call on that device, which also looks
 * up the area's device address.  That first call can therefore fail with
 * MXFP4_ERR_CUDA (out of memory) or synchronise the device: make it at
 * initialisation, before the caller's allocator reserves the device's memory and
 * before any stream capture.
 * All calls share the one area and it keeps the previous call's contents (every
 * byte this path reads is rewritten first); calls that may overlap on the GPU (for
 * example on two streams without ordering) race on it and must be serialised.
 * Nothing here calls cudaMalloc, cudaFree or any allocating library routine. */
mxfp4_status mxfp4_linear_fprop_noalloc(const void* x, const void* w, int64_t M, int64_t N, int64_t K,
                                        const mxfp4_config* cfg, void* y, mxfp4_tensor* save_xT,
                                        mxfp4_tensor* save_wT, mxfp4_stream_t stream);
/* Size in bytes of the scratch area used by mxfp4_linear_fprop_noalloc. */
size_t mxfp4_noalloc_scratch_bytes(void);

/* Synchronises `stream`, then returns and clears the current device's status word:
 * MXFP4_OK, MXFP4_ERR_TIMEOUT if a kernel's bounded wait expired since the last call,
 * or MXFP4_ERR_CUDA if a GEMM kernel found its shared memory misaligned for its tile
 * layout.  In both error cases that kernel returned early and its output is invalid. */
mxfp4_status mxfp4_device_status(mxfp4_stream_t stream);

/* Bounded-wait limit in nanoseconds for kernels launched afterwards by this host
 * thread (default 2e9 = 2 s; 0 restores the default). */
void mxfp4_set_wait_limit_ns(uint64_t ns);

/* Failure-detection test hook: the next `launches` mxfp4_gemm launches made by this
 * host thread never load their first K stage, so the tensor-core issuer's bounded
 * wait expires; the kernel records MXFP4_ERR_TIMEOUT (read with
 * mxfp4_device_status), drains its copies, frees its TMEM and returns.  Its output
 * is then invalid.  0 cancels.  Not for production use. */
void mxfp4_test_inject_gemm_fault(int launches);

const char* mxfp4_status_string(mxfp4_status status);
/* Message for the last error returned on this host thread ("" if none). */
const char* mxfp4_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MXFP4_H */
