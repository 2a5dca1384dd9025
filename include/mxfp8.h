/*
 * mxfp8.h - C ABI of the GB300 (sm_103a) MXFP8 quantizer and block-scaled GEMMs.
 *
 * The method: "End-to-End MXFP8 RL on Blackwell: What Matching Buys, When It Pays Off,
 * and How It Fails" (verl blog post). Section "The pipeline", paragraph "The format":
 * MXFP8 is the OCP microscaling FP8 format - E4M3 elements in blocks of 32 along the
 * reduction dimension, each block sharing one power-of-two E8M0 scale. The learner
 * paragraph of the same section: each linear layer runs three GEMMs (forward, data
 * gradient, weight gradient) on quantized operands, some quantized along the token
 * dimension, with token counts padded to multiples of 32. The weight-synchronization
 * paragraph: the synced weights are the forward GEMM's weight quantization, byte for
 * byte. Section "Where the time goes": scales are rearranged into the layout the GEMM
 * reads; here the quantizer writes that layout directly.
 *
 * Conventions shared by every call:
 *  - Pointers named *_dev are device pointers; the caller allocates and owns every
 *    buffer. The library allocates no device memory in any call. Its only state is a
 *    per-device status word (see mxfp8_get_device_status) and per-device capability
 *    flags, set up on the first call on each device.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *    Every compute call only enqueues work on `stream` and returns; none synchronizes
 *    except mxfp8_get_device_status. Kernels are launched with programmatic stream
 *    serialization: one may be scheduled while the previous kernel of its stream is
 *    still running, and it waits inside the kernel, before its first read or write of
 *    global memory, until that kernel has completed. Stream order therefore holds as
 *    for a plain launch, against any kernel before it. MXFP8_PDL=0 in the environment
 *    (read once per process) launches them plainly.
 *  - Return value: an mxfp8_status. Arguments are checked on the host before anything
 *    is enqueued; a failed check returns its code and enqueues nothing. Errors found
 *    by a kernel (bad expert offsets, a pipeline wait that ran out) are latched in the
 *    device status word and read with mxfp8_get_device_status. No call throws.
 *  - Matrices are row-major with packed rows (leading dimension = number of columns).
 *    BF16 and E4M3 tensors must start on a 16-byte boundary, scale tensors too.
 *  - Quantization rule (OCP, floor form): per block of 32, e = max(-127,
 *    floor(log2 amax) - 8); scale byte = e + 127; element = E4M3(v * 2^-e), round to
 *    nearest even, saturating at +-448, sign of zero kept. A block holding a NaN or an
 *    infinity gets scale 0xFF and every element 0x7F | (its sign bit).
 *  - Scale layouts. LINEAR: scales [S_rows][S_cols] row-major, one byte per block.
 *    SWIZZLED: the tensor cores' 128 x 4 tiles - byte offset of scale (r, c) is
 *    ((r / 128) * ceil(S_cols / 4) + c / 4) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4
 *    + (c % 4); the padding bytes of partial tiles are written as 0x00. The GEMMs read
 *    SWIZZLED scales only.
 */
#ifndef MXFP8_H_
#define MXFP8_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MXFP8_ABI_VERSION 1

typedef enum mxfp8_status {
  MXFP8_OK = 0,
  MXFP8_ERR_INVALID_ARG = 1,      /* null pointer, negative or unsupported size/enum */
  MXFP8_ERR_ALIGNMENT = 2,        /* a blocked dim not a multiple of 32, or a pointer
                                     not 16-byte aligned */
  MXFP8_ERR_UNSUPPORTED_ARCH = 3, /* current device is not compute capability 10.3 */
  MXFP8_ERR_CUDA = 4,             /* a CUDA runtime/driver call failed */
  MXFP8_ERR_BAD_OFFSETS = 5,      /* (device) expert offsets not 0-based, non-decreasing,
                                     32-aligned and ending at total_rows */
  MXFP8_ERR_TIMEOUT = 6           /* (device) a pipeline wait in a kernel ran out; the
                                     kernel abandoned its work */
} mxfp8_status;

typedef enum mxfp8_axis {
  MXFP8_AXIS_ROW = 0, /* blocks along the contiguous (last) dim: out [rows][cols] */
  MXFP8_AXIS_COL = 1  /* blocks along the first dim, emitted transposed: out [cols][rows] */
} mxfp8_axis;

typedef enum mxfp8_scale_layout {
  MXFP8_SCALES_LINEAR = 0,
  MXFP8_SCALES_SWIZZLED = 1
} mxfp8_scale_layout;

typedef enum mxfp8_scale_rule {
  MXFP8_RULE_FLOOR = 0, /* OCP: e = floor(log2 amax) - 8; the largest elements may saturate */
  MXFP8_RULE_CEIL = 1   /* round-up power of two: smallest e with amax <= 448 * 2^e; never
                           saturates (block-wise FP8 recipes' power-of-two scales) */
} mxfp8_scale_rule;

typedef enum mxfp8_op {
  MXFP8_OP_FPROP = 0, /* Y  = X  . W^T   A = X  rows,  B = W  rows          */
  MXFP8_OP_DGRAD = 1, /* dX = dY . W     A = dY rows,  B = W  cols (= W^T)  */
  MXFP8_OP_WGRAD = 2  /* dW = dY^T . X   A = dY cols,  B = X  cols (tokens) */
} mxfp8_op;

typedef enum mxfp8_out_dtype {
  MXFP8_OUT_BF16 = 0,
  MXFP8_OUT_FP32 = 1
} mxfp8_out_dtype;

/* ABI version of the loaded library (MXFP8_ABI_VERSION). */
int mxfp8_version(void);

/* Static text for a status code; never NULL. */
const char* mxfp8_status_string(int status);

/*
 * Bytes of the scale tensor that mxfp8_quantize writes for a [rows][cols] BF16 input.
 * S_rows x S_cols = rows x cols/32 (ROW) or cols x rows/32 (COL); LINEAR is
 * S_rows * S_cols bytes, SWIZZLED is ceil(S_rows/128) * ceil(S_cols/4) * 512 bytes.
 * Returns 0 for invalid arguments (negative sizes, a blocked dim not a multiple of 32,
 * unknown enums, a size that does not fit in int64).
 */
size_t mxfp8_scale_bytes(int64_t rows, int64_t cols, int axis, int scale_layout);

/*
 * MXFP8-quantize a BF16 matrix ("The pipeline" - "The format"; column-wise copies for
 * the weight-gradient GEMM: the learner paragraph).
 *   src_dev      BF16 [rows][cols], read only.
 *   axis ROW     requires cols % 32 == 0; out_dev E4M3 [rows][cols]; scales for
 *                [rows][cols/32].
 *   axis COL     requires rows % 32 == 0 and cols % 8 == 0; out_dev E4M3 [cols][rows]
 *                (the transpose, blocked along its contiguous dim); scales for
 *                [cols][rows/32].
 *   scales_dev   mxfp8_scale_bytes(rows, cols, axis, scale_layout) bytes, written in
 *                full (padding included).
 * rows == 0 or cols == 0 is a no-op. Deterministic: the same input gives the same bytes
 * from every call, which is what makes the synchronized weights equal the forward
 * weights byte for byte (section "The grid, byte for byte").
 */
int mxfp8_quantize(const void* src_dev, int64_t rows, int64_t cols, int axis,
                   void* out_dev, void* scales_dev, int scale_layout, void* stream);

/*
 * mxfp8_quantize with an explicit scale rule (mxfp8_scale_rule). The pages contrast the
 * MXFP8 grid with block-wise FP8 recipes whose power-of-two scales round the other way
 * (section "A different grid, and drift"); MXFP8_RULE_CEIL produces that grid on the same
 * 1x32 blocks so the two can be compared byte for byte. Bytes differ from the floor rule
 * exactly in blocks whose amax exceeds 448 * 2^e_floor (scale byte one higher there).
 * MXFP8_RULE_FLOOR gives the bytes of mxfp8_quantize.
 */
int mxfp8_quantize_rule(const void* src_dev, int64_t rows, int64_t cols, int axis,
                        void* out_dev, void* scales_dev, int scale_layout, int scale_rule,
                        void* stream);

/*
 * Both copies of one BF16 matrix from a single read of it: the row-wise copy (as
 * mxfp8_quantize ROW) into row_out_dev / row_scales_dev and the column-wise copy (as
 * mxfp8_quantize COL) into col_out_dev / col_scales_dev. The learner needs both for X and
 * dY (forward/dgrad operands blocked along K, wgrad operands blocked along tokens:
 * "The pipeline", learner paragraph). Requires rows % 32 == 0 and cols % 32 == 0. Bytes
 * are identical to the two separate calls.
 */
int mxfp8_quantize_dual(const void* src_dev, int64_t rows, int64_t cols, void* row_out_dev,
                        void* row_scales_dev, void* col_out_dev, void* col_scales_dev,
                        int scale_layout, void* stream);

/*
 * One job of mxfp8_quantize_dual_multi: the arguments of one mxfp8_quantize_dual call.
 * All pointers are device pointers owned by the caller.
 */
typedef struct mxfp8_dual_job {
  const void* src;     /* BF16 [rows][cols] */
  int64_t rows, cols;  /* rows % 32 == 0, cols % 32 == 0 */
  void* row_out;       /* E4M3 [rows][cols] */
  void* row_scales;    /* mxfp8_scale_bytes(rows, cols, MXFP8_AXIS_ROW, layout) bytes */
  void* col_out;       /* E4M3 [cols][rows] */
  void* col_scales;    /* mxfp8_scale_bytes(rows, cols, MXFP8_AXIS_COL, layout) bytes */
} mxfp8_dual_job;

#define MXFP8_MAX_DUAL_JOBS 8

/*
 * Several mxfp8_quantize_dual calls in one launch. The tensors' 128 x 128 tiles form one
 * grid, so a small tensor's partly filled last wave of CTAs is shared with the others
 * instead of running alone. Typical use: a linear layer's activations and weight,
 * quantized together before the forward GEMM. "The pipeline" (learner paragraph) gives
 * the quantized operands; the batching is this library's.
 *   jobs        host array of num_jobs descriptors (1 <= num_jobs <= MXFP8_MAX_DUAL_JOBS),
 *               read during the call only; every job is checked as mxfp8_quantize_dual
 *               checks its arguments, and nothing is launched if one fails. Jobs with
 *               rows == 0 or cols == 0 are skipped.
 * Bytes are identical to one mxfp8_quantize_dual call per job. Outputs of different jobs
 * must not overlap.
 */
int mxfp8_quantize_dual_multi(const mxfp8_dual_job* jobs, int num_jobs, int scale_layout,
                              void* stream);

/* Scale choice of the FP8 block-wise recipe (mxfp8_quantize_blockwise). */
typedef enum {
  MXFP8_BW_SCALE_FP32 = 0, /* quantization factor 448 / amax in single precision */
  MXFP8_BW_SCALE_POW2 = 1  /* power-of-two factor 2^-ceil(log2(amax / 448)) */
} mxfp8_blockwise_scale;

/*
 * Number of float scales mxfp8_quantize_blockwise writes for a [rows][cols] weight:
 * ceil(rows/128) * ceil(cols/128). Returns 0 for invalid arguments, including a count
 * that does not fit in int64.
 */
size_t mxfp8_blockwise_scale_count(int64_t rows, int64_t cols);

/*
 * FP8 block-wise weight quantization, the recipe the pages contrast with MXFP8 ("A
 * different grid, and drift": on Blackwell the block-wise learner must use power-of-two
 * block scales while its sampler uses FP32 scales, so the two sides round the same BF16
 * weight differently; "The pipeline", "The format": TE emulates that recipe with MXFP8
 * GEMMs). One scale per 128 x 128 block (the pages give no block size; 128 x 128 is the
 * block-wise weight recipe's usual one):
 *   amax = max |v| over the block;
 *   s = 448 / amax in IEEE single precision (largest finite float if that overflows),
 *       or 2^-e with e = ceil(log2(amax / 448)) >= -127 for MXFP8_BW_SCALE_POW2;
 *       s = 1 for an all-zero block;
 *   code = E4M3(v * s), the product rounded to single precision, then to nearest even,
 *          saturating at 448;
 *   scale_inv = 1 / s in single precision (exactly 2^e for POW2);
 *   a block holding a NaN or an infinity: scale_inv NaN, codes 0x7F with each sign.
 *   src_dev        BF16 [rows][cols], cols % 8 == 0, 16-byte aligned
 *   out_dev        E4M3 [rows][cols], 16-byte aligned
 *   scale_inv_dev  float [ceil(rows/128)][ceil(cols/128)], 4-byte aligned
 * Errors: MXFP8_ERR_INVALID_ARG (bad scale_type, negative or too large sizes, null
 * pointers), MXFP8_ERR_ALIGNMENT (cols % 8, misaligned pointers).
 */
int mxfp8_quantize_blockwise(const void* src_dev, int64_t rows, int64_t cols, void* out_dev,
                             float* scale_inv_dev, int scale_type, void* stream);

/*
 * `batch` independent matrices [batch][rows][cols] quantized as by mxfp8_quantize, each
 * with its own scale block of mxfp8_scale_bytes(rows, cols, axis, layout) bytes; the
 * scale blocks are concatenated in batch order. Used for per-expert MoE weights.
 */
int mxfp8_quantize_batched(const void* src_dev, int64_t batch, int64_t rows, int64_t cols,
                           int axis, void* out_dev, void* scales_dev, int scale_layout,
                           void* stream);

/*
 * Capacity (bytes) to allocate for the scales of mxfp8_quantize_grouped on a
 * [total_rows][cols] input split into at most num_experts token segments. It is an
 * upper bound that needs no expert counts on the host:
 *   ROW: (ceil(total_rows/128) + num_experts) * ceil(cols/128) * 512
 *   COL: ceil(cols/128) * (ceil(total_rows/128) + num_experts) * 512
 * Returns 0 for invalid arguments, including a size that does not fit in int64.
 */
size_t mxfp8_grouped_scale_bytes(int64_t total_rows, int64_t cols, int num_experts, int axis);

/*
 * MXFP8-quantize a token-segmented (MoE) BF16 matrix [total_rows][cols]; expert e owns
 * rows [off[e], off[e+1]) (section "A held-out workload, and end to end", Table 4).
 *   expert_offsets_dev  int32 [num_experts + 1] on the device: off[0] = 0,
 *                       non-decreasing, multiples of 32, off[E] = total_rows. Checked
 *                       on the device; a violation latches MXFP8_ERR_BAD_OFFSETS and
 *                       the scales are left unspecified.
 *   axis ROW  out_dev [total_rows][cols] (cols % 32 == 0); scales: expert e's SWIZZLED
 *             block for its [cnt_e][cols/32] scales, rows padded to 128.
 *   axis COL  out_dev [cols][total_rows] (cols % 8 == 0); scales: expert e's SWIZZLED
 *             block for its [cols][cnt_e/32] scales, token blocks padded to 4.
 *   Blocks are concatenated in expert order (empty experts take no bytes) inside
 *   scales_dev, whose capacity is mxfp8_grouped_scale_bytes(...); bytes past the last
 *   block are not written. The element bytes equal those of mxfp8_quantize.
 */
int mxfp8_quantize_grouped(const void* src_dev, int64_t total_rows, int64_t cols, int axis,
                           const int32_t* expert_offsets_dev, int num_experts,
                           void* out_dev, void* scales_dev, void* stream);

/*
 * mxfp8_quantize_grouped ROW and COL from one read of the input (cols % 32 == 0);
 * each copy's scales go to its own buffer, sized by mxfp8_grouped_scale_bytes for its
 * axis.
 */
int mxfp8_quantize_grouped_dual(const void* src_dev, int64_t total_rows, int64_t cols,
                                const int32_t* expert_offsets_dev, int num_experts,
                                void* row_out_dev, void* row_scales_dev, void* col_out_dev,
                                void* col_scales_dev, void* stream);

/*
 * Block-scaled GEMM on tcgen05 (kind::mxf8f6f4, E4M3 x E4M3, UE8M0 scales, FP32
 * accumulation): C[M][N] = sum_k deq(A)[m][k] * deq(B)[n][k] ("The pipeline", learner
 * paragraph: the three GEMMs of a linear layer).
 *   A_dev, sA_dev  E4M3 [M][K] and its SWIZZLED scales (rows M, K/32 blocks);
 *   B_dev, sB_dev  E4M3 [N][K] and its SWIZZLED scales (rows N, K/32 blocks);
 *   C_dev          [M][N], BF16 or FP32 (out_dtype), fully overwritten.
 * Both operands are K-major ("TN"); `op` names which quantized copies are passed
 * (see mxfp8_op) and does not change the arithmetic. Requires K % 32 == 0,
 * M % 16 == 0 and N % 16 == 0. Accuracy: |C - C_exact| <= 2^-9 * sum_k |a_k b_k| per
 * element before the output rounding.
 * Empty sizes read no operand, so A, B and their scales may then be NULL:
 *  - M == 0 or N == 0 writes nothing and returns MXFP8_OK.
 *  - K == 0 zero-fills C, the empty sum; C must then be valid and 16-byte aligned.
 */
int mxfp8_gemm(const void* A_dev, const void* sA_dev, const void* B_dev, const void* sB_dev,
               void* C_dev, int64_t M, int64_t N, int64_t K, int op, int out_dtype,
               void* stream);

/*
 * mxfp8_gemm with a caller-owned device workspace, which lets the GEMM run its last,
 * partial wave of output tiles as split-K pieces. The rest of the tiles run as usual.
 *  - Split-K: each tile of that wave is cut into 3 ranges of K on separate CTA pairs. Two
 *    pieces leave FP32 partial sums in the workspace, and the third adds them before
 *    rounding.
 *  - Without a workspace: that wave runs as half-width tiles. On deep reductions the
 *    pieces finish it sooner.
 *  - Results: either way they meet the mxfp8_gemm accuracy bound. They are not bit-identical
 *    to mxfp8_gemm's, because the FP32 sums are added in another order.
 * Arguments as for mxfp8_gemm, plus:
 *   workspace_dev    device memory, 32-byte aligned, or NULL; the library allocates nothing.
 *   workspace_bytes  its size. Split-K runs only when it is at least
 *                    mxfp8_gemm_workspace_bytes for the same problem, else the call
 *                    proceeds as mxfp8_gemm.
 * The workspace holds the partial sums and one arrival counter per tile, CTA and epilogue
 * warp. It must be zero-filled before its first use. Each launch sets its counters back to
 * zero, so it needs no reset between calls or CUDA-graph replays. There is one exception:
 * after a call that latched MXFP8_ERR_TIMEOUT, zero-fill it again. Only one GEMM may use a
 * workspace at a time, so GEMMs that can run concurrently (other streams) need workspaces of
 * their own.
 * Errors as for mxfp8_gemm, plus MXFP8_ERR_ALIGNMENT for a misaligned workspace. A piece
 * whose partners do not arrive within the pipeline wait limit latches MXFP8_ERR_TIMEOUT.
 */
int mxfp8_gemm_ws(const void* A_dev, const void* sA_dev, const void* B_dev, const void* sB_dev,
                  void* C_dev, int64_t M, int64_t N, int64_t K, int op, int out_dtype,
                  void* workspace_dev, size_t workspace_bytes, void* stream);

/*
 * Workspace bytes with which mxfp8_gemm_ws runs this GEMM's last wave as split-K pieces
 * on the current device. The size depends on the device's SM count. 0 means the GEMM never
 * splits: its last wave is full or too wide, or K is too shallow (fewer than 120 stages of
 * 128, where the half tiles finish first). The same 0 is returned for arguments mxfp8_gemm
 * would refuse, and for an unsupported device.
 */
size_t mxfp8_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, int op, int out_dtype);

/*
 * Grouped (MoE expert) block-scaled GEMMs over token segments off[e] .. off[e+1]
 * (expert_offsets_dev as for mxfp8_quantize_grouped).
 *   op FPROP / DGRAD:  A [total_rows][K] with grouped ROW scales (one block per expert,
 *                      as written by mxfp8_quantize_grouped ROW); B [E][N][K] with
 *                      batched SWIZZLED scales (mxfp8_quantize_batched); C
 *                      [total_rows][N]: rows of expert e get A_e . B[e]^T. C rows of
 *                      no expert (none when off[E] = total_rows) are not written.
 *   op WGRAD:          A [N][total_rows] and B [K][total_rows] (column-wise copies,
 *                      grouped COL scales); C [E][N][K], C[e] = A[:, seg e] .
 *                      B[:, seg e]^T; an expert with no tokens gets C[e] = 0.
 * Requires K % 32 == 0, N % 16 == 0, total_rows % 32 == 0, and for WGRAD K % 16 == 0.
 * Empty sizes read no operand and run no kernel: A, B and their scales may then be NULL,
 * and the offsets are not read.
 *  - An empty output is a no-op that returns MXFP8_OK: N == 0, or K == 0 for WGRAD, or
 *    total_rows == 0 (no routed tokens) for FPROP / DGRAD.
 *  - A reduction over nothing zero-fills C, which must then be valid and 16-byte aligned:
 *    WGRAD with total_rows == 0, or FPROP / DGRAD with K == 0.
 */
int mxfp8_grouped_gemm(const void* A_dev, const void* sA_dev, const void* B_dev,
                       const void* sB_dev, void* C_dev, const int32_t* expert_offsets_dev,
                       int num_experts, int64_t total_rows, int64_t N, int64_t K, int op,
                       int out_dtype, void* stream);

/*
 * Workspace bytes mxfp8_selfcheck needs for `tokens` random input rows against an
 * [N][K] weight (0 for invalid sizes: tokens % 16, N % 16 and K % 32 must be 0, and the
 * size must fit in 64 bits).
 */
size_t mxfp8_selfcheck_workspace_bytes(int64_t tokens, int64_t N, int64_t K);

/*
 * Post-synchronization self-check of one quantized weight (section "Correctness: how it
 * fails", the post-sync self-check, condition C3). The BF16 input x [tokens][K] is
 * quantized and multiplied, by this library's kernels, with the weight exactly as the
 * GEMM reads it: w_codes_dev (E4M3 [N][K]) and w_scales_dev (SWIZZLED), i.e. the derived
 * layout - one dense layer, or one expert's slice of a batched expert weight. The result
 * is compared with a reference that multiplies the BF16 input with the canonical
 * synchronized weight, ref_codes_dev (E4M3 [N][K]) and ref_scales_dev (LINEAR
 * [N][K/32]), dequantized, with FP32 accumulation. Writes
 * ||Y - Y_ref||_F / ||Y_ref||_F to *rel_err_dev (device float). A healthy weight gives a
 * few percent (the activations' quantization error); a derived layout that is stale or
 * misplaced relative to the synchronized weight gives order 1; the pages' tolerance is
 * 0.25. Requires tokens % 16 == 0, N % 16 == 0, K % 32 == 0 and tokens <= 2097120;
 * sizes whose workspace would not fit in 64 bits are invalid (MXFP8_ERR_INVALID_ARG).
 *   workspace_dev  caller-owned, >= mxfp8_selfcheck_workspace_bytes(tokens, N, K)
 *                  bytes, 256-byte aligned; holds the quantized input, the FP32 output
 *                  and the two reduction sums. Overwritten.
 * Asynchronous on `stream` like the other calls.
 */
int mxfp8_selfcheck(const void* w_codes_dev, const void* w_scales_dev,
                    const void* ref_codes_dev, const void* ref_scales_dev, int64_t N, int64_t K,
                    const void* x_bf16_dev, int64_t tokens, void* workspace_dev,
                    size_t workspace_bytes, float* rel_err_dev, void* stream);

/*
 * mxfp8_selfcheck without a caller-provided workspace, for callers that cannot allocate
 * device memory when the check runs - for instance a serving engine's post-update hook
 * running while the engine's caching allocator holds all free device memory, or a
 * plugin that has no handle to the host framework's allocator. This entry point has no
 * counterpart on the pages; it exists for those callers.
 *   Arguments and result as mxfp8_selfcheck. The workspace is a fixed 8 MiB array
 *   inside the library (every device that loads the library holds it until the process
 *   exits), so mxfp8_selfcheck_workspace_bytes(tokens, N, K) must not exceed
 *   8 MiB (8388608 bytes); larger sizes return MXFP8_ERR_INVALID_ARG.
 *   No device memory is allocated and no allocating library routine is called.
 *   The first call on a device looks up the array's device address on that device
 *   (under a lock, so host threads may make their first calls at the same time); make
 *   that first call before any stream capture.
 *   All calls share the one array: calls that overlap on the GPU (other streams, other
 *   host threads) race on it and must be serialised by the caller. Every call
 *   rewrites what it reads, and clears its two reduction sums itself.
 */
int mxfp8_selfcheck_noalloc(const void* w_codes_dev, const void* w_scales_dev,
                            const void* ref_codes_dev, const void* ref_scales_dev, int64_t N,
                            int64_t K, const void* x_bf16_dev, int64_t tokens,
                            float* rel_err_dev, void* stream);

/*
 * Sets how long a GEMM kernel's pipeline waits (a stage's copies, the tensor cores, the
 * accumulator hand-over) may take before the kernel gives up, for every GEMM launched
 * after the call, in any host thread: `ns` nanoseconds, or the default for ns == 0
 * (MXFP8_WAIT_LIMIT_MS from the environment, else 4 s). Failure detection (the post's
 * section "Correctness: how it fails" lists the failures a pipeline must not hang on): a
 * kernel whose wait runs out latches MXFP8_ERR_TIMEOUT, stops issuing work, waits for the
 * copies and tensor-core operations it has in flight (for at least 2 s, independently of
 * this limit), frees its tensor memory and returns; its outputs are then unspecified. A
 * limit shorter than a tile's computation makes every GEMM time out, which is how the
 * tests exercise that path. The pages have no counterpart for this call. Returns MXFP8_OK.
 */
int mxfp8_set_wait_limit_ns(uint64_t ns);

/*
 * Synchronizes `stream`, then returns and clears the current device's status word:
 * MXFP8_OK, or the first device-side error latched since the last call
 * (MXFP8_ERR_BAD_OFFSETS, MXFP8_ERR_TIMEOUT), or MXFP8_ERR_CUDA if the synchronization
 * itself failed. The word is read and cleared in one atomic exchange, enqueued on
 * `stream` after its earlier work. An error that a kernel on another stream latches
 * concurrently is reported by this call or by the next one; it is never cleared unread.
 */
int mxfp8_get_device_status(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MXFP8_H_ */
