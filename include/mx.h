/*
 * mx.h -- C ABI of the GB300 (sm_103a) block-scaled low-precision linear layer.
 *
 * The library quantizes bf16 tensors into block-scaled FP8/FP4 operands laid
 * out for the 5th-generation tensor core, multiplies them with tcgen05
 * block-scaled MMA, and composes the two into a linear layer's forward,
 * data-gradient and weight-gradient passes.
 *
 * Sources (web pages; cited by title and section):
 *   [MOSS] "MOSS: 用微缩放和自动缩放实现无损 FP8 训练，OLMo-7B 加速 34%":
 *          创新 1 (two-level scaling), Power-of-Two 的关键优势, 两级缩放实现,
 *          GEMM Kernel 优化 (main loop on the tensor core, dequantise once in
 *          the epilogue).
 *   [COAT] "COAT: Compressing Optimizer States and Activation for memory
 *          efficient FP8 Training" (article): FP8 量化最佳化器狀態的難點
 *          (E4M3 range 448 .. 0.00195).
 *   [FAF]  "格式感知融合:让FP4预训练提速两倍的工程实践":
 *          FP4加速为何常常"纸上富贵" (E2M1; nvfp block scaling; MX mxfp),
 *          格式感知融合的设计思路 (producer writes the consumer layout),
 *          两个关键的数值技巧 (stochastic rounding of gradients, fixed-sign
 *          32-point Hadamard on the weight gradient).
 *
 * Conventions shared by every entry point
 *   - Pointers named x, X, W, dY, codes, sf, amax, tensor_scale, C, Y, dX,
 *     dW and workspace are DEVICE pointers; the mx_tensor and mx_bwd_opts
 *     structs themselves live in host memory.
 *   - The caller owns all memory.  The library allocates no device memory.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call
 *     enqueues its work on that stream and returns without synchronising.
 *   - Return value: MX_OK or an mx_status error code.  Argument errors are
 *     found on the host before anything is launched.  A device-side bounded
 *     wait that gives up records MX_ERR_TIMEOUT in a per-device status word
 *     that mx_last_device_status() reads.
 *   - bf16 inputs must be finite; NaN/Inf inputs give unspecified codes.
 *   - Only sm_103 devices are supported (MX_ERR_UNSUPPORTED otherwise);
 *     without a CUDA device calls return MX_ERR_NO_DEVICE.
 */
#ifndef MX_GB300_H
#define MX_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum mx_status {
    MX_OK = 0,
    MX_ERR_INVALID_ARG = 1,  /* null pointer, bad enum, inconsistent shapes */
    MX_ERR_UNSUPPORTED = 2,  /* format/option combination or device not supported */
    MX_ERR_ALIGNMENT = 3,    /* pointer/leading-dimension/K alignment rule broken */
    MX_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
    MX_ERR_TIMEOUT = 5,      /* a device-side bounded wait gave up */
    MX_ERR_NO_DEVICE = 6,    /* no usable CUDA device */
    MX_ERR_WORKSPACE = 7     /* workspace missing or smaller than required */
} mx_status;

/* Block-scaled formats.
 * MXFP8_E4M3: E4M3 codes, one E8M0 (power-of-two) scale per 32 elements along
 *             K ([FAF] mxfp, the MX standard).  No tensor scale.
 * MXFP4_E2M1: E2M1 codes, one E8M0 scale per 32 elements.  No tensor scale.
 * NVFP4:      E2M1 codes, one UE4M3 scale per 16 elements and an FP32 tensor
 *             scale amax / (448 * 6) ([FAF] nvfp, block scaling under a
 *             global scale).
 * MOSS_FP8:   E4M3 codes, FP32 tensor scale amax / 448 times a power-of-two
 *             micro scale per 32 elements ([MOSS] 创新 1, 两级缩放实现).
 * NVFP4_LOCAL: NVFP4 with the FP32 scale local to each region of
 *             MX_LOCAL_REGION (128) consecutive operand rows over all of K
 *             instead of global ([FAF] 格式感知融合的设计思路: "CTA-local" nvfp).
 *             amax and tensor_scale are arrays of mx_scale_count(fmt, rows)
 *             entries; a GEMM applies s_A[i / 128] * s_B[j / 128] per output.
 *             No global amax is needed. */
typedef enum mx_format {
    MX_FMT_MXFP8_E4M3 = 0,
    MX_FMT_MXFP4_E2M1 = 1,
    MX_FMT_NVFP4 = 2,
    MX_FMT_MOSS_FP8 = 3,
    MX_FMT_NVFP4_LOCAL = 4
} mx_format;

/* Operand rows that share one FP32 scale in MX_FMT_NVFP4_LOCAL. */
#define MX_LOCAL_REGION 128

/* RNE: round to nearest, ties to even, saturating at the largest finite
 * value.  SR: stochastic rounding ([FAF] 两个关键的数值技巧; the pages attach it
 * to E2M1, the same rule applies to E4M3, saturating at 448): element
 * L = r*K + k of the K-major operand rounds up iff u16 < p*2^16,
 * p its distance fraction between the two neighbouring grid points and u16
 * the 16-bit half (L odd: high, even: low) of word (L&7)>>1 of
 * Philox4x32-10(counter = {L>>3, L>>35, stream_id, 0}, key = {seed, seed>>32}). */
typedef enum mx_rounding { MX_ROUND_RNE = 0, MX_ROUND_SR = 1 } mx_rounding;

/* Power-of-two scale rule for a block with max |y| = b (Q = 448, emax = 8 for
 * E4M3; Q = 6, emax = 2 for E2M1).  DEFAULT = FLOOR for the MX formats and
 * CEIL for MOSS; NVFP4 accepts DEFAULT only.
 * FLOOR: e = floor(log2 b) - emax.  CEIL: smallest e with b*2^-e <= Q.
 * NEAREST: e = round(log2(b/Q)) ([MOSS] 两级缩放实现's rounding to the
 * nearest power of two).  e is clamped to [-127, 127]; b = 0 gives e = 0. */
typedef enum mx_scale_rule {
    MX_SCALE_DEFAULT = 0,
    MX_SCALE_FLOOR = 1,
    MX_SCALE_CEIL = 2,
    MX_SCALE_NEAREST = 3
} mx_scale_rule;

/* ROWWISE quantizes x[R, C] along C (operand rows = R, K = C).
 * COLWISE quantizes along R and writes the transposed operand
 * (operand rows = C, K = R): the transpose is fused into the producer. */
typedef enum mx_dir { MX_ROWWISE = 0, MX_COLWISE = 1 } mx_dir;

typedef enum mx_out_dtype { MX_OUT_F32 = 0, MX_OUT_BF16 = 1 } mx_out_dtype;

/* A quantized K-major operand.  Device buffers are caller-allocated:
 *   codes        mx_codes_bytes(fmt, rows, k) bytes: row-major [rows, K];
 *                E4M3 one byte per element; E2M1 two per byte, the even k in
 *                the low nibble.  Row stride = K or K/2 bytes.
 *   sf           mx_sf_bytes(fmt, rows, k) bytes: block scales in the tensor
 *                core's scale-factor layout: 512-byte tiles of 128 rows x 4
 *                K-blocks, ordered by row tile then K-block group; row r,
 *                block kb at (r%32)*16 + ((r%128)/32)*4 + kb%4 inside its
 *                tile ([FAF] 格式感知融合的设计思路: the producer writes the
 *                consumer's layout).  Padding bytes are left unwritten.
 *   amax         1 float: max |x| over the tensor (written for NVFP4, MOSS).
 *   tensor_scale 1 float: the FP32 tensor scale (NVFP4, MOSS), else unused.
 * mx_quantize fills rows, k, fmt, block and hadamard. */
typedef struct mx_tensor {
    void* codes;
    uint8_t* sf;
    float* amax;
    float* tensor_scale;
    int64_t rows;
    int64_t k;
    int32_t fmt;
    int32_t block;
    int32_t hadamard;
    int32_t reserved;
} mx_tensor;

/* Byte sizes of an operand's buffers (0 for invalid arguments). */
size_t mx_codes_bytes(int fmt, int64_t rows, int64_t k);
size_t mx_sf_bytes(int fmt, int64_t rows, int64_t k);

/* Entries of an operand's amax and tensor_scale arrays: 1 for MOSS_FP8 and
 * NVFP4, ceil(rows / MX_LOCAL_REGION) (at least 1) for NVFP4_LOCAL, 0 for the
 * formats without a tensor scale and for an invalid fmt. */
size_t mx_scale_count(int fmt, int64_t rows);

/* amax[0] = max |x| over a bf16 matrix x[R, C] with row stride ld elements
 * (ld >= C, ld % 8 == 0, x 16-byte aligned).  [MOSS] 两级缩放实现, level 1. */
int mx_amax(const void* x, int64_t R, int64_t C, int64_t ld, float* amax, void* stream);

/* The fused quantize producer: bf16 x[R, C] (row stride ld elements) ->
 * codes + block scales (+ amax and tensor scale) in *out.
 *   block      32 for MXFP8/MXFP4/MOSS, 16 for NVFP4 (MX_ERR_UNSUPPORTED else).
 *   rounding   MX_ROUND_RNE or MX_ROUND_SR (every format).
 *   hadamard   1: multiply every 32-element K-block by the fixed-sign
 *              Sylvester H32 (unnormalised, five fp32 butterfly stages in
 *              the order h = 1, 2, 4, 8, 16) before scaling ([FAF]
 *              两个关键的数值技巧); MX formats and NVFP4 (K % 32 == 0).  For
 *              NVFP4 the tensor amax is that of the transformed operand,
 *              max |H32 y| over its 32-element groups along K.
 *   amax_in    optional device float holding the tensor amax (max |x|, or
 *              the transformed operand's with hadamard) (skips the amax pass
 *              of NVFP4/MOSS; it is copied to out->amax); NULL = compute it.
 *   seed, stream_id  the SR Philox key and third counter word.
 * Alignment: x 16-byte aligned, ld % 8 == 0, K % block == 0; for COLWISE also
 * R % 32 == 0.  out->codes 16-byte aligned. */
int mx_quantize(const void* x, int64_t R, int64_t C, int64_t ld, int dir, int fmt, int block,
                int rounding, int scale_rule, uint64_t seed, uint32_t stream_id, int hadamard,
                const float* amax_in, mx_tensor* out, void* stream);

/* The dual-direction producer: one read of bf16 x[R, C] emits both the
 * rowwise operand (row_out: rows R, K = C) and the colwise operand (col_out:
 * rows C, K = R), exactly as two mx_quantize calls would, each direction with
 * its own rounding and Hadamard options.  A layer's forward operand and the
 * transposed operand its backward pass needs come from one pass over memory
 * ([FAF] FP4加速为何常常"纸上富贵": operand packing, layout construction and
 * saving backward state are the costs around the GEMM).  Both outputs share
 * the tensor amax and tensor scale (written to both), except NVFP4 with the
 * Hadamard transform on either side: each operand then gets the amax and scale
 * of its own (transformed or plain) values, from a pass of its own over x, and
 * amax_in must be NULL (MX_ERR_UNSUPPORTED).  Requires C % block == 0 and
 * R % 32 == 0; other rules as mx_quantize. */
int mx_quantize_dual(const void* x, int64_t R, int64_t C, int64_t ld, int fmt, int block,
                     int scale_rule, uint64_t seed, uint32_t stream_id, int row_rounding,
                     int row_hadamard, int col_rounding, int col_hadamard, const float* amax_in,
                     mx_tensor* row_out, mx_tensor* col_out, void* stream);

/* out[r, k] (fp32, row-major [rows, K]) = dec(code) * dec(block scale) *
 * tensor scale (if the format has one).  The inverse map of [MOSS]
 * 两级缩放实现's dequantize; a test aid, not on the hot path. */
int mx_dequantize(const mx_tensor* A, float* out, void* stream);

/* The block-scaled GEMM: C[M, N] = alpha * dq(A) dq(B)^T with M = A->rows,
 * N = B->rows, K = A->k = B->k, both operands K-major and of the same format.
 * Block scales are applied inside the tcgen05 MMA; the epilogue multiplies the
 * fp32 accumulator once by alpha = fl32(fl32(tsA * tsB) * e), tsX the tensor
 * scales (1 when the format has none) and e = extra_alpha, times 1/32 when
 * both operands carry the Hadamard transform ((H a)^T (H b) = 32 a^T b)
 * ([MOSS] GEMM Kernel 优化: dequantise once in the epilogue).
 * C is fp32 or bf16 (RNE), row stride ldc elements (ldc >= N, ldc % 8 == 0,
 * C 16-byte aligned); nothing outside the M x N view (columns N .. ldc - 1 of a
 * row, rows past M) is written.  K % 128 == 0 for FP8 formats, K % 256 == 0 for
 * FP4.  A->hadamard must equal B->hadamard.  Asynchronous on `stream`; the
 * call allocates nothing and may be captured into a CUDA graph. */
int mx_gemm(const mx_tensor* A, const mx_tensor* B, float extra_alpha, void* C, int64_t ldc,
            int out_dtype, void* stream);

/* mx_gemm that also returns the output's absolute maximum, reduced in the
 * epilogue from the values as written (after the bf16 rounding for
 * MX_OUT_BF16): *amax_out = max |C[i, j]| over the M x N view, NaN if any
 * element is NaN.  This is the tensor amax that the next quantization of C
 * needs for its tensor scale ([FAF] nvfp: amax / (448 * 6); [MOSS]
 * 两级缩放实现, level 1), so the producer that follows can take it through its
 * amax_in argument instead of a separate reduction pass over C.  amax_out is a
 * device pointer to one float (4-byte aligned) that the call zeroes on
 * `stream` before the GEMM; an empty product (M, N or K zero) gives 0.
 * Errors: MX_ERR_INVALID_ARG for a null amax_out, MX_ERR_ALIGNMENT for a
 * misaligned one, otherwise as mx_gemm.  Allocates nothing; graph-capturable. */
int mx_gemm_amax(const mx_tensor* A, const mx_tensor* B, float extra_alpha, void* C, int64_t ldc,
                 int out_dtype, float* amax_out, void* stream);

/* The block-scaled GEMM with its result quantized in the epilogue into the
 * rowwise MX operand that a following GEMM consumes ([FAF]
 * 格式感知融合的设计思路: the producer writes the consumer's layout, here the
 * GEMM itself is the producer).  out->fmt is MX_FMT_MXFP8_E4M3 or
 * MX_FMT_MXFP4_E2M1; the function sets out->rows = M = A->rows, out->k = N =
 * B->rows, out->block = 32, out->hadamard = 0.  Each 32-column block of a row
 * of v = alpha * acc (the fp32 value mx_gemm would return as fp32, same alpha
 * rule) gets the FLOOR-rule E8M0 scale and round-to-nearest-even codes, exactly
 * as mx_quantize would encode an fp32 input; codes are K-major (out->codes,
 * mx_codes_bytes(out->fmt, M, N) bytes, 16-byte aligned) and scale bytes in the
 * tensor-core layout (out->sf, mx_sf_bytes bytes, 16-byte aligned; the padding
 * is not written).  Requires N % 32 == 0, K > 0 and the mx_gemm rules for A and
 * B.  Errors: MX_ERR_UNSUPPORTED for another output format, MX_ERR_ALIGNMENT
 * for N % 32 != 0 or misaligned buffers, MX_ERR_INVALID_ARG otherwise. */
int mx_gemm_quantized(const mx_tensor* A, const mx_tensor* B, float extra_alpha, mx_tensor* out, void* stream);

/* Workspace bytes for mx_linear_fwd and mx_linear_fwd_save (pass 0),
 * mx_linear_bwd (pass 1) and mx_linear_bwd_saved (pass 2); 0 for another pass
 * or invalid arguments. */
size_t mx_linear_workspace_bytes(int64_t T, int64_t Kin, int64_t Nout, int fmt, int pass);

/* Forward of a linear layer: Y[T, Nout] = X[T, Kin] W[Nout, Kin]^T, both
 * operands quantized rowwise with RNE and the format's default rule, Y in
 * out_dtype with row stride Nout.  workspace: device, >= the size above. */
int mx_linear_fwd(const void* X, const void* W, int64_t T, int64_t Kin, int64_t Nout, int fmt,
                  void* Y, int out_dtype, void* workspace, size_t ws_bytes, void* stream);

/* mx_linear_fwd for callers that cannot allocate device memory (code running
 * inside an allocator or memory-pool callback, processes whose device memory
 * is reserved up front, plugin interfaces that pass only input and output
 * pointers).  The pages have no counterpart to this entry point.
 * Same arguments and result as mx_linear_fwd minus the workspace: the
 * quantized operands go to a fixed 32 MiB array in the library's device
 * memory (held by every GPU that loads the library until the process exits).
 * Returns MX_ERR_WORKSPACE, launching nothing, when
 * mx_linear_workspace_bytes(T, Kin, Nout, fmt, 0) exceeds 32 MiB.
 * It calls no allocator.  The first call on a device looks up the array's
 * device address for that device (make that first call before any stream
 * capture).  All calls share the one array: calls whose work overlaps on the
 * GPU (other streams, other host threads) race on it and must be ordered by
 * the caller. */
int mx_linear_fwd_noalloc(const void* X, const void* W, int64_t T, int64_t Kin, int64_t Nout,
                          int fmt, void* Y, int out_dtype, void* stream);

/* Backward options ([FAF] 两个关键的数值技巧: stochastic rounding of the
 * gradient and a fixed-sign Hadamard-32 preconditioning of the weight
 * gradient, both on the mxfp route; the same options are offered on NVFP4). */
typedef struct mx_bwd_opts {
    int32_t wgrad_hadamard;   /* 1: H32 along tokens on both wgrad operands (MX formats, NVFP4) */
    int32_t wgrad_dy_rounding;/* mx_rounding for dY^T in wgrad */
    uint64_t seed;            /* SR Philox key */
    uint32_t stream_id;       /* SR Philox counter word 2 */
    int32_t reserved;
} mx_bwd_opts;

/* Backward of the same layer (opts NULL = RNE, no Hadamard):
 *   dgrad dX[T, Kin]  = dY[T, Nout] W[Nout, Kin]   (dY rowwise, W colwise)
 *   wgrad dW[Nout, Kin] = dY^T X                    (dY, X colwise)
 * dX or dW may be NULL to skip that GEMM.  Outputs are row-major with row
 * strides Kin, in dx_dtype / dw_dtype.
 * With both dX and dW the weight gradient (X^T's producer and its GEMM) runs
 * on a side stream of the library that waits for the work issued to `stream`
 * before the fork and that `stream` waits for before the call returns (an
 * event join, which graph capture records as a fork and a join), so the two
 * GEMMs fill each other's last partial wave; the results are the same either
 * way.  The side stream and its two events are created once per host thread
 * and device, on the first such call made outside graph capture, and kept
 * until the process exits; a call captured before then runs on `stream`
 * alone.  Work the caller issues to
 * `stream` after the call is ordered after both gradients. */
int mx_linear_bwd(const void* dY, const void* X, const void* W, int64_t T, int64_t Kin,
                  int64_t Nout, int fmt, const mx_bwd_opts* opts, void* dX, int dx_dtype,
                  void* dW, int dw_dtype, void* workspace, size_t ws_bytes, void* stream);

/* Bytes of the saved backward state of one layer (mx_linear_fwd_save ->
 * mx_linear_bwd_saved): the colwise operands X^T [Kin, T] and W^T [Kin, Nout]
 * with their scale bytes and tensor scales; 0 for invalid arguments. */
size_t mx_linear_saved_bytes(int64_t T, int64_t Kin, int64_t Nout, int fmt);

/* Forward of a linear layer that also keeps what its backward pass needs
 * ([FAF] FP4加速为何常常"纸上富贵": saving backward state is one of the costs
 * around the GEMM; 格式感知融合的设计思路: each producer writes its consumer's
 * layout).  One read of X emits the forward operand X (rowwise) and X^T
 * (colwise, for the weight gradient); one read of W emits W and W^T (for the
 * data gradient).  Y[T, Nout] = X W^T exactly as mx_linear_fwd computes it;
 * X^T and W^T go to `saved` (device, mx_linear_saved_bytes bytes, caller-owned,
 * to be passed unchanged to mx_linear_bwd_saved).
 *   x_amax, w_amax  optional device floats holding max |X|, max |W| (NVFP4,
 *                   MOSS): the tensor amax then needs no pass of its own
 *                   (e.g. taken from the operation that produced X, or from a
 *                   weight-scale predictor).  NULL = reduce it from the tensor.
 *                   NVFP4_LOCAL takes NULL only (MX_ERR_UNSUPPORTED else).
 *   opts            the options the backward pass will use (NULL = RNE, no
 *                   Hadamard); wgrad_hadamard decides whether X^T carries the
 *                   Hadamard transform.
 *   workspace       device, >= mx_linear_workspace_bytes(.., pass 0).
 * Requires T % 32 == 0 and Nout % 32 == 0 (the colwise operands' K) besides
 * the rules of mx_quantize and mx_gemm.  Errors: MX_ERR_WORKSPACE for a missing
 * or short workspace or saved buffer, otherwise as mx_quantize_dual/mx_gemm. */
int mx_linear_fwd_save(const void* X, const void* W, int64_t T, int64_t Kin, int64_t Nout, int fmt,
                       const float* x_amax, const float* w_amax, const mx_bwd_opts* opts, void* Y, int out_dtype,
                       void* workspace, size_t ws_bytes, void* saved, size_t saved_bytes, void* stream);

/* Backward of the layer from its saved state: one read of dY emits dY
 * (rowwise, RNE) and dY^T (colwise, opts' rounding and Hadamard), then
 *   dgrad dX[T, Kin] = dY W (against the saved W^T),
 *   wgrad dW[Nout, Kin] = dY^T X (against the saved X^T).
 * Results are bit-identical to mx_linear_bwd with the same opts.  `saved` is
 * the buffer mx_linear_fwd_save filled (read only), `opts` must be the ones
 * given to it.  dy_amax as x_amax above.  dX or dW may be NULL to skip that
 * GEMM.  workspace: device, >= mx_linear_workspace_bytes(.., pass 2).  With
 * both dX and dW the weight-gradient GEMM runs on the side stream, forked and
 * joined as in mx_linear_bwd. */
int mx_linear_bwd_saved(const void* dY, int64_t T, int64_t Kin, int64_t Nout, int fmt, const float* dy_amax,
                        const mx_bwd_opts* opts, const void* saved, size_t saved_bytes, void* dX, int dx_dtype,
                        void* dW, int dw_dtype, void* workspace, size_t ws_bytes, void* stream);

/* Human-readable text of an mx_status. */
const char* mx_strerror(int status);

/* Synchronises `stream`, then returns and clears the device status word of
 * the current device (MX_OK or MX_ERR_TIMEOUT). */
int mx_last_device_status(void* stream);

/* Self-test of the bounded-wait path: launches one block that waits on an
 * mbarrier nothing ever arrives at, giving up after limit_ns nanoseconds.
 * Synchronises the stream and returns MX_ERR_TIMEOUT when the wait gave up as
 * designed (and the status word then reads MX_ERR_TIMEOUT), MX_OK never. */
int mx_selftest_bounded_wait(uint64_t limit_ns, void* stream);

/* Number of CUDA kernels this library has launched in the calling process
 * (memset/memcpy nodes not counted).  Lets a caller count device work. */
uint64_t mx_launch_count(void);

/* Test hook: the quantizer's division by a shared divisor (q_fast, computed
 * from the divisor's correctly rounded reciprocal plus residual corrections)
 * next to CUDA's IEEE division (q_ieee), for n device pairs v[i] / d[i]. */
int mx_debug_divide(const float* v, const float* d, int64_t n, float* q_fast, float* q_ieee, void* stream);

/* Test hook: choose the producer implementation for later calls made by the
 * calling host thread (other threads keep their own choice, initially 0):
 * 0 automatic (the tile producer, except for NVFP4 with the Hadamard
 * transform), 1 direct-load row/col kernels, 2 the shared-memory tile producer
 * for both directions.  Outputs are identical; only the speed differs. */
void mx_debug_set_quant_impl(int impl);

/* Test hook for the tile producer's bounded waits: for later quantize calls
 * made by the calling host thread, the last thread of every producer CTA
 * treats its wait for that CTA's tile number `tile` (0-based, in the CTA's own
 * order) as timed out.  The pass then stops, waits for its own copies in
 * flight and reports MX_ERR_TIMEOUT through the status word
 * (mx_last_device_status); outputs of such a pass are unspecified.  -1 (the
 * initial value) turns it off.  Nothing faults or hangs. */
void mx_debug_set_tile_fail_at(int64_t tile);

/* Test and tuning hook: 0 runs both gradients of mx_linear_bwd /
 * mx_linear_bwd_saved on the caller's stream, one after the other; 1 (the
 * initial setting) forks the weight gradient onto the side stream.  Per host
 * thread. */
void mx_debug_set_bwd_fork(int on);

/* Test hook: force one GEMM kernel variant for later mx_gemm / mx_linear_*
 * calls made by the calling host thread (other threads keep their own choice,
 * initially 0): 0 automatic, 1 single-CTA 128 x 128 tiles, 2 single-CTA
 * 128 x 256 tiles, 3 CTA-pair (cluster of two) 256 x 256 tiles, 4 the
 * warp-specialised CTA pair (scale-factor stores and the epilogue in separate
 * warps; the automatic choice for large shapes). */
void mx_debug_set_gemm_variant(int variant);

/* Test/benchmark hook: the GEMM variant (numbered as above, never 0) that the
 * calling host thread's most recent mx_gemm / mx_linear_* call launched; 0
 * before any. */
int mx_debug_last_gemm_variant(void);

#ifdef __cplusplus
}
#endif
#endif /* MX_GB300_H */
