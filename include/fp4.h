/*
 * fp4.h -- C ABI of the GB300 (sm_103a) block-scaled FP4 library.
 *
 * The library quantizes bf16/fp32 tensors to E2M1 FP4 with a shared per-block
 * scale and runs the block-scaled GEMMs that consume them, following these
 * pages on FP4 LLM training (cited by short name):
 *
 *   [grad]    aicoding.csdn.net "深度学习中的梯度计算基础": Q(x) = s*round(x/s)
 *             (§2.1), the straight-through estimator (§3.1), block size (§4.2)
 *   [lowprec] framerc.cn "低精度训练技术概述": E4M3 / E8M0 / MXFP4 / NVFP4
 *             (§1.1), stochastic rounding (§1.2, §3.2), the unsupported-format
 *             error of the quantize_to_fp4 snippet (§3.2)
 *   [outlier] devpress.csdn.net "大模型4位训练中的异常值动态分析与优化实践":
 *             E2M1 range (§1.1), hot-channel compensation (§3.1-3.2), forward
 *             RTN + 1D scaling / backward SR + 16x16 2D scaling + RHT (§4.1-4.2)
 *   [msr]     lsdiaocha.cn write-up of the MSR FP4 training paper: E2M1 (§一),
 *             the differentiable gradient estimator and its 3.0 clamp (§二),
 *             GEMMs are >95% of the compute (§四), the FP4 LUT kernel (§六)
 *
 * Conventions shared by every call
 * --------------------------------
 *  - All pointers named x, codes, scales, out, ... are DEVICE pointers owned by
 *    the caller.  The library allocates only the context (fp4_create).
 *  - A pointer may be NULL when the buffer it names holds no elements (a zero
 *    extent); such calls validate their arguments and enqueue nothing.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream).  The return value reports argument validation and
 *    launch errors synchronously; FP4_OK means the work was enqueued.
 *  - A device-side wait that gives up (see FP4_ERR_TIMEOUT) sets a status word
 *    in the context; fp4_sync_status() reports and clears it.
 *  - A context serves one stream at a time (it holds scratch used by NVFP4
 *    quantization).  Use one context per concurrently used stream.
 *  - Tensors are row-major.  `ld*` arguments are row pitches in elements.
 *  - Codes: uint8 [rows][k/2]; element 2j in the low nibble, 2j+1 in the high
 *    nibble; 4-bit E2M1 code = sign<<3 | exponent<<1 | mantissa.
 *  - Scales: one byte per block of `block` consecutive elements along k:
 *    MXFP4 = E8M0 exponent byte (scale 2^(byte-127)), block 32;
 *    NVFP4 = E4M3 byte, block 16, times the fp32 per-tensor scale g.
 *    Layout FP4_SF_ROWMAJOR: [rows][k/block].
 *    Layout FP4_SF_MMA (what fp4_gemm reads): rows padded to 128 and k padded
 *    to 256 elements; 512-byte atoms of 128 rows x 4 scales, atom (rt, kt) at
 *    byte ((rt * (kpad/block/4)) + kt) * 512, element (r, j) inside the atom
 *    at (r % 32) * 16 + ((r / 32) % 4) * 4 + (j % 4).  Padding bytes are 0.
 *    A call that reads FP4_SF_MMA scales (an fp4_operand) wants them 16-byte
 *    aligned (FP4_ERR_MISALIGNED otherwise), as it wants the codes.
 */
#ifndef FP4_GB300_H
#define FP4_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
enum {
  FP4_OK = 0,
  FP4_ERR_INVALID_ARG = 1,  /* null pointer, bad size, bad enum value        */
  FP4_ERR_UNSUPPORTED = 2,  /* format/block/mode combination not supported
                               (the "Unsupported format" error of [lowprec]
                               §3.2's quantize_to_fp4)                         */
  FP4_ERR_MISALIGNED = 3,   /* pointer or pitch not 16-byte aligned           */
  FP4_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed              */
  FP4_ERR_TIMEOUT = 5,      /* a device-side wait gave up (bounded wait)       */
  FP4_ERR_TOO_LARGE = 6     /* input exceeds a fixed scratch limit (see
                               fp4_hcp_select_noalloc)                        */
};

/* ---- enums --------------------------------------------------------------- */
enum { FP4_FMT_MXFP4 = 0, FP4_FMT_NVFP4 = 1 };           /* [lowprec] §1.1 */
enum { FP4_ROUND_RTN = 0, FP4_ROUND_SR = 1 };            /* [outlier] §4.1 */
enum { FP4_SCALING_1D = 0, FP4_SCALING_2D = 1 };         /* [outlier] §4.1 */
enum { FP4_SF_ROWMAJOR = 0, FP4_SF_MMA = 1 };
enum { FP4_DTYPE_BF16 = 0, FP4_DTYPE_F32 = 1 };
enum { FP4_HCP_SINGLE = 0, FP4_HCP_TWO = 1, FP4_HCP_TWO_FP8 = 2, FP4_HCP_SINGLE_MXFP8 = 3 };  /* [outlier] §3.1 */

typedef struct fp4_ctx fp4_ctx;

/* Quantization parameters: Q(x) = s * round(x / s)  ([grad] §2.1).
 *  format    FP4_FMT_MXFP4 (E8M0 scales) or FP4_FMT_NVFP4 (E4M3 scales x fp32
 *            tensor scale).
 *  block     elements per scale: the format's own (32 MXFP4, 16 NVFP4), or
 *            16, 32, 64, 128 for either format ([grad] §4.2 studies 16-128)
 *            with transpose 0, 1D scaling and FP4_SF_ROWMAJOR (fp4_quantize
 *            only; such operands are read by fp4_dequantize and
 *            fp4_quant_error_stats, not by the GEMMs); else FP4_ERR_UNSUPPORTED.
 *  rounding  RTN (ties to even) or SR (Philox4x32-10, 16 random bits per
 *            element: round up iff u16 < frac * 65536).
 *  scaling   1D (one scale per `block` elements along the blocked axis) or
 *            2D (one scale per 16x16 tile; NVFP4 only; the scale is repeated
 *            for each of the tile's 16 output rows).
 *  transpose 0: blocks along cols, output [rows][cols/2];
 *            1: blocks along rows, output [cols][rows/2] (the operand layout
 *            of dgrad/wgrad).
 *  rht       1: apply the 16-point random Hadamard transform along the
 *            blocked axis before quantizing ([outlier] §4.1).
 *  SR random bits: element at linear output index i uses Philox call
 *  n = sr_offset + i/8 with counter (n lo, n hi, 0, sr_stream) and key
 *  (sr_seed lo, sr_seed hi), 16-bit lane i % 8.
 *  RHT signs: bit j of word 0 of Philox(counter 0, key rht_seed) set -> -1. */
typedef struct {
  int32_t format;
  int32_t block;
  int32_t rounding;
  int32_t scaling;
  int32_t transpose;
  int32_t rht;
  int32_t sf_layout;
  uint32_t sr_stream;
  uint64_t sr_seed;
  uint64_t sr_offset;
  uint64_t rht_seed;
} fp4_quant_params;

/* A quantized GEMM operand: `rows` x `k` FP4 values, blocks along k. */
typedef struct {
  const uint8_t* codes;        /* [rows][k/2]                                  */
  const uint8_t* scales;       /* layout `sf_layout`                           */
  const float* tensor_scale;   /* NVFP4: device fp32 g; MXFP4: NULL            */
  int32_t format;
  int32_t sf_layout;
  int64_t rows;
  int64_t k;
  int32_t block;               /* elements per scale; 0 = the format's own.
                                  Other blocks (16-128, row-major scales) only
                                  for fp4_dequantize / fp4_quant_error_stats;
                                  every other call -> FP4_ERR_UNSUPPORTED     */
} fp4_operand;

/* ---- context --------------------------------------------------------------
 * fp4_create allocates a small device scratch (status word, amax slots) on the
 * current device.  Returns FP4_ERR_CUDA if no device is usable.               */
int fp4_create(fp4_ctx** out);
void fp4_destroy(fp4_ctx* ctx);
/* Synchronize `stream`, then read and clear the context's device status word.
 * Returns FP4_ERR_TIMEOUT if any kernel of this context gave up a wait.      */
int fp4_sync_status(fp4_ctx* ctx, void* stream);
const char* fp4_status_string(int status);

/* Bytes of the scale buffer for a rows x k operand in the given layout and
 * block (0 = the format's own). */
size_t fp4_scales_bytes(int64_t rows, int64_t k, int32_t format, int32_t sf_layout, int32_t block);

/* ---- per-tensor amax ([lowprec] §1.1 "tensor scaling"; NVFP4's fp32 level)
 * *amax_out = max |x| over a rows x cols tensor, after an optional RHT16
 * along `rht_axis` (-1 none, 1 along cols, 0 along rows).  Overwrites
 * *amax_out (device fp32).  Exposed so that a caller can reduce the amax over
 * shards and pass it back as `given_amax`.                                   */
int fp4_amax(fp4_ctx* ctx, const void* x, int32_t x_dtype, int64_t rows, int64_t cols,
             int64_t ldx, int32_t rht_axis, uint64_t rht_seed, float* amax_out, void* stream);

/* ---- quantize ([grad] §2.1; [lowprec] §1.1-1.2, §3.2; [outlier] §4.1-4.2;
 *      [msr] §六 "maps any float to the nearest of the 16 FP4 values")
 * x: rows x cols, dtype bf16 or fp32, pitch ldx, 16-byte aligned rows.
 * NVFP4: g = amax/2688 (6 * 448) with amax = *given_amax if non-NULL else the
 * tensor's own amax (after the RHT, if any); g is written to *tensor_scale.
 * Block scale sb = E4M3_rn_satfinite(amax_b / (6 g)); s = dec(sb) * g;
 * codes = E2M1(x * (1/s)), all zero when s == 0.
 * MXFP4: scale 2^e, e = floor(log2 amax_b) - 2 clamped to [-127, 127];
 * tensor_scale may be NULL.
 * Requirements: blocked extent % block == 0 (and % 16 with rht or 2D).    */
int fp4_quantize(fp4_ctx* ctx, const void* x, int32_t x_dtype, int64_t rows, int64_t cols,
                 int64_t ldx, const fp4_quant_params* params, const float* given_amax,
                 uint8_t* codes, uint8_t* scales, float* tensor_scale, void* stream);

/* Both operand layouts of one tensor from a single read (the dY of a linear
 * layer feeds dgrad with blocks along cols and wgrad with blocks along rows;
 * X and W feed the forward GEMM in one layout and a backward GEMM in the
 * other).  p_rows must have transpose 0, p_cols transpose 1, same format; each
 * has its own rounding, RHT, scale layout and 1D or 16x16 2D scaling (2D needs
 * its output rows in groups of 16).  The results equal two fp4_quantize calls
 * with the same parameters, bit for bit.                                   */
int fp4_quantize_dual(fp4_ctx* ctx, const void* x, int32_t x_dtype, int64_t rows, int64_t cols,
                      int64_t ldx, const fp4_quant_params* p_rows, const fp4_quant_params* p_cols,
                      const float* given_amax_rows, const float* given_amax_cols,
                      uint8_t* codes_rows, uint8_t* scales_rows, float* tensor_scale_rows,
                      uint8_t* codes_cols, uint8_t* scales_cols, float* tensor_scale_cols,
                      void* stream);

/* ---- dequantize ([grad] §2.1 x_hat = s * code value)
 * out[r][j] = cv * 2^e (MXFP4) or fp32(fp32(cv * dec(sb)) * g) (NVFP4), stored
 * as fp32 or bf16 (round to nearest even), pitch ldo.                        */
int fp4_dequantize(fp4_ctx* ctx, const fp4_operand* q, int32_t out_dtype, void* out,
                   int64_t ldo, void* stream);

/* ---- 16-point random Hadamard transform ([outlier] §4.1)
 * y = 1/4 H16 diag(sigma) x on consecutive 16-element chunks along `axis`
 * (1: along cols, 0: along rows); fp32 butterfly, strides 1,2,4,8.  y is fp32
 * with pitch cols.                                                            */
int fp4_rht16(fp4_ctx* ctx, const void* x, int32_t x_dtype, int64_t rows, int64_t cols,
              int64_t ldx, int32_t axis, uint64_t seed, float* y, void* stream);

/* ---- differentiable gradient estimator backward ([msr] §二)
 * dx = dy * f'(x/s), f'(xs) = min(clamp, (1/k)|u|^(1/k-1)) with u the local
 * coordinate of |xs| inside its E2M1 interval (u = 0 -> clamp); |xs| >= 6 ->
 * `outside` (1 = straight-through, [grad] §3.1).  x/s is formed exactly as the
 * quantizer formed it from the stored scales `q` (q->codes unused, may be
 * NULL; blocks along cols, no RHT).  dy bf16 or fp32; dx fp32.             */
int fp4_dge_backward(fp4_ctx* ctx, const void* x, int32_t x_dtype, int64_t ldx,
                     const fp4_operand* q, const void* dy, int32_t dy_dtype, int64_t lddy,
                     float* dx, int64_t lddx, float k, float clamp, float outside, void* stream);

/* ---- sigmoid-smoothed quantizer ([grad] §3.2)
 * Over the signed E2M1 levels q_0..q_14 = -6..6, with thresholds
 * c_i = (q_i + q_{i+1})/2 and steps v_i = q_{i+1} - q_i (i = 0..13):
 *   Q_soft(xs)  = q_0 + sum_i v_i sigma(beta (xs - c_i))        (-> RTN as beta -> inf)
 *   Q_soft'(xs) = beta sum_i v_i sigma(z_i) (1 - sigma(z_i)),   z_i = beta (xs - c_i).
 * xs = x/s is formed exactly as the quantizer formed it from the stored scales
 * `q` (q->codes unused, may be NULL; blocks along cols, no RHT); s is held
 * constant.  fp4_soft_forward: y = s Q_soft(x/s).  fp4_soft_backward:
 * dx = dy Q_soft'(x/s); dy bf16 or fp32.  Outputs fp32, 16-byte aligned.
 * 0 < beta <= 1e6.  For beta >= 9.71 / 19.41 / 38.82 only the 4 / 2 / 1
 * thresholds nearest x/s on each side are evaluated: the terms left out are
 * below 2^-23 of Q_soft' and 2^-26 in absolute value for Q_soft.             */
int fp4_soft_forward(fp4_ctx* ctx, const void* x, int32_t x_dtype, int64_t ldx, const fp4_operand* q,
                     float* y, int64_t ldy, float beta, void* stream);
int fp4_soft_backward(fp4_ctx* ctx, const void* x, int32_t x_dtype, int64_t ldx, const fp4_operand* q,
                      const void* dy, int32_t dy_dtype, int64_t lddy, float* dx, int64_t lddx, float beta,
                      void* stream);

/* ---- outlier clamping and compensation, OCC ([msr] §三, §六)
 * The largest 1% of activation magnitudes are outliers: X is clamped to
 * [-tau, tau] at the 99% quantile tau before it is quantized, and the part
 * clamped away, dX = X - clamp(X) (a sparse matrix), is multiplied in high
 * precision beside the FP4 GEMM:  Y = alpha Q(X_c) Q(W)^T + dX W^T.
 *
 * fp4_occ_threshold: tau = the ceil(q n)-th smallest |x| over the n = rows*cols
 * elements (nearest rank, 0 < q <= 1; q = 0.99 is the page's choice), written
 * to *tau (device fp32); *n_outliers (device int64) = #{|x| > tau}.  x bf16 or
 * fp32, cols % 8 == 0, n / 8 < 2^31.  Integer selection: exact.  Caller
 * workspace of fp4_occ_threshold_workspace_bytes(x_dtype) bytes.
 * fp4_occ_max_outliers: n - ceil(q n), the most elements |x| > tau can hold
 * (the capacity fp4_occ_gemm needs; host arithmetic in double).           */
size_t fp4_occ_threshold_workspace_bytes(int32_t x_dtype);
int64_t fp4_occ_max_outliers(int64_t rows, int64_t cols, double q);
int fp4_occ_threshold(fp4_ctx* ctx, const void* x, int32_t x_dtype, int64_t rows, int64_t cols, int64_t ldx,
                      double q, float* tau, int64_t* n_outliers, void* workspace, size_t ws_bytes, void* stream);

/* fp4_occ_quantize: quantize X_c = clamp(x, -tau, tau) (tau device fp32) like
 * fp4_quantize with transpose = 0, rht = 0 and 1D scaling (other params ->
 * FP4_ERR_UNSUPPORTED).  NVFP4: g = tau / 2688 (tau is the amax of X_c).
 * col_counts (device float[cols], may be NULL): overwritten with the number of
 * outliers |x| > tau in each column (exact integers).                      */
int fp4_occ_quantize(fp4_ctx* ctx, const void* x, int32_t x_dtype, int64_t rows, int64_t cols, int64_t ldx,
                     const fp4_quant_params* p, const float* tau, uint8_t* codes, uint8_t* scales,
                     float* tensor_scale, float* col_counts, void* stream);

/* fp4_occ_gemm: Y[M,N] = alpha Q(X_c) Q(W)^T + dX W^T with xq = fp4_occ_quantize's
 * output (FP4_SF_MMA), wq = W quantized (FP4_SF_MMA), w_bf16 = W itself [N][K]
 * (pitch ldw) and x = the unclamped activations [M][K] (bf16 or fp32, pitch
 * ldx).  dX W^T is computed in two parts:
 *  - the k_dense columns with the most outliers (col_counts from
 *    fp4_occ_quantize; ties to the lower index) become extra bf16 K columns of
 *    the FP4 GEMM: A_ext = bf16(dX_H / alpha), B_ext = W_H (alpha = gX gW,
 *    1 for MXFP4), accumulated with the FP4 part on the tensor cores;
 *  - every other outlier (|x| > tau) is listed per row, and after the GEMM
 *    stored Y a second pass adds v * W^T[k, :] to its row of Y in fp32, in
 *    list order (a bf16 Y is rounded once before and once after: each
 *    rounding within 2^-9).
 * k_dense = 0 sends all outliers to the second part (col_counts may be NULL).
 * An outlier so large that dX / alpha leaves the bf16 range makes its extra
 * column infinite (|x| / tau ~ 1e28 for weights of amax 1e-3).
 * max_outliers bounds the outliers of the second part (fp4_occ_max_outliers
 * is always enough); a list that would outgrow it sets the context's status
 * (fp4_sync_status -> FP4_ERR_TOO_LARGE) and the rows that did not fit are not
 * compensated.  out_dtype bf16 or fp32, pitch ldy (16-byte rows).  Caller
 * workspace of fp4_occ_gemm_workspace_bytes(M, N, K, k_dense, max_outliers). */
size_t fp4_occ_gemm_workspace_bytes(int64_t m, int64_t n, int64_t k, int32_t k_dense, int64_t max_outliers);
int fp4_occ_gemm(fp4_ctx* ctx, const void* x, int32_t x_dtype, int64_t ldx, const void* w_bf16, int64_t ldw,
                 const fp4_operand* xq, const fp4_operand* wq, const float* tau, const float* col_counts,
                 int32_t k_dense, int64_t max_outliers, int32_t out_dtype, void* y, int64_t ldy, void* workspace,
                 size_t ws_bytes, void* stream);

/* ---- quantization quality ([msr] §三 reports cosine similarity, MSE, SNR;
 *      [grad] §5.1 a relative error per block size)
 * sums (device double[4], overwritten) = sum x^2, sum x_hat^2, sum x x_hat,
 * sum (x - x_hat)^2 over the rows x k tensor x (blocks along cols, any block
 * of 16-128, k % 16 == 0) and its quantization q, with
 *   beta == 0: x_hat = dequant(q) (+ x - clamp(x, -tau, tau) when tau is
 *              non-NULL: the OCC reconstruction);
 *   beta > 0:  x_hat = s Q_soft(x / s), the sigmoid-smoothed value with q's
 *              scales (q->codes unused; tau must be NULL).
 * fp64 accumulation.
 * stats (device double[4], may be NULL) = the quality numbers of those pages,
 * formed on the device from the sums with n = rows * k:
 *   stats[0] cosine similarity  s2 / sqrt(s0 s1)
 *   stats[1] mean squared error s3 / n
 *   stats[2] SNR in dB          10 log10(s0 / s3)   (+inf when s3 = 0)
 *   stats[3] relative L2 error  sqrt(s3 / s0)
 * A ratio with a zero denominator otherwise gives NaN.                     */
int fp4_quant_error_stats(fp4_ctx* ctx, const void* x, int32_t x_dtype, int64_t ldx, const fp4_operand* q,
                          const float* tau, float beta, double* sums, double* stats, void* stream);

/* ---- block-scaled FP4 GEMM ([msr] §四: the GEMMs are >95% of the compute)
 * C[M,N] = alpha * sum_k A[m,k] * B[n,k]  (TN: both operands K-major), FP32
 * accumulation on tcgen05 tensor cores, alpha = gA * gB (NVFP4) or 1 (MXFP4).
 * accumulate = 1: C += result.  out_dtype bf16 or fp32, pitch ldc.
 * Requirements: A and B same format, sf_layout FP4_SF_MMA, k % 32 == 0,
 * code and output pointers 16-byte aligned, ldc*size % 16 == 0.             */
int fp4_gemm(fp4_ctx* ctx, const fp4_operand* A, const fp4_operand* B, int32_t out_dtype,
             void* C, int64_t ldc, int32_t accumulate, void* stream);

/* fp4_gemm_quant_a: C = Q(X) B^T with the activation's quantization fused into
 * the GEMM's operand producer ([outlier] §4.1's forward operand: round to
 * nearest, 1D blocks along K, which needs no tensor-wide amax).  X is bf16
 * [m][k] with pitch ldx (a multiple of 8 elements, 16-byte aligned), k = B->k;
 * inside the GEMM each tile quantizes its rows of X as fp4_quantize does with
 * MXFP4, block 32, RTN (Q(x) = s round(x / s), [grad] §2.1; E8M0 scale,
 * [lowprec] §1.1) and multiplies them with B, an MXFP4 operand in the
 * FP4_SF_MMA layout.  Every 256 output columns quantize X's rows again.
 * a_codes / a_scales: both NULL, or both given (16-byte aligned) to receive
 * X's quantization as well: codes [m][k/2] and FP4_SF_MMA scales of
 * fp4_scales_bytes(m, k, FP4_FMT_MXFP4, FP4_SF_MMA, 0) bytes, padding
 * included, the same bytes fp4_quantize writes; written only when B has rows.
 * out_dtype, C and ldc as fp4_gemm (no accumulate).  C equals fp4_quantize
 * followed by fp4_gemm bit for bit.  FP4_ERR_UNSUPPORTED for an NVFP4 B.   */
int fp4_gemm_quant_a(fp4_ctx* ctx, const void* x_bf16, int64_t m, int64_t ldx, const fp4_operand* B,
                     int32_t out_dtype, void* C, int64_t ldc, uint8_t* a_codes, uint8_t* a_scales, void* stream);

/* ---- hot-channel compensation ([outlier] §3.1-3.2, §4.1)
 * fp4_hcp_num_hot: h = ceil(ratio * k), the number of hot channels out of k
 * when the "top 9%" ([outlier] §4.1: ratio 0.09) are compensated; the product
 * is taken in double precision.  Returns h (0 <= h <= k), or -1 when k < 0 or
 * ratio lies outside [0, 1].  Host arithmetic only.                        */
int32_t fp4_hcp_num_hot(int64_t k, double ratio);

/* fp4_hcp_select: e_c = sum_m (X[m,c] - X_hat[m,c])^2 over the M rows of the
 * bf16 activation X (pitch ldx) and its quantization xq (blocks along K);
 * writes the k_hot channels with the largest e_c, ascending, to hot_idx
 * (device int32[k_hot]); ties go to the lower index.  Caller workspace of
 * fp4_hcp_select_workspace_bytes(K) bytes.                                  */
size_t fp4_hcp_select_workspace_bytes(int64_t k);
int fp4_hcp_select(fp4_ctx* ctx, const void* x_bf16, int64_t ldx, const fp4_operand* xq,
                   int32_t k_hot, int32_t* hot_idx, void* workspace, size_t ws_bytes,
                   void* stream);

/* fp4_hcp_quantize_zeroed: quantize X with the k_hot columns hot_idx (device
 * int32, ascending, as fp4_hcp_select writes them) set to zero, like
 * fp4_quantize with transpose 0, rht 0, 1D scaling and the format's own block
 * (else FP4_ERR_UNSUPPORTED); NVFP4: g from the amax of the zeroed tensor.
 * The operand of fp4_hcp_gemm's order 0.                                   */
int fp4_hcp_quantize_zeroed(fp4_ctx* ctx, const void* x, int32_t x_dtype, int64_t rows, int64_t cols, int64_t ldx,
                            const fp4_quant_params* p, const int32_t* hot_idx, int32_t k_hot, uint8_t* codes,
                            uint8_t* scales, float* tensor_scale, void* stream);

/* fp4_hcp_gemm: Y = alpha * (X_hat W_hat^T + A_ext B_ext^T) with bf16 extra K
 * columns on the hot channels H (order 2, "S-O2-B"):
 *   A_ext = [X - X_hat | X]_H,  B_ext = [W_hat | W - W_hat]_H / alpha
 * (order 1 = the page's literal concat: A_ext = X_H, B_ext = (W - W_hat)_H / alpha;
 *  order 0 = hot channels zeroed: xq from fp4_hcp_quantize_zeroed, A_ext = X_H,
 *  B_ext = W_H / alpha, so Y = alpha Q(X_0) W_hat^T + X_H W_H^T).
 * mode FP4_HCP_SINGLE: one kernel, FP4 K-steps then bf16 K-steps into one
 * TMEM accumulator; FP4_HCP_TWO: the FP4 GEMM, then a bf16 GEMM with C +=;
 * FP4_HCP_TWO_FP8: the FP4 GEMM, then an E4M3 GEMM (tcgen05 kind::f8f6f4)
 * over the same columns without the 1/alpha, each row of A_ext and B_ext
 * scaled by its own fp32 amax/448 ([msr] §六 runs its compensation in FP8):
 * C += s_A[m] s_B[n] sum_j a8[m,j] b8[n,j];  FP4_HCP_SINGLE_MXFP8: one kernel,
 * the bf16 tail's columns (B / alpha) as MXFP8 in the FP4 accumulator
 * (tcgen05 kind::mxf8f6f4): each part padded to 32 columns, blocks of 32 with
 * an E8M0 scale 2^e, e the smallest exponent keeping the block amax <= 448,
 * and E4M3 elements (nearest, ties to even).
 * X (M x K) and W (N x K) bf16 with pitches ldx, ldw; xq, wq their
 * quantizations (FP4_SF_MMA).  Workspace: fp4_hcp_workspace_bytes().       */
size_t fp4_hcp_workspace_bytes(int64_t m, int64_t n, int32_t k_hot, int32_t order);
int fp4_hcp_gemm(fp4_ctx* ctx, const void* x_bf16, int64_t ldx, const void* w_bf16, int64_t ldw,
                 const fp4_operand* xq, const fp4_operand* wq, const int32_t* hot_idx,
                 int32_t k_hot, int32_t mode, int32_t order, void* workspace, size_t ws_bytes,
                 int32_t out_dtype, void* y, int64_t ldy, void* stream);

/* fp4_hcp_select_noalloc: the same selection as fp4_hcp_select, for callers
 * that must not allocate device memory.  Some callers cannot: a framework that
 * hands every byte of the GPU to its own caching pool, a serving loop whose
 * latency budget cannot absorb the device-wide synchronization cudaMalloc and
 * cudaFree may cause, or code running where the allocator is off limits.  This
 * entry point needs neither a context nor a workspace: its scratch (per-channel
 * errors and flags) is a fixed array inside the library, FP4_NOALLOC_MAX_CHANNELS
 * channels (512 KiB), which every GPU that loads the library keeps until the
 * process exits.  The pages have no counterpart; it exists for such callers.
 *  - K > FP4_NOALLOC_MAX_CHANNELS returns FP4_ERR_TOO_LARGE (nothing launched).
 *  - Every call looks up the array's device address on the current device
 *    (cudaGetSymbolAddress).  The first call on a device may thereby load the
 *    library's device code, which puts the module and its array in device
 *    memory outside any caller pool; make that first call before any stream
 *    capture.  Later calls allocate nothing.
 *  - All calls share the one array: calls that overlap on the GPU (different
 *    streams, or different host threads, on the same device) race and give
 *    wrong results.  Each call clears the error sums it accumulates.
 *  - Calls no cudaMalloc, cudaFree or other allocating routine.
 * Arguments, validation, layout and result as fp4_hcp_select.              */
#define FP4_NOALLOC_MAX_CHANNELS 65536
int fp4_hcp_select_noalloc(const void* x_bf16, int64_t ldx, const fp4_operand* xq, int32_t k_hot,
                           int32_t* hot_idx, void* stream);

/* ---- element encoders (the "nearest of the 16 FP4 values" step, [msr] §六)
 * fp4_encode_e2m1: codes[i] = RTN E2M1 code of xs[i] (one code per byte).
 *   method 0: the hardware cvt.rn.satfinite.e2m1x2 conversion;
 *   method 1: a compare chain against the grid midpoints.
 * fp4_encode_e4m3: out[i] = E4M3 byte of t[i], round to nearest even,
 *   saturating at 448 (the NVFP4 block-scale encoding).                      */
int fp4_encode_e2m1(fp4_ctx* ctx, const float* xs, uint8_t* codes, int64_t n, int32_t method,
                    void* stream);
int fp4_encode_e4m3(fp4_ctx* ctx, const float* t, uint8_t* out, int64_t n, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* FP4_GB300_H */
