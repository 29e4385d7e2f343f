// C ABI entry points: argument validation, context handling and dispatch to
// the kernels.  See include/fp4.h for the contract of each call.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <new>

#include "fp4_internal.h"

using namespace fp4;

namespace {

constexpr int kDefaultSms = 148;

int esize(int dt) { return dt == FP4_DTYPE_BF16 ? 2 : 4; }
bool dtype_ok(int dt) { return dt == FP4_DTYPE_BF16 || dt == FP4_DTYPE_F32; }
bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
int block_of(int fmt) { return fmt == FP4_FMT_MXFP4 ? 32 : 16; }
bool block_ok(int b) { return b == 16 || b == 32 || b == 64 || b == 128; }
// elements per scale of an operand (0 = the format's own block)
int op_block(const fp4_operand* q) { return q->block ? q->block : block_of(q->format); }
bool native_block(const fp4_operand* q) { return op_block(q) == block_of(q->format); }

// Philox4x32-10 word 0 for counter 0 (host side, for the RHT sign bits)
uint32_t rht_signs_host(uint64_t seed) {
  uint32_t c[4] = {0, 0, 0, 0};
  uint32_t k0 = (uint32_t)seed, k1 = (uint32_t)(seed >> 32);
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    uint64_t p0 = (uint64_t)0xD2511F53u * c[0], p1 = (uint64_t)0xCD9E8D57u * c[2];
    uint32_t n0 = (uint32_t)(p1 >> 32) ^ c[1] ^ k0, n1 = (uint32_t)p1;
    uint32_t n2 = (uint32_t)(p0 >> 32) ^ c[3] ^ k1, n3 = (uint32_t)p0;
    c[0] = n0; c[1] = n1; c[2] = n2; c[3] = n3;
  }
  return c[0] & 0xFFFFu;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? FP4_OK : FP4_ERR_CUDA; }

// format / block / enum checks shared by the quantize calls
int check_params(const fp4_quant_params* p) {
  if (!p) return FP4_ERR_INVALID_ARG;
  if (p->format != FP4_FMT_MXFP4 && p->format != FP4_FMT_NVFP4) return FP4_ERR_UNSUPPORTED;
  if (!block_ok(p->block)) return FP4_ERR_UNSUPPORTED;
  if (p->rounding != FP4_ROUND_RTN && p->rounding != FP4_ROUND_SR) return FP4_ERR_INVALID_ARG;
  if (p->scaling != FP4_SCALING_1D && p->scaling != FP4_SCALING_2D) return FP4_ERR_INVALID_ARG;
  if (p->scaling == FP4_SCALING_2D && p->format != FP4_FMT_NVFP4) return FP4_ERR_UNSUPPORTED;
  if ((p->transpose != 0 && p->transpose != 1) || (p->rht != 0 && p->rht != 1)) return FP4_ERR_INVALID_ARG;
  if (p->sf_layout != FP4_SF_ROWMAJOR && p->sf_layout != FP4_SF_MMA) return FP4_ERR_INVALID_ARG;
  // blocks other than the format's own: row layout, 1D, row-major scales only
  if (p->block != block_of(p->format) &&
      (p->transpose || p->scaling != FP4_SCALING_1D || p->sf_layout != FP4_SF_ROWMAJOR))
    return FP4_ERR_UNSUPPORTED;
  return FP4_OK;
}

// a pointer may be NULL only when the buffer it names has no elements
bool present(const void* p, bool empty) { return p != nullptr || empty; }

int check_input(const void* x, int dt, int64_t rows, int64_t cols, int64_t ldx) {
  if (rows < 0 || cols < 0 || ldx < cols || !dtype_ok(dt)) return FP4_ERR_INVALID_ARG;
  if (!present(x, rows == 0 || cols == 0)) return FP4_ERR_INVALID_ARG;
  if (rows > 0 && cols > 0 && (!al16(x) || (ldx * esize(dt)) % 16 != 0)) return FP4_ERR_MISALIGNED;
  return FP4_OK;
}

int check_operand(const fp4_operand* q, bool need_codes) {
  if (!q || q->rows < 0 || q->k < 0) return FP4_ERR_INVALID_ARG;
  const bool empty = q->rows == 0 || q->k == 0;
  if (!present(q->scales, empty) || (need_codes && !present(q->codes, empty))) return FP4_ERR_INVALID_ARG;
  if (q->format != FP4_FMT_MXFP4 && q->format != FP4_FMT_NVFP4) return FP4_ERR_UNSUPPORTED;
  if (q->sf_layout != FP4_SF_ROWMAJOR && q->sf_layout != FP4_SF_MMA) return FP4_ERR_INVALID_ARG;
  if (q->block != 0 && !block_ok(q->block)) return FP4_ERR_UNSUPPORTED;
  if (!native_block(q) && q->sf_layout != FP4_SF_ROWMAJOR) return FP4_ERR_UNSUPPORTED;
  if (q->k % op_block(q) != 0) return FP4_ERR_INVALID_ARG;
  if (q->format == FP4_FMT_NVFP4 && !present(q->tensor_scale, empty)) return FP4_ERR_INVALID_ARG;
  if (need_codes && !al16(q->codes)) return FP4_ERR_MISALIGNED;
  // MMA-layout scales are read by TMA and by 32-bit loads (one word = 4 scales)
  if (!empty && q->sf_layout == FP4_SF_MMA && !al16(q->scales)) return FP4_ERR_MISALIGNED;
  return FP4_OK;
}

// a new amax generation for the context's tagged slots (never 0); when the
// 32-bit count wraps, the slots are zeroed once on the stream, so that values
// left by the high generations before the wrap cannot win
uint32_t next_gen(fp4_ctx* ctx, cudaStream_t st) {
  if (++ctx->amax_gen == 0) {
    ctx->amax_gen = 1;
    (void)cudaMemsetAsync(ctx->scratch->amax, 0, sizeof(ctx->scratch->amax), st);
  }
  return ctx->amax_gen;
}

QuantOut make_out(const fp4_quant_params* p, uint8_t* codes, uint8_t* scales, float* ts, const float* amax,
                  int64_t out_rows, int64_t blocked) {
  QuantOut o{};
  o.codes = codes;
  o.scales = scales;
  o.tensor_scale = ts;
  o.amax = amax;
  o.out_rows = out_rows;
  o.out_cols = blocked;
  o.nsf_row = blocked / p->block;
  o.nsf_pad = nsf_padded(blocked, p->format);
  o.sf_layout = p->sf_layout;
  o.rounding = p->rounding;
  o.rht = p->rht;
  o.sr_stream = p->sr_stream;
  o.sr_seed = p->sr_seed;
  o.sr_offset = p->sr_offset;
  o.rht_signs = p->rht ? rht_signs_host(p->rht_seed) : 0u;
  o.keys = philox_round_keys(p->sr_seed);
  return o;
}

// zero the padding of an MMA-layout scale buffer (only when there is any)
cudaError_t clear_sf_padding(const fp4_quant_params* p, uint8_t* scales, int64_t out_rows, int64_t blocked,
                             cudaStream_t st) {
  if (p->sf_layout != FP4_SF_MMA) return cudaSuccess;
  if (out_rows % 128 == 0 && blocked % 256 == 0) return cudaSuccess;
  return cudaMemsetAsync(scales, 0, fp4_scales_bytes(out_rows, blocked, p->format, FP4_SF_MMA, 0), st);
}

// argument checks of the hot-channel selection, shared by both of its entry
// points so that they accept and reject the same calls
int check_hcp_select(const void* x_bf16, int64_t ldx, const fp4_operand* xq, int32_t k_hot, const int32_t* hot_idx) {
  if (k_hot > 0 && !hot_idx) return FP4_ERR_INVALID_ARG;
  int s = check_operand(xq, true);
  if (s) return s;
  if (!native_block(xq)) return FP4_ERR_UNSUPPORTED;
  s = check_input(x_bf16, FP4_DTYPE_BF16, xq->rows, xq->k, ldx);
  if (s) return s;
  if (k_hot < 0 || k_hot > xq->k) return FP4_ERR_INVALID_ARG;
  return FP4_OK;
}

}  // namespace

namespace fp4 {
int validate_hcp_select(const void* x_bf16, int64_t ldx, const fp4_operand* xq, int32_t k_hot,
                        const int32_t* hot_idx) {
  return check_hcp_select(x_bf16, ldx, xq, k_hot, hot_idx);
}
}  // namespace fp4

extern "C" {

const char* fp4_status_string(int s) {
  switch (s) {
    case FP4_OK: return "ok";
    case FP4_ERR_INVALID_ARG: return "invalid argument";
    case FP4_ERR_UNSUPPORTED: return "unsupported format/block/mode combination";
    case FP4_ERR_MISALIGNED: return "pointer or pitch not 16-byte aligned";
    case FP4_ERR_CUDA: return "CUDA call failed";
    case FP4_ERR_TIMEOUT: return "device wait timed out";
    case FP4_ERR_TOO_LARGE: return "input exceeds the fixed scratch limit of this entry point";
    default: return "unknown status";
  }
}

size_t fp4_scales_bytes(int64_t rows, int64_t k, int32_t format, int32_t sf_layout, int32_t block) {
  if (rows <= 0 || k <= 0) return 0;
  int B = block ? block : block_of(format);
  if (!block_ok(B) || (sf_layout == FP4_SF_MMA && B != block_of(format))) return 0;
  if (sf_layout == FP4_SF_ROWMAJOR) return (size_t)(rows * (k / B));
  return (size_t)(cdiv(rows, 128) * 128 * nsf_padded(k, format));
}

int fp4_create(fp4_ctx** out) {
  if (!out) return FP4_ERR_INVALID_ARG;
  *out = nullptr;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FP4_ERR_CUDA;
  fp4_ctx* c = new (std::nothrow) fp4_ctx{};
  if (!c) return FP4_ERR_CUDA;
  c->device = dev;
  if (cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) c->num_sms = kDefaultSms;
  if (cudaMalloc(&c->scratch, sizeof(fp4_ctx_scratch)) != cudaSuccess) {
    delete c;
    return FP4_ERR_CUDA;
  }
  if (cudaMemset(c->scratch, 0, sizeof(fp4_ctx_scratch)) != cudaSuccess) {
    cudaFree(c->scratch);
    delete c;
    return FP4_ERR_CUDA;
  }
  *out = c;
  return FP4_OK;
}

void fp4_destroy(fp4_ctx* ctx) {
  if (!ctx) return;
  cudaFree(ctx->scratch);
  delete ctx;
}

int fp4_sync_status(fp4_ctx* ctx, void* stream) {
  if (!ctx) return FP4_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return FP4_ERR_CUDA;
  unsigned int status = 0;
  if (cudaMemcpy(&status, &ctx->scratch->status, sizeof(status), cudaMemcpyDeviceToHost) != cudaSuccess)
    return FP4_ERR_CUDA;
  if (status) {
    if (cudaMemset(&ctx->scratch->status, 0, sizeof(unsigned int)) != cudaSuccess) return FP4_ERR_CUDA;
    if (status & FP4_DEVICE_TIMEOUT) return FP4_ERR_TIMEOUT;
    if (status & FP4_DEVICE_OVERFLOW) return FP4_ERR_TOO_LARGE;
  }
  return FP4_OK;
}

int fp4_amax(fp4_ctx* ctx, const void* x, int32_t x_dtype, int64_t rows, int64_t cols, int64_t ldx,
             int32_t rht_axis, uint64_t rht_seed, float* amax_out, void* stream) {
  if (!ctx || !amax_out) return FP4_ERR_INVALID_ARG;
  int s = check_input(x, x_dtype, rows, cols, ldx);
  if (s) return s;
  if (rht_axis < -1 || rht_axis > 1) return FP4_ERR_INVALID_ARG;
  if ((rht_axis == 1 && cols % 16) || (rht_axis == 0 && rows % 16)) return FP4_ERR_INVALID_ARG;
  uint32_t signs = rht_axis >= 0 ? rht_signs_host(rht_seed) : 0u;
  return cuda_status(launch_amax(x, x_dtype, rows, cols, ldx, rht_axis, signs, amax_out, 0u, ctx->num_sms,
                                 static_cast<cudaStream_t>(stream)));
}

int fp4_quantize(fp4_ctx* ctx, const void* x, int32_t x_dtype, int64_t rows, int64_t cols, int64_t ldx,
                 const fp4_quant_params* p, const float* given_amax, uint8_t* codes, uint8_t* scales,
                 float* tensor_scale, void* stream) {
  if (!ctx || !present(codes, rows == 0 || cols == 0) || !present(scales, rows == 0 || cols == 0))
    return FP4_ERR_INVALID_ARG;
  int s = check_params(p);
  if (s) return s;
  s = check_input(x, x_dtype, rows, cols, ldx);
  if (s) return s;
  const int64_t out_rows = p->transpose ? cols : rows, blocked = p->transpose ? rows : cols;
  if (blocked % p->block) return FP4_ERR_INVALID_ARG;
  if (p->scaling == FP4_SCALING_2D && out_rows % 16) return FP4_ERR_INVALID_ARG;
  if (!al16(codes)) return FP4_ERR_MISALIGNED;
  if (rows == 0 || cols == 0) return FP4_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const float* amax = given_amax;
  if (p->format == FP4_FMT_NVFP4 && !amax) {
    float* slot = reinterpret_cast<float*>(&ctx->scratch->amax[0]);
    int axis = p->rht ? (p->transpose ? 0 : 1) : -1;
    cudaError_t e = launch_amax(x, x_dtype, rows, cols, ldx, axis, rht_signs_host(p->rht_seed), slot, next_gen(ctx, st),
                                ctx->num_sms, st);
    if (e != cudaSuccess) return FP4_ERR_CUDA;
    amax = slot;
  }
  if (clear_sf_padding(p, scales, out_rows, blocked, st) != cudaSuccess) return FP4_ERR_CUDA;
  QuantOut o = make_out(p, codes, scales, tensor_scale, amax, out_rows, blocked);
  cudaError_t e;
  if (p->transpose && p->scaling == FP4_SCALING_1D && p->block == block_of(p->format) &&
      mx_tiled_supported(x_dtype, p->format, nullptr, &o, rows, cols, ldx))
    return cuda_status(launch_quant_mx_tiled(x, rows, cols, ldx, nullptr, &o, &ctx->scratch->status, ctx->num_sms, st));
  if (p->block != block_of(p->format))
    e = launch_quant_rows_blk(x, x_dtype, rows, cols, ldx, p->format, p->block, o, ctx->num_sms, st);
  else if (!p->transpose && p->scaling == FP4_SCALING_1D)
    e = launch_quant_rows(x, x_dtype, rows, cols, ldx, p->format, o, ctx->num_sms, st);
  else
    e = launch_quant_tile(x, x_dtype, rows, cols, ldx, p->format, p->scaling == FP4_SCALING_2D, p->transpose != 0, o,
                          ctx->num_sms, st);
  return cuda_status(e);
}

int fp4_quantize_dual(fp4_ctx* ctx, const void* x, int32_t x_dtype, int64_t rows, int64_t cols, int64_t ldx,
                      const fp4_quant_params* pr, const fp4_quant_params* pc, const float* given_amax_rows,
                      const float* given_amax_cols, uint8_t* codes_rows, uint8_t* scales_rows, float* ts_rows,
                      uint8_t* codes_cols, uint8_t* scales_cols, float* ts_cols, void* stream) {
  const bool empty = rows == 0 || cols == 0;
  if (!ctx || !present(codes_rows, empty) || !present(scales_rows, empty) || !present(codes_cols, empty) ||
      !present(scales_cols, empty))
    return FP4_ERR_INVALID_ARG;
  int s = check_params(pr);
  if (s) return s;
  s = check_params(pc);
  if (s) return s;
  if (pr->format != pc->format || pr->transpose != 0 || pc->transpose != 1) return FP4_ERR_INVALID_ARG;
  if (pr->block != block_of(pr->format) || pc->block != block_of(pc->format)) return FP4_ERR_UNSUPPORTED;
  s = check_input(x, x_dtype, rows, cols, ldx);
  if (s) return s;
  if (cols % pr->block || rows % pc->block) return FP4_ERR_INVALID_ARG;
  // 16x16 2D scaling: output rows in groups of 16 (rows of x for the row
  // layout, cols of x for the transposed one)
  if ((pr->scaling == FP4_SCALING_2D && rows % 16) || (pc->scaling == FP4_SCALING_2D && cols % 16))
    return FP4_ERR_INVALID_ARG;
  if (!al16(codes_rows) || !al16(codes_cols)) return FP4_ERR_MISALIGNED;
  if (rows == 0 || cols == 0) return FP4_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const float* amax_r = given_amax_rows;
  const float* amax_c = given_amax_cols;
  if (pr->format == FP4_FMT_NVFP4 && (!amax_r || !amax_c)) {
    float* sr = reinterpret_cast<float*>(&ctx->scratch->amax[0]);
    float* sc = reinterpret_cast<float*>(&ctx->scratch->amax[1]);
    cudaError_t e = launch_amax_dual(x, x_dtype, rows, cols, ldx, rht_signs_host(pr->rht_seed),
                                     rht_signs_host(pc->rht_seed), pr->rht != 0, pc->rht != 0, sr, sc, next_gen(ctx, st),
                                     ctx->num_sms, st);
    if (e != cudaSuccess) return FP4_ERR_CUDA;
    if (!amax_r) amax_r = sr;
    if (!amax_c) amax_c = sc;
  }
  if (clear_sf_padding(pr, scales_rows, rows, cols, st) != cudaSuccess) return FP4_ERR_CUDA;
  if (clear_sf_padding(pc, scales_cols, cols, rows, st) != cudaSuccess) return FP4_ERR_CUDA;
  QuantOut orow = make_out(pr, codes_rows, scales_rows, ts_rows, amax_r, rows, cols);
  QuantOut ocol = make_out(pc, codes_cols, scales_cols, ts_cols, amax_c, cols, rows);
  if (pr->scaling == FP4_SCALING_1D && pc->scaling == FP4_SCALING_1D &&
      mx_tiled_supported(x_dtype, pr->format, &orow, &ocol, rows, cols, ldx))
    return cuda_status(launch_quant_mx_tiled(x, rows, cols, ldx, &orow, &ocol, &ctx->scratch->status, ctx->num_sms, st));
  return cuda_status(launch_quant_dual(x, x_dtype, rows, cols, ldx, pr->format, orow, ocol,
                                      pr->scaling == FP4_SCALING_2D, pc->scaling == FP4_SCALING_2D, ctx->num_sms, st));
}

int fp4_dequantize(fp4_ctx* ctx, const fp4_operand* q, int32_t out_dtype, void* out, int64_t ldo, void* stream) {
  if (!ctx || !dtype_ok(out_dtype)) return FP4_ERR_INVALID_ARG;
  int s = check_operand(q, true);
  if (s) return s;
  if (ldo < q->k || !present(out, q->rows == 0 || q->k == 0)) return FP4_ERR_INVALID_ARG;
  if (!al16(out) || (ldo * esize(out_dtype)) % 16) return FP4_ERR_MISALIGNED;
  return cuda_status(launch_dequant(*q, out_dtype, out, ldo, ctx->num_sms, static_cast<cudaStream_t>(stream)));
}

int fp4_rht16(fp4_ctx* ctx, const void* x, int32_t x_dtype, int64_t rows, int64_t cols, int64_t ldx, int32_t axis,
              uint64_t seed, float* y, void* stream) {
  if (!ctx || !present(y, rows == 0 || cols == 0) || (axis != 0 && axis != 1)) return FP4_ERR_INVALID_ARG;
  int s = check_input(x, x_dtype, rows, cols, ldx);
  if (s) return s;
  if ((axis == 1 && cols % 16) || (axis == 0 && rows % 16)) return FP4_ERR_INVALID_ARG;
  if (!al16(y) || (cols * 4) % 16) return FP4_ERR_MISALIGNED;
  return cuda_status(launch_rht16(x, x_dtype, rows, cols, ldx, axis, rht_signs_host(seed), y, ctx->num_sms,
                                  static_cast<cudaStream_t>(stream)));
}

int fp4_dge_backward(fp4_ctx* ctx, const void* x, int32_t x_dtype, int64_t ldx, const fp4_operand* q, const void* dy,
                     int32_t dy_dtype, int64_t lddy, float* dx, int64_t lddx, float k, float clamp, float outside,
                     void* stream) {
  if (!ctx || !(k > 1.0f) || !(clamp > 0.0f)) return FP4_ERR_INVALID_ARG;
  int s = check_operand(q, false);
  if (s) return s;
  if (!native_block(q)) return FP4_ERR_UNSUPPORTED;
  if (!present(dx, q->rows == 0 || q->k == 0)) return FP4_ERR_INVALID_ARG;
  s = check_input(x, x_dtype, q->rows, q->k, ldx);
  if (s) return s;
  s = check_input(dy, dy_dtype, q->rows, q->k, lddy);
  if (s) return s;
  if (lddx < q->k) return FP4_ERR_INVALID_ARG;
  if (!al16(dx) || (lddx * 4) % 16) return FP4_ERR_MISALIGNED;
  return cuda_status(launch_dge(x, x_dtype, ldx, *q, dy, dy_dtype, lddy, dx, lddx, k, clamp, outside, ctx->num_sms,
                                static_cast<cudaStream_t>(stream)));
}

static bool soft_beta_ok(float beta) { return beta > 0.0f && beta <= 1e6f; }

int fp4_soft_forward(fp4_ctx* ctx, const void* x, int32_t x_dtype, int64_t ldx, const fp4_operand* q, float* y,
                     int64_t ldy, float beta, void* stream) {
  if (!ctx || !soft_beta_ok(beta)) return FP4_ERR_INVALID_ARG;
  int s = check_operand(q, false);
  if (s) return s;
  if (!native_block(q)) return FP4_ERR_UNSUPPORTED;
  if (!present(y, q->rows == 0 || q->k == 0)) return FP4_ERR_INVALID_ARG;
  s = check_input(x, x_dtype, q->rows, q->k, ldx);
  if (s) return s;
  if (ldy < q->k) return FP4_ERR_INVALID_ARG;
  if (!al16(y) || (ldy * 4) % 16) return FP4_ERR_MISALIGNED;
  return cuda_status(launch_soft(x, x_dtype, ldx, *q, nullptr, 0, 0, y, ldy, beta, ctx->num_sms,
                                 static_cast<cudaStream_t>(stream)));
}

int fp4_soft_backward(fp4_ctx* ctx, const void* x, int32_t x_dtype, int64_t ldx, const fp4_operand* q,
                      const void* dy, int32_t dy_dtype, int64_t lddy, float* dx, int64_t lddx, float beta,
                      void* stream) {
  if (!ctx || !soft_beta_ok(beta)) return FP4_ERR_INVALID_ARG;
  int s = check_operand(q, false);
  if (s) return s;
  if (!native_block(q)) return FP4_ERR_UNSUPPORTED;
  if (!present(dx, q->rows == 0 || q->k == 0)) return FP4_ERR_INVALID_ARG;
  s = check_input(x, x_dtype, q->rows, q->k, ldx);
  if (s) return s;
  s = check_input(dy, dy_dtype, q->rows, q->k, lddy);
  if (s) return s;
  if (lddx < q->k) return FP4_ERR_INVALID_ARG;
  if (!al16(dx) || (lddx * 4) % 16) return FP4_ERR_MISALIGNED;
  return cuda_status(launch_soft(x, x_dtype, ldx, *q, dy, dy_dtype, lddy, dx, lddx, beta, ctx->num_sms,
                                 static_cast<cudaStream_t>(stream)));
}

// ---- OCC -------------------------------------------------------------------
static uint64_t occ_rank(int64_t n, double q) {
  const double r = std::ceil(q * (double)n);
  return r < 1.0 ? 1u : (uint64_t)r;
}

size_t fp4_occ_threshold_workspace_bytes(int32_t x_dtype) {
  return dtype_ok(x_dtype) ? occ_threshold_ws_bytes(x_dtype) : 0;
}

int64_t fp4_occ_max_outliers(int64_t rows, int64_t cols, double q) {
  if (rows <= 0 || cols <= 0 || !(q > 0.0 && q <= 1.0)) return 0;
  const int64_t n = rows * cols;
  return n - (int64_t)occ_rank(n, q);
}

int fp4_occ_threshold(fp4_ctx* ctx, const void* x, int32_t x_dtype, int64_t rows, int64_t cols, int64_t ldx,
                      double q, float* tau, int64_t* n_outliers, void* workspace, size_t ws_bytes, void* stream) {
  if (!ctx || !tau || !n_outliers || !(q > 0.0 && q <= 1.0)) return FP4_ERR_INVALID_ARG;
  int s = check_input(x, x_dtype, rows, cols, ldx);
  if (s) return s;
  if (cols % 8) return FP4_ERR_INVALID_ARG;
  if (rows * cols / 8 >= (int64_t(1) << 31)) return FP4_ERR_TOO_LARGE;
  if (!workspace || ws_bytes < occ_threshold_ws_bytes(x_dtype)) return FP4_ERR_INVALID_ARG;
  if (!al16(workspace)) return FP4_ERR_MISALIGNED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (rows == 0 || cols == 0) {
    if (cudaMemsetAsync(tau, 0, sizeof(float), st) != cudaSuccess) return FP4_ERR_CUDA;
    return cuda_status(cudaMemsetAsync(n_outliers, 0, sizeof(int64_t), st));
  }
  return cuda_status(launch_occ_threshold(x, x_dtype, rows, cols, ldx, occ_rank(rows * cols, q), workspace, tau,
                                          reinterpret_cast<long long*>(n_outliers), ctx->num_sms, st));
}

int fp4_occ_quantize(fp4_ctx* ctx, const void* x, int32_t x_dtype, int64_t rows, int64_t cols, int64_t ldx,
                     const fp4_quant_params* p, const float* tau, uint8_t* codes, uint8_t* scales,
                     float* tensor_scale, float* col_counts, void* stream) {
  const bool empty = rows == 0 || cols == 0;
  if (!ctx || !tau || !present(codes, empty) || !present(scales, empty)) return FP4_ERR_INVALID_ARG;
  int s = check_params(p);
  if (s) return s;
  if (p->transpose || p->rht || p->scaling != FP4_SCALING_1D || p->block != block_of(p->format))
    return FP4_ERR_UNSUPPORTED;
  s = check_input(x, x_dtype, rows, cols, ldx);
  if (s) return s;
  if (cols % p->block) return FP4_ERR_INVALID_ARG;
  if (rows * (cols / p->block) >= (int64_t(1) << 31)) return FP4_ERR_TOO_LARGE;
  if (!al16(codes)) return FP4_ERR_MISALIGNED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (col_counts && cols > 0 && cudaMemsetAsync(col_counts, 0, sizeof(float) * cols, st) != cudaSuccess)
    return FP4_ERR_CUDA;
  if (empty) return FP4_OK;
  if (clear_sf_padding(p, scales, rows, cols, st) != cudaSuccess) return FP4_ERR_CUDA;
  QuantOut o = make_out(p, codes, scales, tensor_scale, tau, rows, cols);
  o.clamp = tau;
  o.col_counts = col_counts;
  return cuda_status(launch_quant_rows_clamped(x, x_dtype, rows, cols, ldx, p->format, o, ctx->num_sms, st));
}

size_t fp4_occ_gemm_workspace_bytes(int64_t m, int64_t n, int64_t k, int32_t k_dense, int64_t max_outliers) {
  if (m <= 0 || n <= 0 || k <= 0 || k_dense < 0 || max_outliers < 0) return 0;
  return occ_layout(m, n, k, k_dense, max_outliers).bytes;
}

int fp4_occ_gemm(fp4_ctx* ctx, const void* x, int32_t x_dtype, int64_t ldx, const void* w_bf16, int64_t ldw,
                 const fp4_operand* xq, const fp4_operand* wq, const float* tau, const float* col_counts,
                 int32_t k_dense, int64_t max_outliers, int32_t out_dtype, void* y, int64_t ldy, void* workspace,
                 size_t ws_bytes, void* stream) {
  if (!ctx || !tau || !dtype_ok(out_dtype)) return FP4_ERR_INVALID_ARG;
  int s = check_operand(xq, true);
  if (s) return s;
  if (!native_block(xq)) return FP4_ERR_UNSUPPORTED;
  s = check_operand(wq, true);
  if (s) return s;
  if (!native_block(wq)) return FP4_ERR_UNSUPPORTED;
  if (xq->format != wq->format || xq->k != wq->k) return FP4_ERR_INVALID_ARG;
  if (xq->sf_layout != FP4_SF_MMA || wq->sf_layout != FP4_SF_MMA) return FP4_ERR_UNSUPPORTED;
  const int64_t M = xq->rows, N = wq->rows, K = xq->k;
  if (K % 32 || (K == 0 && M > 0 && N > 0)) return FP4_ERR_INVALID_ARG;
  if (M > INT32_MAX || N > INT32_MAX) return FP4_ERR_INVALID_ARG;
  if (k_dense < 0 || k_dense > K || (k_dense > 0 && !col_counts)) return FP4_ERR_INVALID_ARG;
  if (max_outliers < 0 || max_outliers >= (int64_t(1) << 31)) return FP4_ERR_INVALID_ARG;
  s = check_input(x, x_dtype, M, K, ldx);
  if (s) return s;
  s = check_input(w_bf16, FP4_DTYPE_BF16, N, K, ldw);
  if (s) return s;
  if (ldy < N || !present(y, M == 0 || N == 0)) return FP4_ERR_INVALID_ARG;
  if (!al16(y) || (ldy * esize(out_dtype)) % 16) return FP4_ERR_MISALIGNED;
  if (M == 0 || N == 0) return FP4_OK;
  const OccLayout L = occ_layout(M, N, K, k_dense, max_outliers);
  if (!workspace || ws_bytes < L.bytes) return FP4_ERR_INVALID_ARG;
  if (!al16(workspace)) return FP4_ERR_MISALIGNED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_occ_prepare(x, x_dtype, ldx, static_cast<const uint16_t*>(w_bf16), ldw, *xq, *wq, tau,
                                     col_counts, k_dense, max_outliers, workspace, L, &ctx->scratch->status,
                                     ctx->num_sms, st);
  if (e != cudaSuccess) return FP4_ERR_CUDA;
  GemmArgs g{};
  g.A = xq;
  g.B = wq;
  g.fp4_part = true;
  g.out_dtype = out_dtype;
  g.C = y;
  g.ldc = ldy;
  g.status = &ctx->scratch->status;
  g.num_sms = ctx->num_sms;
  uint8_t* base = static_cast<uint8_t*>(workspace);
  if (k_dense > 0) {
    g.a_ext = reinterpret_cast<const uint16_t*>(base + L.a_ext);
    g.b_ext = reinterpret_cast<const uint16_t*>(base + L.b_ext);
    g.kx = L.kx;
  }
  s = launch_gemm(g, st);   // the clamped FP4 product and the dense columns
  if (s) return s;
  return cuda_status(launch_occ_correct(y, ldy, out_dtype, M, N, workspace, L, ctx->num_sms, st));
}

int fp4_quant_error_stats(fp4_ctx* ctx, const void* x, int32_t x_dtype, int64_t ldx, const fp4_operand* q,
                          const float* tau, float beta, double* sums, double* stats, void* stream) {
  if (!ctx || !sums || !(beta >= 0.0f && beta <= 1e6f) || (tau && beta > 0.0f)) return FP4_ERR_INVALID_ARG;
  int s = check_operand(q, beta == 0.0f);
  if (s) return s;
  if (q->k % 16) return FP4_ERR_INVALID_ARG;
  s = check_input(x, x_dtype, q->rows, q->k, ldx);
  if (s) return s;
  return cuda_status(launch_error_stats(x, x_dtype, ldx, *q, op_block(q), tau, beta, sums, stats, ctx->num_sms,
                                        static_cast<cudaStream_t>(stream)));
}

int fp4_gemm(fp4_ctx* ctx, const fp4_operand* A, const fp4_operand* B, int32_t out_dtype, void* C, int64_t ldc,
             int32_t accumulate, void* stream) {
  if (!ctx || !dtype_ok(out_dtype)) return FP4_ERR_INVALID_ARG;
  int s = check_operand(A, true);
  if (s) return s;
  if (!native_block(A)) return FP4_ERR_UNSUPPORTED;
  s = check_operand(B, true);
  if (s) return s;
  if (!native_block(B)) return FP4_ERR_UNSUPPORTED;
  if (!present(C, A->rows == 0 || B->rows == 0)) return FP4_ERR_INVALID_ARG;
  if (A->format != B->format || A->k != B->k) return FP4_ERR_INVALID_ARG;
  if (A->sf_layout != FP4_SF_MMA || B->sf_layout != FP4_SF_MMA) return FP4_ERR_UNSUPPORTED;
  if (A->k % 32) return FP4_ERR_INVALID_ARG;
  if (A->rows > 0 && B->rows > 0 && A->k == 0) return FP4_ERR_INVALID_ARG;
  if (ldc < B->rows) return FP4_ERR_INVALID_ARG;
  // alignment matters only for an output with elements (as for inputs)
  if (A->rows > 0 && B->rows > 0 && (!al16(C) || (ldc * esize(out_dtype)) % 16)) return FP4_ERR_MISALIGNED;
  if (A->rows > INT32_MAX || B->rows > INT32_MAX) return FP4_ERR_INVALID_ARG;
  GemmArgs g{};
  g.A = A;
  g.B = B;
  g.fp4_part = true;
  g.out_dtype = out_dtype;
  g.C = C;
  g.ldc = ldc;
  g.accumulate = accumulate ? 1 : 0;
  g.status = &ctx->scratch->status;
  g.num_sms = ctx->num_sms;
  return launch_gemm(g, static_cast<cudaStream_t>(stream));
}

int fp4_gemm_quant_a(fp4_ctx* ctx, const void* x_bf16, int64_t m, int64_t ldx, const fp4_operand* B,
                     int32_t out_dtype, void* C, int64_t ldc, uint8_t* a_codes, uint8_t* a_scales, void* stream) {
  if (!ctx || !dtype_ok(out_dtype) || m < 0) return FP4_ERR_INVALID_ARG;
  int s = check_operand(B, true);
  if (s) return s;
  if (!native_block(B) || B->format != FP4_FMT_MXFP4 || B->sf_layout != FP4_SF_MMA) return FP4_ERR_UNSUPPORTED;
  const int64_t k = B->k, n = B->rows;
  if (k % 32) return FP4_ERR_INVALID_ARG;
  if (m > 0 && n > 0 && k == 0) return FP4_ERR_INVALID_ARG;
  s = check_input(x_bf16, FP4_DTYPE_BF16, m, k, ldx);
  if (s) return s;
  if (!present(C, m == 0 || n == 0) || ldc < n) return FP4_ERR_INVALID_ARG;
  if ((a_codes == nullptr) != (a_scales == nullptr)) return FP4_ERR_INVALID_ARG;
  if (m > INT32_MAX || n > INT32_MAX || k > INT32_MAX) return FP4_ERR_INVALID_ARG;
  // nothing to compute (an empty X has a NULL pointer; an empty output any pitch)
  if (m == 0 || n == 0) return FP4_OK;
  if (!al16(C) || (ldc * esize(out_dtype)) % 16 || !al16(a_codes) || !al16(a_scales)) return FP4_ERR_MISALIGNED;
  GemmArgs g{};
  g.B = B;
  g.quant_a = true;
  g.fp4_part = true;
  g.out_dtype = out_dtype;
  g.C = C;
  g.ldc = ldc;
  g.status = &ctx->scratch->status;
  g.num_sms = ctx->num_sms;
  g.x_bf16 = x_bf16;
  g.ldx = ldx;
  g.m = m;
  g.qa_codes = a_codes;
  g.qa_scales = a_scales;
  return launch_gemm_pair(g, static_cast<cudaStream_t>(stream));
}

int fp4_hcp_quantize_zeroed(fp4_ctx* ctx, const void* x, int32_t x_dtype, int64_t rows, int64_t cols, int64_t ldx,
                            const fp4_quant_params* p, const int32_t* hot_idx, int32_t k_hot, uint8_t* codes,
                            uint8_t* scales, float* tensor_scale, void* stream) {
  const bool empty = rows == 0 || cols == 0;
  if (!ctx || !present(codes, empty) || !present(scales, empty)) return FP4_ERR_INVALID_ARG;
  int s = check_params(p);
  if (s) return s;
  if (p->transpose || p->rht || p->scaling != FP4_SCALING_1D || p->block != block_of(p->format))
    return FP4_ERR_UNSUPPORTED;
  s = check_input(x, x_dtype, rows, cols, ldx);
  if (s) return s;
  if (cols % p->block || k_hot < 0 || k_hot > cols || (k_hot > 0 && !hot_idx)) return FP4_ERR_INVALID_ARG;
  if (rows * (cols / 16) >= (int64_t(1) << 31)) return FP4_ERR_TOO_LARGE;
  if (!al16(codes)) return FP4_ERR_MISALIGNED;
  if (empty) return FP4_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  float* slot = reinterpret_cast<float*>(&ctx->scratch->amax[0]);
  if (p->format == FP4_FMT_NVFP4) {
    cudaError_t e = launch_amax_zeroed(x, x_dtype, rows, cols, ldx, hot_idx, k_hot, slot, next_gen(ctx, st),
                                       ctx->num_sms, st);
    if (e != cudaSuccess) return FP4_ERR_CUDA;
  }
  if (clear_sf_padding(p, scales, rows, cols, st) != cudaSuccess) return FP4_ERR_CUDA;
  QuantOut o = make_out(p, codes, scales, tensor_scale, slot, rows, cols);
  o.zero_idx = hot_idx;
  o.zero_n = k_hot;
  return cuda_status(launch_quant_rows_zeroed(x, x_dtype, rows, cols, ldx, p->format, o, ctx->num_sms, st));
}

size_t fp4_hcp_select_workspace_bytes(int64_t k) { return k > 0 ? (size_t)k * 8 : 0; }

int32_t fp4_hcp_num_hot(int64_t k, double ratio) {
  if (k < 0 || !(ratio >= 0.0 && ratio <= 1.0)) return -1;
  const double h = std::ceil(ratio * (double)k);
  return (int32_t)std::min<double>(h, (double)std::min<int64_t>(k, INT32_MAX));
}

int fp4_hcp_select(fp4_ctx* ctx, const void* x_bf16, int64_t ldx, const fp4_operand* xq, int32_t k_hot,
                   int32_t* hot_idx, void* workspace, size_t ws_bytes, void* stream) {
  if (!ctx) return FP4_ERR_INVALID_ARG;
  int s = check_hcp_select(x_bf16, ldx, xq, k_hot, hot_idx);
  if (s) return s;
  if (ws_bytes < fp4_hcp_select_workspace_bytes(xq->k) || (xq->k > 0 && !workspace)) return FP4_ERR_INVALID_ARG;
  if (k_hot == 0 || xq->k == 0) return FP4_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  float* err = static_cast<float*>(workspace);
  cudaError_t e = launch_hcp_channel_errors(static_cast<const uint16_t*>(x_bf16), ldx, *xq, err, ctx->num_sms, st);
  if (e == cudaSuccess) e = launch_hcp_topk(err, xq->k, k_hot, hot_idx, st);
  return cuda_status(e);
}

static int64_t hcp_kx(int32_t k_hot, int32_t order) { return cdiv((int64_t)(order == 2 ? 2 : 1) * k_hot, 64) * 64; }

// E4M3 extra columns: K padded to 128 (one 128-byte stage row)
static int64_t hcp_kx8(int32_t k_hot, int32_t order) { return cdiv((int64_t)(order == 2 ? 2 : 1) * k_hot, 128) * 128; }

// MXFP8 extra columns: each part padded to 32 columns, the whole to 128 (one stage)
static int64_t hcp_kxm(int32_t k_hot, int32_t order) {
  return cdiv((int64_t)(order == 2 ? 2 : 1) * cdiv(k_hot, 32) * 32, 128) * 128;
}
// MXFP8 layout: [a8 | b8 | sa | sb], scales of rows padded to 128
static int64_t hcp_mx8_bytes(int64_t m, int64_t n, int64_t kxm, int64_t* off_b8, int64_t* off_sa, int64_t* off_sb) {
  const int64_t b8 = cdiv(m * kxm, 256) * 256;
  const int64_t sa = b8 + cdiv(n * kxm, 256) * 256;
  const int64_t sb = sa + cdiv(m, 128) * 128 * (kxm / 32);
  if (off_b8) *off_b8 = b8;
  if (off_sa) *off_sa = sa;
  if (off_sb) *off_sb = sb;
  return sb + cdiv(n, 128) * 128 * (kxm / 32);
}

// the largest of the bf16 layout [A_ext | B_ext], the E4M3 one [a8 | b8 | sa | sb]
// and the MXFP8 one
size_t fp4_hcp_workspace_bytes(int64_t m, int64_t n, int32_t k_hot, int32_t order) {
  if (m <= 0 || n <= 0 || k_hot <= 0) return 0;
  const int64_t kx = hcp_kx(k_hot, order), kx8 = hcp_kx8(k_hot, order);
  const int64_t bf16 = cdiv(m * kx * 2, 256) * 256 + n * kx * 2;
  const int64_t fp8 = cdiv(m * kx8, 256) * 256 + cdiv(n * kx8, 256) * 256 + cdiv(m * 4, 256) * 256 + n * 4;
  const int64_t mx8 = hcp_mx8_bytes(m, n, hcp_kxm(k_hot, order), nullptr, nullptr, nullptr);
  return (size_t)std::max(std::max(bf16, fp8), mx8);
}

int fp4_hcp_gemm(fp4_ctx* ctx, const void* x_bf16, int64_t ldx, const void* w_bf16, int64_t ldw,
                 const fp4_operand* xq, const fp4_operand* wq, const int32_t* hot_idx, int32_t k_hot, int32_t mode,
                 int32_t order, void* workspace, size_t ws_bytes, int32_t out_dtype, void* y, int64_t ldy,
                 void* stream) {
  if (!ctx || !dtype_ok(out_dtype)) return FP4_ERR_INVALID_ARG;
  if (mode != FP4_HCP_SINGLE && mode != FP4_HCP_TWO && mode != FP4_HCP_TWO_FP8 && mode != FP4_HCP_SINGLE_MXFP8)
    return FP4_ERR_INVALID_ARG;
  if (order < 0 || order > 2) return FP4_ERR_INVALID_ARG;
  int s = check_operand(xq, true);
  if (s) return s;
  if (!native_block(xq)) return FP4_ERR_UNSUPPORTED;
  s = check_operand(wq, true);
  if (s) return s;
  if (!native_block(wq)) return FP4_ERR_UNSUPPORTED;
  if (xq->format != wq->format || xq->k != wq->k) return FP4_ERR_INVALID_ARG;
  if (xq->sf_layout != FP4_SF_MMA || wq->sf_layout != FP4_SF_MMA) return FP4_ERR_UNSUPPORTED;
  if (xq->k % 32 || xq->k == 0) return FP4_ERR_INVALID_ARG;
  if (k_hot < 0 || k_hot > xq->k || (k_hot > 0 && !hot_idx)) return FP4_ERR_INVALID_ARG;
  s = check_input(x_bf16, FP4_DTYPE_BF16, xq->rows, xq->k, ldx);
  if (s) return s;
  s = check_input(w_bf16, FP4_DTYPE_BF16, wq->rows, wq->k, ldw);
  if (s) return s;
  if (ldy < wq->rows || !present(y, xq->rows == 0 || wq->rows == 0)) return FP4_ERR_INVALID_ARG;
  if (!al16(y) || (ldy * esize(out_dtype)) % 16) return FP4_ERR_MISALIGNED;
  const int64_t M = xq->rows, N = wq->rows;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  GemmArgs g{};
  g.A = xq;
  g.B = wq;
  g.fp4_part = true;
  g.out_dtype = out_dtype;
  g.C = y;
  g.ldc = ldy;
  g.status = &ctx->scratch->status;
  g.num_sms = ctx->num_sms;
  if (k_hot == 0 || M == 0 || N == 0) return launch_gemm(g, st);
  if (ws_bytes < fp4_hcp_workspace_bytes(M, N, k_hot, order) || !workspace || !al16(workspace))
    return FP4_ERR_INVALID_ARG;
  if (mode == FP4_HCP_SINGLE_MXFP8) {
    const int64_t kxm = hcp_kxm(k_hot, order);
    int64_t ob8, osa, osb;
    hcp_mx8_bytes(M, N, kxm, &ob8, &osa, &osb);
    uint8_t* base = static_cast<uint8_t*>(workspace);
    cudaError_t e = launch_hcp_gather_mx8(static_cast<const uint16_t*>(x_bf16), ldx,
                                          static_cast<const uint16_t*>(w_bf16), ldw, *xq, *wq, hot_idx, k_hot, order,
                                          kxm, base, base + osa, base + ob8, base + osb, ctx->num_sms, st);
    if (e != cudaSuccess) return FP4_ERR_CUDA;
    g.a_ext = base;
    g.b_ext = base + ob8;
    g.a_ext_sf = base + osa;
    g.b_ext_sf = base + osb;
    g.kx = kxm;
    g.ext_mx8 = true;
    return launch_gemm(g, st);
  }
  if (mode == FP4_HCP_TWO_FP8) {
    const int64_t kx8 = hcp_kx8(k_hot, order);
    uint8_t* base = static_cast<uint8_t*>(workspace);
    uint8_t* a8 = base;
    uint8_t* b8 = a8 + cdiv(M * kx8, 256) * 256;
    float* sa = reinterpret_cast<float*>(b8 + cdiv(N * kx8, 256) * 256);
    float* sb = sa + cdiv(M * 4, 256) * 64;
    cudaError_t e = launch_hcp_gather_fp8(static_cast<const uint16_t*>(x_bf16), ldx,
                                          static_cast<const uint16_t*>(w_bf16), ldw, *xq, *wq, hot_idx, k_hot, order,
                                          kx8, a8, b8, sa, sb, ctx->num_sms, st);
    if (e != cudaSuccess) return FP4_ERR_CUDA;
    s = launch_gemm(g, st);   // base FP4 GEMM
    if (s) return s;
    g.fp4_part = false;       // E4M3 residual GEMM: C += sa[m] sb[n] acc
    g.a_ext = a8;
    g.b_ext = b8;
    g.kx = kx8;
    g.ext_fp8 = true;
    g.row_scale = sa;
    g.col_scale = sb;
    g.accumulate = 1;
    return launch_gemm(g, st);
  }
  const int64_t kx = hcp_kx(k_hot, order);
  uint16_t* a_ext = static_cast<uint16_t*>(workspace);
  uint16_t* b_ext = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(workspace) + cdiv(M * kx * 2, 256) * 256);
  cudaError_t e = launch_hcp_gather(static_cast<const uint16_t*>(x_bf16), ldx, static_cast<const uint16_t*>(w_bf16),
                                    ldw, *xq, *wq, hot_idx, k_hot, order, kx, a_ext, b_ext, ctx->num_sms, st);
  if (e != cudaSuccess) return FP4_ERR_CUDA;
  g.a_ext = a_ext;
  g.b_ext = b_ext;
  if (mode == FP4_HCP_SINGLE) {
    g.kx = kx;
    return launch_gemm(g, st);
  }
  s = launch_gemm(g, st);  // base FP4 GEMM
  if (s) return s;
  g.fp4_part = false;      // residual bf16 GEMM, C +=
  g.kx = kx;
  g.accumulate = 1;
  return launch_gemm(g, st);
}

int fp4_encode_e2m1(fp4_ctx* ctx, const float* xs, uint8_t* codes, int64_t n, int32_t method, void* stream) {
  if (!ctx || !present(xs, n == 0) || !present(codes, n == 0) || n < 0 || (method != 0 && method != 1))
    return FP4_ERR_INVALID_ARG;
  return cuda_status(launch_encode_e2m1(xs, codes, n, method, static_cast<cudaStream_t>(stream)));
}

int fp4_encode_e4m3(fp4_ctx* ctx, const float* t, uint8_t* out, int64_t n, void* stream) {
  if (!ctx || !present(t, n == 0) || !present(out, n == 0) || n < 0) return FP4_ERR_INVALID_ARG;
  return cuda_status(launch_encode_e4m3(t, out, n, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
