// Internal declarations shared by the library's translation units.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/fp4.h"

// Bits of the context's device status word.
#define FP4_DEVICE_TIMEOUT 1u
#define FP4_DEVICE_OVERFLOW 2u   // a device-filled list outgrew its caller-sized buffer

// Device scratch owned by a context: status word + amax slots.  The slots
// hold (generation << 32) | fp32 bits: each amax launch of the context takes
// a new generation, so a slot needs no zeroing before it is reused (the low
// word read as a float is the amax).
struct fp4_ctx_scratch {
  unsigned int status;
  unsigned int pad[3];
  unsigned long long amax[4];
};

struct fp4_ctx {
  int device;
  int num_sms;
  fp4_ctx_scratch* scratch;  // device memory
  uint32_t amax_gen;         // last generation handed out (0 is never used)
};

namespace fp4 {

// Philox4x32-10 round keys (Salmon et al., SC'11): round r uses
// (seed_lo + r * 0x9E3779B9, seed_hi + r * 0xBB67AE85).  They depend on the
// seed only, so the host computes them once and the kernels read them from
// their parameters instead of holding twenty registers.
struct PhiloxRoundKeys {
  uint32_t k0[10], k1[10];
};
__host__ __device__ inline PhiloxRoundKeys philox_round_keys(uint64_t seed) {
  PhiloxRoundKeys k;
  uint32_t a = (uint32_t)seed, b = (uint32_t)(seed >> 32);
  for (int r = 0; r < 10; ++r) {
    k.k0[r] = a;
    k.k1[r] = b;
    a += 0x9E3779B9u;
    b += 0xBB67AE85u;
  }
  return k;
}

struct QuantOut {
  uint8_t* codes;
  uint8_t* scales;
  float* tensor_scale;   // NVFP4 only (may be null)
  const float* amax;     // device amax the NVFP4 scale is derived from
  int64_t out_rows;      // rows of the output layout
  int64_t out_cols;      // elements per output row (the blocked extent)
  int64_t nsf_row;       // scales per output row
  int64_t nsf_pad;       // MMA layout: scales per row padded to 256 elements
  int sf_layout;
  int rounding;
  int rht;
  uint32_t sr_stream;
  uint64_t sr_seed, sr_offset;
  uint32_t rht_signs;    // 16 sign bits
  PhiloxRoundKeys keys;  // of sr_seed
  const float* clamp;    // row quantizer only: device tau, x is clamped to [-tau, tau] (null: no clamp)
  float* col_counts;     // with clamp: per-column count of |x| > tau, added to (null: not counted)
  const int32_t* zero_idx;  // row quantizer only: ascending columns set to 0 before quantizing
  int zero_n;
};

// Launchers (quant.cu).  All return cudaError_t of the launch.
// gen: 0 = amax_out is a float that is zeroed first; else the generation for a
// tagged 64-bit context slot (see fp4_ctx_scratch)
cudaError_t launch_amax(const void* x, int dt, int64_t rows, int64_t cols, int64_t ldx, int rht_axis,
                        uint32_t rht_signs, float* amax_out, uint32_t gen, int num_sms, cudaStream_t st);
cudaError_t launch_amax_dual(const void* x, int dt, int64_t rows, int64_t cols, int64_t ldx,
                             uint32_t signs_rows, uint32_t signs_cols, bool rht_rows, bool rht_cols,
                             float* amax_rows, float* amax_cols, uint32_t gen, int num_sms, cudaStream_t st);
cudaError_t launch_quant_rows(const void* x, int dt, int64_t rows, int64_t cols, int64_t ldx, int fmt,
                              const QuantOut& o, int num_sms, cudaStream_t st);
// the row quantizer with o.clamp set (32-bit block ids: rows * cols / block < 2^31)
cudaError_t launch_quant_rows_clamped(const void* x, int dt, int64_t rows, int64_t cols, int64_t ldx, int fmt,
                                      const QuantOut& o, int num_sms, cudaStream_t st);
cudaError_t launch_quant_tile(const void* x, int dt, int64_t rows, int64_t cols, int64_t ldx, int fmt,
                              bool two_d, bool transpose, const QuantOut& o, int num_sms, cudaStream_t st);
cudaError_t launch_quant_dual(const void* x, int dt, int64_t rows, int64_t cols, int64_t ldx, int fmt,
                              const QuantOut& orow, const QuantOut& ocol, bool two_d_rows, bool two_d_cols,
                              int num_sms, cudaStream_t st);
cudaError_t launch_dequant(const fp4_operand& q, int out_dt, void* out, int64_t ldo, int num_sms,
                           cudaStream_t st);
cudaError_t launch_rht16(const void* x, int dt, int64_t rows, int64_t cols, int64_t ldx, int axis,
                         uint32_t signs, float* y, int num_sms, cudaStream_t st);
cudaError_t launch_dge(const void* x, int xdt, int64_t ldx, const fp4_operand& q, const void* dy, int dydt,
                       int64_t lddy, float* dx, int64_t lddx, float k, float clamp, float outside,
                       int num_sms, cudaStream_t st);
// Q_soft forward (dy == NULL: out = s Q_soft(x/s)) or backward (out = dy Q_soft'(x/s))
cudaError_t launch_soft(const void* x, int xdt, int64_t ldx, const fp4_operand& q, const void* dy, int dydt,
                        int64_t lddy, float* out, int64_t ldo, float beta, int num_sms, cudaStream_t st);
// thresholds evaluated on each side of x/s for this beta (0: all of them)
int soft_window(float beta);
cudaError_t launch_encode_e2m1(const float* xs, uint8_t* codes, int64_t n, int method, cudaStream_t st);
cudaError_t launch_encode_e4m3(const float* t, uint8_t* out, int64_t n, cudaStream_t st);

// GEMM (gemm.cu).  Extra bf16 K columns (the hot-channel tail) are optional.
struct GemmArgs {
  const fp4_operand* A;
  const fp4_operand* B;
  const void* a_ext;       // [M][kx] bf16 (or E4M3 bytes with ext_fp8 / ext_mx8), or null
  const void* b_ext;       // [N][kx]
  int64_t kx;              // extra K (multiple of 64; of 128 with ext_fp8 / ext_mx8), 0 if none
  bool ext_fp8;            // extra columns are E4M3 (kind::f8f6f4), per-row scales in the epilogue
  bool ext_mx8;            // extra columns are MXFP8: E4M3 with E8M0 block scales (CTA-pair kernel,
  const uint8_t* a_ext_sf; //   kind::mxf8f6f4 into the FP4 accumulator); their scales, MMA layout
  const uint8_t* b_ext_sf;
  const float* row_scale;  // [M] and [N]: C (+)= row_scale[m] col_scale[n] acc (no alpha); null: alpha
  const float* col_scale;
  bool fp4_part;           // false: only the bf16 columns (two-kernel residual GEMM)
  int out_dtype;
  void* C;
  int64_t ldc;
  int accumulate;
  unsigned int* status;
  int num_sms;
  // quantize fused into the operand producer (CTA-pair kernel, MXFP4 RTN), when
  // quant_a: A is the bf16 activation x_bf16 [m][B.k] (pitch ldx, a multiple of
  // 8) and g.A is unused; its codes / MMA-layout scales are written to qa_* if
  // non-null
  bool quant_a;
  const void* x_bf16;
  int64_t ldx;
  int64_t m;
  uint8_t* qa_codes;
  uint8_t* qa_scales;
};
int launch_gemm(const GemmArgs& g, cudaStream_t st);  // returns fp4 status
// the CTA-pair kernel (gemm2.cu): plain FP4 GEMM or bf16 extra columns, no C +=;
// with g.x_bf16 the quantize-fused variant
int launch_gemm_pair(const GemmArgs& g, cudaStream_t st);

// Hot-channel compensation (hcp.cu)
cudaError_t launch_hcp_channel_errors(const uint16_t* x, int64_t ldx, const fp4_operand& q, float* err,
                                      int num_sms, cudaStream_t st);
cudaError_t launch_hcp_topk(const float* err, int64_t k, int k_hot, int32_t* hot_idx, cudaStream_t st);
// argument checks of fp4_hcp_select (api.cu), also used by fp4_hcp_select_noalloc
int validate_hcp_select(const void* x_bf16, int64_t ldx, const fp4_operand* xq, int32_t k_hot,
                        const int32_t* hot_idx);
// E4M3 extra columns [M][kx] / [N][kx] (kx a multiple of 128) with row scales sa / sb
// MXFP8 extra columns (E4M3 codes [rows][kxm], E8M0 scales in the MMA layout)
cudaError_t launch_hcp_gather_mx8(const uint16_t* x, int64_t ldx, const uint16_t* w, int64_t ldw,
                                  const fp4_operand& xq, const fp4_operand& wq, const int32_t* hot, int k_hot,
                                  int order, int64_t kxm, uint8_t* a8, uint8_t* sa, uint8_t* b8, uint8_t* sb,
                                  int num_sms, cudaStream_t st);
cudaError_t launch_hcp_gather_fp8(const uint16_t* x, int64_t ldx, const uint16_t* w, int64_t ldw,
                                  const fp4_operand& xq, const fp4_operand& wq, const int32_t* hot, int k_hot,
                                  int order, int64_t kx, uint8_t* a8, uint8_t* b8, float* sa, float* sb, int num_sms,
                                  cudaStream_t st);
cudaError_t launch_hcp_gather(const uint16_t* x, int64_t ldx, const uint16_t* w, int64_t ldw,
                              const fp4_operand& xq, const fp4_operand& wq, const int32_t* hot,
                              int k_hot, int order, int64_t kx, uint16_t* a_ext, uint16_t* b_ext,
                              int num_sms, cudaStream_t st);

// Outlier clamping and compensation (occ.cu).  Workspace layout of fp4_occ_gemm
// (byte offsets).
struct OccLayout {
  int64_t kx;    // extra bf16 K columns (k_dense rounded up to 64)
  int64_t ldt;   // pitch of W^T (N rounded up to 8)
  size_t counts, hot, flags, a_ext, b_ext, wt, row_start, row_len, cursor, entries, bytes;
};
size_t occ_threshold_ws_bytes(int dt);
cudaError_t launch_occ_threshold(const void* x, int dt, int64_t rows, int64_t cols, int64_t ldx, uint64_t rank,
                                 void* ws, float* tau, long long* n_out, int num_sms, cudaStream_t st);
OccLayout occ_layout(int64_t m, int64_t n, int64_t k, int k_dense, int64_t max_outliers);
// top-k columns, their extra GEMM columns, W^T and the per-row scattered outliers
cudaError_t launch_occ_prepare(const void* x, int xdt, int64_t ldx, const uint16_t* w, int64_t ldw,
                               const fp4_operand& xq, const fp4_operand& wq, const float* tau, const float* col_counts,
                               int k_dense, int64_t max_outliers, void* ws, const OccLayout& L, unsigned int* status,
                               int num_sms, cudaStream_t st);
// after the GEMM stored Y [m][n] (pitch ldy): the scattered outliers' product
cudaError_t launch_occ_correct(void* y, int64_t ldy, int out_dtype, int64_t m, int64_t n, const void* ws,
                               const OccLayout& L, int num_sms, cudaStream_t st);
// quality sums over q with any block (16-128); tau: OCC reconstruction; beta > 0:
// the sigmoid-smoothed reconstruction instead of the codes
// stats (may be null): cosine, MSE, SNR (dB) and relative L2 error from the sums
cudaError_t launch_error_stats(const void* x, int xdt, int64_t ldx, const fp4_operand& q, int block,
                               const float* tau, float beta, double* sums, double* stats, int num_sms,
                               cudaStream_t st);
// the row quantizer with the columns o.zero_idx[0..o.zero_n) set to 0 (32-bit block ids)
cudaError_t launch_quant_rows_zeroed(const void* x, int dt, int64_t rows, int64_t cols, int64_t ldx, int fmt,
                                     const QuantOut& o, int num_sms, cudaStream_t st);
// amax of x with the ascending columns hot[0..n) left out, into a tagged slot
cudaError_t launch_amax_zeroed(const void* x, int dt, int64_t rows, int64_t cols, int64_t ldx, const int32_t* hot,
                               int n, float* amax_out, uint32_t gen, int num_sms, cudaStream_t st);
// MXFP4 RTN quantization of bf16 in the row layout (orow), the transposed
// layout (ocol) or both (either may be null), 64 x 256 TMA tiles (quant_mx.cu)
bool mx_tiled_supported(int dt, int fmt, const QuantOut* orow, const QuantOut* ocol, int64_t rows, int64_t cols,
                        int64_t ldx);
cudaError_t launch_quant_mx_tiled(const void* x, int64_t rows, int64_t cols, int64_t ldx, const QuantOut* orow,
                                  const QuantOut* ocol, unsigned int* status, int num_sms, cudaStream_t st);
// row quantizer for any block of 16-128 elements (row-major scales, no transpose)
cudaError_t launch_quant_rows_blk(const void* x, int dt, int64_t rows, int64_t cols, int64_t ldx, int fmt, int block,
                                  const QuantOut& o, int num_sms, cudaStream_t st);

__host__ __device__ inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
// scales per row in the MMA layout: k padded to 256 elements
__host__ __device__ inline int64_t nsf_padded(int64_t k, int fmt) {
  return cdiv(k, 256) * (256 / (fmt == FP4_FMT_MXFP4 ? 32 : 16));
}

}  // namespace fp4
