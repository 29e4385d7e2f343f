// Quantization-side kernels: per-tensor amax, block-scaled FP4 quantize in the
// row and transposed layouts (1D and 16x16 2D scaling, optional RHT16, RTN or
// Philox SR), dequantize, the standalone RHT16, the DGE backward and the
// element encoders.  All are HBM-bound streaming kernels.
//
// Q(x) = s * round(x / s)  ([grad] §2.1); E2M1 elements ([outlier] §1.1, [msr] §一);
// E8M0 / E4M3 block scales, NVFP4 per-tensor scale ([lowprec] §1.1);
// RTN forward, SR + 16x16 2D + RHT backward ([outlier] §4.1-4.2);
// SR as floor + (rand < frac) ([lowprec] §3.2); DGE derivative clamped at 3.0
// ([msr] §二).
#include <cuda_bf16.h>

#include <algorithm>

#include "fp4_device.cuh"

using namespace fp4dev;

namespace fp4 {
namespace {

constexpr int kThreads = 256;

inline int grid_for(int64_t work_items, int per_block, int num_sms, int blocks_per_sm = 8) {
  int64_t need = cdiv(work_items, per_block);
  int64_t cap = (int64_t)num_sms * blocks_per_sm;
  return (int)(need < 1 ? 1 : (need < cap ? need : cap));
}

// ----------------------------------------------------------------------------
// Encode the B values of one block (already RHT'ed if requested) and store
// codes + scale.  `first_elem` is the linear output index of v[0] (SR counter).
// ----------------------------------------------------------------------------
template <int FMT, int B>
__device__ __forceinline__ uint32_t encode_block_codes(const float* v, float g, const QuantOut& o,
                                                       int64_t out_row, int64_t out_col0, float amax_b,
                                                       bool sr) {
  uint32_t byte;
  float r;
  bool zero;
  block_scale<FMT>(amax_b, g, byte, r, zero);
  uint32_t packed[B / 8];
  if (!sr) {
#pragma unroll
    for (int q = 0; q < B / 8; ++q) {
      uint32_t w = 0;
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        float a = __fmul_rn(v[8 * q + 2 * p], r), b = __fmul_rn(v[8 * q + 2 * p + 1], r);
        w |= e2m1x2_hw(a, b) << (8 * p);
      }
      packed[q] = zero ? 0u : w;
    }
  } else {
    int64_t first_elem = out_row * o.out_cols + out_col0;
#pragma unroll
    for (int q = 0; q < B / 8; ++q) {
      uint4 bits = sr_bits8(o.keys, o.sr_offset, o.sr_stream, (uint64_t)(first_elem + 8 * q));
      uint32_t w = 0;
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const float y0 = e2m1_sr_value(__fmul_rn(v[8 * q + 2 * p], r), u16_lane_shl6(bits, 2 * p));
        const float y1 = e2m1_sr_value(__fmul_rn(v[8 * q + 2 * p + 1], r), u16_lane_shl6(bits, 2 * p + 1));
        w |= e2m1x2_hw(y0, y1) << (8 * p);
      }
      packed[q] = zero ? 0u : w;
    }
  }
  uint8_t* dst = o.codes + out_row * (o.out_cols >> 1) + (out_col0 >> 1);
  if constexpr (B == 16) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(packed[0], packed[1]);
  } else {
    *reinterpret_cast<uint4*>(dst) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  }
  return byte;
}

template <int FMT, int B>
__device__ __forceinline__ void encode_store_block(const float* v, float g, const QuantOut& o,
                                                   int64_t out_row, int64_t out_col0, float amax_b,
                                                   bool sr) {
  const uint32_t byte = encode_block_codes<FMT, B>(v, g, o, out_row, out_col0, amax_b, sr);
  o.scales[sf_offset(o.sf_layout, out_row, out_col0 / B, o.nsf_row, o.nsf_pad)] = (uint8_t)byte;
}


__device__ __forceinline__ float load_g(const QuantOut& o, int fmt) {
  if (fmt != FP4_FMT_NVFP4) return 0.0f;
  float g = nvfp4_tensor_scale(*o.amax);
  if (blockIdx.x == 0 && threadIdx.x == 0 && o.tensor_scale) *o.tensor_scale = g;
  return g;
}

// ----------------------------------------------------------------------------
// Row quantizer for any block of SB = 16 * G elements (16-128; [grad] §4.2),
// either scale format, row-major scales: one thread per 16 elements, the G
// threads of a block share its amax through shuffles, the first stores the
// scale byte.  The warp-uniform loop keeps every lane in the shuffles.
// ----------------------------------------------------------------------------
template <int FMT, int DT, int G>
__global__ void __launch_bounds__(kThreads) quant_rows_blk_kernel(const void* __restrict__ x, int64_t rows,
                                                                  int64_t cols, int64_t ldx, QuantOut o) {
  const float g = load_g(o, FMT);
  const bool sr = o.rounding == FP4_ROUND_SR;
  const int lane = threadIdx.x & 31;
  const int64_t units_row = cols / 16, total = rows * units_row;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t base = blockIdx.x * (int64_t)blockDim.x + (threadIdx.x & ~31); base < total; base += stride) {
    const int64_t u = base + lane;
    const bool act = u < total;
    const int64_t r = act ? u / units_row : 0, c0 = act ? (u - r * units_row) * 16 : 0;
    float v[16];
    if (act) {
      load8<DT>(x, r * ldx + c0, v);
      load8<DT>(x, r * ldx + c0 + 8, v + 8);
      if (o.rht) rht16(v, o.rht_signs);
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = 0.0f;
    }
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(v[j]));
#pragma unroll
    for (int m = 1; m < G; m <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, m));
    if (act) {
      const uint32_t byte = encode_block_codes<FMT, 16>(v, g, o, r, c0, amax, sr);
      if ((lane & (G - 1)) == 0) o.scales[r * (cols / (16 * G)) + c0 / (16 * G)] = (uint8_t)byte;
    }
  }
}

// ----------------------------------------------------------------------------
// amax over a row-blocked tensor (plain or RHT16 along cols); cols % 16 == 0,
// rows 16-byte aligned.  One thread per 16-element chunk.
// ----------------------------------------------------------------------------
template <int DT, bool RHT>
__global__ void __launch_bounds__(kThreads) amax_rows_kernel(const void* __restrict__ x, int64_t rows,
                                                             int64_t cols, int64_t ldx, uint32_t signs,
                                                             float* amax_out, uint32_t gen) {
  int64_t nchunk_row = cols >> 4;
  int64_t total = rows * nchunk_row;
  float m = 0.0f;
  for (int64_t c = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; c < total;
       c += (int64_t)gridDim.x * blockDim.x) {
    int64_t r = c / nchunk_row, k0 = (c - r * nchunk_row) << 4;
    float v[16];
    load8<DT>(x, r * ldx + k0, v);
    load8<DT>(x, r * ldx + k0 + 8, v + 8);
    if (RHT) rht16(v, signs);
#pragma unroll
    for (int j = 0; j < 16; ++j) m = fmaxf(m, fabsf(v[j]));
  }
  block_amax_atomic(m, amax_out, gen);
}

// Same reduction with 32-bit chunk ids (fewer than 2^31 chunks): a chunk's
// address is 16 c when rows are contiguous, else (c / nch) ldx + 16 (c % nch)
// with a precomputed divider; two chunks per iteration keep 64 bytes of bf16
// in flight per thread.
// Bit j set iff column k0 + j (j < 16) is in the ascending list hot[0..n):
// binary search for the first entry >= k0, then the few entries below k0 + 16.
__device__ __forceinline__ uint32_t hot_mask16(const int32_t* __restrict__ hot, int n, uint32_t k0) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if ((uint32_t)hot[mid] < k0) lo = mid + 1;
    else hi = mid;
  }
  uint32_t m = 0;
  for (int i = lo; i < n && (uint32_t)hot[i] < k0 + 16u; ++i) m |= 1u << ((uint32_t)hot[i] - k0);
  return m;
}

template <int DT, bool RHT>
__global__ void __launch_bounds__(kThreads) amax_rows32_kernel(const void* __restrict__ x, int64_t ldx, FastDiv nch,
                                                               uint32_t total, int contiguous, uint32_t signs,
                                                               float* amax_out, uint32_t gen) {
  float m = 0.0f;
  const uint32_t stride = gridDim.x * blockDim.x;
  auto addr = [&](uint32_t c) -> int64_t {
    if (contiguous) return (int64_t)c << 4;
    const uint32_t r = fast_div(c, nch);
    return (int64_t)r * ldx + ((int64_t)(c - r * nch.d) << 4);
  };
  for (uint32_t c = blockIdx.x * blockDim.x + threadIdx.x; c < total; c += 2 * stride) {
    const uint32_t c2 = c + stride;
    const bool two = c2 < total && c2 > c;
    float v[16], w[16];
    const int64_t e = addr(c);
    load8<DT, true>(x, e, v);
    load8<DT, true>(x, e + 8, v + 8);
    if (two) {
      const int64_t e2 = addr(c2);
      load8<DT, true>(x, e2, w);
      load8<DT, true>(x, e2 + 8, w + 8);
    }
    if (RHT) rht16(v, signs);
#pragma unroll
    for (int j = 0; j < 16; ++j) m = fmaxf(m, fabsf(v[j]));
    if (two) {
      if (RHT) rht16(w, signs);
#pragma unroll
      for (int j = 0; j < 16; ++j) m = fmaxf(m, fabsf(w[j]));
    }
  }
  block_amax_atomic(m, amax_out, gen);
}

// Column bitmask of the list hot[0..n) in shared memory (rows up to
// kZeroSmemCols columns), built by the CTA before use; longer rows search the
// list per 16 columns instead.
constexpr int kZeroSmemCols = 65536;
__device__ __forceinline__ void build_hot_bits(uint32_t* bits, int64_t cols, const int32_t* hot, int n) {
  const int words = (int)((cols + 31) >> 5);
  for (int i = threadIdx.x; i < words; i += blockDim.x) bits[i] = 0u;
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const uint32_t c = (uint32_t)hot[i];
    if (c < (uint32_t)cols) atomicOr(&bits[c >> 5], 1u << (c & 31));
  }
  __syncthreads();
}
__device__ __forceinline__ uint32_t hot_bits16(const uint32_t* bits, const int32_t* hot, int n, uint32_t k0) {
  return bits ? (bits[k0 >> 5] >> (k0 & 31)) & 0xFFFFu : hot_mask16(hot, n, k0);
}

// amax of x with the ascending columns hot[0..n) left out (16 elements per step)
template <int DT>
__global__ void __launch_bounds__(kThreads) amax_zeroed_kernel(const void* __restrict__ x, int64_t ldx, FastDiv nch,
                                                               uint32_t total, const int32_t* __restrict__ hot, int n,
                                                               float* amax_out, uint32_t gen) {
  extern __shared__ uint32_t zbits_smem[];
  const uint32_t* bits = nullptr;
  if ((int64_t)nch.d * 16 <= kZeroSmemCols) {   // uniform over the grid
    build_hot_bits(zbits_smem, (int64_t)nch.d * 16, hot, n);
    bits = zbits_smem;
  }
  float m = 0.0f;
  for (uint32_t c = blockIdx.x * blockDim.x + threadIdx.x; c < total; c += gridDim.x * blockDim.x) {
    const uint32_t r = fast_div(c, nch), k0 = (c - r * nch.d) << 4;
    float v[16];
    load8<DT, true>(x, (int64_t)r * ldx + k0, v);
    load8<DT, true>(x, (int64_t)r * ldx + k0 + 8, v + 8);
    const uint32_t hm = hot_bits16(bits, hot, n, k0);
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (!((hm >> j) & 1u)) m = fmaxf(m, fabsf(v[j]));
  }
  block_amax_atomic(m, amax_out, gen);
}

// ----------------------------------------------------------------------------
// Row quantizer: blocks along cols, output [rows][cols/2].  One thread per block.
// ----------------------------------------------------------------------------
template <int FMT, int DT>
__global__ void __launch_bounds__(kThreads) quant_rows_kernel(const void* __restrict__ x, int64_t rows,
                                                              int64_t cols, int64_t ldx, QuantOut o) {
  constexpr int B = FMT == FP4_FMT_MXFP4 ? 32 : 16;
  const float g = load_g(o, FMT);
  const bool sr = o.rounding == FP4_ROUND_SR;
  const bool rht = o.rht != 0;
  const int64_t nblk_row = cols / B;
  const int64_t total = rows * nblk_row;
  const bool small = total < (int64_t(1) << 31);  // 32-bit index math
  auto split = [&](int64_t blk, int64_t& r, int64_t& k0) {
    if (small) {
      const uint32_t b32 = (uint32_t)blk, n32 = (uint32_t)nblk_row, r32 = b32 / n32;
      r = r32;
      k0 = (int64_t)(b32 - r32 * n32) * B;
    } else {
      r = blk / nblk_row;
      k0 = (blk - r * nblk_row) * B;
    }
  };
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  // two blocks per iteration: both blocks' loads are in flight together
  for (int64_t blk = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; blk < total; blk += 2 * stride) {
    const int64_t blk2 = blk + stride;
    const bool two = blk2 < total;
    int64_t r, k0, r2 = 0, k2 = 0;
    split(blk, r, k0);
    if (two) split(blk2, r2, k2);
    float v[B], w[B];
#pragma unroll
    for (int q = 0; q < B / 8; ++q) load8<DT>(x, r * ldx + k0 + 8 * q, v + 8 * q);
    if (two) {
#pragma unroll
      for (int q = 0; q < B / 8; ++q) load8<DT>(x, r2 * ldx + k2 + 8 * q, w + 8 * q);
    }
    if (rht) {
#pragma unroll
      for (int h = 0; h < B / 16; ++h) rht16(v + 16 * h, o.rht_signs);
    }
    float amax_b = 0.0f;
#pragma unroll
    for (int j = 0; j < B; ++j) amax_b = fmaxf(amax_b, fabsf(v[j]));
    encode_store_block<FMT, B>(v, g, o, r, k0, amax_b, sr);
    if (two) {
      if (rht) {
#pragma unroll
        for (int h = 0; h < B / 16; ++h) rht16(w + 16 * h, o.rht_signs);
      }
      float amax2 = 0.0f;
#pragma unroll
      for (int j = 0; j < B; ++j) amax2 = fmaxf(amax2, fabsf(w[j]));
      encode_store_block<FMT, B>(w, g, o, r2, k2, amax2, sr);
    }
  }
}

// Row quantizer with 32-bit block ids (fewer than 2^31 blocks): one thread per
// block, two blocks per iteration with all four loads in flight; the block's
// row and position come from a precomputed divider, and its input starts at
// B * blk when rows are contiguous.  Loads allocate in L1 so that a thread's
// second 16 bytes of each 32-byte sector do not fetch the sector again.
// PLAIN: RTN without RHT (the forward path), compiled without the SR and RHT
// code so that its register count, and so its occupancy, is not set by them.
// CLAMP: x is first clamped to [-tau, tau], tau = *o.clamp (outlier clamping,
// [msr] §三), and the elements with |x| > tau are counted per column: in
// shared memory (counts_s, merged once per CTA) when the row fits, else by
// global atomics
constexpr int kClampSmemCols = 8192;
template <bool CLAMP, int B>
__device__ __forceinline__ void clamp_block(float* v, float tau, float* col_counts, uint32_t* counts_s, uint32_t k0) {
  if constexpr (CLAMP) {
#pragma unroll
    for (int j = 0; j < B; ++j) {
      if (fabsf(v[j]) > tau) {
        if (counts_s) atomicAdd(counts_s + k0 + j, 1u);
        else if (col_counts) atomicAdd(col_counts + k0 + j, 1.0f);
        v[j] = copysignf(tau, v[j]);
      }
    }
  }
}

// ZERO: the columns o.zero_idx[0..o.zero_n) are set to 0 before quantizing
// (hot channels routed around the FP4 operand)
template <bool ZERO, int B>
__device__ __forceinline__ void zero_block(float* v, const QuantOut& o, const uint32_t* bits, uint32_t k0) {
  if constexpr (ZERO) {
#pragma unroll
    for (int h = 0; h < B / 16; ++h) {
      const uint32_t m = hot_bits16(bits, o.zero_idx, o.zero_n, k0 + 16 * h);
      if (m) {
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if ((m >> j) & 1u) v[16 * h + j] = 0.0f;
      }
    }
  }
}

template <int FMT, int DT, bool PLAIN, bool CLAMP = false, bool ZERO = false>
__global__ void __launch_bounds__(kThreads) quant_rows32_kernel(const void* __restrict__ x, int64_t ldx, FastDiv nblk,
                                                                uint32_t total, int contiguous, QuantOut o) {
  constexpr int B = FMT == FP4_FMT_MXFP4 ? 32 : 16;
  const float g = load_g(o, FMT);
  const float tau = CLAMP ? *o.clamp : 0.0f;
  extern __shared__ uint32_t counts_smem[];
  uint32_t* counts_s = nullptr;
  uint32_t* zero_bits = nullptr;
  if constexpr (ZERO) {
    if (o.out_cols <= kZeroSmemCols) {   // uniform over the grid
      zero_bits = counts_smem;
      build_hot_bits(zero_bits, o.out_cols, o.zero_idx, o.zero_n);
    }
  }
  if constexpr (CLAMP) {
    if (o.col_counts && o.out_cols <= kClampSmemCols) {   // uniform over the grid
      counts_s = counts_smem;
      for (int b = threadIdx.x; b < (int)o.out_cols; b += blockDim.x) counts_s[b] = 0u;
      __syncthreads();
    }
  }
  const bool sr = !PLAIN && o.rounding == FP4_ROUND_SR;
  const bool rht = !PLAIN && o.rht != 0;
  const uint32_t stride = gridDim.x * blockDim.x;
  for (uint32_t blk = blockIdx.x * blockDim.x + threadIdx.x; blk < total; blk += 2 * stride) {
    const uint32_t blk2 = blk + stride;
    const bool two = blk2 < total && blk2 > blk;
    const uint32_t r = fast_div(blk, nblk), k0 = (blk - r * nblk.d) * B;
    uint32_t r2 = 0, k2 = 0;
    if (two) {
      r2 = fast_div(blk2, nblk);
      k2 = (blk2 - r2 * nblk.d) * B;
    }
    const int64_t e = contiguous ? (int64_t)blk * B : (int64_t)r * ldx + k0;
    const int64_t e2 = contiguous ? (int64_t)blk2 * B : (int64_t)r2 * ldx + k2;
    float v[B], w[B];
#pragma unroll
    for (int q = 0; q < B / 8; ++q) load8<DT, true>(x, e + 8 * q, v + 8 * q);
    if (two) {
#pragma unroll
      for (int q = 0; q < B / 8; ++q) load8<DT, true>(x, e2 + 8 * q, w + 8 * q);
    }
    clamp_block<CLAMP, B>(v, tau, o.col_counts, counts_s, k0);
    if (two) clamp_block<CLAMP, B>(w, tau, o.col_counts, counts_s, k2);
    zero_block<ZERO, B>(v, o, zero_bits, k0);
    if (two) zero_block<ZERO, B>(w, o, zero_bits, k2);
    if (rht) {
#pragma unroll
      for (int h = 0; h < B / 16; ++h) rht16(v + 16 * h, o.rht_signs);
    }
    float amax_b = 0.0f;
#pragma unroll
    for (int j = 0; j < B; ++j) amax_b = fmaxf(amax_b, fabsf(v[j]));
    encode_store_block<FMT, B>(v, g, o, r, k0, amax_b, sr);
    if (two) {
      if (rht) {
#pragma unroll
        for (int h = 0; h < B / 16; ++h) rht16(w + 16 * h, o.rht_signs);
      }
      float amax2 = 0.0f;
#pragma unroll
      for (int j = 0; j < B; ++j) amax2 = fmaxf(amax2, fabsf(w[j]));
      encode_store_block<FMT, B>(w, g, o, r2, k2, amax2, sr);
    }
  }
  if constexpr (CLAMP) {
    if (counts_s) {
      __syncthreads();
      for (int b = threadIdx.x; b < (int)o.out_cols; b += blockDim.x)
        if (counts_s[b]) atomicAdd(o.col_counts + b, (float)counts_s[b]);
    }
  }
}

// ----------------------------------------------------------------------------
// Tiled kernels: a TR x 64 tile of the input is staged in shared memory (fp32)
// so that both the row-blocked and the column-blocked (transposed) outputs are
// read and written coalesced.  TR = 4 blocks (64 rows for NVFP4, 128 for MXFP4).
// ----------------------------------------------------------------------------
enum TileMode { T_AMAX_COLS = 0, T_AMAX_DUAL = 1, T_Q_COLS = 2, T_Q_DUAL = 3, T_Q_ROWS2D = 4 };

constexpr int TC = 64;
constexpr int TSTRIDE = TC + 1;

template <int DT, int TR>
__device__ __forceinline__ void load_tile(const void* __restrict__ x, int64_t rows, int64_t cols,
                                          int64_t ldx, int64_t r0, int64_t c0, float* tile) {
  const bool full = (r0 + TR <= rows) && (c0 + TC <= cols);
  constexpr int CH = TR * TC / 8;  // 8-element chunks
  for (int q = threadIdx.x; q < CH; q += blockDim.x) {
    int rr = q / (TC / 8), cc = (q % (TC / 8)) * 8;
    float v[8];
    if (full) {
      load8<DT>(x, (r0 + rr) * ldx + c0 + cc, v);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        int64_t R = r0 + rr, C = c0 + cc + i;
        v[i] = (R < rows && C < cols) ? load1<DT>(x, R * ldx + C) : 0.0f;
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) tile[rr * TSTRIDE + cc + i] = v[i];
  }
}

// Register copy of one full tile's raw input (no bounds checks): each thread
// holds CPT 8-element chunks, fetched while the previous tile is processed.
template <int DT, int TR>
struct TileRegs {
  static constexpr int CPT = TR * TC / 8 / kThreads;   // chunks per thread
  static constexpr int W = DT == FP4_DTYPE_BF16 ? 1 : 2;
  uint4 r[CPT * W];
};

template <int DT, int TR>
__device__ __forceinline__ void tile_fetch(const void* __restrict__ x, int64_t ldx, int64_t r0, int64_t c0,
                                           TileRegs<DT, TR>& t) {
  constexpr int ES = DT == FP4_DTYPE_BF16 ? 2 : 4;
#pragma unroll
  for (int i = 0; i < TileRegs<DT, TR>::CPT; ++i) {
    const int q = threadIdx.x + i * kThreads;
    const int rr = q / (TC / 8), cc = (q % (TC / 8)) * 8;
    const char* src = static_cast<const char*>(x) + ((r0 + rr) * ldx + c0 + cc) * ES;
    t.r[i * TileRegs<DT, TR>::W] = ld_nc_v4(src);
    if (TileRegs<DT, TR>::W == 2) t.r[i * TileRegs<DT, TR>::W + 1] = ld_nc_v4(src + 16);
  }
}

template <int DT, int TR>
__device__ __forceinline__ void tile_store(const TileRegs<DT, TR>& t, float* tile) {
#pragma unroll
  for (int i = 0; i < TileRegs<DT, TR>::CPT; ++i) {
    const int q = threadIdx.x + i * kThreads;
    const int rr = q / (TC / 8), cc = (q % (TC / 8)) * 8;
    float v[8];
    if (DT == FP4_DTYPE_BF16) {
      const uint4 w = t.r[i];
      const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[2 * j] = __uint_as_float(u[j] << 16);
        v[2 * j + 1] = __uint_as_float(u[j] & 0xFFFF0000u);
      }
    } else {
      const uint4 a = t.r[i * 2], b = t.r[i * 2 + 1];
      v[0] = __uint_as_float(a.x); v[1] = __uint_as_float(a.y); v[2] = __uint_as_float(a.z); v[3] = __uint_as_float(a.w);
      v[4] = __uint_as_float(b.x); v[5] = __uint_as_float(b.y); v[6] = __uint_as_float(b.z); v[7] = __uint_as_float(b.w);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) tile[rr * TSTRIDE + cc + j] = v[j];
  }
}

template <int FMT, int DT, int MODE>
__global__ void __launch_bounds__(kThreads) tile_kernel(const void* __restrict__ x, int64_t rows,
                                                        int64_t cols, int64_t ldx, QuantOut oc,
                                                        QuantOut orr, int two_d, uint32_t signs_c,
                                                        uint32_t signs_r, int rht_c, int rht_r,
                                                        float* amax_c, float* amax_r, uint32_t gen = 0) {
  constexpr int B = FMT == FP4_FMT_MXFP4 ? 32 : 16;
  constexpr int TR = 4 * B;
  __shared__ float tile[TR * TSTRIDE];
  constexpr bool QUANT = MODE >= T_Q_COLS;
  constexpr bool DO_COLS = MODE == T_AMAX_COLS || MODE == T_AMAX_DUAL || MODE == T_Q_COLS || MODE == T_Q_DUAL;
  constexpr bool DO_ROWS = MODE == T_AMAX_DUAL || MODE == T_Q_DUAL || MODE == T_Q_ROWS2D;
  float g_c = 0.0f, g_r = 0.0f;
  if constexpr (QUANT) {
    if (DO_COLS) g_c = load_g(oc, FMT);
    if (DO_ROWS) g_r = load_g(orr, FMT);
  }
  float m_c = 0.0f, m_r = 0.0f;
  // tile ids in 32 bits (the launcher guarantees fewer than 2^31 tiles): a
  // 64-bit division per tile costs more than the tile's element work
  const uint32_t ntc = (uint32_t)cdiv(cols, TC), ntiles = (uint32_t)(cdiv(rows, TR) * ntc);
  const int t = threadIdx.x;
  // full tiles are fetched into registers one iteration ahead; ragged edge
  // tiles are loaded element by element when their turn comes
  TileRegs<DT, TR> pre;
  auto is_full = [&](uint32_t tr, uint32_t tc) {
    return (int64_t)(tr + 1) * TR <= rows && (int64_t)(tc + 1) * TC <= cols;
  };
  uint32_t tr_n = blockIdx.x / ntc, tc_n = blockIdx.x - tr_n * ntc;   // next tile's coordinates
  bool pre_full = false;
  if (blockIdx.x < ntiles && is_full(tr_n, tc_n)) {
    tile_fetch<DT, TR>(x, ldx, (int64_t)tr_n * TR, (int64_t)tc_n * TC, pre);
    pre_full = true;
  }
  for (uint32_t tid = blockIdx.x; tid < ntiles; tid += gridDim.x) {
    const int64_t r0 = (int64_t)tr_n * TR, c0 = (int64_t)tc_n * TC;
    if (pre_full)
      tile_store<DT, TR>(pre, tile);
    else
      load_tile<DT, TR>(x, rows, cols, ldx, r0, c0, tile);
    __syncthreads();
    const uint32_t nxt = tid + gridDim.x;
    tr_n = nxt / ntc;
    tc_n = nxt - tr_n * ntc;
    pre_full = nxt < ntiles && is_full(tr_n, tc_n);
    if (pre_full) tile_fetch<DT, TR>(x, ldx, (int64_t)tr_n * TR, (int64_t)tc_n * TC, pre);
    if constexpr (DO_COLS) {
      // column item: column c of the tile, row-block rb (B rows); lanes = columns
      int c = t % TC, rb = t / TC;
      float v[B];
#pragma unroll
      for (int j = 0; j < B; ++j) v[j] = tile[(rb * B + j) * TSTRIDE + c];
      if (rht_c) {
#pragma unroll
        for (int h = 0; h < B / 16; ++h) rht16(v + 16 * h, signs_c);
      }
      float a = 0.0f;
#pragma unroll
      for (int j = 0; j < B; ++j) a = fmaxf(a, fabsf(v[j]));
      bool valid = (c0 + c < cols) && (r0 + rb * B < rows);
      if constexpr (!QUANT) {
        if (valid) m_c = fmaxf(m_c, a);
      } else {
        if (two_d & 1) {  // 16x16 tile: the 16 lanes of consecutive columns share one scale
#pragma unroll
          for (int o = 8; o; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
        }
        if (valid) encode_store_block<FMT, B>(v, g_c, oc, c0 + c, r0 + rb * B, a, oc.rounding == FP4_ROUND_SR);
      }
    }
    if constexpr (DO_ROWS) {
      // row item: row r of the tile, col-block cb; lanes = consecutive rows
      int r = t % TR, cb = t / TR;
      if (cb < TC / B) {
        float v[B];
#pragma unroll
        for (int j = 0; j < B; ++j) v[j] = tile[r * TSTRIDE + cb * B + j];
        if (rht_r) {
#pragma unroll
          for (int h = 0; h < B / 16; ++h) rht16(v + 16 * h, signs_r);
        }
        float a = 0.0f;
#pragma unroll
        for (int j = 0; j < B; ++j) a = fmaxf(a, fabsf(v[j]));
        bool valid = (r0 + r < rows) && (c0 + cb * B < cols);
        if constexpr (!QUANT) {
          if (valid) m_r = fmaxf(m_r, a);
        } else {
          if (MODE == T_Q_ROWS2D || (two_d & 2)) {  // 16x16 tile: 16 lanes of consecutive rows
#pragma unroll
            for (int o = 8; o; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
          }
          if (valid) encode_store_block<FMT, B>(v, g_r, orr, r0 + r, c0 + cb * B, a, orr.rounding == FP4_ROUND_SR);
        }
      }
    }
    __syncthreads();
  }
  if constexpr (!QUANT) {
    if (DO_COLS) block_amax_atomic(m_c, amax_c, gen);
    if (DO_ROWS) {
      __syncthreads();
      block_amax_atomic(m_r, amax_r, gen);
    }
  }
}

// ----------------------------------------------------------------------------
// NVFP4 with bf16 input (the training path): 64 x 128 tiles.
//   row layout   each thread's four 16-byte loads are 32 consecutive elements
//                of one row, i.e. two blocks: quantized straight from registers
//   transposed   the raw bf16 tile is staged in shared memory; each thread
//                reads one 32-bit word (two adjacent columns) from 16 rows and
//                quantizes both columns' blocks
// Shared memory: 68 words per tile row, word w stored at w ^ ((w & 32) >> 2):
// the 16-byte staging stores of a quarter warp (two rows x four threads) and
// the column reads of a warp (32 consecutive words of one row) each hit all
// 32 banks once.
// RHT without the per-element 1/4: the butterfly outputs w of bf16 inputs are
// multiples of 2^-133, so w/4 is exact in fp32 and max|w/4| = max|w|/4; the
// quantizer multiplies by r/4 instead of forming w/4 and then w/4 * r, which
// is the same product as long as r/4 is exact (r >= 2^-124, else the two
// multiplications are done as written).
// ----------------------------------------------------------------------------
constexpr int NV_TR = 64, NV_TC = 128, NV_SW = 68;

// the 16 RHT signs as +-1.0f multipliers (kernel parameters), in the packed
// pairs rht16_x2 takes: s2[k] = (sigma_k, sigma_{k+8}), sigma_k in the low word
struct RhtSigns {
  uint64_t s2[8];
};
inline RhtSigns rht_sign_floats(uint32_t bits) {
  RhtSigns r;
  const uint64_t one = 0x3F800000u, neg_one = 0xBF800000u;
  for (int k = 0; k < 8; ++k)
    r.s2[k] = ((bits >> k) & 1u ? neg_one : one) | (((bits >> (k + 8)) & 1u ? neg_one : one) << 32);
  return r;
}

__device__ __forceinline__ int nv_swz(int w) { return w ^ ((w & 32) >> 2); }

// one NVFP4 block: w = the values (quarter: w = 4x the true values), amax_b =
// the true block amax; codes and scale stored like encode_store_block
__device__ __forceinline__ void encode_nv_block(const float* w, bool quarter, float g, const QuantOut& o,
                                                int64_t out_row, int64_t out_col0, float amax_b, bool sr) {
  uint32_t byte;
  float r;
  bool zero;
  block_scale<FP4_FMT_NVFP4>(amax_b, g, byte, r, zero);
  float xs[16];
  if (quarter && !(r >= 0x1p-124f) && !zero) {
#pragma unroll
    for (int j = 0; j < 16; ++j) xs[j] = __fmul_rn(__fmul_rn(w[j], 0.25f), r);
  } else {
    const float m = quarter ? __fmul_rn(r, 0.25f) : r;
    const uint64_t m2 = f2_pack(m, m);
#pragma unroll
    for (int k = 0; k < 8; ++k) f2_unpack(f2_mul(f2_pack(w[k], w[k + 8]), m2), xs[k], xs[k + 8]);
  }
  uint32_t packed[2];
  if (!sr) {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      uint32_t v = 0;
#pragma unroll
      for (int p = 0; p < 4; ++p) v |= e2m1x2_hw(xs[8 * q + 2 * p], xs[8 * q + 2 * p + 1]) << (8 * p);
      packed[q] = zero ? 0u : v;
    }
  } else {
    const int64_t first_elem = out_row * o.out_cols + out_col0;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const uint4 bits = sr_bits8(o.keys, o.sr_offset, o.sr_stream, (uint64_t)(first_elem + 8 * q));
      uint32_t v = 0;
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const float y0 = e2m1_sr_value_finite(xs[8 * q + 2 * p], u16_lane_shl6_mul(bits, 2 * p));
        const float y1 = e2m1_sr_value_finite(xs[8 * q + 2 * p + 1], u16_lane_shl6_mul(bits, 2 * p + 1));
        v |= e2m1x2_hw(y0, y1) << (8 * p);
      }
      packed[q] = zero ? 0u : v;
    }
  }
  *reinterpret_cast<uint2*>(o.codes + out_row * (o.out_cols >> 1) + (out_col0 >> 1)) = make_uint2(packed[0], packed[1]);
  o.scales[sf_offset(o.sf_layout, out_row, out_col0 / 16, o.nsf_row, o.nsf_pad)] = (uint8_t)byte;
}

// 16-byte global -> shared copy (cp.async, L2 only); bytes past `src_bytes`
// (0..16) are zero-filled and not read
__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// TWO_D: 16x16 blocks in the transposed layout (a template parameter so that
// the 1D kernels are not compiled with its register demand)
template <int MODE, bool TWO_D>
__global__ void __launch_bounds__(kThreads, 4) tile_nv_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t cols,
                                                           int64_t ldx, FastDiv ntc, uint32_t ntiles, QuantOut oc,
                                                           QuantOut orr, RhtSigns sig_c, RhtSigns sig_r, int rht_c,
                                                           int rht_r, float* amax_c, float* amax_r,
                                                           uint32_t gen = 0) {
  constexpr bool QUANT = MODE >= T_Q_COLS;
  constexpr bool DO_ROWS = MODE == T_AMAX_DUAL || MODE == T_Q_DUAL;
  __shared__ __align__(16) uint32_t tile[2][NV_TR * NV_SW];   // double-buffered: the next tile streams in
  float g_c = 0.0f, g_r = 0.0f;
  if constexpr (QUANT) {
    g_c = load_g(oc, FP4_FMT_NVFP4);
    if (DO_ROWS) g_r = load_g(orr, FP4_FMT_NVFP4);
  }
  const bool sr_c = QUANT && oc.rounding == FP4_ROUND_SR;
  const bool sr_r = QUANT && DO_ROWS && orr.rounding == FP4_ROUND_SR;
  float m_c = 0.0f, m_r = 0.0f;  // amax of the values as computed (4x the true values with RHT)
  const int t = threadIdx.x;
  const int rr = t >> 2, q = t & 3;      // row role: row rr, columns 32q .. 32q+31
  const int pw = t & 63, rb = t >> 6;    // column role: columns 2pw, 2pw+1 of rows 16rb .. 16rb+15

  // this thread's 4 x 16 bytes of tile `id`: row r0 + rr, columns c0 + 32q .. +31
  auto fetch = [&](uint32_t id, uint32_t* buf) {
    const uint32_t tr = fast_div(id, ntc), tc = id - tr * ntc.d;
    const int64_t r = (int64_t)tr * NV_TR + rr, c = (int64_t)tc * NV_TC + 32 * q;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t cc = c + 8 * i;
      const int64_t avail = r < rows ? cols - cc : 0;
      const uint32_t nb = avail <= 0 ? 0u : avail >= 8 ? 16u : (uint32_t)(2 * avail);
      cp_async16(&buf[rr * NV_SW + nv_swz(16 * q + 4 * i)], nb ? x + r * ldx + cc : x, nb);
    }
    cp_async_commit();
  };

  if (blockIdx.x < ntiles) fetch(blockIdx.x, tile[0]);
  int b = 0;
  for (uint32_t id = blockIdx.x; id < ntiles; id += gridDim.x, b ^= 1) {
    const uint32_t tr = fast_div(id, ntc), tc = id - tr * ntc.d;
    const int64_t r0 = (int64_t)tr * NV_TR, c0 = (int64_t)tc * NV_TC;
    const uint32_t nid = id + gridDim.x;
    if (nid < ntiles) {
      fetch(nid, tile[b ^ 1]);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const uint32_t* cur = tile[b];

    if constexpr (DO_ROWS) {
      const bool row_ok = r0 + rr < rows;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint4 w0 = *reinterpret_cast<const uint4*>(&cur[rr * NV_SW + nv_swz(16 * q + 8 * h)]);
        const uint4 w1 = *reinterpret_cast<const uint4*>(&cur[rr * NV_SW + nv_swz(16 * q + 8 * h + 4)]);
        const uint32_t wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
        float v[16];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          v[2 * i] = __uint_as_float(wv[i] << 16);
          v[2 * i + 1] = __uint_as_float(wv[i] & 0xFFFF0000u);
        }
        float a = 0.0f;
        const int64_t col0 = c0 + 32 * q + 16 * h;
        if constexpr (!QUANT) {
          if (rht_r) {
            a = rht16_amax_x2(v, sig_r.s2);
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) a = fmaxf(a, fabsf(v[j]));
          }
          m_r = fmaxf(m_r, a);   // zeros past the edges do not raise it
        } else {
          if (rht_r) rht16_x2(v, sig_r.s2);
#pragma unroll
          for (int j = 0; j < 16; ++j) a = fmaxf(a, fabsf(v[j]));
          if (row_ok && col0 < cols)
            encode_nv_block(v, rht_r != 0, g_r, orr, r0 + rr, col0, rht_r ? __fmul_rn(a, 0.25f) : a, sr_r);
        }
      }
    }
    const int64_t orow = c0 + 2 * pw, ocol0 = r0 + 16 * rb;   // transposed output row / first column
    if constexpr (!QUANT || !TWO_D) {
      // the two columns, each from its own re-read of the staged words; the
      // loop is unrolled so that the compiler can overlap the second column's
      // reads and Philox rounds with the first's (dY dual: 150 -> 147 us)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float v[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const uint32_t wd = cur[(16 * rb + j) * NV_SW + nv_swz(pw)];
          v[j] = __uint_as_float(e ? (wd & 0xFFFF0000u) : (wd << 16));
        }
        float a = 0.0f;
        if constexpr (!QUANT) {
          if (rht_c) {
            a = rht16_amax_x2(v, sig_c.s2);
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) a = fmaxf(a, fabsf(v[j]));
          }
          m_c = fmaxf(m_c, a);
        } else {
          if (rht_c) rht16_x2(v, sig_c.s2);
#pragma unroll
          for (int j = 0; j < 16; ++j) a = fmaxf(a, fabsf(v[j]));
          if (ocol0 < rows && orow + e < cols)
            encode_nv_block(v, rht_c != 0, g_c, oc, orow + e, ocol0, rht_c ? __fmul_rn(a, 0.25f) : a, sr_c);
        }
      }
    } else {
      // 16 x 16 blocks: 8 lanes of adjacent column pairs x 16 rows share one
      // scale, so both columns' maxima come first
      float va[16], vb[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const uint32_t wd = cur[(16 * rb + j) * NV_SW + nv_swz(pw)];
        va[j] = __uint_as_float(wd << 16);
        vb[j] = __uint_as_float(wd & 0xFFFF0000u);
      }
      if (rht_c) {
        rht16_x2(va, sig_c.s2);
        rht16_x2(vb, sig_c.s2);
      }
      float a2 = 0.0f;
#pragma unroll
      for (int j = 0; j < 16; ++j) a2 = fmaxf(a2, fmaxf(fabsf(va[j]), fabsf(vb[j])));
#pragma unroll
      for (int o = 4; o; o >>= 1) a2 = fmaxf(a2, __shfl_xor_sync(0xFFFFFFFFu, a2, o));
      if (rht_c) a2 = __fmul_rn(a2, 0.25f);
      if (ocol0 < rows) {
        if (orow < cols) encode_nv_block(va, rht_c != 0, g_c, oc, orow, ocol0, a2, sr_c);
        if (orow + 1 < cols) encode_nv_block(vb, rht_c != 0, g_c, oc, orow + 1, ocol0, a2, sr_c);
      }
    }
    __syncthreads();   // every thread is done with tile[b] before it is refilled
  }
  if constexpr (!QUANT) {
    if (amax_c) block_amax_atomic(rht_c ? __fmul_rn(m_c, 0.25f) : m_c, amax_c, gen);
    if (DO_ROWS) {
      __syncthreads();
      block_amax_atomic(rht_r ? __fmul_rn(m_r, 0.25f) : m_r, amax_r, gen);
    }
  }
}

// ----------------------------------------------------------------------------
// dequantize: one thread per block
// ----------------------------------------------------------------------------
// Dequantize with any block of 16-128 elements (row-major scales): one thread
// per 16 elements, block index = column >> sb_log2.
template <int FMT, int ODT>
__global__ void __launch_bounds__(kThreads) dequant_blk_kernel(fp4_operand q, int sb_log2, void* out, int64_t ldo) {
  const float g = FMT == FP4_FMT_NVFP4 ? *q.tensor_scale : 1.0f;
  const int64_t units_row = q.k / 16, total = q.rows * units_row, nsf_row = q.k >> sb_log2;
  for (int64_t u = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; u < total; u += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = u / units_row, c0 = (u - r * units_row) * 16;
    const uint32_t sb = q.scales[r * nsf_row + (c0 >> sb_log2)];
    const float s = FMT == FP4_FMT_MXFP4 ? e8m0_scale(sb) : e4m3_decode(sb);
    const uint2 cw = *reinterpret_cast<const uint2*>(q.codes + r * (q.k >> 1) + (c0 >> 1));
    const uint32_t w[2] = {cw.x, cw.y};
    float v[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const uint32_t c = (w[e >> 3] >> (4 * (e & 7))) & 15u;
      const uint32_t m = c & 7u;
      const float mag = m < 4 ? 0.5f * (float)m : (m == 4 ? 2.0f : m == 5 ? 3.0f : m == 6 ? 4.0f : 6.0f);
      float val = __fmul_rn(mag, s);
      if (FMT == FP4_FMT_NVFP4) val = __fmul_rn(val, g);
      v[e] = (c & 8u) ? -val : val;
    }
    const int64_t o0 = r * ldo + c0;
    if constexpr (ODT == FP4_DTYPE_F32) {
      float4* o4 = reinterpret_cast<float4*>(static_cast<float*>(out) + o0);
#pragma unroll
      for (int e = 0; e < 4; ++e) o4[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
    } else {
      uint4* o4 = reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + o0);
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        uint32_t pw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const __nv_bfloat162 h = __floats2bfloat162_rn(v[8 * e + 2 * i], v[8 * e + 2 * i + 1]);
          pw[i] = *reinterpret_cast<const uint32_t*>(&h);
        }
        o4[e] = make_uint4(pw[0], pw[1], pw[2], pw[3]);
      }
    }
  }
}

// one block of codes -> B values (code * s exactly, then * g for NVFP4), stored
template <int FMT, int ODT, int B>
__device__ __forceinline__ void dequant_store(const uint32_t* w, uint32_t sb, float g, void* out, int64_t base) {
  const float s = FMT == FP4_FMT_MXFP4 ? e8m0_scale(sb) : e4m3_decode(sb);
  // each code (sign included) exactly as f16 by the hardware conversion, then
  // code * s (exact: short significands; MXFP4 a power of two), then * g (NVFP4)
  float v[B];
#pragma unroll
  for (int e = 0; e < B / 2; ++e) {
    float lo, hi;
    e2m1x2_decode((w[e >> 2] >> (8 * (e & 3))) & 0xFFu, lo, hi);
    v[2 * e] = __fmul_rn(lo, s);
    v[2 * e + 1] = __fmul_rn(hi, s);
    if (FMT == FP4_FMT_NVFP4) {
      v[2 * e] = __fmul_rn(v[2 * e], g);
      v[2 * e + 1] = __fmul_rn(v[2 * e + 1], g);
    }
  }
  if constexpr (ODT == FP4_DTYPE_F32) {
    float4* o4 = reinterpret_cast<float4*>(static_cast<float*>(out) + base);
#pragma unroll
    for (int e = 0; e < B / 4; ++e) o4[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
  } else {
    uint4* o4 = reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + base);
#pragma unroll
    for (int e = 0; e < B / 8; ++e) {
      uint32_t pk[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 h = __floats2bfloat162_rn(v[8 * e + 2 * i], v[8 * e + 2 * i + 1]);
        pk[i] = *reinterpret_cast<uint32_t*>(&h);
      }
      o4[e] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    }
  }
}

template <int B>
__device__ __forceinline__ void load_codes(const uint8_t* cp, uint32_t* w) {
  if constexpr (B == 16) {
    const uint2 u = *reinterpret_cast<const uint2*>(cp);
    w[0] = u.x; w[1] = u.y;
  } else {
    const uint4 u = *reinterpret_cast<const uint4*>(cp);
    w[0] = u.x; w[1] = u.y; w[2] = u.z; w[3] = u.w;
  }
}

// Two blocks per thread and step, both blocks' loads in flight before either
// is decoded; 32-bit block ids (rows row0 ..) with the multiply-shift divider.
template <int FMT, int ODT>
__global__ void __launch_bounds__(kThreads) dequant_kernel(fp4_operand q, void* out, int64_t ldo, int64_t row0,
                                                           FastDiv nblk, uint32_t total) {
  constexpr int B = FMT == FP4_FMT_MXFP4 ? 32 : 16;
  const int64_t nsf_row = nblk.d, nsf_pad = nsf_padded(q.k, FMT);
  const float g = FMT == FP4_FMT_NVFP4 ? *q.tensor_scale : 1.0f;
  const uint32_t stride = gridDim.x * blockDim.x;
  for (uint32_t blk = blockIdx.x * blockDim.x + threadIdx.x; blk < total; blk += 2 * stride) {
    const uint32_t blk2 = blk + stride;
    const bool two = blk2 < total && blk2 > blk;
    const uint32_t ra = fast_div(blk, nblk), ja = blk - ra * nblk.d;
    const int64_t r = row0 + ra;
    uint32_t rb = 0, jb = 0;
    if (two) {
      rb = fast_div(blk2, nblk);
      jb = blk2 - rb * nblk.d;
    }
    const int64_t r2 = row0 + rb;
    uint32_t w[B / 8], w2[B / 8];
    const uint32_t sb = q.scales[sf_offset(q.sf_layout, r, ja, nsf_row, nsf_pad)];
    load_codes<B>(q.codes + r * (q.k >> 1) + (int64_t)ja * (B / 2), w);
    uint32_t sb2 = 0;
    if (two) {
      sb2 = q.scales[sf_offset(q.sf_layout, r2, jb, nsf_row, nsf_pad)];
      load_codes<B>(q.codes + r2 * (q.k >> 1) + (int64_t)jb * (B / 2), w2);
    }
    dequant_store<FMT, ODT, B>(w, sb, g, out, r * ldo + (int64_t)ja * B);
    if (two) dequant_store<FMT, ODT, B>(w2, sb2, g, out, r2 * ldo + (int64_t)jb * B);
  }
}

// ----------------------------------------------------------------------------
// standalone RHT16 (fp32 out, pitch cols)
// ----------------------------------------------------------------------------
template <int DT>
__global__ void __launch_bounds__(kThreads) rht_rows_kernel(const void* __restrict__ x, int64_t rows,
                                                            int64_t cols, int64_t ldx, uint32_t signs,
                                                            float* y) {
  int64_t nch = cols >> 4, total = rows * nch;
  for (int64_t c = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; c < total;
       c += (int64_t)gridDim.x * blockDim.x) {
    int64_t r = c / nch, k0 = (c - r * nch) << 4;
    float v[16];
    load8<DT>(x, r * ldx + k0, v);
    load8<DT>(x, r * ldx + k0 + 8, v + 8);
    rht16(v, signs);
    float4* o = reinterpret_cast<float4*>(y + r * cols + k0);
#pragma unroll
    for (int e = 0; e < 4; ++e) o[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
  }
}

template <int DT>
__global__ void __launch_bounds__(kThreads) rht_cols_kernel(const void* __restrict__ x, int64_t rows,
                                                            int64_t cols, int64_t ldx, uint32_t signs,
                                                            float* y) {
  int64_t nrb = rows >> 4, total = nrb * cols;
  for (int64_t it = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; it < total;
       it += (int64_t)gridDim.x * blockDim.x) {
    int64_t rb = it / cols, c = it - rb * cols;  // lanes = consecutive columns
    float v[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = load1<DT>(x, (rb * 16 + j) * ldx + c);
    rht16(v, signs);
#pragma unroll
    for (int j = 0; j < 16; ++j) y[(rb * 16 + j) * cols + c] = v[j];
  }
}

// ----------------------------------------------------------------------------
// DGE backward ([msr] §二): dx = dy * min(clamp, (1/k)|u|^(1/k-1)), one thread
// per block of x (blocks along cols)
// ----------------------------------------------------------------------------
// Branch-free: with step 2^(e-1), e = [a >= 2] + [a >= 4], t = a / step is exact
// and u = 2 (t - floor(t)) - 1 is the local coordinate.  powf(0, negative) is
// +inf, so u = 0 lands on the clamp without a special case.
//
// K5: k = 5 (the pages' value), y = |u|^(-4/5) without powf.  y solves
// y^5 u^4 = 1; a fast estimate y0 = __powf(|u|, -0.8) (relative error ~1e-6)
// takes one Newton step for that equation, y1 = y0 (1 + (1 - y0^5 u^4) / 5),
// which squares the relative error (to ~1e-12) and needs no division; what is
// left is the fp32 rounding of the few products, a few ulp.  |u| is 0 or at
// least 2^-24 (t has 24 significant bits), so u^4 >= 2^-96 stays normal; u = 0
// gives y0 = inf and a NaN step, which fminf turns into the clamp, the same
// value the general path reaches through powf(0, negative) = inf.
template <bool K5>
__device__ __forceinline__ float dge_fprime(float xs, float inv_k, float expo, float clamp, float outside) {
  const float a = fabsf(xs);
  const uint32_t e = (a >= 2.0f) + (a >= 4.0f);
  const float t = __fmul_rn(a, __uint_as_float((128u - e) << 23));
  // 2 (t - floor t) - 1 as one fma: 2 (t - floor t) is exact, so the single
  // rounding is the rounding of the subtraction
  const float au = fabsf(__fmaf_rn(__fsub_rn(t, floorf(t)), 2.0f, -1.0f));
  float y;
  if constexpr (K5) {
    const float y0 = __powf(au, -0.8f);
    const float u2 = __fmul_rn(au, au), u4 = __fmul_rn(u2, u2);
    const float y2 = __fmul_rn(y0, y0), y5 = __fmul_rn(__fmul_rn(y2, y2), y0);
    const float e5 = __fmul_rn(y5, u4);
    y = __fmul_rn(y0, __fmaf_rn(-0.2f, e5, 1.2f));
  } else {
    y = powf(au, expo);
  }
  const float f = fminf(clamp, __fmul_rn(inv_k, y));
  return a >= 6.0f ? outside : f;
}

// ----------------------------------------------------------------------------
// Sigmoid-smoothed quantizer ([grad] §3.2) on the signed E2M1 grid
//   q_0..q_14 = -6..6, thresholds c_i = (q_i + q_{i+1}) / 2, steps v_i = q_{i+1} - q_i,
//   Q_soft(xs) = q_0 + sum_i v_i sigma(beta (xs - c_i)),
//   Q_soft'(xs) = beta sum_i v_i sigma(z_i) (1 - sigma(z_i)),  z_i = beta (xs - c_i).
// ----------------------------------------------------------------------------
// Q_soft is odd and Q_soft' even, so both are evaluated at a = |xs|.  With
// t = e^-|z| <= 1: sigma(z) = 1 / (1 + t) for z >= 0 and t / (1 + t) below, and
// sigma (1 - sigma) = t / (1 + t)^2, which keeps full relative precision in the
// tails.  The derivative's terms are summed as one fraction N / D, with
// D = prod (1 + t_i)^2 in [1, 4^14], so the whole sum costs one division.
//
// Window: thresholds are >= 0.5 apart, so the k-th threshold on one side of a
// lies >= 0.5 (k - 1) beyond the nearest one on that side.  Keeping the W
// nearest on each side leaves out terms below 16 e^(-beta W / 2) / (1 - e^(-beta / 2))
// of a kept one (16 = the ratio of the largest to the smallest step, times the
// 4 between e^-|z| and sigma (1 - sigma)); with beta W >= 56 ln 2 that is
// below 2^-24 per side.  W = 0 evaluates all 14 thresholds.
__host__ __device__ constexpr float e2m1_level(int k) {  // k = 0..7
  return k < 4 ? 0.5f * k : (k < 6 ? float(k - 2) : float(2 * k - 8));
}
__host__ __device__ constexpr float soft_level(int i) {  // q_i, i = 0..14
  return i >= 7 ? e2m1_level(i - 7) : -e2m1_level(7 - i);
}
// table entry i: (c_i, v_i) and q_i, the level just below c_i; past the last
// threshold the entries contribute nothing (c = 1e30, v = 0).  (c, v) pairs
// are read per term (8 bytes: two shared-memory wavefronts per warp), q once.
constexpr int kSoftTab = 18;
struct SoftTable {
  float2 cv[kSoftTab];
  float q[kSoftTab];
};
__host__ __device__ constexpr float2 soft_cv(int i) {
  return i < 14 ? float2{0.5f * (soft_level(i) + soft_level(i + 1)), soft_level(i + 1) - soft_level(i)}
                : float2{1e30f, 0.0f};
}
__host__ __device__ constexpr float soft_q(int i) { return i < 14 ? soft_level(i) : 6.0f; }
template <int W>
__device__ __forceinline__ float2 soft_term(const SoftTable* tab, int i0, int m) {
  if constexpr (W == 0) {
    return soft_cv(m);
  } else {
    return tab->cv[i0 + m];
  }
}

// 2^x, PTX ex2.approx.ftz.f32 (relative error ~2^-22; results below 2^-126 flush to 0)
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// index of the first threshold of a's window: thresholds 0..6 are negative,
// so 7 + (number of positive thresholds <= a) is the first one above a
template <int W>
__device__ __forceinline__ int soft_window_start(float a) {
  const int above = (a >= 0.25f) + (a >= 0.75f) + (a >= 1.25f) + (a >= 1.75f) + (a >= 2.5f) + (a >= 3.5f) +
                    (a >= 5.0f);
  return 7 + above - W;
}

// Terms of the 7 negative thresholds -c_p (all below a = |xs| >= 0): the
// exponent of each is beta (a + c_p), so t = e^(-beta a) e^(-beta c_p) -- one ex2
// per element and a launch constant kneg[p] = e^(-beta c_p) per threshold
// instead of one ex2 per term.  The exponent's rounding is of the same order as
// in the direct form (both carry beta (a + c_p)).  Used when all 14 thresholds
// are evaluated (W = 0).
struct SoftNegConst {
  float kneg[7];   // e^(-beta c_p), c_p = 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5
};

// Q_soft'(xs); nbl = -beta log2(e)
template <int W>
__device__ __forceinline__ float soft_grad(float xs, float beta, float nbl, const SoftTable* tab,
                                           const SoftNegConst& kc) {
  const float a = fabsf(xs);
  constexpr int n = W == 0 ? 14 : 2 * W;
  const int i0 = W == 0 ? 0 : soft_window_start<W>(a);
  const float ea = W == 0 ? ex2_approx(a * nbl) : 0.0f;
  float num = 0.0f, den = 1.0f;
#pragma unroll
  for (int m = 0; m < n; ++m) {
    const float2 e = soft_term<W>(tab, i0, m);
    const float t = (W == 0 && m < 7) ? ea * kc.kneg[6 - m] : ex2_approx(fabsf(a - e.x) * nbl);
    const float w = fmaf(t, t + 2.0f, 1.0f);              // (1 + t)^2
    num = fmaf(num, w, e.y * t * den);
    den *= w;
  }
  return beta * __fdividef(num, den);
}

// Q_soft(xs)
template <int W>
__device__ __forceinline__ float soft_value(float xs, float nbl, const SoftTable* tab, const SoftNegConst& kc) {
  const float a = fabsf(xs);
  constexpr int n = W == 0 ? 14 : 2 * W;
  const int i0 = W == 0 ? 0 : soft_window_start<W>(a);
  const float ea = W == 0 ? ex2_approx(a * nbl) : 0.0f;
  float acc = W == 0 ? -6.0f : tab->q[i0];                // the level below the window
#pragma unroll
  for (int m = 0; m < n; ++m) {
    const float2 e = soft_term<W>(tab, i0, m);
    const float d = a - e.x;
    const float t = (W == 0 && m < 7) ? ea * kc.kneg[6 - m] : ex2_approx(fabsf(d) * nbl);
    acc = fmaf(e.y, __fdividef(d >= 0.0f ? 1.0f : t, 1.0f + t), acc);
  }
  return xs < 0.0f ? -acc : acc;
}

// ----------------------------------------------------------------------------
// Maps of the scaled input xs = x / s, one thread per block of x (blocks along
// cols): DGE backward ([msr] §二), Q_soft forward and backward.  xs is formed
// exactly as the quantizer formed it from the stored scale.  Each op gives the
// output element from (xs, s, dy element); ops without kDy take no dy (DYDT < 0).
// ----------------------------------------------------------------------------
template <bool K5>
struct DgeOp {
  float inv_k, expo, clamp, outside;
  static constexpr bool kTable = false, kScale = false, kDy = true;
  __device__ float operator()(float xs, float, float d, const SoftTable*) const {
    return __fmul_rn(d, dge_fprime<K5>(xs, inv_k, expo, clamp, outside));
  }
};
template <int W>
struct SoftGradOp {
  float beta, nbl;
  SoftNegConst kc;
  static constexpr bool kTable = W != 0, kScale = false, kDy = true;
  __device__ float operator()(float xs, float, float d, const SoftTable* tab) const {
    return d * soft_grad<W>(xs, beta, nbl, tab, kc);
  }
};
template <int W>
struct SoftValueOp {
  float nbl;
  SoftNegConst kc;
  static constexpr bool kTable = W != 0, kScale = true, kDy = false;
  __device__ float operator()(float xs, float s, float, const SoftTable* tab) const {
    return s * soft_value<W>(xs, nbl, tab, kc);
  }
};

// Work unit: 8 consecutive elements of a row (16 bytes of bf16 x), so that the
// lanes of a warp read and write contiguous memory; the unit's block scale is
// looked up per unit (the lanes of one block read the same byte).  U units per
// thread per iteration keep their loads in flight together.
constexpr int kMapUnits = 2;
template <int FMT, int XDT, int DYDT, class Op>
__global__ void __launch_bounds__(kThreads) scaled_map_kernel(const void* __restrict__ x, int64_t ldx, fp4_operand q,
                                                              const void* __restrict__ dy, int64_t lddy, float* out,
                                                              int64_t ldo, Op op, FastDiv upr_div) {
  constexpr int B = FMT == FP4_FMT_MXFP4 ? 32 : 16;
  constexpr int U = kMapUnits;
  __shared__ SoftTable tab_s;
  const SoftTable* tab = &tab_s;
  if constexpr (Op::kTable) {
    if (threadIdx.x < kSoftTab) {
      tab_s.cv[threadIdx.x] = soft_cv(threadIdx.x);
      tab_s.q[threadIdx.x] = soft_q(threadIdx.x);
    }
    __syncthreads();
  }
  const int64_t nsf_row = q.k / B, nsf_pad = nsf_padded(q.k, FMT);
  const float g = FMT == FP4_FMT_NVFP4 ? *q.tensor_scale : 0.0f;
  const int64_t upr = q.k / 8, total = q.rows * upr;
  const bool small = total < (int64_t(1) << 31);  // 32-bit unit ids, multiply-shift division
  auto split = [&](int64_t u, int64_t& r, int64_t& c0) {
    if (small) {
      const uint32_t r32 = fast_div((uint32_t)u, upr_div);
      r = r32;
      c0 = (int64_t)((uint32_t)u - r32 * upr_div.d) * 8;
    } else {
      r = u / upr;
      c0 = (u - r * upr) * 8;
    }
  };
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t u0 = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; u0 < total; u0 += U * stride) {
    int64_t r[U], c0[U];
    bool act[U];
    float v[U][8], d[U][8];
    uint32_t sb[U];
#pragma unroll
    for (int i = 0; i < U; ++i) {
      const int64_t u = u0 + i * stride;
      act[i] = u < total;
      r[i] = 0;
      c0[i] = 0;
      if (act[i]) split(u, r[i], c0[i]);
    }
#pragma unroll
    for (int i = 0; i < U; ++i) {
      if (act[i]) {
        load8<XDT>(x, r[i] * ldx + c0[i], v[i]);
        if constexpr (DYDT >= 0) load8<DYDT>(dy, r[i] * lddy + c0[i], d[i]);
        sb[i] = q.scales[sf_offset(q.sf_layout, r[i], c0[i] / B, nsf_row, nsf_pad)];
      }
    }
#pragma unroll
    for (int i = 0; i < U; ++i) {
      if (!act[i]) continue;
      // xs = x * mult exactly as the quantizer formed it; s the block scale
      float mult, sv;
      if (FMT == FP4_FMT_MXFP4) {
        mult = e8m0_inv_scale(sb[i]);
        sv = Op::kScale ? e8m0_scale(sb[i]) : 0.0f;
      } else {
        sv = __fmul_rn(e4m3_decode(sb[i]), g);
        mult = sv == 0.0f ? 0.0f : __frcp_rn(sv);
      }
      float o[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = op(__fmul_rn(v[i][e], mult), sv, DYDT >= 0 ? d[i][e] : 0.0f, tab);
      float4* dst = reinterpret_cast<float4*>(out + r[i] * ldo + c0[i]);
      dst[0] = make_float4(o[0], o[1], o[2], o[3]);
      dst[1] = make_float4(o[4], o[5], o[6], o[7]);
    }
  }
}

// ----------------------------------------------------------------------------
// Quantization quality ([msr] §三 cosine / MSE / SNR; [grad] §5.1 relative
// error): sums of x^2, x_hat^2, x x_hat, (x - x_hat)^2 in fp64 over a tensor and
// its quantization (any block of 16-128), one thread per 16 elements.
//   x_hat = dequant(code)                    (+ x - clamp(x, tau) with OCC)
//   x_hat = s Q_soft(x / s)                  (SOFT: the sigmoid-smoothed value)
// ----------------------------------------------------------------------------
__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

template <int FMT, int XDT, bool SOFT>
__global__ void __launch_bounds__(256) error_stats_kernel(const void* __restrict__ x, int64_t ldx, fp4_operand q,
                                                          int sb_log2, const float* __restrict__ tau_p, float nbl,
                                                          double* sums) {
  const int64_t nsf_row = q.k >> sb_log2, nsf_pad = nsf_padded(q.k, FMT);
  const float g = FMT == FP4_FMT_NVFP4 ? *q.tensor_scale : 0.0f;
  const bool occ = tau_p != nullptr;
  const float tau = occ ? *tau_p : 0.0f;
  const int64_t units_row = q.k / 16, total = q.rows * units_row;
  SoftNegConst kc;
  if constexpr (SOFT) {
    const float cp[7] = {0.25f, 0.75f, 1.25f, 1.75f, 2.5f, 3.5f, 5.0f};
#pragma unroll
    for (int i = 0; i < 7; ++i) kc.kneg[i] = ex2_approx(nbl * cp[i]);
  }
  double sxx = 0.0, shh = 0.0, sxh = 0.0, see = 0.0;
  for (int64_t u = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; u < total; u += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = u / units_row, c0 = (u - r * units_row) * 16;
    const uint32_t sb = q.scales[sf_offset(q.sf_layout, r, c0 >> sb_log2, nsf_row, nsf_pad)];
    float v[16];
    load8<XDT>(x, r * ldx + c0, v);
    load8<XDT>(x, r * ldx + c0 + 8, v + 8);
    float h32[16];
    if constexpr (SOFT) {
      float s, mult;
      if (FMT == FP4_FMT_MXFP4) {
        s = e8m0_scale(sb);
        mult = e8m0_inv_scale(sb);
      } else {
        s = __fmul_rn(e4m3_decode(sb), g);
        mult = s == 0.0f ? 0.0f : __frcp_rn(s);
      }
#pragma unroll
      for (int e = 0; e < 16; ++e) h32[e] = s * soft_value<0>(__fmul_rn(v[e], mult), nbl, nullptr, kc);
    } else {
      const float s = FMT == FP4_FMT_MXFP4 ? e8m0_scale(sb) : e4m3_decode(sb);
      const uint2 cw = *reinterpret_cast<const uint2*>(q.codes + r * (q.k >> 1) + (c0 >> 1));
      const uint32_t w[2] = {cw.x, cw.y};
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const uint32_t code = (w[e >> 3] >> (4 * (e & 7))) & 15u;
        const uint32_t mc = code & 7u;
        const float mag = mc < 4 ? 0.5f * (float)mc : (mc == 4 ? 2.0f : mc == 5 ? 3.0f : mc == 6 ? 4.0f : 6.0f);
        float d = __fmul_rn(mag, s);
        if (FMT == FP4_FMT_NVFP4) d = __fmul_rn(d, g);
        h32[e] = (code & 8u) ? -d : d;
      }
    }
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      double h = (double)h32[e];
      if (!SOFT && occ && fabsf(v[e]) > tau) h += (double)__fsub_rn(v[e], copysignf(tau, v[e]));
      const double xv = (double)v[e], ev = xv - h;
      sxx = fma(xv, xv, sxx);
      shh = fma(h, h, shh);
      sxh = fma(xv, h, sxh);
      see = fma(ev, ev, see);
    }
  }
  __shared__ double part[4][8];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  sxx = warp_sum_d(sxx);
  shh = warp_sum_d(shh);
  sxh = warp_sum_d(sxh);
  see = warp_sum_d(see);
  if (lane == 0) {
    part[0][w] = sxx;
    part[1][w] = shh;
    part[2][w] = sxh;
    part[3][w] = see;
  }
  __syncthreads();
  if (threadIdx.x < 4) {
    double t = 0.0;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) t += part[threadIdx.x][i];
    atomicAdd(&sums[threadIdx.x], t);
  }
}

// cosine = s2 / sqrt(s0 s1), MSE = s3 / n, SNR = 10 log10(s0 / s3) dB and the
// relative L2 error sqrt(s3 / s0) from the four sums (one thread); an
// undefined ratio (a zero denominator) gives NaN, a zero error an infinite SNR
__global__ void error_stats_finalize_kernel(const double* sums, double n, double* stats) {
  const double sxx = sums[0], shh = sums[1], sxh = sums[2], see = sums[3];
  const double nan = __longlong_as_double(0x7FF8000000000000ll), inf = __longlong_as_double(0x7FF0000000000000ll);
  stats[0] = (sxx > 0.0 && shh > 0.0) ? sxh / sqrt(sxx * shh) : nan;
  stats[1] = n > 0.0 ? see / n : nan;
  stats[2] = (sxx > 0.0 && see > 0.0) ? 10.0 * log10(sxx / see) : (sxx > 0.0 ? inf : nan);
  stats[3] = sxx > 0.0 ? sqrt(see / sxx) : nan;
}

// ----------------------------------------------------------------------------
// element encoders
// ----------------------------------------------------------------------------
__global__ void encode_e2m1_kernel(const float* xs, uint8_t* codes, int64_t n, int method) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    float v = xs[i];
    codes[i] = (uint8_t)(method == 0 ? e2m1x2_hw(v, 0.0f) & 15u : e2m1_sw(v));
  }
}
__global__ void encode_e4m3_kernel(const float* t, uint8_t* out, int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    out[i] = (uint8_t)e4m3_rn_satfinite(t[i]);
}

}  // namespace

// ============================================================================
// launchers
// ============================================================================
#define FP4_DISPATCH_DT(dt, DT, ...)          \
  if ((dt) == FP4_DTYPE_BF16) {               \
    constexpr int DT = FP4_DTYPE_BF16;        \
    __VA_ARGS__;                              \
  } else {                                    \
    constexpr int DT = FP4_DTYPE_F32;         \
    __VA_ARGS__;                              \
  }
#define FP4_DISPATCH_FMT(fmt, FMT, ...)       \
  if ((fmt) == FP4_FMT_MXFP4) {               \
    constexpr int FMT = FP4_FMT_MXFP4;        \
    __VA_ARGS__;                              \
  } else {                                    \
    constexpr int FMT = FP4_FMT_NVFP4;        \
    __VA_ARGS__;                              \
  }

cudaError_t launch_amax(const void* x, int dt, int64_t rows, int64_t cols, int64_t ldx, int rht_axis,
                        uint32_t rht_signs, float* amax_out, uint32_t gen, int num_sms, cudaStream_t st) {
  // rht_axis: -1 none, 1 along cols (needs cols % 16 == 0), 0 along rows (rows % 16 == 0)
  if (!gen) {  // a plain float output is zeroed first; a tagged slot needs no zeroing
    cudaError_t e = cudaMemsetAsync(amax_out, 0, sizeof(float), st);
    if (e != cudaSuccess) return e;
  }
  if (rows == 0 || cols == 0) return cudaSuccess;
  if (rht_axis != 0 && cols % 16 == 0) {
    const int64_t nch = cols / 16, total = rows * nch;
    if (total < (int64_t(1) << 31)) {
      int grid = grid_for(cdiv(total, 2), kThreads, num_sms);
      const FastDiv fd = make_fastdiv((uint32_t)nch);
      const int contiguous = ldx == cols;
      FP4_DISPATCH_DT(dt, DT,
        if (rht_axis == 1) amax_rows32_kernel<DT, true><<<grid, kThreads, 0, st>>>(x, ldx, fd, (uint32_t)total, contiguous, rht_signs, amax_out, gen);
        else amax_rows32_kernel<DT, false><<<grid, kThreads, 0, st>>>(x, ldx, fd, (uint32_t)total, contiguous, rht_signs, amax_out, gen));
      return cudaGetLastError();
    }
    int grid = grid_for(total, kThreads, num_sms);
    FP4_DISPATCH_DT(dt, DT,
      if (rht_axis == 1) amax_rows_kernel<DT, true><<<grid, kThreads, 0, st>>>(x, rows, cols, ldx, rht_signs, amax_out, gen);
      else amax_rows_kernel<DT, false><<<grid, kThreads, 0, st>>>(x, rows, cols, ldx, rht_signs, amax_out, gen));
    return cudaGetLastError();
  }
  // transform along rows, or a plain amax of a tensor whose cols are not a
  // multiple of 16: column items of a tiled kernel
  QuantOut none{};
  if (dt == FP4_DTYPE_BF16) {
    const int64_t ntc = cdiv(cols, NV_TC), nt = cdiv(rows, NV_TR) * ntc;
    if (nt >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
    tile_nv_kernel<T_AMAX_COLS, false><<<grid_for(nt, 1, num_sms), kThreads, 0, st>>>(
        static_cast<const uint16_t*>(x), rows, cols, ldx, make_fastdiv((uint32_t)ntc), (uint32_t)nt, none, none,
        rht_sign_floats(rht_signs), rht_sign_floats(0u), rht_axis == 0 ? 1 : 0, 0, amax_out, nullptr, gen);
    return cudaGetLastError();
  }
  int64_t ntiles = cdiv(rows, 64) * cdiv(cols, TC);
  if (ntiles >= (int64_t(1) << 31)) return cudaErrorInvalidValue;  // tile ids are 32-bit
  int grid = grid_for(ntiles, 1, num_sms);
  FP4_DISPATCH_DT(dt, DT, tile_kernel<FP4_FMT_NVFP4, DT, T_AMAX_COLS><<<grid, kThreads, 0, st>>>(
      x, rows, cols, ldx, none, none, 0, rht_signs, 0u, rht_axis == 0 ? 1 : 0, 0, amax_out, nullptr, gen));
  return cudaGetLastError();
}

cudaError_t launch_amax_dual(const void* x, int dt, int64_t rows, int64_t cols, int64_t ldx,
                             uint32_t signs_rows, uint32_t signs_cols, bool rht_rows, bool rht_cols,
                             float* amax_rows, float* amax_cols, uint32_t gen, int num_sms, cudaStream_t st) {
  // amax_rows: the tensor that is blocked along cols (RHT along cols, "row items")
  cudaError_t e = cudaSuccess;
  if (!gen) {
    e = cudaMemsetAsync(amax_rows, 0, sizeof(float), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(amax_cols, 0, sizeof(float), st);
  }
  if (e != cudaSuccess || rows == 0 || cols == 0) return e;
  QuantOut none{};
  if (dt == FP4_DTYPE_BF16) {
    const int64_t ntc = cdiv(cols, NV_TC), nt = cdiv(rows, NV_TR) * ntc;
    if (nt >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
    tile_nv_kernel<T_AMAX_DUAL, false><<<grid_for(nt, 1, num_sms), kThreads, 0, st>>>(
        static_cast<const uint16_t*>(x), rows, cols, ldx, make_fastdiv((uint32_t)ntc), (uint32_t)nt, none, none,
        rht_sign_floats(signs_cols), rht_sign_floats(signs_rows), rht_cols ? 1 : 0, rht_rows ? 1 : 0, amax_cols,
        amax_rows, gen);
    return cudaGetLastError();
  }
  int64_t ntiles = cdiv(rows, 64) * cdiv(cols, TC);
  if (ntiles >= (int64_t(1) << 31)) return cudaErrorInvalidValue;  // tile ids are 32-bit
  int grid = grid_for(ntiles, 1, num_sms);
  FP4_DISPATCH_DT(dt, DT, tile_kernel<FP4_FMT_NVFP4, DT, T_AMAX_DUAL><<<grid, kThreads, 0, st>>>(
      x, rows, cols, ldx, none, none, 0, signs_cols, signs_rows, rht_cols, rht_rows, amax_cols, amax_rows, gen));
  return cudaGetLastError();
}

cudaError_t launch_quant_rows(const void* x, int dt, int64_t rows, int64_t cols, int64_t ldx, int fmt,
                              const QuantOut& o, int num_sms, cudaStream_t st) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  int B = fmt == FP4_FMT_MXFP4 ? 32 : 16;
  const int64_t nblk = cols / B, total = rows * nblk;
  if (total < (int64_t(1) << 31)) {
    int grid = grid_for(cdiv(total, 2), kThreads, num_sms);
    const FastDiv fd = make_fastdiv((uint32_t)nblk);
    const int contiguous = ldx == cols;
    const bool plain = o.rounding == FP4_ROUND_RTN && !o.rht;
    FP4_DISPATCH_FMT(fmt, FMT, FP4_DISPATCH_DT(dt, DT,
      if (plain) quant_rows32_kernel<FMT, DT, true><<<grid, kThreads, 0, st>>>(x, ldx, fd, (uint32_t)total, contiguous, o);
      else quant_rows32_kernel<FMT, DT, false><<<grid, kThreads, 0, st>>>(x, ldx, fd, (uint32_t)total, contiguous, o)));
    return cudaGetLastError();
  }
  int grid = grid_for(total, kThreads, num_sms);
  FP4_DISPATCH_FMT(fmt, FMT, FP4_DISPATCH_DT(dt, DT,
      quant_rows_kernel<FMT, DT><<<grid, kThreads, 0, st>>>(x, rows, cols, ldx, o)));
  return cudaGetLastError();
}

cudaError_t launch_quant_rows_clamped(const void* x, int dt, int64_t rows, int64_t cols, int64_t ldx, int fmt,
                                      const QuantOut& o, int num_sms, cudaStream_t st) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  int B = fmt == FP4_FMT_MXFP4 ? 32 : 16;
  const int64_t nblk = cols / B, total = rows * nblk;
  if (total >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
  int grid = grid_for(cdiv(total, 2), kThreads, num_sms);
  const FastDiv fd = make_fastdiv((uint32_t)nblk);
  const int contiguous = ldx == cols;
  const bool plain = o.rounding == FP4_ROUND_RTN && !o.rht;
  const size_t smem = (o.col_counts && cols <= kClampSmemCols) ? sizeof(uint32_t) * cols : 0;
  FP4_DISPATCH_FMT(fmt, FMT, FP4_DISPATCH_DT(dt, DT,
    if (plain) quant_rows32_kernel<FMT, DT, true, true><<<grid, kThreads, smem, st>>>(x, ldx, fd, (uint32_t)total, contiguous, o);
    else quant_rows32_kernel<FMT, DT, false, true><<<grid, kThreads, smem, st>>>(x, ldx, fd, (uint32_t)total, contiguous, o)));
  return cudaGetLastError();
}

cudaError_t launch_quant_rows_zeroed(const void* x, int dt, int64_t rows, int64_t cols, int64_t ldx, int fmt,
                                     const QuantOut& o, int num_sms, cudaStream_t st) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  int B = fmt == FP4_FMT_MXFP4 ? 32 : 16;
  const int64_t nblk = cols / B, total = rows * nblk;
  if (total >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
  int grid = grid_for(cdiv(total, 2), kThreads, num_sms);
  const FastDiv fd = make_fastdiv((uint32_t)nblk);
  const int contiguous = ldx == cols;
  const bool plain = o.rounding == FP4_ROUND_RTN && !o.rht;
  const size_t smem = cols <= kZeroSmemCols ? sizeof(uint32_t) * (size_t)cdiv(cols, 32) : 0;
  FP4_DISPATCH_FMT(fmt, FMT, FP4_DISPATCH_DT(dt, DT,
    if (plain) quant_rows32_kernel<FMT, DT, true, false, true><<<grid, kThreads, smem, st>>>(x, ldx, fd, (uint32_t)total, contiguous, o);
    else quant_rows32_kernel<FMT, DT, false, false, true><<<grid, kThreads, smem, st>>>(x, ldx, fd, (uint32_t)total, contiguous, o)));
  return cudaGetLastError();
}

cudaError_t launch_amax_zeroed(const void* x, int dt, int64_t rows, int64_t cols, int64_t ldx, const int32_t* hot,
                               int n, float* amax_out, uint32_t gen, int num_sms, cudaStream_t st) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  const int64_t nch = cols / 16, total = rows * nch;
  if (total >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
  const int grid = grid_for(total, kThreads, num_sms);
  const FastDiv fd = make_fastdiv((uint32_t)nch);
  const size_t smem = cols <= kZeroSmemCols ? sizeof(uint32_t) * (size_t)cdiv(cols, 32) : 0;
  FP4_DISPATCH_DT(dt, DT, amax_zeroed_kernel<DT><<<grid, kThreads, smem, st>>>(x, ldx, fd, (uint32_t)total, hot, n,
                                                                              amax_out, gen));
  return cudaGetLastError();
}

cudaError_t launch_quant_tile(const void* x, int dt, int64_t rows, int64_t cols, int64_t ldx, int fmt,
                              bool two_d, bool transpose, const QuantOut& o, int num_sms, cudaStream_t st) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  int TRv = fmt == FP4_FMT_MXFP4 ? 128 : 64;
  int64_t ntiles = cdiv(rows, TRv) * cdiv(cols, TC);
  if (ntiles >= (int64_t(1) << 31)) return cudaErrorInvalidValue;  // tile ids are 32-bit
  int grid = grid_for(ntiles, 1, num_sms);
  if (transpose && fmt == FP4_FMT_NVFP4 && dt == FP4_DTYPE_BF16) {
    const int64_t ntc = cdiv(cols, NV_TC), nt = cdiv(rows, NV_TR) * ntc;
    if (nt >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
    const FastDiv fd = make_fastdiv((uint32_t)ntc);
    const int grid = grid_for(nt, 1, num_sms);
    const auto* xs = static_cast<const uint16_t*>(x);
    if (two_d)
      tile_nv_kernel<T_Q_COLS, true><<<grid, kThreads, 0, st>>>(xs, rows, cols, ldx, fd, (uint32_t)nt, o, o,
                                                                rht_sign_floats(o.rht_signs), rht_sign_floats(0u),
                                                                o.rht, 0, nullptr, nullptr);
    else
      tile_nv_kernel<T_Q_COLS, false><<<grid, kThreads, 0, st>>>(xs, rows, cols, ldx, fd, (uint32_t)nt, o, o,
                                                                 rht_sign_floats(o.rht_signs), rht_sign_floats(0u),
                                                                 o.rht, 0, nullptr, nullptr);
    return cudaGetLastError();
  }
  if (transpose) {
    FP4_DISPATCH_FMT(fmt, FMT, FP4_DISPATCH_DT(dt, DT, tile_kernel<FMT, DT, T_Q_COLS><<<grid, kThreads, 0, st>>>(
        x, rows, cols, ldx, o, o, two_d ? 1 : 0, o.rht_signs, 0u, o.rht, 0, nullptr, nullptr)));
  } else {  // 2D, blocks along cols
    FP4_DISPATCH_FMT(fmt, FMT, FP4_DISPATCH_DT(dt, DT, tile_kernel<FMT, DT, T_Q_ROWS2D><<<grid, kThreads, 0, st>>>(
        x, rows, cols, ldx, o, o, 1, 0u, o.rht_signs, 0, o.rht, nullptr, nullptr)));
  }
  return cudaGetLastError();
}

cudaError_t launch_quant_dual(const void* x, int dt, int64_t rows, int64_t cols, int64_t ldx, int fmt,
                              const QuantOut& orow, const QuantOut& ocol, bool two_d_rows, bool two_d_cols,
                              int num_sms, cudaStream_t st) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  if (fmt == FP4_FMT_NVFP4 && dt == FP4_DTYPE_BF16 && !two_d_rows) {
    const int64_t ntc = cdiv(cols, NV_TC), nt = cdiv(rows, NV_TR) * ntc;
    if (nt >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
    const FastDiv fd = make_fastdiv((uint32_t)ntc);
    const int grid = grid_for(nt, 1, num_sms);
    const auto* xs = static_cast<const uint16_t*>(x);
    if (two_d_cols)
      tile_nv_kernel<T_Q_DUAL, true><<<grid, kThreads, 0, st>>>(xs, rows, cols, ldx, fd, (uint32_t)nt, ocol, orow,
                                                                rht_sign_floats(ocol.rht_signs),
                                                                rht_sign_floats(orow.rht_signs), ocol.rht, orow.rht,
                                                                nullptr, nullptr);
    else
      tile_nv_kernel<T_Q_DUAL, false><<<grid, kThreads, 0, st>>>(xs, rows, cols, ldx, fd, (uint32_t)nt, ocol, orow,
                                                                 rht_sign_floats(ocol.rht_signs),
                                                                 rht_sign_floats(orow.rht_signs), ocol.rht, orow.rht,
                                                                 nullptr, nullptr);
    return cudaGetLastError();
  }
  int TRv = fmt == FP4_FMT_MXFP4 ? 128 : 64;
  int64_t ntiles = cdiv(rows, TRv) * cdiv(cols, TC);
  if (ntiles >= (int64_t(1) << 31)) return cudaErrorInvalidValue;  // tile ids are 32-bit
  int grid = grid_for(ntiles, 1, num_sms);
  FP4_DISPATCH_FMT(fmt, FMT, FP4_DISPATCH_DT(dt, DT, tile_kernel<FMT, DT, T_Q_DUAL><<<grid, kThreads, 0, st>>>(
      x, rows, cols, ldx, ocol, orow, (two_d_cols ? 1 : 0) | (two_d_rows ? 2 : 0), ocol.rht_signs, orow.rht_signs,
      ocol.rht, orow.rht, nullptr, nullptr)));
  return cudaGetLastError();
}

static int log2_block(int b) { return b == 16 ? 4 : b == 32 ? 5 : b == 64 ? 6 : 7; }

cudaError_t launch_quant_rows_blk(const void* x, int dt, int64_t rows, int64_t cols, int64_t ldx, int fmt, int block,
                                  const QuantOut& o, int num_sms, cudaStream_t st) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  const int grid = grid_for(rows * (cols / 16), kThreads, num_sms);
#define FP4_BLK(G)                                                                                         \
  FP4_DISPATCH_FMT(fmt, FMT, FP4_DISPATCH_DT(dt, DT,                                                       \
    quant_rows_blk_kernel<FMT, DT, G><<<grid, kThreads, 0, st>>>(x, rows, cols, ldx, o)))
  switch (block) {
    case 16: FP4_BLK(1); break;
    case 32: FP4_BLK(2); break;
    case 64: FP4_BLK(4); break;
    default: FP4_BLK(8); break;
  }
#undef FP4_BLK
  return cudaGetLastError();
}

static cudaError_t launch_error_sums(const void* x, int xdt, int64_t ldx, const fp4_operand& q, int block,
                                     const float* tau, float beta, double* sums, int num_sms, cudaStream_t st) {
  const int64_t total = q.rows * (q.k / 16);
  const int grid = grid_for(total, 256, num_sms);
  const int sbl = log2_block(block);
  const float nbl = -beta * 1.4426950408889634f;
  FP4_DISPATCH_FMT(q.format, FMT, FP4_DISPATCH_DT(xdt, XDT,
    if (beta > 0.0f) error_stats_kernel<FMT, XDT, true><<<grid, 256, 0, st>>>(x, ldx, q, sbl, nullptr, nbl, sums);
    else error_stats_kernel<FMT, XDT, false><<<grid, 256, 0, st>>>(x, ldx, q, sbl, tau, 0.0f, sums)));
  return cudaGetLastError();
}

cudaError_t launch_error_stats(const void* x, int xdt, int64_t ldx, const fp4_operand& q, int block,
                               const float* tau, float beta, double* sums, double* stats, int num_sms,
                               cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(sums, 0, 4 * sizeof(double), st);
  if (e != cudaSuccess) return e;
  const int64_t total = q.rows * (q.k / 16);
  if (total > 0) {
    e = launch_error_sums(x, xdt, ldx, q, block, tau, beta, sums, num_sms, st);
    if (e != cudaSuccess) return e;
  }
  if (!stats) return cudaSuccess;
  error_stats_finalize_kernel<<<1, 1, 0, st>>>(sums, (double)q.rows * (double)q.k, stats);
  return cudaGetLastError();
}

cudaError_t launch_dequant(const fp4_operand& q, int out_dt, void* out, int64_t ldo, int num_sms,
                           cudaStream_t st) {
  int B = q.format == FP4_FMT_MXFP4 ? 32 : 16;
  if (q.block && q.block != B) {
    const int64_t units = q.rows * (q.k / 16);
    if (units == 0) return cudaSuccess;
    const int grid = grid_for(units, kThreads, num_sms);
    const int sbl = log2_block(q.block);
    FP4_DISPATCH_FMT(q.format, FMT,
      if (out_dt == FP4_DTYPE_F32) dequant_blk_kernel<FMT, FP4_DTYPE_F32><<<grid, kThreads, 0, st>>>(q, sbl, out, ldo);
      else dequant_blk_kernel<FMT, FP4_DTYPE_BF16><<<grid, kThreads, 0, st>>>(q, sbl, out, ldo));
    return cudaGetLastError();
  }
  const int64_t nsf_row = q.k / B;
  if (q.rows == 0 || nsf_row == 0) return cudaSuccess;
  // launches of at most 2^31 blocks (32-bit block ids)
  const int64_t rows_per = std::max<int64_t>(1, ((int64_t(1) << 31) - 1) / nsf_row);
  const FastDiv fd = make_fastdiv((uint32_t)nsf_row);
  for (int64_t r0 = 0; r0 < q.rows; r0 += rows_per) {
    const int64_t total = std::min(rows_per, q.rows - r0) * nsf_row;
    const int grid = grid_for(cdiv(total, 2), kThreads, num_sms);
    FP4_DISPATCH_FMT(q.format, FMT,
      if (out_dt == FP4_DTYPE_F32)
        dequant_kernel<FMT, FP4_DTYPE_F32><<<grid, kThreads, 0, st>>>(q, out, ldo, r0, fd, (uint32_t)total);
      else dequant_kernel<FMT, FP4_DTYPE_BF16><<<grid, kThreads, 0, st>>>(q, out, ldo, r0, fd, (uint32_t)total));
  }
  return cudaGetLastError();
}

cudaError_t launch_rht16(const void* x, int dt, int64_t rows, int64_t cols, int64_t ldx, int axis,
                         uint32_t signs, float* y, int num_sms, cudaStream_t st) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  if (axis == 1) {
    int grid = grid_for(rows * (cols / 16), kThreads, num_sms);
    FP4_DISPATCH_DT(dt, DT, rht_rows_kernel<DT><<<grid, kThreads, 0, st>>>(x, rows, cols, ldx, signs, y));
  } else {
    int grid = grid_for((rows / 16) * cols, kThreads, num_sms);
    FP4_DISPATCH_DT(dt, DT, rht_cols_kernel<DT><<<grid, kThreads, 0, st>>>(x, rows, cols, ldx, signs, y));
  }
  return cudaGetLastError();
}

template <class Op>
cudaError_t launch_scaled_map(const void* x, int xdt, int64_t ldx, const fp4_operand& q, const void* dy, int dydt,
                              int64_t lddy, float* out, int64_t ldo, const Op& op, int num_sms, cudaStream_t st) {
  const int64_t total = q.rows * (q.k / 8);   // 8-element units
  if (total == 0) return cudaSuccess;
  const int grid = grid_for(cdiv(total, kMapUnits), kThreads, num_sms);
  const FastDiv fd = make_fastdiv((uint32_t)std::min<int64_t>(q.k / 8, 0x7FFFFFFF));
  FP4_DISPATCH_FMT(q.format, FMT, FP4_DISPATCH_DT(xdt, XDT,
    if constexpr (!Op::kDy)
      scaled_map_kernel<FMT, XDT, -1, Op><<<grid, kThreads, 0, st>>>(x, ldx, q, dy, lddy, out, ldo, op, fd);
    else if (dydt == FP4_DTYPE_BF16)
      scaled_map_kernel<FMT, XDT, FP4_DTYPE_BF16, Op><<<grid, kThreads, 0, st>>>(x, ldx, q, dy, lddy, out, ldo, op, fd);
    else
      scaled_map_kernel<FMT, XDT, FP4_DTYPE_F32, Op><<<grid, kThreads, 0, st>>>(x, ldx, q, dy, lddy, out, ldo, op, fd)));
  return cudaGetLastError();
}

cudaError_t launch_dge(const void* x, int xdt, int64_t ldx, const fp4_operand& q, const void* dy, int dydt,
                       int64_t lddy, float* dx, int64_t lddx, float k, float clamp, float outside,
                       int num_sms, cudaStream_t st) {
  const float inv_k = 1.0f / k, expo = 1.0f / k - 1.0f;
  if (k == 5.0f)
    return launch_scaled_map(x, xdt, ldx, q, dy, dydt, lddy, dx, lddx, DgeOp<true>{inv_k, expo, clamp, outside},
                             num_sms, st);
  return launch_scaled_map(x, xdt, ldx, q, dy, dydt, lddy, dx, lddx, DgeOp<false>{inv_k, expo, clamp, outside},
                           num_sms, st);
}

// Window per side from beta (beta W >= 56 ln 2 = 38.816; W = 0: all thresholds).
int soft_window(float beta) {
  return beta >= 38.82f ? 1 : beta >= 19.41f ? 2 : beta >= 9.71f ? 4 : 0;
}

static SoftNegConst soft_neg_const(float nbl) {
  static const float c[7] = {0.25f, 0.75f, 1.25f, 1.75f, 2.5f, 3.5f, 5.0f};
  SoftNegConst k;
  for (int p = 0; p < 7; ++p) k.kneg[p] = exp2f(nbl * c[p]);
  return k;
}

cudaError_t launch_soft(const void* x, int xdt, int64_t ldx, const fp4_operand& q, const void* dy, int dydt,
                        int64_t lddy, float* out, int64_t ldo, float beta, int num_sms, cudaStream_t st) {
  const float nbl = -beta * 1.4426950408889634f;  // -beta log2(e)
  const SoftNegConst kc = soft_neg_const(nbl);
#define FP4_SOFT_LAUNCH(W)                                                                                         \
  return dy ? launch_scaled_map(x, xdt, ldx, q, dy, dydt, lddy, out, ldo, SoftGradOp<W>{beta, nbl, kc}, num_sms, st) \
            : launch_scaled_map(x, xdt, ldx, q, nullptr, 0, 0, out, ldo, SoftValueOp<W>{nbl, kc}, num_sms, st)
  switch (soft_window(beta)) {
    case 1: FP4_SOFT_LAUNCH(1);
    case 2: FP4_SOFT_LAUNCH(2);
    case 4: FP4_SOFT_LAUNCH(4);
    default: FP4_SOFT_LAUNCH(0);
  }
#undef FP4_SOFT_LAUNCH
}

cudaError_t launch_encode_e2m1(const float* xs, uint8_t* codes, int64_t n, int method, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  int grid = (int)std::min<int64_t>(cdiv(n, kThreads), 4096);
  encode_e2m1_kernel<<<grid, kThreads, 0, st>>>(xs, codes, n, method);
  return cudaGetLastError();
}
cudaError_t launch_encode_e4m3(const float* t, uint8_t* out, int64_t n, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  int grid = (int)std::min<int64_t>(cdiv(n, kThreads), 4096);
  encode_e4m3_kernel<<<grid, kThreads, 0, st>>>(t, out, n);
  return cudaGetLastError();
}

}  // namespace fp4
