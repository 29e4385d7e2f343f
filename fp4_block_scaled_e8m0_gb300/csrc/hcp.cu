// Hot-channel compensation ([outlier] §3.1-3.2, §4.1).
//
// The quantized product splits into the exact product, first-order and
// second-order error terms ([outlier] §3.1, error-decomposition equation).
// On the k_hot channels with the largest quantization error ("top 9% of
// channels", [outlier] §4.1) the GEMM gets bf16 extra K columns that restore
// those terms: with dX = X - X_hat and dW = W - W_hat,
//   order 2:  A_ext = [dX_H | X_H],  B_ext = [W_hat_H | dW_H] / alpha
//   order 1:  A_ext = [X_H],         B_ext = [dW_H] / alpha  (the page's concat)
//   order 0:  A_ext = [X_H],         B_ext = [W_H] / alpha   (hot channels zeroed in
//             X before it was quantized: their whole product runs in bf16)
// B_ext is divided by alpha = gX * gW so that the GEMM epilogue multiplies the
// whole accumulator (FP4 part and bf16 part) by alpha.
//
// Kernels: per-channel squared error (selection metric), rank-based top-k
// selection (ties to the lower index), and the gather of the extra columns.
#include <cuda_bf16.h>

#include "fp4_device.cuh"

using namespace fp4dev;

namespace fp4 {
namespace {

template <int FMT>
__device__ __forceinline__ float dequant_elem(const fp4_operand& q, int64_t r, int64_t c, float g, int64_t nsf_row,
                                              int64_t nsf_pad) {
  constexpr int B = FMT == FP4_FMT_MXFP4 ? 32 : 16;
  uint32_t byte = q.codes[r * (q.k >> 1) + (c >> 1)];
  uint32_t code = (c & 1) ? (byte >> 4) : (byte & 15u);
  uint32_t sb = q.scales[sf_offset(q.sf_layout, r, c / B, nsf_row, nsf_pad)];
  uint32_t m = code & 7u;
  float mag = m < 4 ? 0.5f * (float)m : (m == 4 ? 2.0f : m == 5 ? 3.0f : m == 6 ? 4.0f : 6.0f);
  float v;
  if (FMT == FP4_FMT_MXFP4) {
    v = __fmul_rn(mag, e8m0_scale(sb));
  } else {
    v = __fmul_rn(__fmul_rn(mag, e4m3_decode(sb)), g);
  }
  return (code & 8u) ? -v : v;
}

// err[c] += sum over this CTA's rows of (x - x_hat)^2.  threadIdx.x: a block of
// B consecutive channels (row-contiguous lanes: a warp reads whole 512-byte
// runs of a row), threadIdx.y: a row group; rows strided over the grid's y
// extent, two rows' loads in flight.  The row groups' sums meet in shared
// memory, and each CTA adds one value per channel to err.
template <int FMT>
__global__ void __launch_bounds__(512) channel_err_kernel(const uint16_t* __restrict__ x, int64_t ldx, fp4_operand q,
                                                          float* err) {
  constexpr int B = FMT == FP4_FMT_MXFP4 ? 32 : 16;
  __shared__ float part[512];
  const int64_t nblk = q.k / B;
  const int64_t cb = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  const bool live = cb < nblk;
  const int64_t nsf_row = nblk, nsf_pad = nsf_padded(q.k, FMT);
  const float g = FMT == FP4_FMT_NVFP4 ? *q.tensor_scale : 0.0f;
  float acc[B];
#pragma unroll
  for (int j = 0; j < B; ++j) acc[j] = 0.0f;
  if (live) {
#pragma unroll 2
    for (int64_t r = blockIdx.y * (int64_t)blockDim.y + threadIdx.y; r < q.rows; r += (int64_t)gridDim.y * blockDim.y) {
      const uint32_t sb = q.scales[sf_offset(q.sf_layout, r, cb, nsf_row, nsf_pad)];
      const float s = FMT == FP4_FMT_MXFP4 ? e8m0_scale(sb) : e4m3_decode(sb);
      float v[B];
#pragma unroll
      for (int h = 0; h < B / 8; ++h) load8<FP4_DTYPE_BF16>(x, r * ldx + cb * B + 8 * h, v + 8 * h);
      // the block's B/2 code bytes in one 8- or 16-byte load
      uint32_t cw[B / 8];
      const uint8_t* cp = q.codes + r * (q.k >> 1) + cb * (B / 2);
      if constexpr (B == 16) {
        const uint2 u = *reinterpret_cast<const uint2*>(cp);
        cw[0] = u.x;
        cw[1] = u.y;
      } else {
        const uint4 u = *reinterpret_cast<const uint4*>(cp);
        cw[0] = u.x;
        cw[1] = u.y;
        cw[2] = u.z;
        cw[3] = u.w;
      }
      // x_hat of two elements from each code byte: the signed E2M1 values by
      // the hardware decode, times the block scale (and g)
#pragma unroll
      for (int j2 = 0; j2 < B / 2; ++j2) {
        float h0, h1;
        e2m1x2_decode(cw[j2 >> 2] >> (8 * (j2 & 3)), h0, h1);
        h0 = __fmul_rn(h0, s);
        h1 = __fmul_rn(h1, s);
        if (FMT == FP4_FMT_NVFP4) {
          h0 = __fmul_rn(h0, g);
          h1 = __fmul_rn(h1, g);
        }
        const float d0 = __fsub_rn(v[2 * j2], h0), d1 = __fsub_rn(v[2 * j2 + 1], h1);
        acc[2 * j2] = __fmaf_rn(d0, d0, acc[2 * j2]);
        acc[2 * j2 + 1] = __fmaf_rn(d1, d1, acc[2 * j2 + 1]);
      }
    }
  }
  // the row groups' sums, channel by channel, then one atomic add per channel
  const int t = threadIdx.y * blockDim.x + threadIdx.x;
#pragma unroll
  for (int j = 0; j < B; ++j) {
    part[t] = acc[j];
    __syncthreads();
    if (threadIdx.y == 0 && live) {
      float sum = part[threadIdx.x];
      for (int y = 1; y < (int)blockDim.y; ++y) sum += part[y * blockDim.x + threadIdx.x];
      atomicAdd(&err[cb * B + j], sum);
    }
    __syncthreads();
  }
}

// rank[c] += the number of channels j in this CTA's slice of 256 that beat c
// (larger error, or equal error and lower index); rank is zeroed first.  The
// grid covers (channels / 256)^2 tiles, so the k^2 comparisons spread over the
// whole GPU.
constexpr int kRankSlice = 256;
__global__ void __launch_bounds__(256) rank_kernel(const float* __restrict__ err, int64_t k, int* rank) {
  __shared__ float chunk[kRankSlice];
  const int64_t c = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  const int64_t base = blockIdx.y * (int64_t)kRankSlice;
  for (int i = threadIdx.x; i < kRankSlice; i += blockDim.x) chunk[i] = base + i < k ? err[base + i] : -1.0f;
  __syncthreads();
  if (c >= k) return;
  const float e = err[c];
  const int n = (int)min((int64_t)kRankSlice, k - base);
  int r = 0;
  if (base + n <= c) {            // every j of the slice has a lower index
    for (int i = 0; i < n; ++i) r += chunk[i] >= e;
  } else if (base > c) {          // every j has a higher index
    for (int i = 0; i < n; ++i) r += chunk[i] > e;
  } else {
    for (int i = 0; i < n; ++i) {
      const float o = chunk[i];
      r += (o > e) || (o == e && base + i < c);
    }
  }
  if (r) atomicAdd(&rank[c], r);
}

// hot_idx = ascending list of the channels with rank < k_hot (one CTA,
// block-wide scan)
__global__ void __launch_bounds__(1024) compact_kernel(const int* __restrict__ rank, int64_t k, int k_hot,
                                                       int32_t* hot_idx) {
  __shared__ int warp_sums[32];
  __shared__ int carry;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  for (int64_t base = 0; base < k; base += blockDim.x) {
    const int64_t c = base + threadIdx.x;
    int f = c < k ? (rank[c] < k_hot ? 1 : 0) : 0;
    int x = f;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[w] = x;
    __syncthreads();
    if (w == 0) {
      int s = lane < (int)(blockDim.x >> 5) ? warp_sums[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xFFFFFFFFu, s, o);
        if (lane >= o) s += y;
      }
      warp_sums[lane] = s;
    }
    __syncthreads();
    int excl = carry + (w ? warp_sums[w - 1] : 0) + x - f;
    if (f) hot_idx[excl] = (int32_t)c;
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) carry = excl + f;
    __syncthreads();
  }
}

// Extra K columns.  One thread per output element (row, j), j in [0, kx).
template <int FMT>
__global__ void __launch_bounds__(256) gather_kernel(const uint16_t* __restrict__ src, int64_t ld, fp4_operand q,
                                                     const int32_t* __restrict__ hot, int k_hot, int order, int64_t kx,
                                                     bool is_a, const float* ts_other, uint16_t* __restrict__ out) {
  constexpr int B = FMT == FP4_FMT_MXFP4 ? 32 : 16;
  const int64_t nsf_row = q.k / B, nsf_pad = nsf_padded(q.k, FMT);
  const float g = FMT == FP4_FMT_NVFP4 ? *q.tensor_scale : 0.0f;
  // B columns are divided by alpha = fp32(gX * gW): inv_alpha = fp32(1 / alpha)
  const float inv_alpha = (FMT == FP4_FMT_NVFP4 && !is_a) ? __frcp_rn(__fmul_rn(*ts_other, g)) : 1.0f;
  const int64_t total = q.rows * kx;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / kx, j = i - r * kx;
    float v = 0.0f;
    const int nterm = order == 2 ? 2 : 1;
    if (j < (int64_t)nterm * k_hot) {
      const int part = (int)(j / k_hot);            // 0: first half, 1: second half
      const int64_t c = hot[j - (int64_t)part * k_hot];
      const float x = bf16_bits_to_float(src[r * ld + c]);
      // which term this column holds
      //   A, order 2: part 0 -> x - x_hat, part 1 -> x ;  A, order 1: x
      //   B, order 2: part 0 -> x_hat/alpha, part 1 -> (x - x_hat)/alpha ;  B, order 1: (x - x_hat)/alpha
      bool want_delta, want_hat;
      if (is_a) {
        want_delta = order == 2 && part == 0;
        want_hat = false;
      } else {
        want_hat = order == 2 && part == 0;
        want_delta = !want_hat && order != 0;   // order 0 (hot channels zeroed): w / alpha
      }
      if (want_delta || want_hat) {
        const float xh = dequant_elem<FMT>(q, r, c, g, nsf_row, nsf_pad);
        v = want_hat ? xh : __fsub_rn(x, xh);
      } else {
        v = x;
      }
      if (!is_a) v = __fmul_rn(v, inv_alpha);
    }
    __nv_bfloat16 h = __float2bfloat16_rn(v);
    out[i] = *reinterpret_cast<uint16_t*>(&h);
  }
}

// E4M3 extra columns: one warp per row of A_ext (rows < M) or B_ext.  The
// row's values are those of the bf16 tail without 1/alpha (order 2: [dX | X]
// and [W_hat | dW]; order 1: X and dW; order 0: X and W); the row gets
// s = amax / 448 and the E4M3 bytes of v / s (nearest, ties to even,
// saturating, sign kept), zero-padded to kx; all-zero rows get s = 0.
template <int FMT>
__global__ void __launch_bounds__(256) gather_fp8_kernel(const uint16_t* __restrict__ x, int64_t ldx,
                                                         const uint16_t* __restrict__ w, int64_t ldw, fp4_operand xq,
                                                         fp4_operand wq, const int32_t* __restrict__ hot, int k_hot,
                                                         int order, int64_t kx, uint8_t* a8, uint8_t* b8, float* sa,
                                                         float* sb) {
  constexpr int B = FMT == FP4_FMT_MXFP4 ? 32 : 16;
  const int64_t nsf_row = xq.k / B, nsf_pad = nsf_padded(xq.k, FMT);
  const float gx = FMT == FP4_FMT_NVFP4 ? *xq.tensor_scale : 0.0f;
  const float gw = FMT == FP4_FMT_NVFP4 ? *wq.tensor_scale : 0.0f;
  const int lane = threadIdx.x & 31;
  const int ncols = (order == 2 ? 2 : 1) * k_hot;
  const int64_t rows = xq.rows + wq.rows;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t row = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5; row < rows; row += nwarps) {
    const bool is_a = row < xq.rows;
    const int64_t r = is_a ? row : row - xq.rows;
    auto value = [&](int j) -> float {
      const int part = j >= k_hot ? 1 : 0;
      const int64_t c = hot[j - part * k_hot];
      if (is_a) {
        const float xv = bf16_bits_to_float(x[r * ldx + c]);
        if (order == 2 && part == 0) return __fsub_rn(xv, dequant_elem<FMT>(xq, r, c, gx, nsf_row, nsf_pad));
        return xv;
      }
      const float wv = bf16_bits_to_float(w[r * ldw + c]);
      if (order == 0) return wv;
      const float wh = dequant_elem<FMT>(wq, r, c, gw, nsf_row, nsf_pad);
      if (order == 2 && part == 0) return wh;
      return __fsub_rn(wv, wh);
    };
    float amax = 0.0f;
    for (int j = lane; j < ncols; j += 32) amax = fmaxf(amax, fabsf(value(j)));
    amax = warp_max(amax);
    const float sc = __fdiv_rn(amax, 448.0f);
    uint8_t* dst = (is_a ? a8 : b8) + r * kx;
    for (int64_t j0 = 0; j0 < kx; j0 += 128) {
      uint32_t word = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = (int)(j0 + 4 * lane + e);
        uint32_t byte = 0;
        if (j < ncols && sc > 0.0f) {
          const float v = value(j);
          byte = e4m3_rn_satfinite(__fdiv_rn(fabsf(v), sc)) | (signbit(v) ? 0x80u : 0u);
        }
        word |= byte << (8 * e);
      }
      *reinterpret_cast<uint32_t*>(dst + j0 + 4 * lane) = word;
    }
    if (lane == 0) (is_a ? sa : sb)[r] = sc;
  }
}

// MXFP8 extra columns for the single-kernel tail: one warp per (row, 32-column
// block) of A_ext or B_ext, rows padded to a multiple of 128 (padding rows get
// scale bytes 0 and no codes).  The values are gather_kernel's (B divided by
// alpha), each part padded with zeros to kp = 32 * ceil(k_hot / 32) columns and
// the whole to kxm; a block's E8M0 exponent is the smallest e with
// amax / 2^e <= 448 (E4M3's largest value), clamped to [-127, 127] (amax 0:
// -127), and each element the E4M3 byte of |v| * 2^-e (one fp32 rounding, then
// nearest, ties to even) with v's sign in bit 7.  Scales in the MMA layout.
template <int FMT>
__global__ void __launch_bounds__(256) gather_mx8_kernel(const uint16_t* __restrict__ src, int64_t ld, fp4_operand q,
                                                         const int32_t* __restrict__ hot, int k_hot, int order,
                                                         int64_t kxm, bool is_a, const float* ts_other,
                                                         uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
  constexpr int B = FMT == FP4_FMT_MXFP4 ? 32 : 16;
  const int64_t nsf_row = q.k / B, nsf_pad = nsf_padded(q.k, FMT);
  const float g = FMT == FP4_FMT_NVFP4 ? *q.tensor_scale : 0.0f;
  const float inv_alpha = (FMT == FP4_FMT_NVFP4 && !is_a) ? __frcp_rn(__fmul_rn(*ts_other, g)) : 1.0f;
  const int lane = threadIdx.x & 31;
  const int64_t nblk = kxm / 32, kp = cdiv(k_hot, 32) * 32;
  const int parts = order == 2 ? 2 : 1;
  const int64_t units = cdiv(q.rows, 128) * 128 * nblk;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t u = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5; u < units; u += nwarps) {
    const int64_t r = u / nblk, jb = u - r * nblk;
    const int64_t col = jb * 32 + lane;
    const int part = (int)(col / kp);
    const int64_t idx = col - (int64_t)part * kp;
    float v = 0.0f;
    if (r < q.rows && part < parts && idx < k_hot) {
      const int64_t c = hot[idx];
      const float x = bf16_bits_to_float(src[r * ld + c]);
      // A, order 2: part 0 -> x - x_hat, part 1 -> x ;  A, orders 1 and 0: x
      // B, order 2: part 0 -> x_hat, part 1 -> x - x_hat ;  B, order 1: x - x_hat ;  B, order 0: x  (all / alpha)
      const bool want_hat = !is_a && order == 2 && part == 0;
      const bool want_delta = is_a ? (order == 2 && part == 0) : (!want_hat && order != 0);
      if (want_delta || want_hat) {
        const float xh = dequant_elem<FMT>(q, r, c, g, nsf_row, nsf_pad);
        v = want_hat ? xh : __fsub_rn(x, xh);
      } else {
        v = x;
      }
      if (!is_a) v = __fmul_rn(v, inv_alpha);
    }
    float m = fabsf(v);
#pragma unroll
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    // amax = 1.f * 2^(E - 127) = (1.f / 2) * 2^(E - 126): e = E - 126 - 9, + 1 when 1.f > 1.75
    const uint32_t bits = __float_as_uint(m);
    int e = (int)(bits >> 23) - 135 + ((bits & 0x7FFFFFu) > 0x600000u ? 1 : 0);
    e = max(-127, min(127, e));
    if (lane == 0)
      scales[((r >> 7) * (nblk >> 2) + (jb >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (jb & 3)] =
          (uint8_t)(e + 127);
    if (r < q.rows) {
      const float t = __fmul_rn(fabsf(v), __uint_as_float((uint32_t)(127 - e) << 23));   // |v| * 2^-e
      codes[r * kxm + col] = (uint8_t)(e4m3_rn_satfinite(t) | (signbit(v) ? 0x80u : 0u));
    }
  }
}

// 16- and 4-byte global -> shared copies (cp.async) and their completion
__device__ __forceinline__ void cpa16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cpa4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cpa_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cpa_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// gather_mx8_kernel with each row staged first: a warp copies its row's bf16
// values (and, where x_hat is used - A at order 2, B at orders 1 and 2 - its FP4
// codes and block scales) into shared memory with 16-byte cp.async copies (with ~9% of the channels hot, nearly
// every 32-byte sector of the row is needed, and the per-block warps of the
// kernel above fetched each hot value, code and scale on its own), then each
// lane forms one whole 32-column block of the row from shared memory (no
// shuffles).  Each warp has two row buffers: the copies of its next row are in
// flight while it forms the current one, so the loads are never waited for
// one at a time.  The hot list is kept in the CTA's shared memory transposed,
// ht[i][b] = channel of column 32 b + i, so that the lanes of a warp read
// consecutive words.  Same bytes as gather_mx8_kernel.  (Lane = element of a
// block with a warp reduction for the block amax measured slower: the lanes'
// byte stores and the reductions' latency outweigh the shared reads it saves.)
// The same staging serves the bf16 extra columns (MX8 = false): there each
// lane forms 8 consecutive columns of the row (one 16-byte store), the values
// of gather_kernel.
//   kx: the row width of the output (MXFP8: kxm, bf16: kx)
//   buf_bytes: one row buffer (16-byte multiple): 2K (+ K/2 + the padded
//   scale count when order != 0); shared memory = the hot list (32 kpb words)
//   + 2 buffers a warp
template <int FMT, bool MX8>
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint16_t* __restrict__ src, int64_t ld, fp4_operand q,
                                                          const int32_t* __restrict__ hot, int k_hot, int order,
                                                          int64_t kx, bool is_a, const float* ts_other,
                                                          int64_t buf_bytes, void* __restrict__ out,
                                                          uint8_t* __restrict__ scales) {
  constexpr int B = FMT == FP4_FMT_MXFP4 ? 32 : 16;
  extern __shared__ __align__(16) uint8_t row_smem[];
  const int64_t K = q.k, nsf_row = K / B, nsf_pad = nsf_padded(K, FMT);
  const float g = FMT == FP4_FMT_NVFP4 ? *q.tensor_scale : 0.0f;
  const float inv_alpha = (FMT == FP4_FMT_NVFP4 && !is_a) ? __frcp_rn(__fmul_rn(*ts_other, g)) : 1.0f;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  // 32-bit block arithmetic: a part's columns kp = 32 kpb; blocks beyond the parts are padding
  const int nblk = (int)(kx / 32), kpb = (int)cdiv(k_hot, 32), parts = order == 2 ? 2 : 1;
  const bool need_q = is_a ? order == 2 : order != 0;                 // x_hat is used
  // MX8: [32][kpb], -1 past k_hot; bf16: the list as given
  int32_t* ht = reinterpret_cast<int32_t*>(row_smem);
  uint8_t* wbase = row_smem + cdiv((int64_t)32 * kpb * 4, 16) * 16 + (int64_t)warp * 2 * buf_bytes;
  for (int t = threadIdx.x; t < 32 * kpb; t += blockDim.x) {
    const int b = t / 32, i = t - b * 32;                              // column 32 b + i of a part
    if (MX8) ht[i * kpb + b] = t < k_hot ? hot[t] : -1;
    else ht[t] = t < k_hot ? hot[t] : -1;
  }
  __syncthreads();
  // row r into buffer `buf` (a commit group of its own, empty past the rows)
  auto stage = [&](int64_t r, uint8_t* buf) {
    if (r < q.rows) {
      const uint16_t* xr = src + r * ld;
      for (int64_t c = 8 * lane; c < K; c += 256) cpa16(buf + 2 * c, xr + c);
      if (need_q) {
        const uint8_t* cr = q.codes + r * (K >> 1);
        for (int64_t c = 16 * lane; c < (K >> 1); c += 512) cpa16(buf + 2 * K + c, cr + c);
        // four consecutive scales at a time (one 32-bit word in the MMA layout)
        for (int64_t j = 4 * lane; j < nsf_pad; j += 128)
          cpa4(buf + 2 * K + (K >> 1) + j, q.scales + sf_offset(FP4_SF_MMA, r, j, nsf_row, nsf_pad));
      }
    }
    cpa_commit();
  };
  // MX8: the scales of the rows up to the next multiple of 128 are written too
  const int64_t rows_end = MX8 ? cdiv(q.rows, 128) * 128 : q.rows, rstep = (int64_t)gridDim.x * nw;
  int64_t r = (int64_t)blockIdx.x * nw + warp;
  stage(r, wbase);
  for (int pb = 0; r < rows_end; r += rstep, pb ^= 1) {
    stage(r + rstep, wbase + (pb ^ 1) * buf_bytes);                    // the next row streams in
    cpa_wait<1>();                                                     // this lane's copies of row r
    __syncwarp();                                                      // ... and every lane's
    const uint8_t* buf = wbase + pb * buf_bytes;
    const uint16_t* xs = reinterpret_cast<const uint16_t*>(buf);
    const uint8_t* cs = buf + 2 * K;
    const uint8_t* ss = cs + (K >> 1);
    const bool real = r < q.rows;
    if constexpr (MX8) {
      for (int jb = lane; jb < nblk; jb += 32) {
        const int part = jb >= kpb ? 1 : 0;
        const int b = jb - part * kpb;                                   // block within the part
        // A, order 2: x - x_hat | x;  A, orders 1, 0: x;
        // B, order 2: x_hat | x - x_hat;  B, order 1: x - x_hat;  B, order 0: x  (B / alpha)
        const bool want_hat = !is_a && order == 2 && part == 0;
        const bool want_delta = is_a ? (order == 2 && part == 0) : (!want_hat && order != 0);
        const bool live = real && jb < parts * kpb;
        // branch-free per element (the two parts' lanes take different forms,
        // and a branch per element would run them one after the other): every
        // lane reads a valid column (0 for padding), forms x and, where x_hat is
        // used, x_hat (the signed E2M1 value by the hardware decode, times the
        // block scale), then selects
        float v[32];
        float m = 0.0f;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int c = live ? ht[i * kpb + b] : -1;
          const int cc = max(c, 0);
          float x = bf16_bits_to_float(xs[cc]);
          if (need_q) {
            float xh, unused;
            e2m1x2_decode((uint32_t)cs[cc >> 1] >> ((cc & 1) << 2), xh, unused);
            const uint32_t sb = ss[cc / B];
            xh = FMT == FP4_FMT_MXFP4 ? __fmul_rn(xh, e8m0_scale(sb)) : __fmul_rn(__fmul_rn(xh, e4m3_decode(sb)), g);
            x = want_hat ? xh : want_delta ? __fsub_rn(x, xh) : x;
          }
          if (!is_a) x = __fmul_rn(x, inv_alpha);
          x = c >= 0 ? x : 0.0f;
          v[i] = x;
          m = fmaxf(m, fabsf(x));
        }
        const uint32_t bits = __float_as_uint(m);
        int e = (int)(bits >> 23) - 135 + ((bits & 0x7FFFFFu) > 0x600000u ? 1 : 0);
        e = max(-127, min(127, e));
        scales[((r >> 7) * (nblk >> 2) + (jb >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (jb & 3)] =
            (uint8_t)(e + 127);
        if (real) {
          const float inv = __uint_as_float((uint32_t)(127 - e) << 23);     // 2^-e
          uint32_t w[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            // the signed conversion: RN is symmetric, so each byte is the code
            // of |x| 2^-e with x's sign bit (-0 included)
            const uint32_t lo = e4m3x2_rn_satfinite(__fmul_rn(v[4 * k], inv), __fmul_rn(v[4 * k + 1], inv));
            const uint32_t hi = e4m3x2_rn_satfinite(__fmul_rn(v[4 * k + 2], inv), __fmul_rn(v[4 * k + 3], inv));
            w[k] = lo | (hi << 16);
          }
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(out) + r * kx + (int64_t)jb * 32);
          dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
          dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
        }
      }
    } else {
      // bf16 columns j0 .. j0 + 7 of the row (parts of k_hot columns, no padding
      // between them; zeros past them), branch-free like the blocks above
      const int live_cols = parts * k_hot;
      uint16_t* orow = static_cast<uint16_t*>(out) + r * kx;
      for (int j0 = 8 * lane; j0 < kx; j0 += 256) {
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int j = j0 + e;
          const int part = j >= k_hot ? 1 : 0;
          const bool live = j < live_cols;
          const int c = live ? ht[j - part * k_hot] : -1;
          const int cc = max(c, 0);
          float x = bf16_bits_to_float(xs[cc]);
          if (need_q) {
            float xh, unused;
            e2m1x2_decode((uint32_t)cs[cc >> 1] >> ((cc & 1) << 2), xh, unused);
            const uint32_t sb = ss[cc / B];
            xh = FMT == FP4_FMT_MXFP4 ? __fmul_rn(xh, e8m0_scale(sb)) : __fmul_rn(__fmul_rn(xh, e4m3_decode(sb)), g);
            const bool want_hat = !is_a && order == 2 && part == 0;
            const bool want_delta = is_a ? (order == 2 && part == 0) : (!want_hat && order != 0);
            x = want_hat ? xh : want_delta ? __fsub_rn(x, xh) : x;
          }
          if (!is_a) x = __fmul_rn(x, inv_alpha);
          v[e] = c >= 0 ? x : 0.0f;
        }
        uint32_t pk[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const __nv_bfloat162 h2 = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
          pk[k] = *reinterpret_cast<const uint32_t*>(&h2);
        }
        *reinterpret_cast<uint4*>(orow + j0) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
    }
    __syncwarp();   // every lane is done with this buffer before it is refilled
  }
  cpa_wait<0>();
}

}  // namespace

cudaError_t launch_hcp_gather_fp8(const uint16_t* x, int64_t ldx, const uint16_t* w, int64_t ldw,
                                  const fp4_operand& xq, const fp4_operand& wq, const int32_t* hot, int k_hot,
                                  int order, int64_t kx, uint8_t* a8, uint8_t* b8, float* sa, float* sb, int num_sms,
                                  cudaStream_t st) {
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(cdiv((xq.rows + wq.rows) * 32, 256),
                                                               (int64_t)num_sms * 8));
  if (xq.format == FP4_FMT_MXFP4)
    gather_fp8_kernel<FP4_FMT_MXFP4><<<grid, 256, 0, st>>>(x, ldx, w, ldw, xq, wq, hot, k_hot, order, kx, a8, b8, sa, sb);
  else
    gather_fp8_kernel<FP4_FMT_NVFP4><<<grid, 256, 0, st>>>(x, ldx, w, ldw, xq, wq, hot, k_hot, order, kx, a8, b8, sa, sb);
  return cudaGetLastError();
}

cudaError_t launch_hcp_channel_errors(const uint16_t* x, int64_t ldx, const fp4_operand& q, float* err, int num_sms,
                                      cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(err, 0, sizeof(float) * q.k, st);
  if (e != cudaSuccess || q.rows == 0 || q.k == 0) return e;
  const int B = q.format == FP4_FMT_MXFP4 ? 32 : 16;
  const int64_t nblk = q.k / B;
  // 512 threads: up to 256 channel blocks x the rest as row groups
  const int bx = (int)std::min<int64_t>(256, cdiv(nblk, 32) * 32), by = 512 / bx;
  dim3 block((unsigned)bx, (unsigned)by);
  dim3 grid((unsigned)cdiv(nblk, bx), 1);
  const int64_t want_y = cdiv((int64_t)num_sms * 2, grid.x);   // two CTAs an SM
  grid.y = (unsigned)std::max<int64_t>(1, std::min<int64_t>(want_y, cdiv(q.rows, by)));
  if (q.format == FP4_FMT_MXFP4)
    channel_err_kernel<FP4_FMT_MXFP4><<<grid, block, 0, st>>>(x, ldx, q, err);
  else
    channel_err_kernel<FP4_FMT_NVFP4><<<grid, block, 0, st>>>(x, ldx, q, err);
  return cudaGetLastError();
}

cudaError_t launch_hcp_topk(const float* err, int64_t k, int k_hot, int32_t* hot_idx, cudaStream_t st) {
  if (k == 0 || k_hot == 0) return cudaSuccess;
  int* rank = reinterpret_cast<int*>(const_cast<float*>(err) + k);
  cudaError_t e = cudaMemsetAsync(rank, 0, sizeof(int) * k, st);
  if (e != cudaSuccess) return e;
  rank_kernel<<<dim3((unsigned)cdiv(k, 256), (unsigned)cdiv(k, kRankSlice)), 256, 0, st>>>(err, k, rank);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  compact_kernel<<<1, 1024, 0, st>>>(rank, k, k_hot, hot_idx);
  return cudaGetLastError();
}

// Launch the staged-row gather (MX8: MXFP8 codes + scales; else bf16 columns)
// for A (X's rows) and B (W's rows); false when a row's two buffers do not fit
template <bool MX8>
bool launch_gather_rows(const uint16_t* x, int64_t ldx, const uint16_t* w, int64_t ldw, const fp4_operand& xq,
                        const fp4_operand& wq, const int32_t* hot, int k_hot, int order, int64_t kx, void* a_out,
                        uint8_t* sa, void* b_out, uint8_t* sb, int num_sms, cudaStream_t st, cudaError_t* err) {
  // two buffers a warp (bf16 values; codes and scales for orders 1 and 2:
  // ~10 K bytes a buffer at K = 4096), while at least one warp's buffers and
  // the hot list fit in 100 KB (two CTAs an SM)
  const int64_t buf_bytes =
      cdiv(xq.k * 2 + (order != 0 ? xq.k / 2 + nsf_padded(xq.k, xq.format) : 0), 16) * 16;
  const int64_t hot_bytes = cdiv((int64_t)32 * cdiv(k_hot, 32) * 4, 16) * 16;
  const int warps = (int)std::min<int64_t>(8, ((int64_t)(100 * 1024) - hot_bytes) / (2 * buf_bytes));
  if (warps < 1) return false;
  const int smem = (int)(hot_bytes + warps * 2 * buf_bytes);
  auto grid_rows = [&](int64_t rows) {
    const int64_t rows_end = MX8 ? cdiv(rows, 128) * 128 : rows;
    return (int)std::max<int64_t>(1, std::min<int64_t>(cdiv(rows_end, warps), (int64_t)num_sms * 2));
  };
  auto run = [&](auto kernel) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (xq.rows > 0)
      kernel<<<grid_rows(xq.rows), 32 * warps, smem, st>>>(x, ldx, xq, hot, k_hot, order, kx, true, nullptr,
                                                           buf_bytes, a_out, sa);
    if (wq.rows > 0)
      kernel<<<grid_rows(wq.rows), 32 * warps, smem, st>>>(w, ldw, wq, hot, k_hot, order, kx, false,
                                                           xq.tensor_scale, buf_bytes, b_out, sb);
    return cudaGetLastError();
  };
  *err = xq.format == FP4_FMT_MXFP4 ? run(gather_rows_kernel<FP4_FMT_MXFP4, MX8>)
                                    : run(gather_rows_kernel<FP4_FMT_NVFP4, MX8>);
  return true;
}

cudaError_t launch_hcp_gather_mx8(const uint16_t* x, int64_t ldx, const uint16_t* w, int64_t ldw,
                                  const fp4_operand& xq, const fp4_operand& wq, const int32_t* hot, int k_hot,
                                  int order, int64_t kxm, uint8_t* a8, uint8_t* sa, uint8_t* b8, uint8_t* sb,
                                  int num_sms, cudaStream_t st) {
  // rows staged in shared memory; wider rows read the hot values directly
  cudaError_t e = cudaSuccess;
  if (launch_gather_rows<true>(x, ldx, w, ldw, xq, wq, hot, k_hot, order, kxm, a8, sa, b8, sb, num_sms, st, &e))
    return e;
  auto grid = [&](int64_t rows) {
    return (int)std::max<int64_t>(1, std::min<int64_t>(cdiv(cdiv(rows, 128) * 128 * (kxm / 32) * 32, 256),
                                                        (int64_t)num_sms * 8));
  };
  if (xq.format == FP4_FMT_MXFP4) {
    gather_mx8_kernel<FP4_FMT_MXFP4><<<grid(xq.rows), 256, 0, st>>>(x, ldx, xq, hot, k_hot, order, kxm, true, nullptr,
                                                                    a8, sa);
    gather_mx8_kernel<FP4_FMT_MXFP4><<<grid(wq.rows), 256, 0, st>>>(w, ldw, wq, hot, k_hot, order, kxm, false, nullptr,
                                                                    b8, sb);
  } else {
    gather_mx8_kernel<FP4_FMT_NVFP4><<<grid(xq.rows), 256, 0, st>>>(x, ldx, xq, hot, k_hot, order, kxm, true, nullptr,
                                                                    a8, sa);
    gather_mx8_kernel<FP4_FMT_NVFP4><<<grid(wq.rows), 256, 0, st>>>(w, ldw, wq, hot, k_hot, order, kxm, false,
                                                                    xq.tensor_scale, b8, sb);
  }
  return cudaGetLastError();
}

cudaError_t launch_hcp_gather(const uint16_t* x, int64_t ldx, const uint16_t* w, int64_t ldw, const fp4_operand& xq,
                              const fp4_operand& wq, const int32_t* hot, int k_hot, int order, int64_t kx,
                              uint16_t* a_ext, uint16_t* b_ext, int num_sms, cudaStream_t st) {
  // rows staged in shared memory; wider rows: one thread per output element
  cudaError_t e = cudaSuccess;
  if (launch_gather_rows<false>(x, ldx, w, ldw, xq, wq, hot, k_hot, order, kx, a_ext, nullptr, b_ext, nullptr,
                                num_sms, st, &e))
    return e;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(cdiv(xq.rows * kx, 256), (int64_t)num_sms * 8));
  const int gridb = (int)std::max<int64_t>(1, std::min<int64_t>(cdiv(wq.rows * kx, 256), (int64_t)num_sms * 8));
  if (xq.format == FP4_FMT_MXFP4) {
    gather_kernel<FP4_FMT_MXFP4><<<grid, 256, 0, st>>>(x, ldx, xq, hot, k_hot, order, kx, true, nullptr, a_ext);
    gather_kernel<FP4_FMT_MXFP4><<<gridb, 256, 0, st>>>(w, ldw, wq, hot, k_hot, order, kx, false, nullptr, b_ext);
  } else {
    gather_kernel<FP4_FMT_NVFP4><<<grid, 256, 0, st>>>(x, ldx, xq, hot, k_hot, order, kx, true, nullptr, a_ext);
    gather_kernel<FP4_FMT_NVFP4><<<gridb, 256, 0, st>>>(w, ldw, wq, hot, k_hot, order, kx, false, xq.tensor_scale, b_ext);
  }
  return cudaGetLastError();
}

}  // namespace fp4

// ============================================================================
// fp4_hcp_select_noalloc: selection with a fixed scratch array in the library
// (no context, no workspace, no allocation).  For callers that may not allocate
// device memory: their memory belongs to their own caching pool, or they cannot
// afford the synchronization that cudaMalloc/cudaFree may bring.
// ============================================================================
namespace fp4 {
namespace {

// per-channel fp32 error sums, then one int flag per channel
static __device__ __align__(256) unsigned char g_hcp_select_scratch[FP4_NOALLOC_MAX_CHANNELS * 8];

// Device address of the scratch array on the current device (host code may not
// use the array's name as a device pointer), looked up on every call: after a
// device reset the module may be loaded again at another address.
int noalloc_scratch(void** ptr, int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FP4_ERR_CUDA;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_hcp_select_scratch) != cudaSuccess || !p) return FP4_ERR_CUDA;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  *ptr = p;
  *sms = n;
  return FP4_OK;
}

}  // namespace
}  // namespace fp4

extern "C" int fp4_hcp_select_noalloc(const void* x_bf16, int64_t ldx, const fp4_operand* xq, int32_t k_hot,
                                      int32_t* hot_idx, void* stream) {
  using namespace fp4;
  int s = validate_hcp_select(x_bf16, ldx, xq, k_hot, hot_idx);
  if (s) return s;
  if (xq->k > FP4_NOALLOC_MAX_CHANNELS) return FP4_ERR_TOO_LARGE;
  if (k_hot == 0 || xq->k == 0) return FP4_OK;   // as fp4_hcp_select: rows == 0 still selects (all errors 0)
  void* scratch = nullptr;
  int sms = 0;
  s = noalloc_scratch(&scratch, &sms);
  if (s) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  float* err = static_cast<float*>(scratch);   // cleared by the launcher before accumulating
  cudaError_t e = launch_hcp_channel_errors(static_cast<const uint16_t*>(x_bf16), ldx, *xq, err, sms, st);
  if (e == cudaSuccess) e = launch_hcp_topk(err, xq->k, k_hot, hot_idx, st);
  return e == cudaSuccess ? FP4_OK : FP4_ERR_CUDA;
}
