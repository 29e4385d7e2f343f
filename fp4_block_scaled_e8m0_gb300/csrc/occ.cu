// Outlier clamping and compensation, OCC ([msr] §三, §六).
//
//   tau  = the ceil(q n)-th smallest |x| over the tensor (nearest rank)
//   X_c  = clamp(X, -tau, tau)            quantized by the row quantizer
//   dX   = X - X_c                        sparse: nonzero where |x| > tau
//   Y    = alpha Q(X_c) Q(W)^T + dX W^T
//
// The threshold is an order statistic of the magnitudes, found exactly with
// integer work: a histogram of the magnitude bit patterns (bf16: all 15 bits,
// 32768 bins; fp32: the top 15 bits, then the low 16 bits of the elements in
// the selected bin) and a scan for the bin that holds the rank.
//
// dX W^T is split by column.  The k_dense columns with the most outliers (the
// persistent hot channels of [outlier] §2) become extra bf16 K columns of the
// FP4 GEMM, A_ext = dX_H / alpha and B_ext = W_H, so the tensor cores compute
// them with the FP4 part; the other outliers are gathered per row and the GEMM
// epilogue adds v * W^T[k, :] for each of them to its row of Y, in fp32 before
// the output is rounded (the GEMM's sparse-correction variant).
#include <cuda_bf16.h>

#include <algorithm>

#include "fp4_device.cuh"

using namespace fp4dev;

namespace fp4 {
namespace {

constexpr int kHistBins = 32768;   // 15-bit magnitude keys
constexpr int kLowBins = 65536;    // fp32: the low 16 bits
constexpr int kHistThreads = 1024;

struct OccSelect {
  unsigned long long below;   // elements in bins below the selected one
  unsigned long long in_bin;  // elements in the selected bin
  unsigned int bin;
  unsigned int pad;
};

template <int DT>
__device__ __forceinline__ uint32_t mag_bits_hi(float v) {
  // bf16 values are exact in fp32 with the low 16 bits zero: the top 15 bits
  // below the sign are the whole magnitude
  return (__float_as_uint(v) >> 16) & 0x7FFFu;
}

// Histogram of the top 15 magnitude bits: per-CTA shared-memory counters,
// merged into the global fine histogram (32768 bins) and a coarse one (256
// bins of 128: the exponent) once per CTA.  8 elements per vector.
template <int DT>
__global__ void __launch_bounds__(kHistThreads) occ_hist_kernel(const void* __restrict__ x, int64_t ldx,
                                                                FastDiv vec_per_row, uint32_t total_vecs,
                                                                unsigned long long* fine,
                                                                unsigned long long* coarse) {
  extern __shared__ uint32_t sh[];
  for (int b = threadIdx.x; b < kHistBins; b += blockDim.x) sh[b] = 0u;
  __syncthreads();
  for (uint32_t v = blockIdx.x * blockDim.x + threadIdx.x; v < total_vecs; v += gridDim.x * blockDim.x) {
    const uint32_t r = fast_div(v, vec_per_row), c = (v - r * vec_per_row.d) * 8u;
    float e[8];
    load8<DT>(x, (int64_t)r * ldx + c, e);
#pragma unroll
    for (int j = 0; j < 8; ++j) atomicAdd(&sh[mag_bits_hi<DT>(e[j])], 1u);
  }
  __syncthreads();
  // thread t owns fine bins 32t .. 32t+31, all inside coarse bin t / 4
  constexpr int PER = kHistBins / kHistThreads;
  uint32_t part = 0;
  for (int i = 0; i < PER; ++i) {
    const int b = threadIdx.x * PER + i;
    const uint32_t c = sh[b];
    if (c) atomicAdd(&fine[b], (unsigned long long)c);
    part += c;
  }
  part += __shfl_xor_sync(0xFFFFFFFFu, part, 1);
  part += __shfl_xor_sync(0xFFFFFFFFu, part, 2);
  if ((threadIdx.x & 3) == 0 && part) atomicAdd(&coarse[threadIdx.x >> 2], (unsigned long long)part);
}

// fp32 second pass: low 16 bits of the elements whose top bits are the
// selected bin (fine: 65536 bins, coarse: 256 bins of 256)
__global__ void __launch_bounds__(256) occ_hist_low_kernel(const float* __restrict__ x, int64_t ldx,
                                                           FastDiv vec_per_row, uint32_t total_vecs,
                                                           const OccSelect* sel, unsigned long long* fine,
                                                           unsigned long long* coarse) {
  const uint32_t bin = sel->bin;
  for (uint32_t v = blockIdx.x * blockDim.x + threadIdx.x; v < total_vecs; v += gridDim.x * blockDim.x) {
    const uint32_t r = fast_div(v, vec_per_row), c = (v - r * vec_per_row.d) * 8u;
    float e[8];
    load8<FP4_DTYPE_F32>(x, (int64_t)r * ldx + c, e);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t u = __float_as_uint(e[j]);
      if (((u >> 16) & 0x7FFFu) == bin) {
        atomicAdd(&fine[u & 0xFFFFu], 1ull);
        atomicAdd(&coarse[(u & 0xFFFFu) >> 8], 1ull);
      }
    }
  }
}

__device__ __forceinline__ unsigned long long warp_incl_scan(unsigned long long v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(0xFFFFFFFFu, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

// One warp finds the bin holding rank `target` among `nb` bins starting at
// `h` (nb a multiple of 32, each lane owning nb / 32 consecutive bins): the
// bin index and the count of the bins before it.
__device__ __forceinline__ void warp_find_bin(const unsigned long long* h, int nb, unsigned long long target,
                                              int& bin, unsigned long long& before) {
  const int lane = threadIdx.x & 31, per = nb / 32;
  unsigned long long local = 0;
  for (int i = 0; i < per; ++i) local += h[lane * per + i];
  const unsigned long long incl = warp_incl_scan(local), excl = incl - local;
  const bool mine = excl < target && target <= incl;
  const int owner = __ffs(__ballot_sync(0xFFFFFFFFu, mine)) - 1;
  int b = 0;
  unsigned long long cum = excl;
  if (mine) {
    for (; b < per; ++b) {
      const unsigned long long c = h[lane * per + b];
      if (cum + c >= target) break;
      cum += c;
    }
  }
  bin = __shfl_sync(0xFFFFFFFFu, lane * per + b, owner < 0 ? 0 : owner);
  before = __shfl_sync(0xFFFFFFFFu, cum, owner < 0 ? 0 : owner);
}

// One warp: coarse bin, then the fine bin inside it.  PASS 0 over the 15-bit
// keys (final for bf16), PASS 1 over the low 16 bits (fp32).
template <int PASS, int DT>
__global__ void __launch_bounds__(32) occ_select_kernel(const unsigned long long* __restrict__ fine,
                                                        const unsigned long long* __restrict__ coarse,
                                                        unsigned long long n, unsigned long long rank,
                                                        OccSelect* sel, float* tau, long long* n_out) {
  constexpr int FPC = PASS == 0 ? kHistBins / 256 : kLowBins / 256;   // fine bins per coarse bin
  const unsigned long long target = PASS == 0 ? rank : rank - sel->below;
  int cb, fb;
  unsigned long long before_c, before_f;
  warp_find_bin(coarse, 256, target, cb, before_c);
  warp_find_bin(fine + (int64_t)cb * FPC, FPC, target - before_c, fb, before_f);
  if (threadIdx.x != 0) return;
  const unsigned int bin = (unsigned int)(cb * FPC + fb);
  const unsigned long long cum = before_c + before_f, h = fine[bin];
  if constexpr (PASS == 0) {
    sel->bin = bin;
    sel->below = cum;
    sel->in_bin = h;
    if (DT == FP4_DTYPE_BF16) {
      *tau = __uint_as_float(bin << 16);
      *n_out = (long long)(n - cum - h);
    }
  } else {
    *tau = __uint_as_float((sel->bin << 16) | bin);
    *n_out = (long long)((n - sel->below - sel->in_bin) + (sel->in_bin - cum - h));
  }
}

// ---------------------------------------------------------------------------
// compensation
// ---------------------------------------------------------------------------
template <int DT>
__device__ __forceinline__ float load_elem(const void* x, int64_t i) {
  if constexpr (DT == FP4_DTYPE_BF16) {
    return bf16_bits_to_float(static_cast<const uint16_t*>(x)[i]);
  } else {
    return static_cast<const float*>(x)[i];
  }
}

// dX = x - clamp(x, -tau, tau): exact in fp32 for the values the method meets
__device__ __forceinline__ float clamp_residual(float v, float tau) {
  return fabsf(v) > tau ? __fsub_rn(v, copysignf(tau, v)) : 0.0f;
}

// 1 / alpha for the bf16 extra columns, or 0 when alpha cannot carry them
// (alpha zero, or 1 / alpha not finite): every outlier then takes the scattered
// path.  Both the column gather and the row extraction take this decision from
// the same device values.
template <int FMT>
__device__ __forceinline__ float tail_inv_alpha(const fp4_operand& xq, const fp4_operand& wq) {
  if constexpr (FMT == FP4_FMT_MXFP4) {
    return 1.0f;
  } else {
    const float alpha = __fmul_rn(*xq.tensor_scale, *wq.tensor_scale);
    const float r = __frcp_rn(alpha);
    return (alpha > 0.0f && isfinite(r)) ? r : 0.0f;
  }
}

// dX / alpha as the bf16 value of an extra column.  (An outlier so large that
// dX / alpha leaves the bf16 range gives an infinite column value: |x| / tau
// would have to exceed ~1e28 for weights of amax 1e-3.)
__device__ __forceinline__ uint16_t tail_bits(float dx, float inv_alpha) {
  const __nv_bfloat16 h = __float2bfloat16_rn(__fmul_rn(dx, inv_alpha));
  return *reinterpret_cast<const uint16_t*>(&h);
}

// dense[c / 32] bit c % 32 set for the k_dense chosen columns
__global__ void occ_flags_kernel(const int32_t* __restrict__ hot, int k_dense, uint32_t* dense) {
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j < k_dense) atomicOr(&dense[hot[j] >> 5], 1u << (hot[j] & 31));
}

// A_ext[m][j] = bf16(dX[m, H_j] / alpha) (0 where the outlier is scattered),
// B_ext[n][j] = W[n, H_j]; columns j >= k_dense are zero.  One thread per
// 8 consecutive columns of one row (16-byte stores).
template <int FMT, int XDT>
__global__ void __launch_bounds__(256) occ_tail_kernel(const void* __restrict__ x, int64_t ldx,
                                                       const uint16_t* __restrict__ w, int64_t ldw, fp4_operand xq,
                                                       fp4_operand wq, const float* __restrict__ tau_p,
                                                       const int32_t* __restrict__ hot, int k_dense, int64_t kx,
                                                       uint16_t* __restrict__ a_ext, uint16_t* __restrict__ b_ext) {
  const float tau = *tau_p;
  const float inv_alpha = tail_inv_alpha<FMT>(xq, wq);
  const int64_t per_row = kx / 8;
  const int64_t total = (xq.rows + wq.rows) * per_row;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = i / per_row, j0 = (i - row * per_row) * 8;
    const bool is_a = row < xq.rows;
    uint16_t o[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int64_t j = j0 + e;
      uint16_t bits = 0;
      if (j < k_dense && inv_alpha != 0.0f) {
        const int64_t c = hot[j];
        bits = is_a ? tail_bits(clamp_residual(load_elem<XDT>(x, row * ldx + c), tau), inv_alpha)
                    : w[(row - xq.rows) * ldw + c];
      }
      o[e] = bits;
    }
    uint4 pk;
    pk.x = o[0] | ((uint32_t)o[1] << 16);
    pk.y = o[2] | ((uint32_t)o[3] << 16);
    pk.z = o[4] | ((uint32_t)o[5] << 16);
    pk.w = o[6] | ((uint32_t)o[7] << 16);
    uint16_t* dst = is_a ? a_ext + row * kx + j0 : b_ext + (row - xq.rows) * kx + j0;
    *reinterpret_cast<uint4*>(dst) = pk;
  }
}

// W [N][K] (pitch ldw) -> WT [K][ldt], 64 x 64 tiles through shared memory:
// 16-byte reads along k (8 bf16 of one W row) and 16-byte writes along n (8 bf16
// of one W^T row, gathered from a tile column); W rows are 16-byte aligned,
// k % 32 == 0, ldt % 8 == 0.  The tile's 16-byte chunk q of row r sits at chunk
// q ^ (r / 8 % 8): the column reads of the write-out (8 rows 8 apart, a word
// each) then fall on distinct banks; with padded rows they all hit one bank.
__device__ __forceinline__ int tr_swz(int r, int c) { return ((((c >> 3) ^ (r >> 3)) & 7) << 3) | (c & 7); }
__global__ void __launch_bounds__(256) transpose_bf16_kernel(const uint16_t* __restrict__ w, int64_t ldw, int64_t n,
                                                             int64_t k, uint16_t* __restrict__ wt, int64_t ldt) {
  __shared__ __align__(16) uint16_t tile[64][64];
  const int64_t tiles_k = cdiv(k, 64), tiles = cdiv(n, 64) * tiles_k;
  const int t = threadIdx.x;
  for (int64_t tt = blockIdx.x; tt < tiles; tt += gridDim.x) {
    const int64_t n0 = (tt / tiles_k) * 64, k0 = (tt % tiles_k) * 64;
#pragma unroll
    for (int i = 0; i < 2; ++i) {                 // 512 chunks of 8: row r, k chunk kc
      const int idx = t + 256 * i, r = idx >> 3, kc = (idx & 7) * 8;
      const int64_t nn = n0 + r, kk = k0 + kc;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (nn < n && kk < k) v = __ldg(reinterpret_cast<const uint4*>(w + nn * ldw + kk));   // k % 8 == 0
      *reinterpret_cast<uint4*>(&tile[r][tr_swz(r, kc)]) = v;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 2; ++i) {                 // 512 chunks of 8: W^T row c (= k), n chunk nc
      const int idx = t + 256 * i, c = idx >> 3, nc = (idx & 7) * 8;
      const int64_t kk = k0 + c, nn = n0 + nc;
      if (kk < k && nn < n) {
        uint32_t q[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          q[j] = tile[nc + 2 * j][tr_swz(nc + 2 * j, c)] | ((uint32_t)tile[nc + 2 * j + 1][tr_swz(nc + 2 * j + 1, c)] << 16);
        if (nn + 8 <= n) {
          *reinterpret_cast<uint4*>(wt + kk * ldt + nn) = make_uint4(q[0], q[1], q[2], q[3]);
        } else {
          for (int j = 0; j < 8 && nn + j < n; ++j) wt[kk * ldt + nn + j] = (uint16_t)(q[j >> 1] >> (16 * (j & 1)));
        }
      }
    }
    __syncthreads();
  }
}

struct OccEntry {
  int32_t k;
  float v;
};

// L2 eviction-priority policies (createpolicy) and the loads / stores that
// carry them: the correction streams Y once (evict first) and re-reads the
// rows of W^T that its entries name (evict last), so that W^T stays in L2
// while Y passes through
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint4 ld_v4_hint(const void* ptr, uint64_t pol) {
  uint4 u;
  asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(u.x), "=r"(u.y), "=r"(u.z), "=r"(u.w) : "l"(ptr), "l"(pol));
  return u;
}
__device__ __forceinline__ void st_v4_hint(void* ptr, uint4 v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(ptr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w), "l"(pol)
               : "memory");
}

// The scattered outliers' product ([msr] §三: computed apart from the
// quantized GEMM and added back), after the GEMM stored Y:
//   Y[m, :] += sum over the entries (k, v) of row m of  v * W^T[k, :]
// in fp32 on the stored values, entry by entry in list order (bf16 Y is
// rounded again: the stored value was rounded once).  One thread per 16
// columns of a row, two groups of 8 that share the row's entries (16-byte
// reads of W^T, whose rows are zero-padded to a multiple of 8 columns), the
// threads of a row side by side; rows without entries are not touched.  On a
// 16384 x 4096 Y with 62 202 entries: 79 us; 8 columns a thread 110 us, 32
// columns (124 registers) 110 us, a warp per row passing over its columns
// (one 512-byte load of Y in flight per warp) 176 us.
template <bool BF16>
__global__ void __launch_bounds__(256) occ_correct_kernel(void* __restrict__ y, int64_t ldy, int64_t M, int64_t N,
                                                          FastDiv upr_div, const uint32_t* __restrict__ row_start,
                                                          const uint32_t* __restrict__ row_len,
                                                          const OccEntry* __restrict__ ent,
                                                          const uint16_t* __restrict__ wt, int64_t ldt) {
  constexpr int G = 2;                                 // 8-column groups a thread
  const uint32_t upr = upr_div.d;                      // 8G-column units per row
  const uint32_t total = (uint32_t)M * upr;
  const uint64_t keep = l2_policy_evict_last(), stream = l2_policy_evict_first();
  for (uint32_t u = blockIdx.x * blockDim.x + threadIdx.x; u < total; u += gridDim.x * blockDim.x) {
    const uint32_t m = fast_div(u, upr_div);
    const uint32_t len = row_len[m];
    if (len == 0) continue;
    const uint32_t s0 = row_start[m];
    const int64_t cu = (int64_t)(u - m * upr) * (8 * G);
    float acc[G][8];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const int64_t c = cu + 8 * g;
      const bool full = c + 8 <= N;
      if constexpr (BF16) {
        const uint16_t* yp = static_cast<const uint16_t*>(y) + (int64_t)m * ldy + c;
        if (full) {
          const uint4 q = ld_v4_hint(yp, stream);
          const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            acc[g][2 * k] = __uint_as_float(w[k] << 16);
            acc[g][2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[g][j] = c + j < N ? __uint_as_float((uint32_t)yp[j] << 16) : 0.0f;
        }
      } else {
        const float* yp = static_cast<const float*>(y) + (int64_t)m * ldy + c;
        if (full) {
          const uint4 a = ld_v4_hint(yp, stream), b = ld_v4_hint(yp + 4, stream);
          acc[g][0] = __uint_as_float(a.x); acc[g][1] = __uint_as_float(a.y);
          acc[g][2] = __uint_as_float(a.z); acc[g][3] = __uint_as_float(a.w);
          acc[g][4] = __uint_as_float(b.x); acc[g][5] = __uint_as_float(b.y);
          acc[g][6] = __uint_as_float(b.z); acc[g][7] = __uint_as_float(b.w);
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[g][j] = c + j < N ? yp[j] : 0.0f;
        }
      }
    }
    for (uint32_t i0 = 0; i0 < len; i0 += 4) {
      OccEntry e[4];
      uint4 q[4][G];
#pragma unroll
      for (int j = 0; j < 4; ++j) e[j] = i0 + j < len ? ent[s0 + i0 + j] : OccEntry{0, 0.0f};
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int g = 0; g < G; ++g)   // W^T rows are padded to 8: a group starting below N is readable
          q[j][g] = (i0 + j < len && cu + 8 * g < N) ? ld_v4_hint(wt + (int64_t)e[j].k * ldt + cu + 8 * g, keep)
                                                      : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (i0 + j >= len) break;   // the row's true entries only
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const uint32_t w[4] = {q[j][g].x, q[j][g].y, q[j][g].z, q[j][g].w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            acc[g][2 * k] = fmaf(e[j].v, __uint_as_float(w[k] << 16), acc[g][2 * k]);
            acc[g][2 * k + 1] = fmaf(e[j].v, __uint_as_float(w[k] & 0xFFFF0000u), acc[g][2 * k + 1]);
          }
        }
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const int64_t c = cu + 8 * g;
      if (c >= N) break;
      const bool full = c + 8 <= N;
      if constexpr (BF16) {
        uint16_t* yp = static_cast<uint16_t*>(y) + (int64_t)m * ldy + c;
        uint32_t pk[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const __nv_bfloat162 h = __floats2bfloat162_rn(acc[g][2 * k], acc[g][2 * k + 1]);
          pk[k] = *reinterpret_cast<const uint32_t*>(&h);
        }
        if (full) {
          st_v4_hint(yp, make_uint4(pk[0], pk[1], pk[2], pk[3]), stream);
        } else {
          for (int j = 0; j < 8 && c + j < N; ++j) yp[j] = (uint16_t)(pk[j >> 1] >> (16 * (j & 1)));
        }
      } else {
        float* yp = static_cast<float*>(y) + (int64_t)m * ldy + c;
        if (full) {
          st_v4_hint(yp, make_uint4(__float_as_uint(acc[g][0]), __float_as_uint(acc[g][1]),
                                    __float_as_uint(acc[g][2]), __float_as_uint(acc[g][3])), stream);
          st_v4_hint(yp + 4, make_uint4(__float_as_uint(acc[g][4]), __float_as_uint(acc[g][5]),
                                        __float_as_uint(acc[g][6]), __float_as_uint(acc[g][7])), stream);
        } else {
          for (int j = 0; j < 8 && c + j < N; ++j) yp[j] = acc[g][j];
        }
      }
    }
  }
}

// 8-bit mask of the outliers |x| > tau among 8 consecutive elements.  bf16:
// on the bit patterns, two elements per instruction (for bf16 x, |x| > tau iff
// the magnitude bits exceed those of tau truncated to bf16; NaNs are not
// outliers, as in the clamp).
// Per 16-bit half of q (a bf16 pair): bit 15 / 31 set where taub < |x|_h <=
// 0x7F80 (an outlier, NaN excluded), by subtractions that cannot borrow across
// the halves (magnitudes and taub + 1 are at most 0x8000): in a half,
// (a | 0x8000) - (taub + 1) has bit 15 set iff a > taub, and 0xFF80 - a iff
// a <= 0x7F80.  tau2p1 = (taub + 1) in both halves.
__device__ __forceinline__ uint32_t outlier_halves(uint32_t q, uint32_t tau2p1) {
  const uint32_t a = q & 0x7FFF7FFFu;
  return ((a | 0x80008000u) - tau2p1) & (0xFF80FF80u - a) & 0x80008000u;
}
// the 8 elements' bits (element 2j from word j's low half, 2j + 1 from its high half)
__device__ __forceinline__ uint32_t outlier_mask8_bits(const uint4& u, uint32_t tau2p1) {
  const uint32_t t = (outlier_halves(u.x, tau2p1) >> 15) | (outlier_halves(u.y, tau2p1) >> 13) |
                     (outlier_halves(u.z, tau2p1) >> 11) | (outlier_halves(u.w, tau2p1) >> 9);
  return (t & 0x55u) | ((t >> 15) & 0xAAu);
}

template <int XDT>
__device__ __forceinline__ uint32_t outlier_mask8(const void* x, int64_t off, float tau, uint32_t tau2) {
  if constexpr (XDT == FP4_DTYPE_BF16) {
    // a plain read-only load (not volatile asm), so that the compiler can put
    // the loads of all the row's chunks in flight before the masks
    return outlier_mask8_bits(__ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(x) + off)), tau2);
  } else {
    float e[8];
    load8<FP4_DTYPE_F32, true>(x, off, e);
    uint32_t mask = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) mask |= (fabsf(e[j]) > tau ? 1u : 0u) << j;
    return mask;
  }
}

// One warp per row: the scattered outliers of the row (|x| > tau, in a column
// that the extra GEMM columns do not carry), lane-major: lane l writes the
// outliers of its columns 8l..8l+7, 256+8l.., in order, after the lanes below
// it.  The 8 warps of a CTA claim their segments with one atomic on the global
// cursor.  The row is read twice (count, write); the second read hits the
// caches and touches only the 8-column groups that hold scattered outliers.
template <int FMT, int XDT>
__global__ void __launch_bounds__(256) occ_extract_kernel(const void* __restrict__ x, int64_t ldx, int64_t rows,
                                                          int64_t cols, fp4_operand xq, fp4_operand wq,
                                                          const float* __restrict__ tau_p,
                                                          const uint32_t* __restrict__ dense, uint32_t* cursor,
                                                          uint32_t capacity, uint32_t* row_start, uint32_t* row_len,
                                                          OccEntry* entries, unsigned int* status) {
  __shared__ uint32_t warp_off[8];
  __shared__ uint32_t cta_base;
  const float tau = *tau_p;
  // bf16 x: |x| > tau iff its magnitude bits exceed those of tau truncated to bf16
  const uint32_t taub = (__float_as_uint(tau) >> 16) & 0x7FFFu, tau2 = (taub + 1u) | ((taub + 1u) << 16);
  const bool tail = tail_inv_alpha<FMT>(xq, wq) != 0.0f;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  auto scat_mask = [&](int64_t r, int64_t c0) {
    const uint32_t m = outlier_mask8<XDT>(x, r * ldx + c0, tau, tau2);
    if (!m || !tail) return m;
    return m & ~((dense[c0 >> 5] >> (c0 & 31)) & 0xFFu);
  };
  // rows of up to 16 x 256 columns keep their 16 eight-bit masks in 4 registers
  // between the passes; longer rows recompute them
  const bool short_row = cols <= 16 * 256;
  for (int64_t r0 = blockIdx.x * (int64_t)8; r0 < rows; r0 += (int64_t)gridDim.x * 8) {   // uniform over the CTA
    const int64_t r = r0 + w;
    const bool active = r < rows;
    uint32_t mine = 0;
    uint32_t mk[4] = {0u, 0u, 0u, 0u};
    if (active) {
      if (short_row && XDT == FP4_DTYPE_BF16) {
        // all 16 chunk loads of the row in flight, then the masks
        uint4 raw[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int64_t c0 = 256 * i + 8 * lane;
          raw[i] = c0 < cols ? __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(x) + r * ldx + c0))
                             : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int64_t c0 = 256 * i + 8 * lane;
          uint32_t m = outlier_mask8_bits(raw[i], tau2);
          if (m && tail && c0 < cols) m &= ~((dense[c0 >> 5] >> (c0 & 31)) & 0xFFu);
          mk[i >> 2] |= m << (8 * (i & 3));
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) mine += __popc(mk[i]);
      } else if (short_row) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int64_t c0 = 256 * i + 8 * lane;
          if (c0 < cols) mk[i >> 2] |= scat_mask(r, c0) << (8 * (i & 3));
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) mine += __popc(mk[i]);
      } else {
#pragma unroll 4
        for (int64_t c0 = 8 * lane; c0 < cols; c0 += 256) mine += __popc(scat_mask(r, c0));
      }
    }
    uint32_t incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += t;
    }
    const uint32_t cnt = __shfl_sync(0xFFFFFFFFu, incl, 31);
    if (lane == 0) warp_off[w] = cnt;
    __syncthreads();
    if (threadIdx.x == 0) {
      uint32_t sum = 0;
      for (int i = 0; i < 8; ++i) {
        const uint32_t c = warp_off[i];
        warp_off[i] = sum;
        sum += c;
      }
      cta_base = sum ? atomicAdd(cursor, sum) : 0u;
    }
    __syncthreads();
    const uint32_t base = cta_base + warp_off[w];
    __syncthreads();                       // warp_off / cta_base are rewritten next iteration
    if (!active) continue;
    const bool fits = (uint64_t)base + cnt <= capacity;
    if (lane == 0) {
      row_start[r] = base;
      row_len[r] = fits ? cnt : 0u;
      if (!fits) atomicOr(status, FP4_DEVICE_OVERFLOW);
    }
    if (!mine || !fits) continue;
    uint32_t pos = base + incl - mine;
    auto emit = [&](int64_t c0, uint32_t m) {
      while (m) {
        const int j = __ffs(m) - 1;
        m &= m - 1;
        entries[pos++] = OccEntry{(int32_t)(c0 + j), clamp_residual(load_elem<XDT>(x, r * ldx + c0 + j), tau)};
      }
    };
    if (short_row) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint32_t m = (mk[i >> 2] >> (8 * (i & 3))) & 0xFFu;
        if (m) emit(256 * i + 8 * lane, m);
      }
    } else {
      for (int64_t c0 = 8 * lane; c0 < cols; c0 += 256) emit(c0, scat_mask(r, c0));
    }
  }
}

inline int grid_cap(int64_t items, int per_block, int num_sms, int per_sm = 8) {
  const int64_t need = cdiv(items, per_block), cap = (int64_t)num_sms * per_sm;
  return (int)std::max<int64_t>(1, std::min(need, cap));
}

}  // namespace

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
// workspace: select state, then the fine and coarse histograms of each pass
size_t occ_threshold_ws_bytes(int dt) {
  return 256 + sizeof(unsigned long long) * (kHistBins + 256 + (dt == FP4_DTYPE_F32 ? kLowBins + 256 : 0));
}

cudaError_t launch_occ_threshold(const void* x, int dt, int64_t rows, int64_t cols, int64_t ldx, uint64_t rank,
                                 void* ws, float* tau, long long* n_out, int num_sms, cudaStream_t st) {
  OccSelect* sel = static_cast<OccSelect*>(ws);
  auto* fine = reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(ws) + 256);
  auto* coarse = fine + kHistBins;
  cudaError_t e = cudaMemsetAsync(ws, 0, occ_threshold_ws_bytes(dt), st);
  if (e != cudaSuccess) return e;
  const uint64_t n = (uint64_t)rows * cols;
  const uint32_t total_vecs = (uint32_t)(n / 8);
  const FastDiv fd = make_fastdiv((uint32_t)(cols / 8));
  const size_t smem = kHistBins * sizeof(uint32_t);
  const int grid = grid_cap(total_vecs, kHistThreads, num_sms, 1);
  if (dt == FP4_DTYPE_BF16) {
    e = cudaFuncSetAttribute(occ_hist_kernel<FP4_DTYPE_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    occ_hist_kernel<FP4_DTYPE_BF16><<<grid, kHistThreads, smem, st>>>(x, ldx, fd, total_vecs, fine, coarse);
    occ_select_kernel<0, FP4_DTYPE_BF16><<<1, 32, 0, st>>>(fine, coarse, n, rank, sel, tau, n_out);
  } else {
    e = cudaFuncSetAttribute(occ_hist_kernel<FP4_DTYPE_F32>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    occ_hist_kernel<FP4_DTYPE_F32><<<grid, kHistThreads, smem, st>>>(x, ldx, fd, total_vecs, fine, coarse);
    occ_select_kernel<0, FP4_DTYPE_F32><<<1, 32, 0, st>>>(fine, coarse, n, rank, sel, tau, n_out);
    unsigned long long* fine_low = coarse + 256;
    unsigned long long* coarse_low = fine_low + kLowBins;
    occ_hist_low_kernel<<<grid_cap(total_vecs, 256, num_sms), 256, 0, st>>>(static_cast<const float*>(x), ldx, fd,
                                                                            total_vecs, sel, fine_low, coarse_low);
    occ_select_kernel<1, FP4_DTYPE_F32><<<1, 32, 0, st>>>(fine_low, coarse_low, n, rank, sel, tau, n_out);
  }
  return cudaGetLastError();
}

OccLayout occ_layout(int64_t m, int64_t n, int64_t k, int k_dense, int64_t max_outliers) {
  OccLayout L{};
  auto al = [](size_t v) { return (v + 255) & ~size_t(255); };
  L.kx = k_dense > 0 ? cdiv(k_dense, 64) * 64 : 0;
  L.ldt = cdiv(n, 8) * 8;
  size_t off = 0;
  L.counts = off;    off = al(off + sizeof(float) * 2 * (size_t)k);     // top-k scratch: values + flags
  L.hot = off;       off = al(off + sizeof(int32_t) * (size_t)std::max(k_dense, 1));
  L.flags = off;     off = al(off + sizeof(uint32_t) * (size_t)cdiv(k, 32));
  L.a_ext = off;     off = al(off + 2 * (size_t)m * L.kx);
  L.b_ext = off;     off = al(off + 2 * (size_t)n * L.kx);
  L.wt = off;        off = al(off + 2 * (size_t)k * L.ldt);
  L.row_start = off; off = al(off + sizeof(uint32_t) * (size_t)m);
  L.row_len = off;   off = al(off + sizeof(uint32_t) * (size_t)m);
  L.cursor = off;    off = al(off + sizeof(uint32_t));
  L.entries = off;   off = al(off + sizeof(OccEntry) * (size_t)std::max<int64_t>(max_outliers, 1));
  L.bytes = off;
  return L;
}

cudaError_t launch_occ_prepare(const void* x, int xdt, int64_t ldx, const uint16_t* w, int64_t ldw,
                               const fp4_operand& xq, const fp4_operand& wq, const float* tau, const float* col_counts,
                               int k_dense, int64_t max_outliers, void* ws, const OccLayout& L, unsigned int* status,
                               int num_sms, cudaStream_t st) {
  uint8_t* base = static_cast<uint8_t*>(ws);
  const int64_t M = xq.rows, N = wq.rows, K = xq.k;
  uint32_t* flags = reinterpret_cast<uint32_t*>(base + L.flags);
  cudaError_t e = cudaMemsetAsync(flags, 0, sizeof(uint32_t) * (size_t)cdiv(K, 32), st);
  if (e != cudaSuccess) return e;
  const int32_t* hot = reinterpret_cast<int32_t*>(base + L.hot);
  if (k_dense > 0) {
    float* counts = reinterpret_cast<float*>(base + L.counts);
    e = cudaMemcpyAsync(counts, col_counts, sizeof(float) * K, cudaMemcpyDeviceToDevice, st);
    if (e != cudaSuccess) return e;
    e = launch_hcp_topk(counts, K, k_dense, reinterpret_cast<int32_t*>(base + L.hot), st);
    if (e != cudaSuccess) return e;
    occ_flags_kernel<<<(unsigned)cdiv(k_dense, 256), 256, 0, st>>>(hot, k_dense, flags);
    const int grid = grid_cap((M + N) * (L.kx / 8), 256, num_sms);
    uint16_t* a_ext = reinterpret_cast<uint16_t*>(base + L.a_ext);
    uint16_t* b_ext = reinterpret_cast<uint16_t*>(base + L.b_ext);
#define FP4_OCC_TAIL(FMT, XDT) \
  occ_tail_kernel<FMT, XDT><<<grid, 256, 0, st>>>(x, ldx, w, ldw, xq, wq, tau, hot, k_dense, L.kx, a_ext, b_ext)
    if (xq.format == FP4_FMT_MXFP4) {
      if (xdt == FP4_DTYPE_BF16) FP4_OCC_TAIL(FP4_FMT_MXFP4, FP4_DTYPE_BF16); else FP4_OCC_TAIL(FP4_FMT_MXFP4, FP4_DTYPE_F32);
    } else {
      if (xdt == FP4_DTYPE_BF16) FP4_OCC_TAIL(FP4_FMT_NVFP4, FP4_DTYPE_BF16); else FP4_OCC_TAIL(FP4_FMT_NVFP4, FP4_DTYPE_F32);
    }
#undef FP4_OCC_TAIL
  }
  // W^T for the scattered pass (padding columns zeroed when N is not a multiple of 8)
  uint16_t* wt = reinterpret_cast<uint16_t*>(base + L.wt);
  if (L.ldt != N) {
    e = cudaMemsetAsync(wt, 0, 2 * (size_t)K * L.ldt, st);
    if (e != cudaSuccess) return e;
  }
  transpose_bf16_kernel<<<grid_cap(cdiv(N, 64) * cdiv(K, 64), 1, num_sms, 8), 256, 0, st>>>(w, ldw, N, K, wt, L.ldt);
  uint32_t* cursor = reinterpret_cast<uint32_t*>(base + L.cursor);
  e = cudaMemsetAsync(cursor, 0, sizeof(uint32_t), st);
  if (e != cudaSuccess) return e;
  uint32_t* rs = reinterpret_cast<uint32_t*>(base + L.row_start);
  uint32_t* rl = reinterpret_cast<uint32_t*>(base + L.row_len);
  OccEntry* ent = reinterpret_cast<OccEntry*>(base + L.entries);
  const int grid = grid_cap(cdiv(M, 8), 1, num_sms, 8);
#define FP4_OCC_EXTRACT(FMT, XDT)                                                                       \
  occ_extract_kernel<FMT, XDT><<<grid, 256, 0, st>>>(x, ldx, M, K, xq, wq, tau, flags, cursor, (uint32_t)max_outliers, \
                                                    rs, rl, ent, status)
  if (xq.format == FP4_FMT_MXFP4) {
    if (xdt == FP4_DTYPE_BF16) FP4_OCC_EXTRACT(FP4_FMT_MXFP4, FP4_DTYPE_BF16); else FP4_OCC_EXTRACT(FP4_FMT_MXFP4, FP4_DTYPE_F32);
  } else {
    if (xdt == FP4_DTYPE_BF16) FP4_OCC_EXTRACT(FP4_FMT_NVFP4, FP4_DTYPE_BF16); else FP4_OCC_EXTRACT(FP4_FMT_NVFP4, FP4_DTYPE_F32);
  }
#undef FP4_OCC_EXTRACT
  return cudaGetLastError();
}

cudaError_t launch_occ_correct(void* y, int64_t ldy, int out_dtype, int64_t m, int64_t n, const void* ws,
                               const OccLayout& L, int num_sms, cudaStream_t st) {
  if (m == 0 || n == 0) return cudaSuccess;
  const uint8_t* base = static_cast<const uint8_t*>(ws);
  const auto* rs = reinterpret_cast<const uint32_t*>(base + L.row_start);
  const auto* rl = reinterpret_cast<const uint32_t*>(base + L.row_len);
  const auto* ent = reinterpret_cast<const OccEntry*>(base + L.entries);
  const auto* wt = reinterpret_cast<const uint16_t*>(base + L.wt);
  // 16-column units with 32-bit ids (below 2^31, so that the grid stride
  // cannot wrap): row bands of at most that many units per launch
  const int64_t upr = cdiv(n, 16), band = std::max<int64_t>(1, ((int64_t(1) << 31) - 1) / upr);
  const FastDiv fd = make_fastdiv((uint32_t)upr);
  const int esz = out_dtype == FP4_DTYPE_BF16 ? 2 : 4;
  for (int64_t r0 = 0; r0 < m; r0 += band) {
    const int64_t rows = std::min(band, m - r0);
    void* yb = static_cast<uint8_t*>(y) + r0 * ldy * esz;
    const int grid = grid_cap(rows * upr, 256, num_sms);
    if (out_dtype == FP4_DTYPE_BF16)
      occ_correct_kernel<true><<<grid, 256, 0, st>>>(yb, ldy, rows, n, fd, rs + r0, rl + r0, ent, wt, L.ldt);
    else
      occ_correct_kernel<false><<<grid, 256, 0, st>>>(yb, ldy, rows, n, fd, rs + r0, rl + r0, ent, wt, L.ldt);
  }
  return cudaGetLastError();
}


}  // namespace fp4
