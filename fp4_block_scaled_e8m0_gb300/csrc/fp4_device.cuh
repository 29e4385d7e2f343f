// Device helpers for the block-scaled FP4 kernels (sm_103a).
//
// Number formats ([outlier] §1.1, [msr] §一: E2M1 with 2 exponent bits and 1
// mantissa bit covering [-6, 6]; [lowprec] §1.1: E8M0 and E4M3 scales) and the
// per-element steps of Q(x) = s * round(x / s) ([grad] §2.1).
//
// Every floating-point step that decides a code uses explicitly rounded fp32
// intrinsics (__fmul_rn, __fdiv_rn, __frcp_rn, __fadd_rn) so the compiler can
// neither contract nor reorder it: the results are bit-reproducible.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "fp4_internal.h"

namespace fp4dev {

// ----------------------------------------------------------------------------
// loads
// ----------------------------------------------------------------------------
__device__ __forceinline__ float bf16_bits_to_float(uint32_t h) { return __uint_as_float(h << 16); }

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

// read-only load that allocates in L1: a thread's second 16 bytes of a 32-byte
// sector then hit L1 instead of fetching the sector from L2 again
__device__ __forceinline__ uint4 ld_nc_v4_l1(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

// Division of 32-bit n by a divisor d fixed for the launch (1 <= d < 2^31), as
// a multiply-high and two shifts: Granlund & Montgomery, "Division by
// invariant integers using multiplication" (PLDI 1994), Fig. 4.1, with
// l = ceil(log2 d), m = floor(2^32 (2^l - d) / d) + 1.
struct FastDiv {
  uint32_t d, m, s1, s2;
};
inline FastDiv make_fastdiv(uint32_t d) {
  uint32_t l = 0;
  while ((1ull << l) < d) ++l;
  const uint64_t m = ((1ull << 32) * ((1ull << l) - d)) / d + 1;
  return {d, (uint32_t)m, l < 1 ? 0u : 1u, l < 1 ? 0u : l - 1};
}
__device__ __forceinline__ uint32_t fast_div(uint32_t n, const FastDiv& f) {
  const uint32_t t = __umulhi(f.m, n);
  return (t + ((n - t) >> f.s1)) >> f.s2;
}

// 8 consecutive input elements (16 bytes of bf16 or 32 bytes of fp32) -> fp32
template <int DT, bool L1 = false>
__device__ __forceinline__ void load8(const void* base, int64_t elem, float* v) {
  if constexpr (DT == FP4_DTYPE_BF16) {
    uint4 q = L1 ? ld_nc_v4_l1(static_cast<const uint16_t*>(base) + elem) : ld_nc_v4(static_cast<const uint16_t*>(base) + elem);
    uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  } else {
    const float* p = static_cast<const float*>(base) + elem;
    uint4 a = L1 ? ld_nc_v4_l1(p) : ld_nc_v4(p), b = L1 ? ld_nc_v4_l1(p + 4) : ld_nc_v4(p + 4);
    v[0] = __uint_as_float(a.x); v[1] = __uint_as_float(a.y);
    v[2] = __uint_as_float(a.z); v[3] = __uint_as_float(a.w);
    v[4] = __uint_as_float(b.x); v[5] = __uint_as_float(b.y);
    v[6] = __uint_as_float(b.z); v[7] = __uint_as_float(b.w);
  }
}

template <int DT>
__device__ __forceinline__ float load1(const void* base, int64_t elem) {
  if constexpr (DT == FP4_DTYPE_BF16)
    return bf16_bits_to_float(__ldg(static_cast<const uint16_t*>(base) + elem));
  else
    return __ldg(static_cast<const float*>(base) + elem);
}

// ----------------------------------------------------------------------------
// E2M1 element encoding
// ----------------------------------------------------------------------------
// Hardware conversion of two fp32 values to packed E2M1 (round to nearest even,
// saturating).  `lo` lands in bits 0-3, `hi` in bits 4-7.
__device__ __forceinline__ uint32_t e2m1x2_hw(float lo, float hi) {
  uint32_t r;
  asm("{\n.reg .b8 q;\ncvt.rn.satfinite.e2m1x2.f32 q, %1, %2;\ncvt.u32.u8 %0, q;\n}"
      : "=r"(r) : "f"(hi), "f"(lo));
  return r & 0xFFu;
}

// one byte of two E2M1 codes (low nibble = first element) -> their exact values
// (sign included) by the hardware conversion to f16x2, then to fp32
__device__ __forceinline__ void e2m1x2_decode(uint32_t byte, float& lo, float& hi) {
  uint32_t h2;
  asm("{\n.reg .b8 c;\ncvt.u8.u32 c, %1;\ncvt.rn.f16x2.e2m1x2 %0, c;\n}" : "=r"(h2) : "r"(byte));
  lo = __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
  hi = __half2float(__ushort_as_half((unsigned short)(h2 >> 16)));
}

// Eight bf16 times the power of two rb (a bf16 bit pattern) -> eight E2M1
// codes, element 0 in bits 0-3.  Each product is one fma.rn.f32.bf16 with
// addend -0: the exact product rounded once to fp32 (subnormals kept), the
// same value and sign of zero as fmul.rn of the two converted to fp32; then
// the hardware conversion (round to nearest even, saturating) two at a time,
// and the four code bytes gathered into one word.  The products run on the
// FMA pipe, which leaves the integer pipe to the rest of the quantizer.
// The elements are the halves of w0..w3 in order (H = 2), or half H of each
// of w0..w7 (H = 0: low halves, H = 1: high halves).
#define FP4_E2M1X8_TAIL                                            \
  "cvt.rn.satfinite.e2m1x2.f32 c0, f1, f0;\n\t"                     \
  "cvt.rn.satfinite.e2m1x2.f32 c1, f3, f2;\n\t"                     \
  "cvt.rn.satfinite.e2m1x2.f32 c2, f5, f4;\n\t"                     \
  "cvt.rn.satfinite.e2m1x2.f32 c3, f7, f6;\n\t"                     \
  "cvt.u32.u8 u0, c0;\n\t"                                          \
  "cvt.u32.u8 u1, c1;\n\t"                                          \
  "cvt.u32.u8 u2, c2;\n\t"                                          \
  "cvt.u32.u8 u3, c3;\n\t"                                          \
  "prmt.b32 t0, u0, u1, 0x0040;\n\t"                                \
  "prmt.b32 t1, u2, u3, 0x0040;\n\t"                                \
  "prmt.b32 %0, t0, t1, 0x5410;\n\t"                                \
  "}"
#define FP4_E2M1X8_REGS                                            \
  "{\n\t"                                                           \
  ".reg .b16 r, z, e0, e1, e2, e3, e4, e5, e6, e7;\n\t"             \
  ".reg .f32 mz, f0, f1, f2, f3, f4, f5, f6, f7;\n\t"               \
  ".reg .b8 c0, c1, c2, c3;\n\t"                                    \
  ".reg .b32 u0, u1, u2, u3, t0, t1;\n\t"                           \
  "mov.b32 {r, z}, %1;\n\t"                                         \
  "mov.f32 mz, 0f80000000;\n\t"
#define FP4_E2M1X8_FMA                                              \
  "fma.rn.f32.bf16 f0, e0, r, mz;\n\t"                              \
  "fma.rn.f32.bf16 f1, e1, r, mz;\n\t"                              \
  "fma.rn.f32.bf16 f2, e2, r, mz;\n\t"                              \
  "fma.rn.f32.bf16 f3, e3, r, mz;\n\t"                              \
  "fma.rn.f32.bf16 f4, e4, r, mz;\n\t"                              \
  "fma.rn.f32.bf16 f5, e5, r, mz;\n\t"                              \
  "fma.rn.f32.bf16 f6, e6, r, mz;\n\t"                              \
  "fma.rn.f32.bf16 f7, e7, r, mz;\n\t"

__device__ __forceinline__ uint32_t mx_codes8(uint4 w, uint32_t rb) {
  uint32_t out;
  asm(FP4_E2M1X8_REGS
      "mov.b32 {e0, e1}, %2;\n\t"
      "mov.b32 {e2, e3}, %3;\n\t"
      "mov.b32 {e4, e5}, %4;\n\t"
      "mov.b32 {e6, e7}, %5;\n\t"
      FP4_E2M1X8_FMA FP4_E2M1X8_TAIL
      : "=r"(out) : "r"(rb), "r"(w.x), "r"(w.y), "r"(w.z), "r"(w.w));
  return out;
}

template <int H>
__device__ __forceinline__ uint32_t mx_codes8_half(const uint32_t* w, uint32_t rb) {
  static_assert(H == 0 || H == 1, "half");
  uint32_t out;
  if constexpr (H == 0)
    asm(FP4_E2M1X8_REGS
        "mov.b32 {e0, z}, %2;\n\t" "mov.b32 {e1, z}, %3;\n\t" "mov.b32 {e2, z}, %4;\n\t" "mov.b32 {e3, z}, %5;\n\t"
        "mov.b32 {e4, z}, %6;\n\t" "mov.b32 {e5, z}, %7;\n\t" "mov.b32 {e6, z}, %8;\n\t" "mov.b32 {e7, z}, %9;\n\t"
        FP4_E2M1X8_FMA FP4_E2M1X8_TAIL
        : "=r"(out) : "r"(rb), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]),
          "r"(w[7]));
  else
    asm(FP4_E2M1X8_REGS
        "mov.b32 {z, e0}, %2;\n\t" "mov.b32 {z, e1}, %3;\n\t" "mov.b32 {z, e2}, %4;\n\t" "mov.b32 {z, e3}, %5;\n\t"
        "mov.b32 {z, e4}, %6;\n\t" "mov.b32 {z, e5}, %7;\n\t" "mov.b32 {z, e6}, %8;\n\t" "mov.b32 {z, e7}, %9;\n\t"
        FP4_E2M1X8_FMA FP4_E2M1X8_TAIL
        : "=r"(out) : "r"(rb), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]),
          "r"(w[7]));
  return out;
}
#undef FP4_E2M1X8_TAIL
#undef FP4_E2M1X8_REGS
#undef FP4_E2M1X8_FMA

// Per-half magnitude maximum of bf16 pairs: max(|a|, |b|) on each half with
// the sign bit the xor of the two (max.xorsign.abs.bf16x2, FMA pipe); the
// caller clears the sign bits.  For finite values the larger magnitude is the
// larger magnitude bit pattern, so this is the block amax of the bit-pattern
// form, subnormals included.
__device__ __forceinline__ uint32_t bf16x2_absmax(uint32_t a, uint32_t b) {
  uint32_t m;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m) : "r"(a), "r"(b));
  return m;
}
// magnitude bits of the largest of eight bf16 (the halves of w)
__device__ __forceinline__ uint32_t bf16x8_amax_bits(uint4 w) {
  const uint32_t m = bf16x2_absmax(bf16x2_absmax(w.x, w.y), bf16x2_absmax(w.z, w.w)) & 0x7FFF7FFFu;
  return max(m & 0xFFFFu, m >> 16);
}

// Compare chain against the midpoints of the grid {0,.5,1,1.5,2,3,4,6}; at a
// midpoint the even code wins (0.25->0, 0.75->2, 1.25->2, 1.75->4, 2.5->4,
// 3.5->6, 5->6); the sign bit is kept.
__device__ __forceinline__ uint32_t e2m1_sw(float xs) {
  float a = fabsf(xs);
  uint32_t m = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) +
               (a >= 3.5f) + (a > 5.0f);
  return ((__float_as_uint(xs) >> 28) & 8u) | m;
}

// Stochastic rounding onto the grid ([lowprec] §3.2's floor(x) + (rand < frac)
// on the non-uniform E2M1 grid): lo = largest grid point <= |xs| (|xs| saturated
// at 6), frac = (|xs| - lo) / step, round up iff u16 < frac * 65536.
// Returns the chosen grid value with the sign of xs; the hardware conversion of
// a grid value is exact, so e2m1x2_hw packs the codes.
//
// Bit-level form.  From 1 up, the grid keeps one mantissa bit of each binade,
// so with rem = the 22 mantissa bits below it, frac * 2^22 = rem and the test
// is 64 u16 < rem: adding 0x3FFFFF - 64 u16 to the fp32 bits carries into the
// kept bit exactly then, and masking the 22 bits leaves lo or the next grid
// point (the carry may move into the exponent: 1.5 * 2^e -> 2^(e+1)).  Below 1
// the step is 0.5, which is the step of [1, 2): b = 1 + |xs| rounded up puts
// the value there with rem = ceil(frac * 2^22), and for an integer n,
// n < R iff n < ceil(R), so the same addition decides exactly; 1 is subtracted
// again afterwards (exact).  fminf sends NaN to the saturated 6, like the clamp.
// (e2m1_sr_value_finite below drops the clamp for the block quantizers, where
// |xs| is finite and below 9 by construction of the block scale: from 6 up the
// result is a value >= 6 that the saturating conversion maps to code 7.)
__device__ __forceinline__ float e2m1_sr_value(float xs, uint32_t u16_shl6) {
  const float a = fminf(fabsf(xs), 6.0f);
  const float off = a < 1.0f ? 1.0f : 0.0f;
  const float b = __fadd_ru(a, off);
  const uint32_t n = (__float_as_uint(b) + 0x3FFFFFu - u16_shl6) & 0xFFC00000u;
  const float y = __fsub_rn(__uint_as_float(n), off);
  return __uint_as_float(__float_as_uint(y) | (__float_as_uint(xs) & 0x80000000u));
}

// ----------------------------------------------------------------------------
// E4M3 (NVFP4 block scale) and E8M0 (MXFP4 block scale)
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t e4m3_rn_satfinite(float t) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(t));
  return r & 0xFFu;
}

// two signed values: the E4M3 byte of `lo` in bits 0-7, of `hi` in bits 8-15
__device__ __forceinline__ uint32_t e4m3x2_rn_satfinite(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float e4m3_decode(uint32_t b) {
  uint32_t e = (b >> 3) & 15u, m = b & 7u;
  return e == 0 ? __fmul_rn((float)m, 0.001953125f)            // m * 2^-9
                : __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// E8M0 byte of a non-negative block amax: floor(log2 amax) - 2 + 127, clamped to
// [0, 254]; amax = 0 and subnormal amax give byte 0.
__device__ __forceinline__ uint32_t e8m0_byte(float amax) {
  int E = (int)((__float_as_uint(amax) >> 23) & 0xFFu);
  return E >= 2 ? (uint32_t)(E - 2) : 0u;
}
// 2^(127 - byte): the exact power of two applied to each element
__device__ __forceinline__ float e8m0_inv_scale(uint32_t byte) {
  return __uint_as_float((254u - byte) << 23);
}
__device__ __forceinline__ float e8m0_scale(uint32_t byte) {
  return byte == 0 ? 5.877471754111438e-39f /* 2^-127 */ : __uint_as_float(byte << 23);
}

// MXFP4 block scale from the magnitude bits of a bf16 block amax: the E8M0
// byte is the amax's exponent field minus 2, i.e. floor(log2 amax) - 2 + 127
// (bf16 and fp32 share the exponent field), clamped at the format's minimum
// (fields 0-2, which include the bf16 subnormals and 0, give byte 0); rb =
// 2^(127 - byte), as a bf16, multiplies each element exactly
__device__ __forceinline__ void mx_scale_from_bits(uint32_t amax_bits, uint32_t& byte, uint32_t& rb) {
  const uint32_t e = (amax_bits >> 7) & 0xFFu;
  byte = e >= 2 ? e - 2 : 0u;
  rb = (254u - byte) << 7;   // 2^(127 - byte) as a bf16 bit pattern (the fp32 one's high half)
}

// Block scale of one block: writes the scale byte and the multiplier r with
// xs = x * r (zero_block = codes forced to 0 when the NVFP4 scale is 0).
template <int FMT>
__device__ __forceinline__ void block_scale(float amax_b, float g, uint32_t& byte, float& r,
                                            bool& zero_block) {
  if constexpr (FMT == FP4_FMT_MXFP4) {
    byte = e8m0_byte(amax_b);
    r = e8m0_inv_scale(byte);
    zero_block = false;
  } else {
    if (g == 0.0f) {
      byte = 0;
      r = 0.0f;
      zero_block = true;
      return;
    }
    float d = __fmul_rn(6.0f, g);
    float t = __fdiv_rn(amax_b, d);
    byte = e4m3_rn_satfinite(t);
    float s = __fmul_rn(e4m3_decode(byte), g);
    zero_block = (s == 0.0f);
    r = zero_block ? 0.0f : __frcp_rn(s);
  }
}

__device__ __forceinline__ float nvfp4_tensor_scale(float amax_t) { return __fdiv_rn(amax_t, 2688.0f); }

// ----------------------------------------------------------------------------
// Philox4x32-10 (Salmon et al., SC'11)
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int rnd = 0; rnd < 10; ++rnd) {
    if (rnd) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint64_t p0 = (uint64_t)0xD2511F53u * c.x;   // one wide multiply each
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * c.z;
    c = make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ k0, (uint32_t)p1, (uint32_t)(p0 >> 32) ^ c.w ^ k1, (uint32_t)p0);
  }
  return c;
}

// Philox with precomputed round keys (fp4::philox_round_keys)
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, const fp4::PhiloxRoundKeys& k) {
#pragma unroll
  for (int rnd = 0; rnd < 10; ++rnd) {
    const uint64_t p0 = (uint64_t)0xD2511F53u * c.x;
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * c.z;
    c = make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ k.k0[rnd], (uint32_t)p1, (uint32_t)(p0 >> 32) ^ c.w ^ k.k1[rnd],
                   (uint32_t)p0);
  }
  return c;
}

// Eight 16-bit uniforms for output elements 8n .. 8n+7 (n = offset + i/8).
__device__ __forceinline__ uint4 sr_bits8(uint64_t seed, uint64_t offset, uint32_t stream,
                                          uint64_t first_elem) {
  uint64_t n = offset + (first_elem >> 3);
  return philox4x32_10(make_uint4((uint32_t)n, (uint32_t)(n >> 32), 0u, stream),
                       (uint32_t)seed, (uint32_t)(seed >> 32));
}
__device__ __forceinline__ uint4 sr_bits8(const fp4::PhiloxRoundKeys& keys, uint64_t offset, uint32_t stream,
                                          uint64_t first_elem) {
  uint64_t n = offset + (first_elem >> 3);
  return philox4x32_10(make_uint4((uint32_t)n, (uint32_t)(n >> 32), 0u, stream), keys);
}
__device__ __forceinline__ float e2m1_sr_value_finite(float xs, uint32_t u16_shl6) {
  const float a = fabsf(xs);
  const float off = a < 1.0f ? 1.0f : 0.0f;
  const float b = __fadd_ru(a, off);
  const uint32_t n = (__float_as_uint(b) + 0x3FFFFFu - u16_shl6) & 0xFFC00000u;
  const float y = __fsub_rn(__uint_as_float(n), off);
  return __uint_as_float(__float_as_uint(y) | (__float_as_uint(xs) & 0x80000000u));
}

// 64 * (16-bit lane j of w): the form e2m1_sr_value takes
__device__ __forceinline__ uint32_t u16_lane_shl6(const uint4& w, int j) {
  uint32_t word = (j >> 1) == 0 ? w.x : (j >> 1) == 1 ? w.y : (j >> 1) == 2 ? w.z : w.w;
  return (j & 1) ? ((word >> 10) & 0x3FFFC0u) : ((word << 6) & 0x3FFFC0u);
}
// the same as multiplications, which the FP32/IMAD pipe can take instead of the
// integer pipe: w * 64 and the high word of w * 2^22 (= w >> 10)
__device__ __forceinline__ uint32_t u16_lane_shl6_mul(const uint4& w, int j) {
  uint32_t word = (j >> 1) == 0 ? w.x : (j >> 1) == 1 ? w.y : (j >> 1) == 2 ? w.z : w.w;
  return ((j & 1) ? __umulhi(word, 0x400000u) : word * 64u) & 0x3FFFC0u;
}

// ----------------------------------------------------------------------------
// 16-point random Hadamard transform: y = 1/4 H16 diag(sigma) x, butterfly with
// strides 1, 2, 4, 8 (fixed fp32 order)
// ----------------------------------------------------------------------------
// signs and butterflies only: v becomes H16 diag(sigma) x (4x the transform)
__device__ __forceinline__ void rht16_raw(float* v, uint32_t sign_bits) {
#pragma unroll
  for (int j = 0; j < 16; ++j)
    v[j] = __uint_as_float(__float_as_uint(v[j]) ^ (((sign_bits >> j) & 1u) << 31));
#pragma unroll
  for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i & h) continue;
      float a = v[i], b = v[i + h];
      v[i] = __fadd_rn(a, b);
      v[i + h] = __fsub_rn(a, b);
    }
  }
}
__device__ __forceinline__ void rht16(float* v, uint32_t sign_bits) {
  rht16_raw(v, sign_bits);
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = __fmul_rn(v[j], 0.25f);
}

// ----------------------------------------------------------------------------
// Packed fp32 pairs (add/sub/mul.rn.f32x2): each lane is rounded exactly as the
// scalar .rn instruction rounds it (no flush to zero), one issue slot per pair.
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// rht16_raw with the signs as multipliers sigma = +-1.0f, on the lane pairs
// p[k] = (v_k, v_{k+8}), k = 0..7, with sig2[k] = (sigma_k, sigma_{k+8}) as the
// bit patterns of a packed pair.  Stages 1, 2 and 4 combine elements whose
// indices differ by 1, 2 or 4, the same offset in both lanes, so each packed
// operation is two of the scalar ones; the first stage forms the exact
// products x sigma and then their sum and difference, the same single
// rounding of the same sums as sign flip + add.  Stage 8 combines the two
// lanes of one pair and is left to the caller (rht16_x2 / rht16_amax_x2).
__device__ __forceinline__ void rht16_stages124_x2(uint64_t* p, const uint64_t* sig2) {
#pragma unroll
  for (int k = 0; k < 8; k += 2) {
    const uint64_t a = f2_mul(p[k], sig2[k]), t = f2_mul(p[k + 1], sig2[k + 1]);
    p[k] = f2_add(a, t);
    p[k + 1] = f2_sub(a, t);
  }
#pragma unroll
  for (int h = 2; h < 8; h <<= 1) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (k & h) continue;
      const uint64_t a = p[k], b = p[k + h];
      p[k] = f2_add(a, b);
      p[k + h] = f2_sub(a, b);
    }
  }
}
// v becomes H16 diag(sigma) v, bit-identical to rht16_raw
__device__ __forceinline__ void rht16_x2(float* v, const uint64_t* sig2) {
  uint64_t p[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) p[k] = f2_pack(v[k], v[k + 8]);
  rht16_stages124_x2(p, sig2);
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    float a, b;
    f2_unpack(p[k], a, b);
    v[k] = __fadd_rn(a, b);
    v[k + 8] = __fsub_rn(a, b);
  }
}
// max_j |(H16 diag(sigma) v)_j| without forming the last stage: for the
// stage-8 pair (a, b), max(|fl(a + b)|, |fl(a - b)|) = fl(|a| + |b|), since
// rounding is monotone and symmetric and max(|a + b|, |a - b|) = |a| + |b|
// (a NaN is skipped by fmaxf either way; infinities give the same result).
__device__ __forceinline__ float rht16_amax_x2(const float* v, const uint64_t* sig2) {
  uint64_t p[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) p[k] = f2_pack(v[k], v[k + 8]);
  rht16_stages124_x2(p, sig2);
  float m = 0.0f;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    float a, b;
    f2_unpack(p[k], a, b);
    m = fmaxf(m, __fadd_rn(fabsf(a), fabsf(b)));
  }
  return m;
}

__device__ __forceinline__ uint32_t rht_sign_bits(uint64_t seed) {
  return philox4x32_10(make_uint4(0u, 0u, 0u, 0u), (uint32_t)seed, (uint32_t)(seed >> 32)).x & 0xFFFFu;
}

// ----------------------------------------------------------------------------
// scale-factor addressing
// ----------------------------------------------------------------------------
// MMA layout: rows padded to 128, blocks along k padded to 256 elements; 512-byte
// atoms of 128 rows x 4 scales.
__device__ __forceinline__ int64_t sf_offset(int sf_layout, int64_t r, int64_t j, int64_t nsf_row,
                                             int64_t nsf_pad) {
  if (sf_layout == FP4_SF_ROWMAJOR) return r * nsf_row + j;
  return ((r >> 7) * (nsf_pad >> 2) + (j >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (j & 3);
}

// ----------------------------------------------------------------------------
// reductions and status
// ----------------------------------------------------------------------------
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// block-wide max (blockDim.x multiple of 32, <= 1024), then one atomicMax on
// the fp32 bit pattern (valid for non-negative floats).
// gen == 0: *out is a float the caller zeroed.  gen != 0: out is the low word
// of a 64-bit slot holding (generation << 32) | bits; every block writes
// (gen << 32) | bits with a 64-bit atomicMax, so the first arrival of a new
// generation replaces whatever an older one left and the slot needs no
// zeroing; the low word read as a float is the amax.
__device__ __forceinline__ void block_amax_atomic(float v, float* out, uint32_t gen = 0) {
  __shared__ float red[32];
  v = warp_max(v);
  int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) red[w] = v;
  __syncthreads();
  if (w == 0) {
    v = (l < (int)(blockDim.x >> 5)) ? red[l] : 0.0f;
    v = warp_max(v);
    if (l == 0) {
      if (gen)
        atomicMax(reinterpret_cast<unsigned long long*>(out),
                  ((unsigned long long)gen << 32) | (unsigned long long)__float_as_uint(v));
      else if (v > 0.0f)
        atomicMax(reinterpret_cast<unsigned int*>(out), __float_as_uint(v));
    }
  }
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

}  // namespace fp4dev
