// MXFP4 round-to-nearest quantization of bf16 tensors in the row layout, the
// transposed layout, or both from one read (the forward and backward operand
// layouts of a linear layer: blocks of 32 along the GEMM's reduction axis).
//
// Q(x) = s * round(x / s) ([grad] §2.1) with E2M1 elements and an E8M0 block
// scale s = 2^(floor(log2 amax) - 2) clamped to [2^-127, 2^127] ([lowprec]
// §1.1; MXFP4: 32-element blocks), round to nearest even ([outlier] §4.1:
// RTN in the forward pass).
//
// 64 x 256 bf16 tiles (32 KB) reach shared memory by TMA through a ring of
// MX_NBUF buffers per CTA, so that MX_NBUF - 1 tile loads are in flight while
// one tile is quantized.  Row blocks: a warp takes one tile row per step, each lane 16
// bytes (8 elements), the 4 lanes of a 32-element block share its amax by two
// shuffles, and the warp writes 128 contiguous bytes of codes.  Column blocks:
// a thread reads one 32-bit word (a column pair) from each of 32 rows and
// quantizes both columns' blocks.  The block amax is a packed bf16 magnitude
// maximum (two columns at a time), and the E8M0 byte is the bf16 exponent
// field of the amax minus 2 (bf16 and fp32 share the exponent field): the
// same bytes as the fp32 form of the scale rule.  x / s is formed exactly as
// x * 2^(127 - byte), one fp32 rounding, before the hardware E2M1 conversion.
// Both run on the FMA pipe; the integer pipe, which bound the earlier form of
// this kernel (bit masks, packed integer maxima, unpacking), keeps the rest.
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>

#include "fp4_device.cuh"
#include "tcgen05.cuh"

using namespace fp4dev;

namespace fp4 {
namespace {

constexpr int MX_TR = 64, MX_TC = 256;                  // tile rows x columns (bf16)
constexpr int MX_TILE_BYTES = MX_TR * MX_TC * 2;        // 32 KB
constexpr int MX_THREADS = 256;
constexpr int MX_NBUF = 2;                              // tile buffers per CTA
constexpr int MX_SMEM = MX_NBUF * MX_TILE_BYTES + 128;  // tiles + barriers
constexpr int MX_CTAS_PER_SM = 3;

template <bool ROWS, bool COLS>
__global__ void __launch_bounds__(MX_THREADS, MX_CTAS_PER_SM)
    mx_tile_kernel(const __grid_constant__ CUtensorMap tm_x, int rows, int cols, uint32_t tiles_c, uint32_t ntiles,
                   QuantOut orow, QuantOut ocol, unsigned int* status) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + MX_NBUF * MX_TILE_BYTES);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(full + MX_NBUF);
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  if (t == 0) {
    for (int b = 0; b < MX_NBUF; ++b) tc::mbar_init(&full[b], 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  auto load = [&](uint32_t id, int b) {
    const uint32_t tr = id / tiles_c, tc = id - tr * tiles_c;
    tc::mbar_expect_tx(&full[b], MX_TILE_BYTES);
    tc::tma_load_2d(smem + b * MX_TILE_BYTES, &tm_x, &full[b], (int)(tc * MX_TC), (int)(tr * MX_TR));
  };
  // step i quantizes tile blockIdx.x + i * gridDim.x from buffer i % MX_NBUF;
  // the first MX_NBUF - 1 tiles are requested before the loop
  if (t == 0)
    for (int i = 0; i < MX_NBUF - 1; ++i)
      if (blockIdx.x + i * gridDim.x < ntiles) load(blockIdx.x + i * gridDim.x, i);
  uint32_t it = 0;
  for (uint32_t id = blockIdx.x; id < ntiles; id += gridDim.x, ++it) {
    const int b = it % MX_NBUF;
    // the tile MX_NBUF - 1 steps ahead goes into the buffer released by the
    // barrier that closed the last step
    const uint32_t ahead = id + (MX_NBUF - 1) * gridDim.x;
    if (t == 0 && ahead < ntiles) load(ahead, (it + MX_NBUF - 1) % MX_NBUF);
    if (t == 0) (void)tc::mbar_wait(&full[b], (it / MX_NBUF) & 1, abort_flag, status);
    __syncthreads();
    if (*abort_flag) break;
    const uint32_t tr = id / tiles_c, tc = id - tr * tiles_c;
    const int r0 = (int)tr * MX_TR, c0 = (int)tc * MX_TC;
    const uint8_t* tile = smem + b * MX_TILE_BYTES;

    if constexpr (ROWS) {
      // warp w: tile rows w, w + 8, ...; lane l: columns 8l .. 8l + 7 (block l / 4)
      const int blk = lane >> 2, col = c0 + 8 * lane;
      const bool col_ok = col < cols;
#pragma unroll 2
      for (int i = 0; i < MX_TR / 8; ++i) {
        const int rr = 8 * i + warp, row = r0 + rr;
        const uint4 w = *reinterpret_cast<const uint4*>(tile + rr * (MX_TC * 2) + lane * 16);
        uint32_t m = bf16x8_amax_bits(w);
        m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
        m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
        uint32_t byte, rb;
        mx_scale_from_bits(m, byte, rb);
        const uint32_t codes = mx_codes8(w, rb);
        if (row < rows && col_ok) {
          *reinterpret_cast<uint32_t*>(orow.codes + (int64_t)row * (orow.out_cols >> 1) + (col >> 1)) = codes;
          if ((lane & 3) == 0)
            orow.scales[sf_offset(orow.sf_layout, row, (c0 >> 5) + blk, orow.nsf_row, orow.nsf_pad)] = (uint8_t)byte;
        }
      }
    }
    if constexpr (COLS) {
      // thread t: columns 2p, 2p + 1 (p = t % 128) of tile rows 32h .. 32h + 31 (h = t / 128)
      const int p = t & 127, h = t >> 7;
      const uint32_t* tw = reinterpret_cast<const uint32_t*>(tile) + (32 * h) * (MX_TC / 2) + p;
      uint32_t w[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) w[j] = tw[j * (MX_TC / 2)];
      uint32_t m = w[0];
#pragma unroll
      for (int j = 1; j < 32; ++j) m = bf16x2_absmax(m, w[j]);
      m &= 0x7FFF7FFFu;      // both columns' block amax bits
      const int orow0 = c0 + 2 * p, ocol0 = r0 + 32 * h;   // output row (an input column) and first column
      if (ocol0 < rows) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          if (orow0 + e >= cols) break;
          uint32_t byte, rb;
          mx_scale_from_bits(e ? (m >> 16) : (m & 0xFFFFu), byte, rb);
          uint32_t q[4];
#pragma unroll
          for (int k = 0; k < 4; ++k)   // rows 8k .. 8k + 7 of this column: half e of 8 words
            q[k] = e ? mx_codes8_half<1>(&w[8 * k], rb) : mx_codes8_half<0>(&w[8 * k], rb);
          *reinterpret_cast<uint4*>(ocol.codes + (int64_t)(orow0 + e) * (ocol.out_cols >> 1) + (ocol0 >> 1)) =
              make_uint4(q[0], q[1], q[2], q[3]);
          ocol.scales[sf_offset(ocol.sf_layout, orow0 + e, ocol0 >> 5, ocol.nsf_row, ocol.nsf_pad)] = (uint8_t)byte;
        }
      }
    }
    __syncthreads();   // every thread is done with this buffer before it is refilled
  }
  // no copy may be in flight when the CTA exits: after an abort (the loop left
  // at step `it`, after requesting step it + MX_NBUF - 1), wait (bounded) for
  // the copies of steps it .. it + MX_NBUF - 1
  if (t == 0 && *abort_flag) {
    for (uint32_t k = it; k < it + MX_NBUF; ++k)
      if (blockIdx.x + k * gridDim.x < ntiles) tc::mbar_drain_wait(&full[k % MX_NBUF], (k / MX_NBUF) & 1, nullptr);
  }
}

}  // namespace

bool mx_tiled_supported(int dt, int fmt, const QuantOut* orow, const QuantOut* ocol, int64_t rows, int64_t cols,
                        int64_t ldx) {
  if (dt != FP4_DTYPE_BF16 || fmt != FP4_FMT_MXFP4) return false;
  for (const QuantOut* o : {orow, ocol})
    if (o && (o->rounding != FP4_ROUND_RTN || o->rht)) return false;
  if (rows >= (int64_t(1) << 31) || cols >= (int64_t(1) << 31) || rows * cols >= (int64_t(1) << 40)) return false;
  return ldx % 8 == 0;   // the TMA row pitch is a multiple of 16 bytes
}

cudaError_t launch_quant_mx_tiled(const void* x, int64_t rows, int64_t cols, int64_t ldx, const QuantOut* orow,
                                  const QuantOut* ocol, unsigned int* status, int num_sms, cudaStream_t st) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  CUtensorMap tm{};
  if (!tc::make_map_box(&tm, x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, cols, rows, ldx, MX_TC, MX_TR))
    return cudaErrorInvalidValue;
  const int64_t tiles_c = cdiv(cols, MX_TC), nt = cdiv(rows, MX_TR) * tiles_c;
  if (nt >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(nt, (int64_t)num_sms * MX_CTAS_PER_SM));
  QuantOut none{};
  const QuantOut& r = orow ? *orow : none;
  const QuantOut& c = ocol ? *ocol : none;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(mx_tile_kernel<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, MX_SMEM);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(mx_tile_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, MX_SMEM);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(mx_tile_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, MX_SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  if (orow && ocol)
    mx_tile_kernel<true, true><<<grid, MX_THREADS, MX_SMEM, st>>>(tm, (int)rows, (int)cols, (uint32_t)tiles_c,
                                                                  (uint32_t)nt, r, c, status);
  else if (orow)
    mx_tile_kernel<true, false><<<grid, MX_THREADS, MX_SMEM, st>>>(tm, (int)rows, (int)cols, (uint32_t)tiles_c,
                                                                   (uint32_t)nt, r, c, status);
  else
    mx_tile_kernel<false, true><<<grid, MX_THREADS, MX_SMEM, st>>>(tm, (int)rows, (int)cols, (uint32_t)tiles_c,
                                                                   (uint32_t)nt, r, c, status);
  return cudaGetLastError();
}

}  // namespace fp4
