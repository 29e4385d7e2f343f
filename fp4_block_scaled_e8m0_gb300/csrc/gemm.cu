// Block-scaled FP4 GEMM on the sm_103a tensor cores (tcgen05).
//
//   C[M,N] = alpha * ( sum_k A[m,k] B[n,k]  +  sum_j Aext[m,j] Bext[n,j] )
//
// The FP4 part is the quantized matmul that carries ">95% of the compute"
// ([msr] §四): E2M1 operands with per-block scales (E8M0 / block 32 = MXFP4,
// E4M3 / block 16 = NVFP4, [lowprec] §1.1) multiplied by
// tcgen05.mma.kind::mxf4nvf4.block_scale, FP32 accumulation in tensor memory.
// The optional bf16 part is the hot-channel compensation tail of [outlier]
// §3.1 ("S" mode: extra K columns in the same GEMM), multiplied by
// tcgen05.mma.kind::f16 into the same accumulator.
//
// Kernel structure (one CTA per SM, persistent over 128 x 256 output tiles):
//   warp 0       TMA producer: A/B code slabs (128-byte K slabs, 128B swizzle)
//                into a 4-stage shared-memory ring, and the scale-factor atoms
//                (3-D tensor maps) into a 5-slot ring, one K step ahead of the
//                slabs: the atoms of step g + 1 are loaded with the slabs of
//                step g, so they are in tensor memory before step g + 1's
//                slabs arrive
//   warp 1       TMEM allocator + MMA issuer (one elected lane): 4 MMAs per
//                stage; tcgen05.commit frees the stage
//   warps 2-5    scale-factor stagers, one per TMEM lane quadrant: copy the
//                stage's scale factors shared -> registers -> tensor memory
//                (tcgen05.st), so the copies stay out of the MMA pipe
//   warps 6-21   epilogue, four per lane quadrant (64 columns each): both
//                32-column tcgen05.ld in flight, one wait, the accumulator
//                is released, then * alpha and store from registers
// Every wait is bounded (globaltimer); a wait that gives up sets the context's
// status word and the CTA drains and exits.
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cstdlib>
#include <mutex>

#include "fp4_device.cuh"
#include "tcgen05.cuh"

namespace fp4 {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int STAGES = 4;
constexpr int KSLAB = 128;                 // bytes of K per stage per row
constexpr int A_TILE = BM * KSLAB;         // 16 KB
constexpr int B_TILE = BN * KSLAB;         // 32 KB
constexpr int SF_A_MAX = 4 * 512;          // NVFP4: 4 atoms of 128 rows x 4 scales
constexpr int SF_B_MAX = (BN / 128) * 4 * 512;
constexpr int SLAB_BYTES = A_TILE + B_TILE;              // one slab stage
constexpr int SF_BYTES = SF_A_MAX + SF_B_MAX;              // one scale slot
constexpr int SF_SLOTS = STAGES + 1;   // the scales run one K step ahead of the slabs
constexpr int SMEM_BYTES = STAGES * SLAB_BYTES + SF_SLOTS * SF_BYTES + 1024 /*align*/ + 256 /*barriers*/;
static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
constexpr int NUM_EPI_WARPS = 16;
constexpr int NUM_THREADS = 32 * (6 + NUM_EPI_WARPS);
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TMEM_SF_BASE = BN;      // scale-factor slots after the accumulator
constexpr uint32_t SF_SLOT_COLS = 48;      // 16 (A) + 32 (B) columns per scale slot
static_assert(TMEM_SF_BASE + SF_SLOTS * SF_SLOT_COLS <= TMEM_COLS, "tensor memory");

struct Params {
  int M, N;
  int k_tiles;        // FP4 K stages (256 elements each)
  int ext_tiles;      // extra K stages: 64 bf16 or 128 E4M3 elements each
  int ext_fp8;        // extra columns are E4M3 (kind::f8f6f4) instead of bf16
  int nvfp4;
  int sf_atoms;       // atoms (128 rows x 4 scales) per stage and 128-row group: 4 NVFP4, 2 MXFP4
  const float* ts_a;
  const float* ts_b;
  void* C;
  int64_t ldc;
  int out_bf16;
  int accumulate;
  unsigned int* status;
  int tiles_m, tiles_n;
  const float* row_scale;      // if set: C (+)= row_scale[m] col_scale[n] acc instead of alpha acc
  const float* col_scale;
};

using namespace tc;

// After warp_exchange_hi3 on 32 columns of fp32 accumulators: lane 4b + a
// writes columns col0 + 4b .. +3 of rows row0 + 4v + a (times alpha; C += when
// accumulating), fp32 or bf16 out.
__device__ __forceinline__ void store_exchanged(const Params& p, const uint32_t* w, int row0, int col0, float alpha,
                                                int lane) {
  const int a = lane & 3, c = col0 + 4 * (lane >> 2);
  if (c >= p.N) return;
  const bool full4 = c + 4 <= p.N;
#pragma unroll
  for (int v = 0; v < 8; ++v) {
    const int row = row0 + 4 * v + a;
    if (row >= p.M) break;
    float x[4];
    if (p.row_scale) {   // per-row and per-column scales (E4M3 extra columns)
      const float rs = p.row_scale[row];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        x[k] = __fmul_rn(__uint_as_float(w[4 * v + k]), __fmul_rn(rs, c + k < p.N ? p.col_scale[c + k] : 0.0f));
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k) x[k] = __fmul_rn(__uint_as_float(w[4 * v + k]), alpha);
    }
    if (p.out_bf16) {
      __nv_bfloat16* q = static_cast<__nv_bfloat16*>(p.C) + (int64_t)row * p.ldc + c;
      if (full4 && !p.accumulate) {
        const __nv_bfloat162 h0 = __floats2bfloat162_rn(x[0], x[1]), h1 = __floats2bfloat162_rn(x[2], x[3]);
        *reinterpret_cast<uint2*>(q) =
            make_uint2(*reinterpret_cast<const uint32_t*>(&h0), *reinterpret_cast<const uint32_t*>(&h1));
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          if (c + k >= p.N) break;
          float y = x[k];
          if (p.accumulate) y = __fadd_rn(__bfloat162float(q[k]), y);
          q[k] = __float2bfloat16_rn(y);
        }
      }
    } else {
      float* q = static_cast<float*>(p.C) + (int64_t)row * p.ldc + c;
      if (full4) {
        float4 y = make_float4(x[0], x[1], x[2], x[3]);
        if (p.accumulate) {
          const float4 o = *reinterpret_cast<const float4*>(q);
          y.x = __fadd_rn(o.x, y.x); y.y = __fadd_rn(o.y, y.y); y.z = __fadd_rn(o.z, y.z); y.w = __fadd_rn(o.w, y.w);
        }
        *reinterpret_cast<float4*>(q) = y;
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          if (c + k >= p.N) break;
          q[k] = p.accumulate ? __fadd_rn(q[k], x[k]) : x[k];
        }
      }
    }
  }
}

// bf16 out without accumulation, 64 columns: word i of w packs columns 2i and
// 2i + 1 (scaled and rounded).  After warp_exchange_hi3 lane 4b + a holds
// columns col0 + 8b .. +7 of rows row0 + 4v + a: one 16-byte store each.
__device__ __forceinline__ void store_exchanged_bf16x2(const Params& p, const uint32_t* w, int row0, int col0,
                                                       int lane) {
  const int a = lane & 3, c = col0 + 8 * (lane >> 2);
  if (c >= p.N) return;
  const bool full8 = c + 8 <= p.N;
#pragma unroll
  for (int v = 0; v < 8; ++v) {
    const int row = row0 + 4 * v + a;
    if (row >= p.M) break;
    uint16_t* q = static_cast<uint16_t*>(p.C) + (int64_t)row * p.ldc + c;
    if (full8) {
      *reinterpret_cast<uint4*>(q) = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (c + k >= p.N) break;
        q[k] = (uint16_t)(w[4 * v + (k >> 1)] >> (16 * (k & 1)));
      }
    }
  }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(NUM_THREADS, 1)
    fp4_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                    const __grid_constant__ CUtensorMap tm_sfa, const __grid_constant__ CUtensorMap tm_sfb,
                    const __grid_constant__ CUtensorMap tm_ax, const __grid_constant__ CUtensorMap tm_bx,
                    const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * SLAB_BYTES + SF_SLOTS * SF_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* sf_ready = empty + STAGES;     // a scale slot is in tensor memory
  uint64_t* sf_full = sf_ready + SF_SLOTS; // a scale slot's atoms landed in shared memory
  uint64_t* acc_full = sf_full + SF_SLOTS;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* drain = acc_empty + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto stage_a = [&](int s) { return smem + s * SLAB_BYTES; };
  auto stage_b = [&](int s) { return smem + s * SLAB_BYTES + A_TILE; };
  auto slot_sfa = [&](int j) { return smem + STAGES * SLAB_BYTES + j * SF_BYTES; };
  auto slot_sfb = [&](int j) { return smem + STAGES * SLAB_BYTES + j * SF_BYTES + SF_A_MAX; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int j = 0; j < SF_SLOTS; ++j) {
      mbar_init(&sf_ready[j], 4);
      mbar_init(&sf_full[j], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, NUM_EPI_WARPS);
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_holder)),
                 "r"(TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  const int num_tiles = p.tiles_m * p.tiles_n;
  const int total_k = p.k_tiles + p.ext_tiles;
  const bool nvfp4 = p.nvfp4 != 0;
  const int atoms = p.sf_atoms;
  const uint32_t sfb_off = nvfp4 ? 16u : 8u;  // B scale columns start after A's in a slot

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      int s = 0, j = 0;
      uint32_t phase = 0, sphase = 0;
      bool ok = true;
      int last_j = -1;                 // the slot of the last scale load issued, and its phase
      uint32_t last_sphase = 0;
      const uint32_t sf_bytes = (uint32_t)atoms * 512;             // one 128-row group, one stage
      // The scale atoms of step (tile, kt) into slot j (rows of 128 bytes
      // inside a 128-row group); the extra-column steps have none and only
      // arrive.  Step g + 1's atoms are issued right after step g's slabs: its
      // slot was last used by step g - 4, the previous user of slab stage
      // g mod 4, whose MMAs have completed once empty[g mod 4] is acquired.
      auto load_sf = [&](int tile, int kt) {
        if (kt < p.k_tiles) {
          const int tm = tile % p.tiles_m, tn = tile / p.tiles_m;
          mbar_expect_tx(&sf_full[j], sf_bytes * (1 + BN / 128));
          tma_load_3d(slot_sfa(j), &tm_sfa, &sf_full[j], 0, kt * atoms * 4, tm);
          tma_load_3d(slot_sfb(j), &tm_sfb, &sf_full[j], 0, kt * atoms * 4, tn * (BN / 128));
        } else {
          mbar_arrive(&sf_full[j]);
        }
        last_j = j;
        last_sphase = sphase;
        if (++j == SF_SLOTS) { j = 0; sphase ^= 1; }
      };
      if ((int)blockIdx.x < num_tiles) load_sf(blockIdx.x, 0);
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        const int tm = tile % p.tiles_m, tn = tile / p.tiles_m;
        for (int kt = 0; kt < total_k; ++kt) {
          if (!mbar_wait(&empty[s], phase ^ 1, abort_flag, p.status)) { ok = false; break; }
          mbar_expect_tx(&full[s], A_TILE + B_TILE);
          if (kt < p.k_tiles) {
            tma_load_2d(stage_a(s), &tm_a, &full[s], kt * KSLAB, tm * BM);
            tma_load_2d(stage_b(s), &tm_b, &full[s], kt * KSLAB, tn * BN);
          } else {
            const int kx = kt - p.k_tiles;
            const int ext_elems = p.ext_fp8 ? 128 : 64;   // 128 bytes of K either way
            tma_load_2d(stage_a(s), &tm_ax, &full[s], kx * ext_elems, tm * BM);
            tma_load_2d(stage_b(s), &tm_bx, &full[s], kx * ext_elems, tn * BN);
          }
          if (kt + 1 < total_k) load_sf(tile, kt + 1);
          else if (tile + (int)gridDim.x < num_tiles) load_sf(tile + gridDim.x, 0);
          if (++s == STAGES) { s = 0; phase ^= 1; }
        }
      }
      // Drain: acquire every stage once more, i.e. wait (bounded) until the last
      // data loaded into each stage has been consumed, and wait for the last
      // scale load to land (after an abort it may not have been consumed); then
      // no load is in flight.
      for (int i = 0; i < STAGES; ++i) {
        const uint64_t t0 = fp4dev::globaltimer_ns();
        for (uint32_t n = 1; !mbar_try_wait(&empty[s], phase ^ 1); ++n) {
          if ((n & 1023u) == 0 && fp4dev::globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
            atomicOr(p.status, FP4_DEVICE_TIMEOUT);
            break;
          }
        }
        if (++s == STAGES) { s = 0; phase ^= 1; }
      }
      if (last_j >= 0) {
        const uint64_t t0 = fp4dev::globaltimer_ns();
        for (uint32_t n = 1; !mbar_try_wait(&sf_full[last_j], last_sphase); ++n) {
          if ((n & 1023u) == 0 && fp4dev::globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
            atomicOr(p.status, FP4_DEVICE_TIMEOUT);
            break;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      int s = 0, j = 0;
      uint32_t phase = 0, sphase = 0, acc_phase = 0;
      bool ok = true;
      // Descriptors are built once: stage s and MMA k only move the start
      // address (16-byte units) by s * SLAB_BYTES / 16 + 2 k, which stays inside
      // the 14-bit field; the instruction descriptors are constants.
      const uint64_t da0 = desc_sw128(smem_u32(stage_a(0))), db0 = desc_sw128(smem_u32(stage_b(0)));
      const uint32_t id_even = idesc_fp4(!nvfp4, 0u, BM, BN), id_odd = idesc_fp4(!nvfp4, nvfp4 ? 0u : 2u, BM, BN);
      const uint32_t id_ext = p.ext_fp8 ? idesc_e4m3(BM, BN) : idesc_bf16(BM, BN);
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        if (!mbar_wait(acc_empty, acc_phase ^ 1, abort_flag, p.status)) { ok = false; break; }
        acc_phase ^= 1;
        tc_fence_after();
        for (int kt = 0; kt < total_k; ++kt) {
          if (!mbar_wait(&full[s], phase, abort_flag, p.status) || !mbar_wait(&sf_ready[j], sphase, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t da = da0 + (uint64_t)(s * (SLAB_BYTES >> 4)), db = db0 + (uint64_t)(s * (SLAB_BYTES >> 4));
          const uint32_t acc0 = kt > 0 ? 1u : 0u;
          if (kt < p.k_tiles) {
            const uint32_t slot = tmem + TMEM_SF_BASE + (uint32_t)j * SF_SLOT_COLS;
            if (nvfp4) {
#pragma unroll
              for (int j = 0; j < 4; ++j)
                mma_fp4(tmem, da + 2 * j, db + 2 * j, id_even, slot + 4 * j, slot + 16 + 8 * j, j > 0 ? 1u : acc0, true);
            } else {
#pragma unroll
              for (int j = 0; j < 4; ++j)
                mma_fp4(tmem, da + 2 * j, db + 2 * j, (j & 1) ? id_odd : id_even, slot + 4 * (j >> 1),
                        slot + 8 + 8 * (j >> 1), j > 0 ? 1u : acc0, false);
            }
          } else {
            // 4 MMAs of 32 bytes of K: 16 bf16 or 32 E4M3 elements each
            if (p.ext_fp8) {
#pragma unroll
              for (int j = 0; j < 4; ++j) mma_e4m3(tmem, da + 2 * j, db + 2 * j, id_ext, j > 0 ? 1u : acc0);
            } else {
#pragma unroll
              for (int j = 0; j < 4; ++j) mma_bf16(tmem, da + 2 * j, db + 2 * j, id_ext, j > 0 ? 1u : acc0);
            }
          }
          tc_commit(&empty[s]);
          if (++s == STAGES) { s = 0; phase ^= 1; }
          if (++j == SF_SLOTS) { j = 0; sphase ^= 1; }
        }
        if (!ok) break;
        tc_commit(acc_full);
      }
      // make sure no MMA is in flight before the allocation is released
      tc_commit(drain);
      const uint64_t t0 = fp4dev::globaltimer_ns();
      for (uint32_t n = 1; !mbar_try_wait(drain, 0); ++n) {
        if ((n & 1023u) == 0 && fp4dev::globaltimer_ns() - t0 > WAIT_LIMIT_NS) break;
      }
    }
  } else if (warp < 6) {
    // ---------------- scale-factor stagers (warps 2..5) ----------------
    // The tensor-memory image equals a 32x128b.warpx4 copy of each 512-byte
    // atom: lane 32q+i, columns c..c+3 of the atom's slot hold the 16 bytes of
    // the atom's shared-memory row i, for every lane quadrant q.
    const int quad = warp & 3;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    int j = 0;                 // scale slot, one per K step in turn
    uint32_t sphase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
      for (int kt = 0; kt < total_k; ++kt) {
        bool got = true;
        if (lane == 0) got = mbar_wait(&sf_full[j], sphase, abort_flag, p.status);
        if (__shfl_sync(0xFFFFFFFFu, got ? 1 : 0, 0) == 0) { ok = false; break; }
        if (kt < p.k_tiles) {
          const uint32_t slot = tmem + lane_base + TMEM_SF_BASE + (uint32_t)j * SF_SLOT_COLS;
          uint32_t v[16];
          if (nvfp4) {
#pragma unroll
            for (int a = 0; a < 4; ++a) {
              const uint4 w = *reinterpret_cast<const uint4*>(slot_sfa(j) + a * 512 + lane * 16);
              v[4 * a] = w.x; v[4 * a + 1] = w.y; v[4 * a + 2] = w.z; v[4 * a + 3] = w.w;
            }
            tmem_st16(slot, v);
            // B: column (2a + g) * 4 holds atom a of 128-row group g; two halves of 16 columns
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {
#pragma unroll
              for (int a2 = 0; a2 < 2; ++a2) {
#pragma unroll
                for (int g = 0; g < 2; ++g) {
                  const int a = hb * 2 + a2;
                  const uint4 w = *reinterpret_cast<const uint4*>(slot_sfb(j) + g * 4 * 512 + a * 512 + lane * 16);
                  const int c = (a2 * 2 + g) * 4;
                  v[c] = w.x; v[c + 1] = w.y; v[c + 2] = w.z; v[c + 3] = w.w;
                }
              }
              tmem_st16(slot + sfb_off + 16 * hb, v);
            }
          } else {
#pragma unroll
            for (int a = 0; a < 2; ++a) {
              const uint4 w = *reinterpret_cast<const uint4*>(slot_sfa(j) + a * 512 + lane * 16);
              v[4 * a] = w.x; v[4 * a + 1] = w.y; v[4 * a + 2] = w.z; v[4 * a + 3] = w.w;
            }
            tmem_st8(slot, v);
#pragma unroll
            for (int a = 0; a < 2; ++a) {
#pragma unroll
              for (int g = 0; g < 2; ++g) {
                const uint4 w = *reinterpret_cast<const uint4*>(slot_sfb(j) + g * 2 * 512 + a * 512 + lane * 16);
                const int c = (a * 2 + g) * 4;
                v[c] = w.x; v[c + 1] = w.y; v[c + 2] = w.z; v[c + 3] = w.w;
              }
            }
            tmem_st16(slot + sfb_off, v);
          }
          tmem_st_wait();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sf_ready[j]);
        if (++j == SF_SLOTS) { j = 0; sphase ^= 1; }
      }
    }
  } else {
    // ---------------- epilogue (warps 6..21) ----------------
    // The accumulator is single-buffered, so the MMAs of the next tile wait
    // until every epilogue warp has its columns in registers: each warp loads
    // all of its 64 columns with one wait and releases before it stores.
    const int quad = warp & 3;               // TMEM lanes 32*quad .. 32*quad+31
    const int slice = (warp - 6) >> 2;       // accumulator columns 64*slice .. +63
    uint32_t acc_phase = 0;
    float alpha = 1.0f;
    if (p.nvfp4) alpha = __fmul_rn(*p.ts_a, *p.ts_b);
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      const int tm = tile % p.tiles_m, tn = tile / p.tiles_m;
      bool ok = true;
      if (lane == 0) ok = mbar_wait(acc_full, acc_phase, abort_flag, p.status);
      ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      acc_phase ^= 1;
      tc_fence_after();
      const int row0 = tm * BM + quad * 32;        // this warp's 32 rows
      const int cbase = slice * 64;
      const int colw = tn * BN + cbase;             // first output column of the slice
      const bool any = row0 < p.M && colw < p.N;   // warp-uniform
      const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)cbase;
      if (p.out_bf16 && !p.accumulate) {
        uint32_t r2[2][32];
        tmem_ld32_nowait(taddr, r2[0]);
        tmem_ld32_nowait(taddr + 32, r2[1]);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_empty);
        if (any) {
          // word i packs columns 2i, 2i+1 of the slice
          uint32_t pk[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const uint32_t* r = r2[i >> 4];
            const __nv_bfloat162 h = __floats2bfloat162_rn(__fmul_rn(__uint_as_float(r[2 * (i & 15)]), alpha),
                                                           __fmul_rn(__uint_as_float(r[2 * (i & 15) + 1]), alpha));
            pk[i] = *reinterpret_cast<const uint32_t*>(&h);
          }
          warp_exchange_hi3(pk, lane);
          store_exchanged_bf16x2(p, pk, row0, colw, lane);
        }
      } else if (!p.accumulate) {
        // fp32 out: both halves in registers, release, then exchange and store
        // each (the accumulator is free for the next tile's MMAs meanwhile)
        uint32_t r2[2][32];
        tmem_ld32_nowait(taddr, r2[0]);
        tmem_ld32_nowait(taddr + 32, r2[1]);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_empty);
        if (any) {
          warp_exchange_hi3(r2[0], lane);
          store_exchanged(p, r2[0], row0, colw, alpha, lane);
          warp_exchange_hi3(r2[1], lane);
          store_exchanged(p, r2[1], row0, colw + 32, alpha, lane);
        }
      } else {
        // C += : 32 columns at a time, so the exchange and the
        // read-modify-write fit the register budget (the release waits for
        // the second load)
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          uint32_t r[32];
          tmem_ld32_nowait(taddr + 32 * h, r);
          tmem_ld_wait();
          if (h == 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty);
          }
          if (any) {
            warp_exchange_hi3(r, lane);
            store_exchanged(p, r, row0, colw + 32 * h, alpha, lane);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS));
  }
}

}  // namespace

namespace tc {
// ---------------------------------------------------------------------------
// host side: tensor maps
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// 2-D map over a row-major [rows][inner] matrix with a box of box_rows x 128 bytes
bool make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elem_bytes, int64_t inner, int64_t rows,
              int box_rows) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(inner * elem_bytes)};
  cuuint32_t box[2] = {(cuuint32_t)(128 / elem_bytes), (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D map over a scale buffer in the MMA layout, seen as [group][row][128 bytes]:
// a box of `rows_box` rows x `groups_box` groups is one stage's atoms of
// `groups_box` consecutive 128-row groups
bool make_sf_map(CUtensorMap* m, const void* base, int64_t group_bytes, int64_t groups, int rows_box, int groups_box) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {128, (cuuint64_t)(group_bytes / 128), (cuuint64_t)groups};
  cuuint64_t strides[2] = {128, (cuuint64_t)group_bytes};
  cuuint32_t box[3] = {128, (cuuint32_t)rows_box, (cuuint32_t)groups_box};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_map_box(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elem_bytes, int64_t inner, int64_t rows,
                  int64_t pitch, int box_inner, int box_rows) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(pitch * elem_bytes)};
  cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace tc

int launch_gemm(const GemmArgs& g, cudaStream_t st) {
  const fp4_operand& A = *g.A;
  const fp4_operand& B = *g.B;
  const int64_t M = A.rows, N = B.rows;
  if (M == 0 || N == 0) return FP4_OK;
  // the FP4 GEMM, alone or with bf16 or MXFP8 extra columns, runs on CTA
  // pairs; E4M3 extra columns, row/column scales and C += stay on the one-SM
  // kernel
  if (g.fp4_part && !g.ext_fp8 && !g.row_scale && !g.accumulate) return launch_gemm_pair(g, st);
  if (g.ext_mx8) return FP4_ERR_UNSUPPORTED;   // MXFP8 extra columns exist on the pair kernel only
  Params p{};
  p.M = (int)M;
  p.N = (int)N;
  p.nvfp4 = A.format == FP4_FMT_NVFP4;
  p.k_tiles = g.fp4_part ? (int)cdiv(A.k, 256) : 0;
  p.ext_fp8 = g.ext_fp8 ? 1 : 0;
  p.ext_tiles = (int)(g.kx / (g.ext_fp8 ? 128 : 64));
  p.row_scale = g.row_scale;
  p.col_scale = g.col_scale;
  p.sf_atoms = p.nvfp4 ? 4 : 2;
  p.ts_a = p.nvfp4 ? A.tensor_scale : nullptr;
  p.ts_b = p.nvfp4 ? B.tensor_scale : nullptr;
  p.C = g.C;
  p.ldc = g.ldc;
  p.out_bf16 = g.out_dtype == FP4_DTYPE_BF16;
  p.accumulate = g.accumulate;
  p.status = g.status;
  p.tiles_m = (int)cdiv(M, BM);
  p.tiles_n = (int)cdiv(N, BN);
  if (p.k_tiles + p.ext_tiles == 0) return FP4_ERR_INVALID_ARG;

  CUtensorMap ta{}, tb{}, tsa{}, tsb{}, tax{}, tbx{};
  bool ok = true;
  if (g.fp4_part) {
    const int64_t group_bytes = (int64_t)128 * nsf_padded(A.k, A.format);
    ok &= tc::make_map(&ta, A.codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, A.k / 2, M, BM);
    ok &= tc::make_map(&tb, B.codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, B.k / 2, N, BN);
    ok &= tc::make_sf_map(&tsa, A.scales, group_bytes, cdiv(M, 128), p.sf_atoms * 4, 1);
    ok &= tc::make_sf_map(&tsb, B.scales, group_bytes, cdiv(N, 128), p.sf_atoms * 4, BN / 128);
  }
  if (g.kx > 0) {
    const CUtensorMapDataType edt = g.ext_fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const int eb = g.ext_fp8 ? 1 : 2;
    ok &= tc::make_map(&tax, g.a_ext, edt, eb, g.kx, M, BM);
    ok &= tc::make_map(&tbx, g.b_ext, edt, eb, g.kx, N, BN);
  }
  if (!g.fp4_part) {  // residual-only GEMM: no FP4 stages, the maps are never read
    ta = tax;
    tb = tbx;
    tsa = tax;
    tsb = tbx;
  }
  if (g.kx == 0) {
    tax = ta;
    tbx = tb;
  }
  if (!ok) return FP4_ERR_CUDA;

  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(fp4_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) != cudaSuccess)
      return FP4_ERR_CUDA;
    attr_set = true;
  }
  const int tiles = p.tiles_m * p.tiles_n;
  const int grid = std::min(tiles, g.num_sms);
  fp4_gemm_kernel<<<grid, NUM_THREADS, SMEM_BYTES, st>>>(ta, tb, tsa, tsb, tax, tbx, p);
  return cudaGetLastError() == cudaSuccess ? FP4_OK : FP4_ERR_CUDA;
}

}  // namespace fp4
