// Block-scaled FP4 GEMM on CTA pairs (tcgen05 cta_group::2), sm_103a.
//
//   C[M,N] = alpha * ( sum_k A[m,k] B[n,k]  +  sum_j Aext[m,j] Bext[n,j] )
//
// (TN, both operands K-major; the optional bf16 part is the hot-channel
// compensation tail of [outlier] §3.1, "S" mode: extra K columns multiplied
// by tcgen05.mma.kind::f16 into the same accumulator)
//
// The quantized matmul that carries ">95% of the compute" ([msr] §四), E2M1
// operands with per-block scales (E8M0 / block 32 = MXFP4, E4M3 / block 16 =
// NVFP4, [lowprec] §1.1), FP32 accumulation in tensor memory.
//
// A cluster of two CTAs on two SMs computes one 256 x 256 output tile: CTA r
// holds rows [128 r, 128 r + 128) of the tile's A rows and of its B rows in
// shared memory, and the pair leader (r = 0) issues one M = 256, N = 256 MMA
// per 64 K elements that reads both CTAs' operands; each CTA's tensor memory
// receives its 128 rows x 256 columns of the accumulator.  Per K step of 256
// elements an SM takes in 32 KB of codes for 2 * 128 * 256 * 256 flop, a
// third less than a one-SM 128 x 256 tile, so the stage ring holds more K
// steps and the tensor pipe waits less for operands.
//
// Warp roles in each CTA of the pair (one CTA per SM, persistent over tiles):
//   warp 0       TMA producer: this CTA's A and B slabs (128-byte K slabs,
//                128-byte swizzle), counted on the pair leader's "full"
//                barrier of the stage, and the stage's scale atoms (this
//                CTA's 128 A rows, all 256 B rows of the tile), counted on its
//                own "sf_full" barrier
//   warp 1       tensor-memory allocation (both CTAs); in the leader one lane
//                issues the pair MMAs and commits each stage to both CTAs'
//                "empty" barriers
//   warps 2-5    scale stagers, one per tensor-memory lane quadrant: copy the
//                stage's scale factors shared -> registers -> this CTA's
//                tensor memory (tcgen05.st) and arrive on the leader's "full"
//                barrier, so the MMA thread waits on one barrier per stage
//   warps 6-21   epilogue: 64 accumulator columns each, both 32-column loads
//                in flight, one wait, the accumulator released to the leader,
//                then * alpha and stores
// Fused-quantize variant (MXFP4, round to nearest, blocks of 32 along K: the
// forward operand of [outlier] §4.1, which needs no tensor-wide amax): A is
// the bf16 activation itself.  The producer also brings 128-row x 128-column
// bf16 half-stages of A into a ring of NXS buffers (TMA), and the sixteen
// epilogue warps, idle while a tile's MMAs run, quantize them ([grad] §2.1,
// E8M0 scale of [lowprec] §1.1) straight into the stage's 128-byte-swizzled A
// slab and its scale atoms (optionally writing the codes out as well); they
// run up to STAGES K steps into the next tile before taking the last tile's
// accumulator.  The stagers then stage the scales as above.
// The scales reach tensor memory through tcgen05.st rather than tcgen05.cp:
// a pair copy of a 512-byte atom held the tensor pipe ~90 cycles (NVFP4 has 12
// atoms per stage next to 4 MMAs of ~136 cycles), the stores run beside the MMAs.
// Every wait is bounded (globaltimer); a wait that gives up sets the context's
// status word and the CTA drains and exits.
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>

#include "fp4_device.cuh"
#include "tcgen05.cuh"

namespace fp4 {
namespace {

using namespace tc;

constexpr int P_BM = 128;                 // A rows per CTA (256 per pair)
constexpr int P_BN = 256;                 // output columns per tile (128 B rows per CTA)
constexpr int P_KSLAB = 128;              // bytes of K per stage per row (256 elements)
constexpr int P_A_TILE = 128 * P_KSLAB;   // 16 KB
constexpr int P_B_TILE = 128 * P_KSLAB;   // 16 KB
constexpr int P_EPI_WARPS = 16;
constexpr int P_THREADS = 32 * (6 + P_EPI_WARPS);
constexpr uint32_t P_TMEM_COLS = 512;

template <bool NV>
struct PairCfg {
  static constexpr int ATOMS = NV ? 4 : 2;                  // scale atoms per 128 rows per stage
  static constexpr int SFA_BYTES = ATOMS * 512;             // this CTA's 128 A rows
  static constexpr int SFB_BYTES = 2 * ATOMS * 512;         // all 256 B rows of the tile
  static constexpr int STAGE = P_A_TILE + P_B_TILE + SFA_BYTES + SFB_BYTES;
  static constexpr int STAGES = NV ? 5 : 6;
  static constexpr uint32_t SLOT_COLS = 12 * ATOMS;         // tensor-memory columns of a stage's scales
  static constexpr int BAR_BYTES = 512;
  static constexpr int SMEM = STAGES * STAGE + BAR_BYTES + 1024;
  static_assert(STAGE % 1024 == 0, "stage alignment (128-byte swizzle)");
  static_assert(SMEM <= 232448, "shared memory per CTA");
  static_assert(P_BN + STAGES * SLOT_COLS <= P_TMEM_COLS, "tensor memory");
};

// fused-quantize variant (MXFP4): fewer stages, and a ring of bf16 A half-stages
struct FuseCfg {
  // two K stages of codes and four bf16 half-stages: a half-stage's buffer is
  // refilled while the next stage is quantized (with three half-stages the
  // refill of a stage's second half started only when the stage before it
  // was done, and each stage waited out a whole TMA latency)
  static constexpr int STAGES = 2;
  static constexpr int XS_COLS = 128;                     // bf16 elements of K per half-stage
  static constexpr int XS_BYTES = 128 * XS_COLS * 2;      // 128 rows: 32 KB
  static constexpr int NXS = 4;
  static constexpr int SMEM = STAGES * PairCfg<false>::STAGE + NXS * XS_BYTES + PairCfg<false>::BAR_BYTES + 1024;
  static_assert(SMEM <= 232448, "shared memory per CTA");
};

// Tile order: groups of up to P_GROUP_M row tiles; inside a group the row tile
// runs fastest and the column tile next, so that the pairs working at one time
// share a few A row blocks and B column blocks and re-read them from L2 (with
// the row tile fastest over the whole of M, the output stream evicted A
// between waves: 7x the operand bytes came from DRAM)
constexpr int P_GROUP_M = 16;
__device__ __forceinline__ void tile_coords(int tile, int tiles_m, int tiles_n, int& tm, int& tn) {
  const int per_group = P_GROUP_M * tiles_n;
  const int g = tile / per_group;
  const int first_m = g * P_GROUP_M;
  const int gm = min(P_GROUP_M, tiles_m - first_m);
  const int local = tile - g * per_group;
  tm = first_m + local % gm;
  tn = local / gm;
}

struct PairParams {
  int M, N;
  int k_tiles;        // FP4 K stages (256 elements each)
  int ext_tiles;      // extra bf16 K stages (64 elements each) after the FP4 ones
  const float* ts_a;  // NVFP4 tensor scales (alpha = ts_a * ts_b), null for MXFP4
  const float* ts_b;
  void* C;
  int64_t ldc;
  unsigned int* status;
  int tiles_m, tiles_n;   // 256 x 256 tiles
  // fused-quantize variant: the quantized A written out (null: not written)
  uint8_t* qa_codes;      // [M][K/2]
  uint8_t* qa_scales;     // MMA layout, atoms of 128 rows x 4 scales
  int K;
  int sf_groups;          // scale atoms per 128 rows in qa_scales (K padded to 256, / 128)
  int ext_mx8;            // extra columns are MXFP8 (128 per stage, one scale atom per 128 rows)
};

template <bool NV, bool BF16_OUT, bool FUSE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(P_THREADS, 1)
    fp4_gemm_pair_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                         const __grid_constant__ CUtensorMap tm_sfa, const __grid_constant__ CUtensorMap tm_sfb,
                         const __grid_constant__ CUtensorMap tm_ax, const __grid_constant__ CUtensorMap tm_bx,
                         const __grid_constant__ CUtensorMap tm_sfax, const __grid_constant__ CUtensorMap tm_sfbx,
                         const PairParams p) {
  static_assert(!(NV && FUSE), "the fused quantizer forms MXFP4 operands");
  using Cfg = PairCfg<NV>;
  constexpr int STAGES = FUSE ? FuseCfg::STAGES : Cfg::STAGES;
  constexpr int NXS = FUSE ? FuseCfg::NXS : 0;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* xs_base = smem + STAGES * Cfg::STAGE;                               // bf16 A half-stages (fused)
  uint64_t* full = reinterpret_cast<uint64_t*>(xs_base + NXS * FuseCfg::XS_BYTES);   // leader: slabs landed, scales staged
  uint64_t* empty = full + STAGES;                                             // stage consumed by the MMAs
  uint64_t* sf_full = empty + STAGES;                                          // this CTA's scale atoms landed
  uint64_t* acc_full = sf_full + STAGES;
  uint64_t* acc_empty = acc_full + 1;                                          // leader: both epilogues done
  uint64_t* drain = acc_empty + 1;
  uint64_t* xs_full = drain + 1;                                               // fused: bf16 half-stage landed
  uint64_t* xs_empty = xs_full + NXS;                                          // fused: half-stage quantized
  uint64_t* q_done = xs_empty + NXS;                                           // fused: stage's A codes and scales written
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(q_done + (FUSE ? STAGES : 0));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  auto stage_a = [&](int s) { return smem + s * Cfg::STAGE; };
  auto stage_b = [&](int s) { return smem + s * Cfg::STAGE + P_A_TILE; };
  auto stage_sfa = [&](int s) { return smem + s * Cfg::STAGE + P_A_TILE + P_B_TILE; };
  auto stage_sfb = [&](int s) { return smem + s * Cfg::STAGE + P_A_TILE + P_B_TILE + Cfg::SFA_BYTES; };
  auto stage_x = [&](int x) { return xs_base + x * FuseCfg::XS_BYTES; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1 + 8);              // the leader's producer + 4 stager warps in each CTA
      mbar_init(&empty[s], 1);
      mbar_init(&sf_full[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 2 * P_EPI_WARPS);    // every epilogue warp of both CTAs
    mbar_init(drain, 1);
    for (int x = 0; x < NXS; ++x) {
      mbar_init(&xs_full[x], 1);
      mbar_init(&xs_empty[x], P_EPI_WARPS);    // the quantizing (epilogue) warps
    }
    if (FUSE)
      for (int s = 0; s < STAGES; ++s) mbar_init(&q_done[s], P_EPI_WARPS);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_holder)),
                 "r"(P_TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
  }
  tc_fence_before();
  cluster_sync();            // barriers initialised and tensor memory allocated in both CTAs
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  // the leader's barriers as seen from this CTA
  const uint32_t full_l = mapa_cluster(&full[0], 0);
  const uint32_t acc_empty_l = mapa_cluster(acc_empty, 0);

  const int num_tiles = p.tiles_m * p.tiles_n;
  const int total_k = p.k_tiles + p.ext_tiles;
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      int s = 0, x = 0;
      uint32_t phase = 0, xphase = 0;
      bool ok = true;
      for (int tile = pair; tile < num_tiles && ok; tile += npairs) {
        int tm, tn;
        tile_coords(tile, p.tiles_m, p.tiles_n, tm, tn);
        const int row_a = tm * 256 + (int)rank * 128, row_b = tn * 256 + (int)rank * 128;
        for (int kt = 0; kt < total_k; ++kt) {
          if constexpr (FUSE) {
            // the stage's two bf16 half-stages of this CTA's A rows (zero fill
            // beyond M and K), each into the ring buffer the stagers released
            for (int h = 0; h < 2 && ok; ++h) {
              if (!mbar_wait(&xs_empty[x], xphase ^ 1, abort_flag, p.status)) { ok = false; break; }
              mbar_expect_tx(&xs_full[x], FuseCfg::XS_BYTES);
              tma_load_2d(stage_x(x), &tm_a, &xs_full[x], kt * 256 + h * FuseCfg::XS_COLS, row_a);
              if (++x == NXS) { x = 0; xphase ^= 1; }
            }
            if (!ok) break;
            if (!mbar_wait(&empty[s], phase ^ 1, abort_flag, p.status)) { ok = false; break; }
            if (leader) mbar_expect_tx(&full[s], 2 * P_B_TILE);
            tma_load_2d_pair(stage_b(s), &tm_b, full_l + (uint32_t)s * 8u, kt * P_KSLAB, row_b);
            mbar_expect_tx(&sf_full[s], Cfg::SFB_BYTES);
            tma_load_3d(stage_sfb(s), &tm_sfb, &sf_full[s], 0, kt * Cfg::ATOMS * 4, 2 * tn);
            if (++s == STAGES) { s = 0; phase ^= 1; }
            continue;
          }
          if (!mbar_wait(&empty[s], phase ^ 1, abort_flag, p.status)) { ok = false; break; }
          if (leader) mbar_expect_tx(&full[s], 2 * (P_A_TILE + P_B_TILE));
          const uint32_t fb = full_l + (uint32_t)s * 8u;
          if (kt < p.k_tiles) {
            tma_load_2d_pair(stage_a(s), &tm_a, fb, kt * P_KSLAB, row_a);
            tma_load_2d_pair(stage_b(s), &tm_b, fb, kt * P_KSLAB, row_b);
            mbar_expect_tx(&sf_full[s], Cfg::SFA_BYTES + Cfg::SFB_BYTES);
            tma_load_3d(stage_sfa(s), &tm_sfa, &sf_full[s], 0, kt * Cfg::ATOMS * 4, 2 * tm + (int)rank);
            tma_load_3d(stage_sfb(s), &tm_sfb, &sf_full[s], 0, kt * Cfg::ATOMS * 4, 2 * tn);
          } else if (p.ext_mx8) {
            // MXFP8 extra columns: 128 per stage (128 bytes of K) and their scale
            // atoms (this CTA's 128 A rows, the tile's 256 B rows)
            const int xt = kt - p.k_tiles;
            tma_load_2d_pair(stage_a(s), &tm_ax, fb, xt * 128, row_a);
            tma_load_2d_pair(stage_b(s), &tm_bx, fb, xt * 128, row_b);
            mbar_expect_tx(&sf_full[s], 512 + 1024);
            tma_load_3d(stage_sfa(s), &tm_sfax, &sf_full[s], 0, xt * 4, 2 * tm + (int)rank);
            tma_load_3d(stage_sfb(s), &tm_sfbx, &sf_full[s], 0, xt * 4, 2 * tn);
          } else {
            // extra bf16 columns: 64 per stage (128 bytes of K), no scales
            const int kx = (kt - p.k_tiles) * 64;
            tma_load_2d_pair(stage_a(s), &tm_ax, fb, kx, row_a);
            tma_load_2d_pair(stage_b(s), &tm_bx, fb, kx, row_b);
            mbar_arrive(&sf_full[s]);
          }
          if (++s == STAGES) { s = 0; phase ^= 1; }
        }
      }
      // drain: wait until every stage loaded has been consumed, so that no copy
      // is in flight when the CTA exits
      for (int i = 0; i < STAGES; ++i) {
        mbar_drain_wait(&empty[s], phase ^ 1, p.status);
        if (++s == STAGES) { s = 0; phase ^= 1; }
      }
      // and until every bf16 half-stage requested has landed
      for (int i = 0; i < NXS; ++i) {
        mbar_drain_wait(&xs_full[x], xphase ^ 1, p.status);
        if (++x == NXS) { x = 0; xphase ^= 1; }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (pair leader) ----------------
    if (leader && lane == 0) {
      int s = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      const uint64_t da0 = desc_sw128(smem_u32(stage_a(0))), db0 = desc_sw128(smem_u32(stage_b(0)));
      const uint32_t id_even = idesc_fp4(!NV, 0u, 256, P_BN), id_odd = idesc_fp4(!NV, NV ? 0u : 2u, 256, P_BN);
      const uint32_t id_ext = idesc_bf16(256, P_BN);
      for (int tile = pair; tile < num_tiles && ok; tile += npairs) {
        if (!mbar_wait(acc_empty, acc_phase ^ 1, abort_flag, p.status)) { ok = false; break; }
        acc_phase ^= 1;
        tc_fence_after();
        for (int kt = 0; kt < total_k; ++kt) {
          if (!mbar_wait(&full[s], phase, abort_flag, p.status)) { ok = false; break; }
          tc_fence_after();
          const uint64_t da = da0 + (uint64_t)(s * (Cfg::STAGE >> 4)), db = db0 + (uint64_t)(s * (Cfg::STAGE >> 4));
          const uint32_t slot = tmem + P_BN + (uint32_t)s * Cfg::SLOT_COLS;
          const uint32_t acc0 = kt > 0 ? 1u : 0u;
          if (kt < p.k_tiles) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              // scale columns of 64-element K chunk j: NVFP4 one atom per chunk,
              // MXFP4 one atom per two chunks (bytes 0-1 / 2-3 chosen by the
              // instruction descriptor); B's two 128-row groups side by side
              const uint32_t a_col = NV ? 4u * j : 4u * (j >> 1);
              const uint32_t b_col = 4u * Cfg::ATOMS + (NV ? 8u * j : 8u * (j >> 1));
              mma_fp4_pair<NV>(tmem, da + 2 * j, db + 2 * j, (!NV && (j & 1)) ? id_odd : id_even, slot + a_col,
                               slot + b_col, j > 0 ? 1u : acc0);
            }
          } else if (p.ext_mx8) {
            // 4 MXFP8 MMAs of 32 K elements (32 bytes), scale byte j of the
            // stage's atoms: A's at the slot's first columns, B's two 128-row
            // groups where the FP4 stages keep B's
#pragma unroll
            for (int j = 0; j < 4; ++j)
              mma_mxf8_pair(tmem, da + 2 * j, db + 2 * j, idesc_mxf8((uint32_t)j, 256, P_BN), slot,
                            slot + 4u * Cfg::ATOMS, j > 0 ? 1u : acc0);
          } else {
            // 4 bf16 MMAs of 16 K elements (32 bytes) into the same accumulator
#pragma unroll
            for (int j = 0; j < 4; ++j) mma_bf16_pair(tmem, da + 2 * j, db + 2 * j, id_ext, j > 0 ? 1u : acc0);
          }
          tc_commit_pair(&empty[s], 0x3);
          if (++s == STAGES) { s = 0; phase ^= 1; }
        }
        if (!ok) break;
        tc_commit_pair(acc_full, 0x3);
      }
      // no MMA may be in flight when the allocation is released
      tc_commit_pair(drain, 0x1);
      mbar_drain_wait(drain, 0, nullptr);
    }
  } else if (warp < 6) {
    // ---------------- scale stagers (warps 2..5) ----------------
    // The tensor-memory image of each 512-byte atom equals a 32x128b.warpx4
    // copy: lane 32q + i, columns c..c+3 of the atom's place hold the 16 bytes
    // of the atom's shared-memory row i, for every lane quadrant q.  A stage's
    // slot: A's atoms (4 columns each), then for each atom of B its two
    // 128-row groups side by side (columns 8a + 4g after A's).
    const int quad = warp & 3;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    int s = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int tile = pair; tile < num_tiles && ok; tile += npairs) {
      int tm, tn;
      tile_coords(tile, p.tiles_m, p.tiles_n, tm, tn);
      for (int kt = 0; kt < total_k; ++kt) {
        // one lane polls, the four stager warps meet at a named barrier
        if (warp == 2 && lane == 0) {
          (void)mbar_wait(&sf_full[s], phase, abort_flag, p.status);
          if constexpr (FUSE) (void)mbar_wait(&q_done[s], phase, abort_flag, p.status);   // A's scale atoms
        }
        named_sync(1, 4 * 32);
        if (*abort_flag) { ok = false; break; }
        if constexpr (FUSE) {
          const int rt = 2 * tm + (int)rank;          // 128-row tile of A
          if (p.qa_scales != nullptr && tn == 0 && rt * 128 < p.M) {
            // the stage's two atoms are contiguous in the MMA layout: 8 bytes a thread
            const int t = threadIdx.x - 64;
            *reinterpret_cast<uint2*>(p.qa_scales + ((int64_t)rt * p.sf_groups + 2 * kt) * 512 + t * 8) =
                *reinterpret_cast<const uint2*>(stage_sfa(s) + t * 8);
          }
        }
        const uint32_t slot = tmem + lane_base + P_BN + (uint32_t)s * Cfg::SLOT_COLS;
        uint32_t v[16];
        if (kt >= p.k_tiles) {
          if (p.ext_mx8) {
            // MXFP8 extra columns: A's one atom at the slot's columns 0-3, B's
            // two 128-row groups at 4 * ATOMS + 0-7
            const uint4 wa = *reinterpret_cast<const uint4*>(stage_sfa(s) + lane * 16);
            v[0] = wa.x; v[1] = wa.y; v[2] = wa.z; v[3] = wa.w;
            v[4] = v[5] = v[6] = v[7] = 0u;
            tmem_st8(slot, v);
            const uint4 w0 = *reinterpret_cast<const uint4*>(stage_sfb(s) + lane * 16);
            const uint4 w1 = *reinterpret_cast<const uint4*>(stage_sfb(s) + 512 + lane * 16);
            v[0] = w0.x; v[1] = w0.y; v[2] = w0.z; v[3] = w0.w;
            v[4] = w1.x; v[5] = w1.y; v[6] = w1.z; v[7] = w1.w;
            tmem_st8(slot + 4u * Cfg::ATOMS, v);
            tmem_st_wait();
            tc_fence_before();
          }
          // extra bf16 columns: no scales to stage
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(full_l + (uint32_t)s * 8u);
          if (++s == STAGES) { s = 0; phase ^= 1; }
          continue;
        }
#pragma unroll
        for (int a = 0; a < Cfg::ATOMS; ++a) {
          const uint4 w = *reinterpret_cast<const uint4*>(stage_sfa(s) + a * 512 + lane * 16);
          v[4 * a] = w.x; v[4 * a + 1] = w.y; v[4 * a + 2] = w.z; v[4 * a + 3] = w.w;
        }
        if constexpr (NV) tmem_st16(slot, v);
        else tmem_st8(slot, v);
#pragma unroll
        for (int piece = 0; piece < Cfg::ATOMS / 2; ++piece) {
#pragma unroll
          for (int a2 = 0; a2 < 2; ++a2) {
#pragma unroll
            for (int g = 0; g < 2; ++g) {
              const int a = piece * 2 + a2;
              const uint4 w =
                  *reinterpret_cast<const uint4*>(stage_sfb(s) + g * Cfg::ATOMS * 512 + a * 512 + lane * 16);
              const int c = (a2 * 2 + g) * 4;
              v[c] = w.x; v[c + 1] = w.y; v[c + 2] = w.z; v[c + 3] = w.w;
            }
          }
          tmem_st16(slot + 4u * Cfg::ATOMS + 16u * piece, v);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(full_l + (uint32_t)s * 8u);
        if (++s == STAGES) { s = 0; phase ^= 1; }
      }
    }
  } else {
    // ---------------- epilogue (warps 6..21) ----------------
    const int quad = warp & 3;               // tensor-memory lanes 32*quad .. +31
    const int slice = (warp - 6) >> 2;       // accumulator columns 64*slice .. +63
    uint32_t acc_phase = 0;
    float alpha = 1.0f;
    if (NV) alpha = __fmul_rn(*p.ts_a, *p.ts_b);
    // one tile's accumulator -> C; false when the kernel gave up a wait
    auto epilogue = [&](int tile) -> bool {
      int tm, tn;
      tile_coords(tile, p.tiles_m, p.tiles_n, tm, tn);
      // one lane polls, the sixteen epilogue warps meet at a named barrier
      if (warp == 6 && lane == 0) (void)mbar_wait(acc_full, acc_phase, abort_flag, p.status);
      named_sync(2, P_EPI_WARPS * 32);
      if (*abort_flag) return false;
      acc_phase ^= 1;
      tc_fence_after();
      const int row0 = tm * 256 + (int)rank * 128 + quad * 32;   // this warp's 32 rows
      const int colw = tn * P_BN + slice * 64;                    // first output column of the slice
      const bool any = row0 < p.M && colw < p.N;                  // warp-uniform
      const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(slice * 64);
      uint32_t r2[2][32];
      tmem_ld32_nowait(taddr, r2[0]);
      tmem_ld32_nowait(taddr + 32, r2[1]);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc_empty_l);
      if (!any) return true;
      if constexpr (BF16_OUT) {
        // word i packs columns 2i, 2i + 1 of the slice; after the exchange lane
        // 4b + a holds columns colw + 8b .. +7 of rows row0 + 4v + a
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const uint32_t* r = r2[i >> 4];
          const __nv_bfloat162 h = __floats2bfloat162_rn(__fmul_rn(__uint_as_float(r[2 * (i & 15)]), alpha),
                                                         __fmul_rn(__uint_as_float(r[2 * (i & 15) + 1]), alpha));
          pk[i] = *reinterpret_cast<const uint32_t*>(&h);
        }
        warp_exchange_hi3(pk, lane);
        const int a = lane & 3, c = colw + 8 * (lane >> 2);
        if (c < p.N) {
          const bool full8 = c + 8 <= p.N;
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            const int row = row0 + 4 * v + a;
            if (row >= p.M) break;
            uint16_t* q = static_cast<uint16_t*>(p.C) + (int64_t)row * p.ldc + c;
            if (full8) {
              *reinterpret_cast<uint4*>(q) = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
            } else {
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                if (c + k >= p.N) break;
                q[k] = (uint16_t)(pk[4 * v + (k >> 1)] >> (16 * (k & 1)));
              }
            }
          }
        }
      } else {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t* w = r2[h];
          warp_exchange_hi3(w, lane);
          const int a = lane & 3, c = colw + 32 * h + 4 * (lane >> 2);
          if (c >= p.N) continue;
          const bool full4 = c + 4 <= p.N;
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            const int row = row0 + 4 * v + a;
            if (row >= p.M) break;
            float* q = static_cast<float*>(p.C) + (int64_t)row * p.ldc + c;
            float x[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) x[k] = __fmul_rn(__uint_as_float(w[4 * v + k]), alpha);
            if (full4) {
              *reinterpret_cast<float4*>(q) = make_float4(x[0], x[1], x[2], x[3]);
            } else {
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                if (c + k >= p.N) break;
                q[k] = x[k];
              }
            }
          }
        }
      }
      return true;
    };
    if constexpr (!FUSE) {
      for (int tile = pair; tile < num_tiles; tile += npairs)
        if (!epilogue(tile)) break;
    } else {
      // Quantize A for the MMAs: warp e = warp - 6 takes rows 8e .. 8e + 7 of
      // this CTA's 128, two rows per step (lanes 0-15 and 16-31), each lane 8
      // elements of a 128-element half-stage; 4 lanes share a 32-element block.
      // The last tile's accumulator is taken after the first STAGES K steps of
      // the next tile are quantized: those need only the last tile's MMAs to
      // have released their slots, and the next tile's first MMA needs the
      // accumulator.
      const int e = warp - 6;
      const int cl = lane & 15;
      const int ahead = min(STAGES, p.k_tiles);
      int s = 0, x = 0, prev = -1;
      uint32_t phase = 0, xphase = 0;
      bool ok = true;
      for (int tile = pair; tile < num_tiles && ok; tile += npairs) {
        int tm, tn;
        tile_coords(tile, p.tiles_m, p.tiles_n, tm, tn);
        const int grow0 = tm * 256 + (int)rank * 128;
        for (int kt = 0; kt < p.k_tiles; ++kt) {
          const int x1 = x + 1 == NXS ? 0 : x + 1;
          if (warp == 6 && lane == 0) {
            // the slot is free once its B scales were requested (the producer
            // waits for the MMAs to release it first); the stage's two bf16
            // half-stages have landed
            (void)mbar_wait(&sf_full[s], phase, abort_flag, p.status);
            (void)mbar_wait(&xs_full[x], xphase, abort_flag, p.status);
            (void)mbar_wait(&xs_full[x1], x1 == 0 ? xphase ^ 1 : xphase, abort_flag, p.status);
          }
          named_sync(2, P_EPI_WARPS * 32);
          if (*abort_flag) { ok = false; break; }
          uint8_t* a_slab = stage_a(s);
          uint8_t* sfa = stage_sfa(s);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint8_t* xs = stage_x(h == 0 ? x : x1);
            const int kcol = kt * 256 + h * FuseCfg::XS_COLS + 8 * cl;   // first element of the lane's 8
            const bool write_codes = p.qa_codes != nullptr && tn == 0 && kcol < p.K;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int r = 8 * e + 2 * i + (lane >> 4);                  // row of this CTA's 128
              const uint4 w = *reinterpret_cast<const uint4*>(xs + r * (FuseCfg::XS_COLS * 2) + cl * 16);
              uint32_t m = fp4dev::bf16x8_amax_bits(w);
              m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
              m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
              uint32_t byte, rb;
              fp4dev::mx_scale_from_bits(m, byte, rb);
              const uint32_t codes = fp4dev::mx_codes8(w, rb);
              // 128-byte swizzle: 16-byte chunk c of row r sits at chunk c ^ (r % 8)
              const int chunk = (h * 4 + (cl >> 2)) ^ (r & 7);
              *reinterpret_cast<uint32_t*>(a_slab + r * P_KSLAB + chunk * 16 + (cl & 3) * 4) = codes;
              // scale of block 4h + cl/4 of the stage: atom h, (r % 32) * 16 + ((r / 32) % 4) * 4 + cl / 4
              if ((cl & 3) == 0) sfa[h * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (cl >> 2)] = (uint8_t)byte;
              if (write_codes && grow0 + r < p.M)
                *reinterpret_cast<uint32_t*>(p.qa_codes + (int64_t)(grow0 + r) * (p.K >> 1) + (kcol >> 1)) = codes;
            }
          }
          // the codes were written through the generic proxy; the MMA reads
          // them through the async proxy
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&xs_empty[x]);
            mbar_arrive(&xs_empty[x1]);
            mbar_arrive(&q_done[s]);
          }
          for (int j = 0; j < 2; ++j)
            if (++x == NXS) { x = 0; xphase ^= 1; }
          if (++s == STAGES) { s = 0; phase ^= 1; }
          if (prev >= 0 && kt == ahead - 1) {
            if (!epilogue(prev)) { ok = false; break; }
            prev = -1;
          }
        }
        if (ok) prev = tile;
      }
      if (ok && prev >= 0) (void)epilogue(prev);
    }
  }

  tc_fence_before();
  cluster_sync();            // no peer access (remote arrives, commits, MMAs) after this point
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(P_TMEM_COLS));
  }
}

template <bool NV, bool BF16_OUT, bool FUSE = false>
int launch_pair(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tsa, const CUtensorMap& tsb,
                const CUtensorMap& tax, const CUtensorMap& tbx, const CUtensorMap& tsax, const CUtensorMap& tsbx,
                const PairParams& p, int num_sms, cudaStream_t st) {
  constexpr int SMEM = FUSE ? FuseCfg::SMEM : PairCfg<NV>::SMEM;
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(fp4_gemm_pair_kernel<NV, BF16_OUT, FUSE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM) != cudaSuccess)
      return FP4_ERR_CUDA;
    attr_set = true;
  }
  const int tiles = p.tiles_m * p.tiles_n;
  const int pairs = std::max(1, std::min(tiles, num_sms / 2));
  fp4_gemm_pair_kernel<NV, BF16_OUT, FUSE><<<2 * pairs, P_THREADS, SMEM, st>>>(ta, tb, tsa, tsb, tax, tbx, tsax, tsbx,
                                                                              p);
  return cudaGetLastError() == cudaSuccess ? FP4_OK : FP4_ERR_CUDA;
}

}  // namespace

int launch_gemm_pair(const GemmArgs& g, cudaStream_t st) {
  const fp4_operand& B = *g.B;
  const bool fuse = g.quant_a;                    // A = the bf16 activation, quantized in the kernel
  const int64_t M = fuse ? g.m : g.A->rows, N = B.rows, K = B.k;
  if (M == 0 || N == 0) return FP4_OK;
  const bool nv = B.format == FP4_FMT_NVFP4;
  if (fuse && (nv || g.kx > 0)) return FP4_ERR_UNSUPPORTED;
  PairParams p{};
  p.M = (int)M;
  p.N = (int)N;
  p.k_tiles = (int)cdiv(K, 256);
  p.ts_a = nv ? g.A->tensor_scale : nullptr;
  p.ts_b = nv ? B.tensor_scale : nullptr;
  p.C = g.C;
  p.ldc = g.ldc;
  p.status = g.status;
  p.tiles_m = (int)cdiv(M, 256);
  p.tiles_n = (int)cdiv(N, P_BN);
  p.ext_mx8 = g.ext_mx8 ? 1 : 0;
  p.ext_tiles = (int)(g.kx / (g.ext_mx8 ? 128 : 64));
  p.qa_codes = g.qa_codes;
  p.qa_scales = g.qa_scales;
  p.K = (int)K;
  p.sf_groups = (int)(nsf_padded(K, B.format) / 4);
  if (p.k_tiles == 0) return FP4_ERR_INVALID_ARG;
  const int atoms = nv ? 4 : 2;
  const int64_t group_bytes = (int64_t)128 * nsf_padded(K, B.format);
  CUtensorMap ta{}, tb{}, tsa{}, tsb{};
  bool ok = tc::make_map(&tb, B.codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K / 2, N, 128);
  ok &= tc::make_sf_map(&tsb, B.scales, group_bytes, cdiv(N, 128), atoms * 4, 2);
  if (fuse) {
    // bf16 A in 128-column x 128-row boxes; the A scale map is never read
    ok &= tc::make_map_box(&ta, g.x_bf16, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, K, M, g.ldx, FuseCfg::XS_COLS, 128);
    tsa = tsb;
  } else {
    ok &= tc::make_map(&ta, g.A->codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K / 2, M, P_BM);
    ok &= tc::make_sf_map(&tsa, g.A->scales, group_bytes, cdiv(M, 128), atoms * 4, 1);
  }
  CUtensorMap tax = ta, tbx = tb, tsax = tsb, tsbx = tsb;   // never read without extra columns
  if (g.kx > 0 && g.ext_mx8) {
    // E4M3 codes [rows][kx] and E8M0 scales in the MMA layout (kx / 32 per row)
    ok &= tc::make_map(&tax, g.a_ext, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, g.kx, M, 128);
    ok &= tc::make_map(&tbx, g.b_ext, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, g.kx, N, 128);
    ok &= tc::make_sf_map(&tsax, g.a_ext_sf, 4 * g.kx, cdiv(M, 128), 4, 1);
    ok &= tc::make_sf_map(&tsbx, g.b_ext_sf, 4 * g.kx, cdiv(N, 128), 4, 2);
  } else if (g.kx > 0) {
    ok &= tc::make_map(&tax, g.a_ext, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, g.kx, M, 128);
    ok &= tc::make_map(&tbx, g.b_ext, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, g.kx, N, 128);
  }
  if (!ok) return FP4_ERR_CUDA;
  const bool bf16 = g.out_dtype == FP4_DTYPE_BF16;
  if (fuse) return bf16 ? launch_pair<false, true, true>(ta, tb, tsa, tsb, tax, tbx, tsax, tsbx, p, g.num_sms, st)
                        : launch_pair<false, false, true>(ta, tb, tsa, tsb, tax, tbx, tsax, tsbx, p, g.num_sms, st);
  if (nv) return bf16 ? launch_pair<true, true>(ta, tb, tsa, tsb, tax, tbx, tsax, tsbx, p, g.num_sms, st)
                      : launch_pair<true, false>(ta, tb, tsa, tsb, tax, tbx, tsax, tsbx, p, g.num_sms, st);
  return bf16 ? launch_pair<false, true>(ta, tb, tsa, tsb, tax, tbx, tsax, tsbx, p, g.num_sms, st)
              : launch_pair<false, false>(ta, tb, tsa, tsb, tax, tbx, tsax, tsbx, p, g.num_sms, st);
}

}  // namespace fp4
