// Inline-PTX wrappers for the sm_103a tensor-core GEMMs: mbarriers, TMA tensor
// copies, tcgen05 MMA / commit / tensor-memory loads and stores, and the
// cluster primitives of the CTA-pair (cta_group::2) kernel.
#pragma once
#include <cuda.h>

#include <cstdint>

#include "fp4_device.cuh"

namespace fp4 {
namespace tc {

constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;  // every device-side wait gives up after 2 s

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// ---- mbarriers (shared::cta addresses unless named otherwise) --------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// arrive on an mbarrier of any CTA of the cluster (shared::cluster address).
// Default (CTA-scope) release: the callers signal the completion of
// tensor-memory accesses that tcgen05.wait::ld / wait::st has already
// waited for, ordered by tcgen05.fence::before_thread_sync; a cluster-scope
// release added 0.5-1 us per arrive under load.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}
// Bounded wait: returns false (and raises the abort flag + status word) when the
// barrier phase does not complete within WAIT_LIMIT_NS or another thread of
// the CTA has already aborted.  The time limit and the abort flag are checked
// only every 1024 polls: reading %globaltimer is slow, and a check after every
// failed poll delays the wake-up.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned int* status) {
  auto poll = [&] { return mbar_try_wait(bar, parity); };
  if (poll()) return true;
  uint64_t t0 = 0;
  for (uint32_t n = 1;; ++n) {
    if (poll()) return true;
    if ((n & 1023u) == 0) {
      if (*abort_flag) return false;
      const uint64_t now = fp4dev::globaltimer_ns();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > WAIT_LIMIT_NS) {
        *abort_flag = 1;
        atomicOr(status, FP4_DEVICE_TIMEOUT);
        return false;
      }
    }
  }
}

// wait (bounded, without the abort flag) until a phase completes; used while
// draining, where the wait must run even after an abort
__device__ __forceinline__ void mbar_drain_wait(uint64_t* bar, uint32_t parity, unsigned int* status) {
  const uint64_t t0 = fp4dev::globaltimer_ns();
  for (uint32_t n = 1; !mbar_try_wait(bar, parity); ++n) {
    if ((n & 1023u) == 0 && fp4dev::globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
      if (status) atomicOr(status, FP4_DEVICE_TIMEOUT);
      break;
    }
  }
}

// named barrier `id` (1..15) over `threads` threads (a multiple of 32)
__device__ __forceinline__ void named_sync(uint32_t id, uint32_t threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ---- cluster ----------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// shared::cluster address of the same object in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t mapa_cluster(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
// all threads of every CTA of the cluster
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---- TMA --------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
          smem_u32(dst)),
      "l"(map), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}
// CTA-pair form: the data lands in this CTA's shared memory, the bytes are
// counted on the mbarrier at `bar_cluster` (a shared::cluster address, here the
// pair leader's barrier)
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map, uint32_t bar_cluster, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], "
      "[%2];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(bar_cluster), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d_pair(void* dst, const CUtensorMap* map, uint32_t bar_cluster, int x, int y,
                                                 int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, "
      "%5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(bar_cluster), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(
          smem_u32(dst)),
      "l"(map), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// ---- tcgen05 ----------------------------------------------------------------
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
// CTA-pair commit: one arrive on the mbarrier at this offset in each CTA of `mask`
__device__ __forceinline__ void tc_commit_pair(uint64_t* bar, uint16_t mask) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                   smem_u32(bar)),
               "h"(mask)
               : "memory");
}

// shared-memory matrix descriptor (K-major, 128-byte swizzle; SBO = 1024 B
// between 8-row groups)
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFF);
  d |= (uint64_t)(1) << 16;                  // leading byte offset (unused with swizzle)
  d |= (uint64_t)(1024 >> 4) << 32;          // stride byte offset
  d |= (uint64_t)1 << 46;                    // descriptor version (sm_100 family)
  d |= (uint64_t)2 << 61;                    // 128-byte swizzle
  return d;
}

// instruction descriptors (M = rows of the MMA: 128 per CTA, 256 for a pair)
__device__ __forceinline__ uint32_t idesc_fp4(bool ue8m0, uint32_t sf_id, int m, int n) {
  uint32_t d = 0;
  d |= sf_id << 4;              // B scale-factor byte
  d |= 1u << 7;                 // A: E2M1
  d |= 1u << 10;                // B: E2M1
  d |= (uint32_t)(n >> 3) << 17;
  d |= (ue8m0 ? 1u : 0u) << 23; // scale type: 1 = UE8M0, 0 = UE4M3
  d |= (uint32_t)(m >> 4) << 24;
  d |= sf_id << 29;             // A scale-factor byte
  return d;
}
// kind::mxf8f6f4 with E4M3 A and B (type code 0) and UE8M0 block scales, one
// scale per 32 K elements (scale_vec::1X): the K = 32 MMA j of a 128-element
// stage takes byte j of each 4-scale group (sf_id)
__device__ __forceinline__ uint32_t idesc_mxf8(uint32_t sf_id, int m, int n) {
  uint32_t d = 0;
  d |= sf_id << 4;              // B scale-factor byte
  d |= (uint32_t)(n >> 3) << 17;
  d |= 1u << 23;                // scale type UE8M0
  d |= (uint32_t)(m >> 4) << 24;
  d |= sf_id << 29;             // A scale-factor byte
  return d;
}
// kind::f8f6f4 with E4M3 A and B (type code 0), F32 accumulation
__device__ __forceinline__ uint32_t idesc_e4m3(int m, int n) {
  uint32_t d = 0;
  d |= 1u << 4;                 // accumulate in F32
  d |= (uint32_t)(n >> 3) << 17;
  d |= (uint32_t)(m >> 4) << 24;
  return d;
}
__device__ __forceinline__ uint32_t idesc_bf16(int m, int n) {
  uint32_t d = 0;
  d |= 1u << 4;                 // accumulate in F32
  d |= 1u << 7;                 // A: BF16
  d |= 1u << 10;                // B: BF16
  d |= (uint32_t)(n >> 3) << 17;
  d |= (uint32_t)(m >> 4) << 24;
  return d;
}

__device__ __forceinline__ void mma_fp4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t acc, bool nvfp4) {
  if (nvfp4) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc), "r"(sfa_tmem), "r"(sfb_tmem));
  } else {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%5], [%6], p;\n}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc), "r"(sfa_tmem), "r"(sfb_tmem));
  }
}
// the CTA-pair MMA (M = 256 across the pair), issued by the pair leader
template <bool NV>
__device__ __forceinline__ void mma_fp4_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t acc) {
  if constexpr (NV) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc), "r"(sfa_tmem), "r"(sfb_tmem));
  } else {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%5], [%6], p;\n}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc), "r"(sfa_tmem), "r"(sfb_tmem));
  }
}
__device__ __forceinline__ void mma_mxf8_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                              uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t acc) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n}" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc), "r"(sfa_tmem), "r"(sfb_tmem));
}
__device__ __forceinline__ void mma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                              uint32_t acc) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void mma_e4m3(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void tmem_ld32_nowait(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 32 lanes x 16 / 8 consecutive 32-bit columns of tensor memory, one register each
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t* v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(v[0]), "r"(v[1]),
               "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Accumulator rows -> coalesced stores.  tcgen05.ld (32x32b) gives lane t the
// 32 words of row t; stored as is, every store instruction would touch 32
// rows.  Exchanging lane bits 4..2 with word bits 4..2 (three butterfly
// stages of shfl.xor; at stage m the lanes with bit m set trade their words j,
// j without bit m, for their partner's words j + m) leaves lane 4b + a holding
// w[4v + k] = (row 4v + a, word column 4b + k): each lane has 4 consecutive
// words of one row for every v, and one 16-byte store per lane covers four
// whole 128-byte row segments per warp instruction.
__device__ __forceinline__ void warp_exchange_hi3(uint32_t* w, int lane) {
#pragma unroll
  for (int m = 16; m >= 4; m >>= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (j & m) continue;
      const uint32_t send = upper ? w[j] : w[j + m];
      const uint32_t recv = __shfl_xor_sync(0xFFFFFFFFu, send, m);
      if (upper)
        w[j] = recv;
      else
        w[j + m] = recv;
    }
  }
}

// ---- host side: tensor maps ---------------------------------------------------
bool make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elem_bytes, int64_t inner, int64_t rows,
              int box_rows);
bool make_sf_map(CUtensorMap* m, const void* base, int64_t group_bytes, int64_t groups, int rows_box, int groups_box);
// 2-D map over a [rows][inner] matrix with a row pitch of `pitch` elements and
// a box of box_inner x box_rows elements, no swizzle
bool make_map_box(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elem_bytes, int64_t inner, int64_t rows,
                  int64_t pitch, int box_inner, int box_rows);

}  // namespace tc
}  // namespace fp4
