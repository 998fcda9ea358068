// Fifth-generation tensor core (tcgen05) primitives for the block-scaled
// NVFP4 expert GEMMs (sm_103a): tensor-memory allocation, shared-memory
// matrix descriptors, the kind::mxf4nvf4 MMA with E4M3 scale vectors of 16
// elements, shared -> tensor memory copies of the scale factors, commit to
// an mbarrier, and tensor-memory loads for the epilogue.  Inline PTX only.
//
// Conventions used throughout (one CTA, cta_group::1):
//  * Operands live in shared memory in the K-major layout without swizzle:
//    "core matrices" of 8 rows x 16 bytes (32 E2M1 elements), 128
//    contiguous bytes each, row r of a core matrix at 16 r.  The byte
//    distance between core matrices adjacent along K is the descriptor's
//    leading-dimension offset (LBO), between core matrices adjacent along
//    M / N (8-row groups) its stride-dimension offset (SBO).
//  * One MMA covers K = 64 (32 bytes of each row: two core matrices along
//    K) and four 16-element scale blocks per row.
//  * Scale factors for one MMA sit in a 512-byte shared-memory chunk, row
//    r (= r32 + 32 r4 of up to 128 rows) at byte 16 r32 + 4 r4 + block;
//    tcgen05.cp (32 lanes x 128 bits, replicated to the four lane
//    quadrants) moves a chunk into four tensor-memory columns, whose base
//    column the MMA takes as its scale operand.
//  * The accumulator of an M = 128, N = n tile is tensor-memory lanes
//    0..127 (row m = lane m) x n fp32 columns.
#pragma once

#include <cstdint>

#include "msk_device.cuh"

namespace msk {

// Instruction descriptor of tcgen05.mma .kind::mxf4nvf4: A and B E2M1
// (format code 1), both K-major, fp32 accumulate, UE4M3 scale factors,
// N = n (multiple of 8), M = 128.
__host__ __device__ constexpr uint32_t idesc_mxf4nvf4(int n) {
  return (1u << 7)                      // A format: E2M1
         | (1u << 10)                   // B format: E2M1
         | ((uint32_t)(n >> 3) << 17)   // N >> 3
         | (0u << 23)                   // scale factors UE4M3
         | ((uint32_t)(128 >> 7) << 27);  // M >> 7
}

// Shared-memory matrix descriptor (K-major, no swizzle): start address,
// LBO and SBO in bytes (multiples of 16), descriptor version 1.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}

// --- tensor memory allocation (one full warp) ------------------------------

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// --- ordering between thread synchronisation and tcgen05 operations --------

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// --- issue (one thread) ----------------------------------------------------

// D (tensor memory) = [D +] A B^T with per-16-element E4M3 scales of A and
// B taken from tensor memory (sfa, sfb: base columns of their chunks).
__device__ __forceinline__ void mma_mxf4nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t sfa_tmem, uint32_t sfb_tmem, bool accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p; }"
      ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"((uint32_t)accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

// 32 rows x 16 bytes of shared memory (described by sdesc) into tensor
// memory columns [taddr, taddr + 4) of every lane quadrant.
__device__ __forceinline__ void tc_cp_sf(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Arrives once on the mbarrier when every tcgen05 operation this thread
// issued before has completed.
__device__ __forceinline__ void tc_commit(uint32_t mbar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar) : "memory");
}

// --- epilogue loads (a warp reads its own lane quadrant) --------------------

// 16 consecutive fp32 columns of the warp's 32 lanes: thread i gets lane
// (taddr lane) + i.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 8 consecutive fp32 columns of the warp's 32 lanes.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// 4 consecutive fp32 columns of the warp's 32 lanes.
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, float (&v)[4]) {
  uint32_t r[4];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr)
               : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ uint32_t tmem_lane_addr(uint32_t base, int lane0, int col) {
  return base + ((uint32_t)lane0 << 16) + (uint32_t)col;
}

}  // namespace msk
