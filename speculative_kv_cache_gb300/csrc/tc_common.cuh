// Helpers shared by the tcgen05 / TMA kernels: shared-memory matrix descriptors, 2-D tensor
// loads, tcgen05 fences, and the tensor-map builder.
#pragma once

#include <cuda.h>

#include "ig_common.cuh"

namespace ig {

// 2-D fp16 tensor [rows][cols] (cols contiguous) for TMA: boxes of 64 columns (one 128-byte
// swizzle atom) x box_rows rows, 128B swizzle, zero fill out of bounds.
ig_status make_map(CUtensorMap* m, const void* base, int rows, int cols, int box_rows);

// Shared-memory matrix descriptor of a K-major, 128B-swizzled tile whose 8-row groups are
// 1024 bytes apart: start address >> 4 (bits 0-13), leading offset 16 B (unused for swizzled
// K-major tiles), stride offset 1024 B (bits 32-45), descriptor version 1 (bit 46), layout
// SWIZZLE_128B (bits 61-63 = 2).  Advancing the start address by 32 B selects the next 16-wide
// K step inside the swizzle atom.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

// tma_load_2d with an L2 policy
__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                                 uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
      "%3}], [%4], %5;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(pol)
      : "memory");
}

__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }


}  // namespace ig
