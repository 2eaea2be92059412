// ss2_tma.cuh — inline PTX for the Tensor Memory Accelerator (TMA) and
// shared-memory mbarriers on sm_100-family GPUs, as documented in the PTX
// ISA (cp.async.bulk.tensor, mbarrier, cp.async.bulk.commit_group /
// wait_group, fence.proxy.async).
//
// Every wait on an mbarrier is bounded: it polls at most kSpinLimit times and
// reports failure instead of spinning forever.
#pragma once

#include <cuda.h>
#include <cstdint>

namespace ss2 {

constexpr uint32_t kSpinLimit = 1u << 26;

// Error bits a kernel can raise in the context's error word.
constexpr int kErrTmaTimeout = 1;

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Makes initialised barriers visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity,
                                          uint32_t limit = kSpinLimit) {
  for (uint32_t i = 0; i < limit; ++i)
    if (mbar_test(bar, parity)) return true;
  return false;
}

__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// 4-D tiled load global -> shared, completion counted on bar (bytes).
__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int x, int y, int z, int w) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_addr(dst)),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_addr(bar))
      : "memory");
}

// Non-tensor bulk copy global -> shared of `bytes` bytes (both addresses
// 16-byte aligned, bytes a multiple of 16), completion counted on bar.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes,
                                          uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// 4-D tiled store shared -> global (bulk group); out-of-bounds parts of the
// box are not written.
__device__ __forceinline__ void tma_store_4d(const CUtensorMap *map, const void *src, int x, int y,
                                             int z, int w) {
  asm volatile(
      "cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group"
      " [%0, {%2, %3, %4, %5}], [%1];" ::"l"(map),
      "r"(smem_addr(src)), "r"(x), "r"(y), "r"(z), "r"(w)
      : "memory");
}

// Offset, in 16-byte units, of 16-byte unit u of a tile whose box rows are
// 128 bytes and which a TMA map with 128-byte swizzling moves (the tile
// starting on 1024 bytes): within each row of eight units, the unit index is
// XORed with the row's index modulo 8 (address bits 4-6 XOR bits 7-9).
__device__ __forceinline__ int swz128(int u) { return u ^ ((u >> 3) & 7); }

// The same for box rows of 32 bytes under 32-byte swizzling: the two units
// of a row swap when bit 2 of the row index is set (address bit 4 XOR bit 7).
__device__ __forceinline__ int swz32(int u) { return u ^ ((u >> 3) & 1); }

__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until at most N committed bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until at most N committed bulk groups are incomplete.
template <int N>
__device__ __forceinline__ void bulk_wait() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Orders this thread's generic-proxy shared-memory accesses before later
// async-proxy (TMA) accesses to the same memory: writes before a bulk store
// reads them, and reads before a bulk load overwrites them.
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

}  // namespace ss2
