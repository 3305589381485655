// Shared pieces of the forward and backward rasterisers: tile/pixel mapping and
// the bulk-copy (cp.async.bulk + mbarrier) staging of record batches into shared
// memory.  Each CTA owns one 16x16 tile, one thread per pixel; warp w covers the
// 8x4 pixel block (w & 1, w >> 1) of the tile so that a Gaussian's footprint
// touches few warps.
#pragma once

#include "gs_common.cuh"

namespace gs {

constexpr int kRasterThreads = 256;
constexpr int kBatch = 256;                          // records per shared-memory batch
constexpr uint32_t kBatchBytes = kBatch * sizeof(Rec);  // 12 KB
constexpr int kWaitLimit = 1 << 24;                  // bounded mbarrier wait (iterations)

__device__ __forceinline__ void pixel_of_thread(int tile, int TX, int& px, int& py) {
  const int tx = tile % TX, ty = tile / TX;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  px = tx * kTile + (warp & 1) * 8 + (lane & 7);
  py = ty * kTile + (warp >> 1) * 4 + (lane >> 3);
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// One elected thread: arm the barrier for `bytes` and start the bulk copy
// global -> shared that completes it.  src and dst 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
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

// Wait for phase `parity` of the barrier with an iteration limit; false (and the
// TIMEOUT status bit) if the limit ran out.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t* dev_status) {
  for (int it = 0; it < kWaitLimit; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
  }
  raise_status(dev_status, GS_ERR_TIMEOUT);
  return false;
}

// Staging of the tile's record list [start, start + n) in batches of kBatch.
struct BatchStager {
  const Rec* src;       // first record of the tile
  uint32_t n;           // records in the tile
  Rec* buf0;
  Rec* buf1;
  uint64_t* bar;        // two barriers

  __device__ __forceinline__ uint32_t count(int b) const {
    const uint32_t lo = uint32_t(b) * kBatch;
    return min(uint32_t(kBatch), n - lo);
  }
  __device__ __forceinline__ Rec* buffer(int slot) const { return slot ? buf1 : buf0; }
  // Called by one thread: load batch b into slot `slot`.
  __device__ __forceinline__ void issue(int b, int slot) const {
    bulk_load(buffer(slot), src + size_t(b) * kBatch, count(b) * uint32_t(sizeof(Rec)), bar + slot);
  }
};

}  // namespace gs
