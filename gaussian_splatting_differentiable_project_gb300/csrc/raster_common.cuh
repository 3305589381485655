// Shared pieces of the forward and backward rasterisers: tile/pixel mapping and
// the bulk-copy (cp.async.bulk + mbarrier) staging of record batches into shared
// memory.  Each CTA owns one 8x8 quarter of a 16x16 tile, one thread per pixel,
// two warps of 8x4 pixels each, and walks the whole tile's record list.  Small
// CTAs keep the coupling between warps (one barrier per batch) to two warps and
// let up to 32 CTAs share an SM, so a quarter whose pixels finish early frees its
// slot instead of idling until the slowest pixel of a 256-pixel tile is done.
#pragma once

#include "gs_common.cuh"

namespace gs {

constexpr int kRasterThreads = 64;                   // one 8x8 quarter tile
constexpr int kCtasPerTile = 4;
// Records per shared-memory batch.  The backward stages 64 (3 KB); the forward 96
// (4.5 KB): half as many batch barriers again per record, which paid in the forward
// (0.95x of its time at 64; 80: 0.96x, 112: 0.98x, 128: 0.99x, three slots of 64: 1.0x)
// and not in the backward (1.0x).
constexpr int kBatch = 64;
constexpr int kBatchFwd = 96;
// Both walks index the composited-entry masks by 32-entry chunks of the tile's list, so
// every batch must start on a chunk: a 48-record backward batch broke that and faulted.
static_assert(kBatch % 32 == 0 && kBatchFwd % 32 == 0, "batches start on 32-entry mask chunks");
constexpr int kWaitLimit = 1 << 24;                  // bounded mbarrier wait (iterations)

__device__ __forceinline__ int tile_of_block() { return int(blockIdx.x) / kCtasPerTile; }

__device__ __forceinline__ void pixel_of_thread(int TX, int& px, int& py) {
  const int tile = tile_of_block(), q = int(blockIdx.x) % kCtasPerTile;
  const int tx = tile % TX, ty = tile / TX;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  px = tx * kTile + (q & 1) * 8 + (lane & 7);
  py = ty * kTile + (q >> 1) * 8 + warp * 4 + (lane >> 3);
}

// ------------------------------------------------------------------ composited-entry masks
// The forward records, for every 8x4 block of a tile and every 32-entry chunk of the
// tile's list that the block's warp walks, each pixel's 32-bit mask of the entries it
// composited (bit i: list position 32 c + i of chunk c, counted from the tile's first
// entry).  The backward walks only those entries.  Chunk c of the tile whose list
// starts at `start` is stored at chunk slot (start >> 5) + tile + c: consecutive tiles'
// slots never overlap (the next list starts n entries later, and ceil(n / 32) <=
// floor(n / 32) + 1), and every slot is below capacity_K / 32 + tiles + 1.
constexpr int kBlocksPerTile = 8;  // 8x4 blocks of a 16x16 tile

__device__ __forceinline__ size_t cmask_index(uint32_t start, int tile, uint32_t chunk_pos, int block, int lane) {
  const size_t slot = size_t(start >> 5) + size_t(tile) + size_t(chunk_pos >> 5);
  return (slot * kBlocksPerTile + size_t(block)) * 32 + size_t(lane);
}

// The backward runs one warp per 8x4 block (eight per tile), each warp on its own: its
// own staging buffers and barriers, no barrier with any other warp, so a warp whose
// pixels need fewer entries than its neighbour's finishes and frees its slot (against
// two warps sharing a tile's batches: 0.987x of the backward's time).  Four such warps
// share a CTA, which only pools their shared memory and scheduling (1.51 against
// 1.55 ms for one warp per CTA).
constexpr int kBwdBlocksPerTile = 8;
constexpr int kBwdWarpsPerCta = 4;
static_assert(kBwdBlocksPerTile % kBwdWarpsPerCta == 0, "a tile's blocks fill whole CTAs");

// Pixel-centre bounds of this warp's 8x4 block.
__device__ __forceinline__ void warp_block_bounds(int TX, float& x0, float& x1, float& y0, float& y1) {
  const int tile = tile_of_block(), q = int(blockIdx.x) % kCtasPerTile;
  const int warp = threadIdx.x >> 5;
  const float bx = float((tile % TX) * kTile + (q & 1) * 8);
  const float by = float((tile / TX) * kTile + (q >> 1) * 8 + warp * 4);
  x0 = bx + 0.5f;
  x1 = bx + 7.5f;
  y0 = by + 0.5f;
  y1 = by + 3.5f;
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
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t* dev_status,
                                          int limit = kWaitLimit) {
  for (int it = 0; it < limit; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
  }
  raise_status(dev_status, GS_ERR_TIMEOUT);
  return false;
}

// Staging of the tile's record list [start, start + n) in batches of kB records
// (kB * 48 bytes is a multiple of 16, as the bulk copy needs).
// The two buffers are one shared array of 2 kB records, addressed by offset (not
// chosen between two pointers), so the walk's record loads stay shared-memory loads.
template <int kB>
struct BatchStager {
  const Rec* src;       // first record of the tile
  uint32_t n;           // records in the tile
  Rec* buf;             // [2][kB]
  uint64_t* bar;        // two barriers

  __device__ __forceinline__ uint32_t count(int b) const {
    const uint32_t lo = uint32_t(b) * kB;
    return min(uint32_t(kB), n - lo);
  }
  __device__ __forceinline__ Rec* buffer(int slot) const { return buf + slot * kB; }
  // Called by one thread: load batch b into slot `slot`.
  __device__ __forceinline__ void issue(int b, int slot) const {
    bulk_load(buffer(slot), src + size_t(b) * kB, count(b) * uint32_t(sizeof(Rec)), bar + slot);
  }
};

}  // namespace gs
