// Workspace layout of gs_bin_sort, shared by the entry point that takes a caller's
// workspace and the one whose scratch is a fixed array inside the library.
#pragma once

#include <cstddef>
#include <cstdint>

namespace gs {

constexpr int kScanThreads = 256;
constexpr int kScanItems = 16;
constexpr int kScanBlock = kScanThreads * kScanItems;  // Gaussians per block
constexpr int kSortThreads = 256;
constexpr int kSortWarps = kSortThreads / 32;
constexpr int kSortItems = 16;
constexpr int kPart = kSortThreads * kSortItems;  // keys per onesweep partition
constexpr int kDepthPasses = 4;
constexpr int kMaxTilePasses = 4;
constexpr int kMaxPasses = kDepthPasses + kMaxTilePasses;
constexpr uint32_t kFlagAgg = 1u << 30;
constexpr uint32_t kFlagInc = 2u << 30;
constexpr uint32_t kCountMask = (1u << 30) - 1u;
constexpr int kSpinLimit = 1 << 22;
constexpr int kLookWindow = 4;  // predecessors read at once in a look-back
constexpr size_t kSortSmem = size_t(kPart) * 8 + size_t(kSortWarps) * 256 * 4;  // 40 KB

constexpr size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
constexpr size_t max_sz(size_t a, size_t b) { return a > b ? a : b; }

constexpr int tile_bits(int64_t tiles) {
  int b = 0;
  while ((int64_t(1) << b) < tiles) ++b;
  return b;
}

constexpr int tile_passes(int64_t tiles) { return (tile_bits(tiles) + 7) / 8; }

// Workspace layout.  The depth sort's scratch (keys A and B, values B) and the tile
// sort's (keys A and B, the values buffer that is not bins.ids) share one region of
// three slots, each large enough for either sort's buffers.  The depth-sorted indices
// end in values A (outside the region) or, when the last depth pass is the identity
// and skips its copy, in values B, which the emission reads while it writes the tile
// keys A and values: so values B takes the slot of tile keys B, which nothing writes
// before the first tile pass.
//   slot 0: depth keys A, tile keys A;  slot 1: depth values B, tile keys B;
//   slot 2: depth keys B, the tile sort's other values buffer
struct SortLayout {
  size_t block_vis, block_cnt, block_sums, vcount, dvA, shared, slot, hist, tickets, look_d, look_t, total;
  size_t zero_begin, zero_bytes;
  int64_t n_blocks, n_parts_n, n_parts_k;
  int passes_t;
  // offsets inside the shared region
  size_t dkA() const { return shared; }
  size_t dvB() const { return shared + slot; }
  size_t dkB() const { return shared + 2 * slot; }
  size_t tkA() const { return shared; }
  size_t tkB() const { return shared + slot; }
  size_t tvAlt() const { return shared + 2 * slot; }
};

constexpr SortLayout sort_layout(int64_t n, uint32_t cap, int64_t tiles) {
  SortLayout L{};
  L.n_blocks = (n + kScanBlock - 1) / kScanBlock;
  if (L.n_blocks < 1) L.n_blocks = 1;
  L.n_parts_n = (n + kPart - 1) / kPart;
  if (L.n_parts_n < 1) L.n_parts_n = 1;
  L.n_parts_k = (int64_t(cap) + kPart - 1) / kPart;
  if (L.n_parts_k < 1) L.n_parts_k = 1;
  L.passes_t = tile_passes(tiles);
  size_t off = 0;
  L.block_vis = off;
  off += align256(size_t(L.n_blocks) * 8);
  L.block_cnt = off;
  off += align256(size_t(L.n_blocks) * 8);
  L.block_sums = off;
  off += align256(size_t(L.n_blocks) * 8);
  L.vcount = off;
  off += 256;
  L.dvA = off;
  off += align256(size_t(n) * 4);
  L.shared = off;
  L.slot = max_sz(align256(size_t(n) * 4), align256(size_t(cap) * 4));
  off += 3 * L.slot;
  L.hist = off;
  off += align256(size_t(kMaxPasses) * 256 * 4);
  L.tickets = off;
  off += align256(size_t(kMaxPasses) * 4);
  L.look_d = off;
  off += align256(size_t(kDepthPasses) * size_t(L.n_parts_n) * 256 * 4);
  L.look_t = off;
  off += align256(size_t(L.passes_t) * size_t(L.n_parts_k) * 256 * 4);
  L.total = off;
  L.zero_begin = L.hist;
  L.zero_bytes = L.total - L.hist;
  return L;
}

}  // namespace gs
