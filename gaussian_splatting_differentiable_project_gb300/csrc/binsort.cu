// gs_bin_sort: tile binning.  The result is that of a stable LSD radix sort of the
// 64-bit (tile << 32 | depth bits) keys of every (Gaussian, tile) intersection,
// emitted in Gaussian-index order: per tile, its Gaussians by depth, ties by index.
// It is produced by two onesweep radix sorts that move fewer bytes than one sort of
// the 64-bit keys:
//   1. the visible Gaussians, compacted in index order, sorted stably by their 32-bit
//      depth bits less the smallest visible depth bits (4 passes over V elements);
//   2. one (tile, index) pair per intersection, emitted in that depth order, sorted
//      stably by tile (ceil(tile bits / 8) passes over K elements).
// Within a tile the pairs keep the depth order with ties by index, which is the order
// of the 64-bit keys; the keys themselves are written in the final gather.
//
// Kernels, in stream order:
//   k_bs_prep          per 4096 Gaussians: the visible count, the sum of tile counts
//                      and the smallest visible depth bits; clears histograms,
//                      tickets, look-back words and the tile ranges (the workspace
//                      needs no initialisation)
//   k_bs_scan_sums x2  one block each: exclusive scan of the visible counts -> V and
//                      the smallest depth bits; sum of the tile counts -> K = n_isect
//                      (capacity check)
//   k_bs_compact       visible Gaussians in index order -> (depth bits - smallest,
//                      index); digit histograms of the depth passes
//   k_bs_onesweep x4   depth passes
//   k_bs_sorted_sums   per 4096 depth-sorted Gaussians: sum of tile counts
//   k_bs_scan_sums     one block: exclusive scan of those sums
//   k_bs_emit          per depth-sorted Gaussian, one (tile, index) pair per tile of its
//                      rect at its offset, staged for coalesced writes; digit
//                      histograms of the tile passes
//   k_bs_onesweep xP   tile passes
//   k_bs_ranges_gather per intersection: tile [start, end), the 64-bit key (the depth
//                      is in the record's last slot) and the 48-byte record gathered
// A onesweep pass: CTAs take 4096-key partitions in ticket order, rank their keys
// stably by digit (per-warp digit-class tables, per-warp histograms), publish per-digit
// aggregates and look back over earlier partitions (bounded wait), then scatter
// through shared memory so each digit's run leaves contiguously.  A pass whose
// histogram puts every key at digit 0 is the identity and only copies.
#include "api_util.h"
#include "binsort_layout.h"
#include "block_scan.cuh"
#include "gs_common.cuh"

namespace gs {

// ------------------------------------------------------------------ memory order helpers
// Look-back words hold flag and count in one 32-bit word and publish nothing
// else, so relaxed (L2-coherent, unfenced) accesses suffice.
__device__ __forceinline__ void st_relaxed(uint32_t* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Sum of one 64-bit value per thread over a 256-thread block (valid in thread 0).
__device__ __forceinline__ uint64_t block_sum_256(uint64_t v, uint64_t* s_warp /*8*/) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) s_warp[warp] = v;
  __syncthreads();
  uint64_t t = 0;
  if (threadIdx.x == 0)
    for (int w = 0; w < 8; ++w) t += s_warp[w];
  __syncthreads();
  return t;
}

// ------------------------------------------------------------------ kernels
__global__ void __launch_bounds__(kScanThreads)
    k_bs_prep(const uint32_t* __restrict__ count, const float* __restrict__ depth, int64_t n, int64_t n_blocks,
              uint64_t* __restrict__ block_vis, uint64_t* __restrict__ block_cnt, uint64_t* __restrict__ block_min,
              uint4* __restrict__ zero, int64_t zero_vec, uint2* __restrict__ ranges, int64_t tiles) {
  __shared__ uint64_t s_w[8];
  __shared__ uint32_t s_min[8];
  // clearing (every block takes a grid-strided share)
  const int64_t gstride = int64_t(gridDim.x) * blockDim.x;
  const int64_t gid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  for (int64_t k = gid; k < zero_vec; k += gstride) zero[k] = make_uint4(0u, 0u, 0u, 0u);
  for (int64_t k = gid; k < tiles; k += gstride) ranges[k] = make_uint2(0u, 0u);
  if (blockIdx.x >= n_blocks) return;
  const int64_t base = int64_t(blockIdx.x) * kScanBlock;
  uint64_t s = 0;
  uint32_t v = 0, mn = ~0u;
#pragma unroll 4
  for (int it = 0; it < kScanItems; ++it) {
    const int64_t i = base + int64_t(it) * kScanThreads + threadIdx.x;
    const uint32_t c = (i < n) ? count[i] : 0u;
    s += c;
    v += (c > 0u);
    if (c > 0u) mn = min(mn, __float_as_uint(depth[i]));
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
  if ((threadIdx.x & 31) == 0) s_min[threadIdx.x >> 5] = mn;
  const uint64_t tv = block_sum_256(v, s_w);  // its barriers order s_min
  const uint64_t ts = block_sum_256(s, s_w);
  if (threadIdx.x == 0) {
    for (int w = 0; w < 8; ++w) mn = min(mn, s_min[w]);
    block_vis[blockIdx.x] = tv;
    block_cnt[blockIdx.x] = ts;
    block_min[blockIdx.x] = mn;
  }
}

// One block: exclusive scan of n_blocks 64-bit sums in place; the total goes to
// *total (clamped to 32 bits) when total is not null, with GS_ERR_CAPACITY raised if
// it exceeds cap.  With block_min not null, the smallest of its n_blocks entries
// goes to *min_out as well.
__global__ void __launch_bounds__(1024)
    k_bs_scan_sums(uint64_t* __restrict__ block_sums, int64_t n_blocks, uint32_t* __restrict__ total, uint64_t cap,
                   uint32_t* __restrict__ dev_status, const uint64_t* __restrict__ block_min = nullptr,
                   uint32_t* __restrict__ min_out = nullptr) {
  __shared__ uint64_t s_part[1024];
  __shared__ uint32_t s_min[32];
  const int t = threadIdx.x;
  const int64_t per = (n_blocks + 1023) / 1024;
  const int64_t b0 = int64_t(t) * per, b1 = min(n_blocks, b0 + per);
  uint64_t s = 0;
  for (int64_t b = b0; b < b1; ++b) s += block_sums[b];
  s_part[t] = s;
  if (block_min) {
    uint32_t mn = ~0u;
    for (int64_t b = b0; b < b1; ++b) mn = min(mn, uint32_t(block_min[b]));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    if ((t & 31) == 0) s_min[t >> 5] = mn;
    __syncthreads();
    if (t == 0) {
      for (int w = 0; w < 32; ++w) mn = min(mn, s_min[w]);
      *min_out = mn;
    }
  }
  __syncthreads();
  // Hillis-Steele inclusive scan over 1024 partial sums
  for (int o = 1; o < 1024; o <<= 1) {
    const uint64_t y = (t >= o) ? s_part[t - o] : 0;
    __syncthreads();
    s_part[t] += y;
    __syncthreads();
  }
  uint64_t run = s_part[t] - s;
  for (int64_t b = b0; b < b1; ++b) {
    const uint64_t c = block_sums[b];
    block_sums[b] = run;
    run += c;
  }
  if (t == 1023 && total) {
    const uint64_t K = s_part[1023];
    total[0] = K > 0xFFFFFFFFull ? 0xFFFFFFFFu : uint32_t(K);
    if (K > cap) raise_status(dev_status, GS_ERR_CAPACITY);
  }
}

// Visible Gaussians (count > 0) in index order -> (depth bits - smallest visible depth
// bits, index) at their compacted positions; histograms of the four 8-bit digits of
// those keys.  Positive fp32 depths order like their bits, and subtracting the
// smallest keeps that order; a scene whose depths lie within a factor of about four
// then has keys below 2^24, and the last depth pass finds every digit 0.
__global__ void __launch_bounds__(kScanThreads)
    k_bs_compact(const uint32_t* __restrict__ count, const float* __restrict__ depth, int64_t n,
                 const uint64_t* __restrict__ block_prefix, const uint32_t* __restrict__ key_min,
                 uint32_t* __restrict__ dk, uint32_t* __restrict__ dv, uint32_t* __restrict__ hist) {
  __shared__ uint32_t s_warp[8];
  __shared__ uint32_t s_hist[kDepthPasses * 256];
  for (int k = threadIdx.x; k < kDepthPasses * 256; k += kScanThreads) s_hist[k] = 0;
  uint64_t pos = block_prefix[blockIdx.x];
  const uint32_t kmin = *key_min;
  const int64_t base = int64_t(blockIdx.x) * kScanBlock;
#pragma unroll 1
  for (int r = 0; r < kScanItems; ++r) {
    const int64_t i = base + int64_t(r) * kScanThreads + threadIdx.x;
    const bool f = (i < n) && count[i] > 0u;
    uint32_t total;
    const uint32_t off = block_excl_scan_256(f ? 1u : 0u, s_warp, &total);  // also orders s_hist clear
    if (f) {
      const uint32_t key = __float_as_uint(depth[i]) - kmin;
      dk[pos + off] = key;
      dv[pos + off] = uint32_t(i);
#pragma unroll
      for (int p = 0; p < kDepthPasses; ++p) atomicAdd(&s_hist[p * 256 + ((key >> (8 * p)) & 0xFFu)], 1u);
    }
    pos += total;
  }
  __syncthreads();
  for (int k = threadIdx.x; k < kDepthPasses * 256; k += kScanThreads) {
    const uint32_t v = s_hist[k];
    if (v) atomicAdd(&hist[k], v);
  }
}

// The depth-sorted ids: the last depth pass leaves them in sorted_a, except when its
// digits are all 0 (depths within a factor of about four), in which case it skips its
// copy and they stay in the third pass's output sorted_b.
__device__ __forceinline__ const uint32_t* depth_sorted_ids(const uint32_t* sorted_a, const uint32_t* sorted_b,
                                                            const uint32_t* last_hist, uint32_t V) {
  return last_hist[0] == V ? sorted_b : sorted_a;
}

// Per 4096 depth-sorted Gaussians: the sum of their tile counts.
__global__ void __launch_bounds__(kScanThreads)
    k_bs_sorted_sums(const uint32_t* __restrict__ sorted_a, const uint32_t* __restrict__ sorted_b,
                     const uint32_t* __restrict__ last_hist, const uint32_t* __restrict__ vcount,
                     const uint32_t* __restrict__ count, uint64_t* __restrict__ block_sums) {
  __shared__ uint64_t s_w[8];
  const uint32_t V = *vcount;
  const uint32_t* const sorted_ids = depth_sorted_ids(sorted_a, sorted_b, last_hist, V);
  const int64_t base = int64_t(blockIdx.x) * kScanBlock;
  uint64_t s = 0;
#pragma unroll 4
  for (int it = 0; it < kScanItems; ++it) {
    const int64_t i = base + int64_t(it) * kScanThreads + threadIdx.x;
    if (i < V) s += count[sorted_ids[i]];
  }
  const uint64_t t = block_sum_256(s, s_w);
  if (threadIdx.x == 0) block_sums[blockIdx.x] = t;
}

// Pairs staged in shared memory per write-out chunk.  A round of 256 Gaussians
// averages about 800 pairs, and 2048 keeps a block at 20 KB of shared memory; with
// at most 32 registers a thread, eight blocks fit on an SM and 4M Gaussians (977
// blocks) run in one wave.
constexpr int kEmitStage = 2048;

// Emission: a block owns depth-sorted positions [block * 4096, +4096) and the
// contiguous output range [block_prefix, block_prefix + block total).  It walks them
// in 16 rounds of 256 (one Gaussian per thread); a block scan of the round's counts
// gives each Gaussian's offset, and the round's (tile, index) pairs are staged through
// shared memory so that they leave in contiguous, coalesced runs.  The digit
// histograms of every tile pass are accumulated on the way out.
__global__ void __launch_bounds__(kScanThreads, 8)
    k_bs_emit(const uint32_t* __restrict__ sorted_a, const uint32_t* __restrict__ sorted_b,
              const uint32_t* __restrict__ last_hist, const uint32_t* __restrict__ vcount,
              const uint32_t* __restrict__ count, const uint2* __restrict__ rect,
              const uint64_t* __restrict__ block_prefix, uint32_t* __restrict__ tk, uint32_t* __restrict__ tv,
              uint32_t cap, int TX, int passes, uint32_t* __restrict__ hist) {
  __shared__ uint32_t s_warp[8];
  __shared__ uint32_t s_hist[kMaxTilePasses * 256];
  __shared__ uint32_t s_key[kEmitStage];
  __shared__ uint32_t s_id[kEmitStage];
  for (int k = threadIdx.x; k < passes * 256; k += kScanThreads) s_hist[k] = 0;
  const uint32_t V = *vcount;
  const uint32_t* const sorted_ids = depth_sorted_ids(sorted_a, sorted_b, last_hist, V);
  uint64_t round_base = block_prefix[blockIdx.x];
  const int64_t base = int64_t(blockIdx.x) * kScanBlock;
  // the gathers of round r + 1 (index, then that Gaussian's count and rect) are in
  // flight while round r is scanned and written out
  uint32_t g_next = 0, c_next = 0;
  uint2 rc_next = make_uint2(0u, 0u);
  {
    const int64_t i = base + threadIdx.x;
    if (i < V) {
      g_next = sorted_ids[i];
      c_next = count[g_next];
      rc_next = rect[g_next];
    }
  }
#pragma unroll 1
  for (int r = 0; r < kScanItems; ++r) {
    const uint32_t g = g_next, c = c_next;
    const uint2 rc = rc_next;
    {
      const int64_t i = base + int64_t(r + 1) * kScanThreads + threadIdx.x;
      g_next = 0;
      c_next = 0;
      rc_next = make_uint2(0u, 0u);
      if (r + 1 < kScanItems && i < V) {
        g_next = sorted_ids[i];
        c_next = count[g_next];
        rc_next = rect[g_next];
      }
    }
    const uint32_t tx0 = rc.x & 0xFFFFu, ty0 = rc.x >> 16;
    const uint32_t w = c ? (rc.y & 0xFFFFu) - tx0 + 1u : 1u;
    uint32_t total;
    const uint32_t off = block_excl_scan_256(c, s_warp, &total);  // also orders s_hist clear
#pragma unroll 1
    for (uint32_t c0 = 0; c0 < total; c0 += kEmitStage) {
      // this thread's pairs k in [0, c) whose round offset off + k lies in the chunk
      const uint32_t lo = (c0 > off) ? c0 - off : 0u;
      const uint32_t hi = min(c, (c0 + kEmitStage > off) ? c0 + kEmitStage - off : 0u);
      if (lo < hi) {
        // pair k is tile (tx0 + k % w, ty0 + k / w): one division, then row-major steps
        uint32_t ky = lo / w, kx = lo - ky * w;
        uint32_t t = (ty0 + ky) * uint32_t(TX) + tx0 + kx;
        for (uint32_t k = lo; k < hi; ++k) {
          s_key[off + k - c0] = t;
          s_id[off + k - c0] = g;
          ++t;
          if (++kx == w) {
            kx = 0;
            t += uint32_t(TX) - w;
          }
        }
      }
      __syncthreads();
      const uint32_t m = min(uint32_t(kEmitStage), total - c0);
      for (uint32_t q = threadIdx.x; q < m; q += kScanThreads) {
        const uint64_t o = round_base + c0 + q;
        if (o < cap) {
          const uint32_t key = s_key[q];
          tk[o] = key;
          tv[o] = s_id[q];
          for (int p = 0; p < passes; ++p) atomicAdd(&s_hist[p * 256 + int((key >> (8 * p)) & 0xFFu)], 1u);
        }
      }
      __syncthreads();
    }
    round_base += total;
  }
  for (int k = threadIdx.x; k < passes * 256; k += kScanThreads) {
    const uint32_t v = s_hist[k];
    if (v) atomicAdd(&hist[k], v);
  }
}

// Words of one per-warp digit-class table of the onesweep ranking: 256 digits and the
// out-of-range marker, padded.
constexpr int kMatchWords = 264;
static_assert(kSortWarps * 2 * kMatchWords <= 2 * kPart, "the class tables fit in the key and value staging area");

// One stable 8-bit LSD pass over 32-bit keys with 32-bit values: keys
// [0, min(*n_ptr, cap)) of kin/vin -> kout/vout by digit (key >> shift) & 255.
__global__ void __launch_bounds__(kSortThreads)
    k_bs_onesweep(const uint32_t* __restrict__ kin, const uint32_t* __restrict__ vin, uint32_t* __restrict__ kout,
                  uint32_t* __restrict__ vout, const uint32_t* __restrict__ n_ptr, uint32_t cap, int shift,
                  const uint32_t* __restrict__ hist, uint32_t* __restrict__ look, uint32_t* __restrict__ ticket,
                  uint32_t* __restrict__ dev_status, int spin_limit = kSpinLimit, bool skip_identity = false) {
  extern __shared__ __align__(16) unsigned char smem[];
  uint32_t* s_keys = reinterpret_cast<uint32_t*>(smem);
  uint32_t* s_vals = s_keys + kPart;
  uint32_t* s_whist = s_vals + kPart;  // kSortWarps x 256
  __shared__ uint32_t s_lstart[256], s_gbase[256], s_warp[8];
  __shared__ uint32_t s_part;

  const uint32_t K = min(*n_ptr, cap);
  if (hist[0] == K) {
    // every key has digit 0 here: the stable pass is the identity, so copy (or, when the
    // caller reads the input in that case, do nothing)
    if (skip_identity) return;
    const uint32_t lo = blockIdx.x * uint32_t(kPart), hi = min(K, lo + uint32_t(kPart));
    for (uint32_t i = lo + threadIdx.x; i < hi; i += kSortThreads) {
      kout[i] = kin[i];
      vout[i] = vin[i];
    }
    return;
  }
  if (threadIdx.x == 0) s_part = atomicAdd(ticket, 1u);
  for (int k = threadIdx.x; k < kSortWarps * 256; k += kSortThreads) s_whist[k] = 0;
  __syncthreads();
  const uint32_t part = s_part;
  const uint32_t base = part * uint32_t(kPart);
  if (base >= K) return;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t wbase = base + uint32_t(warp) * (kSortItems * 32);
  uint32_t key[kSortItems];
  uint32_t val[kSortItems];
  uint32_t rank[kSortItems];
#pragma unroll
  for (int it = 0; it < kSortItems; ++it) {
    const uint32_t idx = wbase + uint32_t(it) * 32 + uint32_t(lane);
    if (idx < K) {
      key[it] = kin[idx];
      val[it] = vin[idx];
    } else {
      key[it] = ~0u;
      val[it] = 0u;
    }
  }
  // stable warp-level ranking: item order is (it, lane).  A lane finds the lanes holding
  // its digit by OR-ing its bit into its digit's word of a per-warp table in shared
  // memory (the out-of-range marker 256 has its own word) and reading the word back;
  // the class's lowest lane clears the word and advances the digit's count.  Items
  // alternate between two tables, so a clear of one item's words is ordered before
  // the next use of that table by the next item's warp barrier.  The tables live in
  // the key and value staging area, which the scatter below reuses only after a block
  // barrier.
  uint32_t* wh = s_whist + warp * 256;
  uint32_t* const wm0 = s_keys + warp * (2 * kMatchWords);
  for (int k = lane; k < 2 * kMatchWords; k += 32) wm0[k] = 0u;
  __syncwarp();
  const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
  for (int it = 0; it < kSortItems; ++it) {
    const uint32_t idx = wbase + uint32_t(it) * 32 + uint32_t(lane);
    const uint32_t d = (idx < K) ? (key[it] >> shift) & 0xFFu : 256u;
    uint32_t* const wm = wm0 + (it & 1) * kMatchWords;
    atomicOr(&wm[d], 1u << lane);
    __syncwarp();
    const uint32_t peers = wm[d];
    const uint32_t old = (d < 256u) ? wh[d] : 0u;
    __syncwarp();
    if (lane == __ffs(peers) - 1) {
      wm[d] = 0u;
      if (d < 256u) wh[d] = old + __popc(peers);
    }
    rank[it] = old + __popc(peers & lt);
  }
  __syncthreads();

  // thread d owns digit d: totals, per-warp exclusive prefixes
  const uint32_t d = threadIdx.x;
  uint32_t tot = 0;
#pragma unroll
  for (int w = 0; w < kSortWarps; ++w) {
    const uint32_t c = s_whist[w * 256 + d];
    s_whist[w * 256 + d] = tot;
    tot += c;
  }
  uint32_t* mine = look + size_t(part) * 256 + d;
  st_relaxed(mine, (part == 0 ? kFlagInc : kFlagAgg) | tot);

  const uint32_t gstart = block_excl_scan_256(hist[d], s_warp, nullptr);
  const uint32_t lstart = block_excl_scan_256(tot, s_warp, nullptr);

  // Look back in windows of kLookWindow predecessors: their words are loaded
  // together, then walked from the nearest, adding aggregates up to the first
  // inclusive prefix; a word not yet published is re-read (bounded) until it is.
  uint32_t excl = 0;
  if (part > 0) {
    int64_t j = int64_t(part) - 1;
    int spins = 0;
    bool done = false;
    while (!done) {
      uint32_t w[kLookWindow];
#pragma unroll
      for (int k = 0; k < kLookWindow; ++k)
        w[k] = (j - k >= 0) ? ld_relaxed(look + size_t(j - k) * 256 + d) : kFlagInc;
#pragma unroll
      for (int k = 0; k < kLookWindow; ++k) {
        if (!done) {
          uint32_t v = w[k];
          while ((v & ~kCountMask) == 0u) {
            if (++spins > spin_limit) {
              raise_status(dev_status, GS_ERR_TIMEOUT);
              v = kFlagInc;
              break;
            }
            __nanosleep(32);
            v = ld_relaxed(look + size_t(j - k) * 256 + d);
          }
          excl += v & kCountMask;
          if ((v & ~kCountMask) == kFlagInc || j - k == 0) done = true;
        }
      }
      j -= kLookWindow;
    }
    st_relaxed(mine, kFlagInc | (excl + tot));
  }
  s_gbase[d] = gstart + excl;
  s_lstart[d] = lstart;
  __syncthreads();

#pragma unroll
  for (int it = 0; it < kSortItems; ++it) {
    const uint32_t idx = wbase + uint32_t(it) * 32 + uint32_t(lane);
    if (idx < K) {
      const uint32_t dd = (key[it] >> shift) & 0xFFu;
      const uint32_t pos = s_lstart[dd] + s_whist[warp * 256 + dd] + rank[it];
      s_keys[pos] = key[it];
      s_vals[pos] = val[it];
    }
  }
  __syncthreads();
  const uint32_t nvalid = min(uint32_t(kPart), K - base);
  for (uint32_t i = threadIdx.x; i < nvalid; i += kSortThreads) {
    const uint32_t k = s_keys[i];
    const uint32_t dd = (k >> shift) & 0xFFu;
    const uint32_t dst = s_gbase[dd] + (i - s_lstart[dd]);
    kout[dst] = k;
    vout[dst] = s_vals[i];
  }
}

// Per intersection i: the tile's [start, end) from the neighbouring tile keys, the
// 64-bit key (tile << 32 | depth bits from the record's last slot) and the record.
// A thread takes four intersections per pass and issues all their loads before its
// stores, so each thread keeps four dependent id -> record loads in flight.
__global__ void __launch_bounds__(256)
    k_bs_ranges_gather(const uint32_t* __restrict__ tk, const uint32_t* __restrict__ ids,
                       const uint32_t* __restrict__ n_isect, uint32_t cap, const float4* __restrict__ rec_in,
                       float4* __restrict__ rec_out, uint64_t* __restrict__ keys, uint2* __restrict__ ranges) {
  constexpr int kU = 4;  // intersections per thread per pass, their loads issued together
  const uint32_t K = min(*n_isect, cap);
  const uint32_t stride = gridDim.x * blockDim.x;
  for (uint32_t i0 = blockIdx.x * blockDim.x + threadIdx.x; i0 < K; i0 += kU * stride) {
    uint32_t t[kU], gid[kU];
    float4 a[kU], b[kU], c[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const uint32_t i = i0 + uint32_t(u) * stride;
      t[u] = 0u;
      gid[u] = 0u;
      if (i < K) {
        t[u] = tk[i];
        gid[u] = ids[i];
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const uint32_t i = i0 + uint32_t(u) * stride;
      if (i < K) {
        a[u] = rec_in[3 * size_t(gid[u])];
        b[u] = rec_in[3 * size_t(gid[u]) + 1];
        c[u] = rec_in[3 * size_t(gid[u]) + 2];
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const uint32_t i = i0 + uint32_t(u) * stride;
      if (i < K) {
        if (i == 0 || tk[i - 1] != t[u]) ranges[t[u]].x = i;
        if (i + 1 == K || tk[i + 1] != t[u]) ranges[t[u]].y = i + 1;
        rec_out[3 * size_t(i)] = a[u];
        rec_out[3 * size_t(i) + 1] = b[u];
        rec_out[3 * size_t(i) + 2] = c[u];
        keys[i] = (uint64_t(t[u]) << 32) | __float_as_uint(c[u].w);
      }
    }
  }
}

// ------------------------------------------------------------------ spatial order
// A storage order of the Gaussians along a Morton (Z-order) curve of their means, so
// that Gaussians near each other in space, which share tiles, sit near each other in
// memory.  Per axis, q = floor((mu - lo) * (1023 / (hi - lo)) + 0.5) clamped to
// [0, 1023], with lo, hi the axis's bounds over the Gaussians' finite means and every
// operation an explicit IEEE fp32 one (reproducible off the GPU); the code interleaves
// the three 10-bit q (x in bit 0, y in bit 1, z in bit 2) and the order is the stable
// sort of the codes (ties by index).  A non-finite coordinate counts as lo.
constexpr int kSoThreads = 256;

// Float -> uint32 whose unsigned order is the float order (for atomic min / max).
__device__ __forceinline__ uint32_t so_ordered(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float so_unordered(uint32_t u) {
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u);
}

// ws words: [0, 3) ordered min per axis, [3, 6) ordered max, 6: n; the histograms,
// tickets and look-back words of the four passes are cleared.
__global__ void k_so_init(uint32_t* __restrict__ box, int64_t n, uint4* __restrict__ zero, int64_t zero_vec) {
  const int64_t gid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  for (int64_t k = gid; k < zero_vec; k += int64_t(gridDim.x) * blockDim.x) zero[k] = make_uint4(0u, 0u, 0u, 0u);
  if (gid < 3) {
    box[gid] = 0xFFFFFFFFu;
    box[3 + gid] = 0u;
  }
  if (gid == 0) box[6] = uint32_t(n);
}

__global__ void __launch_bounds__(kSoThreads)
    k_so_bbox(const float* __restrict__ params, int64_t n, int64_t n_pad, uint32_t* __restrict__ box) {
  uint32_t lo[3] = {0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu}, hi[3] = {0u, 0u, 0u};
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += int64_t(gridDim.x) * blockDim.x) {
#pragma unroll
    for (int a = 0; a < 3; ++a) {
      const float v = params[a * n_pad + i];
      if (isfinite(v)) {
        lo[a] = min(lo[a], so_ordered(v));
        hi[a] = max(hi[a], so_ordered(v));
      }
    }
  }
#pragma unroll
  for (int a = 0; a < 3; ++a) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      lo[a] = min(lo[a], __shfl_xor_sync(0xffffffffu, lo[a], o));
      hi[a] = max(hi[a], __shfl_xor_sync(0xffffffffu, hi[a], o));
    }
    if ((threadIdx.x & 31) == 0) {
      atomicMin(&box[a], lo[a]);
      atomicMax(&box[3 + a], hi[a]);
    }
  }
}

__device__ __forceinline__ uint32_t so_spread10(uint32_t x) {
  x &= 0x3FFu;
  x = (x | (x << 16)) & 0x030000FFu;
  x = (x | (x << 8)) & 0x0300F00Fu;
  x = (x | (x << 4)) & 0x030C30C3u;
  x = (x | (x << 2)) & 0x09249249u;
  return x;
}

__global__ void __launch_bounds__(kSoThreads)
    k_so_codes(const float* __restrict__ params, int64_t n, int64_t n_pad, const uint32_t* __restrict__ box,
               uint32_t* __restrict__ keys, uint32_t* __restrict__ vals, uint32_t* __restrict__ hist) {
  __shared__ uint32_t s_hist[4 * 256];
  for (int k = threadIdx.x; k < 4 * 256; k += kSoThreads) s_hist[k] = 0;
  float lo[3], sc[3];
#pragma unroll
  for (int a = 0; a < 3; ++a) {
    const bool any = box[a] <= box[3 + a];
    lo[a] = any ? so_unordered(box[a]) : 0.0f;
    const float ext = any ? __fsub_rn(so_unordered(box[3 + a]), lo[a]) : 0.0f;
    sc[a] = ext > 0.0f ? __fdiv_rn(1023.0f, ext) : 0.0f;
  }
  __syncthreads();
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += int64_t(gridDim.x) * blockDim.x) {
    uint32_t code = 0;
#pragma unroll
    for (int a = 0; a < 3; ++a) {
      const float v = params[a * n_pad + i];
      const float t = isfinite(v) ? __fadd_rn(__fmul_rn(__fsub_rn(v, lo[a]), sc[a]), 0.5f) : 0.0f;
      const uint32_t q = uint32_t(fminf(fmaxf(floorf(t), 0.0f), 1023.0f));
      code |= so_spread10(q) << a;
    }
    keys[i] = code;
    vals[i] = uint32_t(i);
#pragma unroll
    for (int p = 0; p < 4; ++p) atomicAdd(&s_hist[p * 256 + ((code >> (8 * p)) & 0xFFu)], 1u);
  }
  __syncthreads();
  for (int k = threadIdx.x; k < 4 * 256; k += kSoThreads) {
    const uint32_t v = s_hist[k];
    if (v) atomicAdd(&hist[k], v);
  }
}

// dst[p][i] = src[p][perm[i]] for i < n, p < planes (32-bit elements); dst[p][i] =
// src[p][i] for the padding n <= i < n_pad.
__global__ void __launch_bounds__(256)
    k_permute_planes(const uint32_t* __restrict__ perm, int64_t n, int64_t n_pad, int planes,
                     const uint32_t* __restrict__ src, uint32_t* __restrict__ dst) {
  const int64_t total = int64_t(planes) * n_pad;
  for (int64_t k = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; k < total; k += int64_t(gridDim.x) * blockDim.x) {
    const int64_t p = k / n_pad, i = k - p * n_pad;
    const int64_t from = i < n ? int64_t(perm[i]) : i;
    dst[k] = src[p * n_pad + from];
  }
}

}  // namespace gs

extern "C" size_t gs_bin_sort_workspace_bytes(gs_dims dims, uint32_t capacity_K, int32_t width, int32_t height) {
  if (width <= 0 || height <= 0 || dims.n < 0) return 0;
  const int64_t tiles = int64_t((width + GS_TILE - 1) / GS_TILE) * ((height + GS_TILE - 1) / GS_TILE);
  return gs::sort_layout(dims.n, capacity_K, tiles).total;
}

extern "C" gs_status gs_bin_sort(gs_dims dims, const gs_proj* proj, const gs_camera* cam, uint32_t capacity_K,
                                 gs_bins bins, void* workspace, size_t workspace_bytes, uint32_t* dev_status,
                                 cudaStream_t stream) {
  using namespace gs;
  if (!dims_ok(dims) || !camera_ok(cam) || !proj || !dev_status) return GS_ERR_INVALID_ARG;
  if (!proj->depth || !proj->rect || !proj->count || !proj->rec) return GS_ERR_INVALID_ARG;
  if (!bins.keys || !bins.ids || !bins.rec || !bins.ranges || !bins.n_isect || !workspace) return GS_ERR_INVALID_ARG;
  if (capacity_K == 0 || capacity_K > (1u << 30)) return GS_ERR_INVALID_ARG;
  if (!aligned(bins.keys, 8) || !aligned(bins.rec, 16) || !aligned(bins.ranges, 8) || !aligned(workspace, 256) ||
      !aligned(proj->rec, 16) || !aligned(proj->rect, 8))
    return GS_ERR_INVALID_ARG;
  const int64_t tiles = n_tiles(cam);
  if (tiles > (int64_t(1) << 30)) return GS_ERR_INVALID_ARG;
  const SortLayout L = sort_layout(dims.n, capacity_K, tiles);
  if (workspace_bytes < L.total) return GS_ERR_INVALID_ARG;
  char* ws = static_cast<char*>(workspace);
  uint64_t* block_vis = reinterpret_cast<uint64_t*>(ws + L.block_vis);
  uint64_t* block_cnt = reinterpret_cast<uint64_t*>(ws + L.block_cnt);
  uint64_t* block_sums = reinterpret_cast<uint64_t*>(ws + L.block_sums);
  uint32_t* vcount = reinterpret_cast<uint32_t*>(ws + L.vcount);
  uint32_t* hist = reinterpret_cast<uint32_t*>(ws + L.hist);
  uint32_t* tickets = reinterpret_cast<uint32_t*>(ws + L.tickets);
  uint32_t* look_d = reinterpret_cast<uint32_t*>(ws + L.look_d);
  uint32_t* look_t = reinterpret_cast<uint32_t*>(ws + L.look_t);
  const CamDev cd = cam_dev(*cam);

  // 1. per-block visible counts and tile-count sums + clearing
  const int clear_blocks = sm_count() * 4;
  const int b1 = int(L.n_blocks > clear_blocks ? L.n_blocks : clear_blocks);
  // (block_sums is free until step 5 and holds the per-block smallest depth bits)
  k_bs_prep<<<b1, kScanThreads, 0, stream>>>(proj->count, proj->depth, dims.n, L.n_blocks, block_vis, block_cnt,
                                              block_sums, reinterpret_cast<uint4*>(ws + L.zero_begin),
                                              int64_t(L.zero_bytes / 16), reinterpret_cast<uint2*>(bins.ranges),
                                              tiles);
  // 2. V (and the compaction offsets), the smallest visible depth bits; K (capacity check)
  k_bs_scan_sums<<<1, 1024, 0, stream>>>(block_vis, L.n_blocks, vcount, ~0ull, dev_status, block_sums, vcount + 1);
  k_bs_scan_sums<<<1, 1024, 0, stream>>>(block_cnt, L.n_blocks, bins.n_isect, capacity_K, dev_status);
  // 3. compaction + depth digit histograms, 4. depth passes (even: ends in A; in B when
  //    the last pass is the identity, which then skips its copy)
  uint32_t* dkA = reinterpret_cast<uint32_t*>(ws + L.dkA());
  uint32_t* dvA = reinterpret_cast<uint32_t*>(ws + L.dvA);
  uint32_t* dkB = reinterpret_cast<uint32_t*>(ws + L.dkB());
  uint32_t* dvB = reinterpret_cast<uint32_t*>(ws + L.dvB());
  k_bs_compact<<<int(L.n_blocks), kScanThreads, 0, stream>>>(proj->count, proj->depth, dims.n, block_vis,
                                                             vcount + 1, dkA, dvA, hist);
  {
    uint32_t *ka = dkA, *va = dvA, *kb = dkB, *vb = dvB;
    for (int p = 0; p < kDepthPasses; ++p) {
      k_bs_onesweep<<<int(L.n_parts_n), kSortThreads, kSortSmem, stream>>>(
          ka, va, kb, vb, vcount, uint32_t(dims.n), 8 * p, hist + 256 * p, look_d + size_t(p) * L.n_parts_n * 256,
          tickets + p, dev_status, kSpinLimit, p == kDepthPasses - 1);
      uint32_t* t = ka;
      ka = kb;
      kb = t;
      t = va;
      va = vb;
      vb = t;
    }
  }
  // 5. offsets of the depth-sorted Gaussians' pairs
  const uint32_t* last_hist = hist + 256 * (kDepthPasses - 1);
  k_bs_sorted_sums<<<int(L.n_blocks), kScanThreads, 0, stream>>>(dvA, dvB, last_hist, vcount, proj->count,
                                                                  block_sums);
  k_bs_scan_sums<<<1, 1024, 0, stream>>>(block_sums, L.n_blocks, nullptr, 0, dev_status);
  // 6. emit (tile, index) pairs into the buffers that make the last tile pass land in
  //    bins.ids
  uint32_t* tkA = reinterpret_cast<uint32_t*>(ws + L.tkA());
  uint32_t* tkB = reinterpret_cast<uint32_t*>(ws + L.tkB());
  uint32_t* tvAlt = reinterpret_cast<uint32_t*>(ws + L.tvAlt());
  const bool even = (L.passes_t % 2) == 0;
  uint32_t *ka = tkA, *kb = tkB;
  uint32_t* va = even ? bins.ids : tvAlt;
  uint32_t* vb = even ? tvAlt : bins.ids;
  k_bs_emit<<<int(L.n_blocks), kScanThreads, 0, stream>>>(dvA, dvB, last_hist, vcount, proj->count,
                                                          reinterpret_cast<const uint2*>(proj->rect), block_sums, ka,
                                                          va, capacity_K, cd.TX, L.passes_t, hist + 256 * kDepthPasses);
  // 7. tile passes
  for (int p = 0; p < L.passes_t; ++p) {
    k_bs_onesweep<<<int(L.n_parts_k), kSortThreads, kSortSmem, stream>>>(
        ka, va, kb, vb, bins.n_isect, capacity_K, 8 * p, hist + 256 * (kDepthPasses + p),
        look_t + size_t(p) * L.n_parts_k * 256, tickets + kDepthPasses + p, dev_status);
    uint32_t* t = ka;
    ka = kb;
    kb = t;
    t = va;
    va = vb;
    vb = t;
  }
  // 8. ranges, 64-bit keys and the record gather
  const int g = grid_for(capacity_K, 256, sm_count() * 4);
  k_bs_ranges_gather<<<g, 256, 0, stream>>>(ka, bins.ids, bins.n_isect, capacity_K,
                                            reinterpret_cast<const float4*>(proj->rec),
                                            reinterpret_cast<float4*>(bins.rec), bins.keys,
                                            reinterpret_cast<uint2*>(bins.ranges));
  return launch_status();
}


namespace {
// Workspace of gs_spatial_order: keys A and B, values B (the values A are the caller's
// perm), the box and count words, then histograms, tickets and look-back words of four
// passes (cleared by k_so_init).
struct SoLayout {
  size_t kA, kB, vB, box, hist, tickets, look, total;
  int64_t parts;
};
SoLayout so_layout(int64_t n) {
  using namespace gs;
  SoLayout L{};
  L.parts = (n + kPart - 1) / kPart;
  if (L.parts < 1) L.parts = 1;
  size_t off = 0;
  L.kA = off;
  off += align256(size_t(n) * 4);
  L.kB = off;
  off += align256(size_t(n) * 4);
  L.vB = off;
  off += align256(size_t(n) * 4);
  L.box = off;
  off += 256;
  L.hist = off;
  off += align256(size_t(4) * 256 * 4);
  L.tickets = off;
  off += 256;
  L.look = off;
  off += align256(size_t(4) * size_t(L.parts) * 256 * 4);
  L.total = off;
  return L;
}
}  // namespace

extern "C" size_t gs_spatial_order_workspace_bytes(gs_dims dims) {
  if (dims.n < 0) return 0;
  return so_layout(dims.n).total;
}

extern "C" gs_status gs_spatial_order(gs_dims dims, const float* params, uint32_t* perm, void* workspace,
                                      size_t workspace_bytes, uint32_t* dev_status, cudaStream_t stream) {
  using namespace gs;
  if (!dims_ok(dims) || !params || !perm || !workspace || !dev_status) return GS_ERR_INVALID_ARG;
  if (!aligned(workspace, 256) || !aligned(perm, 4)) return GS_ERR_INVALID_ARG;
  const SoLayout L = so_layout(dims.n);
  if (workspace_bytes < L.total) return GS_ERR_INVALID_ARG;
  if (dims.n == 0) return GS_OK;
  char* ws = static_cast<char*>(workspace);
  uint32_t* kA = reinterpret_cast<uint32_t*>(ws + L.kA);
  uint32_t* kB = reinterpret_cast<uint32_t*>(ws + L.kB);
  uint32_t* vB = reinterpret_cast<uint32_t*>(ws + L.vB);
  uint32_t* box = reinterpret_cast<uint32_t*>(ws + L.box);
  uint32_t* hist = reinterpret_cast<uint32_t*>(ws + L.hist);
  uint32_t* tickets = reinterpret_cast<uint32_t*>(ws + L.tickets);
  uint32_t* look = reinterpret_cast<uint32_t*>(ws + L.look);
  const int64_t zero_vec = int64_t(L.total - L.hist) / 16;
  k_so_init<<<sm_count() * 4, 256, 0, stream>>>(box, dims.n, reinterpret_cast<uint4*>(ws + L.hist), zero_vec);
  const int g = grid_for(dims.n, kSoThreads, sm_count() * 8);
  k_so_bbox<<<g, kSoThreads, 0, stream>>>(params, dims.n, dims.n_pad, box);
  k_so_codes<<<g, kSoThreads, 0, stream>>>(params, dims.n, dims.n_pad, box, kA, perm, hist);
  // four stable 8-bit passes over the 30-bit codes; an even count ends in (kA, perm)
  uint32_t *ka = kA, *va = perm, *kb = kB, *vb = vB;
  for (int p = 0; p < 4; ++p) {
    k_bs_onesweep<<<int(L.parts), kSortThreads, kSortSmem, stream>>>(ka, va, kb, vb, box + 6, uint32_t(dims.n), 8 * p,
                                                                    hist + 256 * p, look + size_t(p) * L.parts * 256,
                                                                    tickets + p, dev_status);
    uint32_t* t = ka;
    ka = kb;
    kb = t;
    t = va;
    va = vb;
    vb = t;
  }
  return launch_status();
}

extern "C" gs_status gs_permute_planes(gs_dims dims, int32_t planes, const uint32_t* perm, const void* src, void* dst,
                                       cudaStream_t stream) {
  using namespace gs;
  if (!dims_ok(dims) || planes <= 0 || !perm || !src || !dst || src == dst) return GS_ERR_INVALID_ARG;
  if (!aligned(src, 4) || !aligned(dst, 4)) return GS_ERR_INVALID_ARG;
  const int64_t total = int64_t(planes) * dims.n_pad;
  if (total == 0) return GS_OK;
  k_permute_planes<<<grid_for(total, 256, sm_count() * 16), 256, 0, stream>>>(
      perm, dims.n, dims.n_pad, planes, static_cast<const uint32_t*>(src), static_cast<uint32_t*>(dst));
  return launch_status();
}

// ------------------------------------------------------------------ wait probe
// A onesweep pass whose first partition never runs: its look-back word is never
// published, so the one CTA (partition 1) waits on it until spin_limit runs out, raises
// GS_ERR_TIMEOUT and finishes its scatter (in bounds: with nothing added from the
// look-back each key lands inside its digit's range).  Scratch: keys and values in and
// out for two partitions, the histogram, the count, the ticket and two partitions'
// look-back words.
namespace {
constexpr size_t kProbeKeys = 2 * size_t(gs::kPart);
constexpr size_t kProbeBytes = (4 * kProbeKeys + 256 + 2 + 2 * 256) * sizeof(uint32_t);

__global__ void k_probe_init(uint32_t* __restrict__ w) {
  uint32_t* kin = w;
  uint32_t* vin = kin + kProbeKeys;
  uint32_t* hist = vin + 3 * kProbeKeys;  // after kout, vout
  uint32_t* n = hist + 256;
  uint32_t* ticket = n + 1;
  uint32_t* look = ticket + 1;
  for (uint32_t i = threadIdx.x; i < kProbeKeys; i += blockDim.x) {
    kin[i] = i & 255u;
    vin[i] = i;
  }
  for (uint32_t d = threadIdx.x; d < 256; d += blockDim.x) hist[d] = uint32_t(kProbeKeys / 256);
  for (uint32_t k = threadIdx.x; k < 2 * 256; k += blockDim.x) look[k] = 0u;
  if (threadIdx.x == 0) {
    *n = uint32_t(kProbeKeys);
    *ticket = 1u;  // partition 0 is never taken
  }
}
}  // namespace

extern "C" size_t gs_util_lookback_probe_bytes(void) { return kProbeBytes; }

extern "C" gs_status gs_util_lookback_probe(int32_t spin_limit, void* scratch, size_t scratch_bytes,
                                            uint32_t* dev_status, cudaStream_t stream) {
  using namespace gs;
  if (spin_limit <= 0 || !scratch || scratch_bytes < kProbeBytes || !dev_status || !aligned(scratch, 16))
    return GS_ERR_INVALID_ARG;
  uint32_t* w = static_cast<uint32_t*>(scratch);
  uint32_t *kin = w, *vin = kin + kProbeKeys, *kout = vin + kProbeKeys, *vout = kout + kProbeKeys;
  uint32_t* hist = vout + kProbeKeys;
  uint32_t* n = hist + 256;
  uint32_t* ticket = n + 1;
  uint32_t* look = ticket + 1;
  k_probe_init<<<1, 256, 0, stream>>>(w);
  k_bs_onesweep<<<1, kSortThreads, kSortSmem, stream>>>(kin, vin, kout, vout, n, uint32_t(kProbeKeys), 0, hist, look,
                                                        ticket, dev_status, spin_limit);
  return launch_status();
}
