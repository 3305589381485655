// gs_bin_sort: tile binning with a onesweep LSD radix sort of 64-bit
// (tile << 32 | depth bits) keys.
//
// Kernels, in stream order:
//   k_bs_count_sums   per-block sums of the per-Gaussian tile counts; also clears
//                     the sort's histograms, tickets, look-back words and the tile
//                     ranges (so the workspace needs no initialisation)
//   k_bs_scan_sums    one block: exclusive scan of the block sums -> K
//   k_bs_emit         per Gaussian, its offset (block scan + block prefix) and one
//                     key per tile of its rect, in index order, staged through
//                     shared memory for coalesced writes; digit histograms of
//                     every radix pass accumulated on the way
//   k_bs_onesweep     one launch per 8-bit digit: stable ranking of 2048 keys per
//                     CTA, decoupled look-back (bounded wait) across CTAs taken in
//                     ticket order, scatter through shared memory
//   k_bs_ranges_gather per intersection: tile [start, end) and the 48-byte record
//                     gathered into key order
#include <mutex>

#include "api_util.h"
#include "gs_common.cuh"

namespace gs {

constexpr int kScanThreads = 256;
constexpr int kScanItems = 16;
constexpr int kScanBlock = kScanThreads * kScanItems;  // Gaussians per scan block
constexpr int kSortThreads = 256;
constexpr int kSortWarps = kSortThreads / 32;
constexpr int kSortItems = 8;
constexpr int kPart = kSortThreads * kSortItems;  // keys per onesweep partition
constexpr int kMaxPasses = 8;
constexpr uint32_t kFlagAgg = 1u << 30;
constexpr uint32_t kFlagInc = 2u << 30;
constexpr uint32_t kCountMask = (1u << 30) - 1u;
constexpr int kSpinLimit = 1 << 22;
constexpr size_t kSortSmem = size_t(kPart) * 8 + size_t(kPart) * 4 + size_t(kSortWarps) * 256 * 4;

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline int tile_bits(int64_t tiles) {
  int b = 0;
  while ((int64_t(1) << b) < tiles) ++b;
  return b;
}

inline int n_passes(int64_t tiles) { return (32 + tile_bits(tiles) + 7) / 8; }

struct SortLayout {
  size_t keys_alt, ids_alt, block_sums, hist, tickets, look, total;
  size_t zero_begin, zero_bytes;
  int64_t n_blocks, n_parts;
  int passes;
};

inline SortLayout sort_layout(int64_t n, uint32_t cap, int64_t tiles) {
  SortLayout L;
  L.n_blocks = (n + kScanBlock - 1) / kScanBlock;
  if (L.n_blocks < 1) L.n_blocks = 1;
  L.n_parts = (int64_t(cap) + kPart - 1) / kPart;
  L.passes = n_passes(tiles);
  size_t off = 0;
  L.keys_alt = off;
  off += align256(size_t(cap) * 8);
  L.ids_alt = off;
  off += align256(size_t(cap) * 4);
  L.block_sums = off;
  off += align256(size_t(L.n_blocks) * 8);
  L.hist = off;
  off += align256(size_t(kMaxPasses) * 256 * 4);
  L.tickets = off;
  off += align256(size_t(kMaxPasses) * 4);
  L.look = off;
  off += align256(size_t(L.passes) * size_t(L.n_parts) * 256 * 4);
  L.total = off;
  L.zero_begin = L.hist;
  L.zero_bytes = L.total - L.hist;
  return L;
}

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

// Exclusive scan of one value per thread over a 256-thread block.
__device__ __forceinline__ uint32_t block_excl_scan_256(uint32_t v, uint32_t* s_warp /*8*/, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  uint32_t wpre = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const uint32_t c = s_warp[w];
    if (w < warp) wpre += c;
    tot += c;
  }
  __syncthreads();
  if (total) *total = tot;
  return wpre + x - v;
}

// ------------------------------------------------------------------ kernels
__global__ void __launch_bounds__(kScanThreads)
    k_bs_count_sums(const uint32_t* __restrict__ count, int64_t n, int64_t n_blocks, uint64_t* __restrict__ block_sums,
                    uint4* __restrict__ zero, int64_t zero_vec, uint2* __restrict__ ranges, int64_t tiles) {
  __shared__ uint32_t s_warp[8];
  // clearing (every block takes a grid-strided share)
  const int64_t gstride = int64_t(gridDim.x) * blockDim.x;
  const int64_t gid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  for (int64_t k = gid; k < zero_vec; k += gstride) zero[k] = make_uint4(0u, 0u, 0u, 0u);
  for (int64_t k = gid; k < tiles; k += gstride) ranges[k] = make_uint2(0u, 0u);
  if (blockIdx.x >= n_blocks) return;
  const int64_t base = int64_t(blockIdx.x) * kScanBlock;
  uint32_t s = 0;
#pragma unroll 4
  for (int it = 0; it < kScanItems; ++it) {
    const int64_t i = base + int64_t(it) * kScanThreads + threadIdx.x;
    if (i < n) s += count[i];
  }
  uint32_t tot;
  block_excl_scan_256(s, s_warp, &tot);
  if (threadIdx.x == 0) block_sums[blockIdx.x] = tot;
}

__global__ void __launch_bounds__(1024)
    k_bs_scan_sums(uint64_t* __restrict__ block_sums, int64_t n_blocks, uint32_t* __restrict__ n_isect, uint32_t cap,
                   uint32_t* __restrict__ dev_status) {
  __shared__ uint64_t s_part[1024];
  const int t = threadIdx.x;
  const int64_t per = (n_blocks + 1023) / 1024;
  const int64_t b0 = int64_t(t) * per, b1 = min(n_blocks, b0 + per);
  uint64_t s = 0;
  for (int64_t b = b0; b < b1; ++b) s += block_sums[b];
  s_part[t] = s;
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
  if (t == 1023) {
    const uint64_t K = s_part[1023];
    n_isect[0] = K > 0xFFFFFFFFull ? 0xFFFFFFFFu : uint32_t(K);
    if (K > cap) raise_status(dev_status, GS_ERR_CAPACITY);
  }
}

constexpr int kEmitStage = 2048;  // keys staged in shared memory per write-out chunk

// Emission: a block owns Gaussians [block * 4096, +4096) and the contiguous output
// range [block_prefix, block_prefix + block total).  It walks them in 16 rounds of
// 256 (one Gaussian per thread, coalesced reads); a block scan of the round's
// counts gives each Gaussian's offset, and the round's keys are staged through
// shared memory in chunks of kEmitStage so that they leave in contiguous,
// coalesced runs.  The digit histograms of every radix pass are accumulated on
// the way out.
__global__ void __launch_bounds__(kScanThreads)
    k_bs_emit(const uint32_t* __restrict__ count, const uint2* __restrict__ rect, const float* __restrict__ depth,
              int64_t n, const uint64_t* __restrict__ block_prefix, uint64_t* __restrict__ keys,
              uint32_t* __restrict__ ids, uint32_t cap, int TX, int passes, uint32_t* __restrict__ hist) {
  __shared__ uint32_t s_warp[8];
  __shared__ uint32_t s_hist[kMaxPasses * 256];
  __shared__ uint64_t s_key[kEmitStage];
  __shared__ uint32_t s_id[kEmitStage];
  for (int k = threadIdx.x; k < passes * 256; k += kScanThreads) s_hist[k] = 0;
  uint64_t round_base = block_prefix[blockIdx.x];
  const int64_t base = int64_t(blockIdx.x) * kScanBlock;
#pragma unroll 1
  for (int r = 0; r < kScanItems; ++r) {
    const int64_t i = base + int64_t(r) * kScanThreads + threadIdx.x;
    const uint32_t c = (i < n) ? count[i] : 0u;
    uint32_t tx0 = 0, ty0 = 0, w = 1;
    uint32_t zb = 0;
    if (c) {
      const uint2 rc = rect[i];
      tx0 = rc.x & 0xFFFFu;
      ty0 = rc.x >> 16;
      w = (rc.y & 0xFFFFu) - tx0 + 1u;
      zb = __float_as_uint(depth[i]);
    }
    uint32_t total;
    const uint32_t off = block_excl_scan_256(c, s_warp, &total);  // also orders s_hist clear
#pragma unroll 1
    for (uint32_t c0 = 0; c0 < total; c0 += kEmitStage) {
      // this thread's keys k in [0, c) whose round offset off + k lies in the chunk
      const uint32_t lo = (c0 > off) ? c0 - off : 0u;
      const uint32_t hi = min(c, (c0 + kEmitStage > off) ? c0 + kEmitStage - off : 0u);
      for (uint32_t k = lo; k < hi; ++k) {
        const uint32_t ty = ty0 + k / w, tx = tx0 + k % w;
        s_key[off + k - c0] = (uint64_t(ty * uint32_t(TX) + tx) << 32) | zb;
        s_id[off + k - c0] = uint32_t(i);
      }
      __syncthreads();
      const uint32_t m = min(uint32_t(kEmitStage), total - c0);
      for (uint32_t q = threadIdx.x; q < m; q += kScanThreads) {
        const uint64_t o = round_base + c0 + q;
        if (o < cap) {
          const uint64_t key = s_key[q];
          keys[o] = key;
          ids[o] = s_id[q];
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

__global__ void __launch_bounds__(kSortThreads)
    k_bs_onesweep(const uint64_t* __restrict__ kin, const uint32_t* __restrict__ vin, uint64_t* __restrict__ kout,
                  uint32_t* __restrict__ vout, const uint32_t* __restrict__ n_isect, uint32_t cap, int shift,
                  const uint32_t* __restrict__ hist, uint32_t* __restrict__ look, uint32_t* __restrict__ ticket,
                  uint32_t* __restrict__ dev_status) {
  extern __shared__ __align__(16) unsigned char smem[];
  uint64_t* s_keys = reinterpret_cast<uint64_t*>(smem);
  uint32_t* s_vals = reinterpret_cast<uint32_t*>(s_keys + kPart);
  uint32_t* s_whist = s_vals + kPart;  // kSortWarps x 256
  __shared__ uint32_t s_lstart[256], s_gbase[256], s_warp[8];
  __shared__ uint32_t s_part;

  const uint32_t K = min(*n_isect, cap);
  if (threadIdx.x == 0) s_part = atomicAdd(ticket, 1u);
  for (int k = threadIdx.x; k < kSortWarps * 256; k += kSortThreads) s_whist[k] = 0;
  __syncthreads();
  const uint32_t part = s_part;
  const uint32_t base = part * uint32_t(kPart);
  if (base >= K) return;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t wbase = base + uint32_t(warp) * (kSortItems * 32);
  uint64_t key[kSortItems];
  uint32_t val[kSortItems];
  uint32_t rank[kSortItems];
#pragma unroll
  for (int it = 0; it < kSortItems; ++it) {
    const uint32_t idx = wbase + uint32_t(it) * 32 + uint32_t(lane);
    if (idx < K) {
      key[it] = kin[idx];
      val[it] = vin[idx];
    } else {
      key[it] = ~0ull;
      val[it] = 0u;
    }
  }
  // stable warp-level ranking: item order is (it, lane)
  uint32_t* wh = s_whist + warp * 256;
  const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
  for (int it = 0; it < kSortItems; ++it) {
    const uint32_t idx = wbase + uint32_t(it) * 32 + uint32_t(lane);
    const uint32_t d = (idx < K) ? uint32_t(key[it] >> shift) & 0xFFu : 256u;
    const uint32_t peers = __match_any_sync(0xffffffffu, d);
    const int leader = __ffs(peers) - 1;
    uint32_t old = 0;
    if (d < 256u && lane == leader) {
      old = wh[d];
      wh[d] = old + __popc(peers);
    }
    old = __shfl_sync(0xffffffffu, old, leader);
    rank[it] = old + __popc(peers & lt);
    __syncwarp();
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

  uint32_t excl = 0;
  if (part > 0) {
    int64_t j = int64_t(part) - 1;
    int spins = 0;
    for (;;) {
      const uint32_t w = ld_relaxed(look + size_t(j) * 256 + d);
      const uint32_t f = w & ~kCountMask;
      if (f == 0u) {
        if (++spins > kSpinLimit) {
          raise_status(dev_status, GS_ERR_TIMEOUT);
          break;
        }
        __nanosleep(32);
        continue;
      }
      excl += w & kCountMask;
      if (f == kFlagInc || j == 0) break;
      --j;
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
      const uint32_t dd = uint32_t(key[it] >> shift) & 0xFFu;
      const uint32_t pos = s_lstart[dd] + s_whist[warp * 256 + dd] + rank[it];
      s_keys[pos] = key[it];
      s_vals[pos] = val[it];
    }
  }
  __syncthreads();
  const uint32_t nvalid = min(uint32_t(kPart), K - base);
  for (uint32_t i = threadIdx.x; i < nvalid; i += kSortThreads) {
    const uint64_t k = s_keys[i];
    const uint32_t dd = uint32_t(k >> shift) & 0xFFu;
    const uint32_t dst = s_gbase[dd] + (i - s_lstart[dd]);
    kout[dst] = k;
    vout[dst] = s_vals[i];
  }
}

__global__ void __launch_bounds__(256)
    k_bs_ranges_gather(const uint64_t* __restrict__ keys, const uint32_t* __restrict__ ids,
                       const uint32_t* __restrict__ n_isect, uint32_t cap, const float4* __restrict__ rec_in,
                       float4* __restrict__ rec_out, uint2* __restrict__ ranges) {
  const uint32_t K = min(*n_isect, cap);
  const uint32_t stride = gridDim.x * blockDim.x;
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < K; i += stride) {
    const uint32_t t = uint32_t(keys[i] >> 32);
    if (i == 0 || uint32_t(keys[i - 1] >> 32) != t) ranges[t].x = i;
    if (i + 1 == K || uint32_t(keys[i + 1] >> 32) != t) ranges[t].y = i + 1;
    const uint32_t g = ids[i];
    const float4 a = rec_in[3 * size_t(g)], b = rec_in[3 * size_t(g) + 1], c = rec_in[3 * size_t(g) + 2];
    rec_out[3 * size_t(i)] = a;
    rec_out[3 * size_t(i) + 1] = b;
    rec_out[3 * size_t(i) + 2] = c;
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
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(k_bs_onesweep, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSortSmem)) !=
        cudaSuccess)
      return GS_ERR_CUDA;
    attr_set = true;
  }
  char* ws = static_cast<char*>(workspace);
  uint64_t* keys_alt = reinterpret_cast<uint64_t*>(ws + L.keys_alt);
  uint32_t* ids_alt = reinterpret_cast<uint32_t*>(ws + L.ids_alt);
  uint64_t* block_sums = reinterpret_cast<uint64_t*>(ws + L.block_sums);
  uint32_t* hist = reinterpret_cast<uint32_t*>(ws + L.hist);
  uint32_t* tickets = reinterpret_cast<uint32_t*>(ws + L.tickets);
  uint32_t* look = reinterpret_cast<uint32_t*>(ws + L.look);
  const CamDev cd = cam_dev(*cam);

  // 1. block sums of the tile counts + clearing
  const int clear_blocks = kSmCount * 4;
  const int b1 = int(L.n_blocks > clear_blocks ? L.n_blocks : clear_blocks);
  k_bs_count_sums<<<b1, kScanThreads, 0, stream>>>(proj->count, dims.n, L.n_blocks, block_sums,
                                                    reinterpret_cast<uint4*>(ws + L.zero_begin),
                                                    int64_t(L.zero_bytes / 16), reinterpret_cast<uint2*>(bins.ranges),
                                                    tiles);
  // 2. scan of the block sums -> K
  k_bs_scan_sums<<<1, 1024, 0, stream>>>(block_sums, L.n_blocks, bins.n_isect, capacity_K, dev_status);
  // 3. emit keys: into the buffer that makes the last pass land in bins.keys
  const bool even = (L.passes % 2) == 0;
  uint64_t* kA = even ? bins.keys : keys_alt;
  uint32_t* vA = even ? bins.ids : ids_alt;
  uint64_t* kB = even ? keys_alt : bins.keys;
  uint32_t* vB = even ? ids_alt : bins.ids;
  k_bs_emit<<<int(L.n_blocks), kScanThreads, 0, stream>>>(proj->count, reinterpret_cast<const uint2*>(proj->rect),
                                                          proj->depth, dims.n, block_sums, kA, vA, capacity_K, cd.TX,
                                                          L.passes, hist);
  // 4. radix passes
  for (int p = 0; p < L.passes; ++p) {
    k_bs_onesweep<<<int(L.n_parts), kSortThreads, kSortSmem, stream>>>(
        kA, vA, kB, vB, bins.n_isect, capacity_K, 8 * p, hist + 256 * p, look + size_t(p) * L.n_parts * 256,
        tickets + p, dev_status);
    uint64_t* tk = kA;
    kA = kB;
    kB = tk;
    uint32_t* tv = vA;
    vA = vB;
    vB = tv;
  }
  // 5. ranges + record gather
  const int g = grid_for(capacity_K, 256, kSmCount * 16);
  k_bs_ranges_gather<<<g, 256, 0, stream>>>(bins.keys, bins.ids, bins.n_isect, capacity_K,
                                            reinterpret_cast<const float4*>(proj->rec),
                                            reinterpret_cast<float4*>(bins.rec), reinterpret_cast<uint2*>(bins.ranges));
  return launch_status();
}

// ---------------------------------------------------------------------------
// gs_bin_sort_noalloc: the same binning for callers that may not allocate device
// memory, e.g. code running inside a host callback or a real-time loop whose
// memory is reserved up front, or a host that forbids device allocation after
// start-up.  The sort's scratch lives in the file-scope array below, which every
// GPU that loads this library holds until the process exits.  Its size covers
// n <= GS_NOALLOC_MAX_N Gaussians, capacity_K <= GS_NOALLOC_MAX_K intersections
// and up to GS_NOALLOC_MAX_TILES tiles (six radix passes).
namespace gs {

constexpr size_t na_align(size_t x) { return (x + 255) & ~size_t(255); }

// The workspace layout of sort_layout() at the maximum sizes.
constexpr size_t kNoAllocBytes =
    na_align(size_t(GS_NOALLOC_MAX_K) * 8) + na_align(size_t(GS_NOALLOC_MAX_K) * 4) +
    na_align(size_t((GS_NOALLOC_MAX_N + kScanBlock - 1) / kScanBlock) * 8) + na_align(size_t(kMaxPasses) * 256 * 4) +
    na_align(size_t(kMaxPasses) * 4) +
    na_align(size_t(6) * size_t((GS_NOALLOC_MAX_K + kPart - 1) / kPart) * 256 * 4);
static_assert(kNoAllocBytes == 15745280, "fixed scratch size changed");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kNoAllocMaxDevices] = {};

}  // namespace gs

extern "C" gs_status gs_bin_sort_noalloc(gs_dims dims, const gs_proj* proj, const gs_camera* cam,
                                         uint32_t capacity_K, gs_bins bins, uint32_t* dev_status,
                                         cudaStream_t stream) {
  using namespace gs;
  if (!dims_ok(dims) || !camera_ok(cam)) return GS_ERR_INVALID_ARG;
  const int64_t tiles = n_tiles(cam);
  if (dims.n > GS_NOALLOC_MAX_N || capacity_K > GS_NOALLOC_MAX_K || tiles > GS_NOALLOC_MAX_TILES)
    return GS_ERR_SCRATCH_LIMIT;
  const size_t need = sort_layout(dims.n, capacity_K, tiles).total;
  if (need > kNoAllocBytes) return GS_ERR_SCRATCH_LIMIT;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) return GS_ERR_CUDA;
  void* scratch = nullptr;
  {
    // once per device, with that device current: the device address of the array
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return GS_ERR_CUDA;
      g_noalloc_ptr[dev] = p;
    }
    scratch = g_noalloc_ptr[dev];
  }
  return gs_bin_sort(dims, proj, cam, capacity_K, bins, scratch, kNoAllocBytes, dev_status, stream);
}
