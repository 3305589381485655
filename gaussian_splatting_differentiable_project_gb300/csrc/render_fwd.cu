// gs_render_fwd: per-tile front-to-back alpha compositing.
//
// One CTA per 8x8 quarter of a 16x16 tile, one thread per pixel.  The tile's
// sorted records are staged into shared memory in batches of 96 (4.5 KB) by
// cp.async.bulk with two mbarrier-tracked buffers, so the next batch streams in
// while the current one is composited; every thread reads the same record
// (shared-memory broadcast).  A pixel stops at its transmittance threshold; the
// CTA stops loading once __syncthreads_count reports no live pixel.  For every
// 32-entry chunk a warp walks it stores each pixel's mask of composited entries, which
// the backward walks instead of re-evaluating the whole list.  The counting
// instantiation (gs_render_fwd_counted) also writes each pixel's number of
// composited entries; the training step runs the one without.
#include "api_util.h"
#include "raster_common.cuh"

namespace gs {

template <bool kCount>
__global__ void __launch_bounds__(kRasterThreads, 20)
    k_render_fwd(const Rec* __restrict__ srec, const uint2* __restrict__ ranges, const uint32_t* __restrict__ n_isect,
                 uint32_t cap, int W, int H, int TX, float bg0, float bg1, float bg2, float* __restrict__ image,
                 float* __restrict__ T_final, uint32_t* __restrict__ n_contrib, uint32_t* __restrict__ n_used,
                 uint32_t* __restrict__ cmask, uint32_t* __restrict__ dev_status) {
  __shared__ __align__(128) Rec s_rec[2][kBatchFwd];
  __shared__ __align__(8) uint64_t s_bar[2];

  const int tile = tile_of_block();
  int pxi, pyi;
  pixel_of_thread(TX, pxi, pyi);
  const bool inside = pxi < W && pyi < H;
  const float px = float(pxi) + 0.5f, py = float(pyi) + 0.5f;
  float bx0, bx1, by0, by1;
  warp_block_bounds(TX, bx0, bx1, by0, by1);
  const int lane = threadIdx.x & 31;
  // this warp's 8x4 block within the tile: row block (q >> 1) * 2 + warp, column q & 1
  const int q = int(blockIdx.x) % kCtasPerTile;
  const int block = (((q >> 1) * 2 + (threadIdx.x >> 5)) << 1) + (q & 1);

  const uint32_t K = min(*n_isect, cap);
  const uint2 rg = ranges[tile];
  const uint32_t start = min(rg.x, K), end = min(max(rg.y, rg.x), K);
  const uint32_t n = end - start;

  float T = 1.0f, C0 = 0.0f, C1 = 0.0f, C2 = 0.0f;
  uint32_t last = 0, used = 0;
  bool done = !inside;

  if (n > 0) {
    BatchStager<kBatchFwd> st{srec + start, n, &s_rec[0][0], s_bar};
    const int nb = int((n + kBatchFwd - 1) / kBatchFwd);
    if (threadIdx.x == 0) {
      mbar_init(&s_bar[0], 1);
      mbar_init(&s_bar[1], 1);
      fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      st.issue(0, 0);
      if (nb > 1) st.issue(1, 1);
    }
    int issued = nb < 2 ? nb : 2;
    for (int b = 0; b < nb; ++b) {
      const int slot = b & 1;
      mbar_wait(&s_bar[slot], uint32_t((b >> 1) & 1), dev_status);
      const Rec* R = st.buffer(slot);
      const int cnt = int(st.count(b));
      const uint32_t pos0 = uint32_t(b) * kBatchFwd;
      // Warp-uniform walk over the batch: 32 entries at a time are culled against
      // the warp's 8x4 block by one ballot, then the warp steps through the set
      // bits in order; every lane takes its skip / stop decisions as predicates,
      // so the warp stays converged.
      if (!__all_sync(0xffffffffu, done)) {
        for (int j0 = 0; j0 < cnt; j0 += 32) {
          uint32_t mask = warp_cull(R, j0, cnt, bx0, bx1, by0, by1);
          uint32_t cm = 0;  // this pixel's composited entries of the chunk
          while (mask) {
            const uint32_t low = mask & (0u - mask);  // the entry's bit
            mask ^= low;
            const int j = j0 + __ffs(low) - 1;
            const float4 ra = R[j].a;  // mx, my, ca, cb
            const float4 rb = R[j].b;  // cc, o, r, g
            const float dx = __fsub_rn(px, ra.x), dy = __fsub_rn(py, ra.y);
            const float power = conic_power(dx, dy, ra.z, ra.w, rb.x);
            if (!done && !(power > 0.0f) && !(power < kPowerSkip)) {
              const float v = __fmul_rn(rb.y, gs_expf_core(power));
              const float alpha = (v < kAlphaMax) ? v : kAlphaMax;
              if (!(alpha < kAlphaMin)) {
                // T (1 - alpha) as T - alpha T, one rounding (the frozen sequence)
                const float Tn = __fmaf_rn(-alpha, T, T);
                if (Tn < kTMin) {
                  done = true;
                } else {
                  const float w = __fmul_rn(alpha, T);
                  C0 = __fmaf_rn(rb.z, w, C0);
                  C1 = __fmaf_rn(rb.w, w, C1);
                  C2 = __fmaf_rn(R[j].c.x, w, C2);
                  T = Tn;
                  cm |= low;
                  if (kCount) ++used;
                }
              }
            }
          }
          cmask[cmask_index(start, tile, pos0 + uint32_t(j0), block, lane)] = cm;
          // the last composited entry so far: the highest bit of this chunk's mask
          if (cm) last = pos0 + uint32_t(j0) + 32u - uint32_t(__clz(cm));
          if (__all_sync(0xffffffffu, done)) break;
        }
      }
      const int alive = __syncthreads_count(!done);
      if (alive == 0) {
        // no pixel needs more: drain copies still in flight before the CTA exits
        for (int q = b + 1; q < issued; ++q) mbar_wait(&s_bar[q & 1], uint32_t((q >> 1) & 1), dev_status);
        break;
      }
      if (b + 2 < nb) {
        if (threadIdx.x == 0) st.issue(b + 2, slot);
        issued = b + 3;
      }
    }
  }
  if (inside) {
    const size_t P = size_t(W) * H;
    const size_t pix = size_t(pyi) * W + pxi;
    image[pix] = __fmaf_rn(T, bg0, C0);
    image[P + pix] = __fmaf_rn(T, bg1, C1);
    image[2 * P + pix] = __fmaf_rn(T, bg2, C2);
    T_final[pix] = T;
    n_contrib[pix] = last;
    if (kCount) n_used[pix] = used;
  }
}

}  // namespace gs

namespace {
gs_status render_fwd_launch(const gs_camera* cam, const gs_bins* bins, uint32_t capacity_K, const float bg[3],
                            float* image, float* T_final, uint32_t* n_contrib, uint32_t* n_used, uint32_t* cmask,
                            size_t cmask_bytes, uint32_t* dev_status, cudaStream_t stream) {
  using namespace gs;
  if (!camera_ok(cam) || !bins || !bg || !image || !T_final || !n_contrib || !cmask || !dev_status)
    return GS_ERR_INVALID_ARG;
  if (!bins->rec || !bins->ranges || !bins->n_isect || capacity_K == 0) return GS_ERR_INVALID_ARG;
  if (!aligned(bins->rec, 16) || !aligned(bins->ranges, 8) || !aligned(cmask, 4)) return GS_ERR_INVALID_ARG;
  if (cmask_bytes < gs_render_cmask_bytes(capacity_K, cam->width, cam->height)) return GS_ERR_INVALID_ARG;
  const int TX = (cam->width + kTile - 1) / kTile;
  const int64_t tiles = n_tiles(cam);
  const Rec* rec = reinterpret_cast<const Rec*>(bins->rec);
  const uint2* ranges = reinterpret_cast<const uint2*>(bins->ranges);
  if (n_used)
    k_render_fwd<true><<<int(tiles * kCtasPerTile), kRasterThreads, 0, stream>>>(
        rec, ranges, bins->n_isect, capacity_K, cam->width, cam->height, TX, bg[0], bg[1], bg[2], image, T_final,
        n_contrib, n_used, cmask, dev_status);
  else
    k_render_fwd<false><<<int(tiles * kCtasPerTile), kRasterThreads, 0, stream>>>(
        rec, ranges, bins->n_isect, capacity_K, cam->width, cam->height, TX, bg[0], bg[1], bg[2], image, T_final,
        n_contrib, nullptr, cmask, dev_status);
  return launch_status();
}
}  // namespace

extern "C" size_t gs_render_cmask_bytes(uint32_t capacity_K, int32_t width, int32_t height) {
  if (width <= 0 || height <= 0) return 0;
  const uint64_t tiles = uint64_t((width + GS_TILE - 1) / GS_TILE) * uint64_t((height + GS_TILE - 1) / GS_TILE);
  const uint64_t slots = uint64_t(capacity_K) / 32 + tiles + 1;
  return size_t(slots * gs::kBlocksPerTile * 32 * sizeof(uint32_t));
}

extern "C" gs_status gs_render_fwd(const gs_camera* cam, const gs_bins* bins, uint32_t capacity_K, const float bg[3],
                                   float* image, float* T_final, uint32_t* n_contrib, uint32_t* cmask,
                                   size_t cmask_bytes, uint32_t* dev_status, cudaStream_t stream) {
  return render_fwd_launch(cam, bins, capacity_K, bg, image, T_final, n_contrib, nullptr, cmask, cmask_bytes,
                           dev_status, stream);
}

extern "C" gs_status gs_render_fwd_counted(const gs_camera* cam, const gs_bins* bins, uint32_t capacity_K,
                                           const float bg[3], float* image, float* T_final, uint32_t* n_contrib,
                                           uint32_t* n_used, uint32_t* cmask, size_t cmask_bytes,
                                           uint32_t* dev_status, cudaStream_t stream) {
  if (!n_used) return GS_ERR_INVALID_ARG;
  return render_fwd_launch(cam, bins, capacity_K, bg, image, T_final, n_contrib, n_used, cmask, cmask_bytes,
                           dev_status, stream);
}

// ------------------------------------------------------------------ wait probe
// The rasterisers' bounded mbarrier wait on a barrier nothing arrives at: phase 0 never
// completes, the wait gives up after wait_limit tries, raises GS_ERR_TIMEOUT and returns.
namespace {
__global__ void k_mbar_probe(int limit, uint32_t* __restrict__ dev_status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    gs::mbar_init(&bar, 1);
    gs::fence_mbar_init();
  }
  __syncthreads();
  gs::mbar_wait(&bar, 0u, dev_status, limit);
}
}  // namespace

extern "C" gs_status gs_util_mbarrier_probe(int32_t wait_limit, uint32_t* dev_status, cudaStream_t stream) {
  using namespace gs;
  if (wait_limit <= 0 || !dev_status) return GS_ERR_INVALID_ARG;
  k_mbar_probe<<<1, 32, 0, stream>>>(wait_limit, dev_status);
  return launch_status();
}
