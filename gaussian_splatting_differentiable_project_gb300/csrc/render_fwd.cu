// gs_render_fwd: per-tile front-to-back alpha compositing.
//
// One CTA per 8x8 quarter of a 16x16 tile, one thread per pixel.  The tile's
// sorted records are staged into shared memory in batches of 96 (4.5 KB) by
// cp.async.bulk with two mbarrier-tracked buffers, so the next batch streams in
// while the current one is composited.  A pixel stops at its transmittance
// threshold; the CTA stops loading once __syncthreads_count reports no live pixel.
//
// Each warp (an 8x4 block) takes a batch 32 entries at a time: one lane per entry
// culls it against the block, and the entries that survive are packed, in order, into
// pairs in the warp's shared memory.  The walk then takes two entries per step: their
// offsets, powers, exponentials and opacity products are formed with the two-wide fp32
// instructions (fma.rn.f32x2 and kin, each half rounded exactly as the scalar
// instruction), and the pair is composited in list order, one entry after the other.
// Every lane reads the same pair (shared-memory broadcast).  A pixel that stops raises
// its alpha threshold to +inf, so it fails every later alpha test.  For every 32-entry
// chunk a warp walks it stores each pixel's mask of composited entries, which the
// backward walks instead of re-evaluating the whole list.  The counting instantiation
// (gs_render_fwd_counted) also writes each pixel's number of composited entries; the
// training step runs the one without.
#include "api_util.h"
#include "raster_common.cuh"

namespace gs {

// gs_expf_core on two arguments at once with the two-wide fp32 instructions: each
// half takes exactly the scalar sequence's roundings (the fused multiply-add, add and
// multiply of a pair round each half as their scalar forms do), and the integer steps
// stay per half.  s - 1.5 * 2^23 is formed as s + (-1.5 * 2^23) and -k ln2 + r as
// k (-ln2) + r, which round identically.
__device__ __forceinline__ float2 gs_expf2_core(float2 x) {
  const float kRound = 12582912.0f;
  const float2 s = __ffma2_rn(x, make_float2(1.44269504088896341f, 1.44269504088896341f), make_float2(kRound, kRound));
  const float2 kf = __fadd2_rn(s, make_float2(-kRound, -kRound));
  float2 r = __ffma2_rn(kf, make_float2(-0.693145751953125f, -0.693145751953125f), x);
  r = __ffma2_rn(kf, make_float2(-1.4286068203094173e-06f, -1.4286068203094173e-06f), r);
  float2 p = __ffma2_rn(make_float2(1.0f / 5040.0f, 1.0f / 5040.0f), r, make_float2(1.0f / 720.0f, 1.0f / 720.0f));
  p = __ffma2_rn(p, r, make_float2(1.0f / 120.0f, 1.0f / 120.0f));
  p = __ffma2_rn(p, r, make_float2(1.0f / 24.0f, 1.0f / 24.0f));
  p = __ffma2_rn(p, r, make_float2(1.0f / 6.0f, 1.0f / 6.0f));
  p = __ffma2_rn(p, r, make_float2(0.5f, 0.5f));
  p = __ffma2_rn(p, r, make_float2(1.0f, 1.0f));
  p = __ffma2_rn(p, r, make_float2(1.0f, 1.0f));
  return make_float2(__uint_as_float(__float_as_uint(p.x) + (__float_as_uint(s.x) << 23)),
                     __uint_as_float(__float_as_uint(p.y) + (__float_as_uint(s.y) << 23)));
}

// conic_power on two entries at once (two-wide instructions, the same roundings).
__device__ __forceinline__ float2 conic_power2(float2 dx, float2 dy, float2 ca, float2 cb, float2 cc) {
  return __ffma2_rn(dx, __ffma2_rn(ca, dx, __fmul2_rn(cb, dy)), __fmul2_rn(__fmul2_rn(cc, dy), dy));
}

// Culled entries of one chunk, packed in pairs: pair p holds the warp's compacted
// entries 2p (.x) and 2p + 1 (.y).  The mean is stored negated, so px + (-mx) gives
// px - mx's bits.
struct __align__(16) EntryPair {
  float2 nmx, nmy;
  float2 ca, cb;
  float2 cc, o;
};

// One entry of the walk, in list order: col holds its colour and, in .w, the bits of
// its position's bit in the chunk.  The frozen compositing decisions of the scalar
// walk, given its power and o e^power, taken as selects rather than branches: every
// value is formed and kept only where the pixel composites the entry (a branch per
// decision cost 0.11 ms of 1.13).
template <bool kCount>
__device__ __forceinline__ void composite_one(float power, float v, const float4& col, float& amin,
                                              float& T, float& C0, float& C1, float& C2, uint32_t& cm,
                                              uint32_t& used) {
  const uint32_t low = __float_as_uint(col.w);  // the entry's bit
  const float alpha = (v < kAlphaMax) ? v : kAlphaMax;
  const float Tn = __fmaf_rn(-alpha, T, T);
  const bool pass = !(power > 0.0f) && !(power < kPowerSkip) && !(alpha < amin);
  const bool stop = Tn < kTMin;
  const bool take = pass && !stop;
  amin = (pass && stop) ? __int_as_float(0x7f800000) : amin;
  const float w = __fmul_rn(alpha, T);
  const float n0 = __fmaf_rn(col.x, w, C0), n1 = __fmaf_rn(col.y, w, C1), n2 = __fmaf_rn(col.z, w, C2);
  C0 = take ? n0 : C0;
  C1 = take ? n1 : C1;
  C2 = take ? n2 : C2;
  T = take ? Tn : T;
  cm |= take ? low : 0u;
  if (kCount) used += take ? 1u : 0u;
}

template <bool kCount>
__global__ void __launch_bounds__(kRasterThreads, 16)
    k_render_fwd(const Rec* __restrict__ srec, const uint2* __restrict__ ranges, const uint32_t* __restrict__ n_isect,
                 uint32_t cap, int W, int H, int TX, float bg0, float bg1, float bg2, float* __restrict__ image,
                 float* __restrict__ T_final, uint32_t* __restrict__ n_contrib, uint32_t* __restrict__ n_used,
                 uint32_t* __restrict__ cmask, uint32_t* __restrict__ dev_status) {
  __shared__ __align__(128) Rec s_rec[2][kBatchFwd];
  __shared__ EntryPair s_pair[kRasterThreads / 32][16];
  __shared__ float4 s_col[kRasterThreads / 32][32];  // compacted entry k: r, g, b, its bit in the chunk
  __shared__ __align__(8) uint64_t s_bar[2];

  const int tile = tile_of_block();
  int pxi, pyi;
  pixel_of_thread(TX, pxi, pyi);
  const bool inside = pxi < W && pyi < H;
  const float px = float(pxi) + 0.5f, py = float(pyi) + 0.5f;
  float bx0, bx1, by0, by1;
  warp_block_bounds(TX, bx0, bx1, by0, by1);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float2 px2 = make_float2(px, px), py2 = make_float2(py, py);
  EntryPair* const my_pair = s_pair[warp];
  float4* const my_col = s_col[warp];
  // this warp's 8x4 block within the tile: row block (q >> 1) * 2 + warp, column q & 1
  const int q = int(blockIdx.x) % kCtasPerTile;
  const int block = (((q >> 1) * 2 + (threadIdx.x >> 5)) << 1) + (q & 1);

  const uint32_t K = min(*n_isect, cap);
  const uint2 rg = ranges[tile];
  const uint32_t start = min(rg.x, K), end = min(max(rg.y, rg.x), K);
  const uint32_t n = end - start;

  float T = 1.0f, C0 = 0.0f, C1 = 0.0f, C2 = 0.0f;
  uint32_t last = 0, used = 0;
  // the alpha threshold of the compositing rule; +inf once the pixel has stopped
  float amin = inside ? kAlphaMin : __int_as_float(0x7f800000);

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
      // Warp-uniform walk over the batch, 32 entries at a time: each lane culls one
      // entry against the warp's 8x4 block and, if it survives, writes it to its
      // compacted slot; the warp then steps through the compacted entries two at a
      // time.  Every lane takes its skip / stop decisions as predicates, so the warp
      // stays converged.
      if (!__all_sync(0xffffffffu, amin > 1.0f)) {
        for (int j0 = 0; j0 < cnt; j0 += 32) {
          const int jl = j0 + lane;
          bool near = false;
          Rec e;
          if (jl < cnt) {
            // the entry may reach one of the warp's pixels when the block of pixel
            // centres lies within its skip radius of its mean (Euclidean distance from
            // the mean to the block); an entry outside it would be skipped by every
            // lane, so culling it changes no decision
            e = R[jl];
            const float ex = fmaxf(fmaxf(bx0 - e.a.x, e.a.x - bx1), 0.0f);
            const float ey = fmaxf(fmaxf(by0 - e.a.y, e.a.y - by1), 0.0f);
            const float r = e.c.z;
            near = (r >= 0.0f) && (ex * ex + ey * ey <= r * r);
          }
          const uint32_t mask = __ballot_sync(0xffffffffu, near);
          __syncwarp();  // the previous chunk's pairs have been read
          if (near) {
            const int k = __popc(mask & ((1u << lane) - 1u));
            float* f = reinterpret_cast<float*>(&my_pair[k >> 1]) + (k & 1);
            f[0] = -e.a.x;
            f[2] = -e.a.y;
            f[4] = e.a.z;
            f[6] = e.a.w;
            f[8] = e.b.x;
            f[10] = e.b.y;
            my_col[k] = make_float4(e.b.z, e.b.w, e.c.x, __uint_as_float(1u << lane));
          }
          __syncwarp();
          const int m = __popc(mask);
          uint32_t cm = 0;  // this pixel's composited entries of the chunk
          for (int k = 0; k < m; k += 2) {
            const EntryPair P = my_pair[k >> 1];
            const float2 dx = __fadd2_rn(px2, P.nmx), dy = __fadd2_rn(py2, P.nmy);
            const float2 power = conic_power2(dx, dy, P.ca, P.cb, P.cc);
            // o e^power for both entries; an entry that the range test skips (or the
            // missing second entry of an odd count) discards its value unused
            const float2 v = __fmul2_rn(P.o, gs_expf2_core(power));
            composite_one<kCount>(power.x, v.x, my_col[k], amin, T, C0, C1, C2, cm, used);
            if (k + 1 < m) composite_one<kCount>(power.y, v.y, my_col[k + 1], amin, T, C0, C1, C2, cm, used);
          }
          cmask[cmask_index(start, tile, pos0 + uint32_t(j0), block, lane)] = cm;
          // the last composited entry so far: the highest bit of this chunk's mask
          if (cm) last = pos0 + uint32_t(j0) + 32u - uint32_t(__clz(cm));
          if (__all_sync(0xffffffffu, amin > 1.0f)) break;
        }
      }
      const int alive = __syncthreads_count(!(amin > 1.0f));
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
