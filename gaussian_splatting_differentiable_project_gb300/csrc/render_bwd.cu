// gs_render_bwd: L1 loss gradient and the compositing backward.
//
// One warp per 8x4 block of a 16x16 tile, one thread per pixel, four independent warps
// to a CTA; each warp stages its tile's records in reverse batches by cp.async.bulk into
// buffers of its own (as the forward does per CTA).  The warp walks back to front only the entries that at least one of its
// pixels composited, as the forward's per-chunk masks record them (the union of the
// block's masks), so entries that every pixel skipped cost nothing and no pixel tests
// whether an entry is in range.  At each entry a pixel that composited it recomputes
// alpha in the forward's fp32 sequence (the same value and the same clamp decision),
// recovers the transmittance before the entry by division by (1 - alpha) and carries
// the normalised colour of everything behind it.  Its nine partials are the opacity and
// colour partials and, for the mean and the conic, the five moments (q dx, q dy,
// q dx^2, q dx dy, q dy^2) of q = dL/dpower; the conic is the Gaussian's own, so the
// projection backward applies it once to the summed moments (10 fewer instructions per
// entry).  A warp with at most kDirectLanes contributing lanes adds them lane by lane
// with vector atomics; a fuller warp reduces them with a shuffle reduce-scatter (14
// shuffles instead of 45 for nine butterflies) and nine lanes add the sums in one
// atomic instruction.  Both land in the Gaussian's interleaved 12-float slot of grad2d
// (two 32-byte sectors instead of nine planes' lines).
#include "api_util.h"
#include "raster_common.cuh"

namespace gs {

// A warp with at most this many contributing lanes skips the reduction: each
// contributing lane adds its own nine partials with three atomics (two float4, one
// scalar) to the Gaussian's slot.  That trades the reduction's 14 shuffles, 14 adds
// and 14 selects for 3 k L2 reductions into one slot (the reduction's one atomic
// instruction reaches L2 as about two requests, its nine addresses lying in two
// sectors).  Those L2 reductions are what limits the walk once k grows.  Measured on the
// 4M-Gaussian isosurface at 2048^2 (backward ms, walking the composited-entry masks):
// thresholds 0 / 4 / 8 / 12 / 14 / 16 / 20 / 24 / 28 give 1.87 / 1.72 / 1.64 / 1.58 /
// 1.56 / 1.55 / 1.61 / 1.85 / 2.15.
constexpr int kDirectLanes = 16;

// Reduce-scatter of nine per-lane values over the warp.  On return lane l with
// (l & 3) == 0 holds the warp sum of value l >> 2 (values 0..7) in *out8 and every
// lane holds the warp sum of value 8 in *out9.
__device__ __forceinline__ void warp_reduce9(const float v[9], float* out8, float* out9) {
  // the adds of each level taken two at a time (two-wide fp32 add, each half rounded
  // as the scalar add, in the same order): value 8 rides along with a pair or with the
  // last single value of every level
  const int lane = threadIdx.x & 31;
  const bool b16 = lane & 16, b8 = lane & 8, b4 = lane & 4;
  float2 w01, w23;
  float z;
  {
    const float s0 = b16 ? v[0] : v[4], k0 = b16 ? v[4] : v[0];
    const float s1 = b16 ? v[1] : v[5], k1 = b16 ? v[5] : v[1];
    const float s2 = b16 ? v[2] : v[6], k2 = b16 ? v[6] : v[2];
    const float s3 = b16 ? v[3] : v[7], k3 = b16 ? v[7] : v[3];
    const float r0 = __shfl_xor_sync(0xffffffffu, s0, 16), r1 = __shfl_xor_sync(0xffffffffu, s1, 16);
    const float r2 = __shfl_xor_sync(0xffffffffu, s2, 16), r3 = __shfl_xor_sync(0xffffffffu, s3, 16);
    const float r8 = __shfl_xor_sync(0xffffffffu, v[8], 16);
    w01 = __fadd2_rn(make_float2(k0, k1), make_float2(r0, r1));
    w23 = __fadd2_rn(make_float2(k2, k3), make_float2(r2, r3));
    z = v[8] + r8;
  }
  float2 xz;  // (x, z) after the next level; x the kept sum of this lane's half
  float x1;
  {
    const float s0 = b8 ? w01.x : w23.x, k0 = b8 ? w23.x : w01.x;
    const float s1 = b8 ? w01.y : w23.y, k1 = b8 ? w23.y : w01.y;
    const float r0 = __shfl_xor_sync(0xffffffffu, s0, 8), r1 = __shfl_xor_sync(0xffffffffu, s1, 8);
    const float r8 = __shfl_xor_sync(0xffffffffu, z, 8);
    const float2 x = __fadd2_rn(make_float2(k0, k1), make_float2(r0, r1));
    xz = make_float2(x.x, z + r8);
    x1 = x.y;
  }
  float2 yz;
  {
    const float send = b4 ? xz.x : x1;
    const float keep = b4 ? x1 : xz.x;
    const float r = __shfl_xor_sync(0xffffffffu, send, 4);
    const float r8 = __shfl_xor_sync(0xffffffffu, xz.y, 4);
    yz = __fadd2_rn(make_float2(keep, xz.y), make_float2(r, r8));
  }
#pragma unroll
  for (int o = 2; o >= 1; o >>= 1)
    yz = __fadd2_rn(yz, make_float2(__shfl_xor_sync(0xffffffffu, yz.x, o), __shfl_xor_sync(0xffffffffu, yz.y, o)));
  *out8 = yz.x;
  *out9 = yz.y;
}


__global__ void __launch_bounds__(32 * kBwdWarpsPerCta)
    k_render_bwd(const Rec* __restrict__ srec, const uint2* __restrict__ ranges, const uint32_t* __restrict__ n_isect,
                 uint32_t cap, int W, int H, int TX, float bg0, float bg1, float bg2, const float* __restrict__ image,
                 const float* __restrict__ target, const float* __restrict__ T_final,
                 const uint32_t* __restrict__ n_contrib, const uint32_t* __restrict__ cmask,
                 float* __restrict__ grad2d, int64_t n_pad, float* __restrict__ loss, float inv3P, float l1w,
                 const float* __restrict__ dLdC_extra, uint32_t* __restrict__ dev_status) {
  __shared__ __align__(128) Rec s_rec_all[kBwdWarpsPerCta][2][kBatch];
  __shared__ __align__(8) uint64_t s_bar_all[kBwdWarpsPerCta][2];

  const int warp = threadIdx.x >> 5;
  const int vb = int(blockIdx.x) * kBwdWarpsPerCta + warp;  // this warp's 8x4 block, over all tiles
  const int tile = vb / kBwdBlocksPerTile;
  const int block = vb % kBwdBlocksPerTile;  // the 8x4 block within the tile
  const int lane = threadIdx.x & 31;
  Rec (*s_rec)[kBatch] = s_rec_all[warp];
  uint64_t* s_bar = s_bar_all[warp];
  const int obx = (tile % TX) * kTile + (block & 1) * 8;
  const int oby = (tile / TX) * kTile + (block >> 1) * 4;
  const int pxi = obx + (lane & 7), pyi = oby + (lane >> 3);
  const bool inside = pxi < W && pyi < H;
  const float px = float(pxi) + 0.5f, py = float(pyi) + 0.5f;

  // per-pixel loss gradient
  float g0 = 0.0f, g1 = 0.0f, g2 = 0.0f, T = 1.0f, lsum = 0.0f;
  uint32_t nc = 0;
  if (inside) {
    const size_t P = size_t(W) * H;
    const size_t pix = size_t(pyi) * W + pxi;
    const float c0 = image[pix], c1 = image[P + pix], c2 = image[2 * P + pix];
    const float t0 = target[pix], t1 = target[P + pix], t2 = target[2 * P + pix];
    // d(l1w L1)/dC = l1w sign(C - C*) / (3 H W), plus any other loss term's gradient
    const float w1 = l1w * inv3P;
    g0 = (c0 > t0) ? w1 : ((c0 < t0) ? -w1 : 0.0f);
    g1 = (c1 > t1) ? w1 : ((c1 < t1) ? -w1 : 0.0f);
    g2 = (c2 > t2) ? w1 : ((c2 < t2) ? -w1 : 0.0f);
    if (dLdC_extra) {
      g0 += dLdC_extra[pix];
      g1 += dLdC_extra[P + pix];
      g2 += dLdC_extra[2 * P + pix];
    }
    lsum = fabsf(c0 - t0) + fabsf(c1 - t1) + fabsf(c2 - t2);
    T = T_final[pix];
    nc = n_contrib[pix];
  }
  // the warp's loss partial and its largest n_contrib
  float ls = lsum;
  uint32_t mx = nc;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    ls += __shfl_xor_sync(0xffffffffu, ls, o);
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  const uint32_t warp_max = mx;
  if (lane == 0) atomicAdd(loss, ls * (l1w * inv3P));

  const uint32_t K = min(*n_isect, cap);
  const uint2 rg = ranges[tile];
  const uint32_t start = min(rg.x, K), end = min(max(rg.y, rg.x), K);
  const uint32_t n_max = min(warp_max, end - start);
  if (n_max == 0) return;

  BatchStager<kBatch> st{srec + start, n_max, &s_rec[0][0], s_bar};
  const int nb = int((n_max + kBatch - 1) / kBatch);
  if (lane == 0) {
    mbar_init(&s_bar[0], 1);
    mbar_init(&s_bar[1], 1);
    fence_mbar_init();
  }
  __syncwarp();
  // batches are consumed last to first; u counts consumption order
  if (lane == 0) {
    st.issue(nb - 1, 0);
    if (nb > 1) st.issue(nb - 2, 1);
  }
  float acc0 = bg0, acc1 = bg1, acc2 = bg2;
  // The chunks are walked from the one holding entry n_max - 1 down to chunk 0; each
  // chunk's masks are loaded one chunk ahead, so the load overlaps the walk before it.
  int chunk = int((n_max - 1) >> 5);
  uint32_t next_mask = cmask[cmask_index(start, tile, uint32_t(chunk) << 5, block, lane)];
  for (int u = 0; u < nb; ++u) {
    const int b = nb - 1 - u;
    const int slot = u & 1;
    mbar_wait(&s_bar[slot], uint32_t((u >> 1) & 1), dev_status);
    const Rec* R = st.buffer(slot);
    const uint32_t pos0 = uint32_t(b) * kBatch;
    const int cnt = int(st.count(b));
    // this warp only needs entries below its largest n_contrib
    const int jmax = int(min(uint32_t(cnt), warp_max > pos0 ? warp_max - pos0 : 0u));
    // 32 entries at a time, from the top: the warp walks, from the highest down, the
    // entries that at least one of its pixels composited in the forward (the union of
    // the pixels' masks for this chunk); a pixel takes part in an entry its own mask has
    for (int j0 = ((jmax - 1) >> 5) << 5; j0 >= 0 && jmax > 0; j0 -= 32) {
      const uint32_t mine = next_mask;  // chunk (pos0 + j0) / 32
      --chunk;
      if (chunk >= 0) next_mask = cmask[cmask_index(start, tile, uint32_t(chunk) << 5, block, lane)];
      uint32_t any = __reduce_or_sync(0xffffffffu, mine);
      while (any) {
        const int hb = 31 - __clz(any);
        any &= ~(1u << hb);
        const int j = j0 + hb;
        const bool contrib = (mine >> hb) & 1u;
        const float4 ra = R[j].a;
        const float4 rb = R[j].b;
        const float4 rc = R[j].c;
        const float dx = __fsub_rn(px, ra.x), dy = __fsub_rn(py, ra.y);
        const float power = conic_power(dx, dy, ra.z, ra.w, rb.x);
        // the forward's decisions, recomputed for a composited entry in the same fp32
        // sequence: alpha and whether it sits at the 0.99 clamp.  Every lane evaluates
        // the entry; a lane that did not composite it carries alpha = 0, which leaves its
        // state unchanged and its partials zero (the warp stays converged).
        const float e = gs_expf_core(contrib ? power : 0.0f);
        const float vv = __fmul_rn(rb.y, e);
        const bool clamped = !(vv < kAlphaMax);
        const float alpha = contrib ? (clamped ? kAlphaMax : vv) : 0.0f;
        const float Ti = __fdividef(T, 1.0f - alpha);
        const float wgt = alpha * Ti;
        float v[9];
        v[6] = g0 * wgt;
        v[7] = g1 * wgt;
        v[8] = g2 * wgt;
        // colour of the entry minus the normalised colour behind it; the carried colour
        // then moves toward the entry's by alpha (acc + alpha (c - acc))
        const float d0 = rb.z - acc0, d1 = rb.w - acc1, d2 = rc.x - acc2;
        const float dLda = Ti * (g0 * d0 + g1 * d1 + g2 * d2);
        acc0 = fmaf(alpha, d0, acc0);
        acc1 = fmaf(alpha, d1, acc1);
        acc2 = fmaf(alpha, d2, acc2);
        T = contrib ? Ti : T;
        const bool lin = contrib && !clamped;
        const float dLdp = lin ? dLda * alpha : 0.0f;
        v[5] = lin ? dLda * e : 0.0f;
        // moments of q = dL/dpower over the offset (dx = px - mx, dy = py - my)
        v[0] = dLdp * dx;
        v[1] = dLdp * dy;
        v[2] = v[0] * dx;
        v[3] = v[0] * dy;
        v[4] = v[1] * dy;
        const uint32_t cm = __ballot_sync(0xffffffffu, contrib);
        float* slot_p = grad2d + int64_t(__float_as_uint(rc.y)) * GS_GRAD2D_STRIDE;
        if (__popc(cm) <= kDirectLanes) {
          // few contributing lanes: each adds its own partials with two vector atomics
          // and one scalar (no more L2 operations than the reduction's nine, without
          // its shuffles)
          if (contrib) {
            atomicAdd(reinterpret_cast<float4*>(slot_p), make_float4(v[0], v[1], v[2], v[3]));
            atomicAdd(reinterpret_cast<float4*>(slot_p) + 1, make_float4(v[4], v[5], v[6], v[7]));
            atomicAdd(slot_p + 8, v[8]);
          }
        } else {
          float s8, s9;
          warp_reduce9(v, &s8, &s9);
          // one atomic instruction: lanes 0, 4, ..., 28 add partials 0..7, lane 1
          // partial 8, all into the Gaussian's 12-float slot
          const bool nine = lane == 1;
          if (((lane & 3) == 0) || nine) atomicAdd(slot_p + (nine ? 8 : (lane >> 2)), nine ? s9 : s8);
        }
      }
    }
    __syncwarp();
    if (u + 2 < nb) {
      if (lane == 0) st.issue(nb - 1 - (u + 2), slot);
    }
  }
}

__global__ void k_zero4(float4* __restrict__ p, int64_t n4, float* __restrict__ scalar) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride)
    p[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  if (blockIdx.x == 0 && threadIdx.x == 0 && scalar) *scalar = 0.0f;
}

}  // namespace gs

extern "C" gs_status gs_render_bwd(gs_dims dims, const gs_camera* cam, const gs_bins* bins, uint32_t capacity_K,
                                   const float bg[3], const float* image, const float* target, const float* T_final,
                                   const uint32_t* n_contrib, const uint32_t* cmask, size_t cmask_bytes,
                                   float l1_weight, const float* dLdC_extra, float* grad2d, float* loss_out,
                                   uint32_t* dev_status, cudaStream_t stream) {
  using namespace gs;
  if (!dims_ok(dims) || !camera_ok(cam) || !bins || !bg || !image || !target || !T_final || !n_contrib || !cmask ||
      !grad2d || !loss_out || !dev_status)
    return GS_ERR_INVALID_ARG;
  if (!bins->rec || !bins->ranges || !bins->n_isect || capacity_K == 0) return GS_ERR_INVALID_ARG;
  if (!aligned(bins->rec, 16) || !aligned(bins->ranges, 8) || !aligned(grad2d, 16) || !aligned(cmask, 4))
    return GS_ERR_INVALID_ARG;
  if (cmask_bytes < gs_render_cmask_bytes(capacity_K, cam->width, cam->height)) return GS_ERR_INVALID_ARG;
  if (!(l1_weight >= 0.0f) || !std::isfinite(l1_weight)) return GS_ERR_INVALID_ARG;
  const int64_t n4 = int64_t(GS_GRAD2D_STRIDE) * dims.n_pad / 4;
  k_zero4<<<grid_for(n4, 256, sm_count() * 8), 256, 0, stream>>>(reinterpret_cast<float4*>(grad2d), n4, loss_out);
  const int TX = (cam->width + kTile - 1) / kTile;
  const int64_t tiles = n_tiles(cam);
  const float inv3P = float(1.0 / (3.0 * double(cam->width) * double(cam->height)));
  k_render_bwd<<<int(tiles * kBwdBlocksPerTile / kBwdWarpsPerCta), 32 * kBwdWarpsPerCta, 0, stream>>>(
      reinterpret_cast<const Rec*>(bins->rec), reinterpret_cast<const uint2*>(bins->ranges), bins->n_isect,
      capacity_K, cam->width, cam->height, TX, bg[0], bg[1], bg[2], image, target, T_final, n_contrib, cmask, grad2d,
      dims.n_pad, loss_out, inv3P, l1_weight, dLdC_extra, dev_status);
  return launch_status();
}
