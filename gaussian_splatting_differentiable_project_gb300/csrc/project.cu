// gs_project: one thread per Gaussian, coalesced reads of the 59 SoA parameter
// planes (each warp reads 128 contiguous bytes per plane), SH read only for
// Gaussians that survive culling, 48-byte record written per visible Gaussian.
#include "api_util.h"
#include "project_frozen.cuh"

namespace gs {

// Skip radius r of a record: at every pixel whose distance from the mean exceeds
// r the entry is skipped by the rasteriser anyway (alpha below 1/255, or power
// below the -5.6 skip threshold), so a warp whose pixels all lie farther than r
// may skip the entry without changing any decision.
//   lam >= the largest eigenvalue of the 2D covariance (the radius eigenvalue, with
//   its 0.1 floor), so the exact inverse gives power <= -|d|^2 / (2 lam).  alpha =
//   o e^power < 1/255 wherever power < -L with L = ln(255 o) (never above 5.54 <
//   5.6).  r^2 = 2.06 lam (L + 0.05) keeps the exact power below -(L + 0.05) by 3%:
//   the fp32 conic differs from the exact inverse by below 0.2% of mu_min while
//   lam <= 1424 (r <= 128 px, which bounds mu_max / mu_min by lam / 0.3), the fp32
//   power by a few ulp of mu_max |d|^2 (< 0.02 here) and the fp32 exponential and
//   product by a few ulp, all inside the 0.05 margin.  An opacity at most
//   0.999/255 is never composited (alpha <= o < 1/255): r = -inf (skip everywhere).
//   Beyond 128 px: +inf (never skip).
__device__ __forceinline__ float skip_radius(float lam, float o) {
  if (!(o * 255.0f > 0.999f)) return -__int_as_float(0x7f7fffff);
  const float L = logf(255.0f * o) + 0.05f;
  const float r = sqrtf(2.06f * lam * L) + 0.1f;
  return r <= 128.0f ? r : __int_as_float(0x7f7fffff);
}

__global__ void __launch_bounds__(256, 2)
    k_project(const float* __restrict__ P, int64_t n, int64_t n_pad, CamDev cam, float4* __restrict__ rec,
              float* __restrict__ depth, int32_t* __restrict__ radius, uint2* __restrict__ rect,
              uint32_t* __restrict__ count, uint32_t* __restrict__ dev_status) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n_pad; i += stride) {
    Geo g;
    g.visible = false;
    g.nonfinite = false;
    if (i < n) project_geo(P, n_pad, i, cam, g);
    bool vis = g.visible;
    bool nonfin = g.nonfinite;
    float o = 0.0f, rgb[3] = {0.0f, 0.0f, 0.0f};
    if (vis) {
      o = opacity_of(ldp(P, n_pad, 10, i));
      float d[3], len;
      view_dir(g.mux, g.muy, g.muz, cam, d, &len);
      float Y[16];
      sh_basis(d[0], d[1], d[2], Y);
      bool cl[3];
      sh_colour(P, n_pad, i, Y, rgb, cl, &nonfin);
      if (nonfin) vis = false;
    }
    if (nonfin) raise_status(dev_status, GS_ERR_NONFINITE);
    if (vis) {
      rec[3 * i + 0] = make_float4(g.mx, g.my, __fmul_rn(-0.5f, g.A), -g.B);
      rec[3 * i + 1] = make_float4(__fmul_rn(-0.5f, g.C), o, rgb[0], rgb[1]);
      rec[3 * i + 2] = make_float4(rgb[2], __uint_as_float(uint32_t(i)), skip_radius(g.lam, o), g.tz);
      depth[i] = g.tz;
      radius[i] = g.radius;
      rect[i] = make_uint2(uint32_t(g.tx0) | (uint32_t(g.ty0) << 16), uint32_t(g.tx1) | (uint32_t(g.ty1) << 16));
      count[i] = uint32_t(g.tx1 - g.tx0 + 1) * uint32_t(g.ty1 - g.ty0 + 1);
    } else {
      depth[i] = 0.0f;
      radius[i] = 0;
      rect[i] = make_uint2(0u, 0u);
      count[i] = 0u;
    }
  }
}

}  // namespace gs

extern "C" gs_status gs_project(gs_dims dims, const float* params, const gs_camera* cam, gs_proj proj,
                                uint32_t* dev_status, cudaStream_t stream) {
  using namespace gs;
  if (!dims_ok(dims) || !camera_ok(cam) || !params || !dev_status) return GS_ERR_INVALID_ARG;
  if (!proj.rec || !proj.depth || !proj.radius || !proj.rect || !proj.count) return GS_ERR_INVALID_ARG;
  if (!aligned(params, 16) || !aligned(proj.rec, 16) || !aligned(proj.rect, 8)) return GS_ERR_INVALID_ARG;
  if (dims.n == 0 && dims.n_pad == 0) return GS_OK;
  const int threads = 256;
  const int blocks = grid_for(dims.n_pad, threads, kSmCount * 64);
  k_project<<<blocks, threads, 0, stream>>>(params, dims.n, dims.n_pad, cam_dev(*cam),
                                            reinterpret_cast<float4*>(proj.rec), proj.depth, proj.radius,
                                            reinterpret_cast<uint2*>(proj.rect), proj.count, dev_status);
  return launch_status();
}
