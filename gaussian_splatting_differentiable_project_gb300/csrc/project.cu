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

constexpr int kProjGroup = 128;                                        // Gaussians per CTA group
constexpr size_t kProjSmem = 2 * size_t(kPlanes) * kProjGroup * sizeof(float);  // two groups of 59 planes: 60416 bytes

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
}

// One CTA takes groups of 128 consecutive Gaussians.  A group's 59 parameter planes
// (30 KB) are copied into shared memory with cp.async, all of them in flight at once,
// so one thread per Gaussian then projects from shared memory without the two
// dependent rounds of global loads (geometry, then SH for the visible) that bound it
// before.  The copies are double-buffered: the next group's planes are in flight while
// this group is projected, three CTAs to an SM.  The frozen operation sequence is
// unchanged.
__global__ void __launch_bounds__(kProjGroup, 3)
    k_project(const float* __restrict__ P, int64_t n, int64_t n_pad, CamDev cam, float4* __restrict__ rec,
              float* __restrict__ depth, int32_t* __restrict__ radius, uint2* __restrict__ rect,
              uint32_t* __restrict__ count, uint32_t* __restrict__ dev_status) {
  extern __shared__ __align__(16) float s_buf[];  // [2][kPlanes][kProjGroup]
  const int tid = threadIdx.x;
  constexpr int kRow4 = kProjGroup / 4;
  const int64_t gstride = int64_t(gridDim.x) * kProjGroup;
  auto stage = [&](int64_t g0, float* dst) {
    for (int e = tid; e < kPlanes * kRow4; e += kProjGroup) {
      const int pl = e / kRow4, q = (e % kRow4) * 4;
      cp_async16(dst + pl * kProjGroup + q, P + int64_t(pl) * n_pad + g0 + q);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  int buf = 0;
  if (int64_t(blockIdx.x) * kProjGroup < n_pad) stage(int64_t(blockIdx.x) * kProjGroup, s_buf);
  for (int64_t b0 = int64_t(blockIdx.x) * kProjGroup; b0 < n_pad; b0 += gstride) {
    float* s_p = s_buf + buf * (kPlanes * kProjGroup);
    if (b0 + gstride < n_pad) {
      stage(b0 + gstride, s_buf + (buf ^ 1) * (kPlanes * kProjGroup));
      asm volatile("cp.async.wait_group 1;" ::: "memory");
    } else {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
    __syncthreads();
    const int64_t i = b0 + tid;
    Geo g;
    g.visible = false;
    g.nonfinite = false;
    if (i < n) project_geo<false>(s_p, kProjGroup, tid, cam, g);
    bool vis = g.visible;
    bool nonfin = g.nonfinite;
    float o = 0.0f, rgb[3] = {0.0f, 0.0f, 0.0f};
    if (vis) {
      o = opacity_of(s_p[10 * kProjGroup + tid]);
      float d[3], len;
      view_dir(g.mux, g.muy, g.muz, cam, d, &len);
      float Y[16];
      sh_basis(d[0], d[1], d[2], Y);
      bool cl[3];
      sh_colour<false>(s_p, kProjGroup, tid, Y, rgb, cl, &nonfin);
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
    __syncthreads();  // the group's planes are read before this buffer is staged again
    buf ^= 1;
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
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(k_project, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kProjSmem)) != cudaSuccess)
      return GS_ERR_CUDA;
    attr_set = true;
  }
  const int blocks = grid_for(dims.n_pad / kProjGroup, 1, sm_count() * 3);
  k_project<<<blocks, kProjGroup, kProjSmem, stream>>>(params, dims.n, dims.n_pad, cam_dev(*cam),
                                                      reinterpret_cast<float4*>(proj.rec), proj.depth, proj.radius,
                                                      reinterpret_cast<uint2*>(proj.rect), proj.count, dev_status);
  return launch_status();
}
