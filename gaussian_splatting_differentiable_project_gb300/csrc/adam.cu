// gs_adam_step: fused Adam over the 59 x n_pad parameter planes.  Streams p, g,
// m, v once (float4 loads) and writes p, m, v once: 28 bytes per parameter.
// n_pad is a multiple of 256, so a float4 never straddles two planes.
#include "api_util.h"
#include "gs_common.cuh"

namespace gs {

struct AdamLr {
  float step[kPlanes];  // lr / (1 - beta1^t) per plane
};

__global__ void __launch_bounds__(256)
    k_adam(float4* __restrict__ p, const float4* __restrict__ g, float4* __restrict__ m, float4* __restrict__ v,
           int64_t n4, int64_t plane4, AdamLr lr, float b1, float c1, float b2, float c2, float eps,
           float inv_sqrt_bc2) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride) {
    const float step = lr.step[i / plane4];
    float4 pp = p[i];
    const float4 gg = __ldcs(g + i);
    float4 mm = m[i], vv = v[i];
#define GS_ADAM1(f)                                           \
  mm.f = b1 * mm.f + c1 * gg.f;                               \
  vv.f = b2 * vv.f + c2 * gg.f * gg.f;                        \
  pp.f -= step * mm.f / (sqrtf(vv.f) * inv_sqrt_bc2 + eps);
    GS_ADAM1(x) GS_ADAM1(y) GS_ADAM1(z) GS_ADAM1(w)
#undef GS_ADAM1
    p[i] = pp;
    __stcs(m + i, mm);
    __stcs(v + i, vv);
  }
}

}  // namespace gs

extern "C" gs_status gs_adam_step(gs_dims dims, float* params, const float* grads, float* m, float* v,
                                  const float lr_plane[GS_N_PLANES], double beta1, double beta2, double eps, int64_t t,
                                  cudaStream_t stream) {
  using namespace gs;
  if (!dims_ok(dims) || !params || !grads || !m || !v || !lr_plane) return GS_ERR_INVALID_ARG;
  if (!aligned(params, 16) || !aligned(grads, 16) || !aligned(m, 16) || !aligned(v, 16)) return GS_ERR_INVALID_ARG;
  if (t < 1 || !(beta1 >= 0.0 && beta1 < 1.0) || !(beta2 >= 0.0 && beta2 < 1.0) || !(eps >= 0.0))
    return GS_ERR_INVALID_ARG;
  const double bc1 = 1.0 - std::pow(beta1, double(t));
  const double bc2 = 1.0 - std::pow(beta2, double(t));
  AdamLr lr;
  for (int k = 0; k < kPlanes; ++k) lr.step[k] = float(double(lr_plane[k]) / bc1);
  const int64_t n4 = int64_t(kPlanes) * dims.n_pad / 4;
  const int blocks = grid_for(n4, 256, kSmCount * 16);
  k_adam<<<blocks, 256, 0, stream>>>(reinterpret_cast<float4*>(params), reinterpret_cast<const float4*>(grads),
                                     reinterpret_cast<float4*>(m), reinterpret_cast<float4*>(v), n4, dims.n_pad / 4, lr,
                                     float(beta1), float(1.0 - beta1), float(beta2), float(1.0 - beta2), float(eps),
                                     float(1.0 / std::sqrt(bc2)));
  return launch_status();
}
