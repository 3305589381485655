// gs_adam_step: fused Adam over the 59 x n_pad parameter planes.  Streams p, g,
// m, v once (float4 loads) and writes p, m, v once: 28 bytes per parameter.
// n_pad is a multiple of 256, so a float4 never straddles two planes.
#include "api_util.h"
#include "adam_common.cuh"

namespace gs {

__global__ void __launch_bounds__(256)
    k_adam(float4* __restrict__ p, const float4* __restrict__ g, float4* __restrict__ m, float4* __restrict__ v,
           int64_t n4, int64_t plane4, AdamParams a) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride) {
    const float step = a.step[i / plane4];
    float4 pp = p[i];
    const float4 gg = __ldcs(g + i);
    float4 mm = m[i], vv = v[i];
    adam_elem(pp.x, mm.x, vv.x, gg.x, step, a);
    adam_elem(pp.y, mm.y, vv.y, gg.y, step, a);
    adam_elem(pp.z, mm.z, vv.z, gg.z, step, a);
    adam_elem(pp.w, mm.w, vv.w, gg.w, step, a);
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
  AdamParams a;
  if (!make_adam_params(lr_plane, beta1, beta2, eps, t, a)) return GS_ERR_INVALID_ARG;
  const int64_t n4 = int64_t(kPlanes) * dims.n_pad / 4;
  const int blocks = grid_for(n4, 256, sm_count() * 16);
  k_adam<<<blocks, 256, 0, stream>>>(reinterpret_cast<float4*>(params), reinterpret_cast<const float4*>(grads),
                                     reinterpret_cast<float4*>(m), reinterpret_cast<float4*>(v), n4, dims.n_pad / 4, a);
  return launch_status();
}
