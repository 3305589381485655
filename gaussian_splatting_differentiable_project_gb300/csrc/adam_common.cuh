// Adam element update shared by gs_adam_step and the fused projection backward +
// Adam, so that both paths apply the same fp32 expression.
#pragma once

#include <cmath>

#include "gs_common.cuh"

namespace gs {

// Hyperparameters as the kernels use them: beta, 1 - beta, the bias corrections
// and lr / (1 - beta1^t) are formed on the host in fp64 and rounded to fp32 once.
struct AdamParams {
  float step[kPlanes];  // lr[plane] / (1 - beta1^t)
  float b1, c1, b2, c2, eps, inv_sqrt_bc2;
};

// Hyperparameters that do not change from step to step (a step count read from
// device memory completes them inside a kernel; see k_project_bwd_adam).
struct AdamHyper {
  float lr[kPlanes];
  double beta1, beta2, eps;
};

inline bool adam_hyper_ok(double beta1, double beta2, double eps) {
  return (beta1 >= 0.0 && beta1 < 1.0) && (beta2 >= 0.0 && beta2 < 1.0) && (eps >= 0.0);
}

// The same fp64 formation on the host (a step count known there) and on the device
// (a step count in device memory, for steps replayed from a CUDA graph).
__host__ __device__ inline void form_adam_params(const float lr_plane[kPlanes], double beta1, double beta2,
                                                 double eps, int64_t t, AdamParams& a) {
  const double bc1 = 1.0 - ::pow(beta1, double(t));
  const double bc2 = 1.0 - ::pow(beta2, double(t));
  for (int k = 0; k < kPlanes; ++k) a.step[k] = float(double(lr_plane[k]) / bc1);
  a.b1 = float(beta1);
  a.c1 = float(1.0 - beta1);
  a.b2 = float(beta2);
  a.c2 = float(1.0 - beta2);
  a.eps = float(eps);
  a.inv_sqrt_bc2 = float(1.0 / ::sqrt(bc2));
}

inline bool make_adam_params(const float lr_plane[kPlanes], double beta1, double beta2, double eps, int64_t t,
                             AdamParams& a) {
  if (t < 1 || !adam_hyper_ok(beta1, beta2, eps)) return false;
  form_adam_params(lr_plane, beta1, beta2, eps, t, a);
  return true;
}

// m = b1 m + (1 - b1) g; v = b2 v + (1 - b2) g^2; p -= step m / (sqrt(v) / sqrt(bc2) + eps)
//
// The square root and the division are the hardware approximations (relative error
// of order 2^-22 each), not the correctly rounded sequences: those made the update
// ALU-bound, and the fused projection backward + Adam ran 1.45x longer with them.
// The update step m / (...) is at most a few lr, so the approximations move p by
// about 1e-6 lr, far inside Adam's tolerance of 1e-5 |p| + 1e-7.  The denominator,
// at most the square root of fp32's largest value plus eps, stays far below 2^126,
// the bound of the range where the approximate division holds.
__device__ __forceinline__ float sqrt_approx(float x) {
  float r;
  asm("sqrt.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ void adam_elem(float& p, float& m, float& v, float g, float step, const AdamParams& a) {
  m = a.b1 * m + a.c1 * g;
  v = a.b2 * v + a.c2 * g * g;
  p -= __fdividef(step * m, sqrt_approx(v) * a.inv_sqrt_bc2 + a.eps);
}

}  // namespace gs
