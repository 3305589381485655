// Frozen fp32 projection of one Gaussian, shared by gs_project and gs_project_bwd.
//
// Follows the projection step of the 3DGS method ("Scaling 3D Gaussian Splatting
// with Distributed Compute", step walkthrough: project locally, SH to RGB before
// compositing): camera transform, Sigma = M M^T with M = R(q) diag(exp(s)), EWA
// 2D covariance with a 0.3 px^2 low-pass, conic, radius, tile rect, opacity,
// degree-3 SH colour.  Every operation that feeds a decision is an explicit
// round-to-nearest intrinsic so that the result is reproducible bit for bit.
#pragma once

#include "gs_common.cuh"

namespace gs {

// Real SH (Condon-Shortley phase) normalisations as polynomials in the unit
// direction: Y00 = 1/(2 sqrt pi); l = 1: sqrt(3/(4 pi)); l = 2: sqrt(15/(4 pi)),
// sqrt(5/(16 pi)), sqrt(15/(16 pi)); l = 3: sqrt(35/(32 pi)), sqrt(105/(4 pi)),
// sqrt(21/(32 pi)), sqrt(7/(16 pi)), sqrt(105/(16 pi)).
constexpr float kSh0 = 0.28209479177387814f;
constexpr float kSh1 = 0.48860251190291992f;
constexpr float kSh2a = 1.0925484305920792f;
constexpr float kSh2b = 0.31539156525252005f;
constexpr float kSh2c = 0.54627421529603959f;
constexpr float kSh3a = 0.59004358992664352f;
constexpr float kSh3b = 2.8906114426405538f;
constexpr float kSh3c = 0.45704579946446572f;
constexpr float kSh3d = 0.37317633259011540f;
constexpr float kSh3e = 1.4453057213202769f;

// The 16 basis values at the unit direction (x, y, z), index l^2 + l + m.
__device__ __forceinline__ void sh_basis(float x, float y, float z, float Y[16]) {
  const float xx = __fmul_rn(x, x), yy = __fmul_rn(y, y), zz = __fmul_rn(z, z);
  const float xy = __fmul_rn(x, y), yz = __fmul_rn(y, z), xz = __fmul_rn(x, z);
  Y[0] = kSh0;
  Y[1] = __fmul_rn(-kSh1, y);
  Y[2] = __fmul_rn(kSh1, z);
  Y[3] = __fmul_rn(-kSh1, x);
  Y[4] = __fmul_rn(kSh2a, xy);
  Y[5] = __fmul_rn(-kSh2a, yz);
  Y[6] = __fmul_rn(kSh2b, __fsub_rn(__fsub_rn(__fmul_rn(2.0f, zz), xx), yy));
  Y[7] = __fmul_rn(-kSh2a, xz);
  Y[8] = __fmul_rn(kSh2c, __fsub_rn(xx, yy));
  Y[9] = __fmul_rn(-kSh3a, __fmul_rn(y, __fsub_rn(__fmul_rn(3.0f, xx), yy)));
  Y[10] = __fmul_rn(kSh3b, __fmul_rn(xy, z));
  const float t4 = __fsub_rn(__fsub_rn(__fmul_rn(4.0f, zz), xx), yy);
  Y[11] = __fmul_rn(-kSh3c, __fmul_rn(y, t4));
  Y[12] = __fmul_rn(kSh3d, __fmul_rn(z, __fsub_rn(__fsub_rn(__fmul_rn(2.0f, zz), __fmul_rn(3.0f, xx)),
                                                   __fmul_rn(3.0f, yy))));
  Y[13] = __fmul_rn(-kSh3c, __fmul_rn(x, t4));
  Y[14] = __fmul_rn(kSh3e, __fmul_rn(z, __fsub_rn(xx, yy)));
  Y[15] = __fmul_rn(-kSh3a, __fmul_rn(x, __fsub_rn(xx, __fmul_rn(3.0f, yy))));
}

// Intermediate and final values of the projection.
struct Geo {
  bool visible;
  bool nonfinite;
  float mux, muy, muz;     // world-space mean
  float tx, ty, tz;        // camera-space mean
  float u, v;              // tx/tz, ty/tz
  float uc, vc;            // clamped abscissae used in the Jacobian
  bool clamp_x, clamp_y;
  float s[3];              // scales
  float qw, qx, qy, qz;    // normalised quaternion
  float qn;                // |q|
  float Rq[9];             // rotation R(q)
  float M[9];              // R diag(s)
  float S00, S01, S02, S11, S12, S22;  // Sigma
  float T0[3], T1[3];      // rows of J W
  float a, b, c, det;      // 2D covariance (+0.3) and its determinant
  float A, B, C;           // conic
  float lam;               // radius eigenvalue mid + sqrt(max(0.1, mid^2 - det))
  float mx, my;            // mean2d
  int radius;
  int tx0, ty0, tx1, ty1;
};

// Parameter load.  kReadOnly uses the read-only data path; kernels that also write
// the parameter planes (the fused projection backward + Adam) or read them from
// shared memory (the staged projection) use plain loads.
template <bool kReadOnly = true>
__device__ __forceinline__ float ldp(const float* P, int64_t n_pad, int plane, int64_t i) {
  if (kReadOnly) return __ldg(P + int64_t(plane) * n_pad + i);
  return P[int64_t(plane) * n_pad + i];
}

// Geometry: everything but opacity and colour.  Sets visible = false when the
// Gaussian is culled (behind the near plane, degenerate quaternion, det <= 0,
// empty tile rect) and nonfinite when a geometric parameter or derived value is
// NaN/Inf.
template <bool kReadOnly = true>
__device__ __forceinline__ void project_geo(const float* P, int64_t n_pad, int64_t i, const CamDev& cam, Geo& g) {
  g.visible = false;
  g.nonfinite = false;
  g.clamp_x = g.clamp_y = false;
  float pv[11];
#pragma unroll
  for (int pl = 0; pl < 11; ++pl) pv[pl] = ldp<kReadOnly>(P, n_pad, pl, i);
  bool fin = true;
#pragma unroll
  for (int pl = 0; pl < 11; ++pl) fin = fin && isfinite(pv[pl]);
  if (!fin) {
    g.nonfinite = true;
    return;
  }
  const float mux = pv[0], muy = pv[1], muz = pv[2];
  g.mux = mux;
  g.muy = muy;
  g.muz = muz;
  const float* R = cam.R;
  g.tx = __fmaf_rn(R[0], mux, __fmaf_rn(R[1], muy, __fmaf_rn(R[2], muz, cam.t[0])));
  g.ty = __fmaf_rn(R[3], mux, __fmaf_rn(R[4], muy, __fmaf_rn(R[5], muz, cam.t[1])));
  g.tz = __fmaf_rn(R[6], mux, __fmaf_rn(R[7], muy, __fmaf_rn(R[8], muz, cam.t[2])));
  if (!(g.tz > cam.near_z)) return;

  // covariance
#pragma unroll
  for (int k = 0; k < 3; ++k) g.s[k] = gs_expf(pv[3 + k]);
  const float qw0 = pv[6], qx0 = pv[7], qy0 = pv[8], qz0 = pv[9];
  const float n2 = __fmaf_rn(qw0, qw0, __fmaf_rn(qx0, qx0, __fmaf_rn(qy0, qy0, __fmul_rn(qz0, qz0))));
  if (!(n2 > 0.0f)) return;
  g.qn = __fsqrt_rn(n2);
  const float w = __fdiv_rn(qw0, g.qn), x = __fdiv_rn(qx0, g.qn), y = __fdiv_rn(qy0, g.qn),
              z = __fdiv_rn(qz0, g.qn);
  g.qw = w;
  g.qx = x;
  g.qy = y;
  g.qz = z;
  const float xx = __fmul_rn(x, x), yy = __fmul_rn(y, y), zz = __fmul_rn(z, z);
  const float xy = __fmul_rn(x, y), xz = __fmul_rn(x, z), yz = __fmul_rn(y, z);
  const float wx = __fmul_rn(w, x), wy = __fmul_rn(w, y), wz = __fmul_rn(w, z);
  g.Rq[0] = __fsub_rn(1.0f, __fmul_rn(2.0f, __fadd_rn(yy, zz)));
  g.Rq[1] = __fmul_rn(2.0f, __fsub_rn(xy, wz));
  g.Rq[2] = __fmul_rn(2.0f, __fadd_rn(xz, wy));
  g.Rq[3] = __fmul_rn(2.0f, __fadd_rn(xy, wz));
  g.Rq[4] = __fsub_rn(1.0f, __fmul_rn(2.0f, __fadd_rn(xx, zz)));
  g.Rq[5] = __fmul_rn(2.0f, __fsub_rn(yz, wx));
  g.Rq[6] = __fmul_rn(2.0f, __fsub_rn(xz, wy));
  g.Rq[7] = __fmul_rn(2.0f, __fadd_rn(yz, wx));
  g.Rq[8] = __fsub_rn(1.0f, __fmul_rn(2.0f, __fadd_rn(xx, yy)));
#pragma unroll
  for (int r = 0; r < 3; ++r)
#pragma unroll
    for (int c = 0; c < 3; ++c) g.M[r * 3 + c] = __fmul_rn(g.Rq[r * 3 + c], g.s[c]);
  const float* M = g.M;
#define GS_SIG(a_, b_) \
  __fmaf_rn(M[(a_)*3 + 0], M[(b_)*3 + 0], __fmaf_rn(M[(a_)*3 + 1], M[(b_)*3 + 1], __fmul_rn(M[(a_)*3 + 2], M[(b_)*3 + 2])))
  g.S00 = GS_SIG(0, 0);
  g.S01 = GS_SIG(0, 1);
  g.S02 = GS_SIG(0, 2);
  g.S11 = GS_SIG(1, 1);
  g.S12 = GS_SIG(1, 2);
  g.S22 = GS_SIG(2, 2);
#undef GS_SIG

  // EWA Jacobian
  g.u = __fdiv_rn(g.tx, g.tz);
  g.v = __fdiv_rn(g.ty, g.tz);
  const float limx = __fmul_rn(1.3f, __fdiv_rn(__fmul_rn(0.5f, float(cam.W)), cam.fx));
  const float limy = __fmul_rn(1.3f, __fdiv_rn(__fmul_rn(0.5f, float(cam.H)), cam.fy));
  float uc = g.u, vc = g.v;
  if (uc > limx) { uc = limx; g.clamp_x = true; }
  if (uc < -limx) { uc = -limx; g.clamp_x = true; }
  if (vc > limy) { vc = limy; g.clamp_y = true; }
  if (vc < -limy) { vc = -limy; g.clamp_y = true; }
  g.uc = uc;
  g.vc = vc;
  const float J00 = __fdiv_rn(cam.fx, g.tz), J02 = -__fdiv_rn(__fmul_rn(cam.fx, uc), g.tz);
  const float J11 = __fdiv_rn(cam.fy, g.tz), J12 = -__fdiv_rn(__fmul_rn(cam.fy, vc), g.tz);
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    g.T0[j] = __fmaf_rn(J00, R[j], __fmul_rn(J02, R[6 + j]));
    g.T1[j] = __fmaf_rn(J11, R[3 + j], __fmul_rn(J12, R[6 + j]));
  }
  const float Sg[3][3] = {{g.S00, g.S01, g.S02}, {g.S01, g.S11, g.S12}, {g.S02, g.S12, g.S22}};
  float V[3], U[3];
#pragma unroll
  for (int r = 0; r < 3; ++r) {
    V[r] = __fmaf_rn(Sg[r][0], g.T0[0], __fmaf_rn(Sg[r][1], g.T0[1], __fmul_rn(Sg[r][2], g.T0[2])));
    U[r] = __fmaf_rn(Sg[r][0], g.T1[0], __fmaf_rn(Sg[r][1], g.T1[1], __fmul_rn(Sg[r][2], g.T1[2])));
  }
  g.a = __fadd_rn(__fmaf_rn(g.T0[0], V[0], __fmaf_rn(g.T0[1], V[1], __fmul_rn(g.T0[2], V[2]))), 0.3f);
  g.b = __fmaf_rn(g.T1[0], V[0], __fmaf_rn(g.T1[1], V[1], __fmul_rn(g.T1[2], V[2])));
  g.c = __fadd_rn(__fmaf_rn(g.T1[0], U[0], __fmaf_rn(g.T1[1], U[1], __fmul_rn(g.T1[2], U[2]))), 0.3f);

  // conic
  g.det = __fmaf_rn(g.a, g.c, -__fmul_rn(g.b, g.b));
  if (!isfinite(g.a) || !isfinite(g.b) || !isfinite(g.c) || !isfinite(g.det)) {
    g.nonfinite = true;
    return;
  }
  if (!(g.det > 0.0f)) return;
  g.A = __fdiv_rn(g.c, g.det);
  g.B = -__fdiv_rn(g.b, g.det);
  g.C = __fdiv_rn(g.a, g.det);

  // radius and mean
  const float mid = __fmul_rn(0.5f, __fadd_rn(g.a, g.c));
  const float disc = __fmaf_rn(mid, mid, -g.det);
  const float lam = __fadd_rn(mid, __fsqrt_rn((0.1f < disc) ? disc : 0.1f));
  g.lam = lam;
  float rf = ceilf(__fmul_rn(3.0f, __fsqrt_rn(lam)));
  if (rf > 16777216.0f) rf = 16777216.0f;
  g.mx = __fmaf_rn(cam.fx, g.u, cam.cx);
  g.my = __fmaf_rn(cam.fy, g.v, cam.cy);
  if (!isfinite(g.mx) || !isfinite(g.my)) {
    g.nonfinite = true;
    return;
  }

  // tile rect
  float fx0 = floorf(__fmul_rn(__fsub_rn(g.mx, rf), 0.0625f));
  float fx1 = floorf(__fmul_rn(__fadd_rn(g.mx, rf), 0.0625f));
  float fy0 = floorf(__fmul_rn(__fsub_rn(g.my, rf), 0.0625f));
  float fy1 = floorf(__fmul_rn(__fadd_rn(g.my, rf), 0.0625f));
  fx0 = (fx0 < 0.0f) ? 0.0f : fx0;
  fy0 = (fy0 < 0.0f) ? 0.0f : fy0;
  const float lastx = float(cam.TX - 1), lasty = float(cam.TY - 1);
  fx1 = (lastx < fx1) ? lastx : fx1;
  fy1 = (lasty < fy1) ? lasty : fy1;
  if (fx0 > fx1 || fy0 > fy1) return;
  g.radius = int(rf);
  g.tx0 = int(fx0);
  g.tx1 = int(fx1);
  g.ty0 = int(fy0);
  g.ty1 = int(fy1);
  g.visible = true;
}

__device__ __forceinline__ float opacity_of(float logit) {
  return __fdiv_rn(1.0f, __fadd_rn(1.0f, gs_expf(-logit)));
}

// Unit view direction from the camera centre, its length, and the SH basis.
__device__ __forceinline__ void view_dir(float mux, float muy, float muz, const CamDev& cam, float d[3],
                                         float* len) {
  const float dx = __fsub_rn(mux, cam.campos[0]), dy = __fsub_rn(muy, cam.campos[1]),
              dz = __fsub_rn(muz, cam.campos[2]);
  const float l = __fsqrt_rn(__fmaf_rn(dx, dx, __fmaf_rn(dy, dy, __fmul_rn(dz, dz))));
  d[0] = __fdiv_rn(dx, l);
  d[1] = __fdiv_rn(dy, l);
  d[2] = __fdiv_rn(dz, l);
  *len = l;
}

// Colour: max(0, sum_k Y_k sh_k + 0.5) per channel, with the clamp flags; sets
// *nonfinite if any SH coefficient is NaN/Inf.
template <bool kReadOnly = true>
__device__ __forceinline__ void sh_colour(const float* __restrict__ P, int64_t n_pad, int64_t i,
                                          const float Y[16], float rgb[3], bool clamped[3], bool* nonfinite) {
  float acc[3];
  bool fin = true;
#pragma unroll
  for (int ch = 0; ch < 3; ++ch) {
    const float sh = ldp<kReadOnly>(P, n_pad, 11 + ch, i);
    fin = fin && isfinite(sh);
    acc[ch] = __fmul_rn(Y[0], sh);
  }
#pragma unroll
  for (int k = 1; k < 16; ++k) {
#pragma unroll
    for (int ch = 0; ch < 3; ++ch) {
      const float sh = ldp<kReadOnly>(P, n_pad, 11 + 3 * k + ch, i);
      fin = fin && isfinite(sh);
      acc[ch] = __fmaf_rn(Y[k], sh, acc[ch]);
    }
  }
#pragma unroll
  for (int ch = 0; ch < 3; ++ch) {
    float c = __fadd_rn(acc[ch], 0.5f);
    clamped[ch] = c < 0.0f;
    rgb[ch] = clamped[ch] ? 0.0f : c;
  }
  if (!fin) *nonfinite = true;
}

}  // namespace gs
