// Plain CPU oracle for one 3D Gaussian Splatting optimisation step.
//
// TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call
// this file: only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg
// use it.  It shares no code, header, table or constant generator with the CUDA
// path; the two meet only through the seeded input generators in gs_inputs/.
//
// What it computes (the step of "3D Gaussian splatting for real-time radiance
// field rendering", Kerbl et al. 2023, which both pages point to as the method;
// the pages' own statement of the step is in "Scaling 3D Gaussian Splatting with
// Distributed Compute", sections on the Gaussian representation, the memory wall
// and the single-step walkthrough):
//
//   project      camera transform, covariance from scale and quaternion, EWA
//                projection to a 2D conic, radius, tile rect, sigmoid opacity,
//                degree-3 real SH colour                      (project_one)
//   bin          per tile, the ordered subsequence of the global (depth, index)
//                sorted list whose tile rect contains the tile (build_tile_lists)
//   render fwd   front-to-back alpha compositing per pixel    (render_pixel_fwd)
//   render bwd   L1 loss gradient, per-pixel analytic backward with explicit
//                suffix sums, per-Gaussian sums in fp64       (render_pixel_bwd)
//   project bwd  full chain rule back to the 59 parameters    (project_bwd_one)
//   adam         textbook Adam recurrence in fp64             (or_adam)
//
// Precision.  Every quantity that decides an integer (radius, tile rect, depth
// key, which entries a pixel composites, where it stops, the clamp at 0.99, the
// sign of the L1 residual) is decided in fp32 by a frozen operation sequence
// that the CUDA kernels follow too: explicit fma where an fma is meant, no
// contraction (this file is compiled with -ffp-contract=off), correctly rounded
// division and square root, and the exponential gs_expf below.  All values that
// do not decide an integer (gradients, suffix sums, Adam) are computed in fp64.
// The whole chain also has an fp64 instantiation, used by the finite-difference
// and closed-form pins.
//
// Readings where the pages are silent (each also listed in the design notes):
//   * low-pass 0.3 px^2 added to the 2D covariance; radius = ceil(3 sqrt(lambda_max))
//     with lambda_max = mid + sqrt(max(0.1, mid^2 - det)); Jacobian abscissae clamped
//     to 1.3 x the half field of view;
//   * alpha = min(0.99, o exp(power)); entries with power > 0 or alpha < 1/255 are
//     skipped; a pixel stops, without compositing, at the first entry that would
//     bring its transmittance below 1e-4; black background by default;
//   * the derivative of the 0.99 clamp is zero where it is active; the derivative
//     of a clamped Jacobian abscissa is zero; colour channels clamped at 0 pass no
//     gradient; radius and rect are constants for differentiation;
//   * pixel (i, j) has its centre at (i + 0.5, j + 0.5); tiles are 16 x 16 pixels.

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <functional>
#include <limits>
#include <thread>
#include <vector>

namespace {

constexpr int kPlanes = 59;   // 3 mean + 3 log-scale + 4 quaternion + 1 logit + 48 SH
constexpr int kTile = 16;     // tile edge in pixels
constexpr int kShCoeffs = 16; // degree 3

// --------------------------------------------------------------------------------
// Camera, in the same field order as the product's camera struct (but declared
// here independently): world->camera rotation (row-major), translation, pinhole
// intrinsics in pixels, image size, camera centre in world space, near plane.
struct OrCamera {
  float R[9];
  float t[3];
  float fx, fy, cx, cy;
  int32_t width, height;
  float campos[3];
  float near_z;
};

// --------------------------------------------------------------------------------
// Threading: a plain chunked parallel-for over [0, n).
int g_threads = 0;
int n_threads() {
  if (g_threads > 0) return g_threads;
  unsigned h = std::thread::hardware_concurrency();
  return h ? int(h) : 1;
}

void parallel_for(int64_t n, const std::function<void(int64_t, int64_t)>& fn) {
  int nt = n_threads();
  if (n <= 0) return;
  if (nt <= 1 || n < 64) {
    fn(0, n);
    return;
  }
  // dynamic chunks so that uneven tiles do not serialise on one thread
  int64_t chunk = std::max<int64_t>(1, n / (int64_t(nt) * 16));
  std::atomic<int64_t> next{0};
  std::vector<std::thread> pool;
  for (int t = 0; t < nt; ++t) {
    pool.emplace_back([&]() {
      for (;;) {
        int64_t b = next.fetch_add(chunk);
        if (b >= n) break;
        fn(b, std::min(n, b + chunk));
      }
    });
  }
  for (auto& th : pool) th.join();
}

// --------------------------------------------------------------------------------
// gs_expf: single-precision exponential from Cody and Waite's argument reduction
// (x = k ln2 + r with ln2 split into a short high part and a low part) and the
// degree-7 Taylor polynomial of e^r in Horner form, scaled by 2^k through the
// exponent field.  k is the integer nearest to x log2(e), rounded once from the exact
// product: fma(x, log2 e, 1.5 2^23) lands on an integer (its ulp is 1), and
// subtracting 1.5 2^23 again is exact.  Then |r| <= ln2/2 plus a rounding, and the
// truncation error r^8/8! <= 5.3e-9 stays below half an fp32 ulp.  Defined on
// [-87, 88], where every result is a normal number, so adding k to the exponent field
// is the exact product with 2^k; below that it returns 0, above +inf.
float gs_expf(float x) {
  if (!(x == x)) return x;
  if (x > 88.0f) return std::numeric_limits<float>::infinity();
  if (x < -87.0f) return 0.0f;
  const float kLog2e = 1.44269504088896341f;
  const float kRound = 12582912.0f;               // 1.5 * 2^23
  const float kLn2Hi = 0.693145751953125f;       // 16 significant bits
  const float kLn2Lo = 1.4286068203094173e-06f;  // ln2 - kLn2Hi
  const float kf = std::fma(x, kLog2e, kRound) - kRound;
  float r = std::fma(-kf, kLn2Hi, x);
  r = std::fma(-kf, kLn2Lo, r);
  float p = 1.0f / 5040.0f;
  p = std::fma(p, r, 1.0f / 720.0f);
  p = std::fma(p, r, 1.0f / 120.0f);
  p = std::fma(p, r, 1.0f / 24.0f);
  p = std::fma(p, r, 1.0f / 6.0f);
  p = std::fma(p, r, 0.5f);
  p = std::fma(p, r, 1.0f);
  p = std::fma(p, r, 1.0f);
  const int32_t k = int32_t(kf);
  uint32_t bits;
  std::memcpy(&bits, &p, 4);
  bits += uint32_t(k) << 23;  // k in [-126, 127]; the result stays normal
  float out;
  std::memcpy(&out, &bits, 4);
  return out;
}

template <class S> S ex(S x);
template <> float ex<float>(float x) { return gs_expf(x); }
template <> double ex<double>(double x) { return std::exp(x); }

template <class S> inline S fma_(S a, S b, S c) { return std::fma(a, b, c); }

// --------------------------------------------------------------------------------
// Real spherical harmonics up to degree 3 with the Condon-Shortley phase, index
// k = l^2 + l + m.  Y_lm = sqrt(2) K_l|m| P_l^|m|(cos t) cos(m phi)      (m > 0)
//                        = sqrt(2) K_l|m| P_l^|m|(cos t) sin(|m| phi)    (m < 0)
//                        = K_l0 P_l(cos t)                                (m = 0)
// with K_lm = sqrt((2l+1)/(4 pi) (l-m)!/(l+m)!).  Written as polynomials in the
// unit direction (x, y, z): sin^m(t) cos(m phi) = Re (x+iy)^m,
// sin^m(t) sin(m phi) = Im (x+iy)^m, cos t = z, and x^2+y^2+z^2 = 1 to put every
// l = 2, 3 polynomial in the homogeneous form used below.
double k_lm(int l, int m) {
  double ratio = 1.0;  // (l+m)! / (l-m)!
  for (int i = l - m + 1; i <= l + m; ++i) ratio *= double(i);
  return std::sqrt((2.0 * l + 1.0) / (4.0 * M_PI) / ratio);
}

struct ShConsts {
  double c0, c1;            // l = 0, 1
  double c2a, c2b, c2c;     // l = 2: xy-type, (2zz-xx-yy), (xx-yy)
  double c3a, c3b, c3c, c3d, c3e;  // l = 3
  ShConsts() {
    const double s2 = std::sqrt(2.0);
    c0 = k_lm(0, 0);
    c1 = k_lm(1, 0);                      // = sqrt(2) K_11; P_1^1 = -sin t
    // l = 2: P_2^2 = 3 sin^2, P_2^1 = -3 sin cos, P_2^0 = (3 cos^2 - 1)/2
    c2a = 3.0 * s2 * k_lm(2, 1);          // -c2a yz, -c2a xz; also 2 * 3 sqrt2 K22 for xy
    c2b = 0.5 * k_lm(2, 0);               // (3zz - 1)/2 = (2zz - xx - yy)/2
    c2c = 3.0 * s2 * k_lm(2, 2);          // Re (x+iy)^2 = xx - yy
    // l = 3: P_3^3 = -15 sin^3, P_3^2 = 15 sin^2 cos, P_3^1 = -(3/2)(5cos^2 - 1) sin,
    //        P_3^0 = (5 cos^3 - 3 cos)/2
    c3a = 15.0 * s2 * k_lm(3, 3);         // Re (x+iy)^3 = x(xx - 3yy), Im = y(3xx - yy)
    c3b = 2.0 * 15.0 * s2 * k_lm(3, 2);   // Im (x+iy)^2 z = 2 xyz
    c3c = 1.5 * s2 * k_lm(3, 1);          // (5zz - 1) = (4zz - xx - yy)
    c3d = 0.5 * k_lm(3, 0);               // z (5zz - 3) = z (2zz - 3xx - 3yy)
    c3e = 15.0 * s2 * k_lm(3, 2);         // Re (x+iy)^2 z = z (xx - yy)
  }
};
const ShConsts& sh_consts() {
  static ShConsts c;
  return c;
}

// The sixteen basis values in the frozen evaluation order.
template <class S>
void sh_basis(S x, S y, S z, S Y[kShCoeffs]) {
  const ShConsts& k = sh_consts();
  const S c0 = S(k.c0), c1 = S(k.c1), c2a = S(k.c2a), c2b = S(k.c2b), c2c = S(k.c2c);
  const S c3a = S(k.c3a), c3b = S(k.c3b), c3c = S(k.c3c), c3d = S(k.c3d), c3e = S(k.c3e);
  // xy-type l = 2 coefficient is twice the Re-part one's sqrt(2) K22 * 3
  const S c2xy = S(2.0 * 3.0 * std::sqrt(2.0) * k_lm(2, 2));
  S xx = x * x, yy = y * y, zz = z * z;
  S xy = x * y, yz = y * z, xz = x * z;
  Y[0] = c0;
  Y[1] = (-c1) * y;
  Y[2] = c1 * z;
  Y[3] = (-c1) * x;
  Y[4] = c2xy * xy;
  Y[5] = (-c2a) * yz;
  Y[6] = c2b * ((S(2) * zz - xx) - yy);
  Y[7] = (-c2a) * xz;
  Y[8] = c2c * (xx - yy);
  Y[9] = (-c3a) * (y * (S(3) * xx - yy));
  Y[10] = c3b * (xy * z);
  Y[11] = (-c3c) * (y * ((S(4) * zz - xx) - yy));
  Y[12] = c3d * (z * ((S(2) * zz - S(3) * xx) - S(3) * yy));
  Y[13] = (-c3c) * (x * ((S(4) * zz - xx) - yy));
  Y[14] = c3e * (z * (xx - yy));
  Y[15] = (-c3a) * (x * (xx - S(3) * yy));
}

// Gradient of each basis polynomial above with respect to (x, y, z), treating the
// three as independent (the normalisation Jacobian removes the radial part).
void sh_basis_grad(double x, double y, double z, double dY[kShCoeffs][3]) {
  const ShConsts& k = sh_consts();
  const double c2xy = 2.0 * 3.0 * std::sqrt(2.0) * k_lm(2, 2);
  double xx = x * x, yy = y * y, zz = z * z;
  auto set = [&](int i, double gx, double gy, double gz) {
    dY[i][0] = gx;
    dY[i][1] = gy;
    dY[i][2] = gz;
  };
  set(0, 0, 0, 0);
  set(1, 0, -k.c1, 0);
  set(2, 0, 0, k.c1);
  set(3, -k.c1, 0, 0);
  set(4, c2xy * y, c2xy * x, 0);
  set(5, 0, -k.c2a * z, -k.c2a * y);
  set(6, -2 * k.c2b * x, -2 * k.c2b * y, 4 * k.c2b * z);
  set(7, -k.c2a * z, 0, -k.c2a * x);
  set(8, 2 * k.c2c * x, -2 * k.c2c * y, 0);
  // y(3xx - yy)
  set(9, -k.c3a * 6 * x * y, -k.c3a * (3 * xx - 3 * yy), 0);
  // xyz
  set(10, k.c3b * y * z, k.c3b * x * z, k.c3b * x * y);
  // y(4zz - xx - yy)
  set(11, -k.c3c * (-2 * x * y), -k.c3c * (4 * zz - xx - 3 * yy), -k.c3c * 8 * y * z);
  // z(2zz - 3xx - 3yy)
  set(12, k.c3d * (-6 * x * z), k.c3d * (-6 * y * z), k.c3d * (6 * zz - 3 * xx - 3 * yy));
  // x(4zz - xx - yy)
  set(13, -k.c3c * (4 * zz - 3 * xx - yy), -k.c3c * (-2 * x * y), -k.c3c * 8 * x * z);
  // z(xx - yy)
  set(14, k.c3e * 2 * x * z, -k.c3e * 2 * y * z, k.c3e * (xx - yy));
  // x(xx - 3yy)
  set(15, -k.c3a * (3 * xx - 3 * yy), -k.c3a * (-6 * x * y), 0);
}

// --------------------------------------------------------------------------------
// Projection of one Gaussian.

template <class S>
struct Proj {
  bool visible = false;
  bool nonfinite = false;
  S mx = 0, my = 0;          // projected mean (pixels)
  S A = 0, B = 0, C = 0;     // conic: inverse of the 2D covariance [[a, b], [b, c]]
  S o = 0;                   // opacity
  S rgb[3] = {0, 0, 0};      // colour after +0.5 and the clamp at 0
  S z = 0;                   // depth (camera-space z)
  S cov_a = 0, cov_b = 0, cov_c = 0;  // 2D covariance incl. the 0.3 low-pass
  int radius = 0, tx0 = 0, ty0 = 0, tx1 = -1, ty1 = -1;
  uint32_t count = 0;
  bool clamp_rgb[3] = {false, false, false};
  bool clamp_x = false, clamp_y = false;
};

inline float param(const float* p, int64_t n_pad, int plane, int64_t i) {
  return p[int64_t(plane) * n_pad + i];
}

template <class S>
Proj<S> project_one(const float* params, int64_t n_pad, int64_t i, const OrCamera& cam) {
  Proj<S> g;
  // 11 geometric parameters must be finite
  for (int pl = 0; pl < 11; ++pl) {
    if (!std::isfinite(param(params, n_pad, pl, i))) {
      g.nonfinite = true;
      return g;
    }
  }
  const S mux = param(params, n_pad, 0, i), muy = param(params, n_pad, 1, i),
          muz = param(params, n_pad, 2, i);
  S Rc[9], Tc[3];
  for (int k = 0; k < 9; ++k) Rc[k] = S(cam.R[k]);
  for (int k = 0; k < 3; ++k) Tc[k] = S(cam.t[k]);
  const S fx = S(cam.fx), fy = S(cam.fy), cx = S(cam.cx), cy = S(cam.cy);

  // 1. camera transform t = R mu + t_c
  const S tx = fma_(Rc[0], mux, fma_(Rc[1], muy, fma_(Rc[2], muz, Tc[0])));
  const S ty = fma_(Rc[3], mux, fma_(Rc[4], muy, fma_(Rc[5], muz, Tc[1])));
  const S tz = fma_(Rc[6], mux, fma_(Rc[7], muy, fma_(Rc[8], muz, Tc[2])));
  if (!(tz > S(cam.near_z))) return g;
  g.z = tz;

  // 2. covariance Sigma = M M^T, M = R(q) diag(exp(log-scale))
  S s[3];
  for (int k = 0; k < 3; ++k) s[k] = ex<S>(S(param(params, n_pad, 3 + k, i)));
  const S qw0 = param(params, n_pad, 6, i), qx0 = param(params, n_pad, 7, i),
          qy0 = param(params, n_pad, 8, i), qz0 = param(params, n_pad, 9, i);
  const S n2 = fma_(qw0, qw0, fma_(qx0, qx0, fma_(qy0, qy0, qz0 * qz0)));
  if (!(n2 > S(0))) return g;
  const S qn = std::sqrt(n2);
  const S w = qw0 / qn, x = qx0 / qn, y = qy0 / qn, z = qz0 / qn;
  const S xx = x * x, yy = y * y, zz = z * z;
  const S xy = x * y, xz = x * z, yz = y * z;
  const S wx = w * x, wy = w * y, wz = w * z;
  S Rq[9];
  Rq[0] = S(1) - S(2) * (yy + zz);
  Rq[1] = S(2) * (xy - wz);
  Rq[2] = S(2) * (xz + wy);
  Rq[3] = S(2) * (xy + wz);
  Rq[4] = S(1) - S(2) * (xx + zz);
  Rq[5] = S(2) * (yz - wx);
  Rq[6] = S(2) * (xz - wy);
  Rq[7] = S(2) * (yz + wx);
  Rq[8] = S(1) - S(2) * (xx + yy);
  S M[9];
  for (int r = 0; r < 3; ++r)
    for (int c = 0; c < 3; ++c) M[r * 3 + c] = Rq[r * 3 + c] * s[c];
  auto sig = [&](int a, int b) {
    return fma_(M[a * 3 + 0], M[b * 3 + 0], fma_(M[a * 3 + 1], M[b * 3 + 1], M[a * 3 + 2] * M[b * 3 + 2]));
  };
  const S S00 = sig(0, 0), S01 = sig(0, 1), S02 = sig(0, 2);
  const S S11 = sig(1, 1), S12 = sig(1, 2), S22 = sig(2, 2);

  // 3. EWA: Jacobian of the perspective map at the mean, abscissae clamped
  const S u = tx / tz, v = ty / tz;
  const S limx = S(1.3) * ((S(0.5) * S(cam.width)) / fx);
  const S limy = S(1.3) * ((S(0.5) * S(cam.height)) / fy);
  S uc = u, vc = v;
  if (uc > limx) { uc = limx; g.clamp_x = true; }
  if (uc < -limx) { uc = -limx; g.clamp_x = true; }
  if (vc > limy) { vc = limy; g.clamp_y = true; }
  if (vc < -limy) { vc = -limy; g.clamp_y = true; }
  const S J00 = fx / tz, J02 = -((fx * uc) / tz);
  const S J11 = fy / tz, J12 = -((fy * vc) / tz);
  // T = J W (2x3), W = camera rotation
  S T0[3], T1[3];
  for (int j = 0; j < 3; ++j) {
    T0[j] = fma_(J00, Rc[0 * 3 + j], J02 * Rc[2 * 3 + j]);
    T1[j] = fma_(J11, Rc[1 * 3 + j], J12 * Rc[2 * 3 + j]);
  }
  const S Sg[3][3] = {{S00, S01, S02}, {S01, S11, S12}, {S02, S12, S22}};
  S V[3], U[3];
  for (int r = 0; r < 3; ++r) {
    V[r] = fma_(Sg[r][0], T0[0], fma_(Sg[r][1], T0[1], Sg[r][2] * T0[2]));
    U[r] = fma_(Sg[r][0], T1[0], fma_(Sg[r][1], T1[1], Sg[r][2] * T1[2]));
  }
  const S a = fma_(T0[0], V[0], fma_(T0[1], V[1], T0[2] * V[2])) + S(0.3);
  const S b = fma_(T1[0], V[0], fma_(T1[1], V[1], T1[2] * V[2]));
  const S c = fma_(T1[0], U[0], fma_(T1[1], U[1], T1[2] * U[2])) + S(0.3);
  g.cov_a = a;
  g.cov_b = b;
  g.cov_c = c;

  // 4. conic
  const S det = fma_(a, c, -(b * b));
  if (!std::isfinite(a) || !std::isfinite(b) || !std::isfinite(c) || !std::isfinite(det)) {
    g.nonfinite = true;
    return g;
  }
  if (!(det > S(0))) return g;
  g.A = c / det;
  g.B = -(b / det);
  g.C = a / det;

  // 5. radius and mean
  const S mid = S(0.5) * (a + c);
  const S disc = fma_(mid, mid, -det);
  const S lam = mid + std::sqrt(std::max(S(0.1), disc));
  S rf = std::ceil(S(3) * std::sqrt(lam));
  if (rf > S(16777216)) rf = S(16777216);
  g.mx = fma_(fx, u, cx);
  g.my = fma_(fy, v, cy);
  if (!std::isfinite(g.mx) || !std::isfinite(g.my)) {
    g.nonfinite = true;
    return g;
  }

  // 6. tile rect: tiles whose pixel span [16t, 16t+16) meets [m - r, m + r]
  const int TX = (cam.width + kTile - 1) / kTile, TY = (cam.height + kTile - 1) / kTile;
  const S inv_tile = S(0.0625);
  S fx0 = std::floor((g.mx - rf) * inv_tile), fx1 = std::floor((g.mx + rf) * inv_tile);
  S fy0 = std::floor((g.my - rf) * inv_tile), fy1 = std::floor((g.my + rf) * inv_tile);
  fx0 = std::max(fx0, S(0));
  fy0 = std::max(fy0, S(0));
  fx1 = std::min(fx1, S(TX - 1));
  fy1 = std::min(fy1, S(TY - 1));
  if (fx0 > fx1 || fy0 > fy1) return g;
  g.radius = int(rf);
  g.tx0 = int(fx0);
  g.tx1 = int(fx1);
  g.ty0 = int(fy0);
  g.ty1 = int(fy1);
  g.count = uint32_t(g.tx1 - g.tx0 + 1) * uint32_t(g.ty1 - g.ty0 + 1);

  // 7. opacity
  g.o = S(1) / (S(1) + ex<S>(-S(param(params, n_pad, 10, i))));

  // 8. colour: view direction from the camera centre, degree-3 SH, +0.5, clamp >= 0
  const S dx = mux - S(cam.campos[0]), dy = muy - S(cam.campos[1]), dz = muz - S(cam.campos[2]);
  const S len = std::sqrt(fma_(dx, dx, fma_(dy, dy, dz * dz)));
  S Y[kShCoeffs];
  sh_basis<S>(dx / len, dy / len, dz / len, Y);
  for (int ch = 0; ch < 3; ++ch) {
    S acc = Y[0] * S(param(params, n_pad, 11 + ch, i));
    for (int k = 1; k < kShCoeffs; ++k) acc = fma_(Y[k], S(param(params, n_pad, 11 + 3 * k + ch, i)), acc);
    for (int k = 0; k < kShCoeffs; ++k)
      if (!std::isfinite(param(params, n_pad, 11 + 3 * k + ch, i))) g.nonfinite = true;
    acc = acc + S(0.5);
    if (acc < S(0)) {
      g.clamp_rgb[ch] = true;
      acc = S(0);
    }
    g.rgb[ch] = acc;
  }
  if (g.nonfinite) {
    g.count = 0;
    return g;
  }
  g.visible = true;
  return g;
}

// --------------------------------------------------------------------------------
// Per-Gaussian projected data consumed by the renderer, in S precision.
template <class S>
struct Splat {
  S mx, my, A, B, C, o, rgb[3], z;
  int tx0, ty0, tx1, ty1;
  uint32_t count;
};

// Per tile: the ordered subsequence of the global (depth, index) order of
// all Gaussians with count > 0 whose rect contains the tile.  The predicate is
// evaluated tile row first (the rows a Gaussian spans), then per tile.
template <class S>
std::vector<std::vector<int32_t>> build_tile_lists(const std::vector<Splat<S>>& sp, int TX, int TY) {
  std::vector<int32_t> order;
  order.reserve(sp.size());
  for (size_t i = 0; i < sp.size(); ++i)
    if (sp[i].count > 0) order.push_back(int32_t(i));
  std::sort(order.begin(), order.end(), [&](int32_t p, int32_t q) {
    if (sp[p].z != sp[q].z) return sp[p].z < sp[q].z;
    return p < q;
  });
  std::vector<std::vector<int32_t>> lists(size_t(TX) * TY);
  parallel_for(TY, [&](int64_t r0, int64_t r1) {
    std::vector<int32_t> row;
    for (int64_t ty = r0; ty < r1; ++ty) {
      row.clear();
      for (int32_t g : order)
        if (sp[g].ty0 <= ty && ty <= sp[g].ty1) row.push_back(g);
      for (int tx = 0; tx < TX; ++tx) {
        auto& L = lists[size_t(ty) * TX + tx];
        for (int32_t g : row)
          if (sp[g].tx0 <= tx && tx <= sp[g].tx1) L.push_back(g);
      }
    }
  });
  return lists;
}

// One entry that a pixel composited, with the clamp decision.
struct Contrib {
  int32_t pos;  // position in the tile list
  bool clamped;
};

// Front-to-back compositing of one pixel in S precision.  Returns colour, final
// transmittance, the count of entries iterated up to the last composited one,
// and (optionally) the entries composited and how many there were.
template <class S>
void render_pixel_fwd(const std::vector<Splat<S>>& sp, const std::vector<int32_t>& L, S px, S py,
                      const S bg[3], S out[3], S* T_out, uint32_t* n_contrib,
                      std::vector<Contrib>* contribs, uint32_t* n_used = nullptr) {
  S T = S(1);
  S Cc[3] = {0, 0, 0};
  uint32_t last = 0, used = 0;
  const S one_255 = S(1) / S(255);
  for (size_t j = 0; j < L.size(); ++j) {
    const Splat<S>& g = sp[L[j]];
    // power = -A/2 dx^2 - B dx dy - C/2 dy^2, as dx (ca dx + cb dy) + cc dy dy with
    // (ca, cb, cc) = (-A/2, -B, -C/2)
    const S dx = px - g.mx, dy = py - g.my;
    const S ca = S(-0.5) * g.A, cb = -g.B, cc = S(-0.5) * g.C;
    const S power = fma_(dx, fma_(ca, dx, cb * dy), (cc * dy) * dy);
    if (power > S(0)) continue;
    const S v = g.o * ex<S>(power);
    const bool clamped = !(v < S(0.99));
    const S alpha = clamped ? S(0.99) : v;
    if (alpha < one_255) continue;
    // T (1 - alpha), evaluated as T - alpha T with one rounding
    const S Tn = fma_(-alpha, T, T);
    if (Tn < S(1e-4)) break;
    const S wgt = alpha * T;
    for (int ch = 0; ch < 3; ++ch) Cc[ch] = fma_(g.rgb[ch], wgt, Cc[ch]);
    T = Tn;
    last = uint32_t(j + 1);
    ++used;
    if (contribs) contribs->push_back({int32_t(j), clamped});
  }
  for (int ch = 0; ch < 3; ++ch) out[ch] = fma_(T, bg[ch], Cc[ch]);
  *T_out = T;
  *n_contrib = last;
  if (n_used) *n_used = used;
}

// Per-pixel backward with explicit suffix sums, all values in fp64.  The
// composited entries and clamp decisions come from the forward.  dLdC is the
// loss gradient with respect to the pixel colour.  Adds, per list position, the
// nine partials (d mean2d x, y; d conic A, B, C; d opacity; d r, g, b).
template <class S>
void render_pixel_bwd(const std::vector<Splat<S>>& sp, const std::vector<int32_t>& L, double px,
                      double py, const double bg[3], const std::vector<Contrib>& cs,
                      const double dLdC[3], double* entry_grads /* 9 per list position */) {
  const size_t m = cs.size();
  if (m == 0) return;
  std::vector<double> alpha(m), G(m), T(m + 1), dxs(m), dys(m);
  T[0] = 1.0;
  for (size_t k = 0; k < m; ++k) {
    const Splat<S>& g = sp[L[cs[k].pos]];
    const double dx = px - double(g.mx), dy = py - double(g.my);
    const double power = -0.5 * (double(g.A) * dx * dx + double(g.C) * dy * dy) - double(g.B) * dx * dy;
    G[k] = std::exp(power);
    alpha[k] = cs[k].clamped ? 0.99 : double(g.o) * G[k];
    dxs[k] = dx;
    dys[k] = dy;
    T[k + 1] = T[k] * (1.0 - alpha[k]);
  }
  // suffix sums S_k = sum_{j>k} c_j alpha_j T_j + T_m bg
  std::vector<double> Ssum(3 * m);
  double run[3] = {T[m] * bg[0], T[m] * bg[1], T[m] * bg[2]};
  for (size_t kk = m; kk-- > 0;) {
    for (int ch = 0; ch < 3; ++ch) Ssum[3 * kk + ch] = run[ch];
    const Splat<S>& g = sp[L[cs[kk].pos]];
    for (int ch = 0; ch < 3; ++ch) run[ch] += double(g.rgb[ch]) * alpha[kk] * T[kk];
  }
  for (size_t k = 0; k < m; ++k) {
    const Splat<S>& g = sp[L[cs[k].pos]];
    double* eg = entry_grads + 9 * size_t(cs[k].pos);
    double dLda = 0.0;
    for (int ch = 0; ch < 3; ++ch) {
      eg[6 + ch] += dLdC[ch] * alpha[k] * T[k];
      dLda += dLdC[ch] * (double(g.rgb[ch]) * T[k] - Ssum[3 * k + ch] / (1.0 - alpha[k]));
    }
    if (cs[k].clamped) continue;
    const double dLdpow = dLda * alpha[k];
    const double dx = dxs[k], dy = dys[k];
    const double A = g.A, B = g.B, C = g.C;
    eg[0] += dLdpow * (A * dx + B * dy);  // d power / d mx
    eg[1] += dLdpow * (B * dx + C * dy);  // d power / d my
    eg[2] += dLdpow * (-0.5 * dx * dx);
    eg[3] += dLdpow * (-dx * dy);
    eg[4] += dLdpow * (-0.5 * dy * dy);
    eg[5] += dLda * G[k];
  }
}

template <class S>
std::vector<Splat<S>> splats_from(int64_t n, const S* proj16, const int32_t* iproj6) {
  std::vector<Splat<S>> sp(static_cast<size_t>(n));
  for (int64_t i = 0; i < n; ++i) {
    const S* p = proj16 + 16 * i;
    const int32_t* q = iproj6 + 6 * i;
    Splat<S>& g = sp[size_t(i)];
    g.mx = p[0];
    g.my = p[1];
    g.A = p[2];
    g.B = p[3];
    g.C = p[4];
    g.o = p[5];
    g.rgb[0] = p[6];
    g.rgb[1] = p[7];
    g.rgb[2] = p[8];
    g.z = p[9];
    g.tx0 = q[1];
    g.ty0 = q[2];
    g.tx1 = q[3];
    g.ty1 = q[4];
    g.count = uint32_t(q[5]);
  }
  return sp;
}

// Forward (and optionally backward) over all tiles.
// The loss is l1_weight * mean |C - C*|; its gradient dL/dC = l1_weight sign(C - C*)
// / (3P) plus dLdC_extra (another loss term's gradient, e.g. D-SSIM), if given.
// n_used, if given, receives each pixel's count of composited entries.
template <class S>
void render_all(int64_t n, const S* proj16, const int32_t* iproj6, int W, int H, const S* bg_in,
                const S* target, S* image, S* T_final, uint32_t* n_contrib, double* grad2d,
                double* loss, double l1_weight = 1.0, const double* dLdC_extra = nullptr,
                uint32_t* n_used = nullptr) {
  const int TX = (W + kTile - 1) / kTile, TY = (H + kTile - 1) / kTile;
  std::vector<Splat<S>> sp = splats_from<S>(n, proj16, iproj6);
  auto lists = build_tile_lists<S>(sp, TX, TY);
  const S bg[3] = {bg_in[0], bg_in[1], bg_in[2]};
  const double bgd[3] = {double(bg_in[0]), double(bg_in[1]), double(bg_in[2])};
  const int64_t P = int64_t(W) * H;
  const bool backward = target != nullptr && grad2d != nullptr;
  std::vector<std::vector<double>> entry_grads(backward ? lists.size() : 0);
  std::vector<double> tile_loss(lists.size(), 0.0);
  const double inv3P = 1.0 / (3.0 * double(P));
  parallel_for(int64_t(lists.size()), [&](int64_t t0, int64_t t1) {
    std::vector<Contrib> cs;
    for (int64_t t = t0; t < t1; ++t) {
      const int tx = int(t % TX), ty = int(t / TX);
      const auto& L = lists[size_t(t)];
      if (backward) entry_grads[size_t(t)].assign(9 * L.size(), 0.0);
      double lsum = 0.0;
      for (int yy = ty * kTile; yy < std::min(H, ty * kTile + kTile); ++yy) {
        for (int xx = tx * kTile; xx < std::min(W, tx * kTile + kTile); ++xx) {
          const S px = S(xx) + S(0.5), py = S(yy) + S(0.5);
          S out[3], T;
          uint32_t nc, nu;
          cs.clear();
          render_pixel_fwd<S>(sp, L, px, py, bg, out, &T, &nc, backward ? &cs : nullptr, &nu);
          const int64_t pix = int64_t(yy) * W + xx;
          for (int ch = 0; ch < 3; ++ch) image[ch * P + pix] = out[ch];
          T_final[pix] = T;
          n_contrib[pix] = nc;
          if (n_used) n_used[pix] = nu;
          if (backward) {
            double dLdC[3];
            for (int ch = 0; ch < 3; ++ch) {
              const S r = out[ch] - target[ch * P + pix];
              // sign of the residual, taken on the S-precision image
              const double sg = (out[ch] > target[ch * P + pix]) ? 1.0 : ((out[ch] < target[ch * P + pix]) ? -1.0 : 0.0);
              lsum += std::fabs(double(out[ch]) - double(target[ch * P + pix]));
              (void)r;
              dLdC[ch] = l1_weight * sg * inv3P + (dLdC_extra ? dLdC_extra[ch * P + pix] : 0.0);
            }
            render_pixel_bwd<S>(sp, L, double(xx) + 0.5, double(yy) + 0.5, bgd, cs, dLdC,
                                entry_grads[size_t(t)].data());
          }
        }
      }
      tile_loss[size_t(t)] = lsum;
    }
  });
  if (backward) {
    std::fill(grad2d, grad2d + 9 * n, 0.0);
    // deterministic merge: tiles in order, entries in list order
    for (size_t t = 0; t < lists.size(); ++t) {
      const auto& L = lists[t];
      const auto& eg = entry_grads[t];
      for (size_t j = 0; j < L.size(); ++j)
        for (int q = 0; q < 9; ++q) grad2d[int64_t(q) * n + L[j]] += eg[9 * j + q];
    }
    double l = 0.0;
    for (double v : tile_loss) l += v;
    if (loss) *loss = l1_weight * l * inv3P;
  }
}

// --------------------------------------------------------------------------------
// Projection backward, fp64 values; decisions (culling, clamps) from the
// S-precision projection.
template <class S>
void project_bwd_one(const float* params, int64_t n_pad, int64_t i, const OrCamera& cam,
                     const double g2[9], double out[kPlanes]) {
  for (int k = 0; k < kPlanes; ++k) out[k] = 0.0;
  const Proj<S> dec = project_one<S>(params, n_pad, i, cam);
  if (!dec.visible) return;
  auto P = [&](int pl) { return double(param(params, n_pad, pl, i)); };
  const double mu[3] = {P(0), P(1), P(2)};
  double W[9], Tc[3];
  for (int k = 0; k < 9; ++k) W[k] = cam.R[k];
  for (int k = 0; k < 3; ++k) Tc[k] = cam.t[k];
  const double fx = cam.fx, fy = cam.fy;
  double t[3];
  for (int r = 0; r < 3; ++r) t[r] = W[3 * r] * mu[0] + W[3 * r + 1] * mu[1] + W[3 * r + 2] * mu[2] + Tc[r];
  const double tz = t[2];
  double s[3];
  for (int k = 0; k < 3; ++k) s[k] = std::exp(P(3 + k));
  const double q0[4] = {P(6), P(7), P(8), P(9)};
  const double qn = std::sqrt(q0[0] * q0[0] + q0[1] * q0[1] + q0[2] * q0[2] + q0[3] * q0[3]);
  const double w = q0[0] / qn, x = q0[1] / qn, y = q0[2] / qn, z = q0[3] / qn;
  const double Rq[9] = {1 - 2 * (y * y + z * z), 2 * (x * y - w * z),     2 * (x * z + w * y),
                        2 * (x * y + w * z),     1 - 2 * (x * x + z * z), 2 * (y * z - w * x),
                        2 * (x * z - w * y),     2 * (y * z + w * x),     1 - 2 * (x * x + y * y)};
  double M[9];
  for (int r = 0; r < 3; ++r)
    for (int c = 0; c < 3; ++c) M[3 * r + c] = Rq[3 * r + c] * s[c];
  double Sg[9];
  for (int r = 0; r < 3; ++r)
    for (int c = 0; c < 3; ++c)
      Sg[3 * r + c] = M[3 * r] * M[3 * c] + M[3 * r + 1] * M[3 * c + 1] + M[3 * r + 2] * M[3 * c + 2];
  const double u = t[0] / tz, v = t[1] / tz;
  const double limx = 1.3 * (0.5 * double(float(cam.width)) / fx);
  const double limy = 1.3 * (0.5 * double(float(cam.height)) / fy);
  const double uc = dec.clamp_x ? (u > 0 ? limx : -limx) : u;
  const double vc = dec.clamp_y ? (v > 0 ? limy : -limy) : v;
  const double J00 = fx / tz, J02 = -fx * uc / tz, J11 = fy / tz, J12 = -fy * vc / tz;
  double T0[3], T1[3];
  for (int j = 0; j < 3; ++j) {
    T0[j] = J00 * W[j] + J02 * W[6 + j];
    T1[j] = J11 * W[3 + j] + J12 * W[6 + j];
  }
  auto quad = [&](const double* p, const double* q) {
    double r = 0;
    for (int a = 0; a < 3; ++a)
      for (int b = 0; b < 3; ++b) r += p[a] * Sg[3 * a + b] * q[b];
    return r;
  };
  const double a = quad(T0, T0) + 0.3, b = quad(T0, T1), c = quad(T1, T1) + 0.3;
  const double det = a * c - b * b;
  const double d2 = det * det;

  // --- conic (A, B, C) -> 2D covariance (a, b, c)
  const double gA = g2[2], gB = g2[3], gC = g2[4];
  const double ga = gA * (-c * c / d2) + gB * (b * c / d2) + gC * (-b * b / d2);
  const double gb = gA * (2 * b * c / d2) + gB * (-(a * c + b * b) / d2) + gC * (2 * a * b / d2);
  const double gc = gA * (-b * b / d2) + gB * (a * b / d2) + gC * (-a * a / d2);

  // --- (a, b, c) -> T rows and Sigma
  double SgT0[3], SgT1[3];
  for (int r = 0; r < 3; ++r) {
    SgT0[r] = Sg[3 * r] * T0[0] + Sg[3 * r + 1] * T0[1] + Sg[3 * r + 2] * T0[2];
    SgT1[r] = Sg[3 * r] * T1[0] + Sg[3 * r + 1] * T1[1] + Sg[3 * r + 2] * T1[2];
  }
  double gT0[3], gT1[3];
  for (int j = 0; j < 3; ++j) {
    gT0[j] = 2 * ga * SgT0[j] + gb * SgT1[j];
    gT1[j] = gb * SgT0[j] + 2 * gc * SgT1[j];
  }
  // dL/dSigma_ij treating entries independently, then symmetrised for M
  double gS[9];
  for (int r = 0; r < 3; ++r)
    for (int cc = 0; cc < 3; ++cc)
      gS[3 * r + cc] = ga * T0[r] * T0[cc] + gb * T0[r] * T1[cc] + gc * T1[r] * T1[cc];

  // --- T = J W -> J entries
  double gJ00 = 0, gJ02 = 0, gJ11 = 0, gJ12 = 0;
  for (int j = 0; j < 3; ++j) {
    gJ00 += gT0[j] * W[j];
    gJ02 += gT0[j] * W[6 + j];
    gJ11 += gT1[j] * W[3 + j];
    gJ12 += gT1[j] * W[6 + j];
  }
  // --- J and mean2d -> camera-space t
  double gt[3] = {0, 0, 0};
  gt[2] += gJ00 * (-fx / (tz * tz)) + gJ11 * (-fy / (tz * tz));
  if (!dec.clamp_x) {
    gt[0] += gJ02 * (-fx / (tz * tz));
    gt[2] += gJ02 * (2 * fx * uc / (tz * tz));
  } else {
    gt[2] += gJ02 * (fx * uc / (tz * tz));
  }
  if (!dec.clamp_y) {
    gt[1] += gJ12 * (-fy / (tz * tz));
    gt[2] += gJ12 * (2 * fy * vc / (tz * tz));
  } else {
    gt[2] += gJ12 * (fy * vc / (tz * tz));
  }
  const double gmx = g2[0], gmy = g2[1];
  gt[0] += gmx * fx / tz;
  gt[1] += gmy * fy / tz;
  gt[2] += gmx * (-fx * t[0] / (tz * tz)) + gmy * (-fy * t[1] / (tz * tz));
  double gmu[3];
  for (int j = 0; j < 3; ++j) gmu[j] = W[j] * gt[0] + W[3 + j] * gt[1] + W[6 + j] * gt[2];

  // --- Sigma = M M^T -> M -> (R(q), s)
  double gM[9];
  for (int r = 0; r < 3; ++r)
    for (int k = 0; k < 3; ++k) {
      double acc = 0;
      for (int j = 0; j < 3; ++j) acc += (gS[3 * r + j] + gS[3 * j + r]) * M[3 * j + k];
      gM[3 * r + k] = acc;
    }
  double gs[3] = {0, 0, 0}, gR[9];
  for (int r = 0; r < 3; ++r)
    for (int k = 0; k < 3; ++k) {
      gs[k] += gM[3 * r + k] * Rq[3 * r + k];
      gR[3 * r + k] = gM[3 * r + k] * s[k];
    }
  for (int k = 0; k < 3; ++k) out[3 + k] = gs[k] * s[k];
  // R(q-hat) partials
  double gq[4];
  gq[0] = gR[1] * (-2 * z) + gR[2] * (2 * y) + gR[3] * (2 * z) + gR[5] * (-2 * x) + gR[6] * (-2 * y) +
          gR[7] * (2 * x);
  gq[1] = gR[1] * (2 * y) + gR[2] * (2 * z) + gR[3] * (2 * y) + gR[4] * (-4 * x) + gR[5] * (-2 * w) +
          gR[6] * (2 * z) + gR[7] * (2 * w) + gR[8] * (-4 * x);
  gq[2] = gR[0] * (-4 * y) + gR[1] * (2 * x) + gR[2] * (2 * w) + gR[3] * (2 * x) + gR[5] * (2 * z) +
          gR[6] * (-2 * w) + gR[7] * (2 * z) + gR[8] * (-4 * y);
  gq[3] = gR[0] * (-4 * z) + gR[1] * (-2 * w) + gR[2] * (2 * x) + gR[3] * (2 * w) + gR[4] * (-4 * z) +
          gR[5] * (2 * y) + gR[6] * (2 * x) + gR[7] * (2 * y);
  const double qh[4] = {w, x, y, z};
  const double dotq = gq[0] * qh[0] + gq[1] * qh[1] + gq[2] * qh[2] + gq[3] * qh[3];
  for (int k = 0; k < 4; ++k) out[6 + k] = (gq[k] - qh[k] * dotq) / qn;

  // --- opacity
  const double o = 1.0 / (1.0 + std::exp(-P(10)));
  out[10] = g2[5] * o * (1.0 - o);

  // --- colour
  const double vd[3] = {mu[0] - double(cam.campos[0]), mu[1] - double(cam.campos[1]),
                        mu[2] - double(cam.campos[2])};
  const double len = std::sqrt(vd[0] * vd[0] + vd[1] * vd[1] + vd[2] * vd[2]);
  const double d[3] = {vd[0] / len, vd[1] / len, vd[2] / len};
  double Y[kShCoeffs];
  sh_basis<double>(d[0], d[1], d[2], Y);
  double dY[kShCoeffs][3];
  sh_basis_grad(d[0], d[1], d[2], dY);
  double gd[3] = {0, 0, 0};
  for (int ch = 0; ch < 3; ++ch) {
    const double gcol = dec.clamp_rgb[ch] ? 0.0 : g2[6 + ch];
    for (int k = 0; k < kShCoeffs; ++k) {
      out[11 + 3 * k + ch] = Y[k] * gcol;
      const double shv = P(11 + 3 * k + ch);
      for (int e = 0; e < 3; ++e) gd[e] += gcol * shv * dY[k][e];
    }
  }
  const double dotd = gd[0] * d[0] + gd[1] * d[1] + gd[2] * d[2];
  for (int e = 0; e < 3; ++e) gmu[e] += (gd[e] - d[e] * dotd) / len;
  for (int e = 0; e < 3; ++e) out[e] = gmu[e];
}

// --------------------------------------------------------------------------------
// SSIM (Wang et al. 2004) with an 11x11 Gaussian window (sigma 1.5), C1 = 0.01^2,
// C2 = 0.03^2, zero padding outside the image, averaged over all pixels and
// channels: the D-SSIM term of the objective ("Scaling 3D Gaussian Splatting with
// Distributed Compute", objective paragraph: a weighted L1 plus D-SSIM; the formula
// was lost from the page, read here as (1 - lambda) L1 + lambda (1 - SSIM)).
// Everything in fp64 by direct summation of the 121-tap window.
struct SsimOut {
  double ssim;
};

void ssim_window(double w[11][11]) {
  double g[11], sum = 0.0;
  for (int k = 0; k < 11; ++k) {
    const double d = double(k - 5);
    g[k] = std::exp(-d * d / (2.0 * 1.5 * 1.5));
    sum += g[k];
  }
  for (int a = 0; a < 11; ++a)
    for (int b = 0; b < 11; ++b) w[a][b] = (g[a] / sum) * (g[b] / sum);
}

// L = lambda (1 - mean SSIM); returns mean SSIM and dL/dx (3 x H x W).
double ssim_and_grad(int W, int H, const double* x, const double* y, double lambda, double* dLdx) {
  const double C1 = 0.01 * 0.01, C2 = 0.03 * 0.03;
  double w[11][11];
  ssim_window(w);
  const int64_t P = int64_t(W) * H;
  std::vector<double> A(3 * P), B(3 * P), C(3 * P), S(3 * P);
  // local statistics and the partial derivatives of S at every pixel
  parallel_for(3 * int64_t(H), [&](int64_t r0, int64_t r1) {
    for (int64_t cr = r0; cr < r1; ++cr) {
      const int c = int(cr / H), i = int(cr % H);
      const double* xc = x + c * P;
      const double* yc = y + c * P;
      for (int j = 0; j < W; ++j) {
        double mx = 0, my = 0, exx = 0, eyy = 0, exy = 0;
        for (int a = -5; a <= 5; ++a) {
          const int ii = i + a;
          if (ii < 0 || ii >= H) continue;
          for (int b = -5; b <= 5; ++b) {
            const int jj = j + b;
            if (jj < 0 || jj >= W) continue;
            const double g = w[a + 5][b + 5];
            const double xv = xc[int64_t(ii) * W + jj], yv = yc[int64_t(ii) * W + jj];
            mx += g * xv;
            my += g * yv;
            exx += g * xv * xv;
            eyy += g * yv * yv;
            exy += g * xv * yv;
          }
        }
        const double sxx = exx - mx * mx, syy = eyy - my * my, sxy = exy - mx * my;
        const double n1 = 2 * mx * my + C1, n2 = 2 * sxy + C2;
        const double d1 = mx * mx + my * my + C1, d2 = sxx + syy + C2;
        const double s = n1 * n2 / (d1 * d2);
        const double dS_dmx = 2 * my * n2 / (d1 * d2) - s * 2 * mx / d1;
        const double dS_dsxx = -s / d2;
        const double dS_dsxy = 2 * n1 / (d1 * d2);
        const double dLdS = -lambda / double(3 * P);
        const int64_t q = c * P + int64_t(i) * W + j;
        S[q] = s;
        A[q] = dLdS * (dS_dmx - 2 * mx * dS_dsxx - my * dS_dsxy);
        B[q] = dLdS * dS_dsxx;
        C[q] = dLdS * dS_dsxy;
      }
    }
  });
  // dL/dx(p) = sum_q G(q - p) [A(q) + 2 x(p) B(q) + y(p) C(q)], q over the image
  parallel_for(3 * int64_t(H), [&](int64_t r0, int64_t r1) {
    for (int64_t cr = r0; cr < r1; ++cr) {
      const int c = int(cr / H), i = int(cr % H);
      for (int j = 0; j < W; ++j) {
        double ga = 0, gb = 0, gc = 0;
        for (int a = -5; a <= 5; ++a) {
          const int ii = i + a;
          if (ii < 0 || ii >= H) continue;
          for (int b = -5; b <= 5; ++b) {
            const int jj = j + b;
            if (jj < 0 || jj >= W) continue;
            const double g = w[a + 5][b + 5];
            const int64_t q = c * P + int64_t(ii) * W + jj;
            ga += g * A[q];
            gb += g * B[q];
            gc += g * C[q];
          }
        }
        const int64_t p = c * P + int64_t(i) * W + j;
        dLdx[p] = ga + 2 * x[p] * gb + y[p] * gc;
      }
    }
  });
  double sum = 0;
  for (double v : S) sum += v;
  return sum / double(3 * P);
}

}  // namespace

// ==================================================================================
// C entry points (ctypes).  Arrays are dense, C order, caller-owned.

extern "C" {

void or_set_threads(int n) { g_threads = n; }
int or_threads() { return n_threads(); }

void or_expf(const float* x, float* y, int64_t n) {
  for (int64_t i = 0; i < n; ++i) y[i] = gs_expf(x[i]);
}

// 16 real SH basis values per direction, fp64.
void or_sh_basis(const double* dirs, double* Y, int64_t n) {
  for (int64_t i = 0; i < n; ++i) sh_basis<double>(dirs[3 * i], dirs[3 * i + 1], dirs[3 * i + 2], Y + 16 * i);
}

// Projection.  proj16: per Gaussian (mx, my, A, B, C, o, r, g, b, z, cov_a, cov_b,
// cov_c, 0, 0, 0); iproj6: (radius, tx0, ty0, tx1, ty1, count); flags bit 0
// visible, bits 1-3 colour clamp r/g/b, bit 4 x clamp, bit 5 y clamp, bit 6
// non-finite input.  Returns the number of non-finite Gaussians.
#define OR_PROJECT_BODY(S)                                                                      \
  std::atomic<int64_t> bad{0};                                                                  \
  parallel_for(n, [&](int64_t b, int64_t e) {                                                   \
    for (int64_t i = b; i < e; ++i) {                                                           \
      Proj<S> g = project_one<S>(params, n_pad, i, *cam);                                       \
      S* p = proj16 + 16 * i;                                                                   \
      const S vals[16] = {g.mx, g.my, g.A, g.B, g.C, g.o, g.rgb[0], g.rgb[1], g.rgb[2], g.z,     \
                          g.cov_a, g.cov_b, g.cov_c, S(0), S(0), S(0)};                         \
      for (int k = 0; k < 16; ++k) p[k] = vals[k];                                              \
      int32_t* q = iproj6 + 6 * i;                                                              \
      q[0] = g.visible ? g.radius : 0;                                                          \
      q[1] = g.tx0;                                                                             \
      q[2] = g.ty0;                                                                             \
      q[3] = g.tx1;                                                                             \
      q[4] = g.ty1;                                                                             \
      q[5] = int32_t(g.visible ? g.count : 0);                                                  \
      flags[i] = uint32_t(g.visible) | (uint32_t(g.clamp_rgb[0]) << 1) |                        \
                 (uint32_t(g.clamp_rgb[1]) << 2) | (uint32_t(g.clamp_rgb[2]) << 3) |            \
                 (uint32_t(g.clamp_x) << 4) | (uint32_t(g.clamp_y) << 5) |                      \
                 (uint32_t(g.nonfinite) << 6);                                                  \
      if (g.nonfinite) bad.fetch_add(1);                                                        \
    }                                                                                           \
  });                                                                                           \
  return bad.load();

int64_t or_project_f32(const float* params, int64_t n, int64_t n_pad, const OrCamera* cam,
                       float* proj16, int32_t* iproj6, uint32_t* flags) {
  OR_PROJECT_BODY(float)
}
int64_t or_project_f64(const float* params, int64_t n, int64_t n_pad, const OrCamera* cam,
                       double* proj16, int32_t* iproj6, uint32_t* flags) {
  OR_PROJECT_BODY(double)
}

// Tile lists as the sorted key/id sequence: keys (tile << 32 | fp32 depth bits),
// ids, and per-tile [start, end).  Returns K (total intersections); writes at most
// cap entries.
int64_t or_tile_lists_f32(int64_t n, const float* proj16, const int32_t* iproj6, int W, int H,
                          uint64_t* keys, uint32_t* ids, uint32_t* ranges, int64_t cap) {
  const int TX = (W + kTile - 1) / kTile, TY = (H + kTile - 1) / kTile;
  std::vector<Splat<float>> sp = splats_from<float>(n, proj16, iproj6);
  auto lists = build_tile_lists<float>(sp, TX, TY);
  int64_t K = 0;
  for (size_t t = 0; t < lists.size(); ++t) {
    ranges[2 * t] = uint32_t(K);
    for (int32_t g : lists[t]) {
      if (K < cap) {
        uint32_t zb;
        std::memcpy(&zb, &sp[size_t(g)].z, 4);
        keys[K] = (uint64_t(t) << 32) | uint64_t(zb);
        ids[K] = uint32_t(g);
      }
      ++K;
    }
    ranges[2 * t + 1] = uint32_t(K);
  }
  return K;
}

// Render forward (and backward if target and grad2d are non-null).
// grad2d is 9 x n: (d mx, d my, d A, d B, d C, d o, d r, d g, d b).  n_used (null, or
// H x W) receives each pixel's count of composited entries.
void or_render_f32(int64_t n, const float* proj16, const int32_t* iproj6, int W, int H, const float* bg,
                   const float* target, float* image, float* T_final, uint32_t* n_contrib,
                   double* grad2d, double* loss, double l1_weight, const double* dLdC_extra, uint32_t* n_used) {
  render_all<float>(n, proj16, iproj6, W, H, bg, target, image, T_final, n_contrib, grad2d, loss, l1_weight,
                    dLdC_extra, n_used);
}
void or_render_f64(int64_t n, const double* proj16, const int32_t* iproj6, int W, int H,
                   const double* bg, const double* target, double* image, double* T_final,
                   uint32_t* n_contrib, double* grad2d, double* loss, double l1_weight,
                   const double* dLdC_extra, uint32_t* n_used) {
  render_all<double>(n, proj16, iproj6, W, H, bg, target, image, T_final, n_contrib, grad2d, loss, l1_weight,
                     dLdC_extra, n_used);
}

// Projection backward: grad2d (9 x n, fp64) -> grads (59 x n, fp64).  prec selects
// the precision the decisions are taken in (32 or 64).
void or_project_bwd(const float* params, int64_t n, int64_t n_pad, const OrCamera* cam, int prec,
                    const double* grad2d, double* grads) {
  parallel_for(n, [&](int64_t b, int64_t e) {
    double g2[9], out[kPlanes];
    for (int64_t i = b; i < e; ++i) {
      for (int q = 0; q < 9; ++q) g2[q] = grad2d[int64_t(q) * n + i];
      if (prec == 64)
        project_bwd_one<double>(params, n_pad, i, *cam, g2, out);
      else
        project_bwd_one<float>(params, n_pad, i, *cam, g2, out);
      for (int k = 0; k < kPlanes; ++k) grads[int64_t(k) * n + i] = out[k];
    }
  });
}

// SSIM of image x against y (3 x H x W each, fp64) and the gradient of
// lambda (1 - SSIM) with respect to x; returns the mean SSIM.
double or_ssim(int W, int H, const double* x, const double* y, double lambda, double* dLdx) {
  return ssim_and_grad(W, H, x, y, lambda, dLdx);
}

// Adam, textbook form in fp64: m = b1 m + (1-b1) g; v = b2 v + (1-b2) g^2;
// m_hat = m / (1 - b1^t); v_hat = v / (1 - b2^t); p -= lr m_hat / (sqrt(v_hat) + eps).
// Arrays are planes x stride; lr is per plane.
void or_adam(double* p, const double* g, double* m, double* v, int planes, int64_t stride,
             const double* lr, double beta1, double beta2, double eps, int64_t t) {
  const double bc1 = 1.0 - std::pow(beta1, double(t));
  const double bc2 = 1.0 - std::pow(beta2, double(t));
  parallel_for(int64_t(planes) * stride, [&](int64_t b, int64_t e) {
    for (int64_t i = b; i < e; ++i) {
      const int pl = int(i / stride);
      m[i] = beta1 * m[i] + (1.0 - beta1) * g[i];
      v[i] = beta2 * v[i] + (1.0 - beta2) * g[i] * g[i];
      const double mh = m[i] / bc1, vh = v[i] / bc2;
      p[i] -= lr[pl] * mh / (std::sqrt(vh) + eps);
    }
  });
}

}  // extern "C"
