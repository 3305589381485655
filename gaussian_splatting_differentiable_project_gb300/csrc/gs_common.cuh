// Device-side helpers shared by the sm_103a kernels of the 3DGS training step.
//
// The frozen fp32 operation sequence: every quantity that decides an integer
// (radius, tile rect, depth key, compositing decisions) is computed with explicit
// round-to-nearest intrinsics (__fmul_rn, __fadd_rn, __fsub_rn, __fmaf_rn,
// __fdiv_rn, __fsqrt_rn), which the compiler never contracts or reassociates, and
// with gs_expf below.  The same sequence written in plain C gives the same bits.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/gs.h"

namespace gs {

constexpr int kPlanes = GS_N_PLANES;
constexpr int kTile = GS_TILE;
constexpr int kTilePixels = kTile * kTile;
constexpr int kRecFloats = GS_REC_FLOATS;

// Record layout (3 x float4 = 48 bytes):
//   a = (mx, my, ca, cb)   b = (cc, opacity, r, g)   c = (b, id bits, 0, 0)
struct __align__(16) Rec {
  float4 a, b, c;
};

// ------------------------------------------------------------------ status bits
__device__ __forceinline__ void raise_status(uint32_t* dev_status, uint32_t bits) {
  if (dev_status) atomicOr(dev_status, bits);
}

// ------------------------------------------------------------------ exponential
// Cody-Waite: x = k ln2 + r, ln2 split into a 16-bit high part and the rest; e^r by
// its degree-7 Taylor polynomial in Horner form; times 2^k in the exponent field.
// k, the integer nearest to x log2(e), comes from one FMA against 1.5 * 2^23 (whose
// ulp is 1, so the sum is rounded to an integer from the exact product) and one exact
// subtraction: no float-to-integer conversions.  The low bits of that sum hold k
// (1.5 * 2^23's low nine bits are zero), so shifting its bits up by 23 gives k << 23,
// which added to the polynomial's bits scales it by 2^k exactly while the result is
// normal: x in [-87, 88].
__device__ __forceinline__ float gs_expf_core(float x) {
  const float kRound = 12582912.0f;  // 1.5 * 2^23
  const float s = __fmaf_rn(x, 1.44269504088896341f, kRound);
  const float kf = __fsub_rn(s, kRound);
  float r = __fmaf_rn(-kf, 0.693145751953125f, x);
  r = __fmaf_rn(-kf, 1.4286068203094173e-06f, r);
  float p = 1.0f / 5040.0f;
  p = __fmaf_rn(p, r, 1.0f / 720.0f);
  p = __fmaf_rn(p, r, 1.0f / 120.0f);
  p = __fmaf_rn(p, r, 1.0f / 24.0f);
  p = __fmaf_rn(p, r, 1.0f / 6.0f);
  p = __fmaf_rn(p, r, 0.5f);
  p = __fmaf_rn(p, r, 1.0f);
  p = __fmaf_rn(p, r, 1.0f);
  return __uint_as_float(__float_as_uint(p) + (__float_as_uint(s) << 23));
}

// Whole real line: NaN passes through, above 88 gives +inf, below -87 gives 0.
__device__ __forceinline__ float gs_expf(float x) {
  if (!(x == x)) return x;
  if (x > 88.0f) return __int_as_float(0x7f800000);
  if (x < -87.0f) return 0.0f;
  return gs_expf_core(x);
}

// ------------------------------------------------------------------ compositing
// Thresholds of the compositing rule.
constexpr float kAlphaMax = 0.99f;
constexpr float kAlphaMin = 1.0f / 255.0f;
constexpr float kTMin = 1e-4f;
// Below this power, o e^power < 1/255 for any opacity o <= 1 (e^-5.6 = 0.00370 <
// 1/255 = 0.00392 with a 6% margin), so the entry is skipped without evaluating
// the exponential.  It changes no decision.
constexpr float kPowerSkip = -5.6f;

// power = ca dx^2 + cb dx dy + cc dy^2 in the frozen order.
__device__ __forceinline__ float conic_power(float dx, float dy, float ca, float cb, float cc) {
  return __fmaf_rn(dx, __fmaf_rn(ca, dx, __fmul_rn(cb, dy)), __fmul_rn(__fmul_rn(cc, dy), dy));
}

// ------------------------------------------------------------------ camera
struct CamDev {
  float R[9];
  float t[3];
  float fx, fy, cx, cy;
  int W, H;
  float campos[3];
  float near_z;
  int TX, TY;
};

inline CamDev cam_dev(const gs_camera& c) {
  CamDev d;
  for (int k = 0; k < 9; ++k) d.R[k] = c.R[k];
  for (int k = 0; k < 3; ++k) d.t[k] = c.t[k];
  d.fx = c.fx;
  d.fy = c.fy;
  d.cx = c.cx;
  d.cy = c.cy;
  d.W = c.width;
  d.H = c.height;
  for (int k = 0; k < 3; ++k) d.campos[k] = c.campos[k];
  d.near_z = c.near_z;
  d.TX = (c.width + kTile - 1) / kTile;
  d.TY = (c.height + kTile - 1) / kTile;
  return d;
}

// ------------------------------------------------------------------ misc
// Streaming multiprocessors of the current device, queried once per device (api.cu);
// grids of the streaming and persistent kernels are sized from it.  Every kernel so
// sized loops over its work with a grid stride, so the count affects speed only.
int sm_count();

inline int grid_for(int64_t items, int threads, int max_blocks) {
  int64_t b = (items + threads - 1) / threads;
  if (b > max_blocks) b = max_blocks;
  if (b < 1) b = 1;
  return int(b);
}

}  // namespace gs
