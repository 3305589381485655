// D-SSIM term of the objective: SSIM with an 11x11 Gaussian window (sigma 1.5,
// separable), C1 = 0.01^2, C2 = 0.03^2, zero padding, averaged over 3 H W values.
//
// Both kernels take a 32x32 output tile per 256-thread CTA, one channel at a time: the
// planes they filter are staged with a 5-pixel halo (42x42, zero outside the image),
// a horizontal 11-tap pass writes the 42 staged rows x 32 columns, and a vertical pass
// finishes in registers.  In each pass a thread produces 4 adjacent outputs from a
// 14-value window held in registers, so a staged value is read once per 4 outputs.
// Staging is by cp.async (4 bytes per value, zero-filled outside the image), so all of
// a channel's loads are in flight together and hold no registers; the next channel's
// staging is issued as soon as the horizontal pass has read the current one, and
// lands while the vertical pass and the per-pixel work run.
//
// gs_ssim_fwd: the local means, variances and covariance, then per pixel the partial
//   derivatives of S times dL/dS = -lambda / (3 H W):
//     a = dL/dS dS/dmu_x,  b = dL/dS dS/ds_xx,  c = dL/dS dS/ds_xy,
//   stored with the local means mu_x, mu_y; the CTA adds its share of mean S.  The
//   moments are taken about a shift per CTA and channel (the tile-centre value of each
//   image; the zero padding is staged as 0 - shift): the window weights sum to 1, so the
//   variance and covariance do not change, while E[x^2] - mu^2 no longer cancels in flat
//   regions (exactly zero there).
// gs_ssim_bwd: with s_x, s_y a shift of its own (the tile-centre values again),
//     dL/dx_j = sum_i g_ij [a_i + 2 (x_j - mu_x,i) b_i + (y_j - mu_y,i) c_i]
//             = G * A + 2 (x_j - s_x) (G * b) + (y_j - s_y) (G * c),
//     A = a - 2 (mu_x - s_x) b - (mu_y - s_y) c,
//   (the window is symmetric, so the transposed filter is G itself).  Folding the means
//   in about the shift rather than about zero keeps the terms that cancel small.
#include <cmath>

#include "api_util.h"
#include "gs_common.cuh"

namespace gs {

constexpr int kSsimTile = 32;                      // output tile edge
constexpr int kSsimHalo = 5;                       // window radius
constexpr int kSsimIn = kSsimTile + 2 * kSsimHalo; // 42 staged rows / columns
constexpr int kSsimInStride = 43;                  // odd: a warp's 14-wide windows hit distinct banks
constexpr int kSsimHStride = 33;                   // horizontal-pass rows: conflict-free column stores
constexpr int kSsimGroup = 4;                      // outputs per thread per pass
constexpr int kSsimWin = kSsimGroup + 10;          // values a group of 4 outputs reads
constexpr int kSsimThreads = 256;
constexpr int kSsimHItems = kSsimIn * (kSsimTile / kSsimGroup);  // 42 rows x 8 column groups
constexpr float kC1 = 0.01f * 0.01f;
constexpr float kC2 = 0.03f * 0.03f;
static_assert(kSsimThreads == kSsimTile * (kSsimTile / kSsimGroup), "one vertical group per thread");

struct SsimWindow {
  float g[11];  // normalised 1D Gaussian, sigma 1.5
};

inline SsimWindow ssim_window() {
  SsimWindow w;
  double sum = 0.0, g[11];
  for (int k = 0; k < 11; ++k) {
    const double d = double(k - 5);
    g[k] = std::exp(-d * d / 4.5);
    sum += g[k];
  }
  for (int k = 0; k < 11; ++k) w.g[k] = float(g[k] / sum);
  return w;
}

// 4-byte cp.async global -> shared; with `in` false nothing is read and the 4 bytes
// are zero-filled (src must still be a valid address).
__device__ __forceinline__ void cp_async4_zfill(float* dst, const float* src, bool in) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(d), "l"(src), "r"(in ? 4 : 0) : "memory");
}
__device__ __forceinline__ void ssim_cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void ssim_cp_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Issue the staging of NQ planes of channel c (plane q at base[q] + c P) with the
// halo into s[q][42][43], values outside the image 0; one commit group.
template <int NQ>
__device__ __forceinline__ void ssim_stage(float (*s)[kSsimIn][kSsimInStride], const float* const (&base)[NQ], int W,
                                           int H, int64_t P, int c, int ox, int oy) {
  // element k = threadIdx.x + 256 i of the 42 x 42 block: (row, column) stepped by
  // (6, 4) per i, with a carry, instead of a division per element
  int r = threadIdx.x / kSsimIn, col = threadIdx.x - r * kSsimIn;
  for (int k = threadIdx.x; k < kSsimIn * kSsimIn; k += kSsimThreads) {
    const int gy = oy - kSsimHalo + r, gx = ox - kSsimHalo + col;
    const bool in = gx >= 0 && gx < W && gy >= 0 && gy < H;
    const int64_t e = in ? int64_t(c) * P + int64_t(gy) * W + gx : 0;
#pragma unroll
    for (int q = 0; q < NQ; ++q) cp_async4_zfill(&s[q][r][col], base[q] + e, in);
    static_assert(kSsimThreads == 6 * kSsimIn + 4, "row / column step of the staging loop");
    col += 4;
    r += 6;
    if (col >= kSsimIn) {
      col -= kSsimIn;
      r += 1;
    }
  }
  ssim_cp_commit();
}

// out[j] += sum_t g[t] v[j + t] for the 4 outputs of a group.
__device__ __forceinline__ void ssim_tap4(float (&out)[kSsimGroup], const float (&v)[kSsimWin], const SsimWindow& w) {
#pragma unroll
  for (int k = 0; k < kSsimWin; ++k)
#pragma unroll
    for (int j = 0; j < kSsimGroup; ++j)
      if (k - j >= 0 && k - j < 11) out[j] = fmaf(w.g[k - j], v[k], out[j]);
}

// ssim_tap4 on two maps at once: out[j] (a pair of maps) += g v[k] (a pair) with the
// two-wide fused multiply-add, each half rounded as fmaf, in the same order.
__device__ __forceinline__ void ssim_tap4x2(float2 (&out)[kSsimGroup], const float2 (&v)[kSsimWin],
                                            const SsimWindow& w) {
#pragma unroll
  for (int k = 0; k < kSsimWin; ++k)
#pragma unroll
    for (int j = 0; j < kSsimGroup; ++j)
      if (k - j >= 0 && k - j < 11) out[j] = __ffma2_rn(make_float2(w.g[k - j], w.g[k - j]), v[k], out[j]);
}

// Four CTAs per SM (at most 64 registers a thread; it needs 51 so, 73 unbounded).
__global__ void __launch_bounds__(kSsimThreads, 4)
    k_ssim_fwd(const float* __restrict__ x, const float* __restrict__ y, int W, int H, SsimWindow w, float dLdS,
               float inv3P, float* __restrict__ maps, float* __restrict__ ssim_out) {
  __shared__ float s_in[2][kSsimIn][kSsimInStride];
  __shared__ float s_h[5][kSsimIn][kSsimHStride];
  __shared__ float s_red[kSsimThreads / 32];
  const int ox = blockIdx.x * kSsimTile, oy = blockIdx.y * kSsimTile;
  const int64_t P = int64_t(W) * H;
  const int vcol = threadIdx.x % kSsimTile, vrow = (threadIdx.x / kSsimTile) * kSsimGroup;
  const int64_t centre = int64_t(min(oy + kSsimTile / 2, H - 1)) * W + min(ox + kSsimTile / 2, W - 1);
  float ssum = 0.0f;
  const float* const planes[2] = {x, y};
  ssim_stage<2>(s_in, planes, W, H, P, 0, ox, oy);
  for (int c = 0; c < 3; ++c) {
    const float shift[2] = {x[c * P + centre], y[c * P + centre]};
    ssim_cp_wait_all();
    __syncthreads();  // channel c staged for every thread; the previous vertical pass done with s_h
    // horizontal: moments of the shifted values (x, y, x^2, y^2, x y) along rows; the
    // shift is taken here (outside the image: 0 - shift)
    for (int i = threadIdx.x; i < kSsimHItems; i += kSsimThreads) {
      const int r = i % kSsimIn, c0 = (i / kSsimIn) * kSsimGroup;
      // (x, y) and (x^2, y^2) as pairs for the two-wide taps, x y alone
      float2 ab[kSsimWin], sq[kSsimWin];
      float xy[kSsimWin];
#pragma unroll
      for (int k = 0; k < kSsimWin; ++k) {
        ab[k] = make_float2(s_in[0][r][c0 + k] - shift[0], s_in[1][r][c0 + k] - shift[1]);
        sq[k] = make_float2(ab[k].x * ab[k].x, ab[k].y * ab[k].y);
        xy[k] = ab[k].x * ab[k].y;
      }
      float2 m01[kSsimGroup], m23[kSsimGroup];
      float m4[kSsimGroup] = {};
#pragma unroll
      for (int j = 0; j < kSsimGroup; ++j) m01[j] = m23[j] = make_float2(0.0f, 0.0f);
      ssim_tap4x2(m01, ab, w);
      ssim_tap4x2(m23, sq, w);
      ssim_tap4(m4, xy, w);
#pragma unroll
      for (int j = 0; j < kSsimGroup; ++j) {
        s_h[0][r][c0 + j] = m01[j].x;
        s_h[1][r][c0 + j] = m01[j].y;
        s_h[2][r][c0 + j] = m23[j].x;
        s_h[3][r][c0 + j] = m23[j].y;
        s_h[4][r][c0 + j] = m4[j];
      }
    }
    __syncthreads();  // s_in read by every thread: the next channel may land there
    if (c + 1 < 3) ssim_stage<2>(s_in, planes, W, H, P, c + 1, ox, oy);
    // vertical: 4 rows of one column per thread
    float m[5][kSsimGroup] = {};
    {
      float2 m01[kSsimGroup], m23[kSsimGroup];
#pragma unroll
      for (int j = 0; j < kSsimGroup; ++j) m01[j] = m23[j] = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int q = 0; q < 4; q += 2) {
        float2 v[kSsimWin];
#pragma unroll
        for (int k = 0; k < kSsimWin; ++k) v[k] = make_float2(s_h[q][vrow + k][vcol], s_h[q + 1][vrow + k][vcol]);
        ssim_tap4x2(q == 0 ? m01 : m23, v, w);
      }
      float v4[kSsimWin];
#pragma unroll
      for (int k = 0; k < kSsimWin; ++k) v4[k] = s_h[4][vrow + k][vcol];
      ssim_tap4(m[4], v4, w);
#pragma unroll
      for (int j = 0; j < kSsimGroup; ++j) {
        m[0][j] = m01[j].x;
        m[1][j] = m01[j].y;
        m[2][j] = m23[j].x;
        m[3][j] = m23[j].y;
      }
    }
#pragma unroll
    for (int j = 0; j < kSsimGroup; ++j) {
      const int px = ox + vcol, py = oy + vrow + j;
      if (px >= W || py >= H) continue;
      const float mx = shift[0] + m[0][j], my = shift[1] + m[1][j];
      const float sxx = m[2][j] - m[0][j] * m[0][j], syy = m[3][j] - m[1][j] * m[1][j];
      const float sxy = m[4][j] - m[0][j] * m[1][j];
      const float n1 = 2.f * mx * my + kC1, n2 = 2.f * sxy + kC2;
      const float d1 = mx * mx + my * my + kC1, d2 = sxx + syy + kC2;
      const float id = 1.0f / (d1 * d2);
      const float S = n1 * n2 * id;
      const float dS_dmx = 2.f * my * n2 * id - S * 2.f * mx / d1;
      const float dS_dsxx = -S / d2;
      const float dS_dsxy = 2.f * n1 * id;
      const int64_t e = int64_t(py) * W + px;
      maps[(0 + c) * P + e] = dLdS * dS_dmx;
      maps[(3 + c) * P + e] = dLdS * dS_dsxx;
      maps[(6 + c) * P + e] = dLdS * dS_dsxy;
      maps[(9 + c) * P + e] = mx;
      maps[(12 + c) * P + e] = my;
      ssum += S;
    }
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) ssum += __shfl_xor_sync(0xffffffffu, ssum, o);
  if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = ssum;
  __syncthreads();  // (s_red is not s_h: no conflict with the last vertical pass)
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int k = 0; k < kSsimThreads / 32; ++k) t += s_red[k];
    atomicAdd(ssim_out, t * inv3P);
  }
}

__global__ void __launch_bounds__(kSsimThreads)
    k_ssim_bwd(const float* __restrict__ x, const float* __restrict__ y, int W, int H, SsimWindow w,
               const float* __restrict__ maps, float* __restrict__ dLdx) {
  // the five maps of a channel (a, b, c, mu_x, mu_y) staged raw (36 KB, dynamic shared
  // memory); A is formed as the horizontal pass reads them (zero outside the image,
  // where every map is 0)
  extern __shared__ __align__(16) float ssim_dyn[];
  float(*s_in)[kSsimIn][kSsimInStride] = reinterpret_cast<float(*)[kSsimIn][kSsimInStride]>(ssim_dyn);
  __shared__ float s_h[3][kSsimIn][kSsimHStride];
  const int ox = blockIdx.x * kSsimTile, oy = blockIdx.y * kSsimTile;
  const int64_t P = int64_t(W) * H;
  const int vcol = threadIdx.x % kSsimTile, vrow = (threadIdx.x / kSsimTile) * kSsimGroup;
  const int64_t centre = int64_t(min(oy + kSsimTile / 2, H - 1)) * W + min(ox + kSsimTile / 2, W - 1);
  const float* const planes[5] = {maps, maps + 3 * P, maps + 6 * P, maps + 9 * P, maps + 12 * P};
  ssim_stage<5>(s_in, planes, W, H, P, 0, ox, oy);
  for (int c = 0; c < 3; ++c) {
    const float sx = x[c * P + centre], sy = y[c * P + centre];
    ssim_cp_wait_all();
    __syncthreads();  // channel c staged for every thread; the previous vertical pass done with s_h
    for (int i = threadIdx.x; i < kSsimHItems; i += kSsimThreads) {
      const int r = i % kSsimIn, c0 = (i / kSsimIn) * kSsimGroup;
      float2 vab[kSsimWin];
      float vc[kSsimWin];
#pragma unroll
      for (int k = 0; k < kSsimWin; ++k) {
        const float vb = s_in[1][r][c0 + k];
        vc[k] = s_in[2][r][c0 + k];
        // A about the shift, paired with b for the two-wide taps
        vab[k] = make_float2(s_in[0][r][c0 + k] - 2.f * (s_in[3][r][c0 + k] - sx) * vb - (s_in[4][r][c0 + k] - sy) * vc[k],
                             vb);
      }
      float2 o01[kSsimGroup];
      float o2[kSsimGroup] = {};
#pragma unroll
      for (int j = 0; j < kSsimGroup; ++j) o01[j] = make_float2(0.0f, 0.0f);
      ssim_tap4x2(o01, vab, w);
      ssim_tap4(o2, vc, w);
#pragma unroll
      for (int j = 0; j < kSsimGroup; ++j) {
        s_h[0][r][c0 + j] = o01[j].x;
        s_h[1][r][c0 + j] = o01[j].y;
        s_h[2][r][c0 + j] = o2[j];
      }
    }
    __syncthreads();  // s_in read by every thread: the next channel may land there
    if (c + 1 < 3) ssim_stage<5>(s_in, planes, W, H, P, c + 1, ox, oy);
    float g[3][kSsimGroup] = {};
    {
      float2 g01[kSsimGroup];
#pragma unroll
      for (int j = 0; j < kSsimGroup; ++j) g01[j] = make_float2(0.0f, 0.0f);
      float2 v[kSsimWin];
      float v2[kSsimWin];
#pragma unroll
      for (int k = 0; k < kSsimWin; ++k) {
        v[k] = make_float2(s_h[0][vrow + k][vcol], s_h[1][vrow + k][vcol]);
        v2[k] = s_h[2][vrow + k][vcol];
      }
      ssim_tap4x2(g01, v, w);
      ssim_tap4(g[2], v2, w);
#pragma unroll
      for (int j = 0; j < kSsimGroup; ++j) {
        g[0][j] = g01[j].x;
        g[1][j] = g01[j].y;
      }
    }
#pragma unroll
    for (int j = 0; j < kSsimGroup; ++j) {
      const int px = ox + vcol, py = oy + vrow + j;
      if (px >= W || py >= H) continue;
      const int64_t e = int64_t(c) * P + int64_t(py) * W + px;
      dLdx[e] = g[0][j] + 2.f * (x[e] - sx) * g[1][j] + (y[e] - sy) * g[2][j];
    }
  }
}

__global__ void k_zero1(float* p) { *p = 0.0f; }

constexpr size_t kSsimBwdDyn = size_t(5) * kSsimIn * kSsimInStride * sizeof(float);  // 36120 bytes

// The backward's dynamic shared-memory opt-in (its 52 KB in all exceed the 48 KB
// default), set on the first call (an eager step before a CUDA graph capture sets it).
bool ssim_bwd_attr_ready() {
  static bool ok = false;
  if (!ok)
    ok = cudaFuncSetAttribute(k_ssim_bwd, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSsimBwdDyn)) ==
         cudaSuccess;
  return ok;
}

}  // namespace gs

extern "C" gs_status gs_ssim_fwd(int32_t width, int32_t height, const float* image, const float* target,
                                 float lambda, float* maps, float* ssim_out, cudaStream_t stream) {
  using namespace gs;
  if (width <= 0 || height <= 0 || !image || !target || !maps || !ssim_out || !(lambda >= 0.0f) ||
      !std::isfinite(lambda))
    return GS_ERR_INVALID_ARG;
  const double P = double(width) * double(height);
  k_zero1<<<1, 1, 0, stream>>>(ssim_out);
  const dim3 grid((width + kSsimTile - 1) / kSsimTile, (height + kSsimTile - 1) / kSsimTile);
  k_ssim_fwd<<<grid, kSsimThreads, 0, stream>>>(image, target, width, height, ssim_window(), float(-double(lambda) / (3.0 * P)),
                                       float(1.0 / (3.0 * P)), maps, ssim_out);
  return launch_status();
}

extern "C" gs_status gs_ssim_bwd(int32_t width, int32_t height, const float* image, const float* target,
                                 const float* maps, float* dLdC, cudaStream_t stream) {
  using namespace gs;
  if (width <= 0 || height <= 0 || !image || !target || !maps || !dLdC) return GS_ERR_INVALID_ARG;
  if (!ssim_bwd_attr_ready()) return GS_ERR_CUDA;
  const dim3 grid((width + kSsimTile - 1) / kSsimTile, (height + kSsimTile - 1) / kSsimTile);
  k_ssim_bwd<<<grid, kSsimThreads, kSsimBwdDyn, stream>>>(image, target, width, height, ssim_window(), maps, dLdC);
  return launch_status();
}
