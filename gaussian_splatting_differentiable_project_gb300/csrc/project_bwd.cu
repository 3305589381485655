// gs_project_bwd: chain rule of the projection, one thread per Gaussian.
//
// The forward quantities (and the decisions: culling, clamped Jacobian abscissae,
// clamped colour channels) are recomputed with the frozen projection, so they
// are exactly those of gs_project; the gradient arithmetic itself is plain fp32.
// Reads the 59 parameter planes and 9 gradient planes, writes 59 gradient
// planes; every access is coalesced across the warp.
#include "api_util.h"
#include "adam_common.cuh"
#include "project_frozen.cuh"

namespace gs {

// d Y_k / d(x, y, z) of the basis polynomials of sh_basis, x, y, z independent.
__device__ __forceinline__ void sh_basis_grad(float x, float y, float z, int k, float g[3]) {
  const float xx = x * x, yy = y * y, zz = z * z;
  switch (k) {
    case 0: g[0] = 0.f; g[1] = 0.f; g[2] = 0.f; break;
    case 1: g[0] = 0.f; g[1] = -kSh1; g[2] = 0.f; break;
    case 2: g[0] = 0.f; g[1] = 0.f; g[2] = kSh1; break;
    case 3: g[0] = -kSh1; g[1] = 0.f; g[2] = 0.f; break;
    case 4: g[0] = kSh2a * y; g[1] = kSh2a * x; g[2] = 0.f; break;
    case 5: g[0] = 0.f; g[1] = -kSh2a * z; g[2] = -kSh2a * y; break;
    case 6: g[0] = -2.f * kSh2b * x; g[1] = -2.f * kSh2b * y; g[2] = 4.f * kSh2b * z; break;
    case 7: g[0] = -kSh2a * z; g[1] = 0.f; g[2] = -kSh2a * x; break;
    case 8: g[0] = 2.f * kSh2c * x; g[1] = -2.f * kSh2c * y; g[2] = 0.f; break;
    case 9: g[0] = -kSh3a * 6.f * x * y; g[1] = -kSh3a * (3.f * xx - 3.f * yy); g[2] = 0.f; break;
    case 10: g[0] = kSh3b * y * z; g[1] = kSh3b * x * z; g[2] = kSh3b * x * y; break;
    case 11: g[0] = kSh3c * 2.f * x * y; g[1] = -kSh3c * (4.f * zz - xx - 3.f * yy); g[2] = -kSh3c * 8.f * y * z; break;
    case 12: g[0] = -kSh3d * 6.f * x * z; g[1] = -kSh3d * 6.f * y * z; g[2] = kSh3d * (6.f * zz - 3.f * xx - 3.f * yy); break;
    case 13: g[0] = -kSh3c * (4.f * zz - 3.f * xx - yy); g[1] = kSh3c * 2.f * x * y; g[2] = -kSh3c * 8.f * x * z; break;
    case 14: g[0] = kSh3e * 2.f * x * z; g[1] = -kSh3e * 2.f * y * z; g[2] = kSh3e * (xx - yy); break;
    default: g[0] = -kSh3a * (3.f * xx - 3.f * yy); g[1] = kSh3a * 6.f * x * y; g[2] = 0.f; break;
  }
}

// Gradients of one Gaussian from its nine 2D gradients: the 11 geometric ones
// (mean, log-scale, quaternion, opacity logit) and the factors of the 48 SH ones
// (d L / d sh[k][ch] = Y[k] gcol[ch]).  Returns false for culled Gaussians and
// padding (all gradients zero).
struct ChainOut {
  float geo[11];
  float Y[16];
  float gcol[3];
};

template <bool kReadOnly = true>
__device__ __forceinline__ bool chain_rule(const float* P, int64_t n, int64_t n_pad, int64_t i, const CamDev& cam,
                                           const uint32_t* __restrict__ count, const float* __restrict__ g2,
                                           ChainOut& o) {
  Geo g;
  g.visible = false;
  if (i < n && count[i] > 0u) project_geo<kReadOnly>(P, n_pad, i, cam, g);
  if (!g.visible) return false;
  float gq2[9];
  {
    // interleaved: the nine partials of Gaussian i at 12 i + 0..8 (three float4)
    const float4* g4 = reinterpret_cast<const float4*>(g2) + 3 * i;
    const float4 x = __ldg(g4), y = __ldg(g4 + 1), z = __ldg(g4 + 2);
    gq2[0] = x.x, gq2[1] = x.y, gq2[2] = x.z, gq2[3] = x.w;
    gq2[4] = y.x, gq2[5] = y.y, gq2[6] = y.z, gq2[7] = y.w;
    gq2[8] = z.x;
  }
  // slots 0..4 hold the moments S1..S5 of q = dL/dpower over the pixel offsets;
  // with the conic: dL/dmx = A S1 + B S2, dL/dmy = B S1 + C S2, dL/dA = -S3/2,
  // dL/dB = -S4, dL/dC = -S5/2
  const float gmx = g.A * gq2[0] + g.B * gq2[1], gmy = g.B * gq2[0] + g.C * gq2[1];
  const float gA = -0.5f * gq2[2], gB = -gq2[3], gC = -0.5f * gq2[4], go = gq2[5];

  // ---- colour: SH coefficients and the view direction
  float d[3], len;
  view_dir(g.mux, g.muy, g.muz, cam, d, &len);
  float Y[16];
  sh_basis(d[0], d[1], d[2], Y);
  float acc[3] = {0.f, 0.f, 0.f};
  float h[3][3] = {{0.f, 0.f, 0.f}, {0.f, 0.f, 0.f}, {0.f, 0.f, 0.f}};
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    float dY[3];
    sh_basis_grad(d[0], d[1], d[2], k, dY);
#pragma unroll
    for (int ch = 0; ch < 3; ++ch) {
      const float sh = ldp<kReadOnly>(P, n_pad, 11 + 3 * k + ch, i);
      acc[ch] = (k == 0) ? __fmul_rn(Y[0], sh) : __fmaf_rn(Y[k], sh, acc[ch]);
      h[ch][0] += sh * dY[0];
      h[ch][1] += sh * dY[1];
      h[ch][2] += sh * dY[2];
    }
  }
  float gcol[3];
#pragma unroll
  for (int ch = 0; ch < 3; ++ch) gcol[ch] = (__fadd_rn(acc[ch], 0.5f) < 0.0f) ? 0.0f : gq2[6 + ch];
#pragma unroll
  for (int k = 0; k < 16; ++k) o.Y[k] = Y[k];
#pragma unroll
  for (int ch = 0; ch < 3; ++ch) o.gcol[ch] = gcol[ch];
  float gd[3];
#pragma unroll
  for (int e = 0; e < 3; ++e) gd[e] = gcol[0] * h[0][e] + gcol[1] * h[1][e] + gcol[2] * h[2][e];
  const float dotd = gd[0] * d[0] + gd[1] * d[1] + gd[2] * d[2];
  const float inv_len = 1.0f / len;
  float gmu[3];
#pragma unroll
  for (int e = 0; e < 3; ++e) gmu[e] = (gd[e] - d[e] * dotd) * inv_len;

  // ---- opacity
  const float op = opacity_of(ldp<kReadOnly>(P, n_pad, 10, i));
  o.geo[10] = go * op * (1.0f - op);

  // ---- conic (A, B, C) -> 2D covariance (a, b, c)
  const float a = g.a, b = g.b, c = g.c;
  const float id2 = 1.0f / (g.det * g.det);
  const float ga = (-gA * c * c + gB * b * c - gC * b * b) * id2;
  const float gb = (2.0f * gA * b * c - gB * (a * c + b * b) + 2.0f * gC * a * b) * id2;
  const float gc = (-gA * b * b + gB * a * b - gC * a * a) * id2;

  // ---- (a, b, c) -> rows of T = J W and Sigma
  const float Sg[3][3] = {{g.S00, g.S01, g.S02}, {g.S01, g.S11, g.S12}, {g.S02, g.S12, g.S22}};
  float ST0[3], ST1[3];
#pragma unroll
  for (int r = 0; r < 3; ++r) {
    ST0[r] = Sg[r][0] * g.T0[0] + Sg[r][1] * g.T0[1] + Sg[r][2] * g.T0[2];
    ST1[r] = Sg[r][0] * g.T1[0] + Sg[r][1] * g.T1[1] + Sg[r][2] * g.T1[2];
  }
  float gT0[3], gT1[3];
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    gT0[j] = 2.0f * ga * ST0[j] + gb * ST1[j];
    gT1[j] = gb * ST0[j] + 2.0f * gc * ST1[j];
  }
  // symmetrised dL/dSigma (gS + gS^T)
  float gSs[3][3];
#pragma unroll
  for (int r = 0; r < 3; ++r)
#pragma unroll
    for (int q = 0; q < 3; ++q)
      gSs[r][q] = 2.0f * ga * g.T0[r] * g.T0[q] + gb * (g.T0[r] * g.T1[q] + g.T1[r] * g.T0[q]) +
                  2.0f * gc * g.T1[r] * g.T1[q];

  // ---- T = J W -> Jacobian entries -> camera-space mean
  const float* W = cam.R;
  float gJ00 = 0.f, gJ02 = 0.f, gJ11 = 0.f, gJ12 = 0.f;
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    gJ00 += gT0[j] * W[j];
    gJ02 += gT0[j] * W[6 + j];
    gJ11 += gT1[j] * W[3 + j];
    gJ12 += gT1[j] * W[6 + j];
  }
  const float fx = cam.fx, fy = cam.fy, tz = g.tz;
  const float itz = 1.0f / tz, itz2 = itz * itz;
  float gtx = 0.f, gty = 0.f, gtz = -(fx * gJ00 + fy * gJ11) * itz2;
  if (!g.clamp_x) {
    gtx -= fx * gJ02 * itz2;
    gtz += 2.0f * fx * g.uc * gJ02 * itz2;
  } else {
    gtz += fx * g.uc * gJ02 * itz2;
  }
  if (!g.clamp_y) {
    gty -= fy * gJ12 * itz2;
    gtz += 2.0f * fy * g.vc * gJ12 * itz2;
  } else {
    gtz += fy * g.vc * gJ12 * itz2;
  }
  gtx += gmx * fx * itz;
  gty += gmy * fy * itz;
  gtz -= (gmx * fx * g.tx + gmy * fy * g.ty) * itz2;
#pragma unroll
  for (int e = 0; e < 3; ++e) gmu[e] += W[e] * gtx + W[3 + e] * gty + W[6 + e] * gtz;
#pragma unroll
  for (int e = 0; e < 3; ++e) o.geo[e] = gmu[e];

  // ---- Sigma = M M^T -> M -> scale and rotation
  float gM[9];
#pragma unroll
  for (int r = 0; r < 3; ++r)
#pragma unroll
    for (int k = 0; k < 3; ++k)
      gM[3 * r + k] = gSs[r][0] * g.M[k] + gSs[r][1] * g.M[3 + k] + gSs[r][2] * g.M[6 + k];
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    const float gs = gM[k] * g.Rq[k] + gM[3 + k] * g.Rq[3 + k] + gM[6 + k] * g.Rq[6 + k];
    o.geo[3 + k] = gs * g.s[k];
  }
  float gR[9];
#pragma unroll
  for (int r = 0; r < 3; ++r)
#pragma unroll
    for (int k = 0; k < 3; ++k) gR[3 * r + k] = gM[3 * r + k] * g.s[k];
  const float w = g.qw, x = g.qx, y = g.qy, z = g.qz;
  float gq[4];
  gq[0] = 2.f * (-z * gR[1] + y * gR[2] + z * gR[3] - x * gR[5] - y * gR[6] + x * gR[7]);
  gq[1] = 2.f * (y * gR[1] + z * gR[2] + y * gR[3] - 2.f * x * gR[4] - w * gR[5] + z * gR[6] + w * gR[7] -
                 2.f * x * gR[8]);
  gq[2] = 2.f * (-2.f * y * gR[0] + x * gR[1] + w * gR[2] + x * gR[3] + z * gR[5] - w * gR[6] + z * gR[7] -
                 2.f * y * gR[8]);
  gq[3] = 2.f * (-2.f * z * gR[0] - w * gR[1] + x * gR[2] + w * gR[3] - 2.f * z * gR[4] + y * gR[5] + x * gR[6] +
                 y * gR[7]);
  const float dq = gq[0] * w + gq[1] * x + gq[2] * y + gq[3] * z;
  const float iqn = 1.0f / g.qn;
  o.geo[6] = (gq[0] - w * dq) * iqn;
  o.geo[7] = (gq[1] - x * dq) * iqn;
  o.geo[8] = (gq[2] - y * dq) * iqn;
  o.geo[9] = (gq[3] - z * dq) * iqn;
  return true;
}

// kAcc: add to G instead of overwriting it (culled Gaussians and padding untouched).
template <bool kAcc>
__global__ void __launch_bounds__(256, 2)
    k_project_bwd(const float* __restrict__ P, int64_t n, int64_t n_pad, CamDev cam, const uint32_t* __restrict__ count,
                  const float* __restrict__ g2, float* __restrict__ G) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n_pad; i += stride) {
    ChainOut o;
    if (!chain_rule(P, n, n_pad, i, cam, count, g2, o)) {
      if (!kAcc) {
#pragma unroll 4
        for (int pl = 0; pl < kPlanes; ++pl) G[int64_t(pl) * n_pad + i] = 0.0f;
      }
      continue;
    }
    if constexpr (!kAcc) {
#pragma unroll
      for (int pl = 0; pl < 11; ++pl) G[int64_t(pl) * n_pad + i] = o.geo[pl];
#pragma unroll
      for (int k = 0; k < 16; ++k)
#pragma unroll
        for (int ch = 0; ch < 3; ++ch) G[int64_t(11 + 3 * k + ch) * n_pad + i] = o.Y[k] * o.gcol[ch];
    } else {
      // accumulate: each group's old values are loaded before any of its stores (the
      // compiler cannot reorder a later plane's load above an earlier plane's store,
      // so one plane at a time would serialise 59 memory round trips)
      {
        float cur[11];
#pragma unroll
        for (int pl = 0; pl < 11; ++pl) cur[pl] = G[int64_t(pl) * n_pad + i];
#pragma unroll
        for (int pl = 0; pl < 11; ++pl) G[int64_t(pl) * n_pad + i] = cur[pl] + o.geo[pl];
      }
#pragma unroll
      for (int k0 = 0; k0 < 16; k0 += 4) {
        float cur[12];
#pragma unroll
        for (int q = 0; q < 12; ++q) cur[q] = G[int64_t(11 + 3 * k0 + q) * n_pad + i];
#pragma unroll
        for (int q = 0; q < 12; ++q)
          G[int64_t(11 + 3 * k0 + q) * n_pad + i] = cur[q] + o.Y[k0 + q / 3] * o.gcol[q % 3];
      }
    }
  }
}

// Fused projection backward + Adam: a CTA takes 256 consecutive Gaussians.  Phase 1:
// each thread derives its Gaussian's gradient factors (11 geometric gradients, the
// 16 SH basis values and 3 colour factors; zeros for culled Gaussians and padding)
// into shared memory.  Phase 2: the CTA streams the 59 planes x 256 parameters as
// float4 (p, m, v read and written once) and applies the Adam element update with
// gradients rebuilt from shared memory, so the gradient planes are never written or
// read.  A CTA's Gaussians occupy whole 1 KB lines of every plane (n_pad and the
// block start are multiples of 256) that no other CTA touches, and phase 1 reads
// them before phase 2 writes them.
constexpr int kFusedBlock = 256;
constexpr int kChunkPlanes = 8;                                       // planes per streamed chunk
constexpr int kChunks = (kPlanes + kChunkPlanes - 1) / kChunkPlanes;  // 8
constexpr int kRow4 = kFusedBlock / 4;                                // float4 per plane row of a group
constexpr size_t kChunkBytes = size_t(kChunkPlanes) * kRow4 * 16;     // one array's share of a chunk
// p, m, v (and the accumulated gradient when there is one), double-buffered: 48 / 64 KB
constexpr size_t fused_dyn_smem(bool acc_in) { return 2 * (acc_in ? 4 : 3) * kChunkBytes; }

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Streams the parameters and moments of one group (and the gradient accumulated by
// earlier views when kAccIn) through shared memory in chunks of kChunkPlanes planes:
// the arrays of chunk c land in buffer c & 1.
template <bool kAccIn>
struct ChunkStream {
  static constexpr int kArrays = kAccIn ? 4 : 3;
  float4* buf;  // [2][kArrays][kChunkPlanes][kRow4]
  __device__ __forceinline__ float4* at(int b, int arr) const {
    return buf + (size_t(b) * kArrays + arr) * (kChunkPlanes * kRow4);
  }
  // every thread: issue its share of chunk c of group b0 into buffer b, one commit group
  __device__ __forceinline__ void issue(int c, int b, const float* P, const float* M, const float* V,
                                        const float* Gin, int64_t n_pad, int64_t b0) const {
    const int pl0 = c * kChunkPlanes;
    const int np = min(kChunkPlanes, kPlanes - pl0);
    for (int e = threadIdx.x; e < np * kRow4; e += kFusedBlock) {
      const int64_t g = int64_t(pl0 + e / kRow4) * n_pad + b0 + int64_t(e % kRow4) * 4;
      cp_async16(at(b, 0) + e, P + g);
      cp_async16(at(b, 1) + e, M + g);
      cp_async16(at(b, 2) + e, V + g);
      if (kAccIn) cp_async16(at(b, 3) + e, Gin + g);
    }
    cp_async_commit();
  }
};

// Fused projection backward + Adam over groups of 256 Gaussians.  Phase 1: one thread
// per Gaussian runs the chain rule and leaves 30 factors in shared memory (11
// geometric gradients, 16 SH basis values, 3 colour factors; an SH coefficient's
// gradient is basis value x colour factor).  Phase 2: the 59 planes of the group
// stream through shared memory in chunks of 8 planes (cp.async, double-buffered,
// the first two chunks issued before phase 1 so that the chain rule overlaps the
// loads); each element gets its gradient from the factors (plus, with kAccIn, the
// gradient that earlier views of a batch accumulated in Gin) and the Adam update, and
// p, m, v are written back.  The gradient planes are never written.
// kDevT: the step count is read from t_dev and the Adam parameters are formed from
// h in fp64 by one thread per CTA (for steps replayed from a CUDA graph, whose
// kernel arguments are fixed); otherwise they arrive ready in a.
template <bool kAccIn, bool kDevT>
__global__ void __launch_bounds__(kFusedBlock, 2)
    k_project_bwd_adam(float* P, int64_t n, int64_t n_pad, CamDev cam, const uint32_t* __restrict__ count,
                       const float* __restrict__ g2, const float* __restrict__ Gin, float* M, float* V,
                       AdamParams a_in, AdamHyper h, const int64_t* __restrict__ t_dev) {
  __shared__ AdamParams s_adam;
  if (kDevT) {
    // the same fp64 expressions as form_adam_params, one plane per thread (fp64
    // division is slow; a single thread forming all 59 would delay every CTA)
    if (threadIdx.x < kPlanes) {
      const double bc1 = 1.0 - ::pow(h.beta1, double(*t_dev));
      s_adam.step[threadIdx.x] = float(double(h.lr[threadIdx.x]) / bc1);
    } else if (threadIdx.x == kPlanes) {
      const double bc2 = 1.0 - ::pow(h.beta2, double(*t_dev));
      s_adam.b1 = float(h.beta1);
      s_adam.c1 = float(1.0 - h.beta1);
      s_adam.b2 = float(h.beta2);
      s_adam.c2 = float(1.0 - h.beta2);
      s_adam.eps = float(h.eps);
      s_adam.inv_sqrt_bc2 = float(1.0 / ::sqrt(bc2));
    }
    __syncthreads();
  }
  const AdamParams& a = kDevT ? s_adam : a_in;
  __shared__ float s_geo[11][kFusedBlock];
  __shared__ float s_Y[16][kFusedBlock];
  __shared__ float s_gc[3][kFusedBlock];
  extern __shared__ __align__(16) unsigned char fused_smem[];
  const ChunkStream<kAccIn> cs{reinterpret_cast<float4*>(fused_smem)};
  const int tid = threadIdx.x;
  const int64_t gstride = int64_t(gridDim.x) * kFusedBlock;
  int64_t b0 = int64_t(blockIdx.x) * kFusedBlock;
  if (b0 < n_pad) {
    cs.issue(0, 0, P, M, V, Gin, n_pad, b0);
    cs.issue(1, 1, P, M, V, Gin, n_pad, b0);
  }
  for (; b0 < n_pad; b0 += gstride) {
    // the next group's first two chunks are issued into the buffers that this
    // group's last two chunks free, so its loads overlap this group's tail and the
    // next chain rule
    const bool has_next = b0 + gstride < n_pad;
    {
      ChainOut o;
      const bool vis = chain_rule<false>(P, n, n_pad, b0 + tid, cam, count, g2, o);
#pragma unroll
      for (int k = 0; k < 11; ++k) s_geo[k][tid] = vis ? o.geo[k] : 0.0f;
#pragma unroll
      for (int k = 0; k < 16; ++k) s_Y[k][tid] = vis ? o.Y[k] : 0.0f;
#pragma unroll
      for (int k = 0; k < 3; ++k) s_gc[k][tid] = vis ? o.gcol[k] : 0.0f;
    }
#pragma unroll 1
    for (int c = 0; c < kChunks; ++c) {
      if (c + 1 < kChunks || has_next)
        cp_async_wait<1>();
      else
        cp_async_wait<0>();
      __syncthreads();  // chunk c landed for every thread; phase 1 factors visible
      const int b = c & 1;
      const int pl0 = c * kChunkPlanes;
      const int np = min(kChunkPlanes, kPlanes - pl0);
      const float4* sp = cs.at(b, 0);
      const float4* sm = cs.at(b, 1);
      const float4* sv = cs.at(b, 2);
      const float4* sg = cs.at(b, kAccIn ? 3 : 2);
      for (int e = tid; e < np * kRow4; e += kFusedBlock) {
        const int pl = pl0 + e / kRow4, q = (e % kRow4) * 4;
        float4 pp = sp[e], mm = sm[e], vv = sv[e];
        float g[4];
        if (pl < 11) {
#pragma unroll
          for (int k = 0; k < 4; ++k) g[k] = s_geo[pl][q + k];
        } else {
          const int kk = (pl - 11) / 3, ch = (pl - 11) % 3;
#pragma unroll
          for (int k = 0; k < 4; ++k) g[k] = s_Y[kk][q + k] * s_gc[ch][q + k];
        }
        if (kAccIn) {
          const float4 gi = sg[e];
          g[0] += gi.x;
          g[1] += gi.y;
          g[2] += gi.z;
          g[3] += gi.w;
        }
        const float step = a.step[pl];
        adam_elem(pp.x, mm.x, vv.x, g[0], step, a);
        adam_elem(pp.y, mm.y, vv.y, g[1], step, a);
        adam_elem(pp.z, mm.z, vv.z, g[2], step, a);
        adam_elem(pp.w, mm.w, vv.w, g[3], step, a);
        const int64_t base = int64_t(pl) * n_pad + b0 + q;
        *reinterpret_cast<float4*>(P + base) = pp;
        *reinterpret_cast<float4*>(M + base) = mm;
        *reinterpret_cast<float4*>(V + base) = vv;
      }
      __syncthreads();  // buffer b free
      if (c + 2 < kChunks)
        cs.issue(c + 2, b, P, M, V, Gin, n_pad, b0);
      else if (has_next)
        cs.issue(c + 2 - kChunks, b, P, M, V, Gin, n_pad, b0 + gstride);
    }
  }
}

}  // namespace gs

namespace {

gs_status project_bwd_launch(gs_dims dims, const float* params, const gs_camera* cam, const gs_proj* proj,
                             const float* grad2d, float* grads, uint32_t* dev_status, cudaStream_t stream, bool acc) {
  using namespace gs;
  if (!dims_ok(dims) || !camera_ok(cam) || !params || !proj || !proj->count || !grad2d || !grads || !dev_status)
    return GS_ERR_INVALID_ARG;
  if (!aligned(params, 16) || !aligned(grads, 16) || !aligned(grad2d, 16)) return GS_ERR_INVALID_ARG;
  const int blocks = grid_for(dims.n_pad, 256, sm_count() * 64);
  if (acc)
    k_project_bwd<true><<<blocks, 256, 0, stream>>>(params, dims.n, dims.n_pad, cam_dev(*cam), proj->count, grad2d,
                                                    grads);
  else
    k_project_bwd<false><<<blocks, 256, 0, stream>>>(params, dims.n, dims.n_pad, cam_dev(*cam), proj->count, grad2d,
                                                     grads);
  return launch_status();
}

// The dynamic shared-memory opt-in of all four fused variants, set together on the
// first call of any of them (an eager step before a CUDA graph capture has then set
// it for the variants the graph uses).
bool fused_attrs_ready() {
  using namespace gs;
  static bool ok = false;
  if (ok) return true;
  ok = cudaFuncSetAttribute(k_project_bwd_adam<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                            int(fused_dyn_smem(false))) == cudaSuccess &&
       cudaFuncSetAttribute(k_project_bwd_adam<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                            int(fused_dyn_smem(true))) == cudaSuccess &&
       cudaFuncSetAttribute(k_project_bwd_adam<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                            int(fused_dyn_smem(false))) == cudaSuccess &&
       cudaFuncSetAttribute(k_project_bwd_adam<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                            int(fused_dyn_smem(true))) == cudaSuccess;
  return ok;
}

template <bool kAccIn, bool kDevT>
gs_status fused_launch(gs_dims dims, float* params, const gs_camera* cam, const gs_proj* proj, const float* grad2d,
                       const float* grads_in, float* m, float* v, const gs::AdamParams& a, const gs::AdamHyper& h,
                       const int64_t* t_dev, cudaStream_t stream) {
  using namespace gs;
  const size_t smem = fused_dyn_smem(kAccIn);
  if (!fused_attrs_ready()) return GS_ERR_CUDA;
  const int blocks = grid_for(dims.n_pad / kFusedBlock, 1, sm_count() * 2);
  k_project_bwd_adam<kAccIn, kDevT><<<blocks, kFusedBlock, smem, stream>>>(
      params, dims.n, dims.n_pad, cam_dev(*cam), proj->count, grad2d, grads_in, m, v, a, h, t_dev);
  return launch_status();
}

__global__ void k_counter_add(int64_t* c, int64_t d) { *c += d; }

}  // namespace

extern "C" gs_status gs_project_bwd(gs_dims dims, const float* params, const gs_camera* cam, const gs_proj* proj,
                                    const float* grad2d, float* grads, uint32_t* dev_status, cudaStream_t stream) {
  return project_bwd_launch(dims, params, cam, proj, grad2d, grads, dev_status, stream, false);
}

extern "C" gs_status gs_project_bwd_accumulate(gs_dims dims, const float* params, const gs_camera* cam,
                                               const gs_proj* proj, const float* grad2d, float* grads,
                                               uint32_t* dev_status, cudaStream_t stream) {
  return project_bwd_launch(dims, params, cam, proj, grad2d, grads, dev_status, stream, true);
}

extern "C" gs_status gs_project_bwd_adam(gs_dims dims, float* params, const gs_camera* cam, const gs_proj* proj,
                                         const float* grad2d, const float* grads_in, float* m, float* v,
                                         const float lr_plane[GS_N_PLANES], double beta1, double beta2, double eps,
                                         int64_t t, uint32_t* dev_status, cudaStream_t stream) {
  using namespace gs;
  if (!dims_ok(dims) || !camera_ok(cam) || !params || !proj || !proj->count || !grad2d || !m || !v || !lr_plane ||
      !dev_status)
    return GS_ERR_INVALID_ARG;
  if (!aligned(params, 16) || !aligned(grad2d, 16) || !aligned(m, 16) || !aligned(v, 16) ||
      (grads_in && !aligned(grads_in, 16)))
    return GS_ERR_INVALID_ARG;
  AdamParams a;
  if (!make_adam_params(lr_plane, beta1, beta2, eps, t, a)) return GS_ERR_INVALID_ARG;
  const AdamHyper h{};
  return grads_in ? fused_launch<true, false>(dims, params, cam, proj, grad2d, grads_in, m, v, a, h, nullptr, stream)
                  : fused_launch<false, false>(dims, params, cam, proj, grad2d, nullptr, m, v, a, h, nullptr, stream);
}

extern "C" gs_status gs_project_bwd_adam_tdev(gs_dims dims, float* params, const gs_camera* cam, const gs_proj* proj,
                                              const float* grad2d, const float* grads_in, float* m, float* v,
                                              const float lr_plane[GS_N_PLANES], double beta1, double beta2,
                                              double eps, const int64_t* t_dev, uint32_t* dev_status,
                                              cudaStream_t stream) {
  using namespace gs;
  if (!dims_ok(dims) || !camera_ok(cam) || !params || !proj || !proj->count || !grad2d || !m || !v || !lr_plane ||
      !t_dev || !dev_status)
    return GS_ERR_INVALID_ARG;
  if (!aligned(params, 16) || !aligned(grad2d, 16) || !aligned(m, 16) || !aligned(v, 16) || !aligned(t_dev, 8) ||
      (grads_in && !aligned(grads_in, 16)))
    return GS_ERR_INVALID_ARG;
  if (!adam_hyper_ok(beta1, beta2, eps)) return GS_ERR_INVALID_ARG;
  AdamHyper h;
  for (int k = 0; k < kPlanes; ++k) h.lr[k] = lr_plane[k];
  h.beta1 = beta1;
  h.beta2 = beta2;
  h.eps = eps;
  const AdamParams a{};
  return grads_in ? fused_launch<true, true>(dims, params, cam, proj, grad2d, grads_in, m, v, a, h, t_dev, stream)
                  : fused_launch<false, true>(dims, params, cam, proj, grad2d, nullptr, m, v, a, h, t_dev, stream);
}

extern "C" gs_status gs_step_counter_add(int64_t* counter, int64_t delta, cudaStream_t stream) {
  using namespace gs;
  if (!counter || !aligned(counter, 8)) return GS_ERR_INVALID_ARG;
  k_counter_add<<<1, 1, 0, stream>>>(counter, delta);
  return launch_status();
}
