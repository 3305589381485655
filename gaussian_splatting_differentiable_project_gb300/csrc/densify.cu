// Adaptive density control.  "Scaling 3D Gaussian Splatting with Distributed
// Compute": adaptive density control clones, splits and prunes Gaussians every
// hundred steps (memory-wall section), from 2D position gradients accumulated over
// the steps (step walkthrough), starting at step 500 (trace section); thresholds and
// the split rule of the cited 3DGS method.
//
//   gs_densify_accumulate  per visible Gaussian: acc += |(g_mx W/2, g_my H/2)|, cnt += 1,
//                          the mean gradient formed from grad2d's moments and the
//                          conic of the Gaussian's record
//   gs_densify_plan        per Gaussian an action (prune / keep / clone / split) and the
//                          offset of its outputs (block scan + one-block scan of the
//                          block sums); the new count
//   gs_densify_apply       the new parameter and moment planes: kept Gaussians and a
//                          clone's original with their moments, a clone's copy and a
//                          split's two children (mu + R S xi, log-scale - ln 1.6) with
//                          zero moments; padding columns cleared
//   gs_opacity_reset       opacity logit clamped, its moments zeroed
// Every decision is an fp32 comparison against a threshold the caller formed in
// fp64 (the sigmoid and exp comparisons are taken on logits and log-scales).
#include "api_util.h"
#include "block_scan.cuh"
#include "gs_common.cuh"

namespace gs {

constexpr int kDenThreads = 256;
constexpr int kDenItems = 16;
constexpr int kDenBlock = kDenThreads * kDenItems;  // Gaussians per plan block
constexpr uint8_t kPrune = 0, kKeep = 1, kClone = 2, kSplit = 3;

__global__ void __launch_bounds__(256)
    k_densify_accum(const uint32_t* __restrict__ count, const float4* __restrict__ rec,
                    const float4* __restrict__ grad2d, int64_t n, float half_w, float half_h,
                    float* __restrict__ acc, uint32_t* __restrict__ cnt) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
    if (count[i] == 0u) continue;
    const float4 s = grad2d[3 * i];  // (S1, S2, S3, S4) of the 12-float slot
    const float4 ra = rec[3 * i];    // (mx, my, -A/2, -B)
    const float cc = reinterpret_cast<const float*>(rec)[12 * i + 4];  // -C/2
    const float A = -2.0f * ra.z, B = -ra.w, C = -2.0f * cc;      // exact
    const float dmx = __fadd_rn(__fmul_rn(A, s.x), __fmul_rn(B, s.y));
    const float dmy = __fadd_rn(__fmul_rn(B, s.x), __fmul_rn(C, s.y));
    const float gx = __fmul_rn(dmx, half_w), gy = __fmul_rn(dmy, half_h);
    acc[i] = __fadd_rn(acc[i], __fsqrt_rn(__fadd_rn(__fmul_rn(gx, gx), __fmul_rn(gy, gy))));
    cnt[i] += 1u;
  }
}

__device__ __forceinline__ uint8_t densify_action(const float* __restrict__ P, int64_t n_pad, int64_t i,
                                                  const float* __restrict__ acc, const uint32_t* __restrict__ cnt,
                                                  const gs_densify_cfg& c) {
  const float logit = P[10 * n_pad + i];
  const float smax = fmaxf(fmaxf(P[3 * n_pad + i], P[4 * n_pad + i]), P[5 * n_pad + i]);
  const uint32_t k = cnt[i];
  const float avg = __fdiv_rn(acc[i], float(k > 0u ? k : 1u));
  const bool prune = (logit < c.logit_prune) || (c.prune_big && smax > c.log_prune_scale);
  if (prune) return kPrune;
  if (!(avg > c.grad_threshold)) return kKeep;
  return (smax <= c.log_grow_scale) ? kClone : kSplit;
}

__device__ __forceinline__ uint32_t outputs_of(uint8_t a) { return a == kPrune ? 0u : (a == kKeep ? 1u : 2u); }

// Per block of 4096 Gaussians: actions and the sum of their output counts.
__global__ void __launch_bounds__(kDenThreads)
    k_densify_plan_sums(const float* __restrict__ P, int64_t n, int64_t n_pad, const float* __restrict__ acc,
                        const uint32_t* __restrict__ cnt, gs_densify_cfg c, uint8_t* __restrict__ action,
                        uint32_t* __restrict__ block_sums) {
  __shared__ uint32_t s_warp[8];
  const int64_t base = int64_t(blockIdx.x) * kDenBlock;
  uint32_t s = 0;
  for (int it = 0; it < kDenItems; ++it) {
    const int64_t i = base + int64_t(it) * kDenThreads + threadIdx.x;
    if (i < n) {
      const uint8_t a = densify_action(P, n_pad, i, acc, cnt, c);
      action[i] = a;
      s += outputs_of(a);
    }
  }
  uint32_t total;
  block_excl_scan_256(s, s_warp, &total);
  if (threadIdx.x == 0) block_sums[blockIdx.x] = total;
}

// One block: exclusive scan of the block sums in place; the total to *n_out.
__global__ void __launch_bounds__(1024)
    k_densify_scan(uint32_t* __restrict__ block_sums, int64_t n_blocks, uint32_t* __restrict__ n_out) {
  __shared__ uint32_t s_part[1024];
  const int t = threadIdx.x;
  const int64_t per = (n_blocks + 1023) / 1024;
  const int64_t b0 = int64_t(t) * per, b1 = min(n_blocks, b0 + per);
  uint32_t s = 0;
  for (int64_t b = b0; b < b1; ++b) s += block_sums[b];
  s_part[t] = s;
  __syncthreads();
  for (int o = 1; o < 1024; o <<= 1) {
    const uint32_t y = (t >= o) ? s_part[t - o] : 0u;
    __syncthreads();
    s_part[t] += y;
    __syncthreads();
  }
  uint32_t run = s_part[t] - s;
  for (int64_t b = b0; b < b1; ++b) {
    const uint32_t v = block_sums[b];
    block_sums[b] = run;
    run += v;
  }
  if (t == 1023) *n_out = s_part[1023];
}

// Per block: the offsets of each Gaussian's outputs (items in (round, thread) order).
__global__ void __launch_bounds__(kDenThreads)
    k_densify_plan_offsets(const uint8_t* __restrict__ action, int64_t n, const uint32_t* __restrict__ block_prefix,
                           uint32_t* __restrict__ offset) {
  __shared__ uint32_t s_warp[8];
  const int64_t base = int64_t(blockIdx.x) * kDenBlock;
  uint32_t run = block_prefix[blockIdx.x];
  for (int it = 0; it < kDenItems; ++it) {
    const int64_t i = base + int64_t(it) * kDenThreads + threadIdx.x;
    const uint32_t o = (i < n) ? outputs_of(action[i]) : 0u;
    uint32_t total;
    const uint32_t off = block_excl_scan_256(o, s_warp, &total);
    if (i < n) offset[i] = run + off;
    run += total;
  }
}

// The new planes.  One thread per source Gaussian writes its outputs (output columns
// increase with the source index, so each plane's writes stay mostly coalesced);
// then the padding columns [n_out, n_pad_dst) are cleared.
__global__ void __launch_bounds__(256)
    k_densify_apply(const float* __restrict__ P, const float* __restrict__ M, const float* __restrict__ V, int64_t n,
                    int64_t n_pad, const uint8_t* __restrict__ action, const uint32_t* __restrict__ offset,
                    const uint32_t* __restrict__ n_out_ptr, const float* __restrict__ randn, float log_shrink,
                    float* __restrict__ Pd, float* __restrict__ Md, float* __restrict__ Vd, int64_t n_pad_dst,
                    uint32_t* __restrict__ dev_status) {
  const uint32_t n_out = *n_out_ptr;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  if (int64_t(n_out) > n_pad_dst) {
    if (blockIdx.x == 0 && threadIdx.x == 0) raise_status(dev_status, GS_ERR_CAPACITY);
    return;
  }
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
    const uint8_t a = action[i];
    if (a == kPrune) continue;
    const int64_t o = offset[i];
    if (a == kKeep || a == kClone) {
      for (int pl = 0; pl < kPlanes; ++pl) {
        Pd[pl * n_pad_dst + o] = P[pl * n_pad + i];
        Md[pl * n_pad_dst + o] = M[pl * n_pad + i];
        Vd[pl * n_pad_dst + o] = V[pl * n_pad + i];
      }
      if (a == kClone) {
        for (int pl = 0; pl < kPlanes; ++pl) {
          Pd[pl * n_pad_dst + o + 1] = P[pl * n_pad + i];
          Md[pl * n_pad_dst + o + 1] = 0.0f;
          Vd[pl * n_pad_dst + o + 1] = 0.0f;
        }
      }
      continue;
    }
    // split: two children at mu + R(q) diag(exp s) xi_k, log-scales shrunk
    float q[4];
    for (int k = 0; k < 4; ++k) q[k] = P[(6 + k) * n_pad + i];
    const float qn = rsqrtf(q[0] * q[0] + q[1] * q[1] + q[2] * q[2] + q[3] * q[3]);
    const float w = q[0] * qn, x = q[1] * qn, y = q[2] * qn, z = q[3] * qn;
    const float R[9] = {1.f - 2.f * (y * y + z * z), 2.f * (x * y - w * z),       2.f * (x * z + w * y),
                        2.f * (x * y + w * z),       1.f - 2.f * (x * x + z * z), 2.f * (y * z - w * x),
                        2.f * (x * z - w * y),       2.f * (y * z + w * x),       1.f - 2.f * (x * x + y * y)};
    float s[3];
    for (int k = 0; k < 3; ++k) s[k] = expf(P[(3 + k) * n_pad + i]);
    for (int c = 0; c < 2; ++c) {
      const int64_t oc = o + c;
      float d[3];
      for (int r = 0; r < 3; ++r) {
        d[r] = 0.0f;
        for (int k = 0; k < 3; ++k) d[r] = fmaf(R[3 * r + k], s[k] * randn[6 * i + 3 * c + k], d[r]);
      }
      for (int k = 0; k < 3; ++k) Pd[k * n_pad_dst + oc] = P[k * n_pad + i] + d[k];
      for (int k = 3; k < 6; ++k) Pd[k * n_pad_dst + oc] = __fsub_rn(P[k * n_pad + i], log_shrink);
      for (int pl = 6; pl < kPlanes; ++pl) Pd[pl * n_pad_dst + oc] = P[pl * n_pad + i];
      for (int pl = 0; pl < kPlanes; ++pl) {
        Md[pl * n_pad_dst + oc] = 0.0f;
        Vd[pl * n_pad_dst + oc] = 0.0f;
      }
    }
  }
  // padding columns of the new planes
  const int64_t pad = n_pad_dst - int64_t(n_out);
  for (int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; e < pad * kPlanes; e += stride) {
    const int64_t pl = e / pad, col = int64_t(n_out) + e % pad;
    Pd[pl * n_pad_dst + col] = 0.0f;
    Md[pl * n_pad_dst + col] = 0.0f;
    Vd[pl * n_pad_dst + col] = 0.0f;
  }
}

__global__ void k_opacity_reset(float* __restrict__ P, float* __restrict__ M, float* __restrict__ V, int64_t n,
                                int64_t n_pad, float logit_max) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
    P[10 * n_pad + i] = fminf(P[10 * n_pad + i], logit_max);
    M[10 * n_pad + i] = 0.0f;
    V[10 * n_pad + i] = 0.0f;
  }
}

inline int64_t densify_blocks(int64_t n) {
  const int64_t b = (n + kDenBlock - 1) / kDenBlock;
  return b < 1 ? 1 : b;
}

}  // namespace gs

extern "C" gs_status gs_densify_accumulate(gs_dims dims, const uint32_t* count, const float* rec, const float* grad2d,
                                           int32_t width, int32_t height, float* grad_acc, uint32_t* vis_cnt,
                                           cudaStream_t stream) {
  using namespace gs;
  if (!dims_ok(dims) || !count || !rec || !grad2d || !grad_acc || !vis_cnt || width <= 0 || height <= 0)
    return GS_ERR_INVALID_ARG;
  if (!aligned(grad2d, 16) || !aligned(rec, 16)) return GS_ERR_INVALID_ARG;
  if (dims.n == 0) return GS_OK;
  k_densify_accum<<<grid_for(dims.n, 256, sm_count() * 16), 256, 0, stream>>>(
      count, reinterpret_cast<const float4*>(rec), reinterpret_cast<const float4*>(grad2d), dims.n,
      0.5f * float(width), 0.5f * float(height), grad_acc, vis_cnt);
  return launch_status();
}

extern "C" size_t gs_densify_workspace_bytes(gs_dims dims) {
  if (dims.n < 0) return 0;
  return size_t(gs::densify_blocks(dims.n)) * 4 + 256;
}

extern "C" gs_status gs_densify_plan(gs_dims dims, const float* params, const float* grad_acc, const uint32_t* vis_cnt,
                                     const gs_densify_cfg* cfg, uint8_t* action, uint32_t* offset, uint32_t* n_out,
                                     void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  using namespace gs;
  if (!dims_ok(dims) || !params || !grad_acc || !vis_cnt || !cfg || !action || !offset || !n_out || !workspace)
    return GS_ERR_INVALID_ARG;
  if (workspace_bytes < gs_densify_workspace_bytes(dims) || !aligned(workspace, 4)) return GS_ERR_INVALID_ARG;
  const int64_t nb = densify_blocks(dims.n);
  if (nb > (int64_t(1) << 24)) return GS_ERR_INVALID_ARG;
  uint32_t* block_sums = static_cast<uint32_t*>(workspace);
  k_densify_plan_sums<<<int(nb), kDenThreads, 0, stream>>>(params, dims.n, dims.n_pad, grad_acc, vis_cnt, *cfg,
                                                           action, block_sums);
  k_densify_scan<<<1, 1024, 0, stream>>>(block_sums, nb, n_out);
  k_densify_plan_offsets<<<int(nb), kDenThreads, 0, stream>>>(action, dims.n, block_sums, offset);
  return launch_status();
}

extern "C" gs_status gs_densify_apply(gs_dims src, int64_t n_pad_dst, const float* params, const float* m,
                                      const float* v, const uint8_t* action, const uint32_t* offset,
                                      const uint32_t* n_out, const float* randn, float log_shrink, float* params_dst,
                                      float* m_dst, float* v_dst, uint32_t* dev_status, cudaStream_t stream) {
  using namespace gs;
  if (!dims_ok(src) || !params || !m || !v || !action || !offset || !n_out || !randn || !params_dst || !m_dst ||
      !v_dst || !dev_status)
    return GS_ERR_INVALID_ARG;
  if (n_pad_dst <= 0 || (n_pad_dst % 256) != 0 || n_pad_dst > (int64_t(1) << 31) || !std::isfinite(log_shrink))
    return GS_ERR_INVALID_ARG;
  const int64_t work = src.n > n_pad_dst ? src.n : n_pad_dst;
  k_densify_apply<<<grid_for(work, 256, sm_count() * 16), 256, 0, stream>>>(
      params, m, v, src.n, src.n_pad, action, offset, n_out, randn, log_shrink, params_dst, m_dst, v_dst, n_pad_dst,
      dev_status);
  return launch_status();
}

extern "C" gs_status gs_opacity_reset(gs_dims dims, float* params, float* m, float* v, float logit_max,
                                      cudaStream_t stream) {
  using namespace gs;
  if (!dims_ok(dims) || !params || !m || !v || !std::isfinite(logit_max)) return GS_ERR_INVALID_ARG;
  if (dims.n == 0) return GS_OK;
  k_opacity_reset<<<grid_for(dims.n, 256, sm_count() * 16), 256, 0, stream>>>(params, m, v, dims.n, dims.n_pad,
                                                                            logit_max);
  return launch_status();
}
