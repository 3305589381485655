// Host-side rules of the method that turn user settings into the scalars the kernels
// take: the Adam hyperparameters of a step over several views, and the density-control
// thresholds.  Both are formed in fp64 here, so the binding above the C ABI only
// marshals arguments.
#include <cmath>

#include "api_util.h"

// "Scaling 3D Gaussian Splatting with Distributed Compute", batch-size section: with B
// views per step the learning rates scale with sqrt(B) and epsilon with 1 / sqrt(B); the
// page's momentum formula did not survive extraction, and is read as the linearisation
// 1 - B (1 - beta) of beta^B, under which beta1 = 0.9 reaches zero at B = 10 as the page
// says, held at zero beyond.
extern "C" gs_status gs_batch_hyper(int32_t batch, const double* lr_plane, double beta1, double beta2, double eps,
                                    double* lr_out, double* beta1_out, double* beta2_out, double* eps_out) {
  if (batch < 1 || !lr_plane || !lr_out || !beta1_out || !beta2_out || !eps_out) return GS_ERR_INVALID_ARG;
  if (!(beta1 >= 0.0 && beta1 < 1.0) || !(beta2 >= 0.0 && beta2 < 1.0) || !(eps >= 0.0) || !std::isfinite(eps))
    return GS_ERR_INVALID_ARG;
  const double root = std::sqrt(double(batch));
  for (int k = 0; k < GS_N_PLANES; ++k) {
    if (!std::isfinite(lr_plane[k])) return GS_ERR_INVALID_ARG;
    lr_out[k] = lr_plane[k] * root;
  }
  const double b1 = 1.0 - double(batch) * (1.0 - beta1);
  const double b2 = 1.0 - double(batch) * (1.0 - beta2);
  *beta1_out = b1 > 0.0 ? b1 : 0.0;
  *beta2_out = b2 > 0.0 ? b2 : 0.0;
  *eps_out = eps / root;
  return GS_OK;
}

// The density-control thresholds of the 3DGS method the pages cite ("Scaling 3D
// Gaussian Splatting with Distributed Compute", memory-wall section: clones, splits and
// prunes every hundred steps), as the comparisons of gs_densify_plan and
// gs_opacity_reset take them: the opacity thresholds as logits and the scale
// thresholds as logs, each formed in fp64 and rounded to fp32 once.
extern "C" gs_status gs_densify_thresholds(double extent, double grow_grad2d, double grow_scale3d,
                                           double prune_opa, double prune_scale3d, double split_shrink,
                                           int32_t prune_big, gs_densify_cfg* cfg, float* log_shrink,
                                           float* logit_reset) {
  if (!cfg || !log_shrink || !logit_reset) return GS_ERR_INVALID_ARG;
  if (!(extent > 0.0) || !std::isfinite(extent) || !(grow_grad2d >= 0.0) || !std::isfinite(grow_grad2d) ||
      !(grow_scale3d > 0.0) || !(prune_scale3d > 0.0) || !(prune_opa > 0.0 && prune_opa < 0.5) ||
      !(split_shrink > 0.0) || !std::isfinite(split_shrink) || !std::isfinite(grow_scale3d) ||
      !std::isfinite(prune_scale3d))
    return GS_ERR_INVALID_ARG;
  cfg->grad_threshold = float(grow_grad2d);
  cfg->logit_prune = float(std::log(prune_opa / (1.0 - prune_opa)));
  cfg->log_grow_scale = float(std::log(grow_scale3d * extent));
  cfg->log_prune_scale = float(std::log(prune_scale3d * extent));
  cfg->prune_big = prune_big ? 1 : 0;
  *log_shrink = float(std::log(split_shrink));
  const double reset = 2.0 * prune_opa;
  *logit_reset = float(std::log(reset / (1.0 - reset)));
  return GS_OK;
}
