/*
 * gs.h -- C ABI of the GB300 (sm_103a) 3D Gaussian Splatting training step.
 *
 * One optimisation step of a scene of anisotropic 3D Gaussians (mean,
 * scale + quaternion covariance, degree-3 SH colour, opacity) for one camera:
 *
 *   gs_project      EWA projection + SH colour, one thread per Gaussian
 *   gs_bin_sort     tile binning: (tile, depth) order by onesweep radix sorts, per-tile
 *                   ranges, records gathered into sorted order
 *   gs_render_fwd   per-tile front-to-back alpha compositing with early termination
 *   gs_render_bwd   L1 loss gradient and the reverse-order compositing backward
 *   gs_project_bwd  chain rule from the 2D gradients to the 59 parameters
 *   gs_adam_step    fused Adam update over every parameter plane
 *   (gs_project_bwd_adam: the last two in one pass; gs_project_bwd_accumulate sums
 *   the gradients of several views of a batch)
 *
 * The method is the one "Toward Distributed 3D Gaussian Splatting for
 * High-Resolution Isosurface Visualization" (section III) trains and "Scaling 3D
 * Gaussian Splatting with Distributed Compute" describes stage by stage: the
 * Gaussian representation and its 59 parameters (memory-wall section), projection
 * as per-Gaussian work and rasterisation as per-pixel work (section on what gsplat
 * distributes), the projected record and SH evaluated before compositing (step
 * walkthrough), tile intersection lists (trace section), gradients flowing back to
 * mean, covariance, colour and opacity, and Adam per parameter.  Thresholds and
 * formulas the pages do not print follow the 3DGS method they cite (Kerbl et al.
 * 2023); each reading is stated at the call it affects.
 *
 * Conventions for every call
 *   - Ownership: the caller owns every buffer (device memory unless stated) and the
 *     stream.  The library never allocates, frees or synchronises.
 *   - Asynchrony: every call only enqueues kernels on `stream` and returns.
 *   - Errors: argument errors (null or misaligned pointers, bad sizes) are
 *     returned at once as a gs_status and nothing is enqueued.  A failed launch
 *     returns GS_ERR_CUDA.  Errors detected on the device (intersection capacity
 *     exceeded, non-finite parameters, a bounded wait that ran out) are OR-ed into
 *     the caller's device word `dev_status` (bits of gs_status) and the kernels
 *     return normally: nothing traps.  Read dev_status after the step.
 *   - Precision: fp32 everywhere.  Quantities that decide an integer (radius, tile
 *     rect, depth key, compositing decisions) follow a frozen fp32 operation
 *     sequence with a Cody-Waite exponential, so they are reproducible bit for bit
 *     by a plain CPU implementation of the same sequence.
 *
 * Parameter layout (`params`, `grads`, `m`, `v`): 59 fp32 planes of stride n_pad
 * (n_pad a multiple of 256, entries [n, n_pad) are padding):
 *   0-2 mean mu, 3-5 log-scale, 6-9 quaternion (w, x, y, z), 10 opacity logit,
 *   11 + 3k + ch: SH coefficient k (< 16) of colour channel ch.
 */
#ifndef GS_H
#define GS_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GS_N_PLANES 59
#define GS_TILE 16          /* tile edge in pixels */
#define GS_REC_FLOATS 12    /* projected record: 48 bytes */
#define GS_N_GRAD2D 9       /* 2D partials per Gaussian */
#define GS_GRAD2D_STRIDE 12 /* floats per Gaussian in grad2d (interleaved, 3 unused) */

typedef enum gs_status {
  GS_OK = 0,
  GS_ERR_INVALID_ARG = 1, /* returned: bad pointer, size or alignment */
  GS_ERR_CUDA = 2,        /* returned: a kernel launch failed */
  GS_ERR_CAPACITY = 4,    /* device: more tile intersections than capacity_K */
  GS_ERR_TIMEOUT = 8,     /* device: a bounded inter-block wait gave up */
  GS_ERR_NONFINITE = 16,  /* device: a Gaussian with NaN/Inf parameters (culled) */
  GS_ERR_SCRATCH_LIMIT = 32 /* returned: sizes exceed gs_bin_sort_noalloc's fixed scratch */
} gs_status;

/* Pinhole camera.  R is the world->camera rotation (row-major) and t the
 * translation, with camera axes x right, y down, z forward.  fx, fy, cx, cy in
 * pixels; pixel (i, j) has its centre at (i + 0.5, j + 0.5).  campos is the camera
 * centre in world space (for the SH view direction).  Gaussians with camera-space
 * z <= near_z are culled. */
typedef struct gs_camera {
  float R[9];
  float t[3];
  float fx, fy, cx, cy;
  int32_t width, height;
  float campos[3];
  float near_z;
} gs_camera;

/* n Gaussians stored in planes of stride n_pad (n_pad % 256 == 0, n <= n_pad). */
typedef struct gs_dims {
  int64_t n;
  int64_t n_pad;
} gs_dims;

/* Per-Gaussian projection output (device arrays of n_pad entries, caller-owned).
 *   rec    12 floats per Gaussian (16-byte aligned): mean2d x, y; (ca, cb, cc) =
 *          (-A/2, -B, -C/2) for the conic [[A, B], [B, C]] (inverse 2D covariance),
 *          so that power = ca dx^2 + cb dx dy + cc dy^2; opacity; r, g, b; the
 *          Gaussian's index (uint32 bits); a skip radius (at pixels farther than it
 *          from the mean the entry's alpha is below the compositing threshold;
 *          +FLT_MAX if not bounded, -FLT_MAX if never composited); camera-space z
 *          (as in depth).  The pages' projected record (means2d, depth, conic,
 *          opacity, colour) minus the radius, which is kept in its own array.
 *   depth  camera-space z.
 *   radius pixel radius ceil(3 sqrt(lambda_max)), 0 if culled.
 *   rect   2 uint32 per Gaussian: (tx0 | ty0 << 16, tx1 | ty1 << 16), inclusive tile
 *          bounds of the box [mean - r, mean + r].
 *   count  number of tiles in rect, 0 if culled. */
typedef struct gs_proj {
  float* rec;
  float* depth;
  int32_t* radius;
  uint32_t* rect;
  uint32_t* count;
} gs_proj;

/* Tile bins (device arrays, caller-owned).
 *   keys     capacity_K uint64 keys (tile << 32 | fp32 depth bits), sorted.
 *   ids      capacity_K uint32 Gaussian indices in key order (ties by index).
 *   rec      capacity_K records (12 floats, 16-byte aligned) in key order.
 *   ranges   2 uint32 per tile: [start, end) of the tile's entries; [0, 0) for a
 *            tile with no entries.
 *   n_isect  1 uint32: the total number of tile intersections K of this view
 *            (may exceed capacity_K, in which case GS_ERR_CAPACITY is raised
 *            and only the first capacity_K entries exist). */
typedef struct gs_bins {
  uint64_t* keys;
  uint32_t* ids;
  float* rec;
  uint32_t* ranges;
  uint32_t* n_isect;
} gs_bins;

/* ---------------------------------------------------------------------------
 * gs_project -- projection of every Gaussian for one camera.
 * "Scaling 3D Gaussian Splatting with Distributed Compute", step walkthrough
 * (project locally: 2D means, depths, conics, radii, visibility; SH evaluated to
 * RGB before compositing).  Per Gaussian: t = R mu + t; cull if t.z <= near_z;
 * Sigma = M M^T with M = R(q / |q|) diag(exp(log-scale)); 2D covariance
 * J W Sigma W^T J^T + 0.3 I with the perspective Jacobian J at the mean (abscissae
 * clamped to 1.3 x the half field of view); conic = its inverse; radius =
 * ceil(3 sqrt(mid + sqrt(max(0.1, mid^2 - det)))); tile rect of the box
 * [mean - r, mean + r], culled if empty; opacity = sigmoid(logit); colour =
 * max(0, sum_k Y_k(dir) sh_k + 0.5) with real SH (Condon-Shortley phase) at the
 * unit direction from campos to mu.
 *   params  59 x n_pad fp32 (read).   proj: outputs (write), n_pad entries each.
 *   dev_status: device uint32 (GS_ERR_NONFINITE may be OR-ed in).
 * Errors: GS_ERR_INVALID_ARG for null/misaligned pointers, n < 0, n > n_pad,
 * n_pad % 256 != 0, width/height <= 0 or not finite intrinsics.  n == 0 is a no-op. */
gs_status gs_project(gs_dims dims, const float* params, const gs_camera* cam, gs_proj proj,
                     uint32_t* dev_status, cudaStream_t stream);

/* Bytes of device scratch gs_bin_sort needs for n Gaussians, capacity_K
 * intersections and the camera's tile grid. */
size_t gs_bin_sort_workspace_bytes(gs_dims dims, uint32_t capacity_K, int32_t width, int32_t height);

/* ---------------------------------------------------------------------------
 * gs_bin_sort -- tile binning.  "Scaling 3D Gaussian Splatting with Distributed
 * Compute", memory-wall section (per-tile sorted lists of Gaussian-to-pixel
 * intersections) and trace section (one tile-intersection pass per Gaussian, one
 * offset pass per intersection).  The result is that of a stable sort of one key
 * (tile_id << 32 | fp32 bits of depth) per tile of each visible Gaussian's rect,
 * emitted in index order: per tile, the ordered subsequence of the global (depth,
 * index) order of the Gaussians whose rect contains the tile.  It is computed by
 * two stable onesweep LSD radix sorts (8-bit digits, decoupled look-back with a
 * bounded wait): the visible Gaussians by depth bits (4 passes), then one
 * (tile, index) pair per intersection, emitted in depth order, by tile
 * (ceil(log2 tiles / 8) passes); then tile ranges, the 64-bit keys and the
 * records gathered into key order.
 *   proj      output of gs_project (read).
 *   workspace device scratch of at least gs_bin_sort_workspace_bytes(), 256-byte
 *             aligned; contents need not be initialised and are clobbered.
 *   bins      outputs (write); keys/ids/rec hold capacity_K entries.
 * Errors: GS_ERR_INVALID_ARG as for gs_project, plus capacity_K == 0 or > 2^30,
 * workspace too small or misaligned.  K > capacity_K sets GS_ERR_CAPACITY on the
 * device; the look-back wait running out sets GS_ERR_TIMEOUT. */
gs_status gs_bin_sort(gs_dims dims, const gs_proj* proj, const gs_camera* cam, uint32_t capacity_K,
                      gs_bins bins, void* workspace, size_t workspace_bytes, uint32_t* dev_status,
                      cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * gs_render_fwd -- per-tile front-to-back alpha compositing.  "Scaling 3D
 * Gaussian Splatting with Distributed Compute", section on what gsplat
 * distributes (rasterisation is per-pixel work per camera) and trace section
 * (tiled rasteriser).  For each pixel over its tile's sorted entries, T = 1:
 * power = ca dx^2 + cb dx dy + cc dy^2 with d = pixel centre - mean2d; skip if
 * power > 0; alpha = min(0.99, o exp(power)); skip if alpha < 1/255; stop,
 * without compositing, if T (1 - alpha) < 1e-4; else C += rgb alpha T and
 * T <- T (1 - alpha).  Output C + T bg.  T (1 - alpha) is formed as the fused
 * T - alpha T (one rounding), part of the frozen fp32 sequence.
 *   bins       from gs_bin_sort (read).   bg: 3 floats (host).
 *   image      3 x H x W fp32 (channel planes), T_final H x W fp32,
 *   n_contrib  H x W uint32: entries iterated up to the last composited (write).
 *   cmask      composited-entry masks for gs_render_bwd (write, 4-byte aligned,
 *              cmask_bytes >= gs_render_cmask_bytes(capacity_K, width, height)):
 *              for every 8x4 pixel block of a tile and every 32-entry chunk of the
 *              tile's list that the block walks, each pixel's 32-bit mask of the
 *              entries it composited.  Chunks past a block's last composited entry
 *              are not written.  Treat the layout as opaque: gs_render_bwd reads it.
 * Errors: GS_ERR_INVALID_ARG for null/misaligned pointers, bad sizes or a short
 * cmask. */
size_t gs_render_cmask_bytes(uint32_t capacity_K, int32_t width, int32_t height);
gs_status gs_render_fwd(const gs_camera* cam, const gs_bins* bins, uint32_t capacity_K, const float bg[3],
                        float* image, float* T_final, uint32_t* n_contrib, uint32_t* cmask, size_t cmask_bytes,
                        uint32_t* dev_status, cudaStream_t stream);

/* gs_render_fwd_counted -- gs_render_fwd that also writes, per pixel, the number of
 * entries it composited (alpha >= 1/255 and not stopped by the transmittance test):
 *   n_used  H x W uint32 (write).
 * The image, T_final, n_contrib and cmask are those of gs_render_fwd, bit for bit.
 * Not part of the training step: it measures how much of the iterated work
 * composites (the mean number of Gaussians composited per pixel of a view).
 * Errors: as gs_render_fwd, plus a null n_used. */
gs_status gs_render_fwd_counted(const gs_camera* cam, const gs_bins* bins, uint32_t capacity_K, const float bg[3],
                                float* image, float* T_final, uint32_t* n_contrib, uint32_t* n_used,
                                uint32_t* cmask, size_t cmask_bytes, uint32_t* dev_status, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * gs_render_bwd -- loss gradient and the compositing backward.  "Scaling 3D
 * Gaussian Splatting with Distributed Compute", objective and gradient-descent
 * section (a weighted L1 and D-SSIM objective between render and ground truth;
 * gradients flow back to mean, covariance, colour and opacity) and step walkthrough
 * (loss computed locally, gradients back through the same stages).
 * dL/dC = l1_weight sign(C - C*) / (3 H W) + dLdC_extra (if non-null, e.g. the D-SSIM
 * term's gradient from gs_ssim_bwd); loss_out = l1_weight mean |C - C*| over the
 * 3 H W values.  Each pixel walks the entries it composited (the forward's cmask) in
 * reverse, recomputing alpha in the forward's fp32 sequence and recovering T by
 * division by (1 - alpha), and produces per entry the partials of the loss with
 * respect to opacity and colour (r, g, b) and, for mean2d and the conic, the five
 * moments of q = dL/dpower over the pixel offset (dx, dy) = (px - mx, py - my); each
 * pixel adds its partials to grad2d with global atomics (summation order is not
 * fixed).  The conic is the Gaussian's own, so its
 * products are applied once to the sums, by the consumers: with power =
 * -(A dx^2 + C dy^2)/2 - B dx dy and S1..S5 the sums of q dx, q dy, q dx^2, q dx dy,
 * q dy^2,  dL/dmx = A S1 + B S2,  dL/dmy = B S1 + C S2,  dL/dA = -S3/2,
 * dL/dB = -S4,  dL/dC = -S5/2.
 *   image, T_final, n_contrib, cmask: outputs of gs_render_fwd for the same bins (read;
 *   cmask_bytes as there).
 *   target      3 x H x W fp32 (read).
 *   l1_weight   weight of the L1 term (1 for the L1 objective, 1 - lambda with D-SSIM).
 *   dLdC_extra  3 x H x W fp32 added to the loss gradient, or null.
 *   grad2d      GS_GRAD2D_STRIDE x n_pad fp32, interleaved (write; zeroed by this
 *               call first): Gaussian i's sums at 12 i + (S1, S2, S3, S4, S5,
 *               d opacity, d r, d g, d b), 12 i + 9..11 unused.  A warp's nine sums
 *               for one Gaussian land in two 32-byte sectors instead of nine planes'
 *               lines.  gs_project_bwd (and the calls built on it) and
 *               gs_densify_accumulate read this layout.
 *   loss_out    1 fp32 (write; zeroed first).
 * Errors: as gs_render_fwd, plus a negative or non-finite l1_weight. */
gs_status gs_render_bwd(gs_dims dims, const gs_camera* cam, const gs_bins* bins, uint32_t capacity_K,
                        const float bg[3], const float* image, const float* target, const float* T_final,
                        const uint32_t* n_contrib, const uint32_t* cmask, size_t cmask_bytes, float l1_weight,
                        const float* dLdC_extra, float* grad2d, float* loss_out, uint32_t* dev_status,
                        cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * gs_ssim_fwd / gs_ssim_bwd -- the D-SSIM term.  "Scaling 3D Gaussian Splatting
 * with Distributed Compute", objective paragraph (a weighted combination of an L1
 * term and a D-SSIM term; the formula did not survive on the page, read as
 * (1 - lambda) L1 + lambda (1 - SSIM)).  SSIM after Wang et al. 2004: an 11x11
 * Gaussian window (sigma 1.5, separable), C1 = 0.01^2, C2 = 0.03^2, zero padding
 * outside the image, averaged over the 3 H W values.
 * gs_ssim_fwd: ssim_out = mean SSIM of image against target (1 fp32, zeroed first);
 *   maps (GS_SSIM_MAPS x H x W fp32, caller-owned scratch) receives, per pixel and
 *   channel, the derivatives of lambda (1 - SSIM) with respect to the local mean of
 *   the image, its variance and the covariance (planes 0-2, 3-5, 6-8), and the local
 *   means of image and target (planes 9-11, 12-14).
 * gs_ssim_bwd: dLdC (3 x H x W fp32, write) = d[lambda (1 - SSIM)] / d image, from maps.
 * Errors: GS_ERR_INVALID_ARG for null pointers, non-positive sizes, lambda < 0. */
#define GS_SSIM_MAPS 15
gs_status gs_ssim_fwd(int32_t width, int32_t height, const float* image, const float* target, float lambda,
                      float* maps, float* ssim_out, cudaStream_t stream);
gs_status gs_ssim_bwd(int32_t width, int32_t height, const float* image, const float* target, const float* maps,
                      float* dLdC, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * gs_project_bwd -- chain rule of gs_project.  "Scaling 3D Gaussian Splatting
 * with Distributed Compute", objective section (gradients reach mu, Sigma, c and
 * alpha as they would the weights of a network).  conic -> 2D covariance ->
 * (Jacobian, Sigma); Jacobian and mean2d -> camera-space mean -> mu; Sigma -> M ->
 * (rotation -> normalised quaternion -> quaternion, scale -> log-scale); sigmoid
 * -> logit; colour -> SH coefficients and view direction -> mu.  Clamped colour
 * channels and clamped Jacobian abscissae pass zero gradient; radius and rect are
 * constants.  Culled Gaussians and padding get zero gradients.
 *   params 59 x n_pad (read); proj from gs_project (read); grad2d as written by
 *   gs_render_bwd (read, 16-byte aligned);
 *   grads  59 x n_pad fp32 (write, every entry).
 * Errors: as gs_project. */
gs_status gs_project_bwd(gs_dims dims, const float* params, const gs_camera* cam, const gs_proj* proj,
                         const float* grad2d, float* grads, uint32_t* dev_status, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * gs_project_bwd_accumulate -- gs_project_bwd adding into grads instead of
 * overwriting it: grads += chain rule of this view's grad2d (entries of culled
 * Gaussians and padding are left as they are).  For a step over a batch of views
 * ("Scaling 3D Gaussian Splatting with Distributed Compute", batch-size section):
 * the first view writes with gs_project_bwd, later ones accumulate, and each view's
 * loss gradient carries its 1 / batch weight through gs_render_bwd's l1_weight.
 *   grads  59 x n_pad fp32 (read and write).  Other arguments and errors as
 *   gs_project_bwd. */
gs_status gs_project_bwd_accumulate(gs_dims dims, const float* params, const gs_camera* cam, const gs_proj* proj,
                                    const float* grad2d, float* grads, uint32_t* dev_status, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * gs_adam_step -- fused Adam over all 59 planes (padding included).  "Scaling 3D
 * Gaussian Splatting with Distributed Compute", DDP background (two moments per
 * parameter) and step walkthrough (Adam over the rank's own parameters).
 *   m = beta1 m + (1 - beta1) g;  v = beta2 v + (1 - beta2) g^2;
 *   p -= (lr[plane] / (1 - beta1^t)) m / (sqrt(v) / sqrt(1 - beta2^t) + eps)
 * The hyperparameters arrive in fp64; 1 - beta, the bias corrections and the
 * per-plane step sizes are formed on the host in fp64 and rounded to fp32 once
 * (so that, e.g., 1 - 0.999 is not taken from an fp32 0.999).  The square root and
 * the division of the update are the hardware approximations (relative error of
 * order 2^-22), which move p by about 1e-6 of the step size.
 *   params, m, v: 59 x n_pad fp32 (read and write, 16-byte aligned);
 *   grads 59 x n_pad (read); lr_plane: 59 floats (host); t >= 1 the step count.
 * Errors: GS_ERR_INVALID_ARG for null/misaligned pointers, bad sizes, t < 1 or
 * betas outside [0, 1). */
gs_status gs_adam_step(gs_dims dims, float* params, const float* grads, float* m, float* v,
                       const float lr_plane[GS_N_PLANES], double beta1, double beta2, double eps, int64_t t,
                       cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * gs_batch_hyper -- the Adam hyperparameters of a step over `batch` views ("Scaling 3D
 * Gaussian Splatting with Distributed Compute", batch-size section): learning rates
 * times sqrt(batch), epsilon divided by sqrt(batch), and each momentum coefficient
 * 1 - batch (1 - beta), the linearisation of beta^batch (the page's formula did not
 * survive extraction; under this reading beta1 = 0.9 reaches zero at batch 10, as the
 * page states), held at zero beyond.  All in fp64; batch 1 returns the inputs.
 * Host-only (no device work).
 *   lr_plane: 59 doubles (host, read); lr_out: 59 doubles (host, write); the three
 *   scalars written through their pointers.
 * Errors: GS_ERR_INVALID_ARG for batch < 1, null pointers, betas outside [0, 1), a
 * negative or non-finite eps or a non-finite learning rate. */
gs_status gs_batch_hyper(int32_t batch, const double* lr_plane, double beta1, double beta2, double eps,
                         double* lr_out, double* beta1_out, double* beta2_out, double* eps_out);

/* ---------------------------------------------------------------------------
 * gs_project_bwd_adam -- gs_project_bwd followed by gs_adam_step in one pass, without
 * materialising the 59 gradient planes.  Same arithmetic as the two calls (each
 * thread derives its Gaussian's gradients in registers and applies the Adam element
 * update of gs_adam_step to all 59 of its parameters, culled and padding ones with
 * gradient 0), so it moves 1456 instead of 2164 bytes per Gaussian.  Use the two
 * separate calls when the gradients themselves are wanted.
 *   params  59 x n_pad (read, then updated in place); proj, grad2d as for
 *   gs_project_bwd; m, v, lr_plane, beta1, beta2, eps, t as for gs_adam_step.
 *   grads_in null, or 59 x n_pad fp32 (read, 16-byte aligned): gradients that earlier
 *   views of a batch accumulated, added to this view's before the update (the last
 *   view of a batch step; the batch's scaled hyperparameters are the caller's).
 * Errors: the union of gs_project_bwd's and gs_adam_step's. */
gs_status gs_project_bwd_adam(gs_dims dims, float* params, const gs_camera* cam, const gs_proj* proj,
                              const float* grad2d, const float* grads_in, float* m, float* v,
                              const float lr_plane[GS_N_PLANES], double beta1, double beta2, double eps, int64_t t,
                              uint32_t* dev_status, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * gs_project_bwd_adam_tdev -- gs_project_bwd_adam with the Adam step count read from
 * device memory when the kernel runs, for steps replayed from a CUDA graph (whose
 * kernel arguments are fixed at capture).  The bias corrections and per-plane step
 * sizes are formed from it in fp64 inside the kernel, as gs_adam_step forms them on
 * the host.  The pages' trace attributes idle GPU time to launch overhead between
 * small kernels ("Scaling 3D Gaussian Splatting with Distributed Compute", trace
 * section); a captured step removes the per-launch host work.
 *   t_dev  1 int64 (device, 8-byte aligned, read): the step count, >= 1 when the
 *          kernel runs (advance it with gs_step_counter_add inside the graph).
 *   Other arguments and errors as gs_project_bwd_adam (lr_plane, beta1, beta2 and
 *   eps are captured by value). */
gs_status gs_project_bwd_adam_tdev(gs_dims dims, float* params, const gs_camera* cam, const gs_proj* proj,
                                   const float* grad2d, const float* grads_in, float* m, float* v,
                                   const float lr_plane[GS_N_PLANES], double beta1, double beta2, double eps,
                                   const int64_t* t_dev, uint32_t* dev_status, cudaStream_t stream);

/* gs_step_counter_add -- *counter += delta on the stream (counter: 1 device int64,
 * 8-byte aligned).  Errors: GS_ERR_INVALID_ARG for a null or misaligned counter. */
gs_status gs_step_counter_add(int64_t* counter, int64_t delta, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Adaptive density control.  "Scaling 3D Gaussian Splatting with Distributed
 * Compute": adaptive density control clones, splits and prunes Gaussians every
 * hundred steps (memory-wall section), from 2D position gradients accumulated over the
 * steps (step walkthrough), starting at step 500 (trace section).  Thresholds and
 * the split rule are the cited 3DGS method's; each threshold is formed in fp64
 * (gs_densify_thresholds) and the kernels compare in fp32:
 *   grow if acc / max(cnt, 1) > grad_threshold (2e-4, the NDC-scaled 2D gradient);
 *   clone if the largest log-scale <= log_grow_scale (ln(0.01 x scene extent)), else
 *   split into two children at mu + R(q) diag(exp s) xi_k with log-scales - log_shrink
 *   (ln 1.6); prune (first) if the opacity logit < logit_prune (ln(0.005 / 0.995)) or,
 *   with prune_big, the largest log-scale > log_prune_scale (ln(0.1 x extent)).
 * gs_densify_thresholds (below) forms them. */
typedef struct gs_densify_cfg {
  float grad_threshold;
  float logit_prune;
  float log_grow_scale;
  float log_prune_scale;
  int32_t prune_big;
} gs_densify_cfg;

#define GS_DENSIFY_PRUNE 0
#define GS_DENSIFY_KEEP 1
#define GS_DENSIFY_CLONE 2
#define GS_DENSIFY_SPLIT 3

/* gs_densify_thresholds -- the configuration above, the split's log_shrink and the
 * opacity reset's logit_max, formed in fp64 from the method's settings and rounded to
 * fp32 once:  grad_threshold = grow_grad2d (2e-4);  logit_prune = logit(prune_opa)
 * (prune_opa = 0.005);  log_grow_scale = ln(grow_scale3d x extent) (0.01);
 * log_prune_scale = ln(prune_scale3d x extent) (0.1);  log_shrink = ln(split_shrink)
 * (1.6);  logit_reset = logit(2 prune_opa).  Host-only (no device work).
 * Errors: GS_ERR_INVALID_ARG for null outputs, a non-positive or non-finite extent,
 * scale factor or shrink, or prune_opa outside (0, 0.5). */
gs_status gs_densify_thresholds(double extent, double grow_grad2d, double grow_scale3d, double prune_opa,
                                double prune_scale3d, double split_shrink, int32_t prune_big, gs_densify_cfg* cfg,
                                float* log_shrink, float* logit_reset);

/* gs_densify_accumulate -- for each Gaussian i < n with count[i] > 0 (visible in
 * this view): grad_acc[i] += |(d mx W/2, d my H/2)|, vis_cnt[i] += 1, with the mean
 * gradient formed from grad2d's sums (gs_render_bwd's layout) and the conic of the
 * Gaussian's record: d mx = A S1 + B S2, d my = B S1 + C S2 (A = -2 rec[2],
 * B = -rec[3], C = -2 rec[4]).  fp32: each product, sum, square and the square root
 * rounded once, in that order.
 *   count, rec (gs_proj.count, gs_proj.rec), grad2d (read); grad_acc n fp32,
 *   vis_cnt n uint32 (read and write; the caller zeroes them after each
 *   refinement).
 * Errors: GS_ERR_INVALID_ARG for bad dims, sizes or pointers. */
gs_status gs_densify_accumulate(gs_dims dims, const uint32_t* count, const float* rec, const float* grad2d,
                                int32_t width, int32_t height, float* grad_acc, uint32_t* vis_cnt,
                                cudaStream_t stream);

/* gs_densify_plan -- per Gaussian i < n its action (GS_DENSIFY_*) and the offset of
 * its outputs in the new arrays (exclusive scan of 0, 1, 2, 2 outputs for prune,
 * keep, clone, split, in index order); *n_out = the new count (device).
 *   params 59 x n_pad (read); action n uint8, offset n uint32, n_out 1 uint32
 *   (write); workspace >= gs_densify_workspace_bytes(dims), 4-byte aligned.
 * Errors: GS_ERR_INVALID_ARG for bad dims, pointers or a small workspace. */
size_t gs_densify_workspace_bytes(gs_dims dims);
gs_status gs_densify_plan(gs_dims dims, const float* params, const float* grad_acc, const uint32_t* vis_cnt,
                          const gs_densify_cfg* cfg, uint8_t* action, uint32_t* offset, uint32_t* n_out,
                          void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* gs_densify_apply -- the new parameter and Adam moment planes (59 x n_pad_dst each)
 * from a plan.  A kept Gaussian and a clone's original keep their moments; a clone's
 * copy and a split's two children start with zero moments; the children's means are
 * mu + R(q) diag(exp s) xi_k with xi = randn[6 i + 3 k .. + 2] (inputs: the method's
 * random draws), their log-scales s - log_shrink, every other plane copied.
 * Columns [n_out, n_pad_dst) are cleared.
 *   n_pad_dst: a multiple of 256 >= *n_out (else GS_ERR_CAPACITY on the device and
 *   nothing is written); the destination arrays must not overlap the sources.
 * Errors: GS_ERR_INVALID_ARG for bad dims, pointers, n_pad_dst or log_shrink. */
gs_status gs_densify_apply(gs_dims src, int64_t n_pad_dst, const float* params, const float* m, const float* v,
                           const uint8_t* action, const uint32_t* offset, const uint32_t* n_out, const float* randn,
                           float log_shrink, float* params_dst, float* m_dst, float* v_dst, uint32_t* dev_status,
                           cudaStream_t stream);

/* gs_opacity_reset -- opacity logit <- min(logit, logit_max) (the method resets
 * opacities to at most 2 x 0.005 periodically) and the opacity plane's Adam moments
 * zeroed, for Gaussians i < n.  Errors: GS_ERR_INVALID_ARG for bad dims, pointers or
 * a non-finite logit_max. */
gs_status gs_opacity_reset(gs_dims dims, float* params, float* m, float* v, float logit_max, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * gs_bin_sort_noalloc -- gs_bin_sort for callers that must not allocate device
 * memory (for example a render loop whose memory is all reserved in advance, or an
 * embedding application whose own allocator owns the GPU).  The paper has no
 * counterpart; this is a library convenience.  Results are identical to
 * gs_bin_sort's.
 *   Scratch: a fixed array inside the library (68.5 MiB), used in place of the
 *   workspace argument; the caller still passes proj and bins.  Under lazy module
 *   loading (the CUDA default) the array is placed on a device by the first call
 *   there, and that placement is itself a device allocation; with
 *   CUDA_MODULE_LOADING=EAGER every process that loads the library holds it on
 *   each GPU it uses.  Either way it stays until the process exits.
 *   Limits: n <= GS_NOALLOC_MAX_N, capacity_K <= GS_NOALLOC_MAX_K, at most
 *   GS_NOALLOC_MAX_TILES tiles; larger sizes return GS_ERR_SCRATCH_LIMIT and
 *   nothing is enqueued.
 *   Set-up: the first call on a device looks up the array's device address (with
 *   that device current) and keeps it.  Make one call during start-up, before the
 *   caller stops allocating and before any stream capture.  The kept address
 *   assumes the device's primary context and no cudaDeviceReset after that call.
 *   Every call on a device shares the one array: calls whose kernels overlap on
 *   the GPU (other streams, other host threads) race and corrupt each other.
 *   Serialise them.  Each call clears what must start at zero itself.
 * Errors: as gs_bin_sort, plus GS_ERR_SCRATCH_LIMIT. */
#define GS_NOALLOC_MAX_N (1 << 22)
#define GS_NOALLOC_MAX_K (1 << 20)
#define GS_NOALLOC_MAX_TILES (1 << 16)
gs_status gs_bin_sort_noalloc(gs_dims dims, const gs_proj* proj, const gs_camera* cam, uint32_t capacity_K,
                              gs_bins bins, uint32_t* dev_status, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * gs_spatial_order -- a storage order of the Gaussians along a Morton (Z-order)
 * curve of their means, for locality: Gaussians near each other in space share
 * tiles, and stored near each other the binning's record gather and the backward's
 * gradient atomics find their lines in L2.  Not a step of the method (the pages give
 * no storage order); a layout applied once, before training and after each density
 * refinement.  A step's result depends on the order only through the index that
 * breaks ties between equal fp32 depths in a tile.
 *   Code of Gaussian i: per axis q = floor((mu - lo) * (1023 / (hi - lo)) + 0.5)
 *   clamped to [0, 1023], each operation in IEEE fp32 in that order, lo and hi the
 *   axis's smallest and largest finite mean (a non-finite coordinate counts as lo;
 *   hi = lo gives q = 0); the 30-bit code interleaves the three q, x in bit 0.
 *   perm: n uint32 (device, written): perm[j] = the index of the Gaussian placed at
 *   j, i.e. the stable sort of the codes (ties by index).
 *   workspace: gs_spatial_order_workspace_bytes(dims) bytes, 256-byte aligned.
 * Errors: GS_ERR_INVALID_ARG for bad dims, null or misaligned pointers, a short
 * workspace; a look-back wait that runs out raises GS_ERR_TIMEOUT in dev_status. */
size_t gs_spatial_order_workspace_bytes(gs_dims dims);
gs_status gs_spatial_order(gs_dims dims, const float* params, uint32_t* perm, void* workspace, size_t workspace_bytes,
                           uint32_t* dev_status, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * gs_permute_planes -- applies a storage order to `planes` planes of 32-bit values
 * (parameters, Adam moments, per-Gaussian accumulators):
 *   dst[p n_pad + j] = src[p n_pad + perm[j]] for j < n; the padding j >= n copied.
 *   src, dst distinct device buffers of planes x n_pad elements, 4-byte aligned;
 *   perm as gs_spatial_order writes it (every entry < n).
 * Errors: GS_ERR_INVALID_ARG for bad dims, planes <= 0, null or aliasing buffers. */
gs_status gs_permute_planes(gs_dims dims, int32_t planes, const uint32_t* perm, const void* src, void* dst,
                            cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * gs_util_expf -- the library's fp32 exponential (Cody-Waite reduction, degree-7
 * Taylor polynomial, 2^k scaling; the one every compositing decision uses), on n
 * device floats, so that callers can check it against another implementation.
 * Errors: GS_ERR_INVALID_ARG for null pointers or n < 0. */
gs_status gs_util_expf(const float* x, float* y, int64_t n, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * gs_util_lookback_probe / gs_util_mbarrier_probe -- make the library's two bounded
 * waits run out, so that callers and tests can see the failure path without a GPU
 * fault or hang.  gs_util_lookback_probe runs one onesweep pass whose first partition
 * never runs: the one CTA's look-back waits on a word nothing publishes for spin_limit
 * tries (the binning's passes use 2^22), raises GS_ERR_TIMEOUT in dev_status and
 * finishes in bounds.  gs_util_mbarrier_probe waits on an mbarrier nothing arrives at
 * for wait_limit tries (the rasterisers use 2^24), raises GS_ERR_TIMEOUT and returns.
 *   scratch: gs_util_lookback_probe_bytes() device bytes, 16-byte aligned.
 * Errors: GS_ERR_INVALID_ARG for a limit <= 0, null pointers, short or misaligned
 * scratch. */
size_t gs_util_lookback_probe_bytes(void);
gs_status gs_util_lookback_probe(int32_t spin_limit, void* scratch, size_t scratch_bytes, uint32_t* dev_status,
                                 cudaStream_t stream);
gs_status gs_util_mbarrier_probe(int32_t wait_limit, uint32_t* dev_status, cudaStream_t stream);

/* gs_sm_count -- the streaming multiprocessor count of the current device, which
 * the library queries once per device and sizes the grids of its streaming and
 * persistent kernels from (those kernels loop over their work with a grid stride, so
 * the count changes speed, never results).  Returns 1 if no device can be queried. */
int32_t gs_sm_count(void);

/* Static description of a status value (several bits: the lowest set one). */
const char* gs_status_str(uint32_t status);

/* Library version, e.g. "gs-gb300 0.1 sm_103a". */
const char* gs_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GS_H */
