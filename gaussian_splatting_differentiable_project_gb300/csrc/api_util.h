// Host-side argument checks shared by the C-ABI entry points.
#pragma once

#include <cmath>
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/gs.h"

namespace gs {

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline bool dims_ok(const gs_dims& d) {
  return d.n >= 0 && d.n_pad >= d.n && d.n_pad > 0 && (d.n_pad % 256) == 0 && d.n_pad <= (int64_t(1) << 31);
}

inline bool camera_ok(const gs_camera* c) {
  if (!c) return false;
  if (c->width <= 0 || c->height <= 0 || c->width > 65535 * 16 || c->height > 65535 * 16) return false;
  const float v[] = {c->fx, c->fy, c->cx, c->cy, c->near_z};
  for (float x : v)
    if (!std::isfinite(x)) return false;
  if (!(c->fx > 0.0f) || !(c->fy > 0.0f)) return false;
  for (int k = 0; k < 9; ++k)
    if (!std::isfinite(c->R[k])) return false;
  for (int k = 0; k < 3; ++k)
    if (!std::isfinite(c->t[k]) || !std::isfinite(c->campos[k])) return false;
  return true;
}

inline int64_t n_tiles(const gs_camera* c) {
  return int64_t((c->width + GS_TILE - 1) / GS_TILE) * int64_t((c->height + GS_TILE - 1) / GS_TILE);
}

inline gs_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? GS_OK : GS_ERR_CUDA;
}

}  // namespace gs
