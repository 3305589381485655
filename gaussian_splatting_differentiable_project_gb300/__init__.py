"""GB300 (sm_103a) 3D Gaussian Splatting training step.

A thin ctypes binding over the C-ABI library ``libgs.so`` (declared in
``include/gs.h``).  Every step of the path runs in the library's CUDA kernels;
this module only marshals arguments: PyTorch tensors supply device memory and the
current CUDA stream.  There is no CPU path: if the library is missing or no GPU is
present, the calls raise.

Entry points (same names as the C ABI, without the ``gs_`` prefix):
- the step: ``project``, ``bin_sort``, ``render_fwd``, ``render_bwd``,
  ``project_bwd``, ``adam_step``, and the fused ``project_bwd_adam``;
  ``render_fwd_counted`` (the forward with per-pixel composited counts);
- the D-SSIM term: ``ssim_fwd``, ``ssim_bwd``;
- batches and graphs: ``project_bwd_accumulate``, ``project_bwd_adam_tdev``,
  ``step_counter_add``;
- density control: ``densify_thresholds``, ``densify_accumulate``, ``densify_plan``,
  ``densify_apply``, ``opacity_reset``;
- the batch step's Adam hyperparameters: ``batch_hyper``;
- storage order: ``spatial_order``, ``permute_planes``;
- sizes and utilities: ``bin_sort_workspace_bytes``, ``densify_workspace_bytes``,
  ``spatial_order_workspace_bytes``, ``bin_sort_noalloc``, ``util_expf``,
  ``sm_count``.
Tensor arguments must be dense CUDA tensors; anything else raises ``GsError``
before a call is made.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

from . import _build

N_PLANES = 59
TILE = 16
REC_FLOATS = 12
N_GRAD2D = 9
GRAD2D_STRIDE = 12  # floats per Gaussian in the interleaved grad2d buffer
SSIM_MAPS = 15  # planes of gs_ssim_fwd's maps: 3 partials and 2 local means per channel


def grad2d_planes(grad2d, n: int) -> np.ndarray:
    """The nine sums of Gaussians [0, n) as (9, n) planes, from the interleaved
    (n_pad, 12) buffer gs_render_bwd writes (host copy): the five moments of
    dL/dpower (S1..S5, see gs.h) and the opacity and colour partials."""
    g = grad2d.detach().cpu().numpy() if hasattr(grad2d, "detach") else np.asarray(grad2d)
    return np.ascontiguousarray(g.reshape(-1, GRAD2D_STRIDE)[:n, :N_GRAD2D].T)


def grad2d_interleaved(planes: np.ndarray) -> np.ndarray:
    """(9, n_pad) planes (moments S1..S5, then opacity and colour partials) -> the
    interleaved (n_pad, 12) layout the projection backward reads (host arrays)."""
    planes = np.asarray(planes, np.float32)
    out = np.zeros((planes.shape[1], GRAD2D_STRIDE), np.float32)
    out[:, :N_GRAD2D] = planes.T
    return out


GS_OK = 0
GS_ERR_INVALID_ARG = 1
GS_ERR_CUDA = 2
GS_ERR_CAPACITY = 4
GS_ERR_TIMEOUT = 8
GS_ERR_NONFINITE = 16
GS_ERR_SCRATCH_LIMIT = 32

_lock = threading.Lock()
_lib = None


class GsError(RuntimeError):
    pass


class GsCamera(ctypes.Structure):
    _fields_ = [("R", ctypes.c_float * 9), ("t", ctypes.c_float * 3),
                ("fx", ctypes.c_float), ("fy", ctypes.c_float),
                ("cx", ctypes.c_float), ("cy", ctypes.c_float),
                ("width", ctypes.c_int32), ("height", ctypes.c_int32),
                ("campos", ctypes.c_float * 3), ("near_z", ctypes.c_float)]


class GsDims(ctypes.Structure):
    _fields_ = [("n", ctypes.c_int64), ("n_pad", ctypes.c_int64)]


class GsProj(ctypes.Structure):
    _fields_ = [("rec", ctypes.c_void_p), ("depth", ctypes.c_void_p), ("radius", ctypes.c_void_p),
                ("rect", ctypes.c_void_p), ("count", ctypes.c_void_p)]


class GsDensifyCfg(ctypes.Structure):
    _fields_ = [("grad_threshold", ctypes.c_float), ("logit_prune", ctypes.c_float),
                ("log_grow_scale", ctypes.c_float), ("log_prune_scale", ctypes.c_float),
                ("prune_big", ctypes.c_int32)]


DENSIFY_PRUNE, DENSIFY_KEEP, DENSIFY_CLONE, DENSIFY_SPLIT = 0, 1, 2, 3


class GsBins(ctypes.Structure):
    _fields_ = [("keys", ctypes.c_void_p), ("ids", ctypes.c_void_p), ("rec", ctypes.c_void_p),
                ("ranges", ctypes.c_void_p), ("n_isect", ctypes.c_void_p)]


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libgs.so (building it in-tree first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if build_if_missing and not _build.up_to_date():
            _build.build()
        if not os.path.exists(_build.LIB):
            raise GsError(f"CUDA library not built: {_build.LIB}")
        lib = ctypes.CDLL(_build.LIB)
        P = ctypes.c_void_p
        st = ctypes.c_int
        lib.gs_project.argtypes = [GsDims, P, ctypes.POINTER(GsCamera), GsProj, P, P]
        lib.gs_project.restype = st
        lib.gs_bin_sort_workspace_bytes.argtypes = [GsDims, ctypes.c_uint32, ctypes.c_int32, ctypes.c_int32]
        lib.gs_bin_sort_workspace_bytes.restype = ctypes.c_size_t
        lib.gs_bin_sort.argtypes = [GsDims, ctypes.POINTER(GsProj), ctypes.POINTER(GsCamera), ctypes.c_uint32,
                                    GsBins, P, ctypes.c_size_t, P, P]
        lib.gs_bin_sort.restype = st
        lib.gs_bin_sort_noalloc.argtypes = [GsDims, ctypes.POINTER(GsProj), ctypes.POINTER(GsCamera),
                                            ctypes.c_uint32, GsBins, P, P]
        lib.gs_bin_sort_noalloc.restype = st
        lib.gs_render_cmask_bytes.argtypes = [ctypes.c_uint32, ctypes.c_int32, ctypes.c_int32]
        lib.gs_render_cmask_bytes.restype = ctypes.c_size_t
        lib.gs_render_fwd.argtypes = [ctypes.POINTER(GsCamera), ctypes.POINTER(GsBins), ctypes.c_uint32,
                                      ctypes.POINTER(ctypes.c_float), P, P, P, P, ctypes.c_size_t, P, P]
        lib.gs_render_fwd.restype = st
        lib.gs_render_fwd_counted.argtypes = [ctypes.POINTER(GsCamera), ctypes.POINTER(GsBins), ctypes.c_uint32,
                                              ctypes.POINTER(ctypes.c_float), P, P, P, P, P, ctypes.c_size_t, P, P]
        lib.gs_render_fwd_counted.restype = st
        lib.gs_render_bwd.argtypes = [GsDims, ctypes.POINTER(GsCamera), ctypes.POINTER(GsBins), ctypes.c_uint32,
                                      ctypes.POINTER(ctypes.c_float), P, P, P, P, P, ctypes.c_size_t, ctypes.c_float,
                                      P, P, P, P, P]
        lib.gs_render_bwd.restype = st
        lib.gs_project_bwd.argtypes = [GsDims, P, ctypes.POINTER(GsCamera), ctypes.POINTER(GsProj), P, P, P, P]
        lib.gs_project_bwd.restype = st
        lib.gs_project_bwd_accumulate.argtypes = [GsDims, P, ctypes.POINTER(GsCamera), ctypes.POINTER(GsProj), P, P,
                                                  P, P]
        lib.gs_project_bwd_accumulate.restype = st
        lib.gs_adam_step.argtypes = [GsDims, P, P, P, P, ctypes.POINTER(ctypes.c_float), ctypes.c_double,
                                     ctypes.c_double, ctypes.c_double, ctypes.c_int64, P]
        lib.gs_adam_step.restype = st
        lib.gs_project_bwd_adam.argtypes = [GsDims, P, ctypes.POINTER(GsCamera), ctypes.POINTER(GsProj), P, P, P, P,
                                            ctypes.POINTER(ctypes.c_float), ctypes.c_double, ctypes.c_double,
                                            ctypes.c_double, ctypes.c_int64, P, P]
        lib.gs_project_bwd_adam.restype = st
        lib.gs_project_bwd_adam_tdev.argtypes = [GsDims, P, ctypes.POINTER(GsCamera), ctypes.POINTER(GsProj), P, P, P,
                                                 P, ctypes.POINTER(ctypes.c_float), ctypes.c_double, ctypes.c_double,
                                                 ctypes.c_double, P, P, P]
        lib.gs_project_bwd_adam_tdev.restype = st
        lib.gs_step_counter_add.argtypes = [P, ctypes.c_int64, P]
        lib.gs_step_counter_add.restype = st
        lib.gs_densify_accumulate.argtypes = [GsDims, P, P, P, ctypes.c_int32, ctypes.c_int32, P, P, P]
        lib.gs_densify_accumulate.restype = st
        lib.gs_densify_workspace_bytes.argtypes = [GsDims]
        lib.gs_densify_workspace_bytes.restype = ctypes.c_size_t
        lib.gs_densify_plan.argtypes = [GsDims, P, P, P, ctypes.POINTER(GsDensifyCfg), P, P, P, P, ctypes.c_size_t, P]
        lib.gs_densify_plan.restype = st
        lib.gs_densify_apply.argtypes = [GsDims, ctypes.c_int64, P, P, P, P, P, P, P, ctypes.c_float, P, P, P, P, P]
        lib.gs_densify_apply.restype = st
        lib.gs_opacity_reset.argtypes = [GsDims, P, P, P, ctypes.c_float, P]
        lib.gs_opacity_reset.restype = st
        lib.gs_ssim_fwd.argtypes = [ctypes.c_int32, ctypes.c_int32, P, P, ctypes.c_float, P, P, P]
        lib.gs_ssim_fwd.restype = st
        lib.gs_ssim_bwd.argtypes = [ctypes.c_int32, ctypes.c_int32, P, P, P, P, P]
        lib.gs_ssim_bwd.restype = st
        lib.gs_util_expf.argtypes = [P, P, ctypes.c_int64, P]
        lib.gs_util_expf.restype = st
        lib.gs_util_lookback_probe_bytes.argtypes = []
        lib.gs_util_lookback_probe_bytes.restype = ctypes.c_size_t
        lib.gs_util_lookback_probe.argtypes = [ctypes.c_int32, P, ctypes.c_size_t, P, P]
        lib.gs_util_lookback_probe.restype = st
        lib.gs_util_mbarrier_probe.argtypes = [ctypes.c_int32, P, P]
        lib.gs_util_mbarrier_probe.restype = st
        lib.gs_spatial_order_workspace_bytes.argtypes = [GsDims]
        lib.gs_spatial_order_workspace_bytes.restype = ctypes.c_size_t
        lib.gs_spatial_order.argtypes = [GsDims, P, P, P, ctypes.c_size_t, P, P]
        lib.gs_spatial_order.restype = st
        lib.gs_permute_planes.argtypes = [GsDims, ctypes.c_int32, P, P, P, P]
        lib.gs_permute_planes.restype = st
        lib.gs_status_str.argtypes = [ctypes.c_uint32]
        lib.gs_status_str.restype = ctypes.c_char_p
        lib.gs_version.restype = ctypes.c_char_p
        D = ctypes.POINTER(ctypes.c_double)
        lib.gs_batch_hyper.argtypes = [ctypes.c_int32, D, ctypes.c_double, ctypes.c_double, ctypes.c_double, D, D, D,
                                       D]
        lib.gs_batch_hyper.restype = st
        lib.gs_densify_thresholds.argtypes = [ctypes.c_double] * 6 + [ctypes.c_int32, ctypes.POINTER(GsDensifyCfg),
                                                                      ctypes.POINTER(ctypes.c_float),
                                                                      ctypes.POINTER(ctypes.c_float)]
        lib.gs_densify_thresholds.restype = st
        lib.gs_sm_count.argtypes = []
        lib.gs_sm_count.restype = ctypes.c_int32
        _lib = lib
        return lib


def status_str(code: int) -> str:
    return load().gs_status_str(int(code)).decode()


def _check(code: int, what: str) -> None:
    if code != GS_OK:
        raise GsError(f"{what}: {status_str(code)} ({code})")


def _stream(stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _p(t) -> ctypes.c_void_p:
    """The device address of a dense CUDA tensor.  The library reads and writes every
    buffer as a dense array in device memory, so a host tensor (whose address a kernel
    cannot dereference) or a strided view (which it would misread) is refused here,
    before anything is enqueued."""
    if not t.is_cuda:
        raise GsError(f"expected a CUDA tensor, got one on {t.device} with shape {tuple(t.shape)}")
    if not t.is_contiguous():
        raise GsError(f"expected a contiguous tensor, got shape {tuple(t.shape)} with strides {t.stride()}")
    return ctypes.c_void_p(t.data_ptr())


# element kinds of _buf: fp32, any 4-byte integer (int32 or uint32 buffers), int64,
# bytes, or any 4-byte type
_KINDS = {
    "f32": ("fp32", lambda t: t.dtype == _torch().float32),
    "i32": ("a 4-byte integer type", lambda t: t.element_size() == 4 and not t.is_floating_point()),
    "i64": ("int64", lambda t: t.dtype == _torch().int64),
    "u8": ("uint8", lambda t: t.dtype == _torch().uint8),
    "any4": ("a 4-byte type", lambda t: t.element_size() == 4),
}


def _torch():
    import torch
    return torch


def _buf(t, count: int, kind: str, what: str) -> ctypes.c_void_p:
    """``_p`` for a buffer the library reads or writes ``count`` elements of: its type
    and size are checked first (a short buffer would be overrun on the device)."""
    name, ok = _KINDS[kind]
    if not ok(t):
        raise GsError(f"{what}: expected {name}, got {t.dtype}")
    if t.numel() < count:
        raise GsError(f"{what}: needs {count} elements, got {t.numel()} (shape {tuple(t.shape)})")
    return _p(t)


def _planes(t, n_pad: int, what: str, planes: int = N_PLANES) -> ctypes.c_void_p:
    return _buf(t, planes * n_pad, "f32", what)


def _check_proj(proj, n_pad: int) -> None:
    if proj.depth.numel() < n_pad:
        raise GsError(f"projection buffers hold {proj.depth.numel()} Gaussians, need {n_pad}")


def _check_bins(bins, cam: GsCamera) -> None:
    if bins.ranges.shape[0] < n_tiles(cam.width, cam.height):
        raise GsError(f"bin buffers hold ranges for {bins.ranges.shape[0]} tiles, the view has "
                      f"{n_tiles(cam.width, cam.height)}")


def camera(cam: dict) -> GsCamera:
    c = GsCamera()
    c.R[:] = [float(v) for v in np.asarray(cam["R"], np.float32).reshape(9)]
    c.t[:] = [float(v) for v in np.asarray(cam["t"], np.float32).reshape(3)]
    c.fx, c.fy, c.cx, c.cy = (float(np.float32(cam[k])) for k in ("fx", "fy", "cx", "cy"))
    c.width, c.height = int(cam["width"]), int(cam["height"])
    c.campos[:] = [float(v) for v in np.asarray(cam["campos"], np.float32).reshape(3)]
    c.near_z = float(np.float32(cam.get("near_z", 0.01)))
    return c


def dims(n: int, n_pad: int) -> GsDims:
    return GsDims(int(n), int(n_pad))


def n_tiles(width: int, height: int) -> int:
    return (-(-width // TILE)) * (-(-height // TILE))


# ----------------------------------------------------------------------------- buffers

class ProjBuffers:
    """Device outputs of ``project`` for n_pad Gaussians."""

    def __init__(self, n_pad: int, device="cuda"):
        import torch
        self.rec = torch.empty((n_pad, REC_FLOATS), dtype=torch.float32, device=device)
        self.depth = torch.empty(n_pad, dtype=torch.float32, device=device)
        self.radius = torch.empty(n_pad, dtype=torch.int32, device=device)
        self.rect = torch.empty((n_pad, 2), dtype=torch.int32, device=device)
        self.count = torch.empty(n_pad, dtype=torch.int32, device=device)

    def c(self) -> GsProj:
        return GsProj(self.rec.data_ptr(), self.depth.data_ptr(), self.radius.data_ptr(), self.rect.data_ptr(),
                      self.count.data_ptr())


class BinBuffers:
    """Device outputs and scratch of ``bin_sort`` for ``capacity`` intersections."""

    def __init__(self, n: int, capacity: int, width: int, height: int, device="cuda"):
        import torch
        self.capacity = int(capacity)
        self.keys = torch.empty(capacity, dtype=torch.int64, device=device)
        self.ids = torch.empty(capacity, dtype=torch.int32, device=device)
        self.rec = torch.empty((capacity, REC_FLOATS), dtype=torch.float32, device=device)
        self.ranges = torch.empty((n_tiles(width, height), 2), dtype=torch.int32, device=device)
        self.n_isect = torch.zeros(2, dtype=torch.int32, device=device)
        ws = bin_sort_workspace_bytes(n, capacity, width, height)
        self.workspace = torch.empty(ws + 256, dtype=torch.uint8, device=device)
        self.ws_bytes = ws
        # the forward's composited-entry masks for this capacity and tile grid (written by
        # render_fwd, read by render_bwd)
        self.cmask_bytes = render_cmask_bytes(capacity, width, height)
        self.cmask = torch.empty(self.cmask_bytes // 4, dtype=torch.int32, device=device)

    def ws_ptr(self) -> int:
        p = self.workspace.data_ptr()
        return (p + 255) & ~255

    def c(self) -> GsBins:
        return GsBins(self.keys.data_ptr(), self.ids.data_ptr(), self.rec.data_ptr(), self.ranges.data_ptr(),
                      self.n_isect.data_ptr())


# ----------------------------------------------------------------------------- entry points

def project(n: int, params, cam: dict, proj: ProjBuffers, dev_status, stream=None) -> None:
    cc = camera(cam)
    n_pad = int(params.shape[1])
    _check_proj(proj, n_pad)
    _check(load().gs_project(dims(n, n_pad), _planes(params, n_pad, "params"), ctypes.byref(cc), proj.c(),
                             _buf(dev_status, 1, "i32", "dev_status"), _stream(stream)), "gs_project")


def bin_sort_workspace_bytes(n: int, capacity: int, width: int, height: int) -> int:
    return int(load().gs_bin_sort_workspace_bytes(dims(n, max(256, n)), int(capacity), int(width), int(height)))


def render_cmask_bytes(capacity: int, width: int, height: int) -> int:
    return int(load().gs_render_cmask_bytes(int(capacity), int(width), int(height)))


def _check_cmask(bins, cc) -> ctypes.c_void_p:
    need = render_cmask_bytes(bins.capacity, cc.width, cc.height)
    return _buf(bins.cmask, need // 4, "i32", "bins.cmask")


def bin_sort(n: int, n_pad: int, proj: ProjBuffers, cam: dict, bins: BinBuffers, dev_status, stream=None) -> None:
    cc = camera(cam)
    _check_proj(proj, n_pad)
    _check_bins(bins, cc)
    pc = proj.c()
    _check(load().gs_bin_sort(dims(n, n_pad), ctypes.byref(pc), ctypes.byref(cc), bins.capacity, bins.c(),
                              ctypes.c_void_p(bins.ws_ptr()), bins.ws_bytes, _buf(dev_status, 1, "i32", "dev_status"),
                              _stream(stream)), "gs_bin_sort")


def bin_sort_noalloc(n: int, n_pad: int, proj: ProjBuffers, cam: dict, bins: BinBuffers, dev_status,
                     stream=None) -> None:
    """gs_bin_sort with the library's fixed scratch instead of bins.workspace (for
    callers that may not allocate device memory; see include/gs.h for the limits)."""
    cc = camera(cam)
    _check_proj(proj, n_pad)
    _check_bins(bins, cc)
    pc = proj.c()
    _check(load().gs_bin_sort_noalloc(dims(n, n_pad), ctypes.byref(pc), ctypes.byref(cc), bins.capacity, bins.c(),
                                      _buf(dev_status, 1, "i32", "dev_status"), _stream(stream)),
           "gs_bin_sort_noalloc")


def _lr(lr_plane):
    lr = [float(x) for x in np.asarray(lr_plane, np.float64).reshape(-1)]
    if len(lr) != N_PLANES:
        raise GsError(f"lr_plane: needs {N_PLANES} learning rates, got {len(lr)}")
    return (ctypes.c_float * N_PLANES)(*lr)


def _bg(bg):
    return (ctypes.c_float * 3)(*[float(x) for x in bg])


def render_fwd(cam: dict, bins: BinBuffers, bg, image, T_final, n_contrib, dev_status, stream=None) -> None:
    cc = camera(cam)
    _check_bins(bins, cc)
    bc = bins.c()
    P = cc.width * cc.height
    cm = _check_cmask(bins, cc)
    _check(load().gs_render_fwd(ctypes.byref(cc), ctypes.byref(bc), bins.capacity, _bg(bg),
                                _buf(image, 3 * P, "f32", "image"), _buf(T_final, P, "f32", "T_final"),
                                _buf(n_contrib, P, "i32", "n_contrib"), cm, bins.cmask_bytes,
                                _buf(dev_status, 1, "i32", "dev_status"), _stream(stream)), "gs_render_fwd")


def render_fwd_counted(cam: dict, bins: BinBuffers, bg, image, T_final, n_contrib, n_used, dev_status,
                       stream=None) -> None:
    """render_fwd that also writes each pixel's number of composited entries."""
    cc = camera(cam)
    _check_bins(bins, cc)
    bc = bins.c()
    P = cc.width * cc.height
    cm = _check_cmask(bins, cc)
    _check(load().gs_render_fwd_counted(ctypes.byref(cc), ctypes.byref(bc), bins.capacity, _bg(bg),
                                        _buf(image, 3 * P, "f32", "image"), _buf(T_final, P, "f32", "T_final"),
                                        _buf(n_contrib, P, "i32", "n_contrib"), _buf(n_used, P, "i32", "n_used"),
                                        cm, bins.cmask_bytes, _buf(dev_status, 1, "i32", "dev_status"),
                                        _stream(stream)), "gs_render_fwd_counted")


def render_bwd(n: int, n_pad: int, cam: dict, bins: BinBuffers, bg, image, target, T_final, n_contrib, grad2d,
               loss, dev_status, stream=None, l1_weight: float = 1.0, dLdC_extra=None) -> None:
    cc = camera(cam)
    _check_bins(bins, cc)
    bc = bins.c()
    P = cc.width * cc.height
    extra = _buf(dLdC_extra, 3 * P, "f32", "dLdC_extra") if dLdC_extra is not None else None
    cm = _check_cmask(bins, cc)
    _check(load().gs_render_bwd(dims(n, n_pad), ctypes.byref(cc), ctypes.byref(bc), bins.capacity, _bg(bg),
                                _buf(image, 3 * P, "f32", "image"), _buf(target, 3 * P, "f32", "target"),
                                _buf(T_final, P, "f32", "T_final"), _buf(n_contrib, P, "i32", "n_contrib"),
                                cm, bins.cmask_bytes, float(l1_weight), extra,
                                _planes(grad2d, n_pad, "grad2d", GRAD2D_STRIDE),
                                _buf(loss, 1, "f32", "loss"), _buf(dev_status, 1, "i32", "dev_status"),
                                _stream(stream)), "gs_render_bwd")


def ssim_fwd(image, target, lam: float, maps, ssim_out, stream=None) -> None:
    """Mean SSIM of image (3 x H x W) against target into ssim_out, and the partial
    derivatives of lam (1 - SSIM) and local means into maps (SSIM_MAPS x H x W)."""
    _, H, W = image.shape
    P = H * W
    _check(load().gs_ssim_fwd(W, H, _buf(image, 3 * P, "f32", "image"), _buf(target, 3 * P, "f32", "target"),
                              float(lam), _buf(maps, SSIM_MAPS * P, "f32", "maps"),
                              _buf(ssim_out, 1, "f32", "ssim_out"), _stream(stream)), "gs_ssim_fwd")


def ssim_bwd(image, target, maps, dLdC, stream=None) -> None:
    """d[lam (1 - SSIM)] / d image into dLdC (3 x H x W), from ssim_fwd's maps."""
    _, H, W = image.shape
    P = H * W
    _check(load().gs_ssim_bwd(W, H, _buf(image, 3 * P, "f32", "image"), _buf(target, 3 * P, "f32", "target"),
                              _buf(maps, SSIM_MAPS * P, "f32", "maps"), _buf(dLdC, 3 * P, "f32", "dLdC"),
                              _stream(stream)), "gs_ssim_bwd")


def project_bwd(n: int, params, cam: dict, proj: ProjBuffers, grad2d, grads, dev_status, stream=None) -> None:
    cc = camera(cam)
    n_pad = int(params.shape[1])
    _check_proj(proj, n_pad)
    pc = proj.c()
    _check(load().gs_project_bwd(dims(n, n_pad), _planes(params, n_pad, "params"), ctypes.byref(cc),
                                 ctypes.byref(pc), _planes(grad2d, n_pad, "grad2d", GRAD2D_STRIDE),
                                 _planes(grads, n_pad, "grads"), _buf(dev_status, 1, "i32", "dev_status"),
                                 _stream(stream)), "gs_project_bwd")


def project_bwd_accumulate(n: int, params, cam: dict, proj: ProjBuffers, grad2d, grads, dev_status,
                           stream=None) -> None:
    """grads += the chain rule of this view's grad2d (a later view of a batch)."""
    cc = camera(cam)
    n_pad = int(params.shape[1])
    _check_proj(proj, n_pad)
    pc = proj.c()
    _check(load().gs_project_bwd_accumulate(dims(n, n_pad), _planes(params, n_pad, "params"), ctypes.byref(cc),
                                            ctypes.byref(pc), _planes(grad2d, n_pad, "grad2d", GRAD2D_STRIDE),
                                            _planes(grads, n_pad, "grads"), _buf(dev_status, 1, "i32", "dev_status"),
                                            _stream(stream)), "gs_project_bwd_accumulate")


def adam_step(n: int, params, grads, m, v, lr_plane, beta1: float, beta2: float, eps: float, t: int,
              stream=None) -> None:
    """Adam step number ``t`` (>= 1); bias corrections are formed inside the call."""
    lr = _lr(lr_plane)
    n_pad = int(params.shape[1])
    _check(load().gs_adam_step(dims(n, n_pad), _planes(params, n_pad, "params"), _planes(grads, n_pad, "grads"),
                               _planes(m, n_pad, "m"), _planes(v, n_pad, "v"), lr, float(beta1), float(beta2),
                               float(eps), int(t), _stream(stream)), "gs_adam_step")


def project_bwd_adam(n: int, params, cam: dict, proj: ProjBuffers, grad2d, m, v, lr_plane, beta1: float,
                     beta2: float, eps: float, t: int, dev_status, stream=None, grads_in=None) -> None:
    """Projection backward and Adam step ``t`` in one pass (no gradient planes);
    ``grads_in``: gradients accumulated by earlier views of a batch, or None."""
    cc = camera(cam)
    n_pad = int(params.shape[1])
    _check_proj(proj, n_pad)
    pc = proj.c()
    lr = _lr(lr_plane)
    gin = _planes(grads_in, n_pad, "grads_in") if grads_in is not None else None
    _check(load().gs_project_bwd_adam(dims(n, n_pad), _planes(params, n_pad, "params"), ctypes.byref(cc),
                                      ctypes.byref(pc), _planes(grad2d, n_pad, "grad2d", GRAD2D_STRIDE), gin,
                                      _planes(m, n_pad, "m"), _planes(v, n_pad, "v"), lr, float(beta1),
                                      float(beta2), float(eps), int(t), _buf(dev_status, 1, "i32", "dev_status"),
                                      _stream(stream)), "gs_project_bwd_adam")


def project_bwd_adam_tdev(n: int, params, cam: dict, proj: ProjBuffers, grad2d, m, v, lr_plane, beta1: float,
                          beta2: float, eps: float, t_dev, dev_status, stream=None, grads_in=None) -> None:
    """project_bwd_adam with the step count read from the device int64 ``t_dev`` when
    the kernel runs (for CUDA graph capture)."""
    cc = camera(cam)
    n_pad = int(params.shape[1])
    _check_proj(proj, n_pad)
    pc = proj.c()
    lr = _lr(lr_plane)
    gin = _planes(grads_in, n_pad, "grads_in") if grads_in is not None else None
    _check(load().gs_project_bwd_adam_tdev(dims(n, n_pad), _planes(params, n_pad, "params"), ctypes.byref(cc),
                                           ctypes.byref(pc), _planes(grad2d, n_pad, "grad2d", GRAD2D_STRIDE), gin,
                                           _planes(m, n_pad, "m"), _planes(v, n_pad, "v"), lr, float(beta1),
                                           float(beta2), float(eps), _buf(t_dev, 1, "i64", "t_dev"),
                                           _buf(dev_status, 1, "i32", "dev_status"), _stream(stream)),
           "gs_project_bwd_adam_tdev")


def step_counter_add(counter, delta: int = 1, stream=None) -> None:
    _check(load().gs_step_counter_add(_buf(counter, 1, "i64", "counter"), int(delta), _stream(stream)),
           "gs_step_counter_add")


def densify_thresholds(extent: float, grow_grad2d: float = 2e-4, grow_scale3d: float = 0.01,
                       prune_opa: float = 0.005, prune_scale3d: float = 0.1, split_shrink: float = 1.6,
                       prune_big: bool = False):
    """The density-control thresholds (gs_densify_thresholds): (the plan's
    configuration, ln split_shrink, the opacity-reset logit of 2 x prune_opa)."""
    cfg = GsDensifyCfg()
    shrink, reset = ctypes.c_float(), ctypes.c_float()
    _check(load().gs_densify_thresholds(float(extent), float(grow_grad2d), float(grow_scale3d), float(prune_opa),
                                        float(prune_scale3d), float(split_shrink), int(bool(prune_big)),
                                        ctypes.byref(cfg), ctypes.byref(shrink), ctypes.byref(reset)),
           "gs_densify_thresholds")
    return cfg, float(shrink.value), float(reset.value)


def batch_hyper(batch: int, lr_plane, beta1: float, beta2: float, eps: float):
    """Adam hyperparameters of a step over ``batch`` views (gs_batch_hyper): (per-plane
    learning rates, beta1, beta2, eps), fp64."""
    lr = np.ascontiguousarray(np.asarray(lr_plane, np.float64).reshape(-1))
    if lr.size != N_PLANES:
        raise GsError(f"lr_plane: needs {N_PLANES} learning rates, got {lr.size}")
    out = np.empty(N_PLANES, np.float64)
    b1, b2, e = ctypes.c_double(), ctypes.c_double(), ctypes.c_double()
    D = ctypes.POINTER(ctypes.c_double)
    _check(load().gs_batch_hyper(int(batch), lr.ctypes.data_as(D), float(beta1), float(beta2), float(eps),
                                 out.ctypes.data_as(D), ctypes.byref(b1), ctypes.byref(b2), ctypes.byref(e)),
           "gs_batch_hyper")
    return out, b1.value, b2.value, e.value


def densify_accumulate(n: int, n_pad: int, proj: "ProjBuffers", grad2d, width: int, height: int, grad_acc, vis_cnt,
                       stream=None) -> None:
    """grad_acc += the NDC-scaled norm of each visible Gaussian's mean2d gradient, formed
    from grad2d's moments and the conic of its record in ``proj``; vis_cnt += 1."""
    _check_proj(proj, n_pad)
    _check(load().gs_densify_accumulate(dims(n, n_pad), _p(proj.count), _p(proj.rec),
                                        _planes(grad2d, n_pad, "grad2d", GRAD2D_STRIDE), int(width), int(height),
                                        _buf(grad_acc, n, "f32", "grad_acc"), _buf(vis_cnt, n, "i32", "vis_cnt"),
                                        _stream(stream)), "gs_densify_accumulate")


def densify_plan(n: int, params, grad_acc, vis_cnt, cfg: GsDensifyCfg, action, offset, n_out, workspace,
                 stream=None) -> None:
    n_pad = int(params.shape[1])
    _check(load().gs_densify_plan(dims(n, n_pad), _planes(params, n_pad, "params"),
                                  _buf(grad_acc, n, "f32", "grad_acc"), _buf(vis_cnt, n, "i32", "vis_cnt"),
                                  ctypes.byref(cfg), _buf(action, n, "u8", "action"), _buf(offset, n, "i32", "offset"),
                                  _buf(n_out, 1, "i32", "n_out"), _p(workspace),
                                  workspace.numel() * workspace.element_size(), _stream(stream)), "gs_densify_plan")


def spatial_order_workspace_bytes(n: int, n_pad: int) -> int:
    return int(load().gs_spatial_order_workspace_bytes(dims(n, n_pad)))


def spatial_order(n: int, params, perm, workspace, dev_status, stream=None) -> None:
    """perm[j] = index of the Gaussian stored at j in Morton order of the means."""
    n_pad = int(params.shape[1])
    _check(load().gs_spatial_order(dims(n, n_pad), _planes(params, n_pad, "params"), _buf(perm, n, "i32", "perm"),
                                   _p(workspace), int(workspace.numel() * workspace.element_size()),
                                   _buf(dev_status, 1, "i32", "dev_status"), _stream(stream)), "gs_spatial_order")


def permute_planes(n: int, perm, src, dst, stream=None) -> None:
    """dst[:, j] = src[:, perm[j]] for j < n, padding copied (src, dst: planes x n_pad,
    any 4-byte element type)."""
    planes = 1 if src.dim() == 1 else int(src.shape[0])
    n_pad = int(src.shape[-1])
    _check(load().gs_permute_planes(dims(n, n_pad), planes, _buf(perm, n, "i32", "perm"),
                                    _buf(src, planes * n_pad, "any4", "src"), _buf(dst, planes * n_pad, "any4", "dst"),
                                    _stream(stream)), "gs_permute_planes")


def densify_workspace_bytes(n: int, n_pad: int) -> int:
    return int(load().gs_densify_workspace_bytes(dims(n, n_pad)))


def densify_apply(n: int, params, m, v, action, offset, n_out, randn, log_shrink: float, params_dst, m_dst, v_dst,
                  dev_status, stream=None) -> None:
    n_pad, n_pad_dst = int(params.shape[1]), int(params_dst.shape[1])
    _check(load().gs_densify_apply(dims(n, n_pad), n_pad_dst, _planes(params, n_pad, "params"),
                                   _planes(m, n_pad, "m"), _planes(v, n_pad, "v"), _buf(action, n, "u8", "action"),
                                   _buf(offset, n, "i32", "offset"), _buf(n_out, 1, "i32", "n_out"),
                                   _buf(randn, 6 * n, "f32", "randn"), float(log_shrink),
                                   _planes(params_dst, n_pad_dst, "params_dst"), _planes(m_dst, n_pad_dst, "m_dst"),
                                   _planes(v_dst, n_pad_dst, "v_dst"), _buf(dev_status, 1, "i32", "dev_status"),
                                   _stream(stream)), "gs_densify_apply")


def opacity_reset(n: int, params, m, v, logit_max: float, stream=None) -> None:
    n_pad = int(params.shape[1])
    _check(load().gs_opacity_reset(dims(n, n_pad), _planes(params, n_pad, "params"), _planes(m, n_pad, "m"),
                                   _planes(v, n_pad, "v"), float(logit_max), _stream(stream)), "gs_opacity_reset")


def util_expf(x, y, stream=None) -> None:
    _check(load().gs_util_expf(_buf(x, 0, "f32", "x"), _buf(y, x.numel(), "f32", "y"), x.numel(), _stream(stream)),
           "gs_util_expf")


def version() -> str:
    return load().gs_version().decode()


def sm_count() -> int:
    """The current device's SM count, as the library queried it for its grids."""
    return int(load().gs_sm_count())


from .trainer import HostTargets, Trainer  # noqa: E402  (re-export)
