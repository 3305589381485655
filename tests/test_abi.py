"""The C-ABI library builds for sm_103a, loads without a GPU, and exports every
function that include/gs.h declares (no compute calls here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        src = open(os.path.join(ROOT, "include", fn)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names.update(re.findall(r"\b(gs_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


def test_header_declares_the_six_stages():
    names = _declared_functions()
    for stage in ("gs_project", "gs_bin_sort", "gs_render_fwd", "gs_render_bwd", "gs_project_bwd", "gs_adam_step"):
        assert stage in names


def test_library_exports_every_declared_symbol():
    from gaussian_splatting_differentiable_project_gb300 import _build
    path = _build.build()
    lib = ctypes.CDLL(path)
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    lib.gs_version.restype = ctypes.c_char_p
    assert b"sm_103a" in lib.gs_version()
    lib.gs_status_str.restype = ctypes.c_char_p
    assert lib.gs_status_str(4) == b"tile intersections exceed capacity"


def test_argument_errors_are_returned_without_a_gpu():
    """Argument checks run on the host before anything is enqueued."""
    import gaussian_splatting_differentiable_project_gb300 as gs
    lib = gs.load()
    cam = gs.camera({"R": [1, 0, 0, 0, 1, 0, 0, 0, 1], "t": [0, 0, 3], "fx": 100, "fy": 100, "cx": 64, "cy": 64,
                     "width": 128, "height": 128, "campos": [0, 0, -3]})
    # n_pad not a multiple of 256
    r = lib.gs_project(gs.dims(10, 100), ctypes.c_void_p(16), ctypes.byref(cam), gs.GsProj(16, 16, 16, 16, 16),
                       ctypes.c_void_p(16), None)
    assert r == gs.GS_ERR_INVALID_ARG
    # null params
    r = lib.gs_project(gs.dims(10, 256), None, ctypes.byref(cam), gs.GsProj(16, 16, 16, 16, 16),
                       ctypes.c_void_p(16), None)
    assert r == gs.GS_ERR_INVALID_ARG
    # zero capacity
    pc = gs.GsProj(16, 16, 16, 16, 16)
    r = lib.gs_bin_sort(gs.dims(10, 256), ctypes.byref(pc), ctypes.byref(cam), 0, gs.GsBins(16, 16, 16, 16, 16),
                        ctypes.c_void_p(256), 1 << 20, ctypes.c_void_p(16), None)
    assert r == gs.GS_ERR_INVALID_ARG
    # workspace too small
    need = lib.gs_bin_sort_workspace_bytes(gs.dims(10, 256), 1000, 128, 128)
    assert need > 0
    r = lib.gs_bin_sort(gs.dims(10, 256), ctypes.byref(pc), ctypes.byref(cam), 1000, gs.GsBins(16, 16, 16, 16, 16),
                        ctypes.c_void_p(256), need - 1, ctypes.c_void_p(16), None)
    assert r == gs.GS_ERR_INVALID_ARG
    # bad camera
    bad = gs.camera({"R": [1, 0, 0, 0, 1, 0, 0, 0, 1], "t": [0, 0, 3], "fx": 0, "fy": 100, "cx": 64, "cy": 64,
                     "width": 128, "height": 128, "campos": [0, 0, -3]})
    r = lib.gs_project(gs.dims(10, 256), ctypes.c_void_p(16), ctypes.byref(bad), gs.GsProj(16, 16, 16, 16, 16),
                       ctypes.c_void_p(16), None)
    assert r == gs.GS_ERR_INVALID_ARG
    # adam: misaligned pointer
    lr = (ctypes.c_float * 59)(*([1e-3] * 59))
    r = lib.gs_adam_step(gs.dims(10, 256), ctypes.c_void_p(20), ctypes.c_void_p(16), ctypes.c_void_p(16),
                         ctypes.c_void_p(16), lr, 0.9, 0.999, 1e-15, 1, None)
    assert r == gs.GS_ERR_INVALID_ARG
    # adam: step count 0
    r = lib.gs_adam_step(gs.dims(10, 256), ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16),
                         ctypes.c_void_p(16), lr, 0.9, 0.999, 1e-15, 0, None)
    assert r == gs.GS_ERR_INVALID_ARG
    # ssim: negative lambda, empty image, null output
    p = ctypes.c_void_p(16)
    assert lib.gs_ssim_fwd(64, 64, p, p, -0.1, p, p, None) == gs.GS_ERR_INVALID_ARG
    assert lib.gs_ssim_fwd(0, 64, p, p, 0.2, p, p, None) == gs.GS_ERR_INVALID_ARG
    assert lib.gs_ssim_bwd(64, 64, p, p, p, None, None) == gs.GS_ERR_INVALID_ARG
    # render backward: negative or non-finite L1 weight
    bins = gs.GsBins(16, 16, 16, 16, 16)
    bg = (ctypes.c_float * 3)(0, 0, 0)
    cmb = lib.gs_render_cmask_bytes(1000, 128, 128)
    # (1000 / 32 + 64 tiles + 1) chunk slots x 8 blocks x 32 pixels x 4 bytes
    assert cmb == (1000 // 32 + 64 + 1) * 8 * 32 * 4
    for w in (-1.0, float("nan"), float("inf")):
        r = lib.gs_render_bwd(gs.dims(10, 256), ctypes.byref(cam), ctypes.byref(bins), 1000, bg, p, p, p, p, p, cmb,
                              w, None, p, p, p, None)
        assert r == gs.GS_ERR_INVALID_ARG, w
    # render forward and backward: a composited-entry mask buffer too short for the view
    r = lib.gs_render_bwd(gs.dims(10, 256), ctypes.byref(cam), ctypes.byref(bins), 1000, bg, p, p, p, p, p, cmb - 4,
                          1.0, None, p, p, p, None)
    assert r == gs.GS_ERR_INVALID_ARG
    assert lib.gs_render_fwd(ctypes.byref(cam), ctypes.byref(bins), 1000, bg, p, p, p, p, cmb - 4, p, None) == \
        gs.GS_ERR_INVALID_ARG
    # spatial order: null perm, short or misaligned workspace; permutation: no planes,
    # aliasing buffers
    need = lib.gs_spatial_order_workspace_bytes(gs.dims(1000, 1024))
    assert need >= 3 * 1000 * 4
    ws = ctypes.c_void_p(256)
    assert lib.gs_spatial_order(gs.dims(1000, 1024), p, None, ws, need, p, None) == gs.GS_ERR_INVALID_ARG
    assert lib.gs_spatial_order(gs.dims(1000, 1024), p, p, ws, need - 1, p, None) == gs.GS_ERR_INVALID_ARG
    assert lib.gs_spatial_order(gs.dims(1000, 1024), p, p, ctypes.c_void_p(272), need, p, None) == \
        gs.GS_ERR_INVALID_ARG
    assert lib.gs_permute_planes(gs.dims(1000, 1024), 0, p, p, ctypes.c_void_p(32), None) == gs.GS_ERR_INVALID_ARG
    assert lib.gs_permute_planes(gs.dims(1000, 1024), 59, p, p, p, None) == gs.GS_ERR_INVALID_ARG
    # wait probes: a non-positive limit, short scratch
    nb = lib.gs_util_lookback_probe_bytes()
    assert nb > 0
    assert lib.gs_util_lookback_probe(0, p, nb, p, None) == gs.GS_ERR_INVALID_ARG
    assert lib.gs_util_lookback_probe(100, p, nb - 1, p, None) == gs.GS_ERR_INVALID_ARG
    assert lib.gs_util_mbarrier_probe(-1, p, None) == gs.GS_ERR_INVALID_ARG


def test_product_package_has_no_oracle_or_cpu_path():
    """The product package never imports the oracle and has no CPU fallback."""
    pkg = os.path.join(ROOT, "gaussian_splatting_differentiable_project_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in src and "from oracle" not in src, f
                assert "gs_oracle" not in src, f


@pytest.mark.parametrize("n", [4096, 4_000_000, 18_000_000])
def test_workspace_query_scales(n):
    import gaussian_splatting_differentiable_project_gb300 as gs
    lib = gs.load()
    pad = -(-n // 256) * 256
    a = lib.gs_bin_sort_workspace_bytes(gs.dims(n, pad), 1 << 20, 2048, 2048)
    b = lib.gs_bin_sort_workspace_bytes(gs.dims(n, pad), 1 << 24, 2048, 2048)
    assert 0 < a < b
    assert b >= (1 << 24) * 12


def test_binding_constants_match_the_header():
    import gaussian_splatting_differentiable_project_gb300 as gs
    src = open(os.path.join(ROOT, "include", "gs.h")).read()
    defs = dict(re.findall(r"#define (GS_[A-Z0-9_]+) (\d+)\b", src))
    assert int(defs["GS_N_PLANES"]) == gs.N_PLANES
    assert int(defs["GS_TILE"]) == gs.TILE
    assert int(defs["GS_REC_FLOATS"]) == gs.REC_FLOATS
    assert int(defs["GS_N_GRAD2D"]) == gs.N_GRAD2D
    assert int(defs["GS_GRAD2D_STRIDE"]) == gs.GRAD2D_STRIDE
    assert int(defs["GS_SSIM_MAPS"]) == gs.SSIM_MAPS


def test_binding_refuses_host_and_strided_tensors():
    """Every buffer crosses the boundary as a device address of a dense array: the
    binding refuses a host tensor (a kernel cannot dereference its address) and a
    strided view (it would be misread) before the library is called."""
    torch = pytest.importorskip("torch")
    import gaussian_splatting_differentiable_project_gb300 as gs
    cam = {"R": [1, 0, 0, 0, 1, 0, 0, 0, 1], "t": [0, 0, 3], "fx": 100, "fy": 100, "cx": 64, "cy": 64,
           "width": 128, "height": 128, "campos": [0, 0, -3]}
    params = torch.zeros((gs.N_PLANES, 256))
    with pytest.raises(gs.GsError, match="CUDA tensor"):
        gs.project(10, params, cam, gs.ProjBuffers(256, "cpu"), torch.zeros(1, dtype=torch.int32))
    with pytest.raises(gs.GsError, match="CUDA tensor"):
        gs.util_expf(torch.zeros(8), torch.zeros(8))
    strided = torch.zeros((4, 8)).t()

    class _OnDevice:
        """A strided view that claims to live on the device (no GPU here)."""
        is_cuda = True
        shape = strided.shape

        def is_contiguous(self):
            return strided.is_contiguous()

        def stride(self):
            return strided.stride()

    with pytest.raises(gs.GsError, match="contiguous"):
        gs._p(_OnDevice())


def test_binding_checks_buffer_types_and_sizes(monkeypatch):
    """A buffer of the wrong type or too small for the call's sizes is refused before
    the library is called (a short buffer would be overrun on the device).  Host
    tensors stand in for device ones here: the address step (whose device check the
    test above covers), the stream and the library are replaced by stubs, so nothing is
    dereferenced and nothing is launched; a call whose buffers all pass reaches the
    stub library and returns."""
    torch = pytest.importorskip("torch")
    import numpy as np
    import gaussian_splatting_differentiable_project_gb300 as gs
    W, H, n, n_pad = 64, 48, 100, 256
    cam = {"R": [1, 0, 0, 0, 1, 0, 0, 0, 1], "t": [0, 0, 3], "fx": 60, "fy": 60, "cx": 32, "cy": 24,
           "width": W, "height": H, "campos": [0, 0, -3]}
    st = torch.zeros(1, dtype=torch.int32)
    proj = gs.ProjBuffers(n_pad, "cpu")
    bins = gs.BinBuffers(n, 4096, W, H, "cpu")

    calls = []

    class _StubLib:
        def __getattr__(self, name):
            return lambda *a: calls.append(name) or 0

    monkeypatch.setattr(gs, "_p", lambda t: ctypes.c_void_p(16))
    monkeypatch.setattr(gs, "_stream", lambda stream=None: None)
    monkeypatch.setattr(gs, "load", lambda *a, **k: _StubLib())

    def refused(match, fn, *a, **k):
        before = len([c for c in calls if not c.endswith("_bytes")])
        with pytest.raises(gs.GsError, match=match):
            fn(*a, **k)
        assert len([c for c in calls if not c.endswith("_bytes")]) == before

    params = torch.zeros((gs.N_PLANES, n_pad))
    img, T, nc = torch.zeros((3, H, W)), torch.zeros((H, W)), torch.zeros((H, W), dtype=torch.int32)
    g2 = torch.zeros((n_pad, gs.GRAD2D_STRIDE))
    lr = np.full(gs.N_PLANES, 1e-3)
    i32 = lambda k: torch.zeros(k, dtype=torch.int32)  # noqa: E731

    # every buffer right: the stub library is reached
    gs.project(n, params, cam, proj, st)
    gs.render_fwd(cam, bins, (0, 0, 0), img, T, nc, st)
    gs.render_bwd(n, n_pad, cam, bins, (0, 0, 0), img, img, T, nc, g2, torch.zeros(1), st, dLdC_extra=img)
    gs.adam_step(n, params, params, params, params, lr, 0.9, 0.999, 1e-15, 1)
    gs.permute_planes(n, i32(n), params, params)
    # (size queries such as gs_render_cmask_bytes are host calls, left out of the count)
    assert [c for c in calls if not c.endswith("_bytes")] == ["gs_project", "gs_render_fwd", "gs_render_bwd",
                                                             "gs_adam_step", "gs_permute_planes"]
    u8 = torch.zeros(n, dtype=torch.uint8)
    i64 = torch.zeros(1, dtype=torch.int64)
    cfg = gs.densify_thresholds(3.0)[0]
    gs.bin_sort(n, n_pad, proj, cam, bins, st)
    gs.bin_sort_noalloc(n, n_pad, proj, cam, bins, st)
    gs.ssim_fwd(img, img, 0.2, torch.zeros((gs.SSIM_MAPS, H, W)), torch.zeros(1))
    gs.ssim_bwd(img, img, torch.zeros((gs.SSIM_MAPS, H, W)), img)
    gs.project_bwd(n, params, cam, proj, g2, params, st)
    gs.project_bwd_accumulate(n, params, cam, proj, g2, params, st)
    gs.project_bwd_adam(n, params, cam, proj, g2, params, params, lr, 0.9, 0.999, 1e-15, 1, st, grads_in=params)
    gs.project_bwd_adam_tdev(n, params, cam, proj, g2, params, params, lr, 0.9, 0.999, 1e-15, i64, st)
    gs.step_counter_add(i64, 1)
    gs.densify_accumulate(n, n_pad, proj, g2, W, H, torch.zeros(n), i32(n))
    gs.densify_plan(n, params, torch.zeros(n), i32(n), cfg, u8, i32(n), i32(1), torch.zeros(16, dtype=torch.uint8))
    gs.densify_apply(n, params, params, params, u8, i32(n), i32(1), torch.zeros((n, 6)), 0.47, params, params, params,
                     st)
    gs.opacity_reset(n, params, params, params, -4.6)
    gs.spatial_order(n, params, i32(n), torch.zeros(16, dtype=torch.uint8), st)
    gs.util_expf(torch.zeros(8), torch.zeros(8))
    gs.render_fwd_counted(cam, bins, (0, 0, 0), img, T, nc, i32(W * H), st)
    gs.batch_hyper(3, lr, 0.9, 0.999, 1e-15)
    # the calls above plus the one inside densify_thresholds
    work = [c for c in calls if not c.endswith("_bytes")]
    assert len(work) == 23 and work.count("gs_densify_thresholds") == 1

    refused("params: expected fp32", gs.project, n, params.double(), cam, proj, st)
    refused("params: needs", gs.project, n, params[:58].contiguous(), cam, proj, st)
    refused("dev_status: expected a 4-byte integer", gs.project, n, params, cam, proj, st.long())
    refused("projection buffers hold", gs.project, n, torch.zeros((gs.N_PLANES, 512)), cam, proj, st)
    refused("tiles", gs.bin_sort, n, n_pad, proj, dict(cam, width=2 * W), bins, st)
    refused("image: needs", gs.render_fwd, cam, bins, (0, 0, 0), torch.zeros((3, H, W - 1)), T, nc, st)
    refused("n_contrib: expected", gs.render_fwd, cam, bins, (0, 0, 0), img, T, nc.float(), st)
    refused("n_used: needs", gs.render_fwd_counted, cam, bins, (0, 0, 0), img, T, nc, i32(W * H - 1), st)
    refused("lr_plane", gs.batch_hyper, 2, lr[:-1], 0.9, 0.999, 1e-15)
    refused("grad2d: needs", gs.render_bwd, n, n_pad, cam, bins, (0, 0, 0), img, img, T, nc,
            torch.zeros((n_pad, gs.N_GRAD2D)), torch.zeros(1), st)
    refused("dLdC_extra: needs", gs.render_bwd, n, n_pad, cam, bins, (0, 0, 0), img, img, T, nc, g2,
            torch.zeros(1), st, dLdC_extra=torch.zeros((2, H, W)))
    refused("maps: needs", gs.ssim_fwd, img, img, 0.2, torch.zeros((gs.SSIM_MAPS - 1, H, W)), torch.zeros(1))
    refused("lr_plane", gs.adam_step, n, params, params, params, params, lr[:-1], 0.9, 0.999, 1e-15, 1)
    refused("v: needs", gs.adam_step, n, params, params, params, params[:, :128].contiguous(), lr, 0.9, 0.999,
            1e-15, 1)
    refused("t_dev: expected int64", gs.project_bwd_adam_tdev, n, params, cam, proj, g2, params, params, lr, 0.9,
            0.999, 1e-15, i32(1), st)
    refused("perm: needs", gs.permute_planes, n, i32(n - 1), params, params)
    refused("dst: expected a 4-byte", gs.permute_planes, n, i32(n), params, params.double())
    refused("randn: needs", gs.densify_apply, n, params, params, params, torch.zeros(n, dtype=torch.uint8), i32(n),
            i32(1), torch.zeros((n, 5)), 0.47, params, params, params, st)
    refused("action: expected uint8", gs.densify_plan, n, params, torch.zeros(n), i32(n),
            gs.densify_thresholds(3.0)[0], i32(n), i32(n), i32(1), torch.zeros(16, dtype=torch.uint8))


@pytest.mark.parametrize("fused,dssim", [(True, 0.0), (False, 0.2)])
def test_trainer_buffers_pass_the_binding_checks(monkeypatch, fused, dssim):
    """Every call the trainer makes (steps, batch steps, density control, storage order)
    hands the binding buffers of the right type and size: run against the stub library
    of the test above, on host tensors."""
    torch = pytest.importorskip("torch")
    import numpy as np
    import gaussian_splatting_differentiable_project_gb300 as gs
    W, H, n, n_pad = 64, 48, 300, 512
    cam = {"R": [1, 0, 0, 0, 1, 0, 0, 0, 1], "t": [0, 0, 3], "fx": 60, "fy": 60, "cx": 32, "cy": 24,
           "width": W, "height": H, "campos": [0, 0, -3]}
    tr = gs.Trainer(np.zeros((gs.N_PLANES, n_pad), np.float32), n, W, H, capacity=4096,
                    lr_plane=np.full(gs.N_PLANES, 1e-3), device="cpu", fused=fused, dssim=dssim)
    calls = []

    class _StubLib:
        def __getattr__(self, name):
            return lambda *a: calls.append(name) or 0

    monkeypatch.setattr(gs, "_p", lambda t: ctypes.c_void_p(16))
    monkeypatch.setattr(gs, "_stream", lambda stream=None: None)
    monkeypatch.setattr(gs, "load", lambda *a, **k: _StubLib())
    target = torch.zeros((3, H, W))
    tr.step(cam, target)
    tr.step_batch([cam, cam, cam], [target] * 3)
    tr.enable_density_control(3.0)
    tr.step(cam, target)
    tr.reorder_spatially()
    tr.reset_opacity()
    stats = tr.refine(randn=torch.zeros((n, 6)))
    assert stats["n"] == 0 and tr.n_pad == 256
    assert "gs_render_bwd" in calls and "gs_densify_apply" in calls and "gs_permute_planes" in calls
    assert ("gs_project_bwd_adam" in calls) == fused and ("gs_ssim_fwd" in calls) == (dssim > 0)


def test_size_and_camera_limits_are_refused_on_the_host():
    """Sizes past the layout's limits and non-finite cameras are refused before
    anything is enqueued: n outside [0, n_pad], n_pad above 2^31, images wider than
    65,535 tiles, non-finite rotation or near plane; null or misaligned raster
    buffers; a density destination whose stride is not a multiple of 256."""
    import gaussian_splatting_differentiable_project_gb300 as gs
    lib = gs.load()
    p = ctypes.c_void_p(16)

    def cam(**kw):
        d = {"R": [1, 0, 0, 0, 1, 0, 0, 0, 1], "t": [0, 0, 3], "fx": 100, "fy": 100, "cx": 64, "cy": 64,
             "width": 128, "height": 128, "campos": [0, 0, -3]}
        d.update(kw)
        return gs.camera(d)

    c = cam()
    pc = gs.GsProj(16, 16, 16, 16, 16)
    bad = gs.GS_ERR_INVALID_ARG
    assert lib.gs_project(gs.dims(300, 256), p, ctypes.byref(c), pc, p, None) == bad
    assert lib.gs_project(gs.dims(-1, 256), p, ctypes.byref(c), pc, p, None) == bad
    assert lib.gs_project(gs.dims(10, (1 << 31) + 256), p, ctypes.byref(c), pc, p, None) == bad
    assert lib.gs_project(gs.dims(10, 256), p, ctypes.byref(cam(width=65535 * 16 + 1)), pc, p, None) == bad
    assert lib.gs_project(gs.dims(10, 256), p, ctypes.byref(cam(R=[float("nan")] + [0] * 8)), pc, p, None) == bad
    assert lib.gs_project(gs.dims(10, 256), p, ctypes.byref(cam(near_z=float("inf"))), pc, p, None) == bad
    bg = (ctypes.c_float * 3)(0, 0, 0)
    bins = gs.GsBins(16, 16, 16, 16, 16)
    cmb = lib.gs_render_cmask_bytes(1000, 128, 128)
    assert lib.gs_render_fwd(ctypes.byref(c), ctypes.byref(bins), 1000, bg, None, p, p, p, cmb, p, None) == bad
    misaligned = gs.GsBins(16, 16, 20, 16, 16)
    assert lib.gs_render_fwd(ctypes.byref(c), ctypes.byref(misaligned), 1000, bg, p, p, p, p, cmb, p, None) == bad
    assert lib.gs_render_fwd(ctypes.byref(c), ctypes.byref(bins), 1000, bg, p, p, p, None, cmb, p, None) == bad
    assert lib.gs_densify_apply(gs.dims(10, 256), 100, p, p, p, p, p, p, p, 0.47, p, p, p, p, None) == bad
    assert lib.gs_opacity_reset(gs.dims(10, 256), p, None, p, -4.0, None) == bad
