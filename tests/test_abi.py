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
    for w in (-1.0, float("nan"), float("inf")):
        r = lib.gs_render_bwd(gs.dims(10, 256), ctypes.byref(cam), ctypes.byref(bins), 1000, bg, p, p, p, p, w, None,
                              p, p, p, None)
        assert r == gs.GS_ERR_INVALID_ARG, w
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
