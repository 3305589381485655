"""The bench's roofline model (CPU): the algorithmic bytes of each stage follow from the
data layout the C ABI declares, the tile sort's pass count from the tile-id width, and
the FP32 peak from the SM count, lanes and clock.  Each byte coefficient is rebuilt here
from the layout's sizes (planes, record, grad2d slot), one unit count at a time."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

F = 4                      # bytes of an fp32 or 32-bit integer value
PLANES = 59                # parameter planes: mean 3, log-scale 3, quaternion 4, opacity 1, SH 48
GEOM = 3 + 3 + 4 + 1       # planes every Gaussian's projection reads
SH = PLANES - GEOM
REC = 12 * F               # projected record
GRAD2D = 12 * F            # interleaved 2D-gradient slot


def _coef(fn, unit, **kw):
    """The coefficient of one unit count in a linear byte model."""
    args = dict(N=0, n_pad=0, V=0, K=0, P=0, E=0)
    args.update(kw)
    base = fn(**args)
    args[unit] = 1
    one = fn(**args)
    return {k: one[k] - base[k] for k in one}


def _stage(**kw):
    return bench.stage_bytes(kw["N"], kw["n_pad"], kw["V"], kw["K"], kw["P"], kw.get("passes", 2),
                             dssim=kw.get("dssim", False), E=kw.get("E", 0))


def test_layout_constants_match_the_binding():
    import gaussian_splatting_differentiable_project_gb300 as gs
    assert gs.N_PLANES == PLANES and gs.REC_FLOATS * F == REC and gs.GRAD2D_STRIDE * F == GRAD2D


def test_projection_bytes():
    # every Gaussian: its geometric planes read; depth, radius, 2-int rect and count written
    assert _coef(_stage, "N")["project"] == GEOM * F + F + F + 2 * F + F
    # every visible Gaussian: its SH planes read and its record written
    assert _coef(_stage, "V")["project"] == SH * F + REC


def test_render_bytes():
    n = _coef(_stage, "n_pad")
    k = _coef(_stage, "K")
    p = _coef(_stage, "P")
    e = _coef(_stage, "E")
    # forward: each intersection's record read once; image (3), T and n_contrib
    # written; a 4-byte mask per pixel and 32 iterated entries written
    assert k["render_fwd"] == REC and p["render_fwd"] == (3 + 1 + 1) * F and e["render_fwd"] == F / 32
    # backward: the grad2d slots cleared, records read once; image and target (3 each),
    # T and n_contrib read; the masks read
    assert n["render_bwd"] == GRAD2D and k["render_bwd"] == REC and e["render_bwd"] == F / 32
    assert p["render_bwd"] == (3 + 3 + 1 + 1) * F
    # with D-SSIM the backward also reads its 3-plane image gradient
    assert _coef(lambda **a: _stage(dssim=True, **a), "P")["render_bwd"] == (3 + 3 + 1 + 1 + 3) * F


def test_projection_backward_and_adam_bytes():
    assert _coef(_stage, "N")["project_bwd"] == F + PLANES * F          # count read, gradients written
    assert _coef(_stage, "V")["project_bwd"] == PLANES * F + GRAD2D     # parameters and grad2d read
    # Adam: p, g, m, v read and p, m, v written, per parameter
    assert _coef(_stage, "n_pad")["adam"] == PLANES * 7 * F
    # fused: the same minus the gradient planes (never written, never read back)
    fused = lambda **a: {"f": bench.fused_bytes(a["N"], a["n_pad"], a["V"])}  # noqa: E731
    assert _coef(fused, "n_pad")["f"] == PLANES * 6 * F
    assert _coef(fused, "V")["f"] == GRAD2D and _coef(fused, "N")["f"] == F


def test_binning_bytes_grow_with_sort_passes():
    a = _coef(lambda **kw: _stage(passes=1, **kw), "K")["bin_sort"]
    b = _coef(lambda **kw: _stage(passes=2, **kw), "K")["bin_sort"]
    # each tile pass reads and writes an 8-byte (key, index) pair per intersection
    assert b - a == 2 * 2 * F
    # one intersection at least: its (tile, index) pair emitted, its 48-byte record
    # gathered and written, its 64-bit key written
    assert a >= 2 * F + 2 * REC + 8


@pytest.mark.parametrize("wh,passes", [((128, 128), 1), ((256, 256), 1), ((257, 256), 2), ((512, 512), 2),
                                       ((2048, 2048), 2), ((8192, 8192), 3)])
def test_tile_sort_passes(wh, passes):
    """ceil(tile-id bits / 8) over 16x16 tiles: 64 tiles take 6 bits, 16,384 take 14."""
    assert bench.passes_for(*wh) == passes


def test_fp32_peak():
    # SMs (queried at run time) x 128 FP32 lanes x 2 FLOP per FMA x the SM clock:
    # 152 SMs at 2070 MHz give 80.5 TFLOP/s
    assert bench.fp32_peak_tflops(2070, 152) == pytest.approx(80.54784)
    assert bench.fp32_peak_tflops(2070, 160) == pytest.approx(80.54784 * 160 / 152)


def test_composited_flop_model():
    """The second work figure: composited pairs the full per-pair count, the other
    iterated pairs their evaluation up to the 1/255 test (17 operations: offset 2,
    power 9, skip test 1, log2(e) 1, exponential 1, opacity product 1, clamp 1, the
    1/255 test 1)."""
    assert bench.FLOP_SKIP_PAIR == 2 + 9 + 1 + 1 + 1 + 1 + 1 + 1
    assert bench.composited_flops(27, 100.0, 100.0) == 2700.0
    assert bench.composited_flops(66, 100.0, 40.0) == 66 * 40 + 17 * 60
    # every iterated pair costs at least its evaluation
    assert bench.composited_flops(66, 100.0, 0.0) == 1700.0
