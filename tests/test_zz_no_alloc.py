"""gs_bin_sort_noalloc: the binning entry point for callers that may not allocate
device memory.

Some callers cannot call cudaMalloc: code that runs where allocation is forbidden or
would stall (a real-time loop whose memory is all reserved at start-up, an embedding
application whose own allocator owns the GPU).  This entry point takes
its sort scratch from a fixed array inside the library instead of a caller-provided
workspace.  Its results must equal gs_bin_sort's bit for bit (sort keys, ids, tile
ranges and gathered records are integer/index work), on consecutive calls that reuse
the array with different sizes, and sizes beyond its fixed limits must be refused
before anything is enqueued.

This file is collected last so that a run stopping at the first failure has already
run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest

import gs_inputs as gi

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import gaussian_splatting_differentiable_project_gb300 as gs  # noqa: E402

DEV = "cuda"


def _both(P, n, cam, capacity):
    """Project once, then bin with the workspace entry point and with the
    fixed-scratch one into separate output buffers."""
    W, H = cam["width"], cam["height"]
    n_pad = P.shape[1]
    params = torch.from_numpy(P).to(DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    proj = gs.ProjBuffers(n_pad, DEV)
    gs.project(n, params, cam, proj, st)
    ref = gs.BinBuffers(n, capacity, W, H, DEV)
    gs.bin_sort(n, n_pad, proj, cam, ref, st)
    out = gs.BinBuffers(n, capacity, W, H, DEV)
    # poison the outputs so that stale or missing writes show
    out.keys.fill_(-1)
    out.ids.fill_(-1)
    out.rec.fill_(float("nan"))
    out.ranges.fill_(-1)
    st2 = torch.zeros(1, dtype=torch.int32, device=DEV)
    # through the C ABI directly
    lib = gs.load()
    cc = gs.camera(cam)
    pc = proj.c()
    r = lib.gs_bin_sort_noalloc(gs.dims(n, n_pad), ctypes.byref(pc), ctypes.byref(cc), capacity, out.c(),
                                ctypes.c_void_p(st2.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert r == gs.GS_OK, gs.status_str(r)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and int(st2.item()) == 0
    K = int(ref.n_isect[0].item())
    assert K > 0 and int(out.n_isect[0].item()) == K
    assert torch.equal(out.keys[:K], ref.keys[:K])
    assert torch.equal(out.ids[:K], ref.ids[:K])
    assert torch.equal(out.ranges, ref.ranges)
    assert np.array_equal(out.rec[:K].cpu().numpy().view(np.uint32), ref.rec[:K].cpu().numpy().view(np.uint32))
    return K


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    """Two calls in a row with different scenes and image sizes: the second must not
    see anything the first left in the shared array."""
    cfg = gi.CONFIGS["tiny"]
    P1 = gi.scene_for(cfg)
    K1 = _both(P1, cfg.n, gi.camera((0.0, 0.0, 3.0), 128, 128), capacity=1 << 16)
    P2 = gi.scene_for(cfg, seed=5, n=3000)
    K2 = _both(P2, 3000, gi.camera((0.4, -0.2, 2.8), 72, 56), capacity=1 << 15)
    assert K1 != K2


def test_noalloc_refuses_sizes_beyond_its_scratch():
    """Sizes above the fixed limits are refused with GS_ERR_SCRATCH_LIMIT on the host."""
    lib = gs.load()
    cfg = gi.CONFIGS["tiny"]
    cam = gs.camera(gi.camera((0.0, 0.0, 3.0), 128, 128))
    proj = gs.ProjBuffers(4096, DEV)
    bins = gs.BinBuffers(4096, 1024, 128, 128, DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    pc = proj.c()
    too_many_isect = (1 << 20) + 1
    r = lib.gs_bin_sort_noalloc(gs.dims(cfg.n, 4096), ctypes.byref(pc), ctypes.byref(cam), too_many_isect,
                                bins.c(), ctypes.c_void_p(st.data_ptr()), None)
    assert r == gs.GS_ERR_SCRATCH_LIMIT
    assert "scratch" in gs.status_str(r)
    big = gs.camera(gi.camera((0.0, 0.0, 3.0), 8192, 8192))  # 262,144 tiles
    r = lib.gs_bin_sort_noalloc(gs.dims(cfg.n, 4096), ctypes.byref(pc), ctypes.byref(big), 1024, bins.c(),
                                ctypes.c_void_p(st.data_ptr()), None)
    assert r == gs.GS_ERR_SCRATCH_LIMIT
