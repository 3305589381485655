"""The layout of gs_render_bwd's grad2d as the header defines it, for the tests: its
slots 0-4 hold the moments S1..S5 of q = dL/dpower over the pixel offset, and the
mean2d and conic partials follow from them with the Gaussian's conic (A, B, C), where
power = -(A dx^2 + C dy^2)/2 - B dx dy:
    dL/dmx = A S1 + B S2,  dL/dmy = B S1 + C S2,  dL/dA = -S3/2,  dL/dB = -S4,
    dL/dC = -S5/2.
Slots 5-8 (opacity, colour) are partials already."""
import numpy as np


def moments_to_partials(planes, conic):
    """(9, n) sums in grad2d's layout -> (9, n) partials (fp64).  conic: (n, 3) (A, B, C)."""
    S = np.asarray(planes, np.float64)
    conic = np.asarray(conic, np.float64)
    conic = np.where(np.isfinite(conic), conic, 0.0)  # culled Gaussians: their sums are 0
    A, B, C = (conic[:, k] for k in range(3))
    out = S.copy()
    out[0] = A * S[0] + B * S[1]
    out[1] = B * S[0] + C * S[1]
    out[2] = -0.5 * S[2]
    out[3] = -S[3]
    out[4] = -0.5 * S[4]
    return out
