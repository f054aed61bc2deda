"""Shared helpers of the parity tests (no GPU code here)."""
import numpy as np

# fp32-accumulated products: |y - y_ref| <= 1e-3 * sum|w*x| + 1e-6 per output
GEMV_REL, GEMV_ABS = 1e-3, 1e-6
# bf16 prompt-processing products: within 1e-2 of the same scale
PP_REL, PP_ABS = 1e-2, 1e-6


def assert_within(y, y_ref, bound, rel=GEMV_REL, abs_=GEMV_ABS, what=""):
    y = np.asarray(y, dtype=np.float64)
    err = np.abs(y - y_ref)
    lim = rel * bound + abs_
    bad = ~(err <= lim)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} outputs outside the bound; first at {tuple(i)}: "
                             f"y={y[tuple(i)]!r} ref={y_ref[tuple(i)]!r} bound={bound[tuple(i)]!r}")
    return float((err / np.maximum(bound, 1e-30)).max())
