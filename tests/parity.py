"""Tolerance checks shared by the GPU parity tests.

The bar for FP16 outputs of quant_gemm (floating point; the GPU accumulates in
FP32 in its own order, the oracle in binary64 in k order):
  * relative L2 error over all outputs  <= 2e-3
  * per output row m: max_n |gpu - ref| <= 1e-2 * max_n |ref[m, n]|
Integer work (packed words, unpacked codes) is compared bit for bit.
Full-size cases are checked on whole sampled rows (the oracle evaluates only
those rows; rows of the output are independent), so the per-row bound is
applied exactly as stated, against each row's own maximum.
"""
import numpy as np

REL_L2 = 2e-3
ROW_MAX_FRAC = 1e-2


def rel_l2(got, ref) -> float:
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(r.ravel())
    return float(np.linalg.norm((g - r).ravel()) / (den if den > 0 else 1.0))


def trajectory_scale(L):
    """Factor on both bars for x_L of a loop block compared from the same x0
    (not iteration by iteration): sqrt(L).  Every iteration is held to the
    unscaled bars on its own inputs (the GPU tests check that iteration by
    iteration); a trajectory from x0 carries one such independent difference
    per iteration on, so the bars grow like a random walk.  Measured on the
    CPU: independent binary32 restatements of the blocks (exact weights as
    the decode kernel; FP16-rounded weights as the tensor-core kernel) drift
    from the oracle by about 9e-4 * sqrt(L) for the SwiGLU block and stay
    inside this bar at L = 1 .. 16
    (tests/test_oracle.py::test_loop_block_fp32_drift_within_trajectory_bar)."""
    return max(1.0, float(L) ** 0.5)


def assert_close(got, ref, what="", scale=1.0):
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.all(np.isfinite(g)), "%s: non-finite output" % what
    e = rel_l2(g, r)
    assert e <= REL_L2 * scale, "%s: rel-L2 %.3e > %.1e" % (what, e, REL_L2 * scale)
    if g.ndim == 1:
        g, r = g[None], r[None]
    rowmax = np.max(np.abs(r), axis=1)
    err = np.max(np.abs(g - r), axis=1)
    bad = err > ROW_MAX_FRAC * scale * rowmax
    assert not np.any(bad), "%s: rows %s exceed the per-row bound (err %s, row max %s)" % (
        what, np.nonzero(bad)[0][:5], err[bad][:5], rowmax[bad][:5])
    return e


def sample_rows(M, count, rng):
    """Up to `count` distinct row indices of an M-row output, sorted; all
    rows when M <= count."""
    if M <= count:
        return np.arange(M)
    return np.sort(rng.choice(M, count, replace=False))
