"""Tolerance checks shared by the GPU parity tests.

The bar for FP16 outputs of quant_gemm (floating point; the GPU accumulates in
FP32 in its own order, the oracle in binary64 in k order):
  * relative L2 error over all outputs  <= 2e-3
  * per output row m: max_n |gpu - ref| <= 1e-2 * max_n |ref[m, n]|
Integer work (packed words, unpacked codes) is compared bit for bit.
"""
import numpy as np

REL_L2 = 2e-3
ROW_MAX_FRAC = 1e-2


def rel_l2(got, ref) -> float:
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(r.ravel())
    return float(np.linalg.norm((g - r).ravel()) / (den if den > 0 else 1.0))


def assert_close(got, ref, what=""):
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.all(np.isfinite(g)), "%s: non-finite output" % what
    e = rel_l2(g, r)
    assert e <= REL_L2, "%s: rel-L2 %.3e > %.1e" % (what, e, REL_L2)
    if g.ndim == 1:
        g, r = g[None], r[None]
    rowmax = np.max(np.abs(r), axis=1)
    err = np.max(np.abs(g - r), axis=1)
    bad = err > ROW_MAX_FRAC * rowmax
    assert not np.any(bad), "%s: rows %s exceed the per-row bound (err %s, row max %s)" % (
        what, np.nonzero(bad)[0][:5], err[bad][:5], rowmax[bad][:5])
    return e


def assert_points_close(got, ref, what=""):
    """Sampled outputs of a full-size case: the same relative-L2 bound over
    the sample, and every sampled value within 1e-2 of the sample's max."""
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(g)), "%s: non-finite output" % what
    e = rel_l2(g, r)
    assert e <= REL_L2, "%s: rel-L2 %.3e > %.1e" % (what, e, REL_L2)
    assert np.max(np.abs(g - r)) <= ROW_MAX_FRAC * np.max(np.abs(r)), what
    return e
