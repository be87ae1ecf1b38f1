"""Comparison helpers for the GPU parity tests (no arithmetic of the method).

Tolerances: bf16 outputs |gpu - ref| <= 2e-2 + 2e-2 |ref| element-wise (the
allclose reading of "abs 2e-2 / rel 2e-2"), plus a scale-aware bound
max|gpu - ref| / max|ref| <= 2e-2 so that outputs far smaller than 2e-2
(long contexts) are still pinned; f32 LSE |gpu - ref| <= 1e-3 with -inf
matching -inf exactly; byte / index work bit-exact.
"""

import numpy as np
import torch

ATOL = 2e-2
RTOL = 2e-2
SCALE_TOL = 2e-2
LSE_ATOL = 1e-3


def to_f64(t: torch.Tensor) -> np.ndarray:
    # Unused split slots hold unspecified bits (possibly signalling NaNs,
    # which raise numpy's "invalid" flag on some hosts); callers mask them.
    with np.errstate(invalid="ignore"):
        return t.detach().float().cpu().numpy().astype(np.float64)


def assert_bf16_close(gpu, ref, what="", mask=None):
    g = to_f64(gpu) if isinstance(gpu, torch.Tensor) else np.asarray(gpu, np.float64)
    r = np.asarray(ref, np.float64)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    if mask is not None:
        g, r = g[mask], r[mask]
    assert np.isfinite(r).all(), what + ": reference has non-finite values"
    assert np.isfinite(g).all(), what + ": GPU result has non-finite values"
    err = np.abs(g - r)
    bad = err > ATOL + RTOL * np.abs(r)
    assert not bad.any(), "%s: %d elements outside abs/rel 2e-2 (max err %.3g)" % (what, bad.sum(), err.max())
    ref_max = np.abs(r).max() if r.size else 0.0
    if ref_max > 0:
        rel = err.max() / ref_max
        assert rel <= SCALE_TOL, "%s: max|err|/max|ref| = %.3g" % (what, rel)
    return float(err.max()) if err.size else 0.0


def assert_lse_close(gpu, ref, what="", mask=None):
    g = to_f64(gpu) if isinstance(gpu, torch.Tensor) else np.asarray(gpu, np.float64)
    r = np.asarray(ref, np.float64)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    if mask is not None:
        g, r = g[mask], r[mask]
    ninf = np.isneginf(r)
    assert np.array_equal(np.isneginf(g), ninf), what + ": -inf pattern differs"
    fin = ~ninf
    assert np.isfinite(g[fin]).all(), what + ": non-finite GPU LSE"
    err = np.abs(g[fin] - r[fin])
    assert (err <= LSE_ATOL).all(), "%s: LSE max err %.3g" % (what, err.max())
    return float(err.max()) if err.size else 0.0
