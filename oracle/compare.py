"""Parity check of a GPU result against the fp64 oracle (test infrastructure).

Tolerance (fixed for this hot path): with s = sqrt(K) * max|A| * max|B|,
  fp32 output:  max |gpu - oracle| / s <= 1e-3
  bf16 output:  |gpu - oracle| <= 1e-3 * s + ulp_bf16(|oracle|)  per element,
where ulp_bf16(x) = 2^(floor(log2 x) - 7) (2^-133 at 0).  For IKBO, K is
Du + Dc, max|A| = max|W| and max|B| = max over U and Cf.  With a bias and /
or SiLU epilogue the same bound applies to the final output (SiLU's slope is
at most ~1.1 and the bias add is exact in fp64).
"""
from __future__ import annotations

import math

import numpy as np


def ulp_bf16(x: np.ndarray) -> np.ndarray:
    ax = np.abs(np.asarray(x, dtype=np.float64))
    out = np.full(ax.shape, 2.0 ** -133)
    nz = ax > 0
    out[nz] = np.exp2(np.floor(np.log2(ax[nz])) - 7)
    return out


def scale(K: int, amax: float, bmax: float) -> float:
    return math.sqrt(K) * float(amax) * float(bmax)


def check(gpu, ref, K: int, amax: float, bmax: float, out_bf16: bool, mask=None):
    """Return (ok, worst_metric, detail).  worst_metric is max|err| / s."""
    g = np.asarray(gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    if mask is not None:
        g = g[mask]
        r = r[mask]
    if g.shape != r.shape:
        return False, float("inf"), "shape %s vs %s" % (g.shape, r.shape)
    if g.size == 0:
        return True, 0.0, "empty"
    if not np.isfinite(g).all():
        bad = np.argwhere(~np.isfinite(g))[:5]
        return False, float("inf"), "non-finite GPU values at %s" % bad.tolist()
    s = scale(K, amax, bmax)
    if s == 0.0:
        s = 1.0
    err = np.abs(g - r)
    metric = float(err.max() / s)
    if out_bf16:
        bound = 1e-3 * s + ulp_bf16(r)
        viol = err > bound
        ok = not viol.any()
        detail = "metric %.3e; %d elements above bound" % (metric, int(viol.sum()))
        if not ok:
            idx = np.unravel_index(np.argmax(err - bound), err.shape)
            detail += "; worst at %s: gpu %r oracle %r" % (tuple(int(i) for i in idx),
                                                          float(g[idx]), float(r[idx]))
    else:
        ok = metric <= 1e-3
        detail = "metric %.3e" % metric
        if not ok:
            idx = np.unravel_index(np.argmax(err), err.shape)
            detail += "; worst at %s: gpu %r oracle %r" % (tuple(int(i) for i in idx),
                                                          float(g[idx]), float(r[idx]))
    return ok, metric, detail
