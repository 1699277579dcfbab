"""Parity metrics and the tolerance gate used by every GPU-vs-oracle test.

Per tensor, with o the fp64 oracle and g the GPU result:
  max_rel  = max|g - o| / max|o|        gate: <= 2e-2
  mean_rel = mean|g - o| / max|o|       gate: <= 2e-3
  norm_rel = sum|g - o| / sum|o|        reported (bf16 rounding floor 2e-3..1e-2)
The gate values are the stated tolerance (max relative error 2e-2, mean
relative error 2e-3 for bf16 operands with fp32 accumulation); the error is
taken relative to the tensor's scale, max|o|, because an element-wise
relative error is unbounded where o crosses zero.
"""
import numpy as np

MAX_REL_TOL = 2e-2
MEAN_REL_TOL = 2e-3


def metrics(g, o):
    g = np.asarray(g, dtype=np.float64)
    o = np.asarray(o, dtype=np.float64)
    assert g.shape == o.shape, (g.shape, o.shape)
    scale = float(np.abs(o).max())
    if scale == 0.0:
        scale = 1.0
    e = np.abs(g - o)
    denom = float(np.abs(o).sum()) or 1.0
    return {
        "max_rel": float(e.max()) / scale if e.size else 0.0,
        "mean_rel": float(e.mean()) / scale if e.size else 0.0,
        "norm_rel": float(e.sum()) / denom,
        "finite": bool(np.isfinite(g).all()),
    }


def assert_close(name, g, o, max_tol=MAX_REL_TOL, mean_tol=MEAN_REL_TOL):
    m = metrics(g, o)
    assert m["finite"], f"{name}: non-finite values"
    assert m["max_rel"] <= max_tol and m["mean_rel"] <= mean_tol, f"{name}: {m}"
    return m
