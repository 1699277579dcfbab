"""Parity metrics and the tolerance gate used by every GPU-vs-oracle test.

Per tensor, with o the fp64 oracle and g the GPU result:
  max_rel  = max|g - o| / max|o|        gate: <= 2e-2
  mean_rel = mean|g - o| / max|o|       gate: <= 2e-3
  norm_rel = sum|g - o| / sum|o|        reported (bf16 rounding floor 2e-3..1e-2)
The gate values are the stated tolerance (max relative error 2e-2, mean
relative error 2e-3 for bf16 operands with fp32 accumulation); the error is
taken relative to the tensor's scale, max|o|, because an element-wise
relative error is unbounded where o crosses zero.

A second, binding bound anchors each tensor on the bf16 rounding floor: the
oracle re-run with bf16 rounding at exactly the GEMM operands of the CUDA path
(oracle/rounding_floor.py, pinned in tests/test_rounding_floor.py) has, on
the same inputs, a norm-wise error F per tensor; the GPU result must have
  norm_rel <= 1.5 F + 2**-16
The factor leaves room for the GPU's roundings falling on slightly different
values than the floor's (same sites, same distribution); 2**-16 covers the
fp32 accumulation and storage that the floor, in float64, does not have
(sqrt(K) 2**-24 for sums of up to K = 2**15 terms).  Both bounds were fixed
before their first GPU run.
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


FLOOR_FACTOR = 1.5
FLOOR_ALLOWANCE = 2.0 ** -16


def floor_bound(floor_norm_rel):
    return FLOOR_FACTOR * floor_norm_rel + FLOOR_ALLOWANCE


def assert_within_floor(name, g, o, floor_norm_rel):
    """The binding floor-anchored bound (norm-wise, see the module docstring)."""
    m = metrics(g, o)
    bound = floor_bound(floor_norm_rel)
    assert m["finite"], f"{name}: non-finite values"
    assert m["norm_rel"] <= bound, f"{name}: norm_rel {m['norm_rel']:.3e} > {bound:.3e} " \
        f"(1.5 x bf16 floor {floor_norm_rel:.3e} + 2^-16)"
    return m


def assert_close(name, g, o, max_tol=MAX_REL_TOL, mean_tol=MEAN_REL_TOL):
    m = metrics(g, o)
    assert m["finite"], f"{name}: non-finite values"
    assert m["max_rel"] <= max_tol and m["mean_rel"] <= mean_tol, f"{name}: {m}"
    return m
