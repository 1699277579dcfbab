"""8-bit floating point (E4M3 and E5M2) for the FP8 GEMM path.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

The Megatron-Core listing (混合精度: FP8 and FP4 training on Blackwell
Ultra; its --fp8-format hybrid flag, E4M3 forward and E5M2 for gradients)
names the formats but gives no scaling recipe.  The formats are the OCP 8-bit
floating-point ones:
  E4M3: 1 sign, 4 exponent bits (bias 7), 3 mantissa bits; no infinity; the
        largest finite value 1.75 * 2^8 = 448; subnormal quantum 2^-9.
  E5M2: 1 sign, 5 exponent bits (bias 15), 2 mantissa bits; the largest
        finite value 1.75 * 2^15 = 57344; subnormal quantum 2^-16.
Reading taken for the scaling (the plainest one, per-tensor "current"
scaling): amax = max |x| in float32, scale = fmax / amax computed in float32
(1 when amax is 0), q = RNE_fp8(float32(x) * scale) saturated to +-fmax, and
scale_inv = 1 / scale is what a GEMM multiplies its fp32 accumulator by.
Everything below is float64 arithmetic on values that the formats represent
exactly, except the two float32 steps that the reading fixes.
"""
from __future__ import annotations

import numpy as np

FORMATS = {
    # name: (mantissa bits, exponent bias, largest finite value)
    "e4m3": (3, 7, 448.0),
    "e5m2": (2, 15, 57344.0),
}


def round_fp8(x: np.ndarray, fmt: str) -> np.ndarray:
    """Round float64 values to the nearest representable value (ties to even
    mantissa), saturating at +-fmax.  Returns float64."""
    m, bias, fmax = FORMATS[fmt]
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    emin = 1 - bias
    # exponent of the binade holding |x| (subnormals use the quantum of emin)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    e = np.maximum(ex - 1, emin)
    quantum = np.ldexp(1.0, e - m)
    r = np.round(a / quantum) * quantum  # np.round: half to even
    r = np.minimum(r, fmax)
    return np.copysign(r, x)


def encode(v: np.ndarray, fmt: str) -> np.ndarray:
    """Byte patterns of values already representable in the format."""
    m, bias, _ = FORMATS[fmt]
    v = np.asarray(v, dtype=np.float64)
    sign = (np.signbit(v)).astype(np.uint8) << 7
    a = np.abs(v)
    emin = 1 - bias
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    e = ex - 1
    normal = (a > 0) & (e >= emin)
    E = np.where(normal, e + bias, 0)
    M = np.where(normal, (a / np.ldexp(1.0, e) - 1.0) * (1 << m), a / np.ldexp(1.0, emin - m))
    assert np.all(M == np.round(M)), "value not representable"
    return (sign | (E.astype(np.uint8) << m) | M.astype(np.uint8)).astype(np.uint8)


def decode(b: np.ndarray, fmt: str) -> np.ndarray:
    """Values of byte patterns (NaN encodings are not produced here)."""
    m, bias, _ = FORMATS[fmt]
    b = np.asarray(b, dtype=np.uint8).astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    E = (b >> m) & ((1 << (7 - m)) - 1)
    M = b & ((1 << m) - 1)
    val = np.where(E > 0, np.ldexp(1.0 + M / (1 << m), E - bias), np.ldexp(M.astype(np.float64), 1 - bias - m))
    return sign * val


def quantize(x: np.ndarray, fmt: str):
    """Per-tensor current scaling (module docstring): returns
    (bytes uint8, scale_inv float32)."""
    _, _, fmax = FORMATS[fmt]
    x32 = np.asarray(x, dtype=np.float32)
    amax = np.float32(np.max(np.abs(x32))) if x32.size else np.float32(0)
    scale = np.float32(fmax) / amax if amax > 0 else np.float32(1.0)
    y = (x32 * scale).astype(np.float32)  # float32 product, as the reading fixes
    q = encode(round_fp8(y.astype(np.float64), fmt), fmt)
    return q, np.float32(1.0) / scale


def gemm_fp8(a_bytes, a_fmt, a_scale_inv, b_bytes, b_fmt, b_scale_inv):
    """C[M, N] = (A B^T) * a_scale_inv * b_scale_inv with A [M, K], B [N, K]
    given as byte patterns: the exact product of the decoded values (one
    matrix product, float64)."""
    A = decode(a_bytes, a_fmt)
    B = decode(b_bytes, b_fmt)
    return (A @ B.T) * (float(a_scale_inv) * float(b_scale_inv))
