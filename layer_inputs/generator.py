"""Counter-based generator for the layer's synthetic inputs.

Recipe (the same for every consumer):

* ``splitmix64`` (Steele, Lea & Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014) evaluated at counters ``base + i`` for i = 0, 1, ...,
  where ``base`` mixes (seed, stream, tensor id).  Stream = layer index in a
  stack; tensor ids are fixed below so every tensor has its own sequence.
* Uniform in (0, 1]: ``((z >> 11) + 1) * 2**-53``.
* Box-Muller on consecutive pairs (u1, u2): ``r = sqrt(-2 ln u1)``,
  ``n0 = r cos(2 pi u2)``, ``n1 = r sin(2 pi u2)``.
* Scale to N(mean, std**2) in float64, round to float32 (nearest-even), then to
  bfloat16 (nearest-even).  The bfloat16 value is *the* input: both the oracle
  (as exact float64) and the GPU (as bf16 or exact fp32) consume that value.

Nothing here computes any part of the transformer layer.
"""
from __future__ import annotations

import concurrent.futures
import dataclasses
import os
from typing import Dict, Optional

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# Draw order / tensor ids of one layer's parameters (fixed so that each tensor
# has its own counter stream regardless of the shape of the others).
PARAM_NAMES = (
    "ln1_g", "ln1_b", "w_qkv", "b_qkv", "w_o", "b_o",
    "ln2_g", "ln2_b", "w_fc1", "b_fc1", "w_fc2", "b_fc2",
)
_TENSOR_ID = {"x": 1, "dy": 2}
_TENSOR_ID.update({n: 16 + i for i, n in enumerate(PARAM_NAMES)})

_CHUNK = 1 << 22


def splitmix64(counters: np.ndarray) -> np.ndarray:
    """splitmix64 output for an array of uint64 counters (wrapping arithmetic)."""
    with np.errstate(over="ignore"):
        z = counters * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def _stream_base(seed: int, stream: int, tensor_id: int) -> np.uint64:
    key = np.array([(seed & 0xFFFFFFFF) << 32 | (stream & 0xFFFF) << 16 | (tensor_id & 0xFFFF)],
                   dtype=np.uint64)
    # One splitmix64 round of the key decorrelates neighbouring streams.
    return splitmix64(key)[0]


def f64_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """float64 -> float32 (nearest-even) -> bfloat16 bits (nearest-even)."""
    f = np.ascontiguousarray(v, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    rounding = np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))
    return ((u + rounding) >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bits to float64."""
    u = bits.astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def _fill_chunk(out: np.ndarray, lo: int, cnt: int, base: np.uint64, mean: float,
                std: float) -> None:
    pairs = (cnt + 1) // 2
    # lo is even (chunks are multiples of _CHUNK), so pairs never straddle.
    idx = np.arange(lo, lo + 2 * pairs, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = splitmix64(base + idx)
    u = ((z >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
    u1, u2 = u[0::2], u[1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    theta = (2.0 * np.pi) * u2
    nrm = np.empty(2 * pairs, dtype=np.float64)
    nrm[0::2] = r * np.cos(theta)
    nrm[1::2] = r * np.sin(theta)
    out[lo:lo + cnt] = f64_to_bf16_bits(mean + std * nrm[:cnt])


def normal_bf16(n: int, seed: int, stream: int, tensor: str, mean: float = 0.0,
                std: float = 1.0) -> np.ndarray:
    """``n`` bfloat16 samples of N(mean, std^2) as uint16 bit patterns.

    Chunks are independent (counter-based), so they are filled by a thread
    pool; the result does not depend on the number of threads.
    """
    out = np.empty(n, dtype=np.uint16)
    if std == 0.0:
        out[:] = f64_to_bf16_bits(np.full(1, mean))[0]
        return out
    base = _stream_base(seed, stream, _TENSOR_ID[tensor])
    starts = list(range(0, n, _CHUNK))
    if len(starts) <= 1:
        for lo in starts:
            _fill_chunk(out, lo, min(_CHUNK, n - lo), base, mean, std)
        return out
    workers = min(len(starts), os.cpu_count() or 1)
    with concurrent.futures.ThreadPoolExecutor(max_workers=workers) as pool:
        futs = [pool.submit(_fill_chunk, out, lo, min(_CHUNK, n - lo), base, mean, std)
                for lo in starts]
        for f in futs:
            f.result()
    return out


@dataclasses.dataclass(frozen=True)
class LayerShape:
    """Shape of one layer call.  ``head_dim`` 0 means hidden // heads."""

    micro_batch: int
    seq_len: int
    hidden: int
    heads: int
    ffn_hidden: int
    tp_parts: int = 1
    head_dim: int = 0

    @property
    def d(self) -> int:
        return self.head_dim if self.head_dim else self.hidden // self.heads

    @property
    def a(self) -> int:
        """Width of the attention block (heads x head_dim)."""
        return self.heads * self.d

    @property
    def tokens(self) -> int:
        return self.micro_batch * self.seq_len

    def param_shapes(self) -> Dict[str, tuple]:
        h, a, f = self.hidden, self.a, self.ffn_hidden
        return {
            "ln1_g": (h,), "ln1_b": (h,), "w_qkv": (3 * a, h), "b_qkv": (3 * a,),
            "w_o": (h, a), "b_o": (h,), "ln2_g": (h,), "ln2_b": (h,),
            "w_fc1": (f, h), "b_fc1": (f,), "w_fc2": (h, f), "b_fc2": (h,),
        }

    def with_tp(self, t: int) -> "LayerShape":
        return dataclasses.replace(self, tp_parts=t)


@dataclasses.dataclass
class LayerInputs:
    """bf16 bit patterns of every input (uint16 arrays), row-major."""

    shape: LayerShape
    x: np.ndarray            # [b, s, h]
    dy: np.ndarray           # [b, s, h]
    params: Dict[str, np.ndarray]

    def f64(self, name: str) -> np.ndarray:
        if name == "x":
            return bf16_bits_to_f64(self.x)
        if name == "dy":
            return bf16_bits_to_f64(self.dy)
        return bf16_bits_to_f64(self.params[name])

    def params_f64(self) -> Dict[str, np.ndarray]:
        return {k: bf16_bits_to_f64(v) for k, v in self.params.items()}


# Distributions of the configurations: activations and upstream gradient
# N(0, 1); weights N(0, 0.02^2); biases 0; LayerNorm gamma 1, beta 0.
DEFAULT_INIT = {
    "x": (0.0, 1.0), "dy": (0.0, 1.0),
    "w_qkv": (0.0, 0.02), "w_o": (0.0, 0.02), "w_fc1": (0.0, 0.02), "w_fc2": (0.0, 0.02),
    "b_qkv": (0.0, 0.0), "b_o": (0.0, 0.0), "b_fc1": (0.0, 0.0), "b_fc2": (0.0, 0.0),
    "ln1_g": (1.0, 0.0), "ln1_b": (0.0, 0.0), "ln2_g": (1.0, 0.0), "ln2_b": (0.0, 0.0),
}

# Variant that exercises the bias and LayerNorm-affine paths (non-zero values).
NONTRIVIAL_INIT = dict(DEFAULT_INIT)
NONTRIVIAL_INIT.update({
    "b_qkv": (0.0, 0.1), "b_o": (0.0, 0.1), "b_fc1": (0.0, 0.1), "b_fc2": (0.0, 0.1),
    "ln1_g": (1.0, 0.1), "ln1_b": (0.0, 0.1), "ln2_g": (1.0, 0.1), "ln2_b": (0.0, 0.1),
})


def make_layer_inputs(shape: LayerShape, seed: int = 0, layer: int = 0,
                      init: Optional[Dict[str, tuple]] = None,
                      with_params: bool = True) -> LayerInputs:
    """Draw x, dy and the layer's parameters for ``layer`` of a stack."""
    init = DEFAULT_INIT if init is None else init
    b, s, h = shape.micro_batch, shape.seq_len, shape.hidden
    x = normal_bf16(b * s * h, seed, 0, "x", *init["x"]).reshape(b, s, h)
    dy = normal_bf16(b * s * h, seed, 0, "dy", *init["dy"]).reshape(b, s, h)
    params = {}
    if with_params:
        for name, shp in shape.param_shapes().items():
            n = int(np.prod(shp))
            params[name] = normal_bf16(n, seed, layer + 1, name, *init[name]).reshape(shp)
    return LayerInputs(shape=shape, x=x, dy=dy, params=params)
