"""The layer with FP8 "hybrid" GEMMs, for the MC_FP8_HYBRID mode.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

The Megatron-Core listing (混合精度; its --fp8-format hybrid flag) runs the
GEMMs on 8-bit floats, E4M3 in the forward pass and E5M2 for gradients; it
gives no scaling recipe, and the one taken (per-tensor current scaling) is
the one of ``oracle/fp8.py``.  This function is the layer at one partition
(the partition sums are pinned elsewhere to equal the unpartitioned
products) with:

* every GEMM operand replaced by its quantise-dequantise value:
  decode(quantize(X)) * scale_inv, with E4M3 for the forward operands (ln1,
  O, ln2, g and the four weight matrices) and E5M2 for the gradient operands
  (dy, dhp, dx1, dQ|dK|dV).  A weight gradient and an input gradient use the
  same quantised tensors as the forward products (one scale per tensor);
* the bf16 rounding sites of the CUDA path (``oracle/rounding_floor.py``)
  where that path stores bf16: ln1, Q|K|V, the softmax probabilities, O, ln2,
  g, hp for GeLU', dhp, dO, P and dS in the attention backward, dQ|dK|dV.
  In this mode dx1 is quantised from fp32, so it has no bf16 site.

Everything else is float64.  With ``quantize=False`` the function is the
rounding-floor layer without the dx1 site, which the tests pin.
"""
from __future__ import annotations

import numpy as np

from . import fp8 as F
from . import layer as L
from .rounding_floor import bf16_round, rounded_attention_backward

E4M3, E5M2 = "e4m3", "e5m2"
FORWARD_OPERANDS = ("w_qkv", "w_o", "w_fc1", "w_fc2", "ln1", "o", "ln2", "g")
GRADIENT_OPERANDS = ("dy", "dhp", "dx1", "dqkv")


def qdq(x: np.ndarray, fmt: str) -> np.ndarray:
    """The values an FP8 product multiplies: per-tensor current scaling,
    round to the format, decode, times the inverse scale (float64)."""
    q, scale_inv = F.quantize(x, fmt)
    return F.decode(q, fmt).reshape(np.shape(x)) * float(scale_inv)


def fp8_forward_backward(shape, P, x, dy, quantize=True):
    """Forward + backward of the layer with FP8 hybrid GEMMs.  Returns
    (y, dx, grads) like ``oracle.layer.layer_forward_backward``."""
    def q(name, t, fmt):
        return qdq(t, fmt) if quantize else t

    b16 = bf16_round
    b, s, h = x.shape
    H, d, a = shape.heads, shape.d, shape.a
    scale = 1.0 / np.sqrt(d)
    W = {k: q(k, P[k], E4M3) for k in ("w_qkv", "w_o", "w_fc1", "w_fc2")}

    ln1, xh1, rs1 = L.layernorm_forward(x, P["ln1_g"], P["ln1_b"])
    ln1 = q("ln1", b16(ln1), E4M3)
    qkv = b16(ln1 @ W["w_qkv"].T + P["b_qkv"])
    o = np.empty((b, s, a))
    lse = np.empty((b, H, s))
    mask = np.tri(s) > 0

    def head(bi, hh, blk):
        return qkv[bi, :, blk * a + hh * d:blk * a + (hh + 1) * d]

    for bi in range(b):
        for hh in range(H):
            sc = np.where(mask, head(bi, hh, 0) @ head(bi, hh, 1).T * scale, -np.inf)
            m = sc.max(1, keepdims=True)
            e = np.exp(sc - m)
            l = e.sum(1, keepdims=True)
            o[bi, :, hh * d:(hh + 1) * d] = (b16(e) @ head(bi, hh, 2)) / l
            lse[bi, hh] = (m + np.log(l))[:, 0]
    o = b16(o)                       # attention output as stored (bf16)
    oq = q("o", o, E4M3)             # its 8-bit operand for the out-projection
    x1 = x + oq @ W["w_o"].T + P["b_o"]
    ln2, xh2, rs2 = L.layernorm_forward(x1, P["ln2_g"], P["ln2_b"])
    ln2 = q("ln2", b16(ln2), E4M3)
    hp = ln2 @ W["w_fc1"].T + P["b_fc1"]
    g = q("g", b16(L.gelu_tanh(hp)), E4M3)
    y = x1 + g @ W["w_fc2"].T + P["b_fc2"]

    G = {}

    def r2(m):
        return m.reshape(-1, m.shape[-1])

    G["b_fc2"] = r2(dy).sum(0)
    dyq = q("dy", dy, E5M2)
    G["w_fc2"] = r2(dyq).T @ r2(g)
    dhp = b16((dyq @ W["w_fc2"]) * L.gelu_tanh_grad(b16(hp)))
    G["b_fc1"] = r2(dhp).sum(0)
    dhpq = q("dhp", dhp, E5M2)
    G["w_fc1"] = r2(dhpq).T @ r2(ln2)
    dd, G["ln2_g"], G["ln2_b"] = L.layernorm_backward(dhpq @ W["w_fc1"], xh2, rs2, P["ln2_g"])
    dx1 = dy + dd
    G["b_o"] = r2(dx1).sum(0)
    dx1q = q("dx1", dx1, E5M2)
    G["w_o"] = r2(dx1q).T @ r2(oq)
    do = b16(dx1q @ W["w_o"])
    dqkv = np.empty_like(qkv)

    def site(name, t):
        return b16(t) if name in ("p_bwd", "ds") else t

    for bi in range(b):
        for hh in range(H):
            c = slice(hh * d, (hh + 1) * d)
            dq, dk, dv = rounded_attention_backward(
                head(bi, hh, 0), head(bi, hh, 1), head(bi, hh, 2), o[bi, :, c], lse[bi, hh],
                do[bi, :, c], site)
            dqkv[bi, :, c] = dq
            dqkv[bi, :, a + hh * d:a + (hh + 1) * d] = dk
            dqkv[bi, :, 2 * a + hh * d:2 * a + (hh + 1) * d] = dv
    dqkv = b16(dqkv)
    G["b_qkv"] = r2(dqkv).sum(0)
    dqkvq = q("dqkv", dqkv, E5M2)
    G["w_qkv"] = r2(dqkvq).T @ r2(ln1)
    dd, G["ln1_g"], G["ln1_b"] = L.layernorm_backward(dqkvq @ W["w_qkv"], xh1, rs1, P["ln1_g"])
    return y, dx1 + dd, G
