"""Diagnostic: the error that bf16 GEMM operands alone cause in the layer.

TEST INFRASTRUCTURE ONLY (never used by the CUDA library).  It re-runs the
layer in float64 but rounds to bfloat16 (round-to-nearest-even) every tensor
that a bf16-operand / fp32-accumulate implementation feeds to a matrix
multiply.  Each rounding happens at a named site; ``GPU_ROUNDING_SITES`` lists
the sites where the CUDA path of this library stores a bf16 operand:

  ln1, ln2    LayerNorm outputs (QKV and fc1 operands)
  qkv         Q | K | V after the bias (attention operands)
  p_fwd       softmax probabilities, unnormalised, before P.V (the row sum
              that divides the product is taken before rounding)
  o           attention output (out-projection operand, delta)
  g           GeLU output (fc2 operand)
  hp          fc1 pre-activation as stored for GeLU'
  dhp         (dy W2) * GeLU'(hp) (fc1 dgrad / wgrad operand)
  dx1         bf16 copy of dx1 (out-projection dgrad / wgrad operand); the
              out-projection bias gradient and the residual use it unrounded
  do          dO (attention backward operand)
  p_bwd       P recomputed in the backward, before dV = P^T dO
  ds          dS = P (dP - delta), before the 1/sqrt(d) scale
  dqkv        dQ | dK | dV (QKV dgrad / wgrad operand)

Sites outside that list are accepted so that a test can show how the floor
moves when a rounding is added where the CUDA path keeps fp32: ``x1`` (the
residual stream after attention) and ``ds_scaled`` (dS rounded after the
1/sqrt(d) scale instead of before).  With ``sites=()`` nothing is rounded and
the function is the plain layer at one partition.

Comparing the result with the exact oracle gives the floor that any such
implementation sits on; the parity tests use it as a second, binding bound.
"""
from __future__ import annotations

import numpy as np

from . import layer as L

GPU_ROUNDING_SITES = ("ln1", "qkv", "p_fwd", "o", "g", "hp", "ln2", "dhp", "dx1", "do",
                      "p_bwd", "ds", "dqkv")
EXTRA_SITES = ("x1", "ds_scaled")


def bf16_round(x: np.ndarray) -> np.ndarray:
    """float64 -> float32 (nearest-even) -> bfloat16 (nearest-even), as float64."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = ((u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)) << np.uint64(16)
    return u.astype(np.uint32).view(np.float32).astype(np.float64).reshape(np.shape(x))


def rounded_attention_backward(q, k, v, o, lse, do, r):
    """One head's attention backward with the rounding sites p_bwd, ds (or
    ds_scaled) applied through ``r(site, tensor)``.  Returns dq, dk, dv
    before the dqkv site."""
    s, d = q.shape
    scale = 1.0 / np.sqrt(d)
    mask = np.tri(s) > 0
    p = np.where(mask, np.exp(q @ k.T * scale - lse[:, None]), 0.0)
    delta = (do * o).sum(1)
    dv = r("p_bwd", p).T @ do
    ds = p * (do @ v.T - delta[:, None])
    ds = r("ds", ds)
    dsc = r("ds_scaled", ds * scale)
    return dsc @ k, dsc.T @ q, dv


def rounded_forward_backward(shape, P, x, dy, sites=GPU_ROUNDING_SITES, rnd=bf16_round):
    """Layer forward + backward at one partition, with ``rnd`` applied at the
    named ``sites``.  Returns (y, dx, grads) like the oracle."""
    unknown = set(sites) - set(GPU_ROUNDING_SITES) - set(EXTRA_SITES)
    assert not unknown, unknown
    on = frozenset(sites)

    def r(site, t):
        return rnd(t) if site in on else t

    b, s, h = x.shape
    H, d, a = shape.heads, shape.d, shape.a
    scale = 1.0 / np.sqrt(d)
    ln1, xh1, rs1 = L.layernorm_forward(x, P["ln1_g"], P["ln1_b"])
    ln1 = r("ln1", ln1)
    qkv = r("qkv", ln1 @ P["w_qkv"].T + P["b_qkv"])
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
            o[bi, :, hh * d:(hh + 1) * d] = (r("p_fwd", e) @ head(bi, hh, 2)) / l
            lse[bi, hh] = (m + np.log(l))[:, 0]
    o = r("o", o)
    x1 = r("x1", x + o @ P["w_o"].T + P["b_o"])
    ln2, xh2, rs2 = L.layernorm_forward(x1, P["ln2_g"], P["ln2_b"])
    ln2 = r("ln2", ln2)
    hp = ln2 @ P["w_fc1"].T + P["b_fc1"]
    g = r("g", L.gelu_tanh(hp))
    y = x1 + g @ P["w_fc2"].T + P["b_fc2"]

    G = {}

    def r2(m):
        return m.reshape(-1, m.shape[-1])

    G["b_fc2"] = r2(dy).sum(0)
    G["w_fc2"] = r2(dy).T @ r2(g)
    dhp = r("dhp", (dy @ P["w_fc2"]) * L.gelu_tanh_grad(r("hp", hp)))
    G["b_fc1"] = r2(dhp).sum(0)
    G["w_fc1"] = r2(dhp).T @ r2(ln2)
    dd, G["ln2_g"], G["ln2_b"] = L.layernorm_backward(dhp @ P["w_fc1"], xh2, rs2, P["ln2_g"])
    dx1 = dy + dd
    G["b_o"] = r2(dx1).sum(0)
    dx1r = r("dx1", dx1)
    G["w_o"] = r2(dx1r).T @ r2(o)
    do = r("do", dx1r @ P["w_o"])
    dqkv = np.empty_like(qkv)
    for bi in range(b):
        for hh in range(H):
            c = slice(hh * d, (hh + 1) * d)
            dq, dk, dv = rounded_attention_backward(
                head(bi, hh, 0), head(bi, hh, 1), head(bi, hh, 2), o[bi, :, c], lse[bi, hh],
                do[bi, :, c], r)
            dqkv[bi, :, c] = dq
            dqkv[bi, :, a + hh * d:a + (hh + 1) * d] = dk
            dqkv[bi, :, 2 * a + hh * d:2 * a + (hh + 1) * d] = dv
    dqkv = r("dqkv", dqkv)
    G["b_qkv"] = r2(dqkv).sum(0)
    G["w_qkv"] = r2(dqkv).T @ r2(ln1)
    dd, G["ln1_g"], G["ln1_b"] = L.layernorm_backward(dqkv @ P["w_qkv"], xh1, rs1, P["ln1_g"])
    return y, dx1 + dd, G


def floor_norm_rel(shape, P, x, dy, exact=None):
    """Per tensor, sum|floor - exact| / sum|exact| (the norm-wise error that
    the rounding sites alone cause).  ``exact`` = (y, dx, grads) of the oracle
    on the same inputs, computed here when not given."""
    if exact is None:
        exact = L.layer_forward_backward(shape, P, x, dy)
    y, dx, G = exact
    yr, dxr, Gr = rounded_forward_backward(shape, P, x, dy)

    def nr(a, b):
        den = float(np.abs(b).sum()) or 1.0
        return float(np.abs(a - b).sum()) / den

    out = {"y": nr(yr, y), "dx": nr(dxr, dx)}
    out.update({k: nr(Gr[k], G[k]) for k in G})
    return out
