"""Diagnostic: the error that bf16 GEMM operands alone cause in the layer.

TEST INFRASTRUCTURE ONLY (never used by the CUDA library).  It re-runs the
layer in float64 but rounds, to bfloat16, every tensor that a bf16-operand /
fp32-accumulate implementation must feed to a matrix multiply: LN1 and LN2
outputs, Q|K|V, the softmax probabilities P, the attention output O, the GeLU
output g, the fc1 pre-activation used for GeLU', dhp, the bf16 copy of dx1,
dO, dS and dQ|dK|dV.  Comparing this with the exact oracle gives the floor
that any such implementation sits on -- used to choose how the stated
tolerance is read (see tests/test_rounding_floor.py).
"""
from __future__ import annotations

import numpy as np

from . import layer as L


def _bf16(x: np.ndarray) -> np.ndarray:
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = ((u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)) << np.uint64(16)
    return u.astype(np.uint32).view(np.float32).astype(np.float64).reshape(x.shape)


def rounded_forward_backward(shape, P, x, dy):
    """Layer forward + backward (t = 1) with bf16 rounding at GEMM operands."""
    b, s, h = x.shape
    H, d, a = shape.heads, shape.d, shape.a
    ln1, xh1, rs1 = L.layernorm_forward(x, P["ln1_g"], P["ln1_b"])
    ln1 = _bf16(ln1)
    qkv = _bf16(ln1 @ P["w_qkv"].T + P["b_qkv"])
    o = np.empty((b, s, a))
    lse = np.empty((b, H, s))
    mask = np.tri(s) > 0
    for bi in range(b):
        for hh in range(H):
            c = slice(hh * d, (hh + 1) * d)
            q, k, v = qkv[bi, :, c], qkv[bi, :, a + hh * d:a + (hh + 1) * d], \
                qkv[bi, :, 2 * a + hh * d:2 * a + (hh + 1) * d]
            sc = np.where(mask, q @ k.T / np.sqrt(d), -np.inf)
            m = sc.max(1, keepdims=True)
            e = np.exp(sc - m)
            l = e.sum(1, keepdims=True)
            o[bi, :, c] = (_bf16(e) @ v) / l
            lse[bi, hh] = (m + np.log(l))[:, 0]
    o = _bf16(o)
    x1 = x + o @ P["w_o"].T + P["b_o"]
    ln2, xh2, rs2 = L.layernorm_forward(x1, P["ln2_g"], P["ln2_b"])
    ln2 = _bf16(ln2)
    hp = ln2 @ P["w_fc1"].T + P["b_fc1"]
    g = _bf16(L.gelu_tanh(hp))
    y = x1 + g @ P["w_fc2"].T + P["b_fc2"]

    G = {}
    r2 = lambda m: m.reshape(-1, m.shape[-1])  # noqa: E731
    G["b_fc2"] = r2(dy).sum(0)
    G["w_fc2"] = r2(dy).T @ r2(g)
    dhp = _bf16((dy @ P["w_fc2"]) * L.gelu_tanh_grad(_bf16(hp)))
    G["b_fc1"] = r2(dhp).sum(0)
    G["w_fc1"] = r2(dhp).T @ r2(ln2)
    dd, G["ln2_g"], G["ln2_b"] = L.layernorm_backward(dhp @ P["w_fc1"], xh2, rs2, P["ln2_g"])
    dx1 = dy + dd
    G["b_o"] = r2(dx1).sum(0)
    dx1r = _bf16(dx1)
    G["w_o"] = r2(dx1r).T @ r2(o)
    do = _bf16(dx1r @ P["w_o"])
    dqkv = np.empty_like(qkv)
    for bi in range(b):
        for hh in range(H):
            c = slice(hh * d, (hh + 1) * d)
            ck, cv = slice(a + hh * d, a + (hh + 1) * d), slice(2 * a + hh * d, 2 * a + (hh + 1) * d)
            q, k, v = qkv[bi, :, c], qkv[bi, :, ck], qkv[bi, :, cv]
            p = np.where(mask, np.exp(q @ k.T / np.sqrt(d) - lse[bi, hh][:, None]), 0.0)
            dsum = (do[bi, :, c] * o[bi, :, c]).sum(1)
            dqkv[bi, :, cv] = _bf16(p).T @ do[bi, :, c]
            ds = _bf16(p * (do[bi, :, c] @ v.T - dsum[:, None]))
            dqkv[bi, :, c] = ds @ k / np.sqrt(d)
            dqkv[bi, :, ck] = ds.T @ q / np.sqrt(d)
    dqkv = _bf16(dqkv)
    G["b_qkv"] = r2(dqkv).sum(0)
    G["w_qkv"] = r2(dqkv).T @ r2(ln1)
    dd, G["ln1_g"], G["ln1_b"] = L.layernorm_backward(dqkv @ P["w_qkv"], xh1, rs1, P["ln1_g"])
    return y, dx1 + dd, G
