"""Sampled outputs of the layer for sequences too long for the full oracle.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Causality makes two sets of outputs computable without the whole layer:
* y at any query row i needs only row i's own path plus K and V of the
  tokens j <= i (computed for all tokens, a [T, h] x [h, 2a] product);
* dx at the last R rows of a sequence depends only on dy at those rows
  (y_i depends on x_j only for i >= j), and the backward through attention
  for those rows reaches keys j only through queries i >= j -- which are all
  in the tail.  So dx for the tail is exact from the tail's forward and
  backward plus the all-token K and V.
Same definitions as ``oracle.layer`` (whose LayerNorm and GeLU functions it
uses), evaluated in float64; the tensor-parallel partition sums are taken
whole (their equality with the unpartitioned products is pinned separately).
"""
from __future__ import annotations

import numpy as np

from . import layer as L


def _split_qkv(P, a):
    W, bias = P["w_qkv"], P["b_qkv"]
    return (W[:a], bias[:a]), (W[a:2 * a], bias[a:2 * a]), (W[2 * a:], bias[2 * a:])


def sampled_rows_and_tail(shape, P, x, dy, rows, tail):
    """Returns (y[:, rows, :], dx[:, s-tail:, :]) for x, dy of shape [b, s, h]."""
    shape = L.oracle_shape(shape)
    b, s, h = x.shape
    H, d, a = shape.heads, shape.d, shape.a
    scale = 1.0 / np.sqrt(d)
    (Wq, bq), (Wk, bk), (Wv, bv) = _split_qkv(P, a)
    ln1, xhat1, rstd1 = L.layernorm_forward(x, P["ln1_g"], P["ln1_b"])
    k_all = ln1 @ Wk.T + bk
    v_all = ln1 @ Wv.T + bv

    def row_forward(ridx):
        """Forward of the given query rows (same rows in every sequence)."""
        q = ln1[:, ridx] @ Wq.T + bq                      # [b, n, a]
        o = np.empty_like(q)
        lse = np.empty((b, H, len(ridx)))
        probs = {}
        last = int(ridx.max()) + 1
        vis = np.arange(last)[None, :] <= ridx[:, None]  # [n, last]
        for bi in range(b):
            for hh in range(H):
                c = slice(hh * d, (hh + 1) * d)
                sc = np.where(vis, (q[bi, :, c] @ k_all[bi, :last, c].T) * scale, -np.inf)
                m = sc.max(axis=1, keepdims=True)
                e = np.exp(sc - m)
                l = e.sum(axis=1, keepdims=True)
                p = e / l
                probs[bi, hh] = p
                o[bi, :, c] = p @ v_all[bi, :last, c]
                lse[bi, hh] = (m + np.log(l))[:, 0]
        x1 = x[:, ridx] + o @ P["w_o"].T + P["b_o"]
        ln2, xhat2, rstd2 = L.layernorm_forward(x1, P["ln2_g"], P["ln2_b"])
        hp = ln2 @ P["w_fc1"].T + P["b_fc1"]
        g = L.gelu_tanh(hp)
        y = x1 + g @ P["w_fc2"].T + P["b_fc2"]
        return y, dict(q=q, o=o, probs=probs, last=last, x1=x1, xhat2=xhat2, rstd2=rstd2, hp=hp)

    y_rows, _ = row_forward(np.asarray(rows))

    t0 = s - tail
    tidx = np.arange(t0, s)
    _, c = row_forward(tidx)
    dy_t = dy[:, t0:]
    dhp = (dy_t @ P["w_fc2"]) * L.gelu_tanh_grad(c["hp"])
    dln2 = dhp @ P["w_fc1"]
    dx1_ln, _, _ = L.layernorm_backward(dln2, c["xhat2"], c["rstd2"], P["ln2_g"])
    dx1 = dy_t + dx1_ln
    do = dx1 @ P["w_o"]
    dq = np.empty((b, tail, a))
    dk = np.empty((b, tail, a))
    dv = np.empty((b, tail, a))
    last = c["last"]                                      # == s
    for bi in range(b):
        for hh in range(H):
            cs = slice(hh * d, (hh + 1) * d)
            p = c["probs"][bi, hh]                        # [tail, s]
            dsum = (do[bi, :, cs] * c["o"][bi, :, cs]).sum(axis=1)
            dp = do[bi, :, cs] @ v_all[bi, :last, cs].T
            ds = p * (dp - dsum[:, None])
            dq[bi, :, cs] = (ds @ k_all[bi, :last, cs]) * scale
            # keys in the tail are reached only by queries in the tail
            dk[bi, :, cs] = (ds[:, t0:].T @ c["q"][bi, :, cs]) * scale
            dv[bi, :, cs] = p[:, t0:].T @ do[bi, :, cs]
    dqkv = np.concatenate([dq, dk, dv], axis=-1)
    dln1 = dqkv @ P["w_qkv"]
    dx_ln, _, _ = L.layernorm_backward(dln1, xhat1[:, t0:], rstd1[:, t0:], P["ln1_g"])
    return y_rows, dx1 + dx_ln
