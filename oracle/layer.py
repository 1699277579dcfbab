"""fp64 CPU oracle of one GPT pre-LN transformer layer, forward and backward.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline leg may import this module.  The CUDA library never
calls it and shares no code with it.

What it computes (plain definitions, evaluated in float64 on the bf16-valued
inputs, no intermediate rounding):

* Layer form (pre-LN GPT block, no dropout)::

      x1 = x + OutProj(Attn(LN1(x)))
      y  = x1 + FC2(GeLU(FC1(LN2(x1))))

* Tensor-parallel split, following the tutorial cf-1.com/news/5344657,
  section 2.2 ("张量并行：把一个大矩阵劈开"): the QKV projection is split by its
  output dimension (partition p owns heads [p H/t, (p+1) H/t)), the first MLP
  linear is split by columns and the second by rows.  The two row-parallel
  linears (attention out-projection and fc2) produce one partial product per
  partition; the partials are summed and the bias is added once after the
  sum.  In the backward pass the two column-parallel linears (QKV and fc1)
  produce one partial input-gradient per partition, which are summed the same
  way.  Each of these sums is written here as an explicit loop over p.
* LayerNorm: biased variance over the hidden dimension, eps = 1e-5.
* GeLU: tanh form 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))).
* Attention: per head, S = q k^T / sqrt(d), causal (key j visible to query i
  iff j <= i), softmax over visible keys, O = P v; LSE = log sum exp(S) over
  visible keys is kept for the backward pass.

The pages write none of these formulas out; the choices above are the plain
readings listed in the design notes (pre-LN, tanh-GeLU, causal, no dropout,
1/sqrt(d) scale, eps 1e-5, biases on all four linears).

Weight layout (PyTorch ``nn.Linear``: y = x W^T + b):
  w_qkv [3a, h] = [Wq; Wk; Wv], each block head-major (head k owns rows
  [k d, (k+1) d) of its block); w_o [h, a]; w_fc1 [f, h]; w_fc2 [h, f].
Activations are [b, s, h] row-major.

Matrix products use numpy's ``@`` (a library matmul) as a single step; rows of
the attention score matrix are formed a block of query rows at a time only to
bound memory -- every row is still the plain definition over its visible keys.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Tuple

import numpy as np

LN_EPS = 1e-5
_GELU_C = np.sqrt(2.0 / np.pi)
_GELU_A = 0.044715

# Query rows per block of the attention score matrix (memory bound only).
_ATTN_ROW_BLOCK = 512


@dataclasses.dataclass(frozen=True)
class OracleShape:
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
        return self.heads * self.d


def oracle_shape(s) -> OracleShape:
    """Accept any object with the shape fields (e.g. a LayerShape)."""
    return OracleShape(s.micro_batch, s.seq_len, s.hidden, s.heads, s.ffn_hidden,
                       s.tp_parts, getattr(s, "head_dim", 0))


# --------------------------------------------------------------------------
# Elementary pieces
# --------------------------------------------------------------------------

def layernorm_forward(x: np.ndarray, gamma: np.ndarray, beta: np.ndarray,
                      eps: float = LN_EPS) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """LayerNorm over the last axis.  Returns (out, xhat, rstd)."""
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    rstd = 1.0 / np.sqrt(var + eps)
    xhat = (x - mu) * rstd
    return xhat * gamma + beta, xhat, rstd


def layernorm_backward(dout: np.ndarray, xhat: np.ndarray, rstd: np.ndarray,
                       gamma: np.ndarray) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Gradient of LayerNorm.  Returns (dx, dgamma, dbeta)."""
    lead = tuple(range(dout.ndim - 1))
    dgamma = (dout * xhat).sum(axis=lead)
    dbeta = dout.sum(axis=lead)
    dxhat = dout * gamma
    m1 = dxhat.mean(axis=-1, keepdims=True)
    m2 = (dxhat * xhat).mean(axis=-1, keepdims=True)
    dx = rstd * (dxhat - m1 - xhat * m2)
    return dx, dgamma, dbeta


def gelu_tanh(x: np.ndarray) -> np.ndarray:
    return 0.5 * x * (1.0 + np.tanh(_GELU_C * (x + _GELU_A * x ** 3)))


def gelu_tanh_grad(x: np.ndarray) -> np.ndarray:
    """d/dx of gelu_tanh, in closed form."""
    th = np.tanh(_GELU_C * (x + _GELU_A * x ** 3))
    return 0.5 * (1.0 + th) + 0.5 * x * (1.0 - th * th) * _GELU_C * (1.0 + 3.0 * _GELU_A * x * x)


def causal_attention_forward(q: np.ndarray, k: np.ndarray, v: np.ndarray
                             ) -> Tuple[np.ndarray, np.ndarray]:
    """One head.  q, k, v: [s, d].  Returns (O [s, d], LSE [s])."""
    s, d = q.shape
    scale = 1.0 / np.sqrt(d)
    out = np.empty_like(q)
    lse = np.empty(s)
    for r0 in range(0, s, _ATTN_ROW_BLOCK):
        r1 = min(s, r0 + _ATTN_ROW_BLOCK)
        sc = (q[r0:r1] @ k[:r1].T) * scale            # [rows, r1]
        rows = np.arange(r0, r1)[:, None]
        cols = np.arange(r1)[None, :]
        sc = np.where(cols <= rows, sc, -np.inf)       # key j visible iff j <= i
        m = sc.max(axis=1, keepdims=True)
        e = np.exp(sc - m)
        l = e.sum(axis=1, keepdims=True)
        out[r0:r1] = (e / l) @ v[:r1]
        lse[r0:r1] = (m + np.log(l))[:, 0]
    return out, lse


def causal_attention_backward(q, k, v, o, lse, do):
    """One head.  Returns (dq, dk, dv), all [s, d]."""
    s, d = q.shape
    scale = 1.0 / np.sqrt(d)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    dsum = (do * o).sum(axis=1)                         # D_i = dO_i . O_i
    for r0 in range(0, s, _ATTN_ROW_BLOCK):
        r1 = min(s, r0 + _ATTN_ROW_BLOCK)
        sc = (q[r0:r1] @ k[:r1].T) * scale
        rows = np.arange(r0, r1)[:, None]
        cols = np.arange(r1)[None, :]
        p = np.where(cols <= rows, np.exp(sc - lse[r0:r1, None]), 0.0)
        dv[:r1] += p.T @ do[r0:r1]
        dp = do[r0:r1] @ v[:r1].T
        ds = p * (dp - dsum[r0:r1, None])
        dq[r0:r1] = (ds @ k[:r1]) * scale
        dk[:r1] += (ds.T @ q[r0:r1]) * scale
    return dq, dk, dv


# --------------------------------------------------------------------------
# Partition helpers (tensor-parallel split)
# --------------------------------------------------------------------------

def head_range(shape: OracleShape, p: int) -> range:
    hp = shape.heads // shape.tp_parts
    return range(p * hp, (p + 1) * hp)


def qkv_rows(shape: OracleShape, p: int) -> np.ndarray:
    """Rows of w_qkv owned by partition p: its heads in the Q, K and V blocks."""
    a, d = shape.a, shape.d
    hr = head_range(shape, p)
    blocks = []
    for blk in range(3):
        blocks.append(np.arange(blk * a + hr.start * d, blk * a + hr.stop * d))
    return np.concatenate(blocks)


def attn_cols(shape: OracleShape, p: int) -> slice:
    """Columns of O (and of w_o) owned by partition p."""
    hr = head_range(shape, p)
    return slice(hr.start * shape.d, hr.stop * shape.d)


def ffn_cols(shape: OracleShape, p: int) -> slice:
    fp = shape.ffn_hidden // shape.tp_parts
    return slice(p * fp, (p + 1) * fp)


def check_divisible(shape: OracleShape) -> None:
    """Hidden size, heads and ffn size must divide by tp_parts.

    Divisibility rule: ai.lansai.wang/82226.html, section 并行度先做整数校验, and
    cf-1.com/news/5344657, section 2.2 (hidden_size and head count divisible by
    the tensor-parallel degree, else a hard error).  The ffn condition follows
    from the column split of the first MLP linear.
    """
    t = shape.tp_parts
    if t < 1:
        raise ValueError("tp_parts must be >= 1")
    if shape.hidden % t or shape.heads % t or shape.ffn_hidden % t:
        raise ValueError(f"hidden={shape.hidden}, heads={shape.heads}, ffn={shape.ffn_hidden} "
                         f"not divisible by tp_parts={t}")
    if shape.head_dim == 0 and shape.hidden % shape.heads:
        raise ValueError("hidden not divisible by heads")


# --------------------------------------------------------------------------
# Layer forward / backward
# --------------------------------------------------------------------------

def layer_forward(shape, params: Dict[str, np.ndarray], x: np.ndarray):
    """Forward pass.  ``x`` [b, s, h] float64.  Returns (y, cache)."""
    shape = oracle_shape(shape)
    check_divisible(shape)
    b, s, h = x.shape
    H, d, a, t = shape.heads, shape.d, shape.a, shape.tp_parts
    P = params

    ln1, xhat1, rstd1 = layernorm_forward(x, P["ln1_g"], P["ln1_b"])

    # Column-parallel QKV: each partition projects onto its own heads.
    q = np.empty((b, s, a))
    k = np.empty((b, s, a))
    v = np.empty((b, s, a))
    for p in range(t):
        rows = qkv_rows(shape, p)
        qkv_p = ln1 @ P["w_qkv"][rows].T + P["b_qkv"][rows]
        n = rows.size // 3
        cols = attn_cols(shape, p)
        q[:, :, cols] = qkv_p[:, :, :n]
        k[:, :, cols] = qkv_p[:, :, n:2 * n]
        v[:, :, cols] = qkv_p[:, :, 2 * n:]

    # Attention, local to each head.
    o = np.empty((b, s, a))
    lse = np.empty((b, H, s))
    for bi in range(b):
        for hh in range(H):
            c = slice(hh * d, (hh + 1) * d)
            o[bi, :, c], lse[bi, hh] = causal_attention_forward(q[bi, :, c], k[bi, :, c], v[bi, :, c])

    # Row-parallel out-projection: one partial per partition, summed, then the
    # bias once and the residual.
    attn_sum = np.zeros((b, s, h))
    for p in range(t):
        cols = attn_cols(shape, p)
        attn_sum += o[:, :, cols] @ P["w_o"][:, cols].T
    x1 = x + attn_sum + P["b_o"]

    ln2, xhat2, rstd2 = layernorm_forward(x1, P["ln2_g"], P["ln2_b"])

    # Column-parallel fc1 + GeLU.
    hp = np.empty((b, s, shape.ffn_hidden))
    for p in range(t):
        cols = ffn_cols(shape, p)
        hp[:, :, cols] = ln2 @ P["w_fc1"][cols].T + P["b_fc1"][cols]
    g = gelu_tanh(hp)

    # Row-parallel fc2: partials summed, bias once, residual.
    mlp_sum = np.zeros((b, s, h))
    for p in range(t):
        cols = ffn_cols(shape, p)
        mlp_sum += g[:, :, cols] @ P["w_fc2"][:, cols].T
    y = x1 + mlp_sum + P["b_fc2"]

    cache = dict(ln1=ln1, xhat1=xhat1, rstd1=rstd1, q=q, k=k, v=v, o=o, lse=lse,
                 x1=x1, ln2=ln2, xhat2=xhat2, rstd2=rstd2, hp=hp, g=g)
    return y, cache


def layer_backward(shape, params: Dict[str, np.ndarray], cache, dy: np.ndarray):
    """Backward pass for upstream gradient ``dy`` [b, s, h].

    Returns (dx, grads) with grads keyed like ``params``.
    """
    shape = oracle_shape(shape)
    b, s, h = dy.shape
    H, d, a, t = shape.heads, shape.d, shape.a, shape.tp_parts
    P = params
    C = cache
    G = {}

    def colsum(m):
        return m.reshape(-1, m.shape[-1]).sum(axis=0)

    def rows2d(m):
        return m.reshape(-1, m.shape[-1])

    # fc2 (row-parallel): per partition weight grad and input grad.
    G["b_fc2"] = colsum(dy)
    G["w_fc2"] = np.empty_like(P["w_fc2"])
    dhp = np.empty_like(C["hp"])
    for p in range(t):
        cols = ffn_cols(shape, p)
        G["w_fc2"][:, cols] = rows2d(dy).T @ rows2d(C["g"][:, :, cols])
        dg_p = dy @ P["w_fc2"][:, cols]
        dhp[:, :, cols] = dg_p * gelu_tanh_grad(C["hp"][:, :, cols])

    # fc1 (column-parallel): the input gradient is a sum over partitions.
    G["b_fc1"] = colsum(dhp)
    G["w_fc1"] = np.empty_like(P["w_fc1"])
    dln2 = np.zeros((b, s, h))
    for p in range(t):
        cols = ffn_cols(shape, p)
        G["w_fc1"][cols] = rows2d(dhp[:, :, cols]).T @ rows2d(C["ln2"])
        dln2 += dhp[:, :, cols] @ P["w_fc1"][cols]

    dx1_ln, G["ln2_g"], G["ln2_b"] = layernorm_backward(dln2, C["xhat2"], C["rstd2"], P["ln2_g"])
    dx1 = dy + dx1_ln

    # Out-projection (row-parallel).
    G["b_o"] = colsum(dx1)
    G["w_o"] = np.empty_like(P["w_o"])
    do = np.empty((b, s, a))
    for p in range(t):
        cols = attn_cols(shape, p)
        G["w_o"][:, cols] = rows2d(dx1).T @ rows2d(C["o"][:, :, cols])
        do[:, :, cols] = dx1 @ P["w_o"][:, cols]

    # Attention backward, per head.
    dq = np.empty((b, s, a))
    dk = np.empty((b, s, a))
    dv = np.empty((b, s, a))
    for bi in range(b):
        for hh in range(H):
            c = slice(hh * d, (hh + 1) * d)
            dq[bi, :, c], dk[bi, :, c], dv[bi, :, c] = causal_attention_backward(
                C["q"][bi, :, c], C["k"][bi, :, c], C["v"][bi, :, c], C["o"][bi, :, c],
                C["lse"][bi, hh], do[bi, :, c])

    # QKV (column-parallel): input gradient summed over partitions.
    G["w_qkv"] = np.empty_like(P["w_qkv"])
    G["b_qkv"] = np.empty_like(P["b_qkv"])
    dln1 = np.zeros((b, s, h))
    for p in range(t):
        rows = qkv_rows(shape, p)
        cols = attn_cols(shape, p)
        dqkv_p = np.concatenate([dq[:, :, cols], dk[:, :, cols], dv[:, :, cols]], axis=-1)
        G["b_qkv"][rows] = colsum(dqkv_p)
        G["w_qkv"][rows] = rows2d(dqkv_p).T @ rows2d(C["ln1"])
        dln1 += dqkv_p @ P["w_qkv"][rows]

    dx_ln, G["ln1_g"], G["ln1_b"] = layernorm_backward(dln1, C["xhat1"], C["rstd1"], P["ln1_g"])
    dx = dx1 + dx_ln
    return dx, G


def layer_forward_backward(shape, params, x, dy):
    y, cache = layer_forward(shape, params, x)
    dx, grads = layer_backward(shape, params, cache, dy)
    return y, dx, grads
