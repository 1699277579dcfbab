"""Pins of the fp64 oracle against things other than itself.

* finite differences of the forward pass (pins the whole backward pass);
* independent library routines: torch float64 ``layer_norm``, causal
  ``scaled_dot_product_attention`` and tanh ``gelu`` with autograd (pins the
  forward pass: variance convention, attention scale, mask direction, GeLU
  form) -- torch is used here only as a checker, never by the CUDA library;
* brute-force attention with explicit Python loops on tiny inputs;
* tensor-parallel invariance (sum of row-parallel partials == unpartitioned
  product; outputs independent of tp_parts);
* causality (rows <= i independent of tokens after i; the gradient statement);
* closed forms (s = 1, zero query weights, constant LayerNorm row, GeLU
  values, all-zero weights).

``test_planted_mistakes`` plants plausible mistakes in the oracle (on the CPU)
and checks that at least one pin fails for each.
"""
import math

import numpy as np
import pytest
import torch

import oracle.layer as L
from layer_inputs import LayerShape, make_layer_inputs
from layer_inputs.generator import NONTRIVIAL_INIT


def _tiny_inputs(shape, seed=1, wstd=0.3):
    init = dict(NONTRIVIAL_INIT)
    for w in ("w_qkv", "w_o", "w_fc1", "w_fc2"):
        init[w] = (0.0, wstd)
    inp = make_layer_inputs(shape, seed=seed, init=init)
    return inp.params_f64(), inp.f64("x"), inp.f64("dy")


def _rel(a, b):
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-300))


# --------------------------------------------------------------------------
# Finite differences
# --------------------------------------------------------------------------

def fd_max_rel_error(shape, P, x, dy, n_probe=40, seed=0):
    """Max relative error of analytic vs central-difference gradients of
    L = sum(y * dy), over every x entry and a sample of each parameter."""
    rng = np.random.default_rng(seed)
    _, dx, G = L.layer_forward_backward(shape, P, x, dy)

    def loss(P_, x_):
        y, _ = L.layer_forward(shape, P_, x_)
        return float((y * dy).sum())

    worst = 0.0
    probes = [("x", idx) for idx in np.ndindex(x.shape)]
    for name, val in P.items():
        flat = rng.choice(val.size, size=min(n_probe, val.size), replace=False)
        probes += [(name, np.unravel_index(i, val.shape)) for i in flat]
    for name, idx in probes:
        base = x if name == "x" else P[name]
        theta = base[idx]
        step = 1e-6 * max(1.0, abs(theta))
        plus = {k: v.copy() for k, v in P.items()}
        minus = {k: v.copy() for k, v in P.items()}
        xp, xm = x.copy(), x.copy()
        if name == "x":
            xp[idx] += step
            xm[idx] -= step
        else:
            plus[name][idx] += step
            minus[name][idx] -= step
        fd = (loss(plus, xp) - loss(minus, xm)) / (2 * step)
        an = dx[idx] if name == "x" else G[name][idx]
        worst = max(worst, abs(fd - an) / max(1.0, abs(an)))
    return worst


@pytest.mark.parametrize("b,s,t", [(1, 1, 1), (1, 2, 2), (2, 5, 1), (2, 5, 2), (1, 5, 2)])
def test_finite_difference_gradients(b, s, t):
    shape = LayerShape(b, s, 8, 2, 16, t)
    P, x, dy = _tiny_inputs(shape)
    assert fd_max_rel_error(shape, P, x, dy) < 1e-6


# --------------------------------------------------------------------------
# Independent library routines (torch float64, autograd)
# --------------------------------------------------------------------------

def torch_layer(shape, P, x, dy):
    """The same layer composed from torch's own routines, with autograd."""
    tp = {k: torch.tensor(v, dtype=torch.float64, requires_grad=True) for k, v in P.items()}
    tx = torch.tensor(x, dtype=torch.float64, requires_grad=True)
    b, s, h = x.shape
    H, d, a = shape.heads, shape.d, shape.a
    F = torch.nn.functional
    ln1 = F.layer_norm(tx, (h,), tp["ln1_g"], tp["ln1_b"], eps=L.LN_EPS)
    qkv = F.linear(ln1, tp["w_qkv"], tp["b_qkv"])
    q, k, v = qkv.split(a, dim=-1)

    def heads(z):
        return z.reshape(b, s, H, d).transpose(1, 2)

    o = F.scaled_dot_product_attention(heads(q), heads(k), heads(v), is_causal=True)
    o = o.transpose(1, 2).reshape(b, s, a)
    x1 = tx + F.linear(o, tp["w_o"], tp["b_o"])
    ln2 = F.layer_norm(x1, (h,), tp["ln2_g"], tp["ln2_b"], eps=L.LN_EPS)
    hmid = F.gelu(F.linear(ln2, tp["w_fc1"], tp["b_fc1"]), approximate="tanh")
    y = x1 + F.linear(hmid, tp["w_fc2"], tp["b_fc2"])
    (y * torch.tensor(dy)).sum().backward()
    return (y.detach().numpy(), tx.grad.numpy(), {k: v.grad.numpy() for k, v in tp.items()})


def torch_max_rel_error(shape, P, x, dy):
    y, dx, G = L.layer_forward_backward(shape, P, x, dy)
    ty, tdx, tG = torch_layer(shape, P, x, dy)
    errs = [_rel(y, ty), _rel(dx, tdx)] + [_rel(G[k], tG[k]) for k in G]
    return max(errs)


@pytest.mark.parametrize("shape", [
    LayerShape(1, 7, 16, 2, 32, 1),
    LayerShape(2, 9, 16, 4, 48, 2),
    LayerShape(1, 33, 64, 4, 128, 4),
    LayerShape(1, 17, 32, 2, 64, 1, head_dim=8),    # a = heads*head_dim != hidden
])
def test_matches_torch_library_routines(shape):
    P, x, dy = _tiny_inputs(shape, wstd=0.2)
    assert torch_max_rel_error(shape, P, x, dy) < 1e-10


def test_config1_shape_matches_torch():
    """The smallest benchmark configuration, default init, both tp values."""
    for t in (1, 2):
        shape = LayerShape(1, 128, 768, 12, 3072, t)
        inp = make_layer_inputs(shape)
        assert torch_max_rel_error(shape, inp.params_f64(), inp.f64("x"), inp.f64("dy")) < 1e-10


# --------------------------------------------------------------------------
# Brute-force attention
# --------------------------------------------------------------------------

def brute_attention(q, k, v):
    s, d = q.shape
    out = np.zeros_like(q)
    for i in range(s):
        scores = [sum(q[i, c] * k[j, c] for c in range(d)) / math.sqrt(d) for j in range(i + 1)]
        m = max(scores)
        w = [math.exp(z - m) for z in scores]
        tot = sum(w)
        for j in range(i + 1):
            out[i] += (w[j] / tot) * v[j]
    return out


def test_attention_brute_force():
    rng = np.random.default_rng(3)
    q, k, v = (rng.standard_normal((6, 4)) for _ in range(3))
    o, _ = L.causal_attention_forward(q, k, v)
    assert _rel(o, brute_attention(q, k, v)) < 1e-13


def test_attention_row_blocks_do_not_matter(monkeypatch):
    rng = np.random.default_rng(4)
    q, k, v, do = (rng.standard_normal((37, 8)) for _ in range(4))
    o, lse = L.causal_attention_forward(q, k, v)
    grads = L.causal_attention_backward(q, k, v, o, lse, do)
    monkeypatch.setattr(L, "_ATTN_ROW_BLOCK", 5)
    o2, lse2 = L.causal_attention_forward(q, k, v)
    grads2 = L.causal_attention_backward(q, k, v, o2, lse2, do)
    assert _rel(o2, o) < 1e-14 and _rel(lse2, lse) < 1e-14
    for g1, g2 in zip(grads, grads2):
        assert _rel(g2, g1) < 1e-13


# --------------------------------------------------------------------------
# Tensor-parallel invariance
# --------------------------------------------------------------------------

def test_partition_sum_equals_unpartitioned_product():
    rng = np.random.default_rng(5)
    o = rng.standard_normal((3, 11, 64))
    w = rng.standard_normal((32, 64))
    full = o @ w.T
    for t in (1, 2, 4, 8):
        shape = L.OracleShape(3, 11, 32, 8, 64, t, head_dim=8)
        acc = np.zeros_like(full)
        for p in range(t):
            cols = L.attn_cols(shape, p)
            acc += o[:, :, cols] @ w[:, cols].T
        assert _rel(acc, full) < 1e-12


def tp_invariance_error(shape, P, x, dy, tps=(1, 2, 4)):
    ref = L.layer_forward_backward(shape.with_tp(1), P, x, dy)
    worst = 0.0
    for t in tps:
        y, dx, G = L.layer_forward_backward(shape.with_tp(t), P, x, dy)
        worst = max([worst, _rel(y, ref[0]), _rel(dx, ref[1])] + [_rel(G[k], ref[2][k]) for k in G])
    return worst


def test_outputs_do_not_depend_on_tp_parts():
    shape = LayerShape(2, 6, 32, 4, 64, 1)
    P, x, dy = _tiny_inputs(shape, wstd=0.2)
    assert tp_invariance_error(shape, P, x, dy) < 1e-12


def test_partitions_cover_heads_and_ffn_exactly_once():
    shape = L.OracleShape(1, 1, 64, 8, 256, 4)
    rows = np.concatenate([L.qkv_rows(shape, p) for p in range(4)])
    assert np.array_equal(np.sort(rows), np.arange(3 * 64))
    cols = np.concatenate([np.arange(256)[L.ffn_cols(shape, p)] for p in range(4)])
    assert np.array_equal(cols, np.arange(256))


@pytest.mark.parametrize("hidden,heads,ffn,t", [(768, 12, 3072, 5), (768, 12, 3070, 4), (64, 3, 128, 2)])
def test_divisibility_rule_rejects(hidden, heads, ffn, t):
    with pytest.raises(ValueError):
        L.check_divisible(L.OracleShape(1, 1, hidden, heads, ffn, t))


# --------------------------------------------------------------------------
# Causality
# --------------------------------------------------------------------------

def test_causal_forward_rows_independent_of_future_tokens():
    shape = LayerShape(2, 9, 16, 2, 32, 2)
    P, x, dy = _tiny_inputs(shape)
    y, _ = L.layer_forward(shape, P, x)
    for i in (0, 3, 7):
        x2 = x.copy()
        x2[:, i + 1:, :] += np.random.default_rng(i).standard_normal(x2[:, i + 1:, :].shape)
        y2, _ = L.layer_forward(shape, P, x2)
        assert np.array_equal(y2[:, :i + 1], y[:, :i + 1])
        if i + 1 < shape.seq_len:
            assert not np.array_equal(y2[:, i + 1:], y[:, i + 1:])


def test_causal_gradient_vanishes_after_last_nonzero_upstream_row():
    shape = LayerShape(1, 8, 16, 2, 32, 1)
    P, x, dy = _tiny_inputs(shape)
    i = 4
    dy = dy.copy()
    dy[:, i + 1:, :] = 0.0
    _, dx, _ = L.layer_forward_backward(shape, P, x, dy)
    assert np.all(dx[:, i + 1:, :] == 0.0)
    assert np.any(dx[:, :i + 1, :] != 0.0)


# --------------------------------------------------------------------------
# Closed forms
# --------------------------------------------------------------------------

def test_single_token_attention_returns_value_row():
    rng = np.random.default_rng(6)
    q, k, v = (rng.standard_normal((1, 8)) for _ in range(3))
    o, lse = L.causal_attention_forward(q, k, v)
    assert np.array_equal(o, v)
    assert lse[0] == pytest.approx(float(q[0] @ k[0]) / math.sqrt(8), rel=1e-15)


def test_zero_scores_give_running_mean_of_values():
    rng = np.random.default_rng(7)
    v = rng.standard_normal((10, 4))
    k = rng.standard_normal((10, 4))
    o, lse = L.causal_attention_forward(np.zeros((10, 4)), k, v)
    running_mean = np.cumsum(v, axis=0) / np.arange(1, 11)[:, None]
    assert _rel(o, running_mean) < 1e-14
    assert np.allclose(lse, np.log(np.arange(1, 11)), rtol=0, atol=1e-14)


def test_constant_layernorm_row_gives_beta():
    x = np.full((3, 8), 0.75)
    beta = np.linspace(-1, 1, 8)
    out, _, _ = L.layernorm_forward(x, np.full(8, 2.0), beta)
    assert np.array_equal(out, np.broadcast_to(beta, (3, 8)))


def test_layernorm_worked_example():
    # x = (1, 2, 3, 4): mean 2.5, biased variance 1.25.
    out, _, rstd = L.layernorm_forward(np.array([1.0, 2.0, 3.0, 4.0]), np.ones(4), np.zeros(4))
    assert rstd[0] == pytest.approx(1.0 / math.sqrt(1.25 + 1e-5), rel=1e-15)
    assert out == pytest.approx(np.array([-1.5, -0.5, 0.5, 1.5]) / math.sqrt(1.25 + 1e-5), rel=1e-14)


def test_gelu_closed_forms():
    assert L.gelu_tanh(np.array(0.0)) == 0.0
    assert L.gelu_tanh_grad(np.array(0.0)) == 0.5
    assert L.gelu_tanh(np.array(10.0)) == 10.0
    assert abs(L.gelu_tanh(np.array(-10.0))) < 1e-30
    xs = np.linspace(-6, 6, 97)
    ref = torch.nn.functional.gelu(torch.tensor(xs), approximate="tanh").numpy()
    assert _rel(L.gelu_tanh(xs), ref) < 1e-15
    tx = torch.tensor(xs, requires_grad=True)
    torch.nn.functional.gelu(tx, approximate="tanh").sum().backward()
    assert _rel(L.gelu_tanh_grad(xs), tx.grad.numpy()) < 1e-14


def test_zero_weights_reduce_to_biases():
    shape = LayerShape(2, 5, 16, 2, 32, 2)
    P, x, _ = _tiny_inputs(shape)
    for w in ("w_qkv", "w_o", "w_fc1", "w_fc2"):
        P[w] = np.zeros_like(P[w])
    y, _ = L.layer_forward(shape, P, x)
    assert _rel(y, x + P["b_o"] + P["b_fc2"]) < 1e-15


# --------------------------------------------------------------------------
# Planted mistakes: every one must trip at least one pin above.
# --------------------------------------------------------------------------

def _pins_trip(shape_fd, shape_lib):
    P, x, dy = _tiny_inputs(shape_fd)
    fd = fd_max_rel_error(shape_fd, P, x, dy, n_probe=8)
    P2, x2, dy2 = _tiny_inputs(shape_lib, wstd=0.2)
    lib = torch_max_rel_error(shape_lib, P2, x2, dy2)
    return fd > 1e-6 or lib > 1e-10


_ORIG_LN_BWD = L.layernorm_backward
_ORIG_ATTN_FWD = L.causal_attention_forward
_ORIG_ATTN_BWD = L.causal_attention_backward


def _mut_gelu_grad_drop_term(x):
    th = np.tanh(L._GELU_C * (x + L._GELU_A * x ** 3))
    return 0.5 * (1.0 + th) + 0.5 * x * (1.0 - th * th) * L._GELU_C


def _mut_ln_unbiased(x, gamma, beta, eps=L.LN_EPS):
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).sum(axis=-1, keepdims=True) / (x.shape[-1] - 1)
    rstd = 1.0 / np.sqrt(var + eps)
    xhat = (x - mu) * rstd
    return xhat * gamma + beta, xhat, rstd


def _mut_ln_bwd_sign(dout, xhat, rstd, gamma):
    dx, dg, db = _ORIG_LN_BWD(dout, xhat, rstd, gamma)
    return dx + 2 * rstd * xhat * (dout * gamma * xhat).mean(axis=-1, keepdims=True), dg, db


def _mut_attn_anticausal(q, k, v):
    o, lse = _ORIG_ATTN_FWD(q[::-1].copy(), k[::-1].copy(), v[::-1].copy())
    return o[::-1].copy(), lse[::-1].copy()


def _mut_attn_bwd_transposed(q, k, v, o, lse, do):
    dq, dk, dv = _ORIG_ATTN_BWD(q, k, v, o, lse, do)
    return dk, dq, dv


@pytest.mark.parametrize("name,mutant", [
    ("gelu_tanh_grad", _mut_gelu_grad_drop_term),
    ("layernorm_forward", _mut_ln_unbiased),
    ("layernorm_backward", _mut_ln_bwd_sign),
    ("causal_attention_forward", _mut_attn_anticausal),
    ("causal_attention_backward", _mut_attn_bwd_transposed),
])
def test_planted_mistakes_are_caught(monkeypatch, name, mutant):
    monkeypatch.setattr(L, name, mutant)
    assert _pins_trip(LayerShape(1, 3, 8, 2, 16, 1), LayerShape(1, 5, 16, 2, 32, 1))


def test_planted_partition_mistake_is_caught(monkeypatch):
    """Adding the row-parallel bias once per partition breaks tp-invariance."""
    shape = LayerShape(1, 4, 16, 2, 32, 1)
    P, x, dy = _tiny_inputs(shape)
    real_forward = L.layer_forward

    def bias_per_partition(shape_, P_, x_):
        y, cache = real_forward(shape_, P_, x_)
        return y + (shape_.tp_parts - 1) * P_["b_fc2"], cache

    monkeypatch.setattr(L, "layer_forward", bias_per_partition)
    assert tp_invariance_error(shape, P, x, dy, tps=(1, 2)) > 1e-6


# --------------------------------------------------------------------------
# Sampled outputs (used for sequences too long for the full oracle)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("shape,rows,tail", [
    (LayerShape(2, 23, 16, 2, 32, 1), [0, 5, 22], 4),
    (LayerShape(1, 40, 32, 4, 64, 2), [3, 39], 7),
    (LayerShape(1, 9, 16, 2, 32, 1), [8], 9),        # tail = whole sequence
])
def test_sampled_rows_and_tail_match_full_oracle(shape, rows, tail):
    from oracle.sampled import sampled_rows_and_tail
    P, x, dy = _tiny_inputs(shape, wstd=0.2)
    y, dx, _ = L.layer_forward_backward(shape, P, x, dy)
    ys, dxs = sampled_rows_and_tail(shape, P, x, dy, rows, tail)
    assert _rel(ys, y[:, rows]) < 1e-12
    assert _rel(dxs, dx[:, -tail:]) < 1e-12
