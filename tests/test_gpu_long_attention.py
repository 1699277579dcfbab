"""Causal attention at the long-sequence configuration's full length
(s = 32768, head_dim 128) against the fp64 oracle, every element.

Two heads run through the fused forward and backward kernels: O, LSE, dQ, dK
and dV are compared element by element with the oracle (so dK and dV of the
earliest keys, the backward kernel's longest loops over 256 query blocks, and
dQ of the middle rows are all checked), and a second run must give the same
bits.  The context-parallel path (cp = 4, chunks of 4096 tokens) is compared
with the same oracle."""
import numpy as np
import pytest
import torch

import oracle.layer as O
from layer_inputs import bf16_bits_to_f64
from megatron_transformer_layer_gb300 import _lib as L
from parity import assert_close

from gpu_util import DEV, bits, check_status, dev_bf16, status, to_f64

pytestmark = pytest.mark.gpu

B, S, H, D = 1, 32768, 2, 128
A = H * D


@pytest.fixture(scope="module")
def case():
    qb = bits(B * S * 3 * A, 61, std=1.8)
    dob = bits(B * S * A, 62)
    q64 = bf16_bits_to_f64(qb).reshape(S, 3 * A)
    do64 = bf16_bits_to_f64(dob).reshape(S, A)
    ref = {}
    for hh in range(H):
        q, k, v = (q64[:, j * A + hh * D:j * A + (hh + 1) * D] for j in range(3))
        o, lse = O.causal_attention_forward(q, k, v)
        dq, dk, dv = O.causal_attention_backward(q, k, v, o, lse, do64[:, hh * D:(hh + 1) * D])
        ref[hh] = dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv)
    return qb, dob, ref


def _compare(label, o, lse, dqkv, ref):
    o = to_f64(o).reshape(S, A)
    lse = to_f64(lse).reshape(H, S)
    g = to_f64(dqkv).reshape(S, 3 * A)
    for hh in range(H):
        r = ref[hh]
        assert_close(f"{label} o head {hh}", o[:, hh * D:(hh + 1) * D], r["o"])
        assert_close(f"{label} lse head {hh}", lse[hh], r["lse"], 1e-4, 1e-5)
        for j, name in enumerate(("dq", "dk", "dv")):
            got = g[:, j * A + hh * D:j * A + (hh + 1) * D]
            assert_close(f"{label} {name} head {hh}", got, r[name])
            # the first and middle blocks on their own, so that an error
            # confined to the longest loops is not averaged away
            for rows in (slice(0, 128), slice(S // 2 - 64, S // 2 + 64)):
                assert_close(f"{label} {name} head {hh} rows {rows}", got[rows], r[name][rows])


def _fused(qkv, dout):
    o = torch.empty(B * S * A, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(B * H * S, dtype=torch.float32, device=DEV)
    dqkv = torch.full((B * S * 3 * A,), float("nan"), dtype=torch.bfloat16, device=DEV)
    delta = torch.empty(B * H * S, dtype=torch.float32, device=DEV)
    st = status()
    assert L.mc_attention_forward(qkv, o, lse, B, S, H, D, st) == 0
    assert L.mc_attention_backward(qkv, o, lse, dout, dqkv, delta, B, S, H, D, st) == 0
    check_status(st)
    return o, lse, dqkv


def test_fused_attention_full_length_every_element(case):
    qb, dob, ref = case
    qkv, dout = dev_bf16(qb), dev_bf16(dob)
    first = _fused(qkv, dout)
    second = _fused(qkv, dout)
    for x, y in zip(first, second):
        assert torch.equal(x, y)
    _compare("fused s32768", *first, ref)


def test_ds_tile_backward_full_length_every_element(case):
    """The backward the layer calls (dQ from the dK/dV kernel's dS tiles,
    256 x 257 / 2 tiles per head, 2.1 GB here) at s = 32768: every element
    against the oracle, bitwise repeatable, dK and dV equal to the
    two-kernel path's."""
    qb, dob, ref = case
    qkv, dout = dev_bf16(qb), dev_bf16(dob)
    o, lse, base = _fused(qkv, dout)
    nbytes = L.mc_attention_backward_ws_bytes(B, S, H, D)
    ws = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device=DEV)
    delta = torch.empty(B * H * S, dtype=torch.float32, device=DEV)
    st = status()
    runs = []
    for _ in range(2):
        dqkv = torch.full((B * S * 3 * A,), float("nan"), dtype=torch.bfloat16, device=DEV)
        assert L.mc_attention_backward_ws(qkv, o, lse, dout, dqkv, delta, B, S, H, D, ws, nbytes,
                                          st) == 0
        check_status(st)
        runs.append(dqkv)
    assert torch.equal(runs[0], runs[1])
    assert torch.equal(runs[0].view(S, 3 * A)[:, A:], base.view(S, 3 * A)[:, A:])
    _compare("dS tiles s32768", o, lse, runs[0], ref)


def test_context_parallel_attention_full_length(case):
    qb, dob, ref = case
    cp = 4
    qkv, dout = dev_bf16(qb), dev_bf16(dob)
    nbytes = L.mc_attention_cp_workspace_bytes(B, S, H, D, cp)
    assert nbytes > 0
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    o = torch.empty(B * S * A, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(B * H * S, dtype=torch.float32, device=DEV)
    dqkv = torch.full((B * S * 3 * A,), float("nan"), dtype=torch.bfloat16, device=DEV)
    delta = torch.empty(B * H * S, dtype=torch.float32, device=DEV)
    st = status()
    assert L.mc_attention_forward_cp(qkv, o, lse, B, S, H, D, cp, ws, nbytes, st) == 0
    assert L.mc_attention_backward_cp(qkv, o, lse, dout, dqkv, delta, B, S, H, D, cp, ws,
                                      nbytes, st) == 0
    check_status(st)
    assert np.isfinite(to_f64(dqkv)).all()
    _compare("cp4 s32768", o, lse, dqkv, ref)
