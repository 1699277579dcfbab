"""Context-parallel attention on the GPU against the fp64 oracle and against
the fused kernels: forward (O, LSE) and backward (dQ, dK, dV) for several
cp_parts, head dims and micro-batches; bitwise repeatable."""
import numpy as np
import pytest
import torch

import oracle.layer as O
from layer_inputs import bf16_bits_to_f64
from megatron_transformer_layer_gb300 import _lib as L
from parity import assert_close

from gpu_util import DEV, bits, check_status, dev_bf16, status, to_f64

pytestmark = pytest.mark.gpu


def _oracle(q64, do64, b, s, H, d, heads=None):
    a = H * d
    o = np.zeros((b, s, a))
    lse = np.zeros((b, H, s))
    g = np.zeros((b, s, 3 * a))
    for bi in range(b):
        for hh in (range(H) if heads is None else heads):
            cq = slice(hh * d, (hh + 1) * d)
            ck, cv = slice(a + hh * d, a + (hh + 1) * d), slice(2 * a + hh * d, 2 * a + (hh + 1) * d)
            q, k, v = q64[bi, :, cq], q64[bi, :, ck], q64[bi, :, cv]
            o[bi, :, cq], lse[bi, hh] = O.causal_attention_forward(q, k, v)
            g[bi, :, cq], g[bi, :, ck], g[bi, :, cv] = O.causal_attention_backward(
                q, k, v, o[bi, :, cq], lse[bi, hh], do64[bi, :, cq])
    return o, lse, g


def _run_cp(qb, dob, b, s, H, d, cp):
    a = H * d
    qkv, dout = dev_bf16(qb), dev_bf16(dob)
    nbytes = L.mc_attention_cp_workspace_bytes(b, s, H, d, cp)
    assert nbytes > 0
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    o = torch.empty(b * s * a, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(b * H * s, dtype=torch.float32, device=DEV)
    dqkv = torch.full((b * s * 3 * a,), float("nan"), dtype=torch.bfloat16, device=DEV)
    delta = torch.empty(b * H * s, dtype=torch.float32, device=DEV)
    st = status()
    assert L.mc_attention_forward_cp(qkv, o, lse, b, s, H, d, cp, ws, nbytes, st) == 0
    assert L.mc_attention_backward_cp(qkv, o, lse, dout, dqkv, delta, b, s, H, d, cp, ws,
                                      nbytes, st) == 0
    check_status(st)
    return o, lse, dqkv


@pytest.mark.parametrize("b,s,H,d,cp", [(1, 1024, 2, 128, 2), (2, 1024, 3, 64, 4),
                                        (1, 768, 2, 128, 3), (1, 512, 1, 128, 1)])
def test_cp_attention_matches_oracle(b, s, H, d, cp):
    a = H * d
    qb = bits(b * s * 3 * a, 40, std=1.8)
    dob = bits(b * s * a, 41)
    q64 = bf16_bits_to_f64(qb).reshape(b, s, 3 * a)
    do64 = bf16_bits_to_f64(dob).reshape(b, s, a)
    o_ref, lse_ref, g_ref = _oracle(q64, do64, b, s, H, d)
    o, lse, dqkv = _run_cp(qb, dob, b, s, H, d, cp)
    assert_close(f"cp{cp} o", to_f64(o).reshape(b, s, a), o_ref)
    assert_close(f"cp{cp} lse", to_f64(lse).reshape(b, H, s), lse_ref, 1e-4, 1e-5)
    got = to_f64(dqkv).reshape(b, s, 3 * a)
    for name, sl in (("dq", slice(0, a)), ("dk", slice(a, 2 * a)), ("dv", slice(2 * a, 3 * a))):
        assert_close(f"cp{cp} {name}", got[:, :, sl], g_ref[:, :, sl])
    # bitwise repeatable
    o2, lse2, dqkv2 = _run_cp(qb, dob, b, s, H, d, cp)
    assert torch.equal(o, o2) and torch.equal(lse, lse2) and torch.equal(dqkv, dqkv2)


def test_cp_attention_long_sequence_against_fused_and_oracle():
    """s = 4096, 8 heads, cp = 4 (chunks of 512): every element close to the
    fused kernels' result; two heads against the oracle."""
    b, s, H, d, cp = 1, 4096, 8, 128, 4
    a = H * d
    qb = bits(b * s * 3 * a, 42, std=1.8)
    dob = bits(b * s * a, 43)
    o, lse, dqkv = _run_cp(qb, dob, b, s, H, d, cp)
    qkv, dout = dev_bf16(qb), dev_bf16(dob)
    of = torch.empty_like(o)
    lf = torch.empty_like(lse)
    gf = torch.empty_like(dqkv)
    delta = torch.empty_like(lse)
    st = status()
    assert L.mc_attention_forward(qkv, of, lf, b, s, H, d, st) == 0
    assert L.mc_attention_backward(qkv, of, lf, dout, gf, delta, b, s, H, d, st) == 0
    check_status(st)
    assert_close("cp vs fused o", to_f64(o), to_f64(of))
    assert_close("cp vs fused lse", to_f64(lse), to_f64(lf), 1e-4, 1e-5)
    assert_close("cp vs fused dqkv", to_f64(dqkv), to_f64(gf))
    q64 = bf16_bits_to_f64(qb).reshape(b, s, 3 * a)
    do64 = bf16_bits_to_f64(dob).reshape(b, s, a)
    heads = (0, 5)
    o_ref, _, g_ref = _oracle(q64, do64, b, s, H, d, heads)
    og = to_f64(o).reshape(b, s, a)
    gg = to_f64(dqkv).reshape(b, s, 3 * a)
    for hh in heads:
        cs = [slice(k * a + hh * d, k * a + (hh + 1) * d) for k in range(3)]
        assert_close(f"cp o head {hh}", og[:, :, cs[0]], o_ref[:, :, cs[0]])
        for name, c in zip(("dq", "dk", "dv"), cs):
            assert_close(f"cp {name} head {hh}", gg[:, :, c], g_ref[:, :, c])


@pytest.mark.parametrize("d", [64, 128])
def test_cp_single_pair_chunks_equal_fused_bitwise(d):
    """A chunk whose result comes from one chunk pair is computed by the same
    blocks in the same order as in the fused kernels, so it matches them bit
    for bit: O and LSE of chunk 0 (its only pair is the diagonal one), and,
    given the same O and LSE, dQ of chunk 0 and dK, dV of the last chunk."""
    b, s, H, cp = 1, 2048, 3, 2
    a, c = H * d, s // (2 * cp)
    qb = bits(b * s * 3 * a, 44, std=1.8)
    dob = bits(b * s * a, 45)
    o, lse, dqkv = _run_cp(qb, dob, b, s, H, d, cp)
    qkv, dout = dev_bf16(qb), dev_bf16(dob)
    of, lf = torch.empty_like(o), torch.empty_like(lse)
    st = status()
    assert L.mc_attention_forward(qkv, of, lf, b, s, H, d, st) == 0
    nbytes = L.mc_attention_backward_ws_bytes(b, s, H, d)
    ds = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    gf = torch.full_like(dqkv, float("nan"))
    delta = torch.empty_like(lse)
    # the fused backward from the context-parallel forward's O and LSE
    assert L.mc_attention_backward_ws(qkv, o, lse, dout, gf, delta, b, s, H, d, ds, nbytes,
                                      st) == 0
    check_status(st)
    assert torch.equal(o.view(s, a)[:c], of.view(s, a)[:c])
    assert torch.equal(lse.view(H, s)[:, :c], lf.view(H, s)[:, :c])
    g, gfv = dqkv.view(s, 3 * a), gf.view(s, 3 * a)
    assert torch.equal(g[:c, :a], gfv[:c, :a])
    assert torch.equal(g[s - c:, a:], gfv[s - c:, a:])
    # and the rest agrees to rounding
    assert_close("cp vs fused dqkv", to_f64(dqkv), to_f64(gf))
