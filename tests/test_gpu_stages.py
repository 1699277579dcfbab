"""Stage parity: each kernel alone, on generator inputs, against the oracle's
functions (fp64).  All calls go through the C ABI."""
import numpy as np
import pytest
import torch

import oracle.layer as O
from layer_inputs import bf16_bits_to_f64
from megatron_transformer_layer_gb300 import _lib as L
from parity import assert_close

from gpu_util import DEV, bits, check_status, dev_bf16, dev_f32_from_bits, status, to_f64

pytestmark = pytest.mark.gpu


# ---------------------------------------------------------------- LayerNorm
@pytest.mark.parametrize("rows,h", [(1, 768), (37, 768), (300, 2048), (64, 8192), (5, 4096)])
def test_layernorm_forward(rows, h):
    xb, gb, bb = bits(rows * h, 1), bits(h, 2, mean=1.0, std=0.1), bits(h, 3, std=0.1)
    x64, g64, b64 = (bf16_bits_to_f64(v) for v in (xb, gb, bb))
    ref, xhat, rstd = O.layernorm_forward(x64.reshape(rows, h), g64, b64)
    x = dev_f32_from_bits(xb)
    out = torch.empty(rows * h, dtype=torch.bfloat16, device=DEV)
    mean = torch.empty(rows, dtype=torch.float32, device=DEV)
    rs = torch.empty(rows, dtype=torch.float32, device=DEV)
    st = status()
    assert L.mc_layernorm_forward(x, dev_bf16(gb), dev_bf16(bb), out, mean, rs, rows, h, st) == 0
    check_status(st)
    assert_close("ln_out", to_f64(out).reshape(rows, h), ref)
    assert_close("mean", to_f64(mean), x64.reshape(rows, h).mean(axis=1), 1e-5, 1e-6)
    assert_close("rstd", to_f64(rs), rstd[:, 0], 1e-5, 1e-6)


@pytest.mark.parametrize("rows,h,accumulate", [(1, 768, 0), (129, 768, 1), (700, 2048, 0),
                                               (33, 4096, 0), (40, 8192, 0),
                                               # more rows than one wave of CTAs at h = 8192
                                               (1000, 8192, 1)])
def test_layernorm_backward(rows, h, accumulate):
    xb, gb, bb = bits(rows * h, 4), bits(h, 5, mean=1.0, std=0.1), bits(h, 6, std=0.1)
    db, rb = bits(rows * h, 7), bits(rows * h, 8)
    x64, g64, b64, d64, r64 = (bf16_bits_to_f64(v) for v in (xb, gb, bb, db, rb))
    x64, d64, r64 = (v.reshape(rows, h) for v in (x64, d64, r64))
    _, xhat, rstd = O.layernorm_forward(x64, g64, b64)
    dxr, dgr, dbr = O.layernorm_backward(d64, xhat, rstd, g64)
    dxr = dxr + r64
    x = dev_f32_from_bits(xb)
    mean = torch.from_numpy(x64.mean(axis=1).astype(np.float32)).to(DEV)
    rs = torch.from_numpy(rstd[:, 0].astype(np.float32)).to(DEV)
    dx = torch.empty(rows * h, dtype=torch.float32, device=DEV)
    dx16 = torch.empty(rows * h, dtype=torch.bfloat16, device=DEV)
    init = 0.5 if accumulate else 0.0
    dgam = torch.full((h,), init, device=DEV)
    dbet = torch.full((h,), init, device=DEV)
    csum = torch.full((h,), init, device=DEV)
    part = torch.empty(L.mc_layernorm_backward_scratch_floats(rows, h), device=DEV)
    st = status()
    assert L.mc_layernorm_backward(dev_f32_from_bits(db), x, mean, rs, dev_bf16(gb),
                                   dev_f32_from_bits(rb), dx, dx16, dgam, dbet, csum, accumulate,
                                   part, rows, h, st) == 0
    check_status(st)
    assert_close("dx", to_f64(dx).reshape(rows, h), dxr)
    assert_close("dx_bf16", to_f64(dx16).reshape(rows, h), dxr)
    assert_close("dgamma", to_f64(dgam) - init, dgr)
    assert_close("dbeta", to_f64(dbet) - init, dbr)
    assert_close("colsum_dx", to_f64(csum) - init, dxr.sum(axis=0))


# ---------------------------------------------------------------- GEMM
def _gemm_case(M, N, K, a_layout, b_layout, epi, k_parts=1, accumulate=0, seed=0):
    ab = bits(M * K, 10 + seed)
    bb = bits(N * K, 11 + seed, std=0.05)
    a = bf16_bits_to_f64(ab).reshape((M, K) if a_layout == 0 else (K, M))
    b = bf16_bits_to_f64(bb).reshape((N, K) if b_layout == 0 else (K, N))
    A = a if a_layout == 0 else a.T
    B = b if b_layout == 0 else b.T
    acc = A @ B.T
    biasb = bits(N, 12 + seed, std=0.5)
    bias64 = bf16_bits_to_f64(biasb)
    auxb = bits(M * N, 13 + seed)
    aux64 = bf16_bits_to_f64(auxb).reshape(M, N)
    lda = K if a_layout == 0 else M
    ldb = K if b_layout == 0 else N
    dA, dB = dev_bf16(ab), dev_bf16(bb)
    st = status()
    f32_out = epi in (L.MC_EPI_STORE_F32, L.MC_EPI_BIAS_RESID_F32)
    out = torch.zeros(M * N, dtype=torch.float32 if f32_out else torch.bfloat16, device=DEV)
    if accumulate:
        out += 0.25
    aux = None
    if epi == L.MC_EPI_BIAS_GELU:
        aux = torch.empty(M * N, dtype=torch.bfloat16, device=DEV)
    elif epi == L.MC_EPI_BIAS_RESID_F32:
        aux = dev_f32_from_bits(auxb)
    elif epi == L.MC_EPI_GELU_BWD:
        aux = dev_bf16(auxb)
    rc = L.mc_gemm(M, N, K, dA, lda, a_layout, dB, ldb, b_layout, out, N, epi,
                   bias=dev_bf16(biasb), aux=aux, ldaux=N, accumulate=accumulate,
                   k_parts=k_parts, status=st)
    assert rc == 0, L.mc_strerror(rc)
    check_status(st)
    got = to_f64(out).reshape(M, N)
    if epi == L.MC_EPI_STORE_F32:
        ref = acc + (0.25 if accumulate else 0.0)
    elif epi == L.MC_EPI_STORE_BF16:
        ref = acc
    elif epi == L.MC_EPI_BIAS_BF16:
        ref = acc + bias64
    elif epi == L.MC_EPI_BIAS_GELU:
        assert_close("gemm_hp", to_f64(aux).reshape(M, N), acc + bias64)
        ref = O.gelu_tanh(acc + bias64)
    elif epi == L.MC_EPI_BIAS_RESID_F32:
        ref = acc + bias64 + aux64
    else:
        ref = acc * O.gelu_tanh_grad(aux64)
    assert_close(f"gemm epi={epi}", got, ref)


@pytest.mark.parametrize("a_layout,b_layout", [(0, 0), (0, 1), (1, 1), (1, 0)])
def test_gemm_store_f32_layouts(a_layout, b_layout):
    # A stored [K, M] has the token count as K, which may be ragged; a K-major B
    # still needs a row stride that is a multiple of 8 elements.
    K = 192 if a_layout == 0 else (100 if b_layout == 1 else 104)
    _gemm_case(200, 320, K, a_layout, b_layout, L.MC_EPI_STORE_F32)


@pytest.mark.parametrize("epi", [L.MC_EPI_STORE_BF16, L.MC_EPI_BIAS_BF16, L.MC_EPI_BIAS_GELU,
                                 L.MC_EPI_BIAS_RESID_F32, L.MC_EPI_GELU_BWD])
def test_gemm_epilogues(epi):
    _gemm_case(130, 192, 128, 0, 0, epi)


def test_gemm_accumulate_and_partitions():
    _gemm_case(64, 128, 100, 1, 1, L.MC_EPI_STORE_F32, accumulate=1)
    _gemm_case(256, 256, 512, 0, 0, L.MC_EPI_STORE_F32, k_parts=4)


@pytest.mark.parametrize("a_layout,b_layout", [(0, 0), (0, 1), (1, 1), (1, 0)])
def test_gemm_wide_tiles(a_layout, b_layout):
    # Enough 128x256 tiles to select the wide-tile variant, which runs on SM
    # pairs (256 x 256 per pair); ragged M.
    _gemm_case(2000, 2560, 256, a_layout, b_layout, L.MC_EPI_STORE_F32, seed=3)


@pytest.mark.parametrize("epi", [L.MC_EPI_STORE_BF16, L.MC_EPI_BIAS_BF16, L.MC_EPI_BIAS_GELU,
                                 L.MC_EPI_BIAS_RESID_F32, L.MC_EPI_GELU_BWD])
def test_gemm_paired_tiles_odd_m_tiles(epi):
    # 17 M-tiles: the last pair's second half lies wholly past M.
    _gemm_case(2100, 2304, 192, 0, 1 if epi == L.MC_EPI_GELU_BWD else 0, epi, seed=4)


def test_gemm_paired_tiles_partitions_and_accumulate():
    _gemm_case(1152, 4608, 512, 0, 0, L.MC_EPI_BIAS_RESID_F32, k_parts=8, seed=5)
    _gemm_case(2048, 2560, 300, 1, 1, L.MC_EPI_STORE_F32, accumulate=1, seed=6)


# ---------------------------------------------------------------- attention
def _qkv_case(b, s, H, d, seed=0):
    a = H * d
    qb = bits(b * s * 3 * a, 20 + seed)
    q64 = bf16_bits_to_f64(qb).reshape(b, s, 3 * a)
    return qb, q64


def _oracle_attention(q64, b, s, H, d, do64=None):
    a = H * d
    o = np.empty((b, s, a))
    lse = np.empty((b, H, s))
    grads = np.empty((b, s, 3 * a)) if do64 is not None else None
    for bi in range(b):
        for hh in range(H):
            c = slice(hh * d, (hh + 1) * d)
            q, k, v = q64[bi, :, c], q64[bi, :, a + hh * d:a + (hh + 1) * d], \
                q64[bi, :, 2 * a + hh * d:2 * a + (hh + 1) * d]
            o[bi, :, c], lse[bi, hh] = O.causal_attention_forward(q, k, v)
            if do64 is not None:
                dq, dk, dv = O.causal_attention_backward(q, k, v, o[bi, :, c], lse[bi, hh],
                                                         do64[bi, :, c])
                grads[bi, :, c] = dq
                grads[bi, :, a + hh * d:a + (hh + 1) * d] = dk
                grads[bi, :, 2 * a + hh * d:2 * a + (hh + 1) * d] = dv
    return o, lse, grads


@pytest.mark.parametrize("b,s,H,d", [(1, 1, 1, 64), (2, 7, 3, 64), (1, 129, 2, 128),
                                     (2, 300, 2, 64), (1, 520, 2, 128),
                                     # (token, head) rows of the delta pass: a ragged last block
                                     (1, 1000, 3, 64)])
def test_attention_forward_backward(b, s, H, d):
    a = H * d
    qb, q64 = _qkv_case(b, s, H, d)
    dob = bits(b * s * a, 30)
    do64 = bf16_bits_to_f64(dob).reshape(b, s, a)
    o_ref, lse_ref, g_ref = _oracle_attention(q64, b, s, H, d, do64)
    qkv = dev_bf16(qb)
    o = torch.empty(b * s * a, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(b * H * s, dtype=torch.float32, device=DEV)
    st = status()
    assert L.mc_attention_forward(qkv, o, lse, b, s, H, d, st) == 0
    check_status(st)
    assert_close("attn_o", to_f64(o).reshape(b, s, a), o_ref)
    assert_close("attn_lse", to_f64(lse).reshape(b, H, s), lse_ref, 1e-4, 1e-5)
    dqkv = torch.full((b * s * 3 * a,), float("nan"), dtype=torch.bfloat16, device=DEV)
    delta = torch.empty(b * H * s, dtype=torch.float32, device=DEV)
    assert L.mc_attention_backward(qkv, o, lse, dev_bf16(dob), dqkv, delta, b, s, H, d, st) == 0
    check_status(st)
    got = to_f64(dqkv).reshape(b, s, 3 * a)
    for name, sl in (("dq", slice(0, a)), ("dk", slice(a, 2 * a)), ("dv", slice(2 * a, 3 * a))):
        assert_close(name, got[:, :, sl], g_ref[:, :, sl])
    # the backward the layer calls: dQ from the dK/dV kernel's dS tiles.  The
    # workspace starts as all-NaN bytes, so a tile read before it was written
    # would poison dQ.
    nbytes = L.mc_attention_backward_ws_bytes(b, s, H, d)
    nb = (s + 127) // 128
    assert nbytes == b * H * nb * (nb + 1) // 2 * 128 * 128 * 2
    ws = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device=DEV)
    dqkv2 = torch.full((b * s * 3 * a,), float("nan"), dtype=torch.bfloat16, device=DEV)
    assert L.mc_attention_backward_ws(qkv, o, lse, dev_bf16(dob), dqkv2, delta, b, s, H, d, ws,
                                      nbytes, st) == 0
    check_status(st)
    got2 = to_f64(dqkv2).reshape(b, s, 3 * a)
    for name, sl in (("dq", slice(0, a)), ("dk", slice(a, 2 * a)), ("dv", slice(2 * a, 3 * a))):
        assert_close(name + " (dS tiles)", got2[:, :, sl], g_ref[:, :, sl])
    # dK, dV come from the same kernel either way
    assert torch.equal(dqkv2.view(b, s, 3 * a)[:, :, a:], dqkv.view(b, s, 3 * a)[:, :, a:])


def test_attention_long_sequence_many_heads():
    """s = 4096 with 64 heads (the 96-layer GPT's shard shape): 32 key blocks
    per heaviest tile and every SM busy, where the last products of a tile can
    trail its softmax.  Bitwise-repeatable over three runs, and sampled heads
    equal to the oracle."""
    b, s, H, d = 1, 4096, 64, 128
    a = H * d
    qb = bits(b * s * 3 * a, 21, std=1.8)
    q64 = bf16_bits_to_f64(qb).reshape(b, s, 3 * a)
    dob = bits(b * s * a, 31)
    qkv, dout = dev_bf16(qb), dev_bf16(dob)
    runs = []
    for _ in range(3):
        o = torch.empty(b * s * a, dtype=torch.bfloat16, device=DEV)
        lse = torch.empty(b * H * s, dtype=torch.float32, device=DEV)
        dqkv = torch.empty(b * s * 3 * a, dtype=torch.bfloat16, device=DEV)
        delta = torch.empty(b * H * s, dtype=torch.float32, device=DEV)
        st = status()
        assert L.mc_attention_forward(qkv, o, lse, b, s, H, d, st) == 0
        assert L.mc_attention_backward(qkv, o, lse, dout, dqkv, delta, b, s, H, d, st) == 0
        check_status(st)
        runs.append((o, lse, dqkv))
    for o, lse, dqkv in runs[1:]:
        assert torch.equal(o, runs[0][0]) and torch.equal(lse, runs[0][1])
        assert torch.equal(dqkv, runs[0][2])
    # the layer's backward (dQ from dS tiles): repeatable, dK and dV equal to
    # the two-kernel path's, dQ checked on the sampled heads below
    nbytes = L.mc_attention_backward_ws_bytes(b, s, H, d)
    ws = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device=DEV)
    tiled = []
    for _ in range(2):
        dq2 = torch.full((b * s * 3 * a,), float("nan"), dtype=torch.bfloat16, device=DEV)
        delta = torch.empty(b * H * s, dtype=torch.float32, device=DEV)
        st = status()
        assert L.mc_attention_backward_ws(qkv, runs[0][0], runs[0][1], dout, dq2, delta, b, s, H,
                                          d, ws, nbytes, st) == 0
        check_status(st)
        tiled.append(dq2)
    assert torch.equal(tiled[0], tiled[1])
    assert torch.equal(tiled[0].view(s, 3 * a)[:, a:], runs[0][2].view(s, 3 * a)[:, a:])
    g2 = to_f64(tiled[0]).reshape(s, 3 * a)
    o = to_f64(runs[0][0]).reshape(s, a)
    g = to_f64(runs[0][2]).reshape(s, 3 * a)
    do64 = bf16_bits_to_f64(dob).reshape(s, a)
    for hh in (0, 9, 40, 63):
        c = slice(hh * d, (hh + 1) * d)
        ck, cv = slice(a + hh * d, a + (hh + 1) * d), slice(2 * a + hh * d, 2 * a + (hh + 1) * d)
        q, k, v = q64[0, :, c], q64[0, :, ck], q64[0, :, cv]
        o_ref, lse_ref = O.causal_attention_forward(q, k, v)
        assert_close(f"attn_o head {hh}", o[:, c], o_ref)
        dq, dk, dv = O.causal_attention_backward(q, k, v, o_ref, lse_ref, do64[:, c])
        assert_close(f"dq head {hh}", g[:, c], dq)
        assert_close(f"dq head {hh} (dS tiles)", g2[:, c], dq)
        assert_close(f"dk head {hh}", g[:, ck], dk)
        assert_close(f"dv head {hh}", g[:, cv], dv)


def test_bounded_wait_reports_timeout_and_context_survives():
    """Failure detection on the GPU without a fault: a wait on a barrier that
    nothing arrives on gives up after its limit, the status word says
    MC_ERR_DEVICE_TIMEOUT at the self-test site, and the next launches run."""
    st = status()
    assert L.mc_selftest_wait_timeout(2_000_000, st) == 0  # 2 ms
    torch.cuda.synchronize()
    assert int(st[0].item()) == L.MC_ERR_DEVICE_TIMEOUT and int(st[1].item()) == 30
    assert L.mc_selftest_wait_timeout(10**9, st) == L.MC_ERR_ARGUMENT  # limits capped
    _gemm_case(130, 192, 128, 0, 0, L.MC_EPI_STORE_BF16)  # the context still works
