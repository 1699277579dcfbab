"""Pins of the E4M3 / E5M2 oracle (oracle/fp8.py) against the formats'
definitions: fixed points of the encodings, exhaustive round trips, ties to
even, saturation, brute-force nearest values, and the scaling reading."""
import numpy as np
import pytest

from oracle import fp8 as F


@pytest.mark.parametrize("fmt,byte,value", [
    ("e4m3", 0x7E, 448.0), ("e4m3", 0x01, 2.0 ** -9), ("e4m3", 0x08, 2.0 ** -6),
    ("e4m3", 0x38, 1.0), ("e4m3", 0xC0, -2.0), ("e4m3", 0x3C, 1.5), ("e4m3", 0x00, 0.0),
    ("e5m2", 0x7B, 57344.0), ("e5m2", 0x01, 2.0 ** -16), ("e5m2", 0x04, 2.0 ** -14),
    ("e5m2", 0x3C, 1.0), ("e5m2", 0xBE, -1.5), ("e5m2", 0x40, 2.0),
])
def test_fixed_points_of_the_encodings(fmt, byte, value):
    assert F.decode(np.array([byte]), fmt)[0] == value
    assert F.encode(np.array([value]), fmt)[0] == byte


def _finite_bytes(fmt):
    b = np.arange(256, dtype=np.uint8)
    if fmt == "e4m3":  # S.1111.111 is NaN
        return b[(b & 0x7F) != 0x7F]
    return b[(b & 0x7C) != 0x7C]  # E5M2 exponent 11111: infinities and NaNs


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_every_finite_byte_round_trips(fmt):
    b = _finite_bytes(fmt)
    assert np.array_equal(F.encode(F.decode(b, fmt), fmt), b)
    assert np.array_equal(F.round_fp8(F.decode(b, fmt), fmt), F.decode(b, fmt))


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_rounding_is_to_the_nearest_value_ties_to_even(fmt):
    vals = np.unique(F.decode(_finite_bytes(fmt), fmt))
    rng = np.random.default_rng(0)
    fmax = F.FORMATS[fmt][2]
    x = np.concatenate([rng.uniform(-fmax, fmax, 4000),
                        rng.standard_normal(4000) * 2.0 ** rng.integers(-18, 4, 4000)])
    r = F.round_fp8(x, fmt)
    d = np.abs(x[:, None] - vals[None, :])
    best = d.min(axis=1)
    assert np.array_equal(np.abs(x - r), best)  # r is a nearest value
    # ties: the midpoints between neighbours go to the one with the even mantissa
    mids = (vals[1:] + vals[:-1]) / 2
    rm = F.round_fp8(mids, fmt)
    codes = F.encode(rm, fmt)
    assert np.all((codes & 1) == 0)


def test_specific_roundings():
    e = lambda v: F.round_fp8(np.array([v]), "e4m3")[0]  # noqa: E731
    assert e(1.0625) == 1.0          # halfway 1 | 1.125 -> even mantissa
    assert e(1.1875) == 1.25         # halfway 1.125 | 1.25 -> even
    assert e(1.07) == 1.125
    assert e(500.0) == 448.0 and e(-1e9) == -448.0   # saturation
    assert e(2.0 ** -10) == 0.0      # half the smallest subnormal -> even (0)
    assert e(3 * 2.0 ** -10) == 2.0 ** -8
    assert F.round_fp8(np.array([60000.0]), "e5m2")[0] == 57344.0


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_quantize_maps_amax_to_fmax_and_scales_back(fmt):
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(5000) * 3.0).astype(np.float32)
    q, sinv = F.quantize(x, fmt)
    v = F.decode(q, fmt)
    fmax = F.FORMATS[fmt][2]
    assert np.max(np.abs(v)) == fmax
    # relative error of the dequantised values: one rounding to m bits
    m = F.FORMATS[fmt][0]
    big = np.abs(x) > np.max(np.abs(x)) * 2.0 ** -5
    rel = np.abs(v[big] * sinv - x[big]) / np.abs(x[big])
    assert rel.max() <= 2.0 ** -(m + 1) * (1 + 1e-6)
    assert F.quantize(np.zeros(8, np.float32), fmt)[1] == 1.0


def test_gemm_is_the_product_of_the_decoded_operands():
    rng = np.random.default_rng(2)
    a, sa = F.quantize(rng.standard_normal((5, 7)).astype(np.float32), "e4m3")
    b, sb = F.quantize(rng.standard_normal((3, 7)).astype(np.float32), "e5m2")
    c = F.gemm_fp8(a, "e4m3", sa, b, "e5m2", sb)
    A, B = F.decode(a, "e4m3"), F.decode(b, "e5m2")
    for i in range(5):
        for j in range(3):
            ref = sum(A[i, k] * B[j, k] for k in range(7)) * float(sa) * float(sb)
            assert abs(c[i, j] - ref) <= 1e-12 * max(1.0, abs(ref))


# --------------------------------------------------------------------------
# The layer with FP8 hybrid GEMMs (oracle/fp8_layer.py)
# --------------------------------------------------------------------------

def _tiny(shape, seed=1):
    from layer_inputs import make_layer_inputs
    from layer_inputs.generator import NONTRIVIAL_INIT
    init = dict(NONTRIVIAL_INIT)
    for w in ("w_qkv", "w_o", "w_fc1", "w_fc2"):
        init[w] = (0.0, 0.3)
    inp = make_layer_inputs(shape, seed=seed, init=init)
    return inp.params_f64(), inp.f64("x"), inp.f64("dy")


@pytest.mark.parametrize("dims", [(1, 5, 16, 2, 32), (2, 33, 32, 4, 64), (2, 9, 16, 1, 48, 1, 8)])
def test_fp8_layer_without_quantisation_is_the_rounding_floor(dims):
    """With the 8-bit rounding turned off the FP8 layer is the pinned bf16
    rounding-floor layer (its sites, except dx1, which this mode quantises
    from fp32)."""
    from layer_inputs import LayerShape
    from oracle import fp8_layer as FL
    from oracle import rounding_floor as RF
    shape = LayerShape(*dims)
    P, x, dy = _tiny(shape)
    got = FL.fp8_forward_backward(shape, P, x, dy, quantize=False)
    ref = RF.rounded_forward_backward(shape, P, x, dy,
                                      sites=tuple(s for s in RF.GPU_ROUNDING_SITES if s != "dx1"))
    for a, b in [(got[0], ref[0]), (got[1], ref[1])] + [(got[2][k], ref[2][k]) for k in ref[2]]:
        assert np.abs(a - b).max() <= 1e-12 * max(1.0, np.abs(b).max())


@pytest.mark.parametrize("fa,fb", [("e4m3", "e4m3"), ("e5m2", "e4m3")])
def test_fp8_layer_products_are_the_gemm_of_the_encoded_operands(fa, fb):
    from oracle import fp8_layer as FL
    rng = np.random.default_rng(4)
    A = rng.standard_normal((6, 32)) * 3
    B = rng.standard_normal((5, 32)) * 0.02
    qa, sa = F.quantize(A, fa)
    qb, sb = F.quantize(B, fb)
    ref = F.gemm_fp8(qa, fa, sa, qb, fb, sb)
    got = FL.qdq(A, fa) @ FL.qdq(B, fb).T
    assert np.abs(got - ref).max() <= 1e-12 * np.abs(ref).max()


def _formats_used(monkeypatch, fl_module, shape, P, x, dy):
    calls = []
    real = F.quantize

    def recording(t, fmt):
        calls.append((np.shape(t), fmt))
        return real(t, fmt)

    monkeypatch.setattr(F, "quantize", recording)
    fl_module.fp8_forward_backward(shape, P, x, dy)
    return calls


def _expected_formats(shape):
    T, h, a, f = shape.micro_batch * shape.seq_len, shape.hidden, shape.a, shape.ffn_hidden
    b, s = shape.micro_batch, shape.seq_len
    fwd = [((3 * a, h), "e4m3"), ((h, a), "e4m3"), ((f, h), "e4m3"), ((h, f), "e4m3"),
           ((b, s, h), "e4m3"), ((b, s, a), "e4m3"), ((b, s, h), "e4m3"), ((b, s, f), "e4m3")]
    bwd = [((b, s, h), "e5m2"), ((b, s, f), "e5m2"), ((b, s, h), "e5m2"), ((b, s, 3 * a), "e5m2")]
    assert T == b * s
    return fwd + bwd


def test_fp8_layer_forward_operands_are_e4m3_and_gradients_e5m2(monkeypatch):
    """The hybrid recipe: the weights and forward activations in E4M3, the
    gradients dy, dhp, dx1 and dQ|dK|dV in E5M2, each quantised once."""
    from layer_inputs import LayerShape
    from oracle import fp8_layer as FL
    shape = LayerShape(2, 5, 32, 2, 64, 1, 8)   # a != h so that the shapes tell the operands apart
    P, x, dy = _tiny(shape)
    assert _formats_used(monkeypatch, FL, shape, P, x, dy) == _expected_formats(shape)


def test_planted_e4m3_gradient_is_caught(monkeypatch):
    from layer_inputs import LayerShape
    from oracle import fp8_layer as FL
    shape = LayerShape(2, 5, 32, 2, 64, 1, 8)
    P, x, dy = _tiny(shape)
    monkeypatch.setattr(FL, "E5M2", "e4m3")   # gradients in the forward format
    assert _formats_used(monkeypatch, FL, shape, P, x, dy) != _expected_formats(shape)


def test_fp8_layer_error_is_an_8_bit_rounding_floor():
    """On config c1 the FP8 layer departs from the exact oracle by about an
    8-bit rounding (E4M3 3 mantissa bits, E5M2 2), far above the bf16 floor
    and far below the tensors' scale."""
    from layer_inputs import LayerShape, make_layer_inputs
    import oracle.layer as OL
    from oracle import fp8_layer as FL
    from oracle import rounding_floor as RF
    from parity import metrics
    shape = LayerShape(1, 128, 768, 12, 3072, 1)
    inp = make_layer_inputs(shape)
    P, x, dy = inp.params_f64(), inp.f64("x"), inp.f64("dy")
    exact = OL.layer_forward_backward(shape, P, x, dy)
    f8 = FL.fp8_forward_backward(shape, P, x, dy)
    bf = RF.rounded_forward_backward(shape, P, x, dy)
    names = ["y", "dx"] + list(exact[2])
    pick = lambda r, k: r[0] if k == "y" else r[1] if k == "dx" else r[2][k]  # noqa: E731
    for k in names:
        if k == "b_fc2":
            continue  # the column sum of dy: no 8-bit operand
        e8 = metrics(pick(f8, k), pick(exact, k))["norm_rel"]
        e16 = metrics(pick(bf, k), pick(exact, k))["norm_rel"]
        assert 2 * e16 < e8 < 0.25, (k, e8, e16)
