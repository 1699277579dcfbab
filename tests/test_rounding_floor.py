"""The bf16 rounding-floor diagnostic: its pins, and how the tolerance is read.

``oracle/rounding_floor.py`` re-runs the layer with bf16 rounding at the
GEMM operands of the CUDA path.  Its floor sets a binding parity bound
(``tests/parity.py``), so it is pinned here against things other than itself:

* its rounding is torch's float64 -> float32 -> bfloat16 conversion, bit for
  bit (a library routine);
* with no rounding site on it equals the oracle (so its arithmetic is the
  layer's and no rounding hides outside the named sites);
* each site, on alone, changes exactly the outputs that the layer's data flow
  puts downstream of that tensor, and nothing else (so a site sits at the
  tensor it names, and it rounds something);
* with K the identity the dQ of the attention backward is dS times the scale,
  so rounding dS before the scale leaves dQ * sqrt(d) a bf16 number;
* planted mistakes (an extra rounding of the residual x1, the rounding of P
  dropped, dS rounded after its scale) each trip one of these pins.

The last test shows why the tolerance is read relative to each tensor's scale
(no GPU involved).
"""
import numpy as np
import pytest
import torch

import oracle.layer as L
import oracle.rounding_floor as RF
from layer_inputs import LayerShape, make_layer_inputs
from layer_inputs.generator import NONTRIVIAL_INIT
from parity import MAX_REL_TOL, MEAN_REL_TOL, metrics

OUTPUTS = ("y", "dx", "ln1_g", "ln1_b", "w_qkv", "b_qkv", "w_o", "b_o", "ln2_g", "ln2_b",
           "w_fc1", "b_fc1", "w_fc2", "b_fc2")
_ATTN_BWD = {"w_qkv", "b_qkv", "ln1_g", "ln1_b", "dx"}
_MLP_BWD = {"b_fc1", "w_fc1", "ln2_g", "ln2_b", "b_o", "w_o"} | _ATTN_BWD
_ALL_BUT_DY_SUM = set(OUTPUTS) - {"b_fc2"}
# Outputs downstream of each rounding site in the layer's data flow (forward
# sites reach y and, through the saved activations, the whole backward; b_fc2
# is the column sum of dy and depends on nothing rounded).
DOWNSTREAM = {
    "ln1": _ALL_BUT_DY_SUM, "qkv": _ALL_BUT_DY_SUM, "p_fwd": _ALL_BUT_DY_SUM,
    "o": _ALL_BUT_DY_SUM, "ln2": _ALL_BUT_DY_SUM,
    "g": {"y", "w_fc2"},
    "hp": _MLP_BWD, "dhp": _MLP_BWD,
    "dx1": {"w_o"} | _ATTN_BWD,
    "do": _ATTN_BWD, "p_bwd": _ATTN_BWD, "ds": _ATTN_BWD, "dqkv": _ATTN_BWD,
}


def _inputs(shape, seed=1):
    init = dict(NONTRIVIAL_INIT)
    for w in ("w_qkv", "w_o", "w_fc1", "w_fc2"):
        init[w] = (0.0, 0.3)
    inp = make_layer_inputs(shape, seed=seed, init=init)
    return inp.params_f64(), inp.f64("x"), inp.f64("dy")


def _flat(y, dx, G):
    out = {"y": y, "dx": dx}
    out.update(G)
    return out


def _rel(a, b):
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-300))


# ---- pins, each a function of the implementation under test ---------------

def identity_error(fb, shape, P, x, dy):
    """Largest relative difference between ``fb`` with no site on and the oracle."""
    got = _flat(*fb(shape, P, x, dy, sites=()))
    ref = _flat(*L.layer_forward_backward(shape, P, x, dy))
    return max(_rel(got[k], ref[k]) for k in OUTPUTS)


def dependency_mismatches(fb, shape, P, x, dy, sites=tuple(DOWNSTREAM)):
    """Sites whose effect (the outputs that change when only that site rounds)
    is not the set the data flow predicts."""
    base = _flat(*fb(shape, P, x, dy, sites=()))
    bad = {}
    for site in sites:
        got = _flat(*fb(shape, P, x, dy, sites=(site,)))
        changed = {k for k in OUTPUTS if not np.array_equal(got[k], base[k])}
        if changed != DOWNSTREAM[site]:
            bad[site] = (sorted(changed ^ DOWNSTREAM[site]))
    return bad


def ds_site_offset(att_bwd, d=8, seed=3):
    """With K = I (s = d) dQ = dS * scale; returns the largest distance of
    dQ * sqrt(d) from a bf16 number, relative to its magnitude (0 when the
    dS site rounds before the scale)."""
    rng = np.random.default_rng(seed)
    q, v, do = (rng.standard_normal((d, d)) for _ in range(3))
    k = np.eye(d)
    o, lse = L.causal_attention_forward(q, k, v)
    dq, _, _ = att_bwd(q, k, v, o, lse, do, lambda site, t: RF.bf16_round(t) if site == "ds" else t)
    z = dq * np.sqrt(d)
    nz = np.abs(z) > 0
    return float((np.abs(RF.bf16_round(z) - z)[nz] / np.abs(z)[nz]).max())


SHAPES = [LayerShape(1, 1, 8, 2, 16, 1), LayerShape(2, 5, 16, 2, 32, 1),
          LayerShape(1, 33, 32, 4, 64, 1), LayerShape(2, 9, 16, 1, 48, 1, 8)]


def test_bf16_round_is_torch_conversion():
    rng = np.random.default_rng(0)
    v = np.concatenate([
        rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000),
        # exact ties between two bf16 neighbours, both parities, both signs
        np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 2 ** -130 * 3, 0.0, -0.0,
                  3.3895313892515355e38, 1e-45, -1e-40]),
    ])
    ref = torch.from_numpy(v).to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    got = RF.bf16_round(v)
    assert np.array_equal(got.view(np.uint64), ref.view(np.uint64))


@pytest.mark.parametrize("shape", SHAPES, ids=str)
def test_no_site_equals_the_oracle(shape):
    P, x, dy = _inputs(shape)
    assert identity_error(RF.rounded_forward_backward, shape, P, x, dy) < 1e-12


@pytest.mark.parametrize("shape", SHAPES[1:], ids=str)
def test_each_site_changes_exactly_its_downstream_outputs(shape):
    P, x, dy = _inputs(shape)
    assert dependency_mismatches(RF.rounded_forward_backward, shape, P, x, dy) == {}


def test_default_sites_are_the_documented_gpu_rounding_points():
    assert set(RF.GPU_ROUNDING_SITES) == set(DOWNSTREAM)
    assert not set(RF.EXTRA_SITES) & set(RF.GPU_ROUNDING_SITES)


def test_ds_is_rounded_before_the_scale():
    assert ds_site_offset(RF.rounded_attention_backward) < 1e-14


# ---- planted mistakes -------------------------------------------------------

def _with_sites(transform):
    def fb(shape, P, x, dy, sites=RF.GPU_ROUNDING_SITES):
        return RF.rounded_forward_backward(shape, P, x, dy, sites=transform(tuple(sites)))
    return fb


def test_planted_extra_rounding_of_x1_is_caught_and_raises_the_floor():
    shape = SHAPES[1]
    P, x, dy = _inputs(shape)
    mutant = _with_sites(lambda s: s + ("x1",))           # rounds x1 whatever it is asked
    assert identity_error(mutant, shape, P, x, dy) > 1e-4
    # and on config c1 it doubles y's floor
    c1 = LayerShape(1, 128, 768, 12, 3072, 1)
    inp = make_layer_inputs(c1)
    P1, x1, dy1 = inp.params_f64(), inp.f64("x"), inp.f64("dy")
    exact = L.layer_forward_backward(c1, P1, x1, dy1)
    good = metrics(RF.rounded_forward_backward(c1, P1, x1, dy1)[0], exact[0])["norm_rel"]
    bad = metrics(mutant(c1, P1, x1, dy1)[0], exact[0])["norm_rel"]
    assert bad > 1.8 * good, (good, bad)


def test_planted_missing_rounding_of_p_is_caught():
    shape = SHAPES[1]
    P, x, dy = _inputs(shape)
    mutant = _with_sites(lambda s: tuple(t for t in s if t != "p_fwd"))
    assert "p_fwd" in dependency_mismatches(mutant, shape, P, x, dy, sites=("p_fwd",))


def test_planted_ds_rounded_after_the_scale_is_caught():
    def mutant(q, k, v, o, lse, do, r):
        return RF.rounded_attention_backward(
            q, k, v, o, lse, do, lambda site, t: r("ds", t) if site == "ds_scaled" else t)
    assert ds_site_offset(mutant) > 1e-4


# ---- the tolerance reading --------------------------------------------------

def test_bf16_operand_floor_vs_tolerance_readings():
    """The stated tolerance is max relative error 2e-2 and mean relative
    error 2e-3 for bf16 operands with fp32 accumulation.  Read norm-wise
    (sum|g - o| / sum|o|) the mean bound sits BELOW what bf16 operands alone
    produce (a weight gradient is a sum of products of two independently
    rounded operands, about 2.3e-3 relative rms), so no bf16-operand
    implementation could meet it.  Read relative to each tensor's scale
    (mean|g - o| / max|o|) it holds with margin."""
    shape = LayerShape(1, 128, 768, 12, 3072, 1)
    inp = make_layer_inputs(shape)
    P, x, dy = inp.params_f64(), inp.f64("x"), inp.f64("dy")
    y, dx, G = L.layer_forward_backward(shape, P, x, dy)
    yr, dxr, Gr = RF.rounded_forward_backward(shape, P, x, dy)
    m = {"y": metrics(yr, y), "dx": metrics(dxr, dx)}
    m.update({k: metrics(Gr[k], G[k]) for k in G})
    over = [k for k, v in m.items() if v["norm_rel"] > MEAN_REL_TOL]
    assert {"w_fc2", "w_fc1", "w_qkv", "w_o"} <= set(over), m
    for k, v in m.items():
        assert v["max_rel"] <= MAX_REL_TOL and v["mean_rel"] <= MEAN_REL_TOL, (k, v)
