"""Parity at the benchmark sizes.

c4 (one layer of the 96-layer GPT, 8 partitions -- the launch configuration
bench.py times) and its single-rank shard are compared element by element
with the full fp64 oracle.

Every tensor must meet the binding floor-anchored bound of tests/parity.py
(norm-wise error <= 1.5 x the pinned bf16 rounding floor of the same inputs
+ 2^-16) and max <= 2e-2.  At these widths (h = 8192, 64 heads) bf16 operands
alone put a few LayerNorm gradients at or above the 2e-3 mean bound: the
rounding floor (oracle/rounding_floor.py, pinned in
tests/test_rounding_floor.py) is there at the same size.  Such a tensor must
meet mean <= 1.25 x its floor's mean instead of 2e-3 and is printed as
outside the stated bound; every tensor's floor and result are printed.  c5 (s = 32768) is too long for the full oracle:
y at sampled rows and dx at the last rows are compared with the sampled
oracle (exact by causality), the fc2 bias gradient with the exact column sum
of dy, and the whole layer at c5's widths with a shorter sequence.
"""
import gc

import numpy as np
import pytest
import torch

import oracle.layer as O
from layer_inputs import LayerShape, make_layer_inputs
from oracle.sampled import sampled_rows_and_tail
from parity import MAX_REL_TOL, MEAN_REL_TOL, assert_close, assert_within_floor, floor_bound, \
    metrics

from gpu_util import run_layer

pytestmark = pytest.mark.gpu


def _full_compare(shape, label):
    inp = make_layer_inputs(shape)
    layer, y, dx, G = run_layer(inp)
    del layer
    gc.collect()
    torch.cuda.empty_cache()
    P, x, dyv = inp.params_f64(), inp.f64("x"), inp.f64("dy")
    y_o, dx_o, G_o = O.layer_forward_backward(shape, P, x, dyv)
    from oracle.rounding_floor import rounded_forward_backward
    yr, dxr, Gr = rounded_forward_backward(shape.with_tp(1), P, x, dyv)
    floor = {"y": metrics(yr, y_o), "dx": metrics(dxr, dx_o)}
    floor.update({k: metrics(Gr[k], G_o[k]) for k in G_o})
    del yr, dxr, Gr
    gc.collect()
    lines, outside = [], []

    def check(name, g, o):
        f = floor[name]
        at_floor = f["mean_rel"] > 0.8 * MEAN_REL_TOL
        mean_tol = max(MEAN_REL_TOL, 1.25 * f["mean_rel"]) if at_floor else MEAN_REL_TOL
        m = assert_close(f"{label} {name} (bf16 floor mean {f['mean_rel']:.2e})", g, o,
                         MAX_REL_TOL, mean_tol)
        assert_within_floor(f"{label} {name}", g, o, f["norm_rel"])
        flag = m["mean_rel"] > MEAN_REL_TOL
        if flag:
            outside.append(name)
        lines.append(f"  {name:6s} max {m['max_rel']:.2e} mean {m['mean_rel']:.2e} "
                     f"(floor {f['mean_rel']:.2e}) | norm {m['norm_rel']:.2e} <= "
                     f"{floor_bound(f['norm_rel']):.2e} (floor {f['norm_rel']:.2e})"
                     + ("  [outside the stated 2e-3 mean bound; at the pinned bf16 floor]"
                        if flag else ""))

    check("y", y, y_o)
    check("dx", dx, dx_o)
    for k in list(G_o):
        check(k, G.pop(k), G_o.pop(k))
        gc.collect()
    print(f"\n{label}:\n" + "\n".join(lines)
          + (f"\n  outside the stated mean bound (at the bf16 floor): {outside}" if outside else ""))


def test_config4_tp8_full_size():
    _full_compare(LayerShape(1, 4096, 8192, 64, 32768, 8), "c4 tp8")


def test_config4_single_rank_shard_full_size():
    _full_compare(LayerShape(1, 4096, 8192, 8, 4096, 1, 128), "c4 shard")


def test_config5_widths_short_sequence():
    _full_compare(LayerShape(1, 2048, 4096, 32, 16384, 1), "c5 widths s2048")


def test_config5_full_size_sampled():
    shape = LayerShape(1, 32768, 4096, 32, 16384, 1)
    inp = make_layer_inputs(shape)
    layer, y, dx, G = run_layer(inp)
    del layer
    torch.cuda.empty_cache()
    rows = [0, 1, 127, 128, 129, 4095, 16384, 30001, 32767]
    tail = 16
    ys, dxs = sampled_rows_and_tail(shape, inp.params_f64(), inp.f64("x"), inp.f64("dy"), rows, tail)
    m_y = assert_close("c5 y rows", y[:, rows], ys)
    m_dx = assert_close("c5 dx tail", dx[:, -tail:], dxs)
    m_b = assert_close("c5 b_fc2", G["b_fc2"], inp.f64("dy").reshape(-1, shape.hidden).sum(axis=0))
    assert np.isfinite(dx).all() and all(np.isfinite(v).all() for v in G.values())
    print(f"\nc5 sampled: y {m_y}\n dx {m_dx}\n b_fc2 {m_b}")
