"""Parity at the benchmark sizes.

c4 (one layer of the 96-layer GPT, 8 partitions -- the launch configuration
bench.py times) and its single-rank shard are compared element by element
with the full fp64 oracle.  c5 (s = 32768) is too long for the full oracle:
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
from parity import assert_close

from gpu_util import run_layer

pytestmark = pytest.mark.gpu


def _full_compare(shape, label):
    inp = make_layer_inputs(shape)
    layer, y, dx, G = run_layer(inp)
    del layer
    gc.collect()
    torch.cuda.empty_cache()
    y_o, dx_o, G_o = O.layer_forward_backward(shape, inp.params_f64(), inp.f64("x"), inp.f64("dy"))
    worst = []
    worst.append(("y", assert_close(f"{label} y", y, y_o)))
    worst.append(("dx", assert_close(f"{label} dx", dx, dx_o)))
    for k in list(G_o):
        worst.append((k, assert_close(f"{label} {k}", G.pop(k), G_o.pop(k))))
        gc.collect()
    name, m = max(worst, key=lambda kv: kv[1]["mean_rel"])
    print(f"\n{label}: worst mean_rel {name} {m}")


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
