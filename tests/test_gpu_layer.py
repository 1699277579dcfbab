"""Layer parity: the whole forward + backward through the C ABI against the
fp64 oracle, on the same seeded inputs; y, dx and all twelve parameter
gradients are checked per tensor, against the stated bounds and against the
bf16 rounding floor of the same inputs (tests/parity.py)."""
import numpy as np
import pytest
import torch

import oracle.layer as O
from layer_inputs import LayerShape, make_layer_inputs
from layer_inputs.generator import NONTRIVIAL_INIT
from oracle.rounding_floor import floor_norm_rel
from parity import assert_close, assert_within_floor, floor_bound, metrics

from gpu_util import DEV, dev_f32_from_bits, run_layer, to_f64

pytestmark = pytest.mark.gpu


def _oracle(inp, t):
    sh = inp.shape.with_tp(t)
    return O.layer_forward_backward(sh, inp.params_f64(), inp.f64("x"), inp.f64("dy"))


def _check_layer(inp, t, label, layer=None):
    _, y, dx, G = run_layer(inp, t, layer=layer)
    y_o, dx_o, G_o = _oracle(inp, t)
    floor = floor_norm_rel(inp.shape.with_tp(1), inp.params_f64(), inp.f64("x"), inp.f64("dy"),
                           exact=(y_o, dx_o, G_o))
    got = {"y": y, "dx": dx, **G}
    ref = {"y": y_o, "dx": dx_o, **G_o}
    lines = []
    for k in ref:
        m = assert_close(f"{label} {k}", got[k], ref[k])
        assert_within_floor(f"{label} {k}", got[k], ref[k], floor[k])
        lines.append(f"  {k:6s} max {m['max_rel']:.2e} mean {m['mean_rel']:.2e} | norm "
                     f"{m['norm_rel']:.2e} <= {floor_bound(floor[k]):.2e} (floor {floor[k]:.2e})")
    print(f"\n{label}:\n" + "\n".join(lines))
    return y, dx, G


@pytest.mark.parametrize("t", [1, 2])
def test_config1(t):
    """b1 s128 h768 H12 f3072, default init (biases 0, gamma 1, beta 0)."""
    _check_layer(make_layer_inputs(LayerShape(1, 128, 768, 12, 3072, t)), t, f"c1 t={t}")


def test_config1_nontrivial_biases_and_affine():
    inp = make_layer_inputs(LayerShape(1, 128, 768, 12, 3072, 2), seed=3, init=NONTRIVIAL_INIT)
    _check_layer(inp, 2, "c1 nontrivial")


@pytest.mark.parametrize("shape", [
    LayerShape(1, 1, 768, 12, 3072, 1),          # single token
    LayerShape(2, 7, 768, 12, 3072, 4),          # ragged, 4 partitions
    LayerShape(2, 129, 1024, 8, 4096, 2),        # head_dim 128, ragged tile tail
    LayerShape(1, 200, 2048, 2, 1024, 1, 128),   # a = heads * head_dim != hidden
])
def test_ragged_and_special_shapes(shape):
    inp = make_layer_inputs(shape, seed=1, init=NONTRIVIAL_INIT)
    _check_layer(inp, shape.tp_parts, str(shape))


def test_gpu_outputs_do_not_depend_on_tp_parts():
    inp = make_layer_inputs(LayerShape(2, 96, 1024, 8, 4096, 1), seed=2, init=NONTRIVIAL_INIT)
    _, y1, dx1, G1 = run_layer(inp, 1)
    for t in (2, 4, 8):
        _, y, dx, G = run_layer(inp, t)
        assert metrics(y, y1)["max_rel"] < 1e-6 and metrics(dx, dx1)["max_rel"] < 1e-6
        for k in G1:
            assert metrics(G[k], G1[k])["max_rel"] < 1e-6, k


def test_gpu_causality():
    shape = LayerShape(1, 150, 768, 12, 3072, 2)
    inp = make_layer_inputs(shape, seed=4)
    layer, y, _, _ = run_layer(inp)
    i = 70
    x2 = inp.x.copy()
    x2[:, i + 1:, :] = inp.x[:, i + 1:, :][:, ::-1, :]          # change every later token
    x = dev_f32_from_bits(x2.reshape(-1, shape.hidden))
    y2 = to_f64(layer.forward(x)).reshape(inp.x.shape)
    torch.cuda.synchronize()
    assert np.array_equal(y2[:, :i + 1], y[:, :i + 1])
    assert not np.array_equal(y2[:, i + 1:], y[:, i + 1:])


def test_accumulate_grads_flag():
    inp = make_layer_inputs(LayerShape(1, 64, 768, 12, 3072, 2), seed=5, init=NONTRIVIAL_INIT)
    layer, _, _, G = run_layer(inp, accumulate=True)
    x = dev_f32_from_bits(inp.x.reshape(-1, 768))
    dy = dev_f32_from_bits(inp.dy.reshape(-1, 768))
    layer.forward(x)
    layer.backward(dy)
    torch.cuda.synchronize()
    for k, v in layer.grads.items():
        assert metrics(to_f64(v), 2 * G[k])["max_rel"] < 1e-6, k


def test_config2_stack_of_12_layers():
    """b4 s512 h768 H12 f3072, tp 2: twelve layers, distinct weights per
    layer, fp32 residual stream between layers, backward in reverse."""
    shape = LayerShape(4, 512, 768, 12, 3072, 2)
    n_layers = 12
    inps = [make_layer_inputs(shape, seed=0, layer=l) for l in range(n_layers)]
    x0, dyN = inps[0].f64("x"), inps[0].f64("dy")
    # oracle
    caches, acts = [], [x0]
    for l in range(n_layers):
        y, c = O.layer_forward(shape, inps[l].params_f64(), acts[-1])
        caches.append(c)
        acts.append(y)
    g = dyN
    grads_o = [None] * n_layers
    for l in reversed(range(n_layers)):
        g, grads_o[l] = O.layer_backward(shape, inps[l].params_f64(), caches[l], g)
    dx_o = g
    # GPU
    from megatron_transformer_layer_gb300.layer import TransformerLayer
    from gpu_util import dev_bf16
    layers = [TransformerLayer(4, 512, 768, 12, 3072, 2,
                               params={k: dev_bf16(v) for k, v in inps[l].params.items()})
              for l in range(n_layers)]
    x = dev_f32_from_bits(inps[0].x.reshape(-1, 768))
    outs = [x]
    for l in range(n_layers):
        outs.append(layers[l].forward(outs[-1]))
    gd = dev_f32_from_bits(inps[0].dy.reshape(-1, 768))
    for l in reversed(range(n_layers)):
        gd = layers[l].backward(gd, x=outs[l])
    torch.cuda.synchronize()
    assert_close("stack y", to_f64(outs[-1]).reshape(x0.shape), acts[-1])
    assert_close("stack dx", to_f64(gd).reshape(x0.shape), dx_o)
    for l in (0, n_layers - 1):
        for k, v in layers[l].grads.items():
            assert_close(f"stack layer{l} {k}", to_f64(v), grads_o[l][k])


@pytest.mark.parametrize("t", [1, 2, 4])
def test_config3(t):
    """b8 s1024 h2048 H16 (d128) f8192."""
    _check_layer(make_layer_inputs(LayerShape(8, 1024, 2048, 16, 8192, t)), t, f"c3 t={t}")


def test_attn_dq_recompute_flag_matches_oracle():
    """MC_ATTN_DQ_RECOMPUTE: the attention backward without the dS tile
    workspace (its dQ kernel forms S and dP again) -- both gates against the
    oracle, the forward bitwise equal to the default mode, a workspace
    smaller by the tiles."""
    from megatron_transformer_layer_gb300.layer import TransformerLayer
    shape = LayerShape(2, 129, 1024, 8, 4096, 2)
    inp = make_layer_inputs(shape, seed=1, init=NONTRIVIAL_INIT)
    lean = TransformerLayer(2, 129, 1024, 8, 4096, 2, attn_dq_recompute=True)
    default, y0, _, _ = run_layer(inp)
    assert lean.ws_bytes < default.ws_bytes
    y1, _, _ = _check_layer(inp, 2, "attn dq recompute", layer=lean)
    assert np.array_equal(y0, y1)


def test_activation_recomputation_matches_default_mode():
    """MC_RECOMPUTE_ACTIVATIONS: nothing saved between the passes, the
    backward re-runs the forward; results identical to the default mode, and
    one workspace shared by a 3-layer stack."""
    from megatron_transformer_layer_gb300.layer import TransformerLayer
    from gpu_util import dev_bf16
    shape = LayerShape(2, 129, 1024, 8, 4096, 2)
    inps = [make_layer_inputs(shape, seed=6, layer=l, init=NONTRIVIAL_INIT) for l in range(3)]
    x = dev_f32_from_bits(inps[0].x.reshape(-1, 1024))
    dy = dev_f32_from_bits(inps[0].dy.reshape(-1, 1024))

    def run(recompute, workspace=None):
        layers = [TransformerLayer(2, 129, 1024, 8, 4096, 2, recompute=recompute,
                                   workspace=workspace,
                                   params={k: dev_bf16(v) for k, v in inp.params.items()})
                  for inp in inps]
        acts = [x]
        for ly in layers:
            acts.append(ly.forward(acts[-1]))
        g = dy
        for i in reversed(range(3)):
            g = layers[i].backward(g, x=acts[i])
        torch.cuda.synchronize()
        assert all(ly.device_status() == 0 for ly in layers)
        return to_f64(acts[-1]), to_f64(g), [{k: to_f64(v) for k, v in ly.grads.items()} for ly in layers]

    y0, dx0, G0 = run(False)
    probe = TransformerLayer(2, 129, 1024, 8, 4096, 2, recompute=True,
                             params={k: dev_bf16(v) for k, v in inps[0].params.items()})
    assert probe.saved is None
    shared = torch.empty(probe.ws_bytes, dtype=torch.uint8, device=DEV)
    y1, dx1, G1 = run(True, shared)
    assert np.array_equal(y0, y1) and np.array_equal(dx0, dx1)
    for a, b in zip(G0, G1):
        for k in a:
            assert np.array_equal(a[k], b[k]), k


def test_cuda_graph_capture_matches_eager():
    """The C ABI enqueues only launches and memsets on the caller's stream, so
    a whole forward + backward can be captured in a CUDA graph (after a first
    uncaptured call has done the one-time set-up) and replayed on new inputs."""
    shape = LayerShape(1, 96, 768, 12, 3072, 2)
    inp = make_layer_inputs(shape, seed=8, init=NONTRIVIAL_INIT)
    inp2 = make_layer_inputs(shape, seed=9, init=NONTRIVIAL_INIT)
    inp2.params = inp.params  # same weights; new x and dy
    layer, _, _, _ = run_layer(inp)
    x = dev_f32_from_bits(inp.x.reshape(-1, 768))
    dy = dev_f32_from_bits(inp.dy.reshape(-1, 768))
    y = torch.empty_like(x)
    dx = torch.empty_like(x)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer.forward(x, y)
        layer.backward(dy, dx, x=x)
    torch.cuda.synchronize()
    # new inputs into the captured buffers, replay, compare with eager
    x.copy_(dev_f32_from_bits(inp2.x.reshape(-1, 768)))
    dy.copy_(dev_f32_from_bits(inp2.dy.reshape(-1, 768)))
    graph.replay()
    torch.cuda.synchronize()
    y_g, dx_g = to_f64(y), to_f64(dx)
    G_g = {k: to_f64(v) for k, v in layer.grads.items()}
    _, y_e, dx_e, G_e = run_layer(inp2, layer=layer)
    assert np.array_equal(y_g.reshape(y_e.shape), y_e)
    assert np.array_equal(dx_g.reshape(dx_e.shape), dx_e)
    for k in G_e:
        assert np.array_equal(G_g[k], G_e[k]), k


@pytest.mark.parametrize("shape", [
    LayerShape(2, 130, 1024, 8, 4096, 4),        # 260 tokens in 4 shards of 65
    LayerShape(1, 256, 768, 12, 3072, 2),        # config c1's widths, 2 shards
])
def test_sequence_parallel_matches_oracle_and_default_mode(shape):
    """MC_SEQUENCE_PARALLEL: LayerNorm, the residual epilogues and the input
    gradients' reduce-scatter run per sequence shard.  The result meets both
    parity gates against the oracle, and equals the default mode up to the
    order of the fp32 sums over shards (the sequence-sharded parameters'
    gradients are the shards' partial sums)."""
    from megatron_transformer_layer_gb300.layer import TransformerLayer
    from gpu_util import dev_bf16
    inp = make_layer_inputs(shape, seed=9, init=NONTRIVIAL_INIT)
    x = dev_f32_from_bits(inp.x.reshape(-1, shape.hidden))
    dy = dev_f32_from_bits(inp.dy.reshape(-1, shape.hidden))
    out = []
    for sp in (False, True):
        ly = TransformerLayer(shape.micro_batch, shape.seq_len, shape.hidden, shape.heads,
                              shape.ffn_hidden, shape.tp_parts, sequence_parallel=sp,
                              params={k: dev_bf16(v) for k, v in inp.params.items()})
        y = ly.forward(x)
        dx = ly.backward(dy)
        torch.cuda.synchronize()
        assert ly.device_status() == 0
        out.append({"y": to_f64(y).reshape(inp.x.shape), "dx": to_f64(dx).reshape(inp.x.shape),
                    **{k: to_f64(v) for k, v in ly.grads.items()}})
    y_o, dx_o, G_o = _oracle(inp, shape.tp_parts)
    ref = {"y": y_o, "dx": dx_o, **G_o}
    floor = floor_norm_rel(shape.with_tp(1), inp.params_f64(), inp.f64("x"), inp.f64("dy"),
                           exact=(y_o, dx_o, G_o))
    for k in ref:
        assert_close(f"sp {k}", out[1][k], ref[k])
        assert_within_floor(f"sp {k}", out[1][k], ref[k], floor[k])
        assert metrics(out[1][k], out[0][k])["max_rel"] < 1e-5, k


def test_c4_layer_is_bitwise_repeatable():
    """The whole layer at the benchmark shape (one layer of the 96-layer GPT,
    8 partitions) twice on the same inputs: y, dx and all twelve gradients
    identical to the bit (no atomics, fixed-order reductions), which would
    expose a race in any kernel of the step."""
    from megatron_transformer_layer_gb300.layer import TransformerLayer
    b, s, h, H, f, t = 1, 4096, 8192, 64, 32768, 8
    g = torch.Generator(device=DEV).manual_seed(11)
    shapes = {"ln1_g": (h,), "ln1_b": (h,), "w_qkv": (3 * h, h), "b_qkv": (3 * h,),
              "w_o": (h, h), "b_o": (h,), "ln2_g": (h,), "ln2_b": (h,), "w_fc1": (f, h),
              "b_fc1": (f,), "w_fc2": (h, f), "b_fc2": (h,)}
    params = {}
    for k, shp in shapes.items():
        std = 0.02 if k.startswith("w_") else 0.1
        mean = 1.0 if k.endswith("_g") else 0.0
        params[k] = (torch.randn(*shp, device=DEV, generator=g) * std + mean).bfloat16()
    x = torch.randn(b * s, h, device=DEV, generator=g).bfloat16().float()
    dy = torch.randn(b * s, h, device=DEV, generator=g).bfloat16().float()
    ly = TransformerLayer(b, s, h, H, f, t, params=params)
    runs = []
    for _ in range(2):
        y = ly.forward(x).clone()
        dx = ly.backward(dy).clone()
        torch.cuda.synchronize()
        assert ly.device_status() == 0
        runs.append((y, dx, {k: v.clone() for k, v in ly.grads.items()}))
    assert torch.equal(runs[0][0], runs[1][0]) and torch.equal(runs[0][1], runs[1][1])
    for k in runs[0][2]:
        assert torch.equal(runs[0][2][k], runs[1][2][k]), k
    assert torch.isfinite(runs[0][0]).all() and torch.isfinite(runs[0][1]).all()


def test_random_params_layer_runs():
    """The convenience initialisation (used in the README) gives a runnable
    layer whose output is finite and whose fc2 bias gradient is the column sum
    of dy."""
    from megatron_transformer_layer_gb300.layer import TransformerLayer
    params = TransformerLayer.random_params(1024, 8, 4096)
    layer = TransformerLayer(1, 256, 1024, 8, 4096, tp_parts=2, params=params)
    x = torch.randn(256, 1024, device=DEV)
    dy = torch.randn(256, 1024, device=DEV).bfloat16().float()
    y = layer.forward(x)
    layer.backward(dy)
    torch.cuda.synchronize()
    assert layer.device_status() == 0 and torch.isfinite(y).all()
    ref = dy.double().sum(0)
    assert torch.allclose(layer.grads["b_fc2"].double(), ref, rtol=1e-5, atol=1e-3)
