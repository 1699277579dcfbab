"""Helpers shared by the GPU tests: uploads generator inputs, runs the C-ABI."""
import numpy as np
import torch

from layer_inputs import bf16_bits_to_f64, normal_bf16
from megatron_transformer_layer_gb300 import _lib as L
from megatron_transformer_layer_gb300.layer import TransformerLayer, bf16_tensor

DEV = "cuda"


def bits(n, stream, tensor="x", mean=0.0, std=1.0, seed=7):
    return normal_bf16(n, seed, stream, tensor, mean, std)


def dev_bf16(b):
    return bf16_tensor(np.ascontiguousarray(b), DEV)


def dev_f32_from_bits(b):
    return torch.from_numpy(bf16_bits_to_f64(b).astype(np.float32)).to(DEV)


def to_f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def status():
    return torch.zeros(64, dtype=torch.int32, device=DEV)


def check_status(st):
    torch.cuda.synchronize()
    code = int(st[0].item())
    assert code == 0, f"device status {code} ({L.mc_strerror(code)}) at site {int(st[1].item())}"


def run_layer(inp, t=None, accumulate=False, layer=None):
    """Forward + backward of one layer on the GPU from generator inputs."""
    sh = inp.shape
    t = sh.tp_parts if t is None else t
    params = {k: dev_bf16(v) for k, v in inp.params.items()}
    if layer is None:
        layer = TransformerLayer(sh.micro_batch, sh.seq_len, sh.hidden, sh.heads, sh.ffn_hidden, t,
                                 sh.head_dim, params=params, accumulate_grads=accumulate)
    else:
        layer.set_params(params)
    x = dev_f32_from_bits(inp.x.reshape(-1, sh.hidden))
    dy = dev_f32_from_bits(inp.dy.reshape(-1, sh.hidden))
    y = layer.forward(x)
    dx = layer.backward(dy)
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    return layer, to_f64(y).reshape(inp.x.shape), to_f64(dx).reshape(inp.x.shape), \
        {k: to_f64(v) for k, v in layer.grads.items()}
