"""fp64 CPU oracle for the GPT transformer layer (forward + backward).

TEST INFRASTRUCTURE ONLY.  This package is the independent reference that the
CUDA library is checked against.  Only ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline / reference leg may import it; the library in
``megatron_transformer_layer_gb300`` never does, and the two share no code.

Parity pins (checked by ``pytest -m "not gpu"``): finite-difference gradients,
independent library routines (torch fp64 LayerNorm / causal SDPA / tanh-GeLU
with autograd), tensor-parallel invariance, causality, closed-form special
cases and the pages' integer worked examples.
"""
from .layer import (  # noqa: F401
    LN_EPS,
    OracleShape,
    layer_forward,
    layer_backward,
    layer_forward_backward,
    layernorm_forward,
    layernorm_backward,
    gelu_tanh,
    gelu_tanh_grad,
    causal_attention_forward,
    causal_attention_backward,
    check_divisible,
)
from . import contracts  # noqa: F401
