"""Seeded synthetic inputs for one GPT pre-LN transformer layer.

This package only draws random numbers and rounds them to bfloat16.  It holds
none of the layer's arithmetic, so both the fp64 oracle (under ``oracle/``)
and the CUDA library can be fed from it without sharing any computation.
"""
from .generator import (  # noqa: F401
    LayerShape,
    LayerInputs,
    make_layer_inputs,
    normal_bf16,
    bf16_bits_to_f64,
    f64_to_bf16_bits,
    splitmix64,
    PARAM_NAMES,
)
