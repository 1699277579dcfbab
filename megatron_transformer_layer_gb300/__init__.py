"""GB300-native GPT pre-LN transformer layer (BF16 forward + backward).

The compute path is ``libmclayer.so`` (hand-written sm_103a CUDA behind the C
ABI in ``include/mc_layer.h``).  ``_lib`` is its ctypes binding (same names as
the C entry points); ``layer.TransformerLayer`` owns the device buffers, which
PyTorch allocates -- PyTorch is used for memory and streams only.
"""
from . import _lib  # noqa: F401
from ._lib import McError  # noqa: F401
