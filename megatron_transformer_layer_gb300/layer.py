"""Device-buffer owner for one layer: torch allocates, libmclayer computes."""
from __future__ import annotations

import torch

from . import _lib as L


def _check(rc: int, where: str) -> None:
    if rc != L.MC_OK:
        raise L.McError(rc, where)


def bf16_tensor(bits, device) -> torch.Tensor:
    """uint16 bf16 bit patterns (numpy) -> bf16 device tensor (bit-exact)."""
    t = torch.from_numpy(bits.astype("int16", copy=False).view("int16").copy())
    return t.view(torch.bfloat16).to(device)


class TransformerLayer:
    """One GPT pre-LN layer on one GPU.

    ``params`` maps parameter names to bf16 device tensors.  Gradients are fp32
    device tensors owned here.  ``forward``/``backward`` enqueue on the current
    torch stream (or ``stream``) and return without synchronising.
    """

    def __init__(self, micro_batch, seq_len, hidden, heads, ffn_hidden, tp_parts=1, head_dim=0,
                 params=None, device="cuda", accumulate_grads=False, recompute=False,
                 workspace=None, sequence_parallel=False, fp8=False, attn_dq_recompute=False):
        # attn_dq_recompute: the attention backward forms S and dP again for
        # dQ instead of keeping dS tiles (whose workspace grows as seq_len^2)
        flags = (L.MC_ACCUMULATE_GRADS if accumulate_grads else 0) | \
            (L.MC_RECOMPUTE_ACTIVATIONS if recompute else 0) | \
            (L.MC_SEQUENCE_PARALLEL if sequence_parallel else 0) | \
            (L.MC_FP8_HYBRID if fp8 else 0) | \
            (L.MC_ATTN_DQ_RECOMPUTE if attn_dq_recompute else 0)
        self.shape = L.make_shape(micro_batch, seq_len, hidden, heads, ffn_hidden, tp_parts,
                                  head_dim, flags)
        _check(L.mc_layer_check_shape(self.shape), "mc_layer_check_shape")
        self.device = torch.device(device)
        self.tokens = micro_batch * seq_len
        self.hidden = hidden
        self.saved_bytes = L.mc_layer_saved_bytes(self.shape)
        self.ws_bytes = L.mc_layer_workspace_bytes(self.shape)
        # uint8 buffers: the caching allocator returns >= 512-byte aligned blocks.
        # With recomputation nothing is saved and a workspace may be shared by
        # the layers of a stack (pass the same `workspace` tensor to each).
        self.saved = (torch.empty(self.saved_bytes, dtype=torch.uint8, device=self.device)
                      if self.saved_bytes else None)
        if workspace is not None:
            assert workspace.numel() >= self.ws_bytes
            self.ws = workspace
        else:
            self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=self.device)
        self.params = params
        self.weights = L.make_weights(params) if params is not None else None
        d = head_dim if head_dim else hidden // heads
        a = heads * d
        shapes = {"ln1_g": (hidden,), "ln1_b": (hidden,), "w_qkv": (3 * a, hidden),
                  "b_qkv": (3 * a,), "w_o": (hidden, a), "b_o": (hidden,), "ln2_g": (hidden,),
                  "ln2_b": (hidden,), "w_fc1": (ffn_hidden, hidden), "b_fc1": (ffn_hidden,),
                  "w_fc2": (hidden, ffn_hidden), "b_fc2": (hidden,)}
        self.grads = {k: torch.zeros(v, dtype=torch.float32, device=self.device)
                      for k, v in shapes.items()}
        self._grads_c = L.make_grads(self.grads)
        self._x = None

    @staticmethod
    def random_params(hidden, heads, ffn_hidden, head_dim=0, device="cuda", seed=0, std=0.02):
        """bf16 parameters in the library's layout: weights N(0, std^2), biases
        0, LayerNorm gains 1 and shifts 0 (the usual GPT initialisation)."""
        d = head_dim if head_dim else hidden // heads
        a = heads * d
        g = torch.Generator(device=device).manual_seed(seed)
        w = {"w_qkv": (3 * a, hidden), "w_o": (hidden, a), "w_fc1": (ffn_hidden, hidden),
             "w_fc2": (hidden, ffn_hidden)}
        p = {k: (torch.randn(*v, device=device, generator=g) * std).bfloat16() for k, v in w.items()}
        for k, n in (("b_qkv", 3 * a), ("b_o", hidden), ("b_fc1", ffn_hidden), ("b_fc2", hidden),
                     ("ln1_b", hidden), ("ln2_b", hidden)):
            p[k] = torch.zeros(n, device=device, dtype=torch.bfloat16)
        for k in ("ln1_g", "ln2_g"):
            p[k] = torch.ones(hidden, device=device, dtype=torch.bfloat16)
        return p

    def set_params(self, params):
        self.params = params
        self.weights = L.make_weights(params)

    def _stream(self, stream):
        return stream if stream is not None else torch.cuda.current_stream(self.device)

    def forward(self, x: torch.Tensor, y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        if y is None:
            y = torch.empty_like(x)
        _check(L.mc_layer_forward(self.shape, self.weights, x, y, self.saved, self.ws,
                                  self.ws_bytes, self._stream(stream)), "mc_layer_forward")
        self._x = x
        return y

    def backward(self, dy: torch.Tensor, dx: torch.Tensor | None = None, x: torch.Tensor | None = None,
                 stream=None) -> torch.Tensor:
        x = self._x if x is None else x
        if dx is None:
            dx = torch.empty_like(dy)
        _check(L.mc_layer_backward(self.shape, self.weights, x, dy, self.saved, dx, self._grads_c,
                                   self.ws, self.ws_bytes, self._stream(stream)),
               "mc_layer_backward")
        return dx

    def device_status(self, stream=None) -> int:
        return L.mc_layer_device_status(self.ws, self._stream(stream))
