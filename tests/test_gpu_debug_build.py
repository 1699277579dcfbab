"""The debug build (libmclayer_debug.so, -DMC_DEBUG) and guard bands.

The debug build checks, on the device, the indices of every global store of
the GEMM, attention and LayerNorm kernels against the extents each kernel
was given; a failed check records MC_ERR_DEVICE_BOUNDS and skips the store.
Here: the index check records that code and touches nothing when an index is
out of range (the self-test kernel, which never dereferences it); ragged and
odd shapes run through the debug build with no check failing and give the
release build's bits; and guard bands around the outputs stay untouched.
"""
import hashlib
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from layer_inputs import LayerShape, make_layer_inputs
from layer_inputs.generator import NONTRIVIAL_INIT
from megatron_transformer_layer_gb300 import _lib as L

from gpu_util import DEV, dev_bf16, dev_f32_from_bits, status

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SHAPES = [(1, 1, 768, 12, 3072, 1), (2, 7, 768, 12, 3072, 4), (2, 129, 1024, 8, 4096, 2),
          (1, 200, 2048, 2, 1024, 1, 128), (1, 300, 1024, 8, 4096, 2)]


def test_index_check_records_bounds_error_and_skips_the_store():
    buf = torch.zeros(5, dtype=torch.int32, device=DEV)
    st = status()
    assert L.mc_selftest_bounds_check(3, 5, buf, st) == L.MC_OK
    torch.cuda.synchronize()
    assert int(st[0].item()) == 0 and buf.tolist() == [0, 0, 0, 1, 0]
    for bad in (5, 7, -1):
        st = status()
        assert L.mc_selftest_bounds_check(bad, 5, buf, st) == L.MC_OK
        torch.cuda.synchronize()
        assert int(st[0].item()) == L.MC_ERR_DEVICE_BOUNDS and int(st[1].item()) == 30
    assert buf.tolist() == [0, 0, 0, 1, 0]


def layer_digest(shape_args, seed=1):
    """Forward + backward of one layer; returns (device status, sha256 of y,
    dx and all gradients) -- run in this process's library."""
    from megatron_transformer_layer_gb300.layer import TransformerLayer
    shape = LayerShape(*shape_args)
    inp = make_layer_inputs(shape, seed=seed, init=NONTRIVIAL_INIT)
    ly = TransformerLayer(*shape_args[:6], head_dim=shape.head_dim,
                          params={k: dev_bf16(v) for k, v in inp.params.items()})
    x = dev_f32_from_bits(inp.x.reshape(-1, shape.hidden))
    dy = dev_f32_from_bits(inp.dy.reshape(-1, shape.hidden))
    y = ly.forward(x)
    dx = ly.backward(dy)
    torch.cuda.synchronize()
    h = hashlib.sha256()
    for t in [y, dx] + [ly.grads[k] for k in sorted(ly.grads)]:
        h.update(t.cpu().numpy().tobytes())
    return ly.device_status(), h.hexdigest()


def test_debug_build_runs_ragged_shapes_clean_and_matches_release():
    code = ("import sys; sys.path[:0] = [%r, %r]\n"
            "from test_gpu_debug_build import layer_digest, SHAPES\n"
            "for s in SHAPES: print(*layer_digest(s))\n") % (ROOT, os.path.join(ROOT, "tests"))
    env = dict(os.environ, MC_LAYER_DEBUG="1")
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                         timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    debug = [ln.split() for ln in out.stdout.strip().splitlines()]
    assert len(debug) == len(SHAPES)
    for shape_args, (st, digest) in zip(SHAPES, debug):
        assert int(st) == 0, (shape_args, st)
        rst, rdigest = layer_digest(shape_args)
        assert rst == 0 and digest == rdigest, shape_args


def test_guard_bands_around_outputs_stay_untouched():
    """y and dx written into the middle of larger buffers whose bands before
    and after hold a fill pattern: the pattern survives forward + backward at
    ragged shapes (an out-of-range store would change it)."""
    from megatron_transformer_layer_gb300.layer import TransformerLayer
    band = 4096
    for shape_args in SHAPES:
        shape = LayerShape(*shape_args)
        inp = make_layer_inputs(shape, seed=2, init=NONTRIVIAL_INIT)
        ly = TransformerLayer(*shape_args[:6], head_dim=shape.head_dim,
                              params={k: dev_bf16(v) for k, v in inp.params.items()})
        n = shape.micro_batch * shape.seq_len * shape.hidden
        x = dev_f32_from_bits(inp.x.reshape(-1, shape.hidden))
        dy = dev_f32_from_bits(inp.dy.reshape(-1, shape.hidden))
        ybuf = torch.full((n + 2 * band,), -7.25, device=DEV)
        dxbuf = torch.full((n + 2 * band,), 3.5e5, device=DEV)
        y = ybuf[band:band + n].view(-1, shape.hidden)
        dx = dxbuf[band:band + n].view(-1, shape.hidden)
        ly.forward(x, y)
        ly.backward(dy, dx, x=x)
        torch.cuda.synchronize()
        assert ly.device_status() == 0
        for buf, fill in ((ybuf, -7.25), (dxbuf, 3.5e5)):
            assert bool((buf[:band] == fill).all()) and bool((buf[band + n:] == fill).all()), \
                shape_args
        assert np.isfinite(y.cpu().numpy()).all() and np.isfinite(dx.cpu().numpy()).all()
