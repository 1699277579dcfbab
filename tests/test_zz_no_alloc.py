"""The allocation-free attention backward (mc_attention_backward_noalloc).

Some callers cannot allocate device memory -- e.g. a plugin whose host
framework forbids cudaMalloc while it runs, or a process whose device memory
another allocator has already reserved -- so they cannot pass the `delta`
scratch buffer that mc_attention_backward takes.  This entry point uses a
fixed scratch array inside the library instead.  Here it is called through the
C ABI twice in a row and must give what the allocating entry point gives, bit
for bit, without changing the device's free memory; a problem larger than its
fixed scratch must be rejected before any launch.
This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import numpy as np
import pytest
import torch

from layer_inputs import bf16_bits_to_f64
from megatron_transformer_layer_gb300 import _lib as L
from parity import assert_close

from gpu_util import DEV, bits, check_status, dev_bf16, status, to_f64

pytestmark = pytest.mark.gpu


def _case(b, s, H, d, seed):
    a = H * d
    qkv = dev_bf16(bits(b * s * 3 * a, 40 + seed))
    dout = dev_bf16(bits(b * s * a, 50 + seed))
    o = torch.empty(b * s * a, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(b * H * s, dtype=torch.float32, device=DEV)
    st = status()
    assert L.mc_attention_forward(qkv, o, lse, b, s, H, d, st) == 0
    ref = torch.empty(b * s * 3 * a, dtype=torch.bfloat16, device=DEV)
    delta = torch.empty(b * H * s, dtype=torch.float32, device=DEV)
    assert L.mc_attention_backward(qkv, o, lse, dout, ref, delta, b, s, H, d, st) == 0
    check_status(st)
    return qkv, o, lse, dout, to_f64(ref)


@pytest.mark.parametrize("b,s,H,d", [(2, 300, 4, 128), (1, 257, 3, 64)])
def test_noalloc_backward_matches_allocating_entry_point_twice(b, s, H, d):
    """Two calls in a row equal the allocating entry point to the bit (the
    same kernels on the same inputs), which is also within the parity
    tolerance; neither call changes the device's free memory or torch's
    reserved pool, i.e. nothing is allocated."""
    qkv, o, lse, dout, ref = _case(b, s, H, d, seed=b + d)
    outs = [torch.full((b * s * 3 * H * d,), float("nan"), dtype=torch.bfloat16, device=DEV)
            for _ in range(2)]
    sts = [status() for _ in range(2)]
    torch.cuda.synchronize()
    free0, reserved0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_reserved()
    for dqkv, st in zip(outs, sts):
        rc = L.mc_attention_backward_noalloc(qkv, o, lse, dout, dqkv, b, s, H, d, st)
        assert rc == L.MC_OK, L.mc_strerror(rc)
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free0
        assert torch.cuda.memory_reserved() == reserved0
    for dqkv, st in zip(outs, sts):
        check_status(st)
        got = to_f64(dqkv)
        assert np.array_equal(got, ref)
        assert_close("noalloc dqkv", got, ref)


def test_noalloc_rejects_problems_beyond_its_scratch():
    # micro_batch * heads * seq_len = 2 * 8 * 65537 > 1,048,576: rejected on the
    # host, nothing launched (the pointers are never dereferenced).
    rc = L.mc_attention_backward_noalloc(0x10000, 0x10000, 0x10000, 0x10000, 0x10000,
                                         2, 65537, 8, 128)
    assert rc == L.MC_ERR_SCRATCH_LIMIT
    assert "scratch" in L.mc_strerror(rc)
