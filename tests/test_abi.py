"""The C-ABI library loads, exports every declared symbol, and rejects bad
arguments on the host before any launch (no GPU needed)."""
import ctypes
import os
import re

import pytest

from megatron_transformer_layer_gb300 import _lib as L

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mc_layer.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mc_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    names = declared_functions()
    assert "mc_layer_forward" in names and "mc_layer_backward" in names
    lib = L.lib()
    for n in names:
        assert hasattr(lib, n), n
        assert n in L._SIGNATURES, f"binding lacks {n}"


@pytest.mark.parametrize("shape,code", [
    ((1, 128, 768, 12, 3072, 1), L.MC_OK),
    ((1, 128, 768, 12, 3072, 2), L.MC_OK),
    ((4, 512, 768, 12, 3072, 2), L.MC_OK),
    ((8, 1024, 2048, 16, 8192, 4), L.MC_OK),
    ((1, 4096, 8192, 64, 32768, 8), L.MC_OK),
    ((1, 4096, 8192, 8, 4096, 1, 128), L.MC_OK),       # one TP=8 rank's shard
    ((1, 32768, 4096, 32, 16384, 1), L.MC_OK),
    ((1, 7, 768, 12, 3072, 4), L.MC_OK),               # 768/4, 12/4 divide
    ((1, 128, 768, 12, 3072, 5), L.MC_ERR_SHAPE),      # hidden % 5
    ((1, 128, 768, 12, 3070, 2), L.MC_ERR_UNSUPPORTED),  # ffn/2 = 1535 not a multiple of 64
    ((1, 128, 4096, 3, 4096, 8), L.MC_ERR_SHAPE),      # 3 heads on 8 partitions
    ((0, 128, 768, 12, 3072, 1), L.MC_ERR_SHAPE),
    ((1, 0, 768, 12, 3072, 1), L.MC_ERR_SHAPE),
    ((1, 128, 768, 12, 3072, 0), L.MC_ERR_SHAPE),
    ((1, 128, 768, 24, 3072, 1), L.MC_ERR_UNSUPPORTED),  # head_dim 32
    ((1, 128, 800, 8, 3072, 1), L.MC_ERR_UNSUPPORTED),   # hidden not a multiple of 64
    ((1, 128, 776, 7, 3072, 1), L.MC_ERR_SHAPE),         # hidden % heads
])
def test_check_shape(shape, code):
    s = L.make_shape(*shape)
    assert L.mc_layer_check_shape(s) == code
    if code == L.MC_OK:
        assert L.mc_layer_saved_bytes(s) > 0 and L.mc_layer_workspace_bytes(s) > 0
        assert L.mc_layer_saved_bytes(s) % 256 == 0
    else:
        assert L.mc_layer_saved_bytes(s) == 0 and L.mc_layer_workspace_bytes(s) == 0


def test_saved_bytes_cover_the_activations():
    b, s, h, H, f = 2, 100, 768, 12, 3072
    T, a = b * s, h
    need = 2 * (T * h * 2 + T * 3 * a + T * a + 2 * T * f) + 4 * (4 * T + b * H * s + T * h)
    assert L.mc_layer_saved_bytes(L.make_shape(b, s, h, H, f, 2)) >= need


def test_unknown_flag_rejected():
    assert L.mc_layer_check_shape(L.make_shape(1, 8, 768, 12, 3072, 1, 0, 32)) == L.MC_ERR_ARGUMENT


def test_strerror_covers_all_codes():
    for code in range(0, -10, -1):
        assert L.mc_strerror(code) != "unknown status code"
    assert L.mc_strerror(-100) == "unknown status code"


def _weights(base=0x10000000):
    return L.mc_layer_weights(*[base + 0x100000 * i for i in range(12)])


def test_forward_rejects_bad_arguments_before_launch():
    s = L.make_shape(1, 16, 768, 12, 3072, 1)
    ws = L.mc_layer_workspace_bytes(s)
    w = _weights()
    x, y, saved, wsp = 0x20000000, 0x30000000, 0x40000000, 0x50000000
    assert L.mc_layer_forward(s, w, None, y, saved, wsp, ws) == L.MC_ERR_NULLPTR
    assert L.mc_layer_forward(s, w, x + 4, y, saved, wsp, ws) == L.MC_ERR_ALIGN
    assert L.mc_layer_forward(s, w, x, y, saved + 16, wsp, ws) == L.MC_ERR_ALIGN
    assert L.mc_layer_forward(s, w, x, y, saved, wsp, ws - 1) == L.MC_ERR_WORKSPACE
    bad_w = _weights()
    bad_w.w_o = None
    assert L.mc_layer_forward(s, bad_w, x, y, saved, wsp, ws) == L.MC_ERR_NULLPTR
    bad_w.w_o = 0x10000008
    assert L.mc_layer_forward(s, bad_w, x, y, saved, wsp, ws) == L.MC_ERR_ALIGN
    assert L.mc_layer_forward(L.make_shape(1, 16, 768, 12, 3072, 5), w, x, y, saved, wsp,
                              ws) == L.MC_ERR_SHAPE


def test_backward_rejects_bad_arguments_before_launch():
    s = L.make_shape(1, 16, 768, 12, 3072, 2)
    ws = L.mc_layer_workspace_bytes(s)
    w = _weights()
    g = L.mc_layer_grads(*[0x60000000 + 0x100000 * i for i in range(12)])
    x, dy, saved, dx, wsp = 0x20000000, 0x21000000, 0x40000000, 0x22000000, 0x50000000
    assert L.mc_layer_backward(s, w, x, dy, saved, dx, g, wsp, ws - 256) == L.MC_ERR_WORKSPACE
    assert L.mc_layer_backward(s, w, x, None, saved, dx, g, wsp, ws) == L.MC_ERR_NULLPTR
    g.b_fc1 = None
    assert L.mc_layer_backward(s, w, x, dy, saved, dx, g, wsp, ws) == L.MC_ERR_NULLPTR
    g.b_fc1 = 0x60000004
    assert L.mc_layer_backward(s, w, x, dy, saved, dx, g, wsp, ws) == L.MC_ERR_ALIGN


def test_stage_calls_reject_bad_arguments_before_launch():
    A, B, C = 0x20000000, 0x30000000, 0x40000000
    # N not a multiple of 64
    assert L.mc_gemm(128, 100, 64, A, 64, 0, B, 64, 0, C, 100, L.MC_EPI_STORE_F32) == L.MC_ERR_UNSUPPORTED
    # K-major A needs K % 64 == 0
    assert L.mc_gemm(128, 128, 100, A, 104, 0, B, 104, 0, C, 128, L.MC_EPI_STORE_F32) == L.MC_ERR_UNSUPPORTED
    assert L.mc_gemm(128, 128, 64, A, 64, 0, B, 64, 0, C, 128, 17) == L.MC_ERR_ARGUMENT
    assert L.mc_gemm(128, 128, 64, A, 64, 0, B, 64, 0, C, 128, L.MC_EPI_BIAS_BF16) == L.MC_ERR_NULLPTR
    assert L.mc_gemm(128, 128, 64, A + 2, 64, 0, B, 64, 0, C, 128, L.MC_EPI_STORE_F32) == L.MC_ERR_ALIGN
    assert L.mc_gemm(128, 128, 64, A, 60, 0, B, 64, 0, C, 128, L.MC_EPI_STORE_F32) == L.MC_ERR_ALIGN
    assert L.mc_gemm(128, 128, 128, A, 64, 0, B, 128, 0, C, 128, L.MC_EPI_STORE_F32) == L.MC_ERR_ARGUMENT
    assert L.mc_gemm(128, 128, 192, A, 192, 0, B, 192, 0, C, 128, L.MC_EPI_STORE_F32,
                     k_parts=5) == L.MC_ERR_ARGUMENT
    assert L.mc_attention_forward(A, B, C, 1, 16, 2, 96) == L.MC_ERR_UNSUPPORTED
    assert L.mc_attention_forward(A, None, C, 1, 16, 2, 64) == L.MC_ERR_NULLPTR
    assert L.mc_layernorm_forward(A, B, C, A, None, None, 4, 100) == L.MC_ERR_UNSUPPORTED
    assert L.mc_layernorm_backward_scratch_floats(10, 768) == 3 * 10 * 768


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(L, "_lib", None)
    monkeypatch.setattr(L, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not found"):
        L.lib()


def test_recompute_flag_plans_no_saved_buffer():
    base = L.make_shape(2, 100, 768, 12, 3072, 2)
    rc = L.make_shape(2, 100, 768, 12, 3072, 2, 0, L.MC_RECOMPUTE_ACTIVATIONS)
    both = L.make_shape(2, 100, 768, 12, 3072, 2, 0,
                        L.MC_RECOMPUTE_ACTIVATIONS | L.MC_ACCUMULATE_GRADS)
    assert L.mc_layer_check_shape(rc) == L.MC_OK and L.mc_layer_check_shape(both) == L.MC_OK
    assert L.mc_layer_saved_bytes(rc) == 0
    assert L.mc_layer_workspace_bytes(rc) >= L.mc_layer_workspace_bytes(base) + \
        L.mc_layer_saved_bytes(base)
    # NULL `saved` is accepted in recompute mode (the checks get past it to the
    # workspace-size rule, still before any launch) and rejected otherwise
    w = _weights()
    wsb = L.mc_layer_workspace_bytes(rc)
    assert L.mc_layer_forward(rc, w, 0x20000000, 0x30000000, None, 0x50000000,
                              wsb - 256) == L.MC_ERR_WORKSPACE
    assert L.mc_layer_forward(base, w, 0x20000000, 0x30000000, None, 0x50000000,
                              wsb) == L.MC_ERR_NULLPTR


def test_sequence_parallel_contract():
    """MC_SEQUENCE_PARALLEL: the tokens must split evenly into tp_parts shards."""
    ok = L.make_shape(2, 6, 768, 12, 3072, 4, 0, L.MC_SEQUENCE_PARALLEL)   # 12 tokens / 4
    bad = L.make_shape(1, 7, 768, 12, 3072, 2, 0, L.MC_SEQUENCE_PARALLEL)  # 7 tokens / 2
    plain = L.make_shape(1, 7, 768, 12, 3072, 2, 0, 0)
    assert L.mc_layer_check_shape(ok) == L.MC_OK
    assert L.mc_layer_check_shape(bad) == L.MC_ERR_SHAPE
    assert L.mc_layer_check_shape(plain) == L.MC_OK
    both = L.make_shape(2, 6, 768, 12, 3072, 4, 0,
                        L.MC_SEQUENCE_PARALLEL | L.MC_RECOMPUTE_ACTIVATIONS)
    assert L.mc_layer_check_shape(both) == L.MC_OK


def test_fp8_hybrid_contract():
    """MC_FP8_HYBRID: tokens a multiple of 16, not combined with the
    sequence-parallel flag; the saved activations grow by exactly the 8-bit
    copies the backward reads (transposed activations and weights, 8 scales)."""
    base = (1, 128, 768, 12, 3072, 2, 0)
    ok = L.make_shape(*base, L.MC_FP8_HYBRID)
    assert L.mc_layer_check_shape(ok) == L.MC_OK
    assert L.mc_layer_check_shape(L.make_shape(1, 100, 768, 12, 3072, 2, 0, L.MC_FP8_HYBRID)) \
        == L.MC_ERR_UNSUPPORTED
    assert L.mc_layer_check_shape(
        L.make_shape(*base, L.MC_FP8_HYBRID | L.MC_SEQUENCE_PARALLEL)) == L.MC_ERR_ARGUMENT
    T, h, a, f = 128, 768, 768, 3072
    extra = sum(-(-n // 256) * 256 for n in (h * T, a * T, h * T, f * T, h * 3 * a, a * h,
                                              h * f, f * h, 8 * 4))
    assert L.mc_layer_saved_bytes(ok) == L.mc_layer_saved_bytes(L.make_shape(*base, 0)) + extra
    assert L.mc_layer_workspace_bytes(ok) > L.mc_layer_workspace_bytes(L.make_shape(*base, 0))


def test_attention_ds_workspace_contract():
    # one 32 KB tile per (query block, key block <= it) pair, per head and batch
    assert L.mc_attention_backward_ws_bytes(1, 4096, 64, 128) == 64 * 32 * 33 // 2 * 32768
    assert L.mc_attention_backward_ws_bytes(2, 129, 3, 64) == 2 * 3 * 3 * 32768
    assert L.mc_attention_backward_ws_bytes(1, 128, 1, 96) == 0
    assert L.mc_attention_backward_ws_bytes(0, 128, 1, 128) == 0
    g = L.lib().mc_attention_backward_ws
    p = 0x10000
    assert g(p, p, p, p, p, p, 1, 256, 2, 128, None, 1 << 30, None, None) == L.MC_ERR_NULLPTR
    assert g(p, p, p, p, p, p, 1, 256, 2, 128, p, 100, None, None) == L.MC_ERR_WORKSPACE
    assert g(p, p, p, p, p, p, 0, 256, 2, 128, p, 1 << 30, None, None) == L.MC_ERR_SHAPE


def test_layer_workspace_holds_the_attention_ds_tiles():
    base = L.mc_layer_workspace_bytes(L.make_shape(1, 512, 1024, 8, 4096, 2))
    tiles = L.mc_attention_backward_ws_bytes(1, 512, 8, 128)
    assert base >= tiles
    # MC_ATTN_DQ_RECOMPUTE leaves the tiles out (up to the 256-byte carving)
    lean = L.mc_layer_workspace_bytes(L.make_shape(1, 512, 1024, 8, 4096, 2, 0,
                                                   L.MC_ATTN_DQ_RECOMPUTE))
    assert lean > 0 and base - tiles - 256 <= lean <= base - tiles
    assert L.mc_layer_check_shape(L.make_shape(1, 512, 1024, 8, 4096, 2, 0,
                                               L.MC_ATTN_DQ_RECOMPUTE | L.MC_FP8_HYBRID)) == 0


def test_fp8_quantize_2d_rejects_on_the_host():
    # rows / cols not multiples of 16, or no output: rejected before any launch
    assert L.lib().mc_fp8_quantize_2d(0x10000, 1, 10, 64, 0, 0x10000, None, 0x10000, 0x10000,
                                      None) == L.MC_ERR_SHAPE
    assert L.lib().mc_fp8_quantize_2d(0x10000, 1, 16, 64, 0, None, None, 0x10000, 0x10000,
                                      None) == L.MC_ERR_NULLPTR
    assert L.lib().mc_fp8_quantize_2d(0x10000, 1, 16, 64, 2, 0x10000, None, 0x10000, 0x10000,
                                      None) == L.MC_ERR_ARGUMENT


def test_build_features():
    """The release library carries the NVTX stage ranges and no index
    checks; the debug library (if built) carries both."""
    from megatron_transformer_layer_gb300 import build
    f = L.lib().mc_build_features()
    assert f & L.MC_BUILD_NVTX
    if os.environ.get("MC_LAYER_DEBUG") != "1":
        assert not f & L.MC_BUILD_DEBUG
    if os.path.exists(build.DEBUG_LIB_PATH):
        dbg = ctypes.CDLL(build.DEBUG_LIB_PATH)
        assert dbg.mc_build_features() == L.MC_BUILD_DEBUG | L.MC_BUILD_NVTX


def test_debug_library_exports_the_same_symbols():
    """libmclayer_debug.so (-DMC_DEBUG) is the same ABI."""
    from megatron_transformer_layer_gb300 import build
    if not os.path.exists(build.DEBUG_LIB_PATH):
        pytest.skip("debug library not built")
    dbg = ctypes.CDLL(build.DEBUG_LIB_PATH)
    for n in declared_functions():
        assert hasattr(dbg, n), n
