"""ctypes binding of ``libmclayer.so`` (the C ABI in ``include/mc_layer.h``).

Argument marshalling only: every function here has the name of the C entry
point it calls and forwards plain integers (device pointers, sizes, a
cudaStream_t handle).  Anything with a ``data_ptr()`` method (a torch tensor)
is accepted where a pointer is expected.  No computation happens in Python.
"""
from __future__ import annotations

import ctypes
import os

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
# MC_LAYER_DEBUG=1 selects the debug build (-DMC_DEBUG: every global store's
# indices are checked on the device; see build.py).
LIB_PATH = os.path.join(PKG_DIR, "libmclayer_debug.so" if os.environ.get("MC_LAYER_DEBUG") == "1"
                        else "libmclayer.so")

MC_OK = 0
MC_ERR_SHAPE = -1
MC_ERR_UNSUPPORTED = -2
MC_ERR_NULLPTR = -3
MC_ERR_ALIGN = -4
MC_ERR_WORKSPACE = -5
MC_ERR_CUDA = -6
MC_ERR_DEVICE_TIMEOUT = -7
MC_ERR_DEVICE_BOUNDS = -8
MC_ERR_ARGUMENT = -9
MC_ERR_SCRATCH_LIMIT = -10

MC_ACCUMULATE_GRADS = 1
MC_RECOMPUTE_ACTIVATIONS = 2
MC_SEQUENCE_PARALLEL = 4
MC_FP8_HYBRID = 8
MC_ATTN_DQ_RECOMPUTE = 16
MC_BUILD_DEBUG = 1
MC_BUILD_NVTX = 2

MC_EPI_STORE_F32 = 0
MC_EPI_STORE_BF16 = 1
MC_EPI_BIAS_BF16 = 2
MC_EPI_BIAS_GELU = 3
MC_EPI_BIAS_RESID_F32 = 4
MC_EPI_GELU_BWD = 5

PARAM_ORDER = ("ln1_g", "ln1_b", "w_qkv", "b_qkv", "w_o", "b_o",
               "ln2_g", "ln2_b", "w_fc1", "b_fc1", "w_fc2", "b_fc2")


class McError(RuntimeError):
    def __init__(self, code: int, where: str = ""):
        self.code = code
        super().__init__(f"{where}: {code} ({mc_strerror(code)})" if where else
                         f"{code} ({mc_strerror(code)})")


class mc_layer_shape(ctypes.Structure):  # noqa: N801 (C name)
    _fields_ = [("micro_batch", ctypes.c_int32), ("seq_len", ctypes.c_int32),
                ("hidden", ctypes.c_int32), ("heads", ctypes.c_int32),
                ("ffn_hidden", ctypes.c_int32), ("tp_parts", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("flags", ctypes.c_uint32)]


class mc_layer_weights(ctypes.Structure):  # noqa: N801
    _fields_ = [(n, ctypes.c_void_p) for n in PARAM_ORDER]


class mc_layer_grads(ctypes.Structure):  # noqa: N801
    _fields_ = [(n, ctypes.c_void_p) for n in PARAM_ORDER]


_lib = None

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_INT = ctypes.c_int
_SZ = ctypes.c_size_t

_SIGNATURES = {
    "mc_layer_check_shape": (_INT, [ctypes.POINTER(mc_layer_shape)]),
    "mc_layer_saved_bytes": (_SZ, [ctypes.POINTER(mc_layer_shape)]),
    "mc_layer_workspace_bytes": (_SZ, [ctypes.POINTER(mc_layer_shape)]),
    "mc_layer_forward": (_INT, [ctypes.POINTER(mc_layer_shape), ctypes.POINTER(mc_layer_weights),
                                _P, _P, _P, _P, _SZ, _P]),
    "mc_layer_backward": (_INT, [ctypes.POINTER(mc_layer_shape), ctypes.POINTER(mc_layer_weights),
                                 _P, _P, _P, _P, ctypes.POINTER(mc_layer_grads), _P, _SZ, _P]),
    "mc_layer_device_status": (_INT, [_P, _P]),
    "mc_strerror": (ctypes.c_char_p, [_INT]),
    "mc_layernorm_forward": (_INT, [_P, _P, _P, _P, _P, _P, _I64, _I32, _P, _P]),
    "mc_layernorm_backward": (_INT, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _INT, _P,
                                     _I64, _I32, _P, _P]),
    "mc_layernorm_backward_scratch_floats": (_SZ, [_I64, _I32]),
    "mc_gemm": (_INT, [_I64, _I64, _I64, _P, _I64, _INT, _P, _I64, _INT, _P, _I64, _INT, _P, _P,
                       _I64, _INT, _INT, _P, _P]),
    "mc_attention_forward": (_INT, [_P, _P, _P, _I32, _I32, _I32, _I32, _P, _P]),
    "mc_attention_backward": (_INT, [_P, _P, _P, _P, _P, _P, _I32, _I32, _I32, _I32, _P, _P]),
    "mc_attention_backward_noalloc": (_INT, [_P, _P, _P, _P, _P, _I32, _I32, _I32, _I32, _P, _P]),
    "mc_attention_backward_ws_bytes": (_SZ, [_I32, _I32, _I32, _I32]),
    "mc_build_features": (_INT, []),
    "mc_attention_backward_ws": (_INT, [_P, _P, _P, _P, _P, _P, _I32, _I32, _I32, _I32, _P, _SZ,
                                        _P, _P]),
    "mc_selftest_wait_timeout": (_INT, [_I64, _P, _P]),
    "mc_selftest_bounds_check": (_INT, [_I64, _I64, _P, _P, _P]),
    "mc_fp8_scratch_floats": (_SZ, []),
    "mc_fp8_quantize": (_INT, [_P, _I32, _I64, _I32, _P, _P, _P, _P, _P]),
    "mc_fp8_quantize_2d": (_INT, [_P, _I32, _I64, _I64, _I32, _P, _P, _P, _P, _P]),
    "mc_gemm_fp8": (_INT, [_I64, _I64, _I64, _P, _I64, _I32, _P, _I64, _I32, _P, _P, _P, _I64,
                           _I32, _P, _P, _I64, _I32, _I32, _P, _P]),
    "mc_cp_schedule": (_INT, [_I32, _I32, _I32, ctypes.POINTER(_I32)]),
    "mc_cp_launch_plan": (_INT, [_I32, ctypes.POINTER(_I32), _I32]),
    "mc_attention_cp_workspace_bytes": (_SZ, [_I32, _I32, _I32, _I32, _I32]),
    "mc_attention_forward_cp": (_INT, [_P, _P, _P, _I32, _I32, _I32, _I32, _I32, _P, _SZ, _P, _P]),
    "mc_attention_backward_cp": (_INT, [_P, _P, _P, _P, _P, _P, _I32, _I32, _I32, _I32, _I32, _P,
                                        _SZ, _P, _P]),
}


def lib() -> ctypes.CDLL:
    """Loads libmclayer.so (or the debug build, see LIB_PATH), built in-tree;
    raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} not found: build it with "
                               "`python -m megatron_transformer_layer_gb300.build` "
                               "(`--debug` for the debug build)")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s) -> int | None:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream  # torch.cuda.Stream


def make_shape(micro_batch, seq_len, hidden, heads, ffn_hidden, tp_parts=1, head_dim=0, flags=0):
    return mc_layer_shape(micro_batch, seq_len, hidden, heads, ffn_hidden, tp_parts, head_dim, flags)


def make_weights(tensors: dict) -> mc_layer_weights:
    return mc_layer_weights(*[_ptr(tensors[n]) for n in PARAM_ORDER])


def make_grads(tensors: dict) -> mc_layer_grads:
    return mc_layer_grads(*[_ptr(tensors[n]) for n in PARAM_ORDER])


# ---- the C entry points, same names ----------------------------------------

def mc_layer_check_shape(shape: mc_layer_shape) -> int:
    return lib().mc_layer_check_shape(ctypes.byref(shape))


def mc_layer_saved_bytes(shape: mc_layer_shape) -> int:
    return lib().mc_layer_saved_bytes(ctypes.byref(shape))


def mc_layer_workspace_bytes(shape: mc_layer_shape) -> int:
    return lib().mc_layer_workspace_bytes(ctypes.byref(shape))


def mc_layer_forward(shape, weights, x, y, saved, ws, ws_bytes, stream=None) -> int:
    return lib().mc_layer_forward(ctypes.byref(shape), ctypes.byref(weights), _ptr(x), _ptr(y),
                                  _ptr(saved), _ptr(ws), ws_bytes, _stream(stream))


def mc_layer_backward(shape, weights, x, dy, saved, dx, grads, ws, ws_bytes, stream=None) -> int:
    return lib().mc_layer_backward(ctypes.byref(shape), ctypes.byref(weights), _ptr(x), _ptr(dy),
                                   _ptr(saved), _ptr(dx), ctypes.byref(grads), _ptr(ws), ws_bytes,
                                   _stream(stream))


def mc_layer_device_status(ws, stream=None) -> int:
    return lib().mc_layer_device_status(_ptr(ws), _stream(stream))


def mc_strerror(code: int) -> str:
    try:
        return lib().mc_strerror(code).decode()
    except RuntimeError:
        return "libmclayer.so not loaded"


def mc_layernorm_forward(x, gamma, beta, out, mean, rstd, rows, h, status=None, stream=None) -> int:
    return lib().mc_layernorm_forward(_ptr(x), _ptr(gamma), _ptr(beta), _ptr(out), _ptr(mean),
                                      _ptr(rstd), rows, h, _ptr(status), _stream(stream))


def mc_layernorm_backward(dout, x, mean, rstd, gamma, resid, dx, dx_bf16, dgamma, dbeta, colsum_dx,
                          accumulate, partials, rows, h, status=None, stream=None) -> int:
    return lib().mc_layernorm_backward(_ptr(dout), _ptr(x), _ptr(mean), _ptr(rstd), _ptr(gamma),
                                       _ptr(resid), _ptr(dx), _ptr(dx_bf16), _ptr(dgamma),
                                       _ptr(dbeta), _ptr(colsum_dx), accumulate, _ptr(partials),
                                       rows, h, _ptr(status), _stream(stream))


def mc_layernorm_backward_scratch_floats(rows: int, h: int) -> int:
    return lib().mc_layernorm_backward_scratch_floats(rows, h)


def mc_gemm(M, N, K, A, lda, a_layout, B, ldb, b_layout, out, ldc, epilogue, bias=None, aux=None,
            ldaux=0, accumulate=0, k_parts=1, status=None, stream=None) -> int:
    return lib().mc_gemm(M, N, K, _ptr(A), lda, a_layout, _ptr(B), ldb, b_layout, _ptr(out), ldc,
                         epilogue, _ptr(bias), _ptr(aux), ldaux, accumulate, k_parts, _ptr(status),
                         _stream(stream))


def mc_attention_forward(qkv, o, lse, micro_batch, seq_len, heads, head_dim, status=None,
                         stream=None) -> int:
    return lib().mc_attention_forward(_ptr(qkv), _ptr(o), _ptr(lse), micro_batch, seq_len, heads,
                                      head_dim, _ptr(status), _stream(stream))


def mc_attention_backward(qkv, o, lse, dout, dqkv, delta, micro_batch, seq_len, heads, head_dim,
                          status=None, stream=None) -> int:
    return lib().mc_attention_backward(_ptr(qkv), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dqkv),
                                       _ptr(delta), micro_batch, seq_len, heads, head_dim,
                                       _ptr(status), _stream(stream))


def mc_attention_backward_ws_bytes(micro_batch, seq_len, heads, head_dim) -> int:
    return lib().mc_attention_backward_ws_bytes(micro_batch, seq_len, heads, head_dim)


def mc_attention_backward_ws(qkv, o, lse, dout, dqkv, delta, micro_batch, seq_len, heads,
                             head_dim, ds_workspace, ds_workspace_bytes, status=None,
                             stream=None) -> int:
    """mc_attention_backward whose dQ is formed from dS^T tiles written by the
    dK/dV kernel into `ds_workspace` (uint8 device tensor)."""
    return lib().mc_attention_backward_ws(_ptr(qkv), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dqkv),
                                          _ptr(delta), micro_batch, seq_len, heads, head_dim,
                                          _ptr(ds_workspace), ds_workspace_bytes, _ptr(status),
                                          _stream(stream))


def mc_attention_backward_noalloc(qkv, o, lse, dout, dqkv, micro_batch, seq_len, heads, head_dim,
                                  status=None, stream=None) -> int:
    """Allocation-free attention backward (fixed in-library scratch)."""
    return lib().mc_attention_backward_noalloc(_ptr(qkv), _ptr(o), _ptr(lse), _ptr(dout),
                                               _ptr(dqkv), micro_batch, seq_len, heads, head_dim,
                                               _ptr(status), _stream(stream))


def mc_cp_schedule(cp_parts, rank, step):
    """(query chunk, key chunk) pairs of a virtual CP rank in a ring step
    (host only); raises on an invalid argument."""
    buf = (_I32 * 8)()
    n = lib().mc_cp_schedule(cp_parts, rank, step, buf)
    if n < 0:
        raise ValueError(mc_strerror(n))
    return [(buf[2 * k], buf[2 * k + 1]) for k in range(n)]


def mc_cp_launch_plan(cp_parts):
    """The context-parallel launch plan (host only): one tuple (launch,
    query chunk, key chunk, mode of the query chunk, mode of the key chunk)
    per chunk pair, in launch order; raises on an invalid argument."""
    n_pairs = cp_parts * (2 * cp_parts + 1) if cp_parts > 0 else 1
    buf = (_I32 * (5 * n_pairs))()
    n = lib().mc_cp_launch_plan(cp_parts, buf, n_pairs)
    if n < 0:
        raise ValueError(mc_strerror(n))
    return [tuple(buf[5 * k + e] for e in range(5)) for k in range(n)]


def mc_attention_cp_workspace_bytes(micro_batch, seq_len, heads, head_dim, cp_parts) -> int:
    return lib().mc_attention_cp_workspace_bytes(micro_batch, seq_len, heads, head_dim, cp_parts)


def mc_attention_forward_cp(qkv, o, lse, micro_batch, seq_len, heads, head_dim, cp_parts,
                            workspace, workspace_bytes, status=None, stream=None) -> int:
    return lib().mc_attention_forward_cp(_ptr(qkv), _ptr(o), _ptr(lse), micro_batch, seq_len,
                                         heads, head_dim, cp_parts, _ptr(workspace),
                                         workspace_bytes, _ptr(status), _stream(stream))


def mc_attention_backward_cp(qkv, o, lse, dout, dqkv, delta, micro_batch, seq_len, heads,
                             head_dim, cp_parts, workspace, workspace_bytes, status=None,
                             stream=None) -> int:
    return lib().mc_attention_backward_cp(_ptr(qkv), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dqkv),
                                          _ptr(delta), micro_batch, seq_len, heads, head_dim,
                                          cp_parts, _ptr(workspace), workspace_bytes,
                                          _ptr(status), _stream(stream))


FP8_E4M3 = 0
FP8_E5M2 = 1


def mc_fp8_scratch_floats() -> int:
    return lib().mc_fp8_scratch_floats()


def mc_fp8_quantize(x, out, scale_inv, scratch, fmt, status=None, stream=None) -> int:
    """Per-tensor current scaling of x (fp32 or bf16 tensor) to 8-bit bytes."""
    import torch
    in_bf16 = 1 if x.dtype == torch.bfloat16 else 0
    return lib().mc_fp8_quantize(_ptr(x), in_bf16, x.numel(), fmt, _ptr(out), _ptr(scale_inv),
                                 _ptr(scratch), _ptr(status), _stream(stream))


def mc_fp8_quantize_2d(x, out, out_t, scale_inv, scratch, fmt, stream=None) -> int:
    """Per-tensor current scaling of a 2-D x (fp32 or bf16) to 8-bit bytes,
    written as is (out) and/or transposed (out_t); either may be None."""
    import torch
    in_bf16 = 1 if x.dtype == torch.bfloat16 else 0
    rows, cols = x.shape
    return lib().mc_fp8_quantize_2d(_ptr(x), in_bf16, rows, cols, fmt, _ptr(out), _ptr(out_t),
                                    _ptr(scale_inv), _ptr(scratch), _stream(stream))


def mc_gemm_fp8(M, N, K, A, lda, a_format, B, ldb, b_format, a_scale_inv, b_scale_inv, out, ldc,
                epilogue, bias=None, aux=None, ldaux=0, accumulate=0, k_parts=1, status=None,
                stream=None) -> int:
    return lib().mc_gemm_fp8(M, N, K, _ptr(A), lda, a_format, _ptr(B), ldb, b_format,
                             _ptr(a_scale_inv), _ptr(b_scale_inv), _ptr(out), ldc, epilogue,
                             _ptr(bias), _ptr(aux), ldaux, accumulate, k_parts, _ptr(status),
                             _stream(stream))


def mc_selftest_bounds_check(index, extent, buf, status, stream=None) -> int:
    """Runs the index check of a debug build on one index (failure-path test)."""
    return lib().mc_selftest_bounds_check(index, extent, _ptr(buf), _ptr(status), _stream(stream))


def mc_selftest_wait_timeout(timeout_ns, status, stream=None) -> int:
    """Runs a kernel whose bounded wait is made to run out (failure-path test)."""
    return lib().mc_selftest_wait_timeout(timeout_ns, _ptr(status), _stream(stream))
