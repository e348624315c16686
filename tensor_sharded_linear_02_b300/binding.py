"""Thin ctypes binding of ``libtp_b300.so`` (the C ABI in ``include/tp.h``).

Argument marshalling only: every function takes torch tensors that already
live on the current CUDA device, reads their pointers, sizes and dtypes, and
calls the C entry point of the same name on the current torch stream.  No
arithmetic of the method happens here, and there is no fallback: if the
library is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtp_b300.so")

TP_OK = 0
TP_ERR_DEVICE_TIMEOUT = 8
TP_F32, TP_BF16 = 0, 1
TP_SPLIT_COLS, TP_SPLIT_ROWS = 0, 1
TP_ACT_NONE, TP_ACT_GELU = 0, 1
TP_MAX_SHARDS = 64
TP_STATIC_WS_BYTES = 32 << 20

_lock = threading.Lock()
_lib = None


class TPError(RuntimeError):
    """A library call returned a status other than TP_OK."""

    def __init__(self, fn: str, status: int, message: str):
        super().__init__(f"{fn}: {message}")
        self.status = status


_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_int = ctypes.c_int

SIGNATURES = {
    "tp_column_linear": ([_vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _int, _int, _int, _vp], _int),
    "tp_column_linear_grouped": ([_vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _int, _int, _int,
                                  _int, _vp], _int),
    "tp_row_linear": ([_vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _int, _int, _vp], _int),
    "tp_sharded_linear": ([_vp, _vp, _vp, _i64, _i64, _i64, _int, _int, _int, _int, _int, _vp],
                          _int),
    "tp_shard_reduce": ([_vp, _vp, _i64, _i64, _int, _int, _vp], _int),
    "tp_shard_concat": ([_vp, _vp, _i64, _i64, _int, _int, _vp], _int),
    "tp_shard_concat_grouped": ([_vp, _vp, _i64, _i64, _int, _int, _int, _vp], _int),
    "tp_mlp_block_workspace_size": ([_i64, _i64, _int], ctypes.c_size_t),
    "tp_mlp_block": ([_vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _i64, _i64, _i64, _int, _int,
                      _int, _vp], _int),
    "tp_mlp_block_static_ws": ([_vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _int, _int, _vp],
                               _int),
    "tp_qkv_linear": ([_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, _int, _int, _int, _vp],
                      _int),
    "tp_column_linear_bias": ([_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _int, _int, _int,
                               _vp], _int),
    "tp_row_linear_bias": ([_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _int, _int, _vp],
                           _int),
    "tp_mlp_block_bias": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _i64, _i64, _i64,
                           _int, _int, _int, _vp], _int),
    "tp_column_linear_backward": ([_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _int, _int,
                                   _vp], _int),
    "tp_row_linear_backward": ([_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _int, _int, _vp],
                               _int),
    "tp_mlp_block_backward_workspace_size": ([_i64, _i64, _int], ctypes.c_size_t),
    "tp_mlp_block_backward": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _i64, _i64,
                               _i64, _int, _int, _int, _vp], _int),
    "tp_get_device_status": ([_vp], _int),
    "tp_selftest_bounded_wait": ([ctypes.c_uint64, _vp], _int),
    "tp_status_string": ([_int], ctypes.c_char_p),
}


def lib() -> ctypes.CDLL:
    """Load the shared library (once) and declare every entry point."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it first (python -c "
                    f"'import __graft_entry__; __graft_entry__.build()')")
            handle = ctypes.CDLL(LIB_PATH)
            for name, (args, res) in SIGNATURES.items():
                fn = getattr(handle, name)
                fn.argtypes = args
                fn.restype = res
            _lib = handle
        return _lib


def _check(fn: str, status: int) -> None:
    if status != TP_OK:
        msg = lib().tp_status_string(status).decode()
        raise TPError(fn, status, msg)


def _dtype_code(t) -> int:
    import torch
    if t == torch.bfloat16:
        return TP_BF16
    if t == torch.float32:
        return TP_F32
    raise TypeError(f"unsupported dtype {t}")


def _ptr(t):
    """Device pointer of a tensor the C ABI reads as a dense row-major array:
    a CPU tensor, a tensor on another device than the current one, or a
    strided view (a transpose, a column slice) would be misread, so all
    three are refused here."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"tensor of shape {tuple(t.shape)} is not on a CUDA device")
    import torch
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"tensor of shape {tuple(t.shape)} is on {t.device}, not on the current "
                         f"device cuda:{torch.cuda.current_device()}")
    if not t.is_contiguous():
        raise ValueError(f"tensor of shape {tuple(t.shape)} and strides {t.stride()} is not "
                         f"contiguous (row-major)")
    return ctypes.c_void_p(t.data_ptr())


def _dims(t, ndim: int, name: str):
    """The sizes of a tensor that must have `ndim` dimensions."""
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions, got shape {tuple(t.shape)}")
    return tuple(int(v) for v in t.shape)


def _expect(t, shape, name: str, dtype=None) -> None:
    """Refuses an optional tensor whose shape (or dtype) is not the one the
    call's sizes imply: the C ABI sees only a pointer and would read or
    write past the end of a smaller buffer."""
    if t is None:
        return
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")


def _same_dtype(names_and_tensors) -> None:
    ts = [(n, t) for n, t in names_and_tensors if t is not None]
    for n, t in ts[1:]:
        if t.dtype != ts[0][1].dtype:
            raise ValueError(f"{n} has dtype {t.dtype}, but {ts[0][0]} has {ts[0][1].dtype}")


def _ws_bytes(ws) -> int:
    if ws is None:
        return 0
    if ws.dim() != 1:
        raise ValueError(f"workspace must be a 1-D buffer, got shape {tuple(ws.shape)}")
    return ws.numel() * ws.element_size()


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _act(act) -> int:
    if act in (None, "none", TP_ACT_NONE):
        return TP_ACT_NONE
    if act in ("gelu", TP_ACT_GELU):
        return TP_ACT_GELU
    raise ValueError(f"unknown activation {act!r}")


def _out_dtype(Y, Ys):
    return (Y if Y is not None else Ys).dtype


# --------------------------------------------------------------- entries ---

def _column_shapes(X, W, Y, Y_shards, n_shards, bias=None):
    M, K = _dims(X, 2, "X")
    K2, N = _dims(W, 2, "W")
    if K2 != K:
        raise ValueError(f"W has {K2} rows, X has {K} columns")
    _same_dtype([("X", X), ("W", W), ("bias", bias)])
    _same_dtype([("Y", Y), ("Y_shards", Y_shards)])
    _expect(Y, (M, N), "Y")
    if Y_shards is not None and n_shards >= 1 and N % n_shards == 0:
        _expect(Y_shards, (n_shards, M, N // n_shards), "Y_shards")
    _expect(bias, (N,), "bias")
    return M, K, N


def tp_column_linear(X, W, Y=None, Y_shards=None, n_shards=1, act=None, stream=None):
    M, K, N = _column_shapes(X, W, Y, Y_shards, n_shards)
    st = lib().tp_column_linear(_ptr(X), _ptr(W), _ptr(Y), _ptr(Y_shards), M, K, N, n_shards,
                                _dtype_code(X.dtype), _dtype_code(_out_dtype(Y, Y_shards)),
                                _act(act), _stream(stream))
    _check("tp_column_linear", st)


def tp_column_linear_grouped(X, W, Y=None, Y_shards=None, n_shards=1, col_groups=1, act=None,
                             stream=None):
    M, K, N = _column_shapes(X, W, Y, Y_shards, n_shards)
    st = lib().tp_column_linear_grouped(_ptr(X), _ptr(W), _ptr(Y), _ptr(Y_shards), M, K, N,
                                        n_shards, col_groups, _dtype_code(X.dtype),
                                        _dtype_code(_out_dtype(Y, Y_shards)), _act(act),
                                        _stream(stream))
    _check("tp_column_linear_grouped", st)


def _row_shapes(X, W, Y, P_out, n_shards, bias=None):
    import torch
    M, K = _dims(X, 2, "X")
    K2, N = _dims(W, 2, "W")
    if K2 != K:
        raise ValueError(f"W has {K2} rows, X has {K} columns")
    _same_dtype([("X", X), ("W", W), ("bias", bias)])
    _expect(Y, (M, N), "Y")
    _expect(P_out, (n_shards, M, N), "P_out", torch.float32)
    _expect(bias, (N,), "bias")
    return M, K, N


def tp_row_linear(X, W, Y=None, P_out=None, n_shards=1, stream=None):
    M, K, N = _row_shapes(X, W, Y, P_out, n_shards)
    out_t = _dtype_code(Y.dtype) if Y is not None else TP_F32
    st = lib().tp_row_linear(_ptr(X), _ptr(W), _ptr(Y), _ptr(P_out), M, K, N, n_shards,
                             _dtype_code(X.dtype), out_t, _stream(stream))
    _check("tp_row_linear", st)


def tp_sharded_linear(X, W, Y, n_shards=1, split=TP_SPLIT_COLS, act=None, stream=None):
    M, K, N = _row_shapes(X, W, Y, None, n_shards)
    st = lib().tp_sharded_linear(_ptr(X), _ptr(W), _ptr(Y), M, K, N, n_shards, split,
                                 _dtype_code(X.dtype), _dtype_code(Y.dtype), _act(act),
                                 _stream(stream))
    _check("tp_sharded_linear", st)


def tp_shard_reduce(P, Y, stream=None):
    import torch
    n, rows, cols = _dims(P, 3, "P")
    _expect(P, (n, rows, cols), "P", torch.float32)
    _expect(Y, (rows, cols), "Y")
    st = lib().tp_shard_reduce(_ptr(P), _ptr(Y), rows, cols, n, _dtype_code(Y.dtype),
                               _stream(stream))
    _check("tp_shard_reduce", st)


def tp_shard_concat(Ys, Y, stream=None):
    n, rows, sc = _dims(Ys, 3, "Ys")
    _expect(Y, (rows, n * sc), "Y", Ys.dtype)
    st = lib().tp_shard_concat(_ptr(Ys), _ptr(Y), rows, sc, n, _dtype_code(Ys.dtype),
                               _stream(stream))
    _check("tp_shard_concat", st)


def tp_shard_concat_grouped(Ys, Y, col_groups=1, stream=None):
    n, rows, sc = _dims(Ys, 3, "Ys")
    _expect(Y, (rows, n * sc), "Y", Ys.dtype)
    st = lib().tp_shard_concat_grouped(_ptr(Ys), _ptr(Y), rows, sc, n, col_groups,
                                       _dtype_code(Ys.dtype), _stream(stream))
    _check("tp_shard_concat_grouped", st)


def tp_mlp_block_workspace_size(M, f, dtype) -> int:
    return int(lib().tp_mlp_block_workspace_size(M, f, _dtype_code(dtype)))


def _mlp_shapes(X, W1, W2, Y, b1=None, b2=None):
    M, d = _dims(X, 2, "X")
    d1, f = _dims(W1, 2, "W1")
    if d1 != d:
        raise ValueError(f"W1 has {d1} rows, X has {d} columns")
    _expect(W2, (f, d), "W2")
    _expect(Y, (M, d), "Y")
    _expect(b1, (f,), "b1")
    _expect(b2, (d,), "b2")
    _same_dtype([("X", X), ("W1", W1), ("W2", W2), ("b1", b1), ("b2", b2)])
    return M, d, f


def tp_mlp_block(X, W1, W2, Y, ws, n_shards=1, stream=None):
    M, d, f = _mlp_shapes(X, W1, W2, Y)
    st = lib().tp_mlp_block(_ptr(X), _ptr(W1), _ptr(W2), _ptr(Y), _ptr(ws),
                            _ws_bytes(ws), M, d, f, n_shards,
                            _dtype_code(X.dtype), _dtype_code(Y.dtype), _stream(stream))
    _check("tp_mlp_block", st)


def tp_qkv_linear(X, W, Y, Y_shards=None, n_q_heads=1, n_kv_heads=1, head_dim=1, n_shards=1,
                  stream=None):
    M, K = _dims(X, 2, "X")
    _same_dtype([("X", X), ("W", W)])
    _same_dtype([("Y", Y), ("Y_shards", Y_shards)])
    N = (n_q_heads + 2 * n_kv_heads) * head_dim
    _expect(W, (K, N), "W")
    _expect(Y, (M, N), "Y")
    if (Y_shards is not None and n_shards >= 1 and n_kv_heads >= 1 and n_q_heads % n_shards == 0
            and (n_kv_heads % n_shards == 0 or n_shards % n_kv_heads == 0)):
        kvs = n_kv_heads // n_shards if n_kv_heads >= n_shards else 1
        _expect(Y_shards, (n_shards, M, (n_q_heads // n_shards + 2 * kvs) * head_dim), "Y_shards")
    st = lib().tp_qkv_linear(_ptr(X), _ptr(W), _ptr(Y), _ptr(Y_shards), M, K, n_q_heads,
                             n_kv_heads, head_dim, n_shards, _dtype_code(X.dtype),
                             _dtype_code(Y.dtype), _stream(stream))
    _check("tp_qkv_linear", st)


def tp_column_linear_bias(X, W, bias, Y=None, Y_shards=None, n_shards=1, act=None, stream=None):
    M, K, N = _column_shapes(X, W, Y, Y_shards, n_shards, bias)
    st = lib().tp_column_linear_bias(_ptr(X), _ptr(W), _ptr(bias), _ptr(Y), _ptr(Y_shards), M, K,
                                     N, n_shards, _dtype_code(X.dtype),
                                     _dtype_code(_out_dtype(Y, Y_shards)), _act(act),
                                     _stream(stream))
    _check("tp_column_linear_bias", st)


def tp_row_linear_bias(X, W, bias, Y=None, P_out=None, n_shards=1, stream=None):
    M, K, N = _row_shapes(X, W, Y, P_out, n_shards, bias)
    out_t = _dtype_code(Y.dtype) if Y is not None else TP_F32
    st = lib().tp_row_linear_bias(_ptr(X), _ptr(W), _ptr(bias), _ptr(Y), _ptr(P_out), M, K, N,
                                  n_shards, _dtype_code(X.dtype), out_t, _stream(stream))
    _check("tp_row_linear_bias", st)


def tp_mlp_block_bias(X, W1, b1, W2, b2, Y, ws, n_shards=1, stream=None):
    M, d, f = _mlp_shapes(X, W1, W2, Y, b1, b2)
    st = lib().tp_mlp_block_bias(_ptr(X), _ptr(W1), _ptr(b1), _ptr(W2), _ptr(b2), _ptr(Y),
                                 _ptr(ws), _ws_bytes(ws), M, d, f, n_shards,
                                 _dtype_code(X.dtype), _dtype_code(Y.dtype), _stream(stream))
    _check("tp_mlp_block_bias", st)


def _grad_dtype(*ts):
    for t in ts:
        if t is not None:
            return _dtype_code(t.dtype)
    return TP_F32


def _linear_backward_shapes(X, W, dY, dX, dW):
    M, K = _dims(X, 2, "X")
    K2, N = _dims(W, 2, "W")
    if K2 != K:
        raise ValueError(f"W has {K2} rows, X has {K} columns")
    _expect(dY, (M, N), "dY")
    _expect(dX, (M, K), "dX")
    _expect(dW, (K, N), "dW")
    _same_dtype([("X", X), ("W", W), ("dY", dY)])
    _same_dtype([("dX", dX), ("dW", dW)])
    return M, K, N


def tp_column_linear_backward(X, W, dY, dX=None, dW=None, n_shards=1, stream=None):
    M, K, N = _linear_backward_shapes(X, W, dY, dX, dW)
    st = lib().tp_column_linear_backward(_ptr(X), _ptr(W), _ptr(dY), _ptr(dX), _ptr(dW), M, K, N,
                                         n_shards, _dtype_code(X.dtype), _grad_dtype(dX, dW),
                                         _stream(stream))
    _check("tp_column_linear_backward", st)


def tp_row_linear_backward(X, W, dY, dX=None, dW=None, n_shards=1, stream=None):
    M, K, N = _linear_backward_shapes(X, W, dY, dX, dW)
    st = lib().tp_row_linear_backward(_ptr(X), _ptr(W), _ptr(dY), _ptr(dX), _ptr(dW), M, K, N,
                                      n_shards, _dtype_code(X.dtype), _grad_dtype(dX, dW),
                                      _stream(stream))
    _check("tp_row_linear_backward", st)


def tp_mlp_block_backward_workspace_size(M, f, dtype) -> int:
    return int(lib().tp_mlp_block_backward_workspace_size(M, f, _dtype_code(dtype)))


def tp_mlp_block_backward(X, W1, W2, dY, ws, dX=None, dW1=None, dW2=None, n_shards=1,
                          stream=None):
    M, d, f = _mlp_shapes(X, W1, W2, dY)
    _same_dtype([("X", X), ("dY", dY)])
    _expect(dX, (M, d), "dX")
    _expect(dW1, (d, f), "dW1")
    _expect(dW2, (f, d), "dW2")
    _same_dtype([("dX", dX), ("dW1", dW1), ("dW2", dW2)])
    st = lib().tp_mlp_block_backward(_ptr(X), _ptr(W1), _ptr(W2), _ptr(dY), _ptr(dX), _ptr(dW1),
                                     _ptr(dW2), _ptr(ws), _ws_bytes(ws), M, d, f,
                                     n_shards, _dtype_code(X.dtype), _grad_dtype(dX, dW1, dW2),
                                     _stream(stream))
    _check("tp_mlp_block_backward", st)


def tp_mlp_block_static_ws(X, W1, W2, Y, n_shards=1, stream=None):
    """tp_mlp_block with the library's fixed scratch instead of a workspace
    (for callers that cannot allocate device memory)."""
    M, d, f = _mlp_shapes(X, W1, W2, Y)
    st = lib().tp_mlp_block_static_ws(_ptr(X), _ptr(W1), _ptr(W2), _ptr(Y), M, d, f, n_shards,
                                      _dtype_code(X.dtype), _dtype_code(Y.dtype),
                                      _stream(stream))
    _check("tp_mlp_block_static_ws", st)


def tp_get_device_status(stream=None) -> int:
    """Synchronise and return the device status code (TP_OK or an error)."""
    return int(lib().tp_get_device_status(_stream(stream)))


def tp_selftest_bounded_wait(limit_ns: int, stream=None) -> None:
    _check("tp_selftest_bounded_wait", lib().tp_selftest_bounded_wait(limit_ns, _stream(stream)))


def tp_status_string(status: int) -> str:
    return lib().tp_status_string(status).decode()
