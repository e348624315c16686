"""fp64 host oracle for the tensor-parallel sharded linear layer and MLP block.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, the smoke check in
``__graft_entry__.py`` and the CPU-baseline / reference arm of ``bench.py``
may import this package.  The CUDA library never calls it and it never calls
the CUDA library; the two share only the seeded input generator, which holds
none of the method's arithmetic.

The arithmetic lives in ``oracle.c`` (plain loops, double accumulation); this
module only compiles it with the host C compiler, loads it and marshals numpy
arrays.  Every function states the passage it follows:

* [TP-topic]  chipfoundryservices.com topic page "Tensor Parallelism":
  "Tensor Parallelism Fundamentals", "Column-Wise Parallelism",
  "Row-Wise Parallelism", "Megatron-LM Tensor Parallelism", SVG figure panel
  "Attention Head Parallelism".
* [Glossary]  aiforbusinessandlife.com glossary "Tensor Parallelism":
  "How it works", "Worked example", "Check your understanding".

Readings taken where the pages are silent or garbled (each is also listed in
the design notes):

* Row split: the Fundamentals bullet prints the per-device product as
  "X_i.W"; the Row-Wise section and the worked example split the contracted
  dimension of both X and W, Y_i = X_i.W_i.  The latter is used.
* Combine after a column split is a concat (Column-Wise section, glossary
  worked example); the figure's "all-reduce" box belongs to the MLP pair.
* The activation is the exact GeLU, x*Phi(x), with the host libm erf.
* Partials are summed in ascending shard order.
* Head-group split for the QKV projection: columns form G blocks (Q|K|V) and
  shard i owns the i-th contiguous slice of each block.
* Sequence parallelism: shard i owns token rows [i*M/n, (i+1)*M/n) outside
  the tensor-parallel block; after the block's all-reduce each shard keeps
  its own token rows (a reduce-scatter over token rows).

Parity pins for each function are in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_fp = ctypes.POINTER(ctypes.c_float)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_i64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with the host C compiler.

    Portable flags only (no -march=native): the library may be built on one
    host and run on another.  No -ffast-math, so every double operation is
    IEEE round-to-nearest and no sum is reassociated.
    """
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp",
               "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        lib.orc_matmul.argtypes = [_dp, _dp, _dp, _i64, _i64, _i64]
        lib.orc_gelu.argtypes = [ctypes.c_double]
        lib.orc_gelu.restype = ctypes.c_double
        lib.orc_gelu_inplace.argtypes = [_dp, _i64]
        lib.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.orc_bf16_to_double.restype = ctypes.c_double
        lib.orc_bf16_from_double.argtypes = [ctypes.c_double]
        lib.orc_bf16_from_double.restype = ctypes.c_uint16
        lib.orc_bf16_to_double_array.argtypes = [_u16p, _dp, _i64]
        lib.orc_double_to_bf16_array.argtypes = [_dp, _u16p, _i64]
        lib.orc_column_linear.argtypes = [_dp, _dp, _dp, _dp, _dp, _i64, _i64, _i64,
                                          _i64, _i64, ctypes.c_int]
        lib.orc_row_linear.argtypes = [_dp, _dp, _dp, _dp, _dp, _i64, _i64, _i64, _i64]
        lib.orc_mlp_block.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp, _i64, _i64, _i64, _i64,
                                      ctypes.c_int]
        lib.orc_qkv_linear.argtypes = [_dp, _dp, _dp, _dp, _i64, _i64, _i64, _i64, _i64, _i64]
        lib.orc_gelu_grad.argtypes = [ctypes.c_double]
        lib.orc_gelu_grad.restype = ctypes.c_double
        lib.orc_column_linear_backward.argtypes = [_dp, _dp, _dp, _dp, _dp, _i64, _i64, _i64,
                                                   _i64]
        lib.orc_row_linear_backward.argtypes = [_dp, _dp, _dp, _dp, _dp, _i64, _i64, _i64, _i64]
        lib.orc_mlp_block_backward.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp, _dp, _i64, _i64,
                                               _i64, _i64]
        _i64p = ctypes.POINTER(ctypes.c_int64)
        lib.orc_mlp_block_backward_sampled.argtypes = [_dp, _dp, _dp, _dp, _i64, _i64, _i64, _i64,
                                                       _i64p, _i64, _i64p, _i64, _i64p, _i64,
                                                       _dp, _dp, _dp]
        lib.orc_shard_reduce.argtypes = [_fp, _dp, _i64, _i64, _i64]
        lib.orc_shard_concat.argtypes = [_dp, _dp, _i64, _i64, _i64, _i64]
        lib.orc_allgather_rows.argtypes = [_dp, _dp, _i64, _i64, _i64]
        lib.orc_reduce_scatter_rows.argtypes = [_dp, _dp, _i64, _i64, _i64]
        lib.orc_seq_parallel_mlp_block.argtypes = [_dp, _dp, _dp, _dp, _i64, _i64, _i64, _i64]
        _lib = lib
        return lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a: np.ndarray, typ=_dp):
    return a.ctypes.data_as(typ) if a is not None else None


def set_threads(n: int) -> None:
    """Number of host threads the OpenMP loops use (row-parallel only)."""
    os.environ["OMP_NUM_THREADS"] = str(int(n))
    try:
        libgomp = ctypes.CDLL("libgomp.so.1")
        libgomp.omp_set_num_threads(ctypes.c_int(int(n)))
    except OSError:
        pass


# ----------------------------------------------------------------- bf16 -----

def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact double values (format definition)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    _load().orc_bf16_to_double_array(_ptr(b, _u16p), _ptr(out), b.size)
    return out


def f64_to_bf16(x: np.ndarray) -> np.ndarray:
    """double -> bf16 bit patterns, round to nearest, ties to even."""
    a = _f64(x)
    out = np.empty(a.shape, dtype=np.uint16)
    _load().orc_double_to_bf16_array(_ptr(a), _ptr(out, _u16p), a.size)
    return out


# ----------------------------------------------------------------- maths ----

def gelu(x) -> np.ndarray:
    """Exact GeLU x*Phi(x) applied elementwise ([TP-topic] Megatron-LM, MLP
    layer splitting: the activation is applied to each shard independently)."""
    a = _f64(x).copy()
    _load().orc_gelu_inplace(_ptr(a), a.size)
    return a


def matmul(X, W) -> np.ndarray:
    """Unsharded Y = X.W ([TP-topic] Fundamentals), naive loops in double."""
    X, W = _f64(X), _f64(W)
    M, K = X.shape
    K2, N = W.shape
    assert K == K2
    Y = np.empty((M, N), dtype=np.float64)
    _load().orc_matmul(_ptr(X), _ptr(W), _ptr(Y), M, K, N)
    return Y


def column_linear(X, W, n_shards: int, col_groups: int = 1, act: str | None = None, bias=None):
    """Column-parallel linear ([TP-topic] "Column-Wise Parallelism").

    Returns (Y, Ys): the concatenated output [M, N] and the shard-major local
    outputs [n_shards, M, N/n_shards].  ``act='gelu'`` applies the exact GeLU
    to each shard's output before the concat; ``bias`` [N] is split with W's
    columns and added by each shard before the activation.
    """
    X, W = _f64(X), _f64(W)
    b = None if bias is None else _f64(bias)
    M, K = X.shape
    _, N = W.shape
    assert N % col_groups == 0 and (N // col_groups) % n_shards == 0
    Y = np.empty((M, N), dtype=np.float64)
    Ys = np.empty((n_shards, M, N // n_shards), dtype=np.float64)
    _load().orc_column_linear(_ptr(X), _ptr(W), _ptr(b), _ptr(Y), _ptr(Ys), M, K, N,
                              n_shards, col_groups, 1 if act == "gelu" else 0)
    return Y, Ys


def qkv_kv_heads_per_shard(hq: int, hkv: int, n_shards: int) -> int:
    """KV heads each shard holds under the GQA split (see qkv_linear)."""
    assert hq % n_shards == 0 and (hkv % n_shards == 0 or n_shards % hkv == 0)
    return hkv // n_shards if hkv >= n_shards else 1


def qkv_linear(X, W, hq: int, hkv: int, hd: int, n_shards: int):
    """QKV projection with grouped-query heads ([TP-topic] SVG figure,
    "Attention Head Parallelism": split Q heads evenly, replicate the shared
    KV heads).  W = [Wq | Wk | Wv] [K, (hq + 2 hkv) hd].  Returns (Y, Ys): the
    full projection [M, (hq+2hkv) hd] and the shard-local outputs
    [n, M, (hq/n + 2 kvs) hd], each ordered Q | K | V."""
    X, W = _f64(X), _f64(W)
    M, K = X.shape
    kvs = qkv_kv_heads_per_shard(hq, hkv, n_shards)
    assert W.shape == (K, (hq + 2 * hkv) * hd)
    Y = np.empty((M, (hq + 2 * hkv) * hd))
    Ys = np.empty((n_shards, M, (hq // n_shards + 2 * kvs) * hd))
    _load().orc_qkv_linear(_ptr(X), _ptr(W), _ptr(Y), _ptr(Ys), M, K, hq, hkv, hd, n_shards)
    return Y, Ys


def row_linear(X, W, n_shards: int, bias=None):
    """Row-parallel linear ([TP-topic] "Row-Wise Parallelism").

    Returns (Y, P): Y = sum of the shard partials (ascending shard order),
    plus ``bias`` [N] once after the sum if given, and the bias-free
    partials P [n_shards, M, N].
    """
    X, W = _f64(X), _f64(W)
    b = None if bias is None else _f64(bias)
    M, K = X.shape
    _, N = W.shape
    assert K % n_shards == 0
    Y = np.empty((M, N), dtype=np.float64)
    P = np.empty((n_shards, M, N), dtype=np.float64)
    _load().orc_row_linear(_ptr(X), _ptr(W), _ptr(b), _ptr(Y), _ptr(P), M, K, N, n_shards)
    return Y, P


def mlp_block(X, W1, W2, n_shards: int, mirror_h_bf16: bool = False, b1=None,
              b2=None) -> np.ndarray:
    """Megatron-style MLP block ([TP-topic] Megatron-LM, "MLP Layer Splitting"):
    Y = sum_i GeLU(X.W1_i + b1_i).W2_i + b2 with W1 (and b1) split by columns
    and W2 by rows; b2 is added once after the sum."""
    X, W1, W2 = _f64(X), _f64(W1), _f64(W2)
    c1 = None if b1 is None else _f64(b1)
    c2 = None if b2 is None else _f64(b2)
    M, d = X.shape
    _, f = W1.shape
    assert W2.shape == (f, d) and f % n_shards == 0
    Y = np.empty((M, d), dtype=np.float64)
    _load().orc_mlp_block(_ptr(X), _ptr(W1), _ptr(c1), _ptr(W2), _ptr(c2), _ptr(Y), M, d, f,
                          n_shards, 1 if mirror_h_bf16 else 0)
    return Y


# ------------------------------------------------------------- backward ----

def gelu_grad(x) -> np.ndarray:
    """GeLU'(x) = Phi(x) + x*phi(x), elementwise."""
    a = _f64(x)
    f = _load().orc_gelu_grad
    return np.vectorize(f, otypes=[np.float64])(a) if a.size else a.copy()


def column_linear_backward(X, W, dY, n_shards: int):
    """Backward of the column-parallel linear ([TP-topic] Megatron-LM,
    "Identity Operators": the forward identity on X is a sum over shards in
    the backward).  Returns (dX [M,K], dW [K,N]); dW's column block i is
    shard i's gradient, dX = sum_i dY_i . W_i^T in ascending shard order."""
    X, W, dY = _f64(X), _f64(W), _f64(dY)
    M, K = X.shape
    _, N = W.shape
    assert dY.shape == (M, N) and N % n_shards == 0
    dX = np.empty((M, K)); dW = np.empty((K, N))
    _load().orc_column_linear_backward(_ptr(X), _ptr(W), _ptr(dY), _ptr(dX), _ptr(dW), M, K, N,
                                       n_shards)
    return dX, dW


def row_linear_backward(X, W, dY, n_shards: int):
    """Backward of the row-parallel linear (the forward sum is an identity in
    the backward: every shard receives the full dY).  Returns (dX [M,K],
    dW [K,N]); shard i owns columns i of dX and rows i of dW."""
    X, W, dY = _f64(X), _f64(W), _f64(dY)
    M, K = X.shape
    _, N = W.shape
    assert dY.shape == (M, N) and K % n_shards == 0
    dX = np.empty((M, K)); dW = np.empty((K, N))
    _load().orc_row_linear_backward(_ptr(X), _ptr(W), _ptr(dY), _ptr(dX), _ptr(dW), M, K, N,
                                    n_shards)
    return dX, dW


def mlp_block_backward(X, W1, W2, dY, n_shards: int):
    """Backward of the MLP block for L = sum(Y * dY): returns (dX, dW1, dW2),
    each shard recomputing its pre-activation, dX summed over shards in
    ascending order ([TP-topic] Megatron-LM, "Identity Operators")."""
    X, W1, W2, dY = _f64(X), _f64(W1), _f64(W2), _f64(dY)
    M, d = X.shape
    _, f = W1.shape
    assert W2.shape == (f, d) and dY.shape == (M, d) and f % n_shards == 0
    dX = np.empty((M, d)); dW1 = np.empty((d, f)); dW2 = np.empty((f, d))
    _load().orc_mlp_block_backward(_ptr(X), _ptr(W1), _ptr(W2), _ptr(dY), _ptr(dX), _ptr(dW1),
                                   _ptr(dW2), M, d, f, n_shards)
    return dX, dW1, dW2


def mlp_block_backward_sampled(X, W1, W2, dY, n_shards: int, dx_rows, dw1_cols, dw2_rows):
    """The MLP block's backward on sampled outputs (for checks at sizes whose
    full fp64 backward is too slow): returns (dX[dx_rows, :],
    dW1[:, dw1_cols], dW2[dw2_rows, :]), each value by the same chain rule
    as mlp_block_backward, written per value."""
    X, W1, W2, dY = _f64(X), _f64(W1), _f64(W2), _f64(dY)
    M, d = X.shape
    _, f = W1.shape
    assert W2.shape == (f, d) and dY.shape == (M, d) and f % n_shards == 0
    rx = np.ascontiguousarray(dx_rows, dtype=np.int64)
    c1 = np.ascontiguousarray(dw1_cols, dtype=np.int64)
    r2 = np.ascontiguousarray(dw2_rows, dtype=np.int64)
    i64p = ctypes.POINTER(ctypes.c_int64)
    dXs = np.empty((rx.size, d)); dW1s = np.empty((d, c1.size)); dW2s = np.empty((r2.size, d))
    _load().orc_mlp_block_backward_sampled(_ptr(X), _ptr(W1), _ptr(W2), _ptr(dY), M, d, f,
                                           n_shards, _ptr(rx, i64p), rx.size, _ptr(c1, i64p),
                                           c1.size, _ptr(r2, i64p), r2.size, _ptr(dXs),
                                           _ptr(dW1s), _ptr(dW2s))
    return dXs, dW1s, dW2s


def shard_reduce(P) -> np.ndarray:
    """Sum of fp32 partials [n, rows, cols] over ascending shard, in double."""
    P = np.ascontiguousarray(P, dtype=np.float32)
    n, rows, cols = P.shape
    Y = np.empty((rows, cols), dtype=np.float64)
    _load().orc_shard_reduce(_ptr(P, _fp), _ptr(Y), rows, cols, n)
    return Y


def shard_concat(Ys, col_groups: int = 1) -> np.ndarray:
    """Concat of shard outputs [n, rows, sc] into [rows, n*sc] (column
    ownership as in column_linear)."""
    Ys = _f64(Ys)
    n, rows, sc = Ys.shape
    assert sc % col_groups == 0
    Y = np.empty((rows, n * sc), dtype=np.float64)
    _load().orc_shard_concat(_ptr(Ys), _ptr(Y), rows, sc, n, col_groups)
    return Y


# ------------------------------------------------- sequence parallelism ----

def allgather_rows(Xs) -> np.ndarray:
    """All-gather of token blocks before the tensor-parallel block
    ([TP-topic] "Sequence Parallelism Extension": every shard needs every
    token): Xs [n, M/n, cols] -> X [M, cols], shard i's rows i*M/n onward."""
    Xs = _f64(Xs)
    n, rb, cols = Xs.shape
    X = np.empty((n * rb, cols), dtype=np.float64)
    _load().orc_allgather_rows(_ptr(Xs), _ptr(X), n, rb, cols)
    return X


def reduce_scatter_rows(P) -> np.ndarray:
    """The combine after the block under sequence parallelism ([TP-topic]
    "Sequence Parallelism Extension"): the all-reduce of the shards'
    partial outputs P [n, M, cols] (ascending shard order), after which
    shard i keeps its own token rows: returns [n, M/n, cols]."""
    P = _f64(P)
    n, M, cols = P.shape
    assert M % n == 0
    Ys = np.empty((n, M // n, cols), dtype=np.float64)
    _load().orc_reduce_scatter_rows(_ptr(P), _ptr(Ys), n, M, cols)
    return Ys


def seq_parallel_mlp_block(Xs, W1, W2) -> np.ndarray:
    """MLP block between two sequence-split regions: token blocks
    Xs [n, M/n, d] are all-gathered, every shard i computes its partial
    GeLU(X.W1_i).W2_i for all tokens, and the partials are reduce-scattered
    over token rows: returns [n, M/n, d]."""
    Xs, W1, W2 = _f64(Xs), _f64(W1), _f64(W2)
    n, rb, d = Xs.shape
    _, f = W1.shape
    assert W1.shape == (d, f) and W2.shape == (f, d) and f % n == 0
    Ys = np.empty((n, rb, d), dtype=np.float64)
    _load().orc_seq_parallel_mlp_block(_ptr(Xs), _ptr(W1), _ptr(W2), _ptr(Ys), n, rb, d, f)
    return Ys
