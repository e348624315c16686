"""Host-side tests of the C ABI (no GPU needed).

The library must load and export every entry point that include/tp.h
declares, and argument validation must reject bad calls synchronously,
before any CUDA call.  Every call here either fails validation or has no
work to do, so none of them reaches a kernel launch (the fake pointers are
never dereferenced)."""
import ctypes
import os
import re

import pytest

from tensor_sharded_linear_02_b300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tp.h")

OK, NULL, SHAPE, DIV, ALIGN, DTYPE, WS, CUDA, TIMEOUT, ALIAS = range(10)
F32, BF16 = 0, 1
A = 0x10000000  # fake, 16-byte aligned device addresses; never dereferenced
B = 0x20000000
C = 0x30000000
D = 0x40000000


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.lib()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+char\s*\*|tp_status|size_t)\s*(tp_\w+)\s*\(",
                                 text, flags=re.M)))


def test_header_declares_the_five_entry_points():
    names = _declared_functions()
    for n in ("tp_column_linear", "tp_row_linear", "tp_shard_reduce", "tp_shard_concat",
              "tp_mlp_block"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), f"{n} declared in tp.h but not exported"
        assert n in binding.SIGNATURES, f"{n} has no binding"


def test_status_strings(lib):
    for code in range(10):
        s = lib.tp_status_string(code).decode()
        assert s.startswith("TP_")
    assert lib.tp_status_string(0).decode() == "TP_OK"
    assert lib.tp_status_string(12345).decode() == "TP_ERR_UNKNOWN"


def test_workspace_size(lib):
    assert lib.tp_mlp_block_workspace_size(2048, 4096, BF16) == 2048 * 4096 * 2
    assert lib.tp_mlp_block_workspace_size(3, 5, BF16) == 256  # rounded up to 256 bytes
    assert lib.tp_mlp_block_workspace_size(3, 5, F32) == 256
    assert lib.tp_mlp_block_workspace_size(-1, 5, F32) == 0
    assert lib.tp_mlp_block_workspace_size(0, 5, F32) == 0


def _col(lib, X=A, W=B, Y=C, Ys=None, M=16, K=32, N=64, n=2, it=BF16, ot=BF16, act=0):
    return lib.tp_column_linear(X, W, Y, Ys, M, K, N, n, it, ot, act, None)


def _row(lib, X=A, W=B, Y=C, P=None, M=16, K=32, N=64, n=2, it=BF16, ot=BF16):
    return lib.tp_row_linear(X, W, Y, P, M, K, N, n, it, ot, None)


def test_column_validation(lib):
    assert _col(lib, X=None) == NULL
    assert _col(lib, Y=None, Ys=None) == NULL
    assert _col(lib, M=-1) == SHAPE
    assert _col(lib, M=1 << 31) == SHAPE
    assert _col(lib, n=0) == DIV
    assert _col(lib, n=65) == DIV
    assert _col(lib, N=64, n=3) == DIV
    assert _col(lib, X=A + 2) == ALIGN           # bf16 path needs 16-byte alignment
    assert _col(lib, K=36) == ALIGN              # row pitch 72 bytes
    assert _col(lib, N=20, n=1) == ALIGN         # row pitch 40 bytes
    assert _col(lib, Ys=D, N=48, n=4) == ALIGN   # shard width 12 columns
    assert _col(lib, it=7) == DTYPE
    assert _col(lib, act=5) == DTYPE
    assert _col(lib, Y=A + 64) == ALIAS          # Y overlaps X
    assert _col(lib, Ys=B) == ALIAS              # Y_shards overlaps W
    assert _col(lib, M=0) == OK                  # nothing to do, no launch
    assert _col(lib, N=0) == OK
    assert lib.tp_column_linear_grouped(A, B, C, None, 16, 32, 64, 2, 3, BF16, BF16, 0, None) == DIV
    assert lib.tp_column_linear_grouped(A, B, C, None, 16, 32, 60, 2, 3, BF16, BF16, 0, None) == ALIGN
    assert lib.tp_column_linear_grouped(A, B, C, None, 16, 32, 96, 2, 0, BF16, BF16, 0, None) == DIV


def test_fp32_path_alignment_is_4_bytes(lib):
    assert _col(lib, X=A + 2, it=F32, ot=F32) == ALIGN
    assert _col(lib, M=0, X=A + 4, K=5, N=6, n=3, it=F32, ot=F32) == OK


def test_row_validation(lib):
    assert _row(lib, W=None) == NULL
    assert _row(lib, Y=None, P=None) == NULL
    assert _row(lib, K=30, n=4) == DIV
    assert _row(lib, P=D, K=32, n=8) == ALIGN    # K/n = 4 columns per shard
    assert _row(lib, Y=B + 16) == ALIAS
    assert _row(lib, P=A) == ALIAS
    assert _row(lib, M=0) == OK
    assert lib.tp_sharded_linear(A, B, C, 16, 32, 64, 2, 1, BF16, BF16, 1, None) == DTYPE
    assert lib.tp_sharded_linear(A, B, C, 16, 32, 64, 2, 9, BF16, BF16, 0, None) == SHAPE


def test_reduce_and_concat_validation(lib):
    assert lib.tp_shard_reduce(None, C, 4, 8, 2, BF16, None) == NULL
    assert lib.tp_shard_reduce(A, C, -1, 8, 2, BF16, None) == SHAPE
    assert lib.tp_shard_reduce(A, C, 4, 8, 0, BF16, None) == DIV
    assert lib.tp_shard_reduce(A + 4, C, 4, 8, 2, BF16, None) == ALIGN
    assert lib.tp_shard_reduce(A, A + 32, 4, 8, 2, BF16, None) == ALIAS
    assert lib.tp_shard_reduce(A, C, 4, 8, 2, 3, None) == DTYPE
    assert lib.tp_shard_reduce(A, C, 0, 8, 2, BF16, None) == OK
    assert lib.tp_shard_concat(A, C, 4, 12, 2, BF16, None) == ALIGN   # 12 bf16 = 24 bytes
    assert lib.tp_shard_concat(A, A + 16, 4, 16, 2, BF16, None) == ALIAS
    assert lib.tp_shard_concat_grouped(A, C, 4, 48, 2, 5, BF16, None) == DIV
    assert lib.tp_shard_concat(A, C, 0, 16, 2, BF16, None) == OK


def test_mlp_validation(lib):
    def mlp(X=A, W1=B, W2=C, Y=D, ws=0x50000000, wsb=1 << 20, M=16, d=32, f=64, n=2,
            it=BF16, ot=BF16):
        return lib.tp_mlp_block(X, W1, W2, Y, ws, wsb, M, d, f, n, it, ot, None)
    assert mlp(W2=None) == NULL
    assert mlp(f=60, n=8) == DIV
    assert mlp(ws=None) == WS
    assert mlp(wsb=16 * 64 * 2 - 1) == WS
    assert mlp(ws=A) == ALIAS
    assert mlp(Y=C) == ALIAS
    assert mlp(d=36) == ALIGN
    assert mlp(M=0) == OK


def test_binding_refuses_host_tensors():
    """The binding hands the C ABI device pointers only: a CPU tensor is
    refused before any call."""
    import torch
    X = torch.zeros(4, 8, dtype=torch.bfloat16)
    W = torch.zeros(8, 16, dtype=torch.bfloat16)
    Y = torch.zeros(4, 16, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        binding.tp_column_linear(X, W, Y, None, n_shards=2)


def test_binding_checks_every_shape_before_the_call():
    """The C ABI sees bare pointers, so an output or second operand smaller
    than the call's sizes imply would be read or written past its end: the
    binding compares every tensor's shape and dtype with the sizes it
    derives from X and W (or W1) and raises before any call.  (CPU tensors:
    the shape checks come first, the device check last.)"""
    import torch
    bf, f32 = torch.bfloat16, torch.float32
    X = torch.zeros(4, 8, dtype=bf)
    W = torch.zeros(8, 16, dtype=bf)
    cases = [
        (lambda: binding.tp_column_linear(X, W, torch.zeros(4, 15, dtype=bf), n_shards=2), "Y"),
        (lambda: binding.tp_column_linear(X, torch.zeros(7, 16, dtype=bf), None,
                                          torch.zeros(2, 4, 8, dtype=bf), n_shards=2), "rows"),
        (lambda: binding.tp_column_linear(X, W, None, torch.zeros(2, 4, 7, dtype=bf),
                                          n_shards=2), "Y_shards"),
        (lambda: binding.tp_column_linear(X, W.float(), torch.zeros(4, 16, dtype=bf)), "dtype"),
        (lambda: binding.tp_column_linear(X, W, torch.zeros(4, 16, dtype=bf),
                                          torch.zeros(2, 4, 8, dtype=f32), n_shards=2), "dtype"),
        (lambda: binding.tp_column_linear_bias(X, W, torch.zeros(15, dtype=bf),
                                               torch.zeros(4, 16, dtype=bf)), "bias"),
        (lambda: binding.tp_row_linear(X, W, torch.zeros(4, 16, dtype=bf),
                                       torch.zeros(2, 4, 16, dtype=bf), n_shards=2), "P_out"),
        (lambda: binding.tp_row_linear(X, W, None, torch.zeros(3, 4, 16, dtype=f32),
                                       n_shards=2), "P_out"),
        (lambda: binding.tp_shard_reduce(torch.zeros(2, 4, 16, dtype=f32),
                                         torch.zeros(4, 8, dtype=bf)), "Y"),
        (lambda: binding.tp_shard_reduce(torch.zeros(2, 4, 16, dtype=bf),
                                         torch.zeros(4, 16, dtype=bf)), "P"),
        (lambda: binding.tp_shard_concat(torch.zeros(2, 4, 8, dtype=bf),
                                         torch.zeros(4, 15, dtype=bf)), "Y"),
        (lambda: binding.tp_shard_concat_grouped(torch.zeros(2, 4, 8, dtype=bf),
                                                 torch.zeros(4, 16, dtype=f32)), "dtype"),
        (lambda: binding.tp_mlp_block(X, W, torch.zeros(16, 7, dtype=bf),
                                      torch.zeros(4, 8, dtype=bf), torch.zeros(256, dtype=torch.uint8)),
         "W2"),
        (lambda: binding.tp_mlp_block(X, W, torch.zeros(16, 8, dtype=bf),
                                      torch.zeros(5, 8, dtype=bf), torch.zeros(256, dtype=torch.uint8)),
         "Y"),
        (lambda: binding.tp_mlp_block(X, W, torch.zeros(16, 8, dtype=f32),
                                      torch.zeros(4, 8, dtype=bf), torch.zeros(256, dtype=torch.uint8)),
         "dtype"),
        (lambda: binding.tp_mlp_block_bias(X, W, torch.zeros(8, dtype=bf), torch.zeros(16, 8, dtype=bf),
                                           None, torch.zeros(4, 8, dtype=bf),
                                           torch.zeros(256, dtype=torch.uint8)), "b1"),
        (lambda: binding.tp_mlp_block_static_ws(X, W, torch.zeros(16, 8, dtype=bf),
                                                torch.zeros(4, 9, dtype=bf)), "Y"),
        (lambda: binding.tp_qkv_linear(X, torch.zeros(8, 6 * 4, dtype=bf),
                                       torch.zeros(4, 6 * 4, dtype=bf), None, n_q_heads=4,
                                       n_kv_heads=2, head_dim=4), "W"),
        (lambda: binding.tp_qkv_linear(X, torch.zeros(8, 8 * 4, dtype=bf),
                                       torch.zeros(4, 8 * 4, dtype=bf),
                                       torch.zeros(2, 4, 12, dtype=bf), n_q_heads=4,
                                       n_kv_heads=2, head_dim=4, n_shards=2), "Y_shards"),
        (lambda: binding.tp_column_linear_backward(X, W, torch.zeros(4, 16, dtype=bf),
                                                   torch.zeros(4, 7, dtype=bf)), "dX"),
        (lambda: binding.tp_row_linear_backward(X, W, torch.zeros(3, 16, dtype=bf)), "dY"),
        (lambda: binding.tp_mlp_block_backward(X, W, torch.zeros(16, 8, dtype=bf),
                                               torch.zeros(4, 8, dtype=bf),
                                               torch.zeros(256, dtype=torch.uint8),
                                               dW2=torch.zeros(8, 16, dtype=bf)), "dW2"),
        (lambda: binding.tp_column_linear(torch.zeros(4, 8, 1, dtype=bf), W, None), "dimensions"),
    ]
    for fn, what in cases:
        with pytest.raises(ValueError, match=what):
            fn()
    # a consistent call gets past the shape checks and stops at the device check
    with pytest.raises(ValueError, match="CUDA"):
        binding.tp_row_linear(X, W, torch.zeros(4, 16, dtype=bf),
                              torch.zeros(2, 4, 16, dtype=f32), n_shards=2)


def test_absurd_sizes_are_refused_without_overflow(lib):
    """Sizes whose products would overflow 64-bit byte counts (or exceed any
    device's memory) are refused with TP_ERR_SHAPE before anything else."""
    big = (1 << 31) - 1
    assert _col(lib, M=big, K=big, N=64) == SHAPE
    assert _col(lib, M=16, K=big, N=big - 7) == SHAPE
    assert _row(lib, M=big, K=32, N=big - 7) == SHAPE
    assert lib.tp_shard_reduce(A, C, 1 << 40, 1 << 30, 2, BF16, None) == SHAPE
    assert lib.tp_shard_concat(A, C, 1 << 40, 1 << 30, 2, BF16, None) == SHAPE
    assert lib.tp_qkv_linear(A, B, C, None, 16, 32, big, big, big, 1, BF16, BF16, None) == SHAPE
    assert lib.tp_mlp_block_workspace_size(1 << 33, 1 << 31, BF16) == 0
    assert lib.tp_mlp_block_workspace_size(big, big, BF16) == 0
    assert lib.tp_mlp_block_backward_workspace_size(big, big, BF16) == 0
    assert lib.tp_mlp_block(A, B, C, D, 0x50000000, 1 << 20, big, big, 8, 2, BF16, BF16,
                            None) == SHAPE
