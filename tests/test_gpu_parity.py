"""GPU parity: the CUDA path, called through the C ABI, against the fp64
oracle on the same seeded input bytes.  Sizes span several tiles with
ragged tails in every dimension and exercise each kernel path (persistent
tcgen05 GEMM with and without wrap-around, the cluster split with the
shared-memory exchange of partial rows, per-shard partial outputs, the CUDA-core fp32
path, the vector and scalar reduce, plain and head-group concat)."""
import numpy as np
import pytest

import oracle
from helpers import (assert_bf16_parity, bf16_dev_to_f64, dev_bits, dev_to_f64, to_dev_bf16,
                     to_dev_f32)
from tensor_sharded_linear_02_b300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tp():
    from tensor_sharded_linear_02_b300 import binding
    binding.lib()
    return binding


def _bf16_inputs(M, K, N, seed, xstd=1.0, wstd=0.02):
    xb = inputs.bf16_normal((M, K), inputs.stream_seed(seed, 0), xstd)
    wb = inputs.bf16_normal((K, N), inputs.stream_seed(seed, 1), wstd)
    return xb, wb


def _status_ok(tp):
    assert tp.tp_get_device_status() == tp.TP_OK


# ----------------------------------------------------------- fp32 exact -----

def test_worked_example_fp32(tp, cuda_device):
    """Glossary worked example on the device: X=[1,2], W rows [3,4,5,6] and
    [7,8,9,10] give [17,20,23,26]; halves [17,20]|[23,26]; row partials."""
    import torch
    X = to_dev_f32([[1, 2]], cuda_device)
    W = to_dev_f32([[3, 4, 5, 6], [7, 8, 9, 10]], cuda_device)
    Y = torch.empty(1, 4, device=cuda_device)
    Ys = torch.empty(2, 1, 2, device=cuda_device)
    tp.tp_column_linear(X, W, Y, Ys, n_shards=2)
    P = torch.empty(2, 1, 4, device=cuda_device)
    Yr = torch.empty(1, 4, device=cuda_device)
    tp.tp_row_linear(X, W, Yr, P, n_shards=2)
    _status_ok(tp)
    assert Y.cpu().tolist() == [[17, 20, 23, 26]]
    assert Ys.cpu().tolist() == [[[17, 20]], [[23, 26]]]
    assert P.cpu().tolist() == [[[3, 4, 5, 6]], [[14, 16, 18, 20]]]
    assert Yr.cpu().tolist() == [[17, 20, 23, 26]]


def test_tiny_integer_config_fp32(tp, cuda_device):
    """X [16,32], W [32,64], integers uniform in [-4,4] from seed 0, two
    shards: the column concat and the row sum both equal X.W exactly."""
    import torch
    X = inputs.int_uniform((16, 32), inputs.stream_seed(0, 0))
    W = inputs.int_uniform((32, 64), inputs.stream_seed(0, 1))
    ref = oracle.matmul(X, W)
    ref_c, ref_s = oracle.column_linear(X, W, 2)
    ref_r, ref_p = oracle.row_linear(X, W, 2)
    Xd, Wd = to_dev_f32(X, cuda_device), to_dev_f32(W, cuda_device)
    Y = torch.empty(16, 64, device=cuda_device)
    Ys = torch.empty(2, 16, 32, device=cuda_device)
    tp.tp_column_linear(Xd, Wd, Y, Ys, n_shards=2)
    Yr = torch.empty(16, 64, device=cuda_device)
    P = torch.empty(2, 16, 64, device=cuda_device)
    tp.tp_row_linear(Xd, Wd, Yr, P, n_shards=2)
    Yf = torch.empty(16, 64, device=cuda_device)
    tp.tp_row_linear(Xd, Wd, Yf, None, n_shards=2)
    Yc = torch.empty(16, 64, device=cuda_device)
    tp.tp_shard_concat(Ys, Yc)
    Yred = torch.empty(16, 64, device=cuda_device)
    tp.tp_shard_reduce(P, Yred)
    _status_ok(tp)
    for got in (Y, Yr, Yf, Yc, Yred):
        np.testing.assert_array_equal(dev_to_f64(got), ref)
    np.testing.assert_array_equal(dev_to_f64(Ys), ref_s)
    np.testing.assert_array_equal(dev_to_f64(P), ref_p)
    np.testing.assert_array_equal(ref_c, ref)
    np.testing.assert_array_equal(ref_r, ref)


@pytest.mark.parametrize("M,K,N,n", [(7, 5, 9, 3), (33, 12, 20, 4), (1, 1, 1, 1)])
def test_fp32_ragged_integer(tp, cuda_device, M, K, N, n):
    import torch
    X = inputs.int_uniform((M, K), inputs.stream_seed(5, 0))
    W = inputs.int_uniform((K, N), inputs.stream_seed(5, 1))
    ref = oracle.matmul(X, W)
    Xd, Wd = to_dev_f32(X, cuda_device), to_dev_f32(W, cuda_device)
    if N % n == 0:
        Y = torch.empty(M, N, device=cuda_device)
        tp.tp_column_linear(Xd, Wd, Y, None, n_shards=n)
        np.testing.assert_array_equal(dev_to_f64(Y), ref)
    if K % n == 0:
        Y = torch.empty(M, N, device=cuda_device)
        tp.tp_row_linear(Xd, Wd, Y, None, n_shards=n)
        np.testing.assert_array_equal(dev_to_f64(Y), ref)
    _status_ok(tp)


def test_fp32_mlp_block(tp, cuda_device):
    """fp32 MLP block on the CUDA-core path, against the oracle."""
    import torch
    M, d, f, n = 24, 16, 32, 4
    X = inputs.f32_normal((M, d), 41)
    W1 = inputs.f32_normal((d, f), 42, 0.2)
    W2 = inputs.f32_normal((f, d), 43, 0.2)
    Y = torch.empty(M, d, device=cuda_device)
    ws = torch.empty(tp.tp_mlp_block_workspace_size(M, f, torch.float32), dtype=torch.uint8,
                     device=cuda_device)
    tp.tp_mlp_block(to_dev_f32(X, cuda_device), to_dev_f32(W1, cuda_device),
                    to_dev_f32(W2, cuda_device), Y, ws, n_shards=n)
    _status_ok(tp)
    np.testing.assert_allclose(dev_to_f64(Y), oracle.mlp_block(X, W1, W2, n), rtol=1e-5,
                               atol=1e-5)


# ------------------------------------------------------ bf16 column split ---

COLUMN_CASES = [
    # M, K, N, n, act      path exercised
    (300, 328, 640, 2, None),     # cluster split, ragged M, K and N tails
    (300, 328, 640, 2, "gelu"),
    (2304, 136, 2080, 4, "gelu"),  # persistent, 162 tiles > SM count (TMEM ring wraps)
    (1280, 200, 2048, 8, None),    # persistent, exactly one tile per CTA or less
    (1, 64, 256, 1, None),         # one row
    (129, 8, 8, 1, "gelu"),        # K one vector, N one vector
]


@pytest.mark.parametrize("M,K,N,n,act", COLUMN_CASES)
def test_column_linear_bf16(tp, cuda_device, M, K, N, n, act):
    import torch
    xb, wb = _bf16_inputs(M, K, N, seed=M + K + N)
    X, W = to_dev_bf16(xb, cuda_device), to_dev_bf16(wb, cuda_device)
    Y = torch.empty(M, N, dtype=torch.bfloat16, device=cuda_device)
    Ys = torch.empty(n, M, N // n, dtype=torch.bfloat16, device=cuda_device)
    tp.tp_column_linear(X, W, Y, Ys, n_shards=n, act=act)
    Y1 = torch.empty(M, N, dtype=torch.bfloat16, device=cuda_device)
    tp.tp_column_linear(X, W, Y1, None, n_shards=1, act=act)
    Yf = torch.empty(M, N, dtype=torch.float32, device=cuda_device)
    tp.tp_column_linear(X, W, Yf, None, n_shards=n, act=act)
    _status_ok(tp)
    ref, ref_s = oracle.column_linear(oracle.bf16_to_f64(xb), oracle.bf16_to_f64(wb), n, act=act)
    assert_bf16_parity(bf16_dev_to_f64(Y), ref, "column Y")
    assert_bf16_parity(dev_to_f64(Yf), ref, "column Y fp32 out", out_bf16=False)
    # concat fused in the store == the shard outputs, bit for bit
    np.testing.assert_array_equal(dev_bits(Ys), dev_bits(Y).reshape(M, n, N // n).transpose(1, 0, 2))
    # sharded == unsharded launch, bit for bit
    np.testing.assert_array_equal(dev_bits(Y), dev_bits(Y1))
    # fp32 output rounds to the bf16 output
    np.testing.assert_array_equal(dev_bits(Yf.to(torch.bfloat16)), dev_bits(Y))


GELU_REL_TOL = 1e-4   # fp32 GeLU, relative, wherever |GeLU(x)| >= 1e-30
GELU_TINY = 1e-30


def _all_bf16_in(lo, hi):
    """Every finite bf16 value in [lo, hi] (bit patterns and values)."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = oracle.bf16_to_f64(bits)
    keep = np.isfinite(vals) & (vals >= lo) & (vals <= hi)
    return bits[keep], vals[keep]


def _bf16_ulp_distance(a_bits, b_bits):
    """Distance in representable bf16 values between two bit patterns
    (sign-magnitude mapped to a monotone integer line)."""
    def line(b):
        b = np.asarray(b).astype(np.uint16).astype(np.int64)
        mag = b & 0x7FFF
        return np.where(b & 0x8000, -mag, mag)
    return np.abs(line(a_bits) - line(b_bits))


def _identity_columns(N):
    """W [8, N] with W[k, j] = 1 for j % 8 == k: X.W copies X's 8 columns
    exactly into every group of 8 output columns."""
    w = np.zeros((8, N), dtype=np.float64)
    w[np.arange(N) % 8, np.arange(N)] = 1.0
    return oracle.f64_to_bf16(w)


def _check_gelu(got, xin, what):
    """fp32 GeLU against the oracle: relative error <= GELU_REL_TOL where
    |GeLU(x)| >= GELU_TINY, absolute error <= GELU_TINY below that."""
    ref = oracle.gelu(xin.ravel()).reshape(xin.shape)
    big = np.abs(ref) >= GELU_TINY
    rel = np.where(big, np.abs(got - ref) / np.where(big, np.abs(ref), 1.0), 0.0)
    worst = int(np.argmax(rel))
    assert rel.flat[worst] <= GELU_REL_TOL, (
        f"{what}: GeLU({xin.flat[worst]!r}) = {got.flat[worst]!r}, oracle {ref.flat[worst]!r}, "
        f"relative error {rel.flat[worst]:.3e}")
    assert np.all(np.abs(got[~big] - ref[~big]) <= GELU_TINY), f"{what}: deep-tail GeLU"
    return ref


def test_gelu_epilogue_accuracy(tp, cuda_device):
    """The epilogue's exact GeLU at every bf16 value in [-12, 12] (and +-32,
    +-128): W = [I_8 | I_8 | ...] makes X.W copy X's entries exactly into an
    fp32 accumulator, so the output is GeLU(x) itself.  Checked relative to
    the value (the negative tail GeLU(x) = x Phi(x) shrinks like
    exp(-x^2/2), so an absolute bound would say nothing there):
      * fp32 output: relative error <= 1e-4 wherever |GeLU(x)| >= 1e-30;
      * bf16 output (TMA stores, and the per-thread stores of the
        shard-major copy): within one bf16 ulp of the round-to-nearest-even
        of the oracle's fp64 GeLU, at every such x;
      * the fp32-input CUDA-core path, the same relative bound."""
    import torch
    bits, vals = _all_bf16_in(-12.0, 12.0)
    extra_bits = np.array([0x4200, 0xC200, 0x4300, 0xC300], dtype=np.uint16)  # +-32, +-128
    xb = np.concatenate([bits, extra_bits])
    xs = np.concatenate([vals, oracle.bf16_to_f64(extra_bits)])
    pad = (-xb.size) % 8
    xb = np.concatenate([xb, np.zeros(pad, np.uint16)])
    xs = np.concatenate([xs, np.zeros(pad)])
    M = xb.size // 8
    N = 8 * 33  # 264 columns: two column tiles, the second ragged
    X, W = to_dev_bf16(xb.reshape(M, 8), cuda_device), to_dev_bf16(_identity_columns(N), cuda_device)
    xin = xs.reshape(M, 8)[:, np.arange(N) % 8]

    Yf = torch.empty(M, N, dtype=torch.float32, device=cuda_device)
    tp.tp_column_linear(X, W, Yf, None, n_shards=1, act="gelu")
    Yb = torch.empty(M, N, dtype=torch.bfloat16, device=cuda_device)
    tp.tp_column_linear(X, W, Yb, None, n_shards=1, act="gelu")
    n = 3
    Ys = torch.empty(n, M, N // n, dtype=torch.bfloat16, device=cuda_device)
    tp.tp_column_linear(X, W, None, Ys, n_shards=n, act="gelu")
    _status_ok(tp)

    ref = _check_gelu(dev_to_f64(Yf), xin, "fp32 output")
    big = np.abs(ref) >= GELU_TINY
    want = oracle.f64_to_bf16(ref)
    for what, got_bits in (("bf16 output", dev_bits(Yb).view(np.uint16)),
                           ("bf16 shard-major output",
                            dev_bits(Ys).view(np.uint16).transpose(1, 0, 2).reshape(M, N))):
        dist = np.where(big, _bf16_ulp_distance(got_bits, want), 0)
        worst = int(np.argmax(dist))
        assert dist.flat[worst] <= 1, (
            f"{what}: GeLU({xin.flat[worst]!r}) -> bf16 {got_bits.flat[worst]:#06x}, RNE of the "
            f"oracle {want.flat[worst]:#06x} ({dist.flat[worst]} ulp apart)")
    # the bf16 output is the RNE of the fp32 one (same epilogue arithmetic)
    np.testing.assert_array_equal(dev_bits(Yf.to(torch.bfloat16)), dev_bits(Yb))

    # fp32 inputs take the CUDA-core path and its scalar GeLU
    Xf = to_dev_f32(xs.reshape(M, 8), cuda_device)
    Wf = to_dev_f32(oracle.bf16_to_f64(_identity_columns(16)), cuda_device)
    Yc = torch.empty(M, 16, dtype=torch.float32, device=cuda_device)
    tp.tp_column_linear(Xf, Wf, Yc, None, n_shards=1, act="gelu")
    _status_ok(tp)
    _check_gelu(dev_to_f64(Yc), xs.reshape(M, 8)[:, np.arange(16) % 8], "fp32 CUDA-core path")


def _with_plan(plan, fn):
    import os
    old = os.environ.get("TP_GEMM_PLAN")
    os.environ["TP_GEMM_PLAN"] = plan
    try:
        return fn()
    finally:
        if old is None:
            del os.environ["TP_GEMM_PLAN"]
        else:
            os.environ["TP_GEMM_PLAN"] = old


@pytest.mark.parametrize("M,K,N,n", [(300, 328, 640, 2), (513, 1024, 392, 4), (1000, 512, 1152, 8)])
def test_tile_plans_agree(tp, cuda_device, M, K, N, n):
    """Every launch plan (256- and 128-wide pair tiles, cluster split over two
    pairs) on the same column (GeLU) and row products: the persistent
    plans accumulate every element in the same order, so their outputs are
    bit-identical; the split plans add slice partials and are held to the
    accuracy bar against the oracle."""
    import torch
    xb, wb = _bf16_inputs(M, K, N, seed=7 * M + N)
    X, W = to_dev_bf16(xb, cuda_device), to_dev_bf16(wb, cuda_device)
    Xd, Wd = oracle.bf16_to_f64(xb), oracle.bf16_to_f64(wb)
    col_ref, _ = oracle.column_linear(Xd, Wd, n, act="gelu")
    row_ref, _ = oracle.row_linear(Xd, Wd, n)
    outs = {}
    for plan in ["256", "128", "split2"]:
        Yc = torch.empty(M, N, dtype=torch.bfloat16, device=cuda_device)
        Yr = torch.empty(M, N, dtype=torch.float32, device=cuda_device)
        _with_plan(plan, lambda: tp.tp_column_linear(X, W, Yc, None, n_shards=n, act="gelu"))
        _with_plan(plan, lambda: tp.tp_row_linear(X, W, Yr, None, n_shards=n))
        _status_ok(tp)
        assert_bf16_parity(bf16_dev_to_f64(Yc), col_ref, f"column, plan {plan}")
        assert_bf16_parity(dev_to_f64(Yr), row_ref, f"row, plan {plan}", out_bf16=False)
        outs[plan] = (dev_bits(Yc), dev_bits(Yr))
    np.testing.assert_array_equal(outs["256"][0], outs["128"][0])
    np.testing.assert_array_equal(outs["256"][1], outs["128"][1])


@pytest.mark.parametrize("M,K,G,n,sw", [(256, 128, 3, 4, 64), (130, 64, 3, 2, 8), (64, 32, 2, 8, 16)])
def test_column_linear_head_groups(tp, cuda_device, M, K, G, n, sw):
    """Head-group split: shard i owns slice i of each of the G column blocks."""
    import torch
    N = G * n * sw
    xb, wb = _bf16_inputs(M, K, N, seed=7 * N)
    X, W = to_dev_bf16(xb, cuda_device), to_dev_bf16(wb, cuda_device)
    Y = torch.empty(M, N, dtype=torch.bfloat16, device=cuda_device)
    Ys = torch.empty(n, M, N // n, dtype=torch.bfloat16, device=cuda_device)
    tp.tp_column_linear_grouped(X, W, Y, Ys, n_shards=n, col_groups=G)
    Yc = torch.empty(M, N, dtype=torch.bfloat16, device=cuda_device)
    tp.tp_shard_concat_grouped(Ys, Yc, col_groups=G)
    _status_ok(tp)
    ref, ref_s = oracle.column_linear(oracle.bf16_to_f64(xb), oracle.bf16_to_f64(wb), n,
                                      col_groups=G)
    assert_bf16_parity(bf16_dev_to_f64(Ys), ref_s, "grouped shard outputs")
    np.testing.assert_array_equal(dev_bits(Yc), dev_bits(Y))
    np.testing.assert_array_equal(bf16_dev_to_f64(Ys), oracle.bf16_to_f64(
        dev_bits(Y).view(np.uint16)).reshape(M, G, n, sw).transpose(2, 0, 1, 3).reshape(n, M, G * sw))


# --------------------------------------------------------- bf16 row split ---

ROW_CASES = [
    (1280, 512, 2048, 4),   # persistent (80 tiles): shards walked in one accumulator
    (256, 1024, 512, 2),    # 4 tiles: cluster of 8, shard groups summed through DSMEM
    (300, 384, 264, 3),     # ragged, cluster split not aligned to shards
    (8, 64, 8, 8),          # shard depth 8 (< one k-block)
]


@pytest.mark.parametrize("M,K,N,n", ROW_CASES)
def test_row_linear_bf16_fused(tp, cuda_device, M, K, N, n):
    import torch
    xb, wb = _bf16_inputs(M, K, N, seed=3 * M + K)
    X, W = to_dev_bf16(xb, cuda_device), to_dev_bf16(wb, cuda_device)
    Y = torch.empty(M, N, dtype=torch.bfloat16, device=cuda_device)
    tp.tp_row_linear(X, W, Y, None, n_shards=n)
    _status_ok(tp)
    ref, _ = oracle.row_linear(oracle.bf16_to_f64(xb), oracle.bf16_to_f64(wb), n)
    assert_bf16_parity(bf16_dev_to_f64(Y), ref, "row fused")


@pytest.mark.parametrize("M,K,N,n", [(300, 384, 264, 3), (256, 1024, 512, 8), (130, 64, 16, 8)])
def test_row_linear_bf16_partials(tp, cuda_device, M, K, N, n):
    """Per-shard fp32 partials P_i = X_i.W_i, then the standalone reduce."""
    import torch
    xb, wb = _bf16_inputs(M, K, N, seed=5 * M + N)
    X, W = to_dev_bf16(xb, cuda_device), to_dev_bf16(wb, cuda_device)
    P = torch.empty(n, M, N, dtype=torch.float32, device=cuda_device)
    Y = torch.empty(M, N, dtype=torch.bfloat16, device=cuda_device)
    tp.tp_row_linear(X, W, Y, P, n_shards=n)
    _status_ok(tp)
    ref, ref_p = oracle.row_linear(oracle.bf16_to_f64(xb), oracle.bf16_to_f64(wb), n)
    for i in range(n):
        rel, mx, rms = assert_bf16_parity(dev_to_f64(P[i]), ref_p[i], f"partial {i}", out_bf16=False)
        assert rel < 1e-5  # fp32 output of an fp32 accumulation
    assert_bf16_parity(bf16_dev_to_f64(Y), ref, "row partials + reduce")


def test_sharded_linear_dispatch(tp, cuda_device):
    import torch
    M, K, N = 200, 256, 512
    xb, wb = _bf16_inputs(M, K, N, seed=99)
    X, W = to_dev_bf16(xb, cuda_device), to_dev_bf16(wb, cuda_device)
    Yc = torch.empty(M, N, dtype=torch.bfloat16, device=cuda_device)
    Yr = torch.empty(M, N, dtype=torch.bfloat16, device=cuda_device)
    tp.tp_sharded_linear(X, W, Yc, n_shards=4, split=tp.TP_SPLIT_COLS)
    tp.tp_sharded_linear(X, W, Yr, n_shards=4, split=tp.TP_SPLIT_ROWS)
    _status_ok(tp)
    ref = oracle.matmul(oracle.bf16_to_f64(xb), oracle.bf16_to_f64(wb))
    assert_bf16_parity(bf16_dev_to_f64(Yc), ref, "dispatch cols")
    assert_bf16_parity(bf16_dev_to_f64(Yr), ref, "dispatch rows")


# ------------------------------------------------------------- MLP block ----

@pytest.mark.parametrize("M,d,f,n", [(200, 256, 512, 2), (2048, 1024, 4096, 2), (384, 512, 1024, 8)])
def test_mlp_block_bf16(tp, cuda_device, M, d, f, n):
    """Megatron MLP block: column GEMM + GeLU, row GEMM with the shard sum
    in the accumulator.  (2048, 1024, 4096, N=2) is the MLP-block workload
    with X ~ N(0,1) and weights ~ N(0, 0.02)."""
    import torch
    xb = inputs.bf16_normal((M, d), inputs.stream_seed(1, 0), 1.0)
    w1b = inputs.bf16_normal((d, f), inputs.stream_seed(1, 1), 0.02)
    w2b = inputs.bf16_normal((f, d), inputs.stream_seed(1, 2), 0.02)
    X, W1, W2 = (to_dev_bf16(b, cuda_device) for b in (xb, w1b, w2b))
    Y = torch.empty(M, d, dtype=torch.bfloat16, device=cuda_device)
    ws = torch.empty(tp.tp_mlp_block_workspace_size(M, f, torch.bfloat16), dtype=torch.uint8,
                     device=cuda_device)
    tp.tp_mlp_block(X, W1, W2, Y, ws, n_shards=n)
    Y2 = torch.empty_like(Y)
    tp.tp_mlp_block(X, W1, W2, Y2, ws, n_shards=n)
    _status_ok(tp)
    ref = oracle.mlp_block(oracle.bf16_to_f64(xb), oracle.bf16_to_f64(w1b),
                           oracle.bf16_to_f64(w2b), n)
    assert_bf16_parity(bf16_dev_to_f64(Y), ref, "MLP block")
    np.testing.assert_array_equal(dev_bits(Y), dev_bits(Y2))  # run-to-run identical
    # the hidden activation in the workspace is GeLU(X.W1) rounded to bf16
    H = ws[: M * f * 2].view(torch.bfloat16).view(M, f)
    Href, _ = oracle.column_linear(oracle.bf16_to_f64(xb), oracle.bf16_to_f64(w1b), n, act="gelu")
    assert_bf16_parity(bf16_dev_to_f64(H), Href, "hidden H")


# -------------------------------------------------------- reduce / concat ---

@pytest.mark.parametrize("n", [1, 2, 3, 4, 8, 16])
@pytest.mark.parametrize("rows,cols", [(64, 96), (7, 5), (1, 8)])
def test_shard_reduce(tp, cuda_device, n, rows, cols):
    import torch
    P = inputs.f32_normal((n, rows, cols), 1000 + n)
    Pd = to_dev_f32(P, cuda_device)
    Yf = torch.empty(rows, cols, dtype=torch.float32, device=cuda_device)
    Yb = torch.empty(rows, cols, dtype=torch.bfloat16, device=cuda_device)
    tp.tp_shard_reduce(Pd, Yf)
    tp.tp_shard_reduce(Pd, Yb)
    _status_ok(tp)
    ref = oracle.shard_reduce(P)
    # recursive fp32 summation: |err| <= (n-1) * 2^-24 * sum_i |P_i|
    bound = (n - 1) * 2.0 ** -24 * np.abs(P.astype(np.float64)).sum(axis=0)
    assert np.all(np.abs(dev_to_f64(Yf) - ref) <= bound + 1e-30)
    # the bf16 output is the round-to-nearest-even of the fp32 sum
    np.testing.assert_array_equal(dev_bits(Yb), oracle.f64_to_bf16(dev_to_f64(Yf)).view(np.int16))


def test_shard_reduce_integer_exact_and_specials(tp, cuda_device):
    import torch
    rng = np.random.default_rng(0)
    P = rng.integers(-50, 50, size=(8, 16, 32)).astype(np.float32)
    P[3, 0, 0] = np.nan
    P[2, 1, 1] = np.inf
    P[5, 2, 2] = -np.inf
    Pd = to_dev_f32(P, cuda_device)
    Y = torch.empty(16, 32, dtype=torch.float32, device=cuda_device)
    tp.tp_shard_reduce(Pd, Y)
    _status_ok(tp)
    got = dev_to_f64(Y)
    ref = oracle.shard_reduce(P)
    assert np.isnan(got[0, 0]) and got[1, 1] == np.inf and got[2, 2] == -np.inf
    mask = np.isfinite(ref)
    np.testing.assert_array_equal(got[mask], ref[mask])


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("n,rows,sc", [(8, 100, 64), (2, 16, 32), (3, 1, 8)])
def test_shard_concat(tp, cuda_device, dtype, n, rows, sc):
    import torch
    Ys = inputs.f32_normal((n, rows, sc), 500 + n)
    if dtype == "bf16":
        bits = oracle.f64_to_bf16(Ys)
        Ysd = to_dev_bf16(bits, cuda_device)
        Y = torch.empty(rows, n * sc, dtype=torch.bfloat16, device=cuda_device)
        src = oracle.bf16_to_f64(bits)
    else:
        Ysd = to_dev_f32(Ys, cuda_device)
        Y = torch.empty(rows, n * sc, dtype=torch.float32, device=cuda_device)
        src = Ys.astype(np.float64)
    tp.tp_shard_concat(Ysd, Y)
    _status_ok(tp)
    np.testing.assert_array_equal(dev_to_f64(Y), oracle.shard_concat(src))


# ------------------------------------------------------- failure handling ---

def test_bounded_wait_reports_timeout(tp, cuda_device):
    """A wait on a barrier nobody arrives on gives up after its limit and the
    host reads TP_ERR_DEVICE_TIMEOUT; the context stays usable."""
    import torch
    assert tp.tp_get_device_status() == tp.TP_OK
    tp.tp_selftest_bounded_wait(20_000_000)  # 20 ms
    assert tp.tp_get_device_status() == tp.TP_ERR_DEVICE_TIMEOUT
    assert tp.tp_get_device_status() == tp.TP_OK  # cleared by the read
    P = torch.ones(2, 8, 8, device=cuda_device)
    Y = torch.empty(8, 8, device=cuda_device)
    tp.tp_shard_reduce(P, Y)
    assert tp.tp_get_device_status() == tp.TP_OK
    assert float(Y.sum()) == 128.0


def test_validation_errors_on_device(tp, cuda_device):
    import torch
    X = torch.zeros(16, 32, dtype=torch.bfloat16, device=cuda_device)
    W = torch.zeros(32, 64, dtype=torch.bfloat16, device=cuda_device)
    Y = torch.zeros(16, 64, dtype=torch.bfloat16, device=cuda_device)
    with pytest.raises(tp.TPError) as e:
        tp.tp_column_linear(X, W, Y, None, n_shards=3)
    assert e.value.status == 3
    big = torch.zeros(16 * 32 + 8, dtype=torch.bfloat16, device=cuda_device)
    Xmis = big[1:1 + 16 * 32].view(16, 32)  # 2-byte offset: not 16-byte aligned
    with pytest.raises(tp.TPError) as e:
        tp.tp_column_linear(Xmis, W, Y, None, n_shards=2)
    assert e.value.status == 4
    buf = torch.zeros(16 * 32 + 16 * 64, dtype=torch.bfloat16, device=cuda_device)
    Xa = buf[:16 * 32].view(16, 32)
    Ya = buf[256:256 + 16 * 64].view(16, 64)  # overlaps Xa
    with pytest.raises(tp.TPError) as e:
        tp.tp_column_linear(Xa, W, Ya, None, n_shards=2)
    assert e.value.status == 9  # output aliases an input
    ws = torch.empty(16, dtype=torch.uint8, device=cuda_device)
    W2 = torch.zeros(64, 32, dtype=torch.bfloat16, device=cuda_device)
    Y2 = torch.zeros(16, 32, dtype=torch.bfloat16, device=cuda_device)
    with pytest.raises(tp.TPError) as e:
        tp.tp_mlp_block(X, W, W2, Y2, ws, n_shards=2)
    assert e.value.status == 6
    assert tp.tp_get_device_status() == tp.TP_OK


def test_empty_inputs(tp, cuda_device):
    import torch
    X = torch.zeros(0, 32, dtype=torch.bfloat16, device=cuda_device)
    W = torch.randn(32, 64, device=cuda_device).to(torch.bfloat16)
    Y = torch.zeros(0, 64, dtype=torch.bfloat16, device=cuda_device)
    tp.tp_column_linear(X, W, Y, None, n_shards=2)
    tp.tp_row_linear(X, W, Y, None, n_shards=2)
    # K = 0: the empty contraction gives zeros (and GeLU(0) = 0)
    X0 = torch.zeros(8, 0, dtype=torch.bfloat16, device=cuda_device)
    W0 = torch.zeros(0, 16, dtype=torch.bfloat16, device=cuda_device)
    Y0 = torch.full((8, 16), 7.0, dtype=torch.bfloat16, device=cuda_device)
    tp.tp_column_linear(X0, W0, Y0, None, n_shards=2, act="gelu")
    P = torch.zeros(4, 0, 8, device=cuda_device)
    R = torch.zeros(0, 8, device=cuda_device)
    tp.tp_shard_reduce(P, R)
    _status_ok(tp)
    assert float(Y0.float().abs().sum()) == 0.0


# ------------------------------------------------------------------ bias ----

@pytest.mark.parametrize("M,K,N,n", [(300, 328, 640, 2), (1000, 512, 1152, 8), (64, 64, 264, 3)])
def test_linear_bias_bf16(tp, cuda_device, M, K, N, n):
    """Column split: each shard adds its slice of the bias before the GeLU;
    row split: the bias is added once after the sum (fused accumulator,
    cluster split and per-shard partials + reduce all agree with the oracle)."""
    import torch
    xb, wb = _bf16_inputs(M, K, N, seed=13 * N + K)
    bb = inputs.bf16_normal((N,), inputs.stream_seed(13 * N + K, 5), 0.5)
    X, W, b = to_dev_bf16(xb, cuda_device), to_dev_bf16(wb, cuda_device), to_dev_bf16(bb, cuda_device)
    Xd, Wd, bd = oracle.bf16_to_f64(xb), oracle.bf16_to_f64(wb), oracle.bf16_to_f64(bb)
    if N % n == 0:
        Yc = torch.empty(M, N, dtype=torch.bfloat16, device=cuda_device)
        Ys = torch.empty(n, M, N // n, dtype=torch.bfloat16, device=cuda_device)
        tp.tp_column_linear_bias(X, W, b, Yc, Ys, n_shards=n, act="gelu")
        Yc1 = torch.empty_like(Yc)
        tp.tp_column_linear_bias(X, W, b, Yc1, None, n_shards=n, act="gelu")
        _status_ok(tp)
        ref, ref_s = oracle.column_linear(Xd, Wd, n, act="gelu", bias=bd)
        assert_bf16_parity(bf16_dev_to_f64(Yc), ref, "column + bias")
        assert_bf16_parity(bf16_dev_to_f64(Ys), ref_s, "column + bias, shard-major")
        np.testing.assert_array_equal(dev_bits(Yc), dev_bits(Yc1))
    if K % n == 0:
        ref, _ = oracle.row_linear(Xd, Wd, n, bias=bd)
        for plan in ["256", "split2"]:
            Yr = torch.empty(M, N, dtype=torch.float32, device=cuda_device)
            _with_plan(plan, lambda: tp.tp_row_linear_bias(X, W, b, Yr, None, n_shards=n))
            _status_ok(tp)
            assert_bf16_parity(dev_to_f64(Yr), ref, f"row + bias, plan {plan}", out_bf16=False)
        if (K // n) % 8 == 0:
            P = torch.empty(n, M, N, dtype=torch.float32, device=cuda_device)
            Yp = torch.empty(M, N, dtype=torch.bfloat16, device=cuda_device)
            tp.tp_row_linear_bias(X, W, b, Yp, P, n_shards=n)
            _status_ok(tp)
            assert_bf16_parity(bf16_dev_to_f64(Yp), ref, "row + bias via partials")
            _, Pref = oracle.row_linear(Xd, Wd, n)
            assert_bf16_parity(dev_to_f64(P), Pref, "bias-free partials", out_bf16=False)


def test_bias_integer_exact_and_empty(tp, cuda_device):
    """Integer-valued fp32 and bf16 inputs with an integer bias: exact; an
    empty contraction (K = 0) gives act(bias) on every row."""
    import torch
    M, K, N, n = 40, 64, 48, 4
    xi = inputs.int_uniform((M, K), inputs.stream_seed(9, 0))
    wi = inputs.int_uniform((K, N), inputs.stream_seed(9, 1))
    bi = inputs.int_uniform((N,), inputs.stream_seed(9, 2))
    ref_c, _ = oracle.column_linear(xi, wi, n, bias=bi)
    ref_r, _ = oracle.row_linear(xi, wi, n, bias=bi)
    for dt in ("f32", "bf16"):
        conv = (lambda a: to_dev_f32(a, cuda_device)) if dt == "f32" else \
            (lambda a: to_dev_bf16(oracle.f64_to_bf16(a), cuda_device))
        X, W, b = conv(xi), conv(wi), conv(bi)
        Yc = torch.empty(M, N, dtype=torch.float32, device=cuda_device)
        Yr = torch.empty(M, N, dtype=torch.float32, device=cuda_device)
        tp.tp_column_linear_bias(X, W, b, Yc, None, n_shards=n)
        tp.tp_row_linear_bias(X, W, b, Yr, None, n_shards=n)
        _status_ok(tp)
        np.testing.assert_array_equal(dev_to_f64(Yc), ref_c)
        np.testing.assert_array_equal(dev_to_f64(Yr), ref_r)
    X0 = torch.zeros(M, 0, dtype=torch.bfloat16, device=cuda_device)
    W0 = torch.zeros(0, N, dtype=torch.bfloat16, device=cuda_device)
    b = to_dev_bf16(oracle.f64_to_bf16(bi), cuda_device)
    Y0 = torch.empty(M, N, dtype=torch.float32, device=cuda_device)
    tp.tp_column_linear_bias(X0, W0, b, Y0, None, n_shards=n, act="gelu")
    _status_ok(tp)
    # the epilogue GeLU's relative bound (GELU_REL_TOL; GeLU(0) = 0 exactly)
    np.testing.assert_allclose(dev_to_f64(Y0), np.tile(oracle.gelu(bi), (M, 1)), rtol=GELU_REL_TOL,
                               atol=0)


def test_binding_refuses_strided_views(tp, cuda_device):
    """A transposed or column-sliced view is not the dense row-major array
    the C ABI reads: the binding refuses it instead of misreading it."""
    import torch
    X = torch.zeros(64, 32, dtype=torch.bfloat16, device=cuda_device)
    Wt = torch.zeros(64, 32, dtype=torch.bfloat16, device=cuda_device)
    W = torch.zeros(32, 32, dtype=torch.bfloat16, device=cuda_device)
    Y = torch.zeros(64, 64, dtype=torch.bfloat16, device=cuda_device)
    with pytest.raises(ValueError, match="contiguous"):
        tp.tp_column_linear(X, Wt.t(), Y, None, n_shards=2)  # W as a transposed view
    with pytest.raises(ValueError, match="contiguous"):
        tp.tp_column_linear(X, W, Y[:, :32], None, n_shards=2)  # Y as a column slice


@pytest.mark.parametrize("M,K,N,n", [(300, 384, 400, 2), (513, 640, 272, 2)])
def test_split_plan_paths(tp, cuda_device, M, K, N, n):
    """The two-pair cluster split forced on every output path it has: an odd
    k-block count (the two K halves differ in length), ragged M and N, bf16
    output through TMA stores with bias and GeLU, the shard-major copy
    (per-thread stores: must equal the plain output's columns bit for bit),
    and fp32 output; integer-valued inputs give the exact product whatever
    the order the two halves are added in."""
    import torch
    xb, wb = _bf16_inputs(M, K, N, seed=31 * M + N)
    bb = inputs.bf16_normal((N,), inputs.stream_seed(31 * M + N, 7), 0.5)
    X, W, b = to_dev_bf16(xb, cuda_device), to_dev_bf16(wb, cuda_device), to_dev_bf16(bb, cuda_device)
    Xd, Wd, bd = oracle.bf16_to_f64(xb), oracle.bf16_to_f64(wb), oracle.bf16_to_f64(bb)
    Yc = torch.empty(M, N, dtype=torch.bfloat16, device=cuda_device)
    Ys = torch.empty(n, M, N // n, dtype=torch.bfloat16, device=cuda_device)
    Yc1 = torch.empty_like(Yc)
    Yr = torch.empty(M, N, dtype=torch.bfloat16, device=cuda_device)
    _with_plan("split2", lambda: tp.tp_column_linear_bias(X, W, b, Yc, Ys, n_shards=n, act="gelu"))
    _with_plan("split2", lambda: tp.tp_column_linear_bias(X, W, b, Yc1, None, n_shards=n,
                                                          act="gelu"))
    _with_plan("split2", lambda: tp.tp_row_linear_bias(X, W, b, Yr, None, n_shards=n))
    _status_ok(tp)
    ref_c, ref_s = oracle.column_linear(Xd, Wd, n, act="gelu", bias=bd)
    ref_r, _ = oracle.row_linear(Xd, Wd, n, bias=bd)
    assert_bf16_parity(bf16_dev_to_f64(Yc), ref_c, "split: column + bias + GeLU, direct stores")
    assert_bf16_parity(bf16_dev_to_f64(Yc1), ref_c, "split: column + bias + GeLU, TMA stores")
    assert_bf16_parity(bf16_dev_to_f64(Yr), ref_r, "split: row + bias, bf16 out")
    np.testing.assert_array_equal(dev_bits(Yc), dev_bits(Yc1))
    ys = dev_bits(Ys)
    yc = dev_bits(Yc)
    for i in range(n):
        np.testing.assert_array_equal(ys[i], yc[:, i * (N // n):(i + 1) * (N // n)])

    xi = inputs.int_uniform((M, K), inputs.stream_seed(31 * M + N, 8))
    wi = inputs.int_uniform((K, N), inputs.stream_seed(31 * M + N, 9))
    Xi = to_dev_bf16(oracle.f64_to_bf16(xi), cuda_device)
    Wi = to_dev_bf16(oracle.f64_to_bf16(wi), cuda_device)
    exact = xi.astype(np.int64) @ wi.astype(np.int64)
    for fn in (tp.tp_column_linear, tp.tp_row_linear):
        Yf = torch.empty(M, N, dtype=torch.float32, device=cuda_device)
        _with_plan("split2", lambda: fn(Xi, Wi, Yf, None, n_shards=n))
        _status_ok(tp)
        np.testing.assert_array_equal(dev_to_f64(Yf), exact)


@pytest.mark.parametrize("M,d,f,n", [(200, 256, 512, 2), (2048, 1024, 4096, 2)])
def test_mlp_block_bias(tp, cuda_device, M, d, f, n):
    import torch
    xb = inputs.bf16_normal((M, d), inputs.stream_seed(17, 0), 1.0)
    w1b = inputs.bf16_normal((d, f), inputs.stream_seed(17, 1), 0.02)
    w2b = inputs.bf16_normal((f, d), inputs.stream_seed(17, 2), 0.02)
    b1b = inputs.bf16_normal((f,), inputs.stream_seed(17, 3), 0.5)
    b2b = inputs.bf16_normal((d,), inputs.stream_seed(17, 4), 0.5)
    X, W1, W2, b1, b2 = (to_dev_bf16(a, cuda_device) for a in (xb, w1b, w2b, b1b, b2b))
    ws = torch.empty(tp.tp_mlp_block_workspace_size(M, f, torch.bfloat16), dtype=torch.uint8,
                     device=cuda_device)
    Y = torch.empty(M, d, dtype=torch.bfloat16, device=cuda_device)
    tp.tp_mlp_block_bias(X, W1, b1, W2, b2, Y, ws, n_shards=n)
    Yn = torch.empty_like(Y)
    tp.tp_mlp_block_bias(X, W1, None, W2, None, Yn, ws, n_shards=n)
    Yp = torch.empty_like(Y)
    tp.tp_mlp_block(X, W1, W2, Yp, ws, n_shards=n)
    _status_ok(tp)
    ref = oracle.mlp_block(*(oracle.bf16_to_f64(a) for a in (xb, w1b, w2b)), n,
                           b1=oracle.bf16_to_f64(b1b), b2=oracle.bf16_to_f64(b2b))
    assert_bf16_parity(bf16_dev_to_f64(Y), ref, "MLP block + biases")
    np.testing.assert_array_equal(dev_bits(Yn), dev_bits(Yp))


# ------------------------------------------------------- GQA head split ----

@pytest.mark.parametrize("M,K,hq,hkv,hd,n", [
    (300, 256, 32, 8, 128, 8),   # KV heads split: one per shard
    (257, 128, 32, 4, 128, 8),   # KV heads replicated on 2 shards each
    (64, 64, 16, 1, 64, 4),      # multi-query: one KV head on every shard
    (100, 64, 8, 8, 64, 4),      # hkv = hq: the head-group split
])
def test_qkv_gqa(tp, cuda_device, M, K, hq, hkv, hd, n):
    """QKV projection with grouped-query heads: the full output against the
    oracle, each shard's [Q_i | K_i | V_i] bit-equal to the matching columns
    of the full output (replicated KV heads in every shard that holds them)
    and within the accuracy bar of the oracle's shard-local products."""
    import torch
    N = (hq + 2 * hkv) * hd
    xb, wb = _bf16_inputs(M, K, N, seed=M + hq + hkv)
    X, W = to_dev_bf16(xb, cuda_device), to_dev_bf16(wb, cuda_device)
    kvs = oracle.qkv_kv_heads_per_shard(hq, hkv, n)
    Y = torch.empty(M, N, dtype=torch.bfloat16, device=cuda_device)
    Ys = torch.empty(n, M, (hq // n + 2 * kvs) * hd, dtype=torch.bfloat16, device=cuda_device)
    tp.tp_qkv_linear(X, W, Y, Ys, n_q_heads=hq, n_kv_heads=hkv, head_dim=hd, n_shards=n)
    _status_ok(tp)
    ref, ref_s = oracle.qkv_linear(oracle.bf16_to_f64(xb), oracle.bf16_to_f64(wb), hq, hkv, hd, n)
    assert_bf16_parity(bf16_dev_to_f64(Y), ref, "QKV full")
    assert_bf16_parity(bf16_dev_to_f64(Ys), ref_s, "QKV shard-local")
    # the shard-local outputs are copies of the full output's columns
    y = dev_bits(Y)
    ys = dev_bits(Ys)
    qs = hq // n
    for i in range(n):
        kv0 = i * kvs if hkv >= n else (i * hkv) // n
        cols = (list(range(i * qs * hd, (i + 1) * qs * hd))
                + list(range((hq + kv0) * hd, (hq + kv0 + kvs) * hd))
                + list(range((hq + hkv + kv0) * hd, (hq + hkv + kv0 + kvs) * hd)))
        np.testing.assert_array_equal(ys[i], y[:, cols])
    if hkv == hq:
        Yg = torch.empty(n, M, N // n, dtype=torch.bfloat16, device=cuda_device)
        tp.tp_column_linear_grouped(X, W, None, Yg, n_shards=n, col_groups=3)
        _status_ok(tp)
        np.testing.assert_array_equal(dev_bits(Yg), ys)


def test_qkv_gqa_validation(tp, cuda_device):
    import torch
    X = torch.zeros(8, 64, dtype=torch.bfloat16, device=cuda_device)
    W = torch.zeros(64, (8 + 2 * 3) * 64, dtype=torch.bfloat16, device=cuda_device)
    Y = torch.zeros(8, (8 + 2 * 3) * 64, dtype=torch.bfloat16, device=cuda_device)
    with pytest.raises(tp.TPError) as e:   # 3 KV heads do not divide 8 Q heads
        tp.tp_qkv_linear(X, W, Y, None, n_q_heads=8, n_kv_heads=3, head_dim=64, n_shards=2)
    assert e.value.status == 2
    W2 = torch.zeros(64, (8 + 2 * 2) * 64, dtype=torch.bfloat16, device=cuda_device)
    Y2 = torch.zeros(8, (8 + 2 * 2) * 64, dtype=torch.bfloat16, device=cuda_device)
    with pytest.raises(tp.TPError) as e:   # 3 shards do not divide 8 Q heads
        tp.tp_qkv_linear(X, W2, Y2, None, n_q_heads=8, n_kv_heads=2, head_dim=64, n_shards=3)
    assert e.value.status == 3
    assert tp.tp_get_device_status() == tp.TP_OK


# ------------------------------------------------- sequence parallelism ----

@pytest.mark.parametrize("n,Mb,d,f", [(4, 128, 256, 1024), (2, 300, 264, 512), (8, 64, 512, 2048)])
def test_sequence_parallel_combines(tp, cuda_device, n, Mb, d, f):
    """Sequence parallelism on one device: shard i's token block is rows
    [i*Mb, (i+1)*Mb) of a row-major [n*Mb, d] buffer, so the all-gather
    before the tensor-parallel block and the reduce-scatter after it move
    no data.  Checked here:
      * the MLP block run on the token blocks' buffer itself yields, block
        by block, the oracle's all-gather -> MLP -> reduce-scatter;
      * the row-parallel product, fused (shard sum in the accumulator) and
        through per-shard partials and the standalone reduce, yields the
        oracle's reduce-scatter of the shards' partials block by block;
      * the column GEMM reads the gathered X as it is: run on the whole
        buffer or on each token block alone, the outputs agree bit for bit
        (same launch plan, same accumulation order for every row)."""
    import torch
    M = n * Mb
    seed = 61 * n + Mb
    xs = inputs.bf16_normal((n, Mb, d), inputs.stream_seed(seed, 0), 1.0)
    w1b = inputs.bf16_normal((d, f), inputs.stream_seed(seed, 1), 0.02)
    w2b = inputs.bf16_normal((f, d), inputs.stream_seed(seed, 2), 0.02)
    Xs = to_dev_bf16(xs, cuda_device)          # [n, Mb, d]: the token blocks
    X = Xs.view(M, d)                          # the all-gathered tokens, same bytes
    W1, W2 = to_dev_bf16(w1b, cuda_device), to_dev_bf16(w2b, cuda_device)
    Xd, W1d, W2d = (oracle.bf16_to_f64(a) for a in (xs, w1b, w2b))

    Y = torch.empty(M, d, dtype=torch.bfloat16, device=cuda_device)
    ws = torch.empty(tp.tp_mlp_block_workspace_size(M, f, torch.bfloat16), dtype=torch.uint8,
                     device=cuda_device)
    tp.tp_mlp_block(X, W1, W2, Y, ws, n_shards=n)
    _status_ok(tp)
    ref = oracle.seq_parallel_mlp_block(Xd, W1d, W2d)
    got = bf16_dev_to_f64(Y.view(n, Mb, d))
    for i in range(n):
        assert_bf16_parity(got[i], ref[i], f"sequence-parallel MLP, token block {i}")

    # the row-parallel product of H (per-shard column blocks) with W2
    H = ws[: M * f * 2].view(torch.bfloat16).view(M, f)
    hb = dev_bits(H).view(np.uint16)
    _, Pref = oracle.row_linear(oracle.bf16_to_f64(hb), W2d, n)
    rs_ref = oracle.reduce_scatter_rows(Pref)
    Yf = torch.empty(M, d, dtype=torch.float32, device=cuda_device)
    tp.tp_row_linear(H, W2, Yf, None, n_shards=n)
    P = torch.empty(n, M, d, dtype=torch.float32, device=cuda_device)
    Yp = torch.empty(M, d, dtype=torch.float32, device=cuda_device)
    tp.tp_row_linear(H, W2, None, P, n_shards=n)
    tp.tp_shard_reduce(P, Yp)
    _status_ok(tp)
    fused, via_p = dev_to_f64(Yf).reshape(n, Mb, d), dev_to_f64(Yp).reshape(n, Mb, d)
    rs_dev = oracle.reduce_scatter_rows(dev_to_f64(P))
    abs_sum = np.abs(dev_to_f64(P)).sum(axis=0).reshape(n, Mb, d)
    for i in range(n):
        assert_bf16_parity(fused[i], rs_ref[i], f"fused row product, token block {i}",
                           out_bf16=False)
        assert_bf16_parity(via_p[i], rs_ref[i], f"partials + reduce, token block {i}",
                           out_bf16=False)
        # the reduce of the device's own partials: the fp32 sum's bound
        assert np.all(np.abs(via_p[i] - rs_dev[i]) <= (n - 1) * 2.0 ** -24 * abs_sum[i] + 1e-30)

    # the column GEMM on the gathered buffer == on each token block alone
    Hg = torch.empty(M, f, dtype=torch.bfloat16, device=cuda_device)
    _with_plan("256", lambda: tp.tp_column_linear(X, W1, Hg, None, n_shards=n, act="gelu"))
    for i in range(n):
        Hi = torch.empty(Mb, f, dtype=torch.bfloat16, device=cuda_device)
        _with_plan("256", lambda: tp.tp_column_linear(Xs[i], W1, Hi, None, n_shards=n,
                                                      act="gelu"))
        _status_ok(tp)
        np.testing.assert_array_equal(dev_bits(Hi), dev_bits(Hg[i * Mb:(i + 1) * Mb]))


def _pairs():
    """CTA pairs of the persistent GEMM on this GPU (one per two SMs)."""
    import torch
    return torch.cuda.get_device_properties(0).multi_processor_count // 2


def test_half_width_last_round(tp, cuda_device):
    """A product whose 256-wide pair tiles fill a few more than one round
    (tiles = pairs + r, 2r <= pairs): the last r tiles run as 2r half-width
    units.  Against the oracle, and bit for bit against the all-128-wide
    plan (same accumulation order per element), for the column GEMM with
    bias and GeLU (TMA stores, and the per-thread stores of the shard-major
    copy), the fused row GEMM and the per-shard fp32 partials."""
    import torch
    P = _pairs()
    mt = P // 8 + 1                       # 8 column tiles per row of tiles
    M, K, N, n = 256 * mt - 37, 264, 8 * 256, 4  # ragged last tile row
    assert 8 * mt > P and 2 * (8 * mt - P) <= P
    xb, wb = _bf16_inputs(M, K, N, seed=77)
    bb = inputs.bf16_normal((N,), inputs.stream_seed(77, 5), 0.5)
    X, W, b = to_dev_bf16(xb, cuda_device), to_dev_bf16(wb, cuda_device), to_dev_bf16(bb, cuda_device)
    Xd, Wd, bd = oracle.bf16_to_f64(xb), oracle.bf16_to_f64(wb), oracle.bf16_to_f64(bb)
    ref_c, ref_s = oracle.column_linear(Xd, Wd, n, act="gelu", bias=bd)
    outs = {}
    for plan in ("256", "128"):
        Yc = torch.empty(M, N, dtype=torch.bfloat16, device=cuda_device)
        Ys = torch.empty(n, M, N // n, dtype=torch.bfloat16, device=cuda_device)
        _with_plan(plan, lambda: tp.tp_column_linear_bias(X, W, b, Yc, None, n_shards=n,
                                                          act="gelu"))
        _with_plan(plan, lambda: tp.tp_column_linear_bias(X, W, b, None, Ys, n_shards=n,
                                                          act="gelu"))
        _status_ok(tp)
        assert_bf16_parity(bf16_dev_to_f64(Yc), ref_c, f"column + bias + GeLU, plan {plan}")
        assert_bf16_parity(bf16_dev_to_f64(Ys), ref_s, f"shard-major, plan {plan}")
        outs[plan] = (dev_bits(Yc), dev_bits(Ys))
    np.testing.assert_array_equal(outs["256"][0], outs["128"][0])
    np.testing.assert_array_equal(outs["256"][1], outs["128"][1])
    # row split: X2 [M, 2048] . W2 [2048, 2048], n = 8 shards, fused and as partials
    x2 = inputs.bf16_normal((M, N), inputs.stream_seed(78, 0), 1.0)
    w2 = inputs.bf16_normal((N, N), inputs.stream_seed(78, 1), 0.02)
    X2, W2 = to_dev_bf16(x2, cuda_device), to_dev_bf16(w2, cuda_device)
    ref_r, ref_p = oracle.row_linear(oracle.bf16_to_f64(x2), oracle.bf16_to_f64(w2), 8)
    routs = {}
    for plan in ("256", "128"):
        Yr = torch.empty(M, N, dtype=torch.float32, device=cuda_device)
        _with_plan(plan, lambda: tp.tp_row_linear(X2, W2, Yr, None, n_shards=8))
        _status_ok(tp)
        assert_bf16_parity(dev_to_f64(Yr), ref_r, f"row, plan {plan}", out_bf16=False)
        routs[plan] = dev_bits(Yr)
    np.testing.assert_array_equal(routs["256"], routs["128"])
    # per-shard partials: one output per shard (k-group), so the units are
    # row tiles x column tiles x shards; one row tile, 8 column tiles and
    # P // 8 + 1 shards leave the same short last round
    Mp = 256
    kg = P // 8 + 1
    x3 = inputs.bf16_normal((Mp, 8 * kg), inputs.stream_seed(79, 0), 1.0)
    w3 = inputs.bf16_normal((8 * kg, N), inputs.stream_seed(79, 1), 0.05)
    X3, W3 = to_dev_bf16(x3, cuda_device), to_dev_bf16(w3, cuda_device)
    Pd = torch.empty(kg, Mp, N, dtype=torch.float32, device=cuda_device)
    tp.tp_row_linear(X3, W3, None, Pd, n_shards=kg)
    _status_ok(tp)
    _, ref_p3 = oracle.row_linear(oracle.bf16_to_f64(x3), oracle.bf16_to_f64(w3), kg)
    assert_bf16_parity(dev_to_f64(Pd), ref_p3, "per-shard partials, short last round",
                       out_bf16=False)


# ------------------------------------------------------ concurrent streams --

def test_concurrent_streams(tp, cuda_device):
    """Independent calls on separate streams (MLP blocks of three shapes,
    one of them on the cluster split path, and a standalone reduce) overlap
    on the GPU and give the same bits as the same calls one after another:
    the kernels share no state but the error word, and the host's
    tensor-map cache is locked."""
    import torch
    cases = [(200, 256, 512, 2), (2048, 1024, 4096, 2), (384, 512, 1024, 8)]
    jobs = []
    for i, (M, d, f, n) in enumerate(cases):
        xb = inputs.bf16_normal((M, d), inputs.stream_seed(40 + i, 0), 1.0)
        w1b = inputs.bf16_normal((d, f), inputs.stream_seed(40 + i, 1), 0.02)
        w2b = inputs.bf16_normal((f, d), inputs.stream_seed(40 + i, 2), 0.02)
        X, W1, W2 = (to_dev_bf16(b, cuda_device) for b in (xb, w1b, w2b))
        ws = torch.empty(tp.tp_mlp_block_workspace_size(M, f, torch.bfloat16),
                         dtype=torch.uint8, device=cuda_device)
        Yser = torch.empty(M, d, dtype=torch.bfloat16, device=cuda_device)
        tp.tp_mlp_block(X, W1, W2, Yser, ws, n_shards=n)
        jobs.append((X, W1, W2, n, Yser, (M, d, f)))
    P = to_dev_f32(inputs.f32_normal((4, 512, 1024), 47), cuda_device)
    Rser = torch.empty(512, 1024, dtype=torch.float32, device=cuda_device)
    tp.tp_shard_reduce(P, Rser)
    torch.cuda.synchronize()

    streams = [torch.cuda.Stream(cuda_device) for _ in range(len(jobs) + 1)]
    outs, wss = [], []
    for X, W1, W2, n, Yser, (M, d, f) in jobs:
        outs.append(torch.full((M, d), float("nan"), dtype=torch.bfloat16, device=cuda_device))
        wss.append(torch.empty(tp.tp_mlp_block_workspace_size(M, f, torch.bfloat16),
                               dtype=torch.uint8, device=cuda_device))
    R = torch.full((512, 1024), float("nan"), dtype=torch.float32, device=cuda_device)
    torch.cuda.synchronize()
    for rep in range(3):
        for s, (X, W1, W2, n, _, _), Y, ws in zip(streams, jobs, outs, wss):
            tp.tp_mlp_block(X, W1, W2, Y, ws, n_shards=n, stream=s)
        tp.tp_shard_reduce(P, R, stream=streams[-1])
    torch.cuda.synchronize()
    _status_ok(tp)
    for (_, _, _, _, Yser, shape), Y in zip(jobs, outs):
        np.testing.assert_array_equal(dev_bits(Y), dev_bits(Yser), err_msg=f"MLP {shape}")
    np.testing.assert_array_equal(R.cpu().numpy().view(np.int32), Rser.cpu().numpy().view(np.int32))


# ------------------------------------------------------- random shapes ------

def _random_shapes(count, seed):
    """Seeded shapes inside the boundary's rules (rows of 16-byte multiples,
    shard widths and depths multiples of 8), from one row up to a few tiles
    with ragged tails; n from {1, 2, 3, 4, 8}."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(count):
        n = int(rng.choice([1, 2, 3, 4, 8]))
        M = int(rng.integers(1, 700))
        K = 8 * n * int(rng.integers(1, max(2, 1100 // (8 * n))))
        N = 8 * n * int(rng.integers(1, max(2, 1100 // (8 * n))))
        out.append((M, K, N, n))
    return out


@pytest.mark.parametrize("M,K,N,n", _random_shapes(8, 20261203))
def test_random_shapes(tp, cuda_device, M, K, N, n):
    """Column GEMM (with GeLU), row GEMM with the fused shard sum and the
    MLP block (d = K, f = N) on seeded random shapes, each against the
    oracle; the column output also bit for bit against the unsharded
    launch."""
    import torch
    seed = 7 * M + 3 * K + N + n
    xb, wb = _bf16_inputs(M, K, N, seed=seed)
    X, W = to_dev_bf16(xb, cuda_device), to_dev_bf16(wb, cuda_device)
    Xd, Wd = oracle.bf16_to_f64(xb), oracle.bf16_to_f64(wb)
    Yc = torch.empty(M, N, dtype=torch.bfloat16, device=cuda_device)
    Yc1 = torch.empty_like(Yc)
    tp.tp_column_linear(X, W, Yc, None, n_shards=n, act="gelu")
    tp.tp_column_linear(X, W, Yc1, None, n_shards=1, act="gelu")
    Yr = torch.empty(M, N, dtype=torch.bfloat16, device=cuda_device)
    tp.tp_row_linear(X, W, Yr, None, n_shards=n)
    w2b = inputs.bf16_normal((N, K), inputs.stream_seed(seed, 2), 0.02)
    W2 = to_dev_bf16(w2b, cuda_device)
    Ym = torch.empty(M, K, dtype=torch.bfloat16, device=cuda_device)
    ws = torch.empty(tp.tp_mlp_block_workspace_size(M, N, torch.bfloat16), dtype=torch.uint8,
                     device=cuda_device)
    tp.tp_mlp_block(X, W, W2, Ym, ws, n_shards=n)
    _status_ok(tp)
    ref_c, _ = oracle.column_linear(Xd, Wd, n, act="gelu")
    assert_bf16_parity(bf16_dev_to_f64(Yc), ref_c, f"column {M}x{K}x{N} n={n}")
    np.testing.assert_array_equal(dev_bits(Yc), dev_bits(Yc1))
    ref_r, _ = oracle.row_linear(Xd, Wd, n)
    assert_bf16_parity(bf16_dev_to_f64(Yr), ref_r, f"row {M}x{K}x{N} n={n}")
    ref_m = oracle.mlp_block(Xd, Wd, oracle.bf16_to_f64(w2b), n)
    assert_bf16_parity(bf16_dev_to_f64(Ym), ref_m, f"MLP {M}x{K}x{N} n={n}")
