"""Parity at the workloads' full sizes, in the launch configuration the
bench uses.  The GPU computes the whole problem; the fp64 oracle computes a
seeded sample of rows, at least one in every 256-row pair tile plus the
first and the last row (every output row depends only on its own input
row, so a sampled row is checked exactly as it would be in the full
problem, and every tile, hence every persistent round, is reached).
Properties that hold at any size (shard outputs == concat columns bit for
bit, sharded == unsharded, run-to-run identity) are checked on everything.
"""
import numpy as np
import pytest

import oracle
from helpers import assert_bf16_parity, bf16_dev_to_f64, dev_bits, dev_to_f64, to_dev_bf16
from tensor_sharded_linear_02_b300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tp():
    from tensor_sharded_linear_02_b300 import binding
    binding.lib()
    return binding


PAIR_TILE_ROWS = 256  # output rows of one tile of a CTA pair


def _rows(M, per_tile, seed):
    """`per_tile` rows of every 256-row pair tile, at seeded random offsets
    (so that the samples fall in different tensor-memory lane quadrants and
    epilogue warps), plus the first and the last row: a fault specific to
    one tile, or to a later persistent round, shows in some sampled row."""
    rng = np.random.default_rng(seed)
    picks = [0, M - 1]
    for t0 in range(0, M, PAIR_TILE_ROWS):
        t1 = min(t0 + PAIR_TILE_ROWS, M)
        picks += [int(r) for r in rng.choice(np.arange(t0, t1), size=min(per_tile, t1 - t0),
                                             replace=False)]
    rows = np.unique(np.array(picks, dtype=np.int64))
    assert len(np.unique(rows // PAIR_TILE_ROWS)) == (M + PAIR_TILE_ROWS - 1) // PAIR_TILE_ROWS
    return rows


def _mlp_case(tp, dev, M, d, f, n_list, std, per_tile, seed):
    import torch
    xb = inputs.bf16_normal((M, d), inputs.stream_seed(seed, 0), 1.0)
    w1b = inputs.bf16_normal((d, f), inputs.stream_seed(seed, 1), std)
    w2b = inputs.bf16_normal((f, d), inputs.stream_seed(seed, 2), std)
    X, W1, W2 = (to_dev_bf16(b, dev) for b in (xb, w1b, w2b))
    ws = torch.empty(tp.tp_mlp_block_workspace_size(M, f, torch.bfloat16), dtype=torch.uint8,
                     device=dev)
    rows = _rows(M, per_tile, seed)
    Xs = oracle.bf16_to_f64(xb[rows])
    W1d, W2d = oracle.bf16_to_f64(w1b), oracle.bf16_to_f64(w2b)
    for n in n_list:
        Y = torch.empty(M, d, dtype=torch.bfloat16, device=dev)
        tp.tp_mlp_block(X, W1, W2, Y, ws, n_shards=n)
        assert tp.tp_get_device_status() == tp.TP_OK
        got = bf16_dev_to_f64(Y[torch.from_numpy(rows).to(dev)])
        ref = oracle.mlp_block(Xs, W1d, W2d, n)
        assert_bf16_parity(got, ref, f"MLP {M}x{d}x{f} N={n} sampled rows")
        H = ws[: M * f * 2].view(torch.bfloat16).view(M, f)
        Hs = bf16_dev_to_f64(H[torch.from_numpy(rows).to(dev)])
        Href, _ = oracle.column_linear(Xs, W1d, n, act="gelu")
        assert_bf16_parity(Hs, Href, f"hidden H N={n} sampled rows")
        Y2 = torch.empty_like(Y)
        tp.tp_mlp_block(X, W1, W2, Y2, ws, n_shards=n)
        assert torch.equal(Y.view(torch.int16), Y2.view(torch.int16))


def test_gpt_mlp_block(tp, cuda_device):
    """GPT-style MLP block: X [4096, 4096], W1 [4096, 16384], W2 [16384, 4096]
    ~ N(0, 0.02), N = 8."""
    _mlp_case(tp, cuda_device, 4096, 4096, 16384, [8], 0.02, per_tile=2, seed=3)


def test_wide_mlp_shard_sweep(tp, cuda_device):
    """Wide MLP block X [4096, 8192], W1 [8192, 28672], W2 [28672, 8192]
    ~ N(0, 0.01), every shard count N in {1, 2, 4, 8, 16}."""
    _mlp_case(tp, cuda_device, 4096, 8192, 28672, [1, 2, 4, 8, 16], 0.01, per_tile=2, seed=5)


def test_attention_projections(tp, cuda_device):
    """QKV projection X [8192, 4096] . Wqkv [4096, 12288] split into 8 head
    groups of 4 heads (Q|K|V column blocks), and the output projection
    C [8192, 4096] . Wo [4096, 4096] split by rows into 8 with the partials
    summed on the device."""
    import torch
    dev = cuda_device
    M, d, n, G = 8192, 4096, 8, 3
    xb = inputs.bf16_normal((M, d), inputs.stream_seed(4, 0), 1.0)
    wqkv = inputs.bf16_normal((d, G * d), inputs.stream_seed(4, 1), 0.02)
    cb = inputs.bf16_normal((M, d), inputs.stream_seed(4, 2), 1.0)
    wo = inputs.bf16_normal((d, d), inputs.stream_seed(4, 3), 0.02)
    X, Wqkv, C, Wo = (to_dev_bf16(b, dev) for b in (xb, wqkv, cb, wo))
    QKV = torch.empty(M, G * d, dtype=torch.bfloat16, device=dev)
    loc = torch.empty(n, M, G * d // n, dtype=torch.bfloat16, device=dev)
    tp.tp_column_linear_grouped(X, Wqkv, QKV, loc, n_shards=n, col_groups=G)
    O = torch.empty(M, d, dtype=torch.bfloat16, device=dev)
    tp.tp_row_linear(C, Wo, O, None, n_shards=n)
    cat = torch.empty_like(QKV)
    tp.tp_shard_concat_grouped(loc, cat, col_groups=G)
    assert tp.tp_get_device_status() == tp.TP_OK
    # all sizes: the standalone concat of the shard outputs rebuilds the fused one
    assert torch.equal(cat.view(torch.int16), QKV.view(torch.int16))
    rows = _rows(M, 1, 4)
    ridx = torch.from_numpy(rows).to(dev)
    ref_qkv, ref_loc = oracle.column_linear(oracle.bf16_to_f64(xb[rows]),
                                            oracle.bf16_to_f64(wqkv), n, col_groups=G)
    assert_bf16_parity(bf16_dev_to_f64(QKV[ridx]), ref_qkv, "QKV sampled rows")
    assert_bf16_parity(bf16_dev_to_f64(loc[:, ridx]), ref_loc, "QKV head-group shards")
    ref_o, _ = oracle.row_linear(oracle.bf16_to_f64(cb[rows]), oracle.bf16_to_f64(wo), n)
    assert_bf16_parity(bf16_dev_to_f64(O[ridx]), ref_o, "Wo row split sampled rows")


def test_standalone_reduce_sweep(tp, cuda_device):
    """N fp32 partials [4096, 8192] -> bf16 for N in {1, 2, 4, 8, 16}, every
    element checked against the oracle's double sum."""
    import torch
    dev = cuda_device
    rows, cols = 4096, 8192
    P16 = inputs.f32_normal((16, rows, cols), 4242)
    Pd = torch.from_numpy(P16).to(dev)
    for n in (1, 2, 4, 8, 16):
        Yb = torch.empty(rows, cols, dtype=torch.bfloat16, device=dev)
        Yf = torch.empty(rows, cols, dtype=torch.float32, device=dev)
        tp.tp_shard_reduce(Pd[:n], Yb)
        tp.tp_shard_reduce(Pd[:n], Yf)
        assert tp.tp_get_device_status() == tp.TP_OK
        ref = oracle.shard_reduce(P16[:n])
        got = dev_to_f64(Yf)
        abs_sum = np.zeros((rows, cols))
        for i in range(n):
            abs_sum += np.abs(P16[i])
        bound = (n - 1) * 2.0 ** -24 * abs_sum
        assert np.all(np.abs(got - ref) <= bound + 1e-30), f"reduce N={n}"
        np.testing.assert_array_equal(dev_bits(Yb), oracle.f64_to_bf16(got).view(np.int16))


def test_gpt_mlp_backward_sampled(tp, cuda_device):
    """Backward of the GPT-style MLP block at full size (X [4096, 4096],
    W1 [4096, 16384], W2 [16384, 4096], N = 8; dY ~ N(0, 1)), as the bench
    runs it: the GPU computes dX, dW1, dW2 whole; the fp64 oracle computes
    dX on rows in every 256-row tile, dW1 on columns and dW2 on rows spread
    over every 256-wide tile of theirs (first and last included).  Two calls
    are bit-identical."""
    import torch
    dev = cuda_device
    M, d, f, n = 4096, 4096, 16384, 8
    xb = inputs.bf16_normal((M, d), inputs.stream_seed(6, 0), 1.0)
    w1b = inputs.bf16_normal((d, f), inputs.stream_seed(6, 1), 0.02)
    w2b = inputs.bf16_normal((f, d), inputs.stream_seed(6, 2), 0.02)
    gb = inputs.bf16_normal((M, d), inputs.stream_seed(6, 3), 1.0)
    X, W1, W2, dY = (to_dev_bf16(b, dev) for b in (xb, w1b, w2b, gb))
    ws = torch.empty(tp.tp_mlp_block_backward_workspace_size(M, f, torch.bfloat16),
                     dtype=torch.uint8, device=dev)
    outs = []
    for _ in range(2):
        dX = torch.empty(M, d, dtype=torch.bfloat16, device=dev)
        dW1 = torch.empty(d, f, dtype=torch.bfloat16, device=dev)
        dW2 = torch.empty(f, d, dtype=torch.bfloat16, device=dev)
        tp.tp_mlp_block_backward(X, W1, W2, dY, ws, dX, dW1, dW2, n_shards=n)
        outs.append((dX, dW1, dW2))
    assert tp.tp_get_device_status() == tp.TP_OK
    for a, b in zip(*outs):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    dX, dW1, dW2 = outs[0]
    rx = _rows(M, 1, 61)            # dX rows: one in every 256-row tile
    c1 = _rows(f, 1, 62)[::2]       # dW1 columns: every other 256-wide tile
    r2 = _rows(f, 1, 63)[1::2]      # dW2 rows: the other tiles
    sX, sW1, sW2 = oracle.mlp_block_backward_sampled(
        *(oracle.bf16_to_f64(b) for b in (xb, w1b, w2b, gb)), n, rx, c1, r2)
    assert_bf16_parity(bf16_dev_to_f64(dX[torch.from_numpy(rx).to(dev)]), sX, "dX sampled rows")
    assert_bf16_parity(bf16_dev_to_f64(dW1[:, torch.from_numpy(c1).to(dev)]), sW1,
                       "dW1 sampled columns")
    assert_bf16_parity(bf16_dev_to_f64(dW2[torch.from_numpy(r2).to(dev)]), sW2,
                       "dW2 sampled rows")
