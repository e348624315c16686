"""GPU parity of the backward pass against the fp64 oracle: the sharded
linears' gradients (bit-exact on integer-valued bf16 inputs, within the
accuracy bar on normal inputs) and the MLP block's (recomputed
pre-activation, GeLU' in the epilogue, shard sum of dX in the accumulator).
The products read X^T and W^T in place through the tensor cores' transposed
operand layouts; ragged sizes exercise the zero-filled tails of those
layouts."""
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


def _int_bf16(shape, seed):
    v = inputs.int_uniform(shape, seed)
    return oracle.f64_to_bf16(v)


@pytest.mark.parametrize("kind", ["column", "row"])
@pytest.mark.parametrize("M,K,N,n", [(300, 264, 640, 2), (513, 128, 392, 4), (64, 520, 256, 8),
                                     (1, 8, 8, 1)])
def test_linear_backward_integer_exact(tp, cuda_device, kind, M, K, N, n):
    """Integer-valued bf16 inputs in [-4, 4]: every product and partial sum is
    an integer below 2^24, so the fp32 gradients equal the oracle's exactly."""
    import torch
    if (kind == "column" and N % n) or (kind == "row" and K % n):
        pytest.skip("shard count does not divide the split axis")
    xb = _int_bf16((M, K), inputs.stream_seed(M + K, 0))
    wb = _int_bf16((K, N), inputs.stream_seed(M + K, 1))
    gb = _int_bf16((M, N), inputs.stream_seed(M + K, 2))
    X, W, dY = (to_dev_bf16(b, cuda_device) for b in (xb, wb, gb))
    dX = torch.empty(M, K, dtype=torch.float32, device=cuda_device)
    dW = torch.empty(K, N, dtype=torch.float32, device=cuda_device)
    fn = tp.tp_column_linear_backward if kind == "column" else tp.tp_row_linear_backward
    fn(X, W, dY, dX, dW, n_shards=n)
    assert tp.tp_get_device_status() == tp.TP_OK
    back = oracle.column_linear_backward if kind == "column" else oracle.row_linear_backward
    rX, rW = back(*(oracle.bf16_to_f64(b) for b in (xb, wb, gb)), n)
    np.testing.assert_array_equal(dev_to_f64(dX), rX)
    np.testing.assert_array_equal(dev_to_f64(dW), rW)


@pytest.mark.parametrize("kind", ["column", "row"])
def test_linear_backward_bf16(tp, cuda_device, kind):
    """Normal inputs, bf16 and fp32 gradients within the accuracy bar; a
    NULL output skips that gradient."""
    import torch
    M, K, N, n = 700, 512, 1032, 4 if kind == "row" else 2
    N = 1032 if kind == "row" else 1040
    xb = inputs.bf16_normal((M, K), inputs.stream_seed(31, 0), 1.0)
    wb = inputs.bf16_normal((K, N), inputs.stream_seed(31, 1), 0.02)
    gb = inputs.bf16_normal((M, N), inputs.stream_seed(31, 2), 1.0)
    X, W, dY = (to_dev_bf16(b, cuda_device) for b in (xb, wb, gb))
    fn = tp.tp_column_linear_backward if kind == "column" else tp.tp_row_linear_backward
    back = oracle.column_linear_backward if kind == "column" else oracle.row_linear_backward
    rX, rW = back(*(oracle.bf16_to_f64(b) for b in (xb, wb, gb)), n)
    dX = torch.empty(M, K, dtype=torch.bfloat16, device=cuda_device)
    dW = torch.empty(K, N, dtype=torch.bfloat16, device=cuda_device)
    fn(X, W, dY, dX, dW, n_shards=n)
    dXf = torch.empty(M, K, dtype=torch.float32, device=cuda_device)
    fn(X, W, dY, dXf, None, n_shards=n)
    assert tp.tp_get_device_status() == tp.TP_OK
    assert_bf16_parity(bf16_dev_to_f64(dX), rX, f"{kind} dX")
    assert_bf16_parity(bf16_dev_to_f64(dW), rW, f"{kind} dW")
    assert_bf16_parity(dev_to_f64(dXf), rX, f"{kind} dX fp32", out_bf16=False)
    np.testing.assert_array_equal(dev_bits(dXf.to(torch.bfloat16)), dev_bits(dX))
    # dX with 256- and 128-wide tiles: the same accumulation order per element
    import os
    outs = []
    for plan in ("256", "128"):
        os.environ["TP_GEMM_PLAN"] = plan
        try:
            dXp = torch.empty(M, K, dtype=torch.float32, device=cuda_device)
            fn(X, W, dY, dXp, None, n_shards=n)
        finally:
            del os.environ["TP_GEMM_PLAN"]
        outs.append(dev_bits(dXp))
    assert tp.tp_get_device_status() == tp.TP_OK
    np.testing.assert_array_equal(outs[0], outs[1])
    np.testing.assert_array_equal(outs[0], dev_bits(dXf))


@pytest.mark.parametrize("M,d,f,n", [(200, 256, 512, 2), (300, 264, 1000, 4),
                                     (2048, 1024, 4096, 2)])
def test_mlp_block_backward(tp, cuda_device, M, d, f, n):
    """dX, dW1, dW2 of the MLP block against the oracle (fp64, per shard,
    pre-activation recomputed exactly); the recomputed H equals the forward
    pass's H bit for bit; two calls give identical results."""
    import torch
    xb = inputs.bf16_normal((M, d), inputs.stream_seed(41, 0), 1.0)
    w1b = inputs.bf16_normal((d, f), inputs.stream_seed(41, 1), 0.02)
    w2b = inputs.bf16_normal((f, d), inputs.stream_seed(41, 2), 0.02)
    gb = inputs.bf16_normal((M, d), inputs.stream_seed(41, 3), 1.0)
    X, W1, W2, dY = (to_dev_bf16(b, cuda_device) for b in (xb, w1b, w2b, gb))
    ws = torch.empty(tp.tp_mlp_block_backward_workspace_size(M, f, torch.bfloat16),
                     dtype=torch.uint8, device=cuda_device)
    outs = []
    for _ in range(2):
        dX = torch.empty(M, d, dtype=torch.bfloat16, device=cuda_device)
        dW1 = torch.empty(d, f, dtype=torch.bfloat16, device=cuda_device)
        dW2 = torch.empty(f, d, dtype=torch.bfloat16, device=cuda_device)
        tp.tp_mlp_block_backward(X, W1, W2, dY, ws, dX, dW1, dW2, n_shards=n)
        outs.append((dX, dW1, dW2))
    assert tp.tp_get_device_status() == tp.TP_OK
    rX, rW1, rW2 = oracle.mlp_block_backward(*(oracle.bf16_to_f64(b) for b in (xb, w1b, w2b, gb)),
                                             n)
    assert_bf16_parity(bf16_dev_to_f64(outs[0][0]), rX, "MLP dX")
    assert_bf16_parity(bf16_dev_to_f64(outs[0][1]), rW1, "MLP dW1")
    assert_bf16_parity(bf16_dev_to_f64(outs[0][2]), rW2, "MLP dW2")
    for a, b in zip(*outs):
        np.testing.assert_array_equal(dev_bits(a), dev_bits(b))
    # the recomputed H (second part of the workspace) is the forward's H
    part = (M * f * 2 + 255) // 256 * 256
    H_bwd = ws[part: part + M * f * 2].view(torch.bfloat16).view(M, f)
    fws = torch.empty(tp.tp_mlp_block_workspace_size(M, f, torch.bfloat16), dtype=torch.uint8,
                      device=cuda_device)
    Y = torch.empty(M, d, dtype=torch.bfloat16, device=cuda_device)
    tp.tp_mlp_block(X, W1, W2, Y, fws, n_shards=n)
    assert tp.tp_get_device_status() == tp.TP_OK
    H_fwd = fws[: M * f * 2].view(torch.bfloat16).view(M, f)
    np.testing.assert_array_equal(dev_bits(H_bwd), dev_bits(H_fwd))


def test_mlp_block_backward_fp32_grads_and_skips(tp, cuda_device):
    """fp32 gradients round to the bf16 ones; NULL outputs are skipped."""
    import torch
    M, d, f, n = 256, 128, 384, 3
    xb = inputs.bf16_normal((M, d), inputs.stream_seed(43, 0), 1.0)
    w1b = inputs.bf16_normal((d, f), inputs.stream_seed(43, 1), 0.05)
    w2b = inputs.bf16_normal((f, d), inputs.stream_seed(43, 2), 0.05)
    gb = inputs.bf16_normal((M, d), inputs.stream_seed(43, 3), 1.0)
    X, W1, W2, dY = (to_dev_bf16(b, cuda_device) for b in (xb, w1b, w2b, gb))
    ws = torch.empty(tp.tp_mlp_block_backward_workspace_size(M, f, torch.bfloat16),
                     dtype=torch.uint8, device=cuda_device)
    dX = torch.empty(M, d, dtype=torch.float32, device=cuda_device)
    dW1 = torch.empty(d, f, dtype=torch.float32, device=cuda_device)
    dW2 = torch.empty(f, d, dtype=torch.float32, device=cuda_device)
    tp.tp_mlp_block_backward(X, W1, W2, dY, ws, dX, dW1, dW2, n_shards=n)
    dW2_only = torch.full((f, d), float("nan"), dtype=torch.float32, device=cuda_device)
    tp.tp_mlp_block_backward(X, W1, W2, dY, ws, None, None, dW2_only, n_shards=n)
    assert tp.tp_get_device_status() == tp.TP_OK
    rX, rW1, rW2 = oracle.mlp_block_backward(*(oracle.bf16_to_f64(b) for b in (xb, w1b, w2b, gb)),
                                             n)
    assert_bf16_parity(dev_to_f64(dX), rX, "dX fp32", out_bf16=False)
    assert_bf16_parity(dev_to_f64(dW1), rW1, "dW1 fp32", out_bf16=False)
    assert_bf16_parity(dev_to_f64(dW2), rW2, "dW2 fp32", out_bf16=False)
    np.testing.assert_array_equal(dev_bits(dW2_only), dev_bits(dW2))


def test_backward_validation(tp, cuda_device):
    import torch
    X = torch.zeros(16, 24, dtype=torch.bfloat16, device=cuda_device)
    W = torch.zeros(24, 40, dtype=torch.bfloat16, device=cuda_device)
    dY = torch.zeros(16, 40, dtype=torch.bfloat16, device=cuda_device)
    dX = torch.zeros(16, 24, dtype=torch.bfloat16, device=cuda_device)
    with pytest.raises(tp.TPError) as e:
        tp.tp_column_linear_backward(X, W, dY, dX, None, n_shards=3)  # 3 does not divide 40
    assert e.value.status == 3
    with pytest.raises(tp.TPError) as e:
        tp.tp_row_linear_backward(X, W, dY, dX, None, n_shards=5)     # 5 does not divide 24
    assert e.value.status == 3
    with pytest.raises(tp.TPError) as e:
        tp.tp_column_linear_backward(X, W, dY, X, None, n_shards=2)   # dX aliases X
    assert e.value.status == 9
    with pytest.raises(tp.TPError) as e:                              # fp32 inputs
        tp.tp_column_linear_backward(X.float(), W.float(), dY.float(), dX.float(), None)
    assert e.value.status == 5
    assert tp.tp_get_device_status() == tp.TP_OK


def test_gelu_grad_epilogue_accuracy(tp, cuda_device):
    """The backward epilogue's GeLU'(z) = Phi(z) + z phi(z) at every bf16 z in
    [-12, 12], isolated: with W1 = [I_8 | I_8 | ...] the recomputed
    pre-activation Z = X.W1 copies X's entries exactly, and with dY = e_0 and
    W2[:, 0] = 1 the product dY.W2^T is 1 everywhere, so the dZ stored in the
    workspace is bf16(GeLU'(z)).  Bound: one bf16 ulp of the round-to-
    nearest-even of the fp64 value, except near the zero of GeLU' (where
    the two terms cancel and only an error relative to their magnitude,
    Phi(z) + |z| phi(z), is meaningful: 2^-8 of the value plus 1e-4 of that
    magnitude), and nothing below 1e-30."""
    import math
    import torch
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = oracle.bf16_to_f64(bits)
    keep = np.isfinite(vals) & (np.abs(vals) <= 12.0)
    xb, xs = bits[keep], vals[keep]
    pad = (-xb.size) % 8
    xb = np.concatenate([xb, np.zeros(pad, np.uint16)])
    xs = np.concatenate([xs, np.zeros(pad)])
    M, d, f = xb.size // 8, 8, 8 * 33
    w1 = np.zeros((d, f))
    w1[np.arange(f) % 8, np.arange(f)] = 1.0
    w2 = np.zeros((f, d))
    w2[:, 0] = 1.0
    g = np.zeros((M, d))
    g[:, 0] = 1.0
    X = to_dev_bf16(xb.reshape(M, d), cuda_device)
    W1, W2, dY = (to_dev_bf16(oracle.f64_to_bf16(a), cuda_device) for a in (w1, w2, g))
    ws = torch.empty(tp.tp_mlp_block_backward_workspace_size(M, f, torch.bfloat16),
                     dtype=torch.uint8, device=cuda_device)
    dX = torch.empty(M, d, dtype=torch.bfloat16, device=cuda_device)
    tp.tp_mlp_block_backward(X, W1, W2, dY, ws, dX, None, None, n_shards=1)
    assert tp.tp_get_device_status() == tp.TP_OK
    part = (M * f * 2 + 255) // 256 * 256
    dZ = ws[2 * part: 2 * part + M * f * 2].view(torch.int16).view(M, f)
    got_bits = dZ.cpu().numpy().view(np.uint16)
    z = xs.reshape(M, d)[:, np.arange(f) % 8]
    ref = oracle.gelu_grad(z.ravel()).reshape(M, f)
    got = oracle.bf16_to_f64(got_bits)
    phi = np.exp(-0.5 * z * z) / math.sqrt(2.0 * math.pi)
    scale = 0.5 * (1.0 + np.vectorize(math.erf)(z / math.sqrt(2.0))) + np.abs(z) * phi
    want = oracle.f64_to_bf16(ref)
    line = lambda b: np.where(b.astype(np.int64) & 0x8000, -(b.astype(np.int64) & 0x7FFF),
                              b.astype(np.int64) & 0x7FFF)
    ulps = np.abs(line(got_bits) - line(want))
    ok = ((ulps <= 1) | (np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-4 * scale)
          | (np.abs(ref) < 1e-30) & (np.abs(got) < 1e-30))
    worst = int(np.argmin(ok))
    assert ok.all(), (f"GeLU'({z.flat[worst]!r}) -> {got.flat[worst]!r}, oracle "
                      f"{ref.flat[worst]!r} ({ulps.flat[worst]} ulp)")
    # where the terms do not cancel, the one-ulp bound holds on its own
    clear = np.abs(ref) >= 0.05 * scale
    assert np.all(ulps[clear & (np.abs(ref) >= 1e-30)] <= 1)


def test_backward_half_width_last_round(tp, cuda_device):
    """Input and weight gradients whose 256-wide tiles fill a few more than
    one round of the GPU's CTA pairs: the last tiles run as half-width
    units, for dX = dY.W^T through the second, half-height tensor map of
    the [N][K] operand, and for dW = X^T.dY.  Against the oracle and bit
    for bit against the all-128-wide plan."""
    import os
    import torch
    P = torch.cuda.get_device_properties(0).multi_processor_count // 2
    mt = P // 8 + 1
    M, K, N, n = 256 * mt - 21, 8 * 256, 264, 2   # dX [M, K]: 8 * mt tiles
    xb = inputs.bf16_normal((M, K), inputs.stream_seed(83, 0), 1.0)
    wb = inputs.bf16_normal((K, N), inputs.stream_seed(83, 1), 0.02)
    gb = inputs.bf16_normal((M, N), inputs.stream_seed(83, 2), 1.0)
    X, W, dY = (to_dev_bf16(b, cuda_device) for b in (xb, wb, gb))
    rX, rW = oracle.column_linear_backward(*(oracle.bf16_to_f64(b) for b in (xb, wb, gb)), n)
    outs = {}
    for plan in ("256", "128"):
        os.environ["TP_GEMM_PLAN"] = plan
        try:
            dX = torch.empty(M, K, dtype=torch.float32, device=cuda_device)
            tp.tp_column_linear_backward(X, W, dY, dX, None, n_shards=n)
        finally:
            del os.environ["TP_GEMM_PLAN"]
        assert tp.tp_get_device_status() == tp.TP_OK
        assert_bf16_parity(dev_to_f64(dX), rX, f"dX, plan {plan}", out_bf16=False)
        outs[plan] = dev_bits(dX)
    np.testing.assert_array_equal(outs["256"], outs["128"])
    # dW = X^T.dY [K', N'] with K' = 256 mt rows of tiles: X2 [M2, 256 mt], dY2 [M2, 8 * 256]
    M2 = 520
    x2 = inputs.bf16_normal((M2, 256 * mt), inputs.stream_seed(84, 0), 1.0)
    g2 = inputs.bf16_normal((M2, 2048), inputs.stream_seed(84, 1), 1.0)
    w2 = inputs.bf16_normal((256 * mt, 2048), inputs.stream_seed(84, 2), 0.02)
    X2, dY2, W2 = (to_dev_bf16(b, cuda_device) for b in (x2, g2, w2))
    _, rW2 = oracle.column_linear_backward(*(oracle.bf16_to_f64(b) for b in (x2, w2, g2)), 1)
    dW = torch.empty(256 * mt, 2048, dtype=torch.float32, device=cuda_device)
    tp.tp_column_linear_backward(X2, W2, dY2, None, dW, n_shards=1)
    assert tp.tp_get_device_status() == tp.TP_OK
    assert_bf16_parity(dev_to_f64(dW), rW2, "dW, short last round", out_bf16=False)


def _random_backward_shapes(count, seed):
    """Seeded shapes inside the boundary's rules (dimensions that are row
    pitches multiples of 8; the split axis a multiple of 8 n), one row up to
    a few tiles with ragged tails."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(count):
        n = int(rng.choice([1, 2, 3, 4, 8]))
        M = int(rng.integers(1, 600))
        d = 8 * int(rng.integers(1, 90))
        f = 8 * n * int(rng.integers(1, max(2, 900 // (8 * n))))
        out.append((M, d, f, n))
    return out


@pytest.mark.parametrize("M,d,f,n", _random_backward_shapes(6, 20261204))
def test_random_shapes_backward(tp, cuda_device, M, d, f, n):
    """The MLP block's gradients and the row linear's (X = H-like input of
    width f, W = W2) on seeded random shapes, each against the oracle."""
    import torch
    seed = 11 * M + 5 * d + f + n
    xb = inputs.bf16_normal((M, d), inputs.stream_seed(seed, 0), 1.0)
    w1b = inputs.bf16_normal((d, f), inputs.stream_seed(seed, 1), 0.02)
    w2b = inputs.bf16_normal((f, d), inputs.stream_seed(seed, 2), 0.02)
    gb = inputs.bf16_normal((M, d), inputs.stream_seed(seed, 3), 1.0)
    hb = inputs.bf16_normal((M, f), inputs.stream_seed(seed, 4), 0.5)
    X, W1, W2, dY, Hx = (to_dev_bf16(b, cuda_device) for b in (xb, w1b, w2b, gb, hb))
    ws = torch.empty(tp.tp_mlp_block_backward_workspace_size(M, f, torch.bfloat16),
                     dtype=torch.uint8, device=cuda_device)
    dX = torch.empty(M, d, dtype=torch.bfloat16, device=cuda_device)
    dW1 = torch.empty(d, f, dtype=torch.bfloat16, device=cuda_device)
    dW2 = torch.empty(f, d, dtype=torch.bfloat16, device=cuda_device)
    tp.tp_mlp_block_backward(X, W1, W2, dY, ws, dX, dW1, dW2, n_shards=n)
    dH = torch.empty(M, f, dtype=torch.bfloat16, device=cuda_device)
    dWr = torch.empty(f, d, dtype=torch.bfloat16, device=cuda_device)
    tp.tp_row_linear_backward(Hx, W2, dY, dH, dWr, n_shards=n)
    assert tp.tp_get_device_status() == tp.TP_OK
    f64 = oracle.bf16_to_f64
    rX, rW1, rW2 = oracle.mlp_block_backward(f64(xb), f64(w1b), f64(w2b), f64(gb), n)
    shape = f"{M}x{d}x{f} n={n}"
    assert_bf16_parity(bf16_dev_to_f64(dX), rX, f"MLP dX {shape}")
    assert_bf16_parity(bf16_dev_to_f64(dW1), rW1, f"MLP dW1 {shape}")
    assert_bf16_parity(bf16_dev_to_f64(dW2), rW2, f"MLP dW2 {shape}")
    rH, rWr = oracle.row_linear_backward(f64(hb), f64(w2b), f64(gb), n)
    assert_bf16_parity(bf16_dev_to_f64(dH), rH, f"row dX {shape}")
    assert_bf16_parity(bf16_dev_to_f64(dWr), rWr, f"row dW {shape}")
