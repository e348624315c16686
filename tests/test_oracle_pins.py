"""Pins of the fp64 oracle against things other than itself (CPU only).

Each test ties one oracle function to something the pages or mathematics fix:
the glossary page's worked example, brute force in plain Python integers,
a library routine (scipy's normal CDF, numpy's concatenate, torch's float32
to bf16 conversion), tabulated values, and the invariant that the sharded
result equals the unsharded one.  The last test plants mistakes in the
oracle's inputs and checks that the pins catch them.
"""
import itertools
import math
import os
import random

import numpy as np
import pytest
import scipy.special

import oracle
from tensor_sharded_linear_02_b300 import inputs

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _read_golden(name):
    rows = {}
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            rows.setdefault(key, []).append([float(v) for v in vals])
    return rows


@pytest.fixture(scope="module")
def worked():
    g = _read_golden("worked_example.txt")
    X = np.array(g["X"])
    W = np.array(g["W"])
    return X, W, g


# ------------------------------------------------------- worked example -----

def test_worked_example_full_product(worked):
    X, W, g = worked
    np.testing.assert_array_equal(oracle.matmul(X, W), np.array(g["Y"]))


def test_worked_example_column_split(worked):
    X, W, g = worked
    Y, Ys = oracle.column_linear(X, W, n_shards=2)
    np.testing.assert_array_equal(Ys[0], np.array([g["column_shard"][0]]))
    np.testing.assert_array_equal(Ys[1], np.array([g["column_shard"][1]]))
    np.testing.assert_array_equal(Y, np.array(g["Y"]))
    np.testing.assert_array_equal(oracle.shard_concat(Ys), np.array(g["Y"]))


def test_worked_example_row_split(worked):
    X, W, g = worked
    Y, P = oracle.row_linear(X, W, n_shards=2)
    np.testing.assert_array_equal(P[0], np.array([g["row_partial"][0]]))
    np.testing.assert_array_equal(P[1], np.array([g["row_partial"][1]]))
    np.testing.assert_array_equal(Y, np.array(g["Y"]))
    np.testing.assert_array_equal(oracle.shard_reduce(P.astype(np.float32)), np.array(g["Y"]))


def test_combine_rule_from_quiz(worked):
    """Glossary "Check your understanding": partials covering the same output
    coordinates are added; outputs covering different coordinates are
    concatenated.  The row split's partials each span all of Y; the column
    split's shard outputs are disjoint and their widths add up to Y's."""
    X, W, _ = worked
    _, P = oracle.row_linear(X, W, 2)
    _, Ys = oracle.column_linear(X, W, 2)
    assert all(p.shape == (1, 4) for p in P)
    assert sum(y.shape[1] for y in Ys) == 4


# ------------------------------------------------------- brute force -------

def _bf_matmul(X, W):
    M, K = len(X), len(X[0]) if X else 0
    N = len(W[0]) if W else 0
    return [[sum(X[i][k] * W[k][j] for k in range(K)) for j in range(N)] for i in range(M)]


def _divisors(n):
    return [d for d in range(1, n + 1) if n % d == 0]


def _rand_int_matrix(rng, r, c):
    return [[rng.randint(-9, 9) for _ in range(c)] for _ in range(r)]


def test_brute_force_integer_shapes():
    """Plain Python integer loops on random tiny shapes, every shard count
    that divides the split axis: exact equality."""
    rng = random.Random(12345)
    for _ in range(60):
        M, K, N = rng.randint(1, 8), rng.randint(1, 8), rng.randint(1, 8)
        X, W = _rand_int_matrix(rng, M, K), _rand_int_matrix(rng, K, N)
        ref = _bf_matmul(X, W)
        np.testing.assert_array_equal(oracle.matmul(X, W), np.array(ref, dtype=np.float64))
        for n in _divisors(N):
            Y, Ys = oracle.column_linear(X, W, n)
            np.testing.assert_array_equal(Y, ref)
            w = N // n
            for i in range(n):
                Wi = [row[i * w:(i + 1) * w] for row in W]
                np.testing.assert_array_equal(Ys[i], _bf_matmul(X, Wi))
        for n in _divisors(K):
            Y, P = oracle.row_linear(X, W, n)
            np.testing.assert_array_equal(Y, ref)
            ks = K // n
            for i in range(n):
                Xi = [row[i * ks:(i + 1) * ks] for row in X]
                Wi = W[i * ks:(i + 1) * ks]
                np.testing.assert_array_equal(P[i], _bf_matmul(Xi, Wi))


def test_brute_force_head_groups():
    """Head-group column split (G column blocks, shard i owns slice i of each
    block): brute force on labelled columns."""
    rng = random.Random(7)
    for G, n, sw in [(3, 2, 1), (3, 2, 2), (3, 4, 1), (2, 2, 3)]:
        N = G * n * sw
        M, K = 3, 4
        X, W = _rand_int_matrix(rng, M, K), _rand_int_matrix(rng, K, N)
        ref = _bf_matmul(X, W)
        Y, Ys = oracle.column_linear(X, W, n, col_groups=G)
        np.testing.assert_array_equal(Y, ref)
        for i in range(n):
            cols = [b * (N // G) + i * sw + j for b in range(G) for j in range(sw)]
            np.testing.assert_array_equal(Ys[i], [[r[c] for c in cols] for r in ref])
        np.testing.assert_array_equal(oracle.shard_concat(Ys, col_groups=G), ref)


def test_mlp_brute_force_with_library_gelu():
    """MLP block on tiny shapes against plain loops whose GeLU is
    x * scipy.special.ndtr(x) (a library normal CDF, not the oracle's erf)."""
    rng = np.random.default_rng(3)
    for M, d, f, n in [(3, 4, 8, 2), (2, 5, 6, 3), (4, 3, 4, 4), (1, 2, 2, 1)]:
        X = rng.standard_normal((M, d))
        W1 = rng.standard_normal((d, f))
        W2 = rng.standard_normal((f, d))
        H = [[sum(X[i, k] * W1[k, j] for k in range(d)) for j in range(f)] for i in range(M)]
        H = [[h * float(scipy.special.ndtr(h)) for h in row] for row in H]
        Y = [[sum(H[i][k] * W2[k, j] for k in range(f)) for j in range(d)] for i in range(M)]
        got = oracle.mlp_block(X, W1, W2, n)
        np.testing.assert_allclose(got, Y, rtol=1e-12, atol=1e-12)


def _bf16_round_py(v):
    """Round a double to the nearest bf16 value, ties to even, by exact
    float arithmetic: frexp gives v = m 2^e with 0.5 <= |m| < 1, m * 2^8 is
    exact, and Python's round() rounds halves to even (normal range only)."""
    if v == 0.0:
        return v
    m, e = math.frexp(v)
    return math.ldexp(round(m * 256.0), e - 8)


def test_mlp_mirror_mode_rounds_hidden_to_bf16():
    """The oracle's diagnostic mode (hidden activation rounded to bf16 before
    the second product) against plain loops: GeLU from scipy's normal CDF,
    each H value rounded to bf16 by _bf16_round_py, then the row product
    and the ascending shard sum.  The mode must also differ from the plain
    oracle (the rounding really happens), by no more than the rounding of H
    allows."""
    rng = np.random.default_rng(11)
    for M, d, f, n in [(3, 4, 8, 2), (2, 5, 6, 3), (4, 8, 16, 4), (1, 2, 2, 1)]:
        X = rng.standard_normal((M, d))
        W1 = rng.standard_normal((d, f))
        W2 = rng.standard_normal((f, d))
        H = [[sum(X[i, k] * W1[k, j] for k in range(d)) for j in range(f)] for i in range(M)]
        H = [[_bf16_round_py(h * float(scipy.special.ndtr(h))) for h in row] for row in H]
        fs = f // n
        Y = [[sum(sum(H[i][s * fs + k] * W2[s * fs + k, j] for k in range(fs)) for s in range(n))
              for j in range(d)] for i in range(M)]
        got = oracle.mlp_block(X, W1, W2, n, mirror_h_bf16=True)
        np.testing.assert_allclose(got, Y, rtol=1e-12, atol=1e-12)
        plain = oracle.mlp_block(X, W1, W2, n)
        assert not np.array_equal(got, plain)
        # |H_bf16 - H| <= 2^-8 |H| (8 significant bits), so
        # |dY| <= 2^-8 sum_k |H_k| |W2_kj|
        Hp = np.array([[h * scipy.special.ndtr(h) for h in row] for row in (X @ W1)])
        bound = 2.0 ** -8 * (np.abs(Hp) @ np.abs(W2)) + 1e-12
        assert np.all(np.abs(got - plain) <= bound)


def test_sequence_parallel_combines_brute_force():
    """Sequence-parallel combines ([TP-topic] "Sequence Parallelism
    Extension") on tiny integer shapes against plain Python: the all-gather
    stacks the token blocks in shard order, and the combine after the block
    gives shard i the sum over all shards' partials of its own token rows
    [i*M/n, (i+1)*M/n).  Planted mistakes (own partial only, another
    shard's rows, a dropped shard) are rejected."""
    rnd = random.Random(5)
    for n, Mb, cols in [(1, 3, 2), (2, 2, 3), (3, 1, 4), (4, 2, 1), (8, 1, 2)]:
        M = n * Mb
        P = [[[rnd.randint(-9, 9) for _ in range(cols)] for _ in range(M)] for _ in range(n)]
        want = [[[sum(P[j][i * Mb + r][c] for j in range(n)) for c in range(cols)]
                 for r in range(Mb)] for i in range(n)]
        got = oracle.reduce_scatter_rows(np.array(P, dtype=np.float64))
        np.testing.assert_array_equal(got, want)
        own_only = [[P[i][i * Mb + r] for r in range(Mb)] for i in range(n)]
        if n > 1:
            assert not np.array_equal(got, own_only)
            assert not np.array_equal(got, np.roll(np.array(want), 1, axis=0))
            dropped = [[[sum(P[j][i * Mb + r][c] for j in range(n - 1)) for c in range(cols)]
                        for r in range(Mb)] for i in range(n)]
            assert not np.array_equal(got, dropped) or not any(
                P[n - 1][r][c] for r in range(M) for c in range(cols))
        Xs = [[[rnd.randint(-9, 9) for _ in range(cols)] for _ in range(Mb)] for _ in range(n)]
        gathered = [row for block in Xs for row in block]
        np.testing.assert_array_equal(oracle.allgather_rows(np.array(Xs, dtype=np.float64)),
                                      gathered)


def test_sequence_parallel_mlp_block_brute_force():
    """The MLP block between two sequence-split regions: token blocks
    all-gathered, each shard's GeLU(X.W1_i).W2_i for every token (GeLU from
    scipy's normal CDF), partials summed and split by token rows; against
    plain loops, for every shard count dividing both the tokens and f."""
    rng = np.random.default_rng(9)
    for n, Mb, d, f in [(1, 3, 4, 4), (2, 2, 3, 4), (3, 1, 2, 6), (4, 2, 2, 8)]:
        M = n * Mb
        Xs = rng.standard_normal((n, Mb, d))
        W1 = rng.standard_normal((d, f))
        W2 = rng.standard_normal((f, d))
        X = [list(Xs[i, r]) for i in range(n) for r in range(Mb)]
        fs = f // n
        P = []
        for s_ in range(n):
            H = [[sum(X[t][k] * W1[k, s_ * fs + j] for k in range(d)) for j in range(fs)]
                 for t in range(M)]
            H = [[h * float(scipy.special.ndtr(h)) for h in row] for row in H]
            P.append([[sum(H[t][j] * W2[s_ * fs + j, c] for j in range(fs)) for c in range(d)]
                      for t in range(M)])
        want = [[[sum(P[s_][i * Mb + r][c] for s_ in range(n)) for c in range(d)]
                 for r in range(Mb)] for i in range(n)]
        got = oracle.seq_parallel_mlp_block(Xs, W1, W2)
        np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_bias_brute_force_integer_shapes():
    """Biases on tiny integer shapes against plain Python loops: the column
    split adds each shard's slice of the bias to its outputs, the row split
    adds the bias once after the sum, for every shard count; a bias added by
    every shard of the row split (n times) is caught."""
    rng = random.Random(777)
    for _ in range(40):
        M, K, N = rng.randint(1, 6), rng.randint(1, 8), rng.randint(1, 8)
        X, W = _rand_int_matrix(rng, M, K), _rand_int_matrix(rng, K, N)
        b = [rng.randint(-4, 4) for _ in range(N)]
        ref = [[v + b[j] for j, v in enumerate(row)] for row in _bf_matmul(X, W)]
        for n in _divisors(N):
            Y, Ys = oracle.column_linear(X, W, n, bias=b)
            np.testing.assert_array_equal(Y, ref)
            w = N // n
            for i in range(n):
                np.testing.assert_array_equal(Ys[i], [row[i * w:(i + 1) * w] for row in ref])
        for n in _divisors(K):
            Y, P = oracle.row_linear(X, W, n, bias=b)
            np.testing.assert_array_equal(Y, ref)
            np.testing.assert_array_equal(P.sum(axis=0), np.array(_bf_matmul(X, W), float))
            if n > 1 and any(b):
                per_shard = P.sum(axis=0) + n * np.array(b, float)
                assert not np.array_equal(per_shard, np.array(ref, float))


def test_mlp_bias_brute_force_with_library_gelu():
    """MLP block with b1 (split with W1, before the GeLU) and b2 (once after
    the sum) against plain loops with scipy's normal CDF."""
    rng = np.random.default_rng(8)
    for M, d, f, n in [(3, 4, 8, 2), (2, 5, 6, 3), (4, 3, 4, 4)]:
        X = rng.standard_normal((M, d))
        W1, W2 = rng.standard_normal((d, f)), rng.standard_normal((f, d))
        b1, b2 = rng.standard_normal(f), rng.standard_normal(d)
        H = [[sum(X[i, k] * W1[k, j] for k in range(d)) + b1[j] for j in range(f)]
             for i in range(M)]
        H = [[h * float(scipy.special.ndtr(h)) for h in row] for row in H]
        Y = [[sum(H[i][k] * W2[k, j] for k in range(f)) + b2[j] for j in range(d)]
             for i in range(M)]
        got = oracle.mlp_block(X, W1, W2, n, b1=b1, b2=b2)
        np.testing.assert_allclose(got, Y, rtol=1e-12, atol=1e-12)


def test_qkv_gqa_brute_force():
    """GQA split on tiny integer shapes against Python-int loops: shard i's
    local output is X times its own Q head columns followed by the K and V
    columns of the KV heads its Q heads use (split when n divides hkv,
    replicated when hkv divides n); with hkv = hq it equals the head-group
    split of column_linear (col_groups = 3), and the full output is X.W."""
    rng = random.Random(99)
    for hq, hkv, hd, n in [(4, 2, 2, 2), (4, 1, 3, 4), (8, 2, 1, 8), (6, 3, 2, 3), (4, 4, 2, 2),
                           (8, 4, 2, 2)]:
        M, K = rng.randint(1, 4), rng.randint(1, 5)
        N = (hq + 2 * hkv) * hd
        X, W = _rand_int_matrix(rng, M, K), _rand_int_matrix(rng, K, N)
        Y, Ys = oracle.qkv_linear(X, W, hq, hkv, hd, n)
        full = _bf_matmul(X, W)
        np.testing.assert_array_equal(Y, full)
        group = hq // hkv  # Q heads per KV head
        for i in range(n):
            qh = list(range(i * hq // n, (i + 1) * hq // n))
            kvh = sorted({h // group for h in qh})   # the KV heads these Q heads read
            cols = ([h * hd + j for h in qh for j in range(hd)]
                    + [hq * hd + h * hd + j for h in kvh for j in range(hd)]
                    + [(hq + hkv) * hd + h * hd + j for h in kvh for j in range(hd)])
            np.testing.assert_array_equal(Ys[i], [[row[c] for c in cols] for row in full])
        if hkv == hq:
            _, Yg = oracle.column_linear(X, W, n, col_groups=3)
            np.testing.assert_array_equal(Ys, Yg)


# --------------------------------------------- sharded == unsharded --------

def test_sharded_equals_unsharded_float():
    """Sharded result equals the unsharded one for every shard count
    ([TP-topic] Implementation Considerations: same results as one device),
    up to double reassociation in the row/MLP sums."""
    rng = np.random.default_rng(11)
    M, K, N = 5, 24, 24
    X = rng.standard_normal((M, K))
    W = rng.standard_normal((K, N))
    ref = oracle.matmul(X, W)
    for n in _divisors(24):
        Y, _ = oracle.column_linear(X, W, n)
        np.testing.assert_array_equal(Y, ref)  # same dot products, same order
        Y, P = oracle.row_linear(X, W, n)
        np.testing.assert_allclose(Y, ref, rtol=1e-12, atol=1e-12)
    W1 = rng.standard_normal((K, 48)) * 0.2
    W2 = rng.standard_normal((48, K)) * 0.2
    ref = oracle.mlp_block(X, W1, W2, 1)
    for n in _divisors(48):
        np.testing.assert_allclose(oracle.mlp_block(X, W1, W2, n), ref, rtol=1e-12, atol=1e-12)


def test_mlp_equals_composed_steps():
    """MLP block = row split of GeLU(column split) with the column output
    never concatenated ([TP-topic] Row-Wise: the input is already split)."""
    rng = np.random.default_rng(5)
    X = rng.standard_normal((6, 8))
    W1 = rng.standard_normal((8, 16))
    W2 = rng.standard_normal((16, 8))
    for n in (1, 2, 4, 8):
        H, _ = oracle.column_linear(X, W1, n, act="gelu")
        Y, _ = oracle.row_linear(H, W2, n)
        np.testing.assert_allclose(oracle.mlp_block(X, W1, W2, n), Y, rtol=1e-13, atol=1e-13)


# --------------------------------------------------------------- GeLU ------

def test_gelu_against_library_cdf():
    x = np.concatenate([np.linspace(-12, 12, 4001), inputs.normal((5000,), 99, 3.0)])
    ref = x * scipy.special.ndtr(x)
    np.testing.assert_allclose(oracle.gelu(x), ref, rtol=1e-13, atol=1e-300)


def test_gelu_textbook_values():
    g = _read_golden("gelu_textbook.txt")
    for x, phi in (row for key, rows in g.items() for row in [[float(key)] + r for r in rows]):
        assert abs(oracle.gelu([x])[0] - x * phi) <= 1e-9 * max(1.0, abs(x))


def test_gelu_special_values():
    assert oracle.gelu([0.0])[0] == 0.0
    x = np.linspace(-8, 8, 257)
    # x*Phi(x) - (-x)*Phi(-x) = x*(Phi(x) + Phi(-x)) = x
    np.testing.assert_allclose(oracle.gelu(x) - oracle.gelu(-x), x, rtol=0, atol=1e-14)
    assert oracle.gelu([40.0])[0] == 40.0
    assert oracle.gelu([-40.0])[0] == 0.0 or abs(oracle.gelu([-40.0])[0]) < 1e-300


# --------------------------------------------------------------- bf16 ------

def test_bf16_hand_cases():
    f = oracle.f64_to_bf16
    cases = [
        (1.0, 0x3F80), (-2.0, 0xC000), (0.0, 0x0000), (-0.0, 0x8000),
        (1.0 + 2.0 ** -8, 0x3F80),            # tie -> even (mantissa 0)
        (1.0 + 3 * 2.0 ** -8, 0x3F82),        # tie -> even (mantissa 2)
        (1.0 + 2.0 ** -8 + 2.0 ** -20, 0x3F81),  # just above the tie
        (3.3895313892515355e38, 0x7F7F),      # largest finite bf16
        (3.4e38, 0x7F80),                     # rounds past the largest finite
        (2.0 ** -133, 0x0001),                # smallest subnormal
        (2.0 ** -134, 0x0000),                # tie between 0 and 2^-133 -> even (0)
        (3 * 2.0 ** -134, 0x0002),            # tie between 1 and 2 quanta -> even
        (2.0 ** -126, 0x0080),                # smallest normal
        (float("inf"), 0x7F80), (float("-inf"), 0xFF80),
    ]
    for x, bits in cases:
        assert int(f(np.array([x]))[0]) == bits, (x, hex(int(f(np.array([x]))[0])), hex(bits))
    assert np.isnan(oracle.bf16_to_f64(f(np.array([float("nan")]))))[0]
    for bits in (0x3F80, 0xC000, 0x0001, 0x0080, 0x7F7F, 0x8001):
        v = oracle.bf16_to_f64(np.array([bits], dtype=np.uint16))[0]
        assert int(f(np.array([v]))[0]) == bits


def test_bf16_against_torch_from_float32():
    """For float32 sources (no double rounding) the oracle's RNE must agree
    with torch's float32 -> bfloat16 conversion bit for bit."""
    import torch
    rng = np.random.default_rng(0)
    bits32 = rng.integers(0, 2 ** 32, size=200000, dtype=np.uint64).astype(np.uint32)
    x32 = bits32.view(np.float32)
    x32 = x32[np.isfinite(x32)]
    ours = oracle.f64_to_bf16(x32.astype(np.float64))
    theirs = torch.from_numpy(x32.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, theirs)
    back = oracle.bf16_to_f64(theirs)
    np.testing.assert_array_equal(back, torch.from_numpy(theirs.view(np.int16).copy()).view(torch.bfloat16).double().numpy())


# ------------------------------------------------------- reduce/concat -----

def test_reduce_integer_exact_and_float_vs_fsum():
    rng = np.random.default_rng(2)
    P = rng.integers(-1000, 1000, size=(5, 7, 9)).astype(np.float32)
    np.testing.assert_array_equal(oracle.shard_reduce(P), P.astype(np.int64).sum(axis=0))
    P = rng.standard_normal((16, 3, 5)).astype(np.float32)
    got = oracle.shard_reduce(P)
    for r, c in itertools.product(range(3), range(5)):
        ref = math.fsum(float(v) for v in P[:, r, c])
        assert abs(got[r, c] - ref) <= 1e-15 * max(1.0, abs(ref))


def test_concat_against_numpy():
    rng = np.random.default_rng(4)
    Ys = rng.standard_normal((4, 6, 8))
    np.testing.assert_array_equal(oracle.shard_concat(Ys), np.concatenate(list(Ys), axis=1))


# ------------------------------------------------------------- backward ----

def test_gelu_grad_against_finite_differences():
    """GeLU' against central differences of the oracle's own GeLU (truncation
    error ~ h^2 times the third derivative, about 1e-10 here), its value at 0
    and the identity GeLU'(z) + GeLU'(-z) = 1 (Phi(z) + Phi(-z) = 1 and
    z*phi(z) is odd)."""
    x = np.linspace(-8.0, 8.0, 321)
    h = 1e-5
    fd = (oracle.gelu(x + h) - oracle.gelu(x - h)) / (2 * h)
    np.testing.assert_allclose(oracle.gelu_grad(x), fd, rtol=0, atol=1e-8)
    assert oracle.gelu_grad([0.0])[0] == 0.5
    np.testing.assert_allclose(oracle.gelu_grad(x) + oracle.gelu_grad(-x), 1.0, atol=1e-15)


def _loss_column(X, W, dY, n):
    Y, _ = oracle.column_linear(X, W, n)
    return float(np.sum(Y * dY))


def _loss_row(X, W, dY, n):
    Y, _ = oracle.row_linear(X, W, n)
    return float(np.sum(Y * dY))


@pytest.mark.parametrize("kind", ["column", "row"])
def test_linear_backward_is_the_forward_derivative(kind):
    """L(X, W) = sum(Y * dY) is linear in X and in W separately, so on small
    integers the change of the forward oracle's L along any integer direction
    E equals <grad, E> exactly.  Checked for every shard count dividing the
    split axis, plus: the sharded gradients equal the one-shard ones."""
    rng = np.random.default_rng(11)
    for M, K, N in [(3, 4, 6), (5, 6, 4), (2, 8, 8)]:
        X = rng.integers(-4, 5, (M, K)).astype(float)
        W = rng.integers(-4, 5, (K, N)).astype(float)
        dY = rng.integers(-4, 5, (M, N)).astype(float)
        axis = N if kind == "column" else K
        back = oracle.column_linear_backward if kind == "column" else oracle.row_linear_backward
        loss = _loss_column if kind == "column" else _loss_row
        ref = back(X, W, dY, 1)
        for n in [s for s in range(1, axis + 1) if axis % s == 0]:
            dX, dW = back(X, W, dY, n)
            np.testing.assert_array_equal(dX, ref[0])
            np.testing.assert_array_equal(dW, ref[1])
            for _ in range(3):
                EX = rng.integers(-3, 4, X.shape).astype(float)
                EW = rng.integers(-3, 4, W.shape).astype(float)
                assert loss(X + EX, W, dY, n) - loss(X, W, dY, n) == float(np.sum(dX * EX))
                assert loss(X, W + EW, dY, n) - loss(X, W, dY, n) == float(np.sum(dW * EW))


def test_mlp_backward_against_finite_differences():
    """dX, dW1, dW2 of the MLP block against central differences of the
    forward oracle's L = sum(Y * dY) along random directions (relative error
    of the difference quotient ~ h^2 ~ 1e-10), for 1, 2 and 4 shards; the
    sharded gradients equal the one-shard ones up to reassociation."""
    rng = np.random.default_rng(5)
    M, d, f = 5, 6, 8
    X = rng.standard_normal((M, d))
    W1 = rng.standard_normal((d, f)) * 0.5
    W2 = rng.standard_normal((f, d)) * 0.5
    dY = rng.standard_normal((M, d))
    ref = oracle.mlp_block_backward(X, W1, W2, dY, 1)
    h = 1e-5

    def L(X_, W1_, W2_, n):
        return float(np.sum(oracle.mlp_block(X_, W1_, W2_, n) * dY))

    for n in (1, 2, 4):
        dX, dW1, dW2 = oracle.mlp_block_backward(X, W1, W2, dY, n)
        for got, want in zip((dX, dW1, dW2), ref):
            np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)
        for _ in range(3):
            E = [rng.standard_normal(a.shape) for a in (X, W1, W2)]
            fd = [
                (L(X + h * E[0], W1, W2, n) - L(X - h * E[0], W1, W2, n)) / (2 * h),
                (L(X, W1 + h * E[1], W2, n) - L(X, W1 - h * E[1], W2, n)) / (2 * h),
                (L(X, W1, W2 + h * E[2], n) - L(X, W1, W2 - h * E[2], n)) / (2 * h),
            ]
            for g, e, q in zip((dX, dW1, dW2), E, fd):
                assert abs(float(np.sum(g * e)) - q) <= 1e-7 * max(1.0, abs(q))


def test_sampled_mlp_backward_matches_full_and_finite_differences():
    """The per-value backward oracle (for full-size checks) against the
    matrix-level backward oracle on small shapes, every shard count, and a
    few of its values against central differences of the forward oracle."""
    rng = np.random.default_rng(21)
    for M, d, f in [(5, 4, 8), (3, 6, 12), (7, 3, 6)]:
        X = rng.standard_normal((M, d))
        W1 = rng.standard_normal((d, f)) * 0.5
        W2 = rng.standard_normal((f, d)) * 0.5
        dY = rng.standard_normal((M, d))
        for n in [k for k in (1, 2, 3, 4, 6) if f % k == 0]:
            rX, rW1, rW2 = oracle.mlp_block_backward(X, W1, W2, dY, n)
            rows = [0, M - 1, M // 2]
            cols = [0, f - 1, f // 3]
            rows2 = [f - 1, 0, f // 2]
            sX, sW1, sW2 = oracle.mlp_block_backward_sampled(X, W1, W2, dY, n, rows, cols, rows2)
            np.testing.assert_allclose(sX, rX[rows], rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(sW1, rW1[:, cols], rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(sW2, rW2[rows2], rtol=1e-12, atol=1e-12)
    # independent of both: L = sum(Y * dY), dL/dX[r, k] by central differences
    M, d, f = 4, 3, 6
    X = rng.standard_normal((M, d)); W1 = rng.standard_normal((d, f)); W2 = rng.standard_normal((f, d))
    dY = rng.standard_normal((M, d))
    sX, sW1, sW2 = oracle.mlp_block_backward_sampled(X, W1, W2, dY, 2, [2], [4], [1])
    h = 1e-6
    def L(X_, W1_, W2_):
        return float(np.sum(oracle.mlp_block(X_, W1_, W2_, 2) * dY))
    for k in range(d):
        E = np.zeros_like(X); E[2, k] = h
        assert abs((L(X + E, W1, W2) - L(X - E, W1, W2)) / (2 * h) - sX[0, k]) < 1e-6
        E1 = np.zeros_like(W1); E1[k, 4] = h
        assert abs((L(X, W1 + E1, W2) - L(X, W1 - E1, W2)) / (2 * h) - sW1[k, 0]) < 1e-6
        E2 = np.zeros_like(W2); E2[1, k] = h
        assert abs((L(X, W1, W2 + E2) - L(X, W1, W2 - E2)) / (2 * h) - sW2[0, k]) < 1e-6


def test_backward_pins_catch_planted_mistakes():
    """Gradients with a dropped GeLU' factor or a missing shard in the
    backward sum fail the finite-difference pin that the oracle passes."""
    rng = np.random.default_rng(6)
    M, d, f = 4, 4, 6
    X, dY = rng.standard_normal((M, d)), rng.standard_normal((M, d))
    W1, W2 = rng.standard_normal((d, f)) * 0.5, rng.standard_normal((f, d)) * 0.5
    h = 1e-5
    EX = rng.standard_normal(X.shape)
    fd = (np.sum(oracle.mlp_block(X + h * EX, W1, W2, 2) * dY)
          - np.sum(oracle.mlp_block(X - h * EX, W1, W2, 2) * dY)) / (2 * h)
    Z = oracle.matmul(X, W1)
    gz = oracle.gelu_grad(Z)
    no_grad_factor = oracle.matmul(oracle.matmul(dY, W2.T), W1.T)
    one_shard_only = oracle.matmul(oracle.matmul(dY, W2[:3].T) * gz[:, :3], W1[:, :3].T)
    dX, _, _ = oracle.mlp_block_backward(X, W1, W2, dY, 2)
    assert abs(np.sum(dX * EX) - fd) < 1e-7 * max(1.0, abs(fd))
    assert abs(np.sum(no_grad_factor * EX) - fd) > 1e-3
    assert abs(np.sum(one_shard_only * EX) - fd) > 1e-3


# ----------------------------------------------- inputs (generator) --------

def test_generator_reproducible_and_shaped():
    a = inputs.bf16_normal((64, 48), inputs.stream_seed(0, 1), 0.02)
    b = inputs.bf16_normal((64, 48), inputs.stream_seed(0, 1), 0.02)
    np.testing.assert_array_equal(a, b)
    v = oracle.bf16_to_f64(a)
    assert abs(v.std() - 0.02) < 0.002 and abs(v.mean()) < 0.002
    ints = inputs.int_uniform((16, 32), inputs.stream_seed(0, 0))
    assert set(np.unique(ints)).issubset(set(range(-4, 5)))
    assert len(np.unique(ints)) == 9
    z = inputs.normal((200000,), 5)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1.0) < 0.01


# ------------------------------------------- planted mistakes are caught ---

def test_pins_catch_planted_mistakes(worked):
    """Feed the oracle the mistakes a wrong implementation would make and
    check that the worked-example pins reject each of them."""
    X, W, g = worked
    Y = np.array(g["Y"])
    # transposed operand: the 2x4 W read as its 4x2 transpose's layout
    Wt = W.T.reshape(2, 4)
    assert not np.array_equal(oracle.matmul(X, Wt), Y)
    # dropped shard in the row-split sum
    _, P = oracle.row_linear(X, W, 2)
    assert not np.array_equal(P[0], Y)
    # wrong row-split pairing: X_0 with W_1 (an index slip)
    assert not np.array_equal(X[:, :1] * W[1:2] + X[:, 1:] * W[0:1], Y)
    # swapped column shards in the concat
    _, Ys = oracle.column_linear(X, W, 2)
    assert not np.array_equal(np.concatenate([Ys[1], Ys[0]], axis=1), Y)
    # a sign error in GeLU's odd part would break x*Phi(x) at x=1
    assert abs(oracle.gelu([1.0])[0] - 0.8413447461) < 1e-9
    assert abs(0.5 * (1 - math.erf(1 / math.sqrt(2))) - 0.8413447461) > 0.1
