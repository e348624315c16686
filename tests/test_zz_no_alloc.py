"""tp_mlp_block_static_ws: the MLP block for callers that cannot allocate
device memory at call time (for example a serving loop that must not call
cudaMalloc once running, or a host that owns all device memory in its own
pool and passes the library only inputs and outputs).  Its scratch is a
fixed array inside the library, so it is checked here against the
caller-workspace entry point, on two calls in a row: the second call must
not be affected by what the first one left in the shared array.  Both entry
points run the same kernels in the same order on the same inputs, so their
outputs must agree bit for bit (and, like every MLP-block result, sit
within the accuracy bar of each other).

This file is collected last on purpose: if it fails, a run that stops at
the first failure has already run every other test.
"""
import numpy as np
import pytest

from helpers import assert_bf16_parity, bf16_dev_to_f64, dev_bits, to_dev_bf16
from tensor_sharded_linear_02_b300 import inputs

pytestmark = pytest.mark.gpu


def _case(tp, dev, M, d, f, n, seed):
    import torch
    xb = inputs.bf16_normal((M, d), inputs.stream_seed(seed, 0), 1.0)
    w1b = inputs.bf16_normal((d, f), inputs.stream_seed(seed, 1), 0.02)
    w2b = inputs.bf16_normal((f, d), inputs.stream_seed(seed, 2), 0.02)
    X, W1, W2 = (to_dev_bf16(b, dev) for b in (xb, w1b, w2b))
    ws = torch.empty(tp.tp_mlp_block_workspace_size(M, f, torch.bfloat16), dtype=torch.uint8,
                     device=dev)
    Y_ref = torch.empty(M, d, dtype=torch.bfloat16, device=dev)
    tp.tp_mlp_block(X, W1, W2, Y_ref, ws, n_shards=n)
    Y = torch.full((M, d), float("nan"), dtype=torch.bfloat16, device=dev)
    tp.tp_mlp_block_static_ws(X, W1, W2, Y, n_shards=n)
    assert tp.tp_get_device_status() == tp.TP_OK
    np.testing.assert_array_equal(dev_bits(Y), dev_bits(Y_ref))
    return bf16_dev_to_f64(Y), bf16_dev_to_f64(Y_ref)


def test_static_ws_matches_workspace_entry(cuda_device):
    from tensor_sharded_linear_02_b300 import binding as tp
    # first call: the MLP-block workload's shape (H = 16 MiB of the 32 MiB)
    got, ref = _case(tp, cuda_device, 2048, 1024, 4096, 2, seed=21)
    assert_bf16_parity(got, ref, "static scratch, call 1")
    # second call, other shape and inputs, reusing the array the first left
    got, ref = _case(tp, cuda_device, 300, 256, 768, 3, seed=22)
    assert_bf16_parity(got, ref, "static scratch, call 2")


def test_static_ws_rejects_oversize(cuda_device):
    import torch
    from tensor_sharded_linear_02_b300 import binding as tp
    M, d, f = 4096, 64, 4104  # H = 4096 * 4104 * 2 bytes > 32 MiB
    assert M * f * 2 > tp.TP_STATIC_WS_BYTES
    X = torch.zeros(M, d, dtype=torch.bfloat16, device=cuda_device)
    W1 = torch.zeros(d, f, dtype=torch.bfloat16, device=cuda_device)
    W2 = torch.zeros(f, d, dtype=torch.bfloat16, device=cuda_device)
    Y = torch.zeros(M, d, dtype=torch.bfloat16, device=cuda_device)
    with pytest.raises(tp.TPError) as e:
        tp.tp_mlp_block_static_ws(X, W1, W2, Y, n_shards=2)
    assert e.value.status == 6  # TP_ERR_WORKSPACE
    assert tp.tp_get_device_status() == tp.TP_OK
