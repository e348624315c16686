"""Shared test helpers: moving generator output to the device and back, and
the accuracy bar for bf16 results.

Accuracy bar (bf16 inputs, fp32 accumulation, compared with the fp64
oracle on the same input bytes):
    relative Frobenius error  ||got - ref||_F / ||ref||_F  <= 5e-3
    elementwise |got - ref|  <= 2e-2 * RMS(ref) + u * |ref|
where u is the unit roundoff of the output format: 2^-8 for a bf16 output
(8 significant bits: half the spacing of bf16 values in [1, 2) is 2^-8),
0 for an fp32 output.  The 2e-2 * RMS term bounds the accumulated error of
the fp32 result; a bf16 output then rounds each element to nearest, which
by itself can move it by half an ulp (up to 2^-8 |y|) -- more than
2e-2 * RMS whenever |y| exceeds about 5 RMS, as in the positive tail of a
GeLU output.  Tests that have both outputs also check that the bf16 output
is exactly the round-to-nearest-even of the fp32 one.
Integer-valued fp32 inputs must match exactly.
"""
import numpy as np

import oracle

REL_FRO_TOL = 5e-3
MAX_ERR_RMS_TOL = 2e-2


def to_dev_bf16(bits, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def to_dev_f32(a, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


def bf16_dev_to_f64(t):
    import torch
    return oracle.bf16_to_f64(t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def dev_to_f64(t):
    import torch
    if t.dtype == torch.bfloat16:
        return bf16_dev_to_f64(t)
    return t.detach().cpu().double().numpy()


def dev_bits(t):
    """Raw bit patterns of a device tensor (for bit-exact comparisons)."""
    import torch
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().copy()
    return t.view(torch.int32).numpy().copy()


def errors(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    nref = np.linalg.norm(ref)
    rel = np.linalg.norm(got - ref) / nref if nref > 0 else np.linalg.norm(got - ref)
    rms = np.sqrt(np.mean(ref ** 2)) if ref.size else 0.0
    mx = np.max(np.abs(got - ref)) if ref.size else 0.0
    return rel, mx, rms


BF16_UNIT_ROUNDOFF = 2.0 ** -8


def assert_bf16_parity(got, ref, what="", out_bf16=True):
    """Check a result of bf16 inputs with fp32 accumulation against the fp64
    oracle (see the module docstring for the bar)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rel, mx, rms = errors(got, ref)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert rel <= REL_FRO_TOL, f"{what}: relative Frobenius error {rel:.3e} > {REL_FRO_TOL}"
    u = BF16_UNIT_ROUNDOFF if out_bf16 else 0.0
    excess = np.abs(got - ref) - (MAX_ERR_RMS_TOL * rms + u * np.abs(ref))
    worst = int(np.argmax(excess)) if excess.size else 0
    assert excess.size == 0 or excess.flat[worst] <= 0, (
        f"{what}: |err| {abs(got.flat[worst] - ref.flat[worst]):.3e} at ref {ref.flat[worst]:.4e} "
        f"exceeds {MAX_ERR_RMS_TOL} * RMS {rms:.3e} + {u:.2e} * |ref|")
    return rel, mx, rms
