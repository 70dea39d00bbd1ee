"""Tolerances of the GPU-vs-oracle comparisons.

bf16 I/O with float32 accumulation: |got - ref| <= 3e-3 + 2e-2 |ref|,
elementwise.  float32 path: |got - ref| <= 1e-4 (|ref| + rms_row(ref)), the
row RMS taken over the head's dv values (a pure relative bound is undefined
at the zero crossings of the output).
"""
import numpy as np

BF16_ATOL = 3e-3
BF16_RTOL = 2e-2
F32_REL = 1e-4


def _np(x):
    if hasattr(x, "detach"):
        x = x.detach().float().cpu().numpy()
    return np.asarray(x, dtype=np.float64)


def bf16_worst(got, ref):
    got, ref = _np(got), _np(ref)
    bound = BF16_ATOL + BF16_RTOL * np.abs(ref)
    ratio = np.abs(got - ref) / bound
    ratio = np.where(np.isfinite(got), ratio, np.inf)
    return float(ratio.max()) if ratio.size else 0.0


def assert_bf16_close(got, ref, what=""):
    got, ref = _np(got), _np(ref)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    bound = BF16_ATOL + BF16_RTOL * np.abs(ref)
    err = np.abs(got - ref)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.unravel_index(np.argmax(np.where(bad, err / bound, 0)), err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements outside 3e-3 + 2e-2|ref|; "
            f"worst at {idx}: got {got[idx]!r} ref {ref[idx]!r}")


def assert_f32_close(got, ref, what=""):
    got, ref = _np(got), _np(ref)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    rms = np.sqrt(np.mean(ref * ref, axis=-1, keepdims=True))
    bound = F32_REL * (np.abs(ref) + rms)
    err = np.abs(got - ref)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.unravel_index(np.argmax(np.where(bad, err / bound, 0)), err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements outside 1e-4(|ref|+rms_row); "
            f"worst at {idx}: got {got[idx]!r} ref {ref[idx]!r}")


GRAD_REL = 1e-4


def assert_grad_close(got, ref, what=""):
    """float32 gradients: |got - ref| <= 1e-4 (|ref| + rms_row(ref) + rms(ref)).

    Rows are the last axis (a head's d or dv values).  The tensor-wide rms
    term covers rows whose exact gradient is zero (the first causal query
    row has a single visible key, so its query gradient vanishes).  Every
    gradient is a sum of at most L products of float32 factors; measured on
    the CPU, float32 autograd of the same forward stays within 1.1e-5 of the
    float64 result in these units, so the bound leaves a 9x margin for the
    kernels' other summation orders.  1-D tensors (dlambda) use the rms of
    the whole vector as their row.
    """
    got, ref = _np(got), _np(ref)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    rms_all = np.sqrt(np.mean(ref * ref)) if ref.size else 0.0
    rms = np.sqrt(np.mean(ref * ref, axis=-1, keepdims=True))
    bound = GRAD_REL * (np.abs(ref) + rms + rms_all)
    err = np.abs(got - ref)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.unravel_index(np.argmax(np.where(bad, err / bound, 0)), err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements outside 1e-4(|ref|+rms_row+rms); "
            f"worst at {idx}: got {got[idx]!r} ref {ref[idx]!r}")


GRAD_BF16_REL = 3e-2


def assert_grad_bf16_close(got, ref, what=""):
    """Tensor-core gradients from bf16 operands:
    |got - ref| <= 3e-2 (|ref| + rms_row(ref) + rms(ref)).

    The kernels round the norm's input gradient and the score gradients
    (W = A1 - lambda A2, dS1, dS2) to bf16 as tensor-core operands.  A float64
    replay of exactly those roundings on the CPU (ragged shapes, groups of 1
    to 4, L up to 512, causal and full) stays within 1.2e-2 of the float64
    gradients in these units, so the bound leaves a 2.5x margin for float32
    accumulation and the kernels' exponentials."""
    got, ref = _np(got), _np(ref)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    rms_all = np.sqrt(np.mean(ref * ref)) if ref.size else 0.0
    rms = np.sqrt(np.mean(ref * ref, axis=-1, keepdims=True))
    bound = GRAD_BF16_REL * (np.abs(ref) + rms + rms_all)
    err = np.abs(got - ref)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.unravel_index(np.argmax(np.where(bad, err / bound, 0)), err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements outside 3e-2(|ref|+rms_row+rms); "
            f"worst at {idx}: got {got[idx]!r} ref {ref[idx]!r}")
