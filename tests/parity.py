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


GRAD_F32_MAG = 2.0 ** -20


def assert_grad_close(got, ref, what="", mag=None):
    """float32 gradients: |got - ref| <= 1e-4 (|ref| + rms_row(ref) + rms(ref)).

    Rows are the last axis (a head's d or dv values).  The tensor-wide rms
    term covers rows whose exact gradient is zero (the first causal query
    row has a single visible key, so its query gradient vanishes).  Every
    gradient is a sum of at most L products of float32 factors; measured on
    the CPU, float32 autograd of the same forward stays within 1.1e-5 of the
    float64 result in these units, so the bound leaves a 9x margin for the
    kernels' other summation orders.  1-D tensors (dlambda) use the rms of
    the whole vector as their row.

    With ``mag`` (the oracle's sum of absolute terms, as for the bf16
    gradients) the bound adds 2^-20 mag, sixteen float32 units of that sum.
    It is needed where a row's output vanishes (lambda = 1 on a causal row
    that sees one key: o = 0 exactly): the norm then scales that row's do by
    (1 - lambda_init) / sqrt(eps), and gradients whose exact value is 0 keep
    the float32 residue of two summation orders of the same dot product
    (measured 2^-27 mag on the GPU).
    """
    got, ref = _np(got), _np(ref)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    rms_all = np.sqrt(np.mean(ref * ref)) if ref.size else 0.0
    rms = np.sqrt(np.mean(ref * ref, axis=-1, keepdims=True))
    bound = GRAD_REL * (np.abs(ref) + rms + rms_all)
    if mag is not None:
        mag = _np(mag)
        assert mag.shape == ref.shape, (mag.shape, ref.shape)
        bound = bound + GRAD_F32_MAG * mag
    err = np.abs(got - ref)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.unravel_index(np.argmax(np.where(bad, err / bound, 0)), err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements outside 1e-4(|ref|+rms_row+rms)"
            f"{' + 2^-20 mag' if mag is not None else ''}; "
            f"worst at {idx}: got {got[idx]!r} ref {ref[idx]!r}")



BF16_MAG = 2.0 ** -7


def assert_bf16_mag_close(got, ref, mag, what=""):
    """bf16 output where the two maps may cancel (lambda near 1):
    |got - ref| <= 3e-3 + 2e-2 |ref| + 2^-7 mag, mag = the oracle's sum of
    absolute terms (oracle.ref_numpy.gda_magnitudes).

    The tensor-core prefill rounds every map weight P to bf16 (relative error
    at most 2^-8) before the value product, so an output element can move by
    up to 2^-8 mag; when o is much smaller than its terms that exceeds the
    elementwise bound.  A float64 replay of that rounding on the CPU (24 cases
    with lambda from -1 to 2, groups of 1 to 7, d = 64 / 128) puts every
    element within 0.75 x 2^-8 mag and within 0.24 of this bound; the plain
    bound fails there for up to 51 elements per case, all at lambda = 1."""
    got, ref, mag = _np(got), _np(ref), _np(mag)
    assert got.shape == ref.shape == mag.shape, (got.shape, ref.shape, mag.shape)
    bound = BF16_ATOL + BF16_RTOL * np.abs(ref) + BF16_MAG * mag
    err = np.abs(got - ref)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.unravel_index(np.argmax(np.where(bad, err / bound, 0)), err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements outside 3e-3 + 2e-2|ref| + 2^-7 mag; "
            f"worst at {idx}: got {got[idx]!r} ref {ref[idx]!r} mag {mag[idx]!r}")

GRAD_BF16_REL = 2e-2
GRAD_BF16_MAG = 2.0 ** -7


def assert_grad_bf16_close(got, ref, mag, what=""):
    """Tensor-core gradients from bf16 operands:
    |got - ref| <= 2e-2 (|ref| + rms_row(ref) + rms(ref)) + 2^-7 mag,
    mag = the oracle's sum of absolute terms of that gradient
    (oracle.ref_torch_grad.gda_grad_magnitudes).

    The kernels round P of the first pass, the norm's input gradient do and the
    score gradients (W = A1 - lambda A2, dS1, dS2) to bf16 (relative error
    at most 2^-8 each).  Two kinds of error follow, and a float64 replay of exactly
    those roundings on the CPU (41 ragged cases, groups of 1 to 4, L up to
    512, causal and full; the replay reproduces the kernel's values to the
    bit where checked) shows both:
    - errors that scale with the output: the rounding of O1 and O2 reaches do
      through o = O1 - lambda O2 and the norm; at most 1.2e-2 (|ref| +
      rms_row + rms) for dv and 1.9e-2 elsewhere;
    - errors that scale with the terms of a cancelling sum: in early causal
      rows a gradient is a short sum of score gradients that add to ~0; there
      the error stays below 0.46 x 2^-8 x mag.
    The sum of the two bounds holds every replayed element with a margin of
    at least 2x on its dominant term."""
    got, ref, mag = _np(got), _np(ref), _np(mag)
    assert got.shape == ref.shape == mag.shape, (got.shape, ref.shape, mag.shape)
    rms_all = np.sqrt(np.mean(ref * ref)) if ref.size else 0.0
    rms = np.sqrt(np.mean(ref * ref, axis=-1, keepdims=True))
    bound = GRAD_BF16_REL * (np.abs(ref) + rms + rms_all) + GRAD_BF16_MAG * mag
    err = np.abs(got - ref)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.unravel_index(np.argmax(np.where(bad, err / bound, 0)), err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements outside 2e-2(|ref|+rms_row+rms) + 2^-7 mag; "
            f"worst at {idx}: got {got[idx]!r} ref {ref[idx]!r} mag {mag[idx]!r}")
