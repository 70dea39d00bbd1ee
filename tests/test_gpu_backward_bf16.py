"""GPU parity of the tensor-core backward (gda_attn_bwd_bf16) against the
float64 autograd oracle (oracle/ref_torch_grad.py) on the same seeded bf16
inputs.

Tolerance (tests/parity.py, assert_grad_bf16_close), every element of the six
gradients: |err| <= 2e-2 (|ref| + rms_row(ref) + rms(ref)) + 2^-7 mag, where
mag is the oracle's sum of the absolute values of the gradient's terms.  Small cases
span several 128-row and 64-row tiles with ragged tails, L = 1, causal and
full attention, groups of 1 to 4; the 3:1 workload's sizes (B 4, L 2048,
12 signal / 4 noise heads, d 64, dv 128) are compared on one whole head
group.
"""
import pytest
import torch

import grouped_differential_attention_gb300 as gda
from grouped_differential_attention_gb300 import workloads as W
from oracle.ref_torch_grad import gda_backward, gda_grad_magnitudes
from parity import assert_grad_bf16_close

pytestmark = pytest.mark.gpu

NAMES = ("dq_sig", "dk_sig", "dq_noise", "dk_noise", "dv", "dlambda")


@pytest.fixture(scope="module", autouse=True)
def device_error_word_stays_clear():
    from grouped_differential_attention_gb300 import build
    build.build()
    gda.gda_device_error(clear=True)
    yield
    assert gda.gda_device_error(clear=True) == 0


def run_bwd(inputs, lam_init, causal=True, eps=1e-5, flags=0):
    q1, k1, q2, k2, v, lam, dy = [t.cuda() for t in inputs]
    grads = gda.gda_attn_bwd_bf16(q1, k1, q2, k2, v, lam, lam_init, dy, causal=causal, eps=eps, flags=flags)
    torch.cuda.synchronize()
    return [g.cpu() for g in grads]


def oracle_grads(inputs, lam_init, causal=True, eps=1e-5, norm=True):
    """(gradients, magnitudes) of the float64 oracle on the bf16 inputs' values."""
    f64 = [t.to(torch.float64) for t in inputs]
    return (gda_backward(*f64[:6], lam_init, f64[6], causal=causal, eps=eps, norm=norm),
            gda_grad_magnitudes(*f64[:6], lam_init, f64[6], causal=causal, eps=eps, norm=norm))


def check(got, oracle, what):
    ref, mag = oracle
    for name, g, r, m in zip(NAMES, got, ref, mag):
        assert torch.isfinite(g).all(), f"{what} {name}: non-finite values"
        assert_grad_bf16_close(g, r, m, f"{what} {name}")


SMALL = [
    # B, L, hs, hn, causal
    (2, 150, 6, 2, True),
    (1, 300, 3, 1, True),
    (2, 100, 4, 4, False),
    (1, 257, 12, 4, True),
    (2, 77, 6, 3, True),
    (1, 130, 4, 2, False),
    (1, 64, 2, 1, True),
]


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "B%d_L%d_h%d+%d_%s" % (*s[:4], "causal" if s[4] else "full"))
def test_bf16_backward_matches_oracle(shape):
    B, L, hs, hn, causal = shape
    inp = W.make_backward_inputs(W.GDA3_PREFILL_L2048, B=B, L=L, h_s=hs, h_n=hn, seed=500 + L + hs)
    got = run_bwd(inp, 0.8, causal)
    check(got, oracle_grads(inp, 0.8, causal), str(shape))


def test_bf16_backward_single_key():
    """L = 1: exact q/k gradients are 0 (one visible key); dv = (1 - lambda) do."""
    inp = W.make_backward_inputs(W.GDA3_PREFILL_L2048, B=2, L=1, h_s=3, h_n=1, seed=40)
    got = run_bwd(inp, 0.7)
    ref, mag = oracle_grads(inp, 0.7)
    for g in got[:4]:
        assert float(g.abs().max()) <= 1e-3
    assert_grad_bf16_close(got[4], ref[4], mag[4], "L=1 dv")


def test_bf16_backward_pre_norm_output():
    inp = W.make_backward_inputs(W.GDA3_PREFILL_L2048, B=2, L=96, h_s=6, h_n=2, seed=41)
    got = run_bwd(inp, 0.8, flags=gda.GDA_FLAG_NO_NORM)
    check(got, oracle_grads(inp, 0.8, norm=False), "no_norm")


def test_bf16_backward_of_equal_maps_at_lambda_one():
    """q2 = q1, k2 = k1, h_n = h_s, lambda = 1, pre-norm output: W = 0 exactly, so
    dv is exactly 0, and the noise gradients are the exact negatives of the
    signal ones (bit-identical statistics and products on both sides)."""
    inp = list(W.make_backward_inputs(W.GDA3_PREFILL_L2048, B=1, L=200, h_s=4, h_n=4, seed=43))
    inp[2], inp[3] = inp[0].clone(), inp[1].clone()
    inp[5] = torch.ones_like(inp[5])
    got = run_bwd(inp, 0.8, flags=gda.GDA_FLAG_NO_NORM)
    assert torch.count_nonzero(got[4]) == 0
    assert torch.equal(got[2], -got[0])
    assert torch.equal(got[3], -got[1])
    check(got, oracle_grads(inp, 0.8, norm=False), "equal maps")


def test_bf16_backward_is_deterministic():
    inp = W.make_backward_inputs(W.GDA3_PREFILL_L2048, B=2, L=300, h_s=6, h_n=2, seed=44)
    a = run_bwd(inp, 0.7)
    b = run_bwd(inp, 0.7)
    for name, x, y in zip(NAMES, a, b):
        assert torch.equal(x, y), name


def test_bf16_backward_agrees_with_float32_backward():
    """The float32 CUDA-core backward on the same (bf16-valued) inputs is
    accurate to 1e-4; the two differ by no more than the bf16 bound."""
    inp = W.make_backward_inputs(W.GDA3_PREFILL_L2048, B=1, L=180, h_s=6, h_n=2, seed=45)
    got = run_bwd(inp, 0.8)
    f32 = [t.float().cuda() for t in inp]
    ref = gda.gda_attn_bwd(*f32[:6], 0.8, f32[6])
    torch.cuda.synchronize()
    _, mag = oracle_grads(inp, 0.8)
    check(got, ([r.cpu().double() for r in ref], mag), "vs float32 backward")


def test_bf16_backward_full_size_one_group():
    """B 4, L 2048, h 12+4, d 64, dv 128: every gradient of noise group 1
    (signal heads 3, 4, 5) against the oracle on that group's slice."""
    w = W.GDA3_PREFILL_L2048
    inp = W.make_backward_inputs(w)
    got = run_bwd(inp, w.lambda_init, w.causal, w.eps)
    r = w.h_s // w.h_n
    g = 1
    sig = slice(g * r, (g + 1) * r)
    dlam = torch.zeros(r, dtype=torch.float64)
    q1, k1, q2, k2, v, lam, dy = inp
    for b in range(w.B):
        sl = [q1[b:b + 1, :, sig], k1[b:b + 1, :, sig], q2[b:b + 1, :, g:g + 1], k2[b:b + 1, :, g:g + 1],
              v[b:b + 1, :, sig], lam[sig], dy[b:b + 1, :, sig]]
        ref, mag = oracle_grads(sl, w.lambda_init, w.causal, w.eps)
        what = f"b{b} group {g}"
        assert_grad_bf16_close(got[0][b:b + 1, :, sig], ref[0], mag[0], what + " dq_sig")
        assert_grad_bf16_close(got[1][b:b + 1, :, sig], ref[1], mag[1], what + " dk_sig")
        assert_grad_bf16_close(got[2][b:b + 1, :, g:g + 1], ref[2], mag[2], what + " dq_noise")
        assert_grad_bf16_close(got[3][b:b + 1, :, g:g + 1], ref[3], mag[3], what + " dk_noise")
        assert_grad_bf16_close(got[4][b:b + 1, :, sig], ref[4], mag[4], what + " dv")
        dlam += ref[5]
        dmag = mag[5] if b == 0 else dmag + mag[5]
    assert_grad_bf16_close(got[5][sig], dlam, dmag, "dlambda group 1")
    for t in got:
        assert torch.isfinite(t).all()


def test_bf16_backward_lambda_zero_noise_gradients_vanish():
    """lambda = 0: the noise map does not reach the output, so the noise
    projections' gradients are exactly 0; dlambda = -sum do . O2 is not."""
    inp = list(W.make_backward_inputs(W.GDA3_PREFILL_L2048, B=1, L=150, h_s=6, h_n=2, seed=46))
    inp[5] = torch.zeros_like(inp[5])
    got = run_bwd(inp, 0.8)
    assert torch.count_nonzero(got[2]) == 0 and torch.count_nonzero(got[3]) == 0
    check(got, oracle_grads(inp, 0.8), "lambda 0")


def test_bf16_backward_sharp_maps():
    """Queries scaled by 4 (exact in bf16): logits up to ~30 / sqrt(d) units,
    nearly one-hot rows, which exercises the saved statistics' range."""
    inp = list(W.make_backward_inputs(W.GDA3_PREFILL_L2048, B=1, L=200, h_s=6, h_n=2, seed=47))
    inp[0] = inp[0] * 4
    inp[2] = inp[2] * 4
    got = run_bwd(inp, 0.8)
    check(got, oracle_grads(inp, 0.8), "sharp maps")
