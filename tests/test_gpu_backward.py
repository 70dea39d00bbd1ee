"""GPU parity of the float32 backward (gda_attn_bwd) against the float64
autograd oracle (oracle/ref_torch_grad.py) on the same seeded inputs.

Tolerance (tests/parity.py, assert_grad_close): |err| <= 1e-4 (|ref| +
rms_row(ref) + rms(ref)) for every element of the six gradients.
Small cases are compared on every element: several 16-row and 32-key tiles
with ragged tails, causal and full attention, every supported (d, dv),
group sizes 1, 2, 3 and 4, and the pre-norm output (GDA_FLAG_NO_NORM).  The
3:1 workload's sizes (B 4, L 2048, 12 signal / 4 noise heads, d 64, dv 128)
are compared on one whole group of heads, whose gradients the oracle computes
exactly from the group's slice of the inputs.
"""
import numpy as np
import pytest
import torch

import grouped_differential_attention_gb300 as gda
from grouped_differential_attention_gb300 import workloads as W
from oracle.ref_torch_grad import gda_backward
from parity import assert_grad_close

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
    grads = gda.gda_attn_bwd(q1, k1, q2, k2, v, lam, lam_init, dy, causal=causal, eps=eps, flags=flags)
    torch.cuda.synchronize()
    return [g.cpu() for g in grads]


def check(got, ref, what):
    for name, g, r in zip(NAMES, got, ref):
        assert torch.isfinite(g).all(), f"{what} {name}: non-finite values"
        assert_grad_close(g, r, f"{what} {name}")


SMALL = [
    # B, L, hs, hn, d, dv, causal
    (2, 77, 6, 2, 64, 128, True),
    (1, 150, 4, 1, 128, 256, True),
    (2, 50, 4, 4, 64, 64, False),
    (1, 129, 8, 2, 128, 128, False),
    (1, 200, 6, 3, 64, 256, True),
    (2, 33, 4, 2, 128, 64, True),
    (1, 77, 3, 1, 64, 128, True),      # odd B * L * h_s: workspace segments stay 16-byte aligned
]


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "B%d_L%d_h%d+%d_d%d_dv%d_%s" % (
    *s[:6], "causal" if s[6] else "full"))
def test_backward_matches_oracle(shape):
    B, L, hs, hn, d, dv, causal = shape
    inp = W.make_backward_inputs(W.DIFF_F32_L128, B=B, L=L, h_s=hs, h_n=hn, d=d, dv=dv,
                                 seed=300 + L + hs)
    got = run_bwd(inp, 0.7, causal)
    ref = gda_backward(*inp[:6], 0.7, inp[6], causal=causal)
    check(got, ref, str(shape))


def test_backward_single_key():
    """L = 1: each row sees one key, both softmax maps are the constant 1, so
    the exact query and key gradients are zero (their float32 values are the
    rounding residue of do . v - do . O, about 1e-8 here).  The pre-norm
    output is (1 - lambda) v, parallel to O2 = v, and the norm's gradient is
    orthogonal to its input up to eps, so dlambda = -do . O2 is itself a
    cancellation residue (2e-4 exactly, from terms of size ~10): it is held
    to 1e-4 absolute.  dv = (1 - lambda) do matches the oracle."""
    inp = W.make_backward_inputs(W.DIFF_F32_L128, B=2, L=1, h_s=3, h_n=1, d=64, dv=128, seed=40)
    got = run_bwd(inp, 0.7, causal=True)
    ref = gda_backward(*inp[:6], 0.7, inp[6], causal=True)
    for name, g, r in zip(NAMES[:4], got[:4], ref[:4]):
        assert float(r.abs().max()) == 0.0, name
        assert float(g.abs().max()) <= 1e-5, name
    assert_grad_close(got[4], ref[4], "L=1 dv")
    assert float((got[5].double() - ref[5]).abs().max()) <= 1e-4


def test_backward_pre_norm_output():
    inp = W.make_backward_inputs(W.DIFF_F32_L128, B=2, L=96, h_s=6, h_n=2, d=64, dv=128, seed=41)
    got = run_bwd(inp, 0.8, causal=True, flags=gda.GDA_FLAG_NO_NORM)
    ref = gda_backward(*inp[:6], 0.8, inp[6], causal=True, norm=False)
    check(got, ref, "no_norm")


def test_backward_norm_eps_and_lambda_init():
    inp = W.make_backward_inputs(W.DIFF_F32_L128, B=1, L=64, h_s=4, h_n=2, d=64, dv=64, seed=42)
    got = run_bwd(inp, 0.2, causal=True, eps=0.5)
    ref = gda_backward(*inp[:6], 0.2, inp[6], causal=True, eps=0.5)
    check(got, ref, "eps 0.5, lambda_init 0.2")


def test_backward_of_equal_maps_at_lambda_one():
    """q2 = q1, k2 = k1, h_n = h_s, lambda = 1, pre-norm output: the two maps
    cancel, so the value gradient is exactly zero and the noise projections'
    gradients are exactly the negated signal ones (both sides compute the
    same numbers in the same order); the signal gradients still match the
    oracle."""
    inp = list(W.make_backward_inputs(W.DIFF_F32_L128, B=1, L=80, h_s=4, h_n=4, d=64, dv=128, seed=43))
    inp[2], inp[3] = inp[0].clone(), inp[1].clone()
    inp[5] = torch.ones_like(inp[5])
    got = run_bwd(inp, 0.8, causal=True, flags=gda.GDA_FLAG_NO_NORM)
    ref = gda_backward(*inp[:6], 0.8, inp[6], causal=True, norm=False)
    assert torch.count_nonzero(got[4]) == 0
    assert torch.equal(got[2], -got[0])
    assert torch.equal(got[3], -got[1])
    check(got, ref, "equal maps")


def test_backward_is_deterministic():
    inp = W.make_backward_inputs(W.DIFF_F32_L128, B=2, L=100, h_s=6, h_n=2, d=64, dv=128, seed=44)
    a = run_bwd(inp, 0.7)
    b = run_bwd(inp, 0.7)
    for name, x, y in zip(NAMES, a, b):
        assert torch.equal(x, y), name


def test_backward_rejects_short_workspace():
    inp = [t.cuda() for t in W.make_backward_inputs(W.DIFF_F32_L128, B=1, L=32, h_s=2, h_n=1, d=64,
                                                        dv=64, seed=45)]
    need = gda.gda_attn_bwd_workspace_size(1, 32, 2, 64, 64)
    ws = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(gda.GDAError):
        gda.gda_attn_bwd(*inp[:6], 0.8, inp[6], workspace=ws)


def test_backward_full_size_one_group():
    """B 4, L 2048, h 12+4, d 64, dv 128 (the 3:1 workload's sizes, float32):
    every gradient of noise group 2 (signal heads 6, 7, 8) against the oracle
    run on that group's slice, one batch element at a time."""
    w = W.GDA3_PREFILL_L2048
    inp = W.make_backward_inputs(w, dtype="f32")
    got = run_bwd(inp, w.lambda_init, w.causal, w.eps)
    r = w.h_s // w.h_n
    g = 2
    sig = slice(g * r, (g + 1) * r)
    dlam = torch.zeros(r, dtype=torch.float64)
    for b in range(w.B):
        q1, k1, q2, k2, v, lam, dy = inp
        sl = (q1[b:b + 1, :, sig], k1[b:b + 1, :, sig], q2[b:b + 1, :, g:g + 1], k2[b:b + 1, :, g:g + 1],
              v[b:b + 1, :, sig], lam[sig])
        ref = gda_backward(*sl, w.lambda_init, dy[b:b + 1, :, sig], causal=w.causal, eps=w.eps)
        what = f"b{b} group {g}"
        assert_grad_close(got[0][b:b + 1, :, sig], ref[0], what + " dq_sig")
        assert_grad_close(got[1][b:b + 1, :, sig], ref[1], what + " dk_sig")
        assert_grad_close(got[2][b:b + 1, :, g:g + 1], ref[2], what + " dq_noise")
        assert_grad_close(got[3][b:b + 1, :, g:g + 1], ref[3], what + " dk_noise")
        assert_grad_close(got[4][b:b + 1, :, sig], ref[4], what + " dv")
        dlam += ref[5]
    assert_grad_close(got[5][sig], dlam, "dlambda group 2")
    for t in got:
        assert torch.isfinite(t).all()


def test_backward_lambda_zero_noise_gradients_vanish():
    inp = list(W.make_backward_inputs(W.DIFF_F32_L128, B=1, L=90, h_s=4, h_n=2, d=64, dv=128, seed=48))
    inp[5] = torch.zeros_like(inp[5])
    got = run_bwd(inp, 0.8)
    assert torch.count_nonzero(got[2]) == 0 and torch.count_nonzero(got[3]) == 0
    check(got, gda_backward(*inp[:6], 0.8, inp[6]), "lambda 0")


def test_backward_sharp_maps():
    inp = list(W.make_backward_inputs(W.DIFF_F32_L128, B=1, L=120, h_s=4, h_n=2, d=64, dv=128, seed=49))
    inp[0] = inp[0] * 4
    inp[2] = inp[2] * 4
    got = run_bwd(inp, 0.8)
    check(got, gda_backward(*inp[:6], 0.8, inp[6]), "sharp maps")
