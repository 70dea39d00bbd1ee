"""Every path with lambda outside [0, 1].

The differential map (softmax(Q1 K1^T/sqrt d) - lambda softmax(Q2 K2^T/sqrt d))
is defined for any real lambda; the re-parameterisation exp(.) - exp(.) +
lambda_init can leave [0, 1] in either direction.  Each kernel takes lambda as
a float32 per signal head, so nothing may clamp it.  Here the heads carry
lambda = -1 ... 2 (0 and 1 included) and every path is compared with the
float64 oracle.  Near lambda = 1 the two maps can nearly cancel, and the
tensor-core prefill, which rounds each map weight to bf16 before the value
product, then moves an output by up to 2^-8 times the sum of its absolute
terms: its bound here is 3e-3 + 2e-2 |ref| + 2^-7 mag (parity.py,
assert_bf16_mag_close).  Decode (float32 weights) keeps 3e-3 + 2e-2 |ref|,
float32 paths 1e-4 (|ref| + rms_row), bf16 gradients as in their backward
tests; the float32 gradients add 2^-20 mag because the lambda = 1 head's first
causal row has o = 0 exactly, which the norm's gradient amplifies by
(1 - lambda_init) / sqrt(eps).
"""
import pytest
import torch

import grouped_differential_attention_gb300 as gda
from grouped_differential_attention_gb300 import workloads as W
from oracle.ref_numpy import gda_magnitudes
from oracle.ref_torch_grad import gda_backward, gda_grad_magnitudes
from parity import (assert_bf16_close, assert_bf16_mag_close, assert_f32_close, assert_grad_bf16_close,
                    assert_grad_close)

pytestmark = pytest.mark.gpu

GRADS = ("dq_sig", "dk_sig", "dq_noise", "dk_noise", "dv", "dlambda")


@pytest.fixture(scope="module", autouse=True)
def device_error_word_stays_clear():
    from grouped_differential_attention_gb300 import build
    build.build()
    gda.gda_device_error(clear=True)
    yield
    assert gda.gda_device_error(clear=True) == 0


def wide_lambda(h_s):
    """Per-head lambda spread over [-1, 2], with 0 and 1 among them when h_s % 3 == 1."""
    return torch.linspace(-1.0, 2.0, h_s, dtype=torch.float32)


@pytest.mark.parametrize("d,dv,single_pass", [(64, 128, False), (128, 256, False), (128, 256, True)])
def test_prefill_bf16_wide_lambda(oracle_mod, d, dv, single_pass):
    q1, k1, q2, k2, v, _ = W.make_prefill_inputs(W.GDA3_PREFILL_L2048, B=2, L=259, h_s=7, h_n=1,
                                                 d=d, dv=dv, seed=71)
    lam = wide_lambda(7)
    inp = (q1, k1, q2, k2, v, lam)
    flags = gda.GDA_FLAG_SINGLE_PASS if single_pass else 0
    got = gda.gda_attn_fwd(*[t.cuda() for t in inp], 0.8, flags=flags)
    torch.cuda.synchronize()
    mag = gda_magnitudes(*[t.double() for t in inp], 0.8)
    assert_bf16_mag_close(got.cpu(), oracle_mod.prefill(*inp, 0.8), mag, "lambda in [-1, 2]")


def test_prefill_2pass_wide_lambda_no_norm(oracle_mod):
    q1, k1, q2, k2, v, _ = W.make_prefill_inputs(W.GDA3_PREFILL_L2048, B=1, L=300, h_s=4, h_n=2,
                                                 seed=72)
    inp = (q1, k1, q2, k2, v, wide_lambda(4))
    got = gda.gda_attn_fwd_2pass(*[t.cuda() for t in inp], 0.8, flags=gda.GDA_FLAG_NO_NORM)
    torch.cuda.synchronize()
    mag = gda_magnitudes(*[t.double() for t in inp], 0.8, norm=False)
    assert_bf16_mag_close(got.cpu(), oracle_mod.prefill(*inp, 0.8, norm=False), mag, "pre-norm, lambda in [-1, 2]")


def test_prefill_f32_wide_lambda(oracle_mod):
    q1, k1, q2, k2, v, _ = W.make_prefill_inputs(W.DIFF_F32_L128, B=1, L=150, h_s=4, h_n=4, seed=73)
    inp = (q1, k1, q2, k2, v, wide_lambda(4))
    got = gda.gda_attn_fwd_f32(*[t.cuda() for t in inp], 0.8)
    torch.cuda.synchronize()
    assert_f32_close(got.cpu(), oracle_mod.prefill(*inp, 0.8), "float32, lambda in [-1, 2]")


def test_decode_wide_lambda(oracle_mod):
    q1, q2, k1c, k2c, vc, lens, _ = W.make_decode_inputs(W.GDA3_DECODE_B64, B=5, Lcap=700, h_s=7, h_n=1,
                                                         seed=74, len_range=(1, 700))
    inp = (q1, q2, k1c, k2c, vc, lens, wide_lambda(7))
    got = gda.gda_attn_decode(*[t.cuda() for t in inp], 0.8)
    torch.cuda.synchronize()
    assert_bf16_close(got.cpu(), oracle_mod.decode(*inp, 0.8), "decode, lambda in [-1, 2]")


def test_backward_bf16_wide_lambda():
    q1, k1, q2, k2, v, _, dy = W.make_backward_inputs(W.GDA3_PREFILL_L2048, B=1, L=200, h_s=4, h_n=1,
                                                      seed=75)
    inp = (q1, k1, q2, k2, v, wide_lambda(4), dy)
    got = gda.gda_attn_bwd_bf16(*[t.cuda() for t in inp[:6]], 0.8, inp[6].cuda())
    torch.cuda.synchronize()
    f64 = [t.to(torch.float64) for t in inp]
    ref = gda_backward(*f64[:6], 0.8, f64[6])
    mag = gda_grad_magnitudes(*f64[:6], 0.8, f64[6])
    for name, g, r, m in zip(GRADS, got, ref, mag):
        assert_grad_bf16_close(g.cpu(), r, m, "bf16 backward, lambda in [-1, 2] " + name)


def test_backward_f32_wide_lambda():
    q1, k1, q2, k2, v, _, dy = W.make_backward_inputs(W.DIFF_F32_L128, B=1, L=90, h_s=4, h_n=2, seed=76)
    inp = (q1, k1, q2, k2, v, wide_lambda(4), dy)
    got = gda.gda_attn_bwd(*[t.cuda() for t in inp[:6]], 0.8, inp[6].cuda())
    torch.cuda.synchronize()
    f64 = [t.to(torch.float64) for t in inp]
    ref = gda_backward(*f64[:6], 0.8, f64[6])
    mag = gda_grad_magnitudes(*f64[:6], 0.8, f64[6])   # row 0 of the lambda = 1 head has o = 0
    for name, g, r, m in zip(GRADS, got, ref, mag):
        assert_grad_close(g.cpu(), r, "float32 backward, lambda in [-1, 2] " + name, mag=m)
