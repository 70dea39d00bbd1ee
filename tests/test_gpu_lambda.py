"""GPU parity of the lambda re-parameterisation against the float64 oracle.

lambda_h = exp(lq1_h . lk1_h) - exp(lq2_h . lk2_h) + lambda_init ("Differential
Attention in Large Language Models ...", section "Learnable Lambda
Re-parameterization").  The kernel forms float32 dot products (fused
multiply-adds over d, then a warp shuffle sum) and calls expf; with |x| <= 2
and d <= 256 the dot products are off by a few float32 ulps of sum |terms|
and expf by <= 2 ulps, so |err| <= 1e-5 (1 + |ref|) holds with margin.
"""
import math

import numpy as np
import pytest
import torch

import grouped_differential_attention_gb300 as gda
from grouped_differential_attention_gb300 import workloads as W
from parity import assert_bf16_close

pytestmark = pytest.mark.gpu


def vectors(hs, d, scale, seed):
    g = torch.Generator().manual_seed(seed)
    return [scale * torch.randn(hs, d, generator=g) for _ in range(4)]


@pytest.mark.parametrize("hs,d,scale", [(12, 64, 0.1), (24, 64, 0.1), (16, 128, 0.05), (1, 1, 0.7),
                                        (5, 33, 0.2), (300, 256, 0.08)])
def test_lambda_reparam_matches_oracle(oracle_mod, hs, d, scale):
    vecs = vectors(hs, d, scale, seed=hs * 7 + d)
    lam_init = oracle_mod.lambda_init_schedule(3)
    got = gda.gda_lambda_reparam(*(t.cuda() for t in vecs), lam_init)
    torch.cuda.synchronize()
    ref = oracle_mod.lambda_reparam(*(t.numpy() for t in vecs), lam_init)
    err = np.abs(got.cpu().double().numpy() - ref)
    assert np.all(err <= 1e-5 * (1 + np.abs(ref))), err.max()


def test_lambda_reparam_zero_vectors_give_lambda_init_exactly():
    z = torch.zeros(12, 64, device="cuda")
    got = gda.gda_lambda_reparam(z, z, z, z, 0.375)
    assert torch.all(got == 0.375)


def test_device_lambda_feeds_the_prefill(oracle_mod):
    """lambda produced on the device drives the prefill without a host copy."""
    inp = W.make_prefill_inputs(W.GDA3_PREFILL_L2048, B=1, L=150, h_s=6, h_n=2, seed=31)
    vecs = vectors(6, 64, 0.1, seed=5)
    # a deep layer's constant, as in the workloads: the bf16 bound's absolute
    # term assumes outputs scaled by 1 - lambda_init <= 0.27 (see the design
    # notes on the bf16 tolerance)
    lam_init = 0.8
    lam_dev = gda.gda_lambda_reparam(*(t.cuda() for t in vecs), lam_init)
    out = gda.gda_attn_fwd(*(t.cuda() for t in inp[:5]), lam_dev, lam_init)
    torch.cuda.synchronize()
    lam_ref = oracle_mod.lambda_reparam(*(t.numpy() for t in vecs), lam_init)
    lam_got = lam_dev.cpu()
    assert np.all(np.abs(lam_got.double().numpy() - lam_ref) <= 1e-5 * (1 + np.abs(lam_ref)))
    # the oracle takes the same float32 lambda values the kernel saw
    ref = oracle_mod.prefill(*inp[:5], lam_got, lam_init)
    assert_bf16_close(out.cpu(), ref, "prefill with the device lambda")
