"""GPU parity of the fp8-cache decode against the float64 dense decode.

The caches hold e4m3 codes with a float32 scale per head; the oracle
dequantises them exactly (codes widened to float64 times the scale) and runs
the decode definition in float64.  bf16 output: |err| <= 3e-3 + 2e-2|ref|.
"""
import numpy as np
import pytest
import torch

import grouped_differential_attention_gb300 as gda
from grouped_differential_attention_gb300 import workloads as W
from oracle.ref_numpy import gda_decode_dense
from parity import assert_bf16_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def device_error_word_stays_clear():
    from grouped_differential_attention_gb300 import build
    build.build()
    gda.gda_device_error(clear=True)
    yield
    assert gda.gda_device_error(clear=True) == 0


def oracle_fp8(inp, lam_init, eps=1e-5):
    q1, q2, k1q, k2q, vq, k1s, k2s, vs, lens, lam = inp
    f64 = lambda t: t.to(torch.float64).numpy()
    return gda_decode_dense(f64(q1), f64(q2), f64(k1q), f64(k2q), f64(vq), lens.numpy(), lam.numpy(),
                            lam_init, eps=eps, k1_scale=k1s.numpy(), k2_scale=k2s.numpy(),
                            v_scale=vs.numpy())


def run_fp8(inp, lam_init, eps=1e-5):
    out = gda.gda_attn_decode_fp8(*(t.cuda() for t in inp), lam_init, eps=eps)
    torch.cuda.synchronize()
    return out.cpu()


@pytest.mark.parametrize("shape", [  # B, Lcap, h_s, h_n, d, dv
    (3, 40, 12, 4, 64, 128),
    (5, 1000, 6, 2, 128, 256),
    (2, 777, 4, 4, 64, 64),
    (2, 300, 16, 4, 128, 256),
    (70, 64, 3, 1, 64, 128),
    (4, 2049, 12, 4, 64, 128),
])
def test_fp8_decode_shapes_and_edge_lengths(shape):
    B, Lcap, hs, hn, d, dv = shape
    inp = W.make_decode_inputs_fp8(W.GDA3_DECODE_B64, B=B, Lcap=Lcap, h_s=hs, h_n=hn, d=d, dv=dv,
                                   seed=B * 37 + Lcap, len_range=(1, Lcap))
    lens = inp[8]
    lens[0] = 1
    lens[-1] = Lcap
    assert_bf16_close(run_fp8(inp, 0.8), oracle_fp8(inp, 0.8), str(shape))


def test_fp8_decode_full_size_workload():
    w = W.GDA3_DECODE_B64
    inp = W.make_decode_inputs_fp8(w)
    assert_bf16_close(run_fp8(inp, w.lambda_init, w.eps), oracle_fp8(inp, w.lambda_init, w.eps), w.name)


def test_fp8_cache_of_representable_values_matches_bf16_decode():
    """Caches whose values are e4m3 codes times 1: the fp8 and bf16 decodes see the same numbers."""
    q1, q2, k1q, k2q, vq, k1s, k2s, vs, lens, lam = W.make_decode_inputs_fp8(
        W.GDA3_DECODE_B64, B=6, Lcap=900, len_range=(1, 900), seed=77)
    ones = [torch.ones_like(t) for t in (k1s, k2s, vs)]
    got = run_fp8((q1, q2, k1q, k2q, vq, *ones, lens, lam), 0.8)
    bf = [t.to(torch.float32).to(torch.bfloat16) for t in (k1q, k2q, vq)]   # exact: e4m3 fits bf16
    ref = gda.gda_attn_decode(*(t.cuda() for t in (q1, q2, *bf, lens, lam)), 0.8)
    torch.cuda.synchronize()
    assert_bf16_close(got, ref.cpu().double().numpy(), "fp8 vs bf16 decode")


def run_paged_fp8(inp, page_size, seed, lam_init=0.8):
    q1, q2, k1q, k2q, vq, k1s, k2s, vs, lens, lam = inp
    k1p, k2p, vp, table = W.page_caches(k1q, k2q, vq, page_size, seed=seed)
    out = gda.gda_attn_decode_paged_fp8(*(t.cuda() for t in (q1, q2, k1p, k2p, vp, k1s, k2s, vs, table, lens, lam)),
                                        lam_init)
    torch.cuda.synchronize()
    return out.cpu()


@pytest.mark.parametrize("shape", [  # B, Lcap, h_s, h_n, d, dv, page_size
    (3, 64, 12, 4, 64, 128, 16),
    (5, 1000, 6, 2, 128, 256, 8),
    (2, 777, 4, 4, 64, 64, 7),
    (70, 64, 3, 1, 64, 128, 1),
])
def test_paged_fp8_decode_matches_oracle(shape):
    """Paged pools of e4m3 codes (seeded random page order) with per-head
    scales: both serving variants at once, against the float64 dense decode
    of the same codes and scales."""
    B, Lcap, hs, hn, d, dv, ps = shape
    Lcap = (Lcap + ps - 1) // ps * ps
    inp = W.make_decode_inputs_fp8(W.GDA3_DECODE_B64, B=B, Lcap=Lcap, h_s=hs, h_n=hn, d=d, dv=dv,
                                   seed=B * 41 + Lcap + ps, len_range=(1, Lcap))
    inp[8][0] = 1
    inp[8][-1] = Lcap
    assert_bf16_close(run_paged_fp8(inp, ps, seed=ps), oracle_fp8(inp, 0.8), str(shape))


def test_paged_fp8_decode_equals_contiguous_fp8_decode():
    """Same positions, same partition over the CTAs, same arithmetic: the
    paged result equals the contiguous one bit for bit."""
    inp = W.make_decode_inputs_fp8(W.GDA3_DECODE_B64, B=8, Lcap=4096, seed=93, len_range=(1, 4096))
    assert torch.equal(run_paged_fp8(inp, 64, seed=7), run_fp8(inp, 0.8))
