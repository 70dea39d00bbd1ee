"""GPU parity of the split-KV decode against the float64 oracle.

bf16 caches, float32 accumulation: |err| <= 3e-3 + 2e-2|ref| elementwise on
every output of the 64-sequence decode workload, plus edge lengths (1 and
Lcap), wide head sets and consistency with the causal prefill's last row.
"""
import pytest
import torch

import grouped_differential_attention_gb300 as gda
from grouped_differential_attention_gb300 import workloads as W
from parity import assert_bf16_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def device_error_word_stays_clear():
    from grouped_differential_attention_gb300 import build
    build.build()
    gda.gda_device_error(clear=True)
    yield
    assert gda.gda_device_error(clear=True) == 0


def run_decode(inputs, lam_init, eps=1e-5):
    q1, q2, k1c, k2c, vc, lens, lam = (t.cuda() for t in inputs)
    out = gda.gda_attn_decode(q1, q2, k1c, k2c, vc, lens, lam, lam_init, eps=eps)
    torch.cuda.synchronize()
    return out.cpu()


def test_decode_workload_all_outputs(oracle_mod):
    w = W.GDA3_DECODE_B64
    inp = W.make_decode_inputs(w)
    got = run_decode(inp, w.lambda_init, w.eps)
    ref = oracle_mod.decode(*inp, w.lambda_init, eps=w.eps)
    assert_bf16_close(got, ref, w.name)


@pytest.mark.parametrize("shape", [  # B, Lcap, h_s, h_n, d, dv
    (3, 40, 12, 4, 64, 128),
    (5, 1000, 6, 2, 128, 256),
    (2, 777, 4, 4, 64, 64),
    (2, 300, 16, 4, 128, 256),     # 832 chunks per row: wide variant
    (70, 64, 3, 1, 64, 128),
])
def test_decode_shapes_and_edge_lengths(oracle_mod, shape):
    B, Lcap, hs, hn, d, dv = shape
    inp = W.make_decode_inputs(W.GDA3_DECODE_B64, B=B, Lcap=Lcap, h_s=hs, h_n=hn, d=d, dv=dv,
                               seed=B * 31 + Lcap, len_range=(1, Lcap))
    lens = inp[5]
    lens[0] = 1
    lens[-1] = Lcap
    got = run_decode(inp, 0.8)
    ref = oracle_mod.decode(*inp, 0.8)
    assert_bf16_close(got, ref, str(shape))


def test_decode_equals_last_prefill_row(oracle_mod):
    """Decoding token n-1 over a cache of n rows = row n-1 of the causal prefill."""
    B, n, hs, hn, d, dv = 1, 515, 6, 2, 64, 128
    q1, k1, q2, k2, v, lam = W.make_prefill_inputs(W.GDA3_PREFILL_L2048, B=B, L=n, h_s=hs,
                                                   h_n=hn, d=d, dv=dv, seed=21)
    pre = gda.gda_attn_fwd(*(t.cuda() for t in (q1, k1, q2, k2, v, lam)), 0.8)
    dec = gda.gda_attn_decode(q1[:, n - 1].cuda(), q2[:, n - 1].cuda(), k1.cuda(), k2.cuda(),
                              v.cuda(), torch.tensor([n], dtype=torch.int32, device="cuda"),
                              lam.cuda(), 0.8)
    torch.cuda.synchronize()
    ref = oracle_mod.prefill_rows(q1, k1, q2, k2, v, lam, 0.8, [n - 1])[:, 0]
    assert_bf16_close(dec.cpu(), ref, "decode")
    assert_bf16_close(pre[:, n - 1].cpu(), ref, "prefill last row")


def test_decode_reuses_its_workspace():
    w = W.GDA3_DECODE_B64
    inp = W.make_decode_inputs(w, B=8, Lcap=512, len_range=(100, 512), seed=4)
    q1, q2, k1c, k2c, vc, lens, lam = (t.cuda() for t in inp)
    ws = torch.full((gda.gda_attn_decode_workspace_size(8, 512, 12, 4, 128),), 255,
                    dtype=torch.uint8, device="cuda")
    a = gda.gda_attn_decode(q1, q2, k1c, k2c, vc, lens, lam, 0.8, workspace=ws).clone()
    b = gda.gda_attn_decode(q1, q2, k1c, k2c, vc, lens, lam, 0.8, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
