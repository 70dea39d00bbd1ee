"""GPU parity of the chunked prefill (queries continuing a cached prefix).

A chunk of L query rows over Lk keys is, by definition, the last L rows of
the prefill over an Lk-row sequence; the oracle evaluates exactly those rows
(oracle.prefill_rows on full-length queries whose last L rows are the
chunk's).  bf16 output: |err| <= 3e-3 + 2e-2|ref|.
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


def chunk_case(B, L, Lk, hs, hn, d, dv, seed):
    q1, k1, q2, k2, v, lam = W.make_prefill_inputs(W.GDA3_PREFILL_L2048, B=B, L=Lk, h_s=hs, h_n=hn, d=d, dv=dv,
                                                   seed=seed)
    return (q1, k1, q2, k2, v, lam)


@pytest.mark.parametrize("shape", [  # B, L, Lk, h_s, h_n, d, dv, causal
    (1, 128, 1000, 12, 4, 64, 128, True),
    (2, 77, 300, 6, 2, 64, 128, True),
    (1, 1, 513, 3, 1, 64, 128, True),
    (2, 200, 200, 4, 2, 128, 256, True),
    (1, 64, 130, 4, 4, 64, 128, False),
    (1, 300, 2048, 8, 2, 128, 128, True),
    # more than 28 key tiles per item: the grouped kernel's per-row output stores instead of
    # the staged (TMA) epilogue, with items of two signal heads and of one
    (4, 640, 4200, 8, 2, 64, 128, True),
    (1, 100, 4500, 3, 1, 64, 128, True),
])
def test_chunked_prefill_matches_oracle(oracle_mod, shape):
    B, L, Lk, hs, hn, d, dv, causal = shape
    full = chunk_case(B, L, Lk, hs, hn, d, dv, seed=L * 3 + Lk)
    q1, k1, q2, k2, v, lam = full
    rows = list(range(Lk - L, Lk))
    chunk = (q1[:, Lk - L:], k1, q2[:, Lk - L:], k2, v, lam)
    got = gda.gda_attn_fwd_chunk(*(t.contiguous().cuda() for t in chunk), 0.8, causal=causal)
    torch.cuda.synchronize()
    ref = oracle_mod.prefill_rows(q1, k1, q2, k2, v, lam, 0.8, rows, causal=causal)
    assert_bf16_close(got.cpu(), ref, str(shape))


def test_prefill_in_chunks_equals_whole_prefill():
    q1, k1, q2, k2, v, lam = (t.cuda() for t in chunk_case(2, 600, 600, 12, 4, 64, 128, seed=17))
    whole = gda.gda_attn_fwd(q1, k1, q2, k2, v, lam, 0.8)
    parts = []
    for a, b in ((0, 256), (256, 512), (512, 600)):
        parts.append(gda.gda_attn_fwd_chunk(q1[:, a:b].contiguous(), k1[:, :b].contiguous(),
                                            q2[:, a:b].contiguous(), k2[:, :b].contiguous(),
                                            v[:, :b].contiguous(), lam, 0.8))
    torch.cuda.synchronize()
    assert_bf16_close(torch.cat(parts, dim=1).cpu(), whole.cpu().double().numpy(), "chunks vs whole")


@pytest.mark.parametrize("two_pass", [True, False], ids=["two_pass", "single_pass"])
@pytest.mark.parametrize("shape", [  # B, L, Lk, h_s, h_n, d, dv, causal
    (1, 100, 700, 4, 1, 64, 256, True),
    (1, 130, 500, 4, 2, 128, 256, False),
    (2, 1, 257, 4, 2, 128, 256, True),
    (2, 77, 300, 6, 2, 64, 128, True),
])
def test_chunked_prefill_both_kernels(oracle_mod, shape, two_pass):
    """gda_attn_fwd_chunk_2pass (two-pass kernels, caller workspace) and
    gda_attn_fwd_chunk (single pass, no workspace) both match the oracle."""
    B, L, Lk, hs, hn, d, dv, causal = shape
    q1, k1, q2, k2, v, lam = chunk_case(B, L, Lk, hs, hn, d, dv, seed=L * 5 + Lk)
    chunk = (q1[:, Lk - L:], k1, q2[:, Lk - L:], k2, v, lam)
    got = gda.gda_attn_fwd_chunk(*(t.contiguous().cuda() for t in chunk), 0.8, causal=causal, two_pass=two_pass)
    torch.cuda.synchronize()
    ref = oracle_mod.prefill_rows(q1, k1, q2, k2, v, lam, 0.8, list(range(Lk - L, Lk)), causal=causal)
    assert_bf16_close(got.cpu(), ref, str(shape))
