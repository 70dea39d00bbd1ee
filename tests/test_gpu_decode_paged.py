"""GPU parity of the paged-cache decode.

Contiguous caches are scattered into page pools under a seeded random page
permutation (workloads.page_caches); the oracle runs the decode definition
on the contiguous caches.  bf16 output: |err| <= 3e-3 + 2e-2|ref|.
"""
import pytest
import torch

import grouped_differential_attention_gb300 as gda
from grouped_differential_attention_gb300 import workloads as W
from parity import assert_bf16_close

pytestmark = pytest.mark.gpu


def paged_case(B, Lcap, hs, hn, d, dv, page_size, seed):
    q1, q2, k1c, k2c, vc, lens, lam = W.make_decode_inputs(
        W.GDA3_DECODE_B64, B=B, Lcap=Lcap, h_s=hs, h_n=hn, d=d, dv=dv, seed=seed, len_range=(1, Lcap))
    lens[0] = 1
    lens[-1] = Lcap
    pools = W.page_caches(k1c, k2c, vc, page_size, seed=seed)
    return (q1, q2, k1c, k2c, vc, lens, lam), pools


def run_paged(contig, pools, lam_init=0.8):
    q1, q2, _, _, _, lens, lam = contig
    k1p, k2p, vp, table = pools
    out = gda.gda_attn_decode_paged(*(t.cuda() for t in (q1, q2, k1p, k2p, vp, table, lens, lam)), lam_init)
    torch.cuda.synchronize()
    return out.cpu()


@pytest.mark.parametrize("shape", [  # B, Lcap, h_s, h_n, d, dv, page_size
    (3, 64, 12, 4, 64, 128, 16),
    (5, 1000, 6, 2, 128, 256, 8),
    (2, 777, 4, 4, 64, 64, 7),
    (4, 2048, 12, 4, 64, 128, 64),
    (70, 64, 3, 1, 64, 128, 1),
    (2, 384, 16, 4, 128, 256, 128),
])
def test_paged_decode_matches_oracle(oracle_mod, shape):
    B, Lcap, hs, hn, d, dv, ps = shape
    Lcap = (Lcap + ps - 1) // ps * ps
    contig, pools = paged_case(B, Lcap, hs, hn, d, dv, ps, seed=B * 13 + Lcap + ps)
    ref = oracle_mod.decode(*contig, 0.8)
    assert_bf16_close(run_paged(contig, pools), ref, str(shape))
    assert gda.gda_device_error(clear=True) == 0


def test_paged_decode_equals_contiguous_decode():
    contig, pools = paged_case(8, 4096, 12, 4, 64, 128, 64, seed=91)
    got = run_paged(contig, pools)
    ref = gda.gda_attn_decode(*(t.cuda() for t in contig), 0.8)
    torch.cuda.synchronize()
    assert_bf16_close(got, ref.cpu().double().numpy(), "paged vs contiguous")


def test_paged_decode_reports_page_ids_outside_the_pool():
    contig, pools = paged_case(2, 256, 6, 2, 64, 128, 32, seed=5)
    k1p, k2p, vp, table = pools
    gda.gda_device_error(clear=True)
    bad = table.clone()
    bad[1, 0] = k1p.shape[0]          # one past the pool: read as page 0 and reported
    out = run_paged(contig, (k1p, k2p, vp, bad))
    assert torch.isfinite(out.float()).all()
    assert gda.gda_device_error(clear=True) & gda.GDA_DEVERR_BAD_PAGE
