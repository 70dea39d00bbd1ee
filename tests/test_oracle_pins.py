"""Pins of the float64 oracle against things other than itself.

Each test ties the oracle to a library routine (PyTorch float64
scaled-dot-product attention, ``rms_norm``), a closed form, an exact
invariant, a value printed on the pages, or an independent brute force.
Together they make a dropped term, a wrong sign, a wrong group index, a
wrong softmax scale, a transposed operand or a wrong mask fail somewhere.

Sources: "Differential Attention in Large Language Models ..." (sections
"The Mechanics of Attention Noise", "Differential Attention Architecture",
"Learnable Lambda Re-parameterization", "Headwise Normalization") and the
"Grouped Differential Attention" abstract.
"""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from grouped_differential_attention_gb300 import workloads
from oracle import ref_numpy

HERE = os.path.dirname(os.path.abspath(__file__))


def case(B, L, hs, hn, d, dv, seed=0, dtype="f32", lam_range=(0.2, 0.8)):
    return workloads.make_prefill_inputs(
        workloads.DIFF_F32_L128, B=B, L=L, h_s=hs, h_n=hn, d=d, dv=dv, seed=seed,
        dtype=dtype, lam_range=lam_range)


def sdpa64(q, k, v, causal):
    """Library attention in float64; tensors are [B, L, H, D]."""
    out = F.scaled_dot_product_attention(
        q.double().permute(0, 2, 1, 3), k.double().permute(0, 2, 1, 3),
        v.double().permute(0, 2, 1, 3), is_causal=causal)
    return out.permute(0, 2, 1, 3).numpy()


SHAPES = [  # B, L, hs, hn, d, dv
    (1, 1, 2, 2, 8, 16),
    (2, 7, 2, 1, 8, 16),
    (1, 19, 6, 2, 16, 32),
    (2, 33, 4, 4, 16, 32),
    (1, 40, 8, 2, 32, 64),
    (1, 24, 12, 4, 64, 128),
]


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("shape", SHAPES)
def test_lambda_zero_is_library_attention(oracle_mod, shape, causal):
    """lambda = 0 leaves the signal map alone: softmax(Q1 K1^T / sqrt d) V."""
    q1, k1, q2, k2, v, lam = case(*shape)
    got = oracle_mod.prefill(q1, k1, q2, k2, v, torch.zeros_like(lam), 0.8,
                             causal=causal, norm=False)
    np.testing.assert_allclose(got, sdpa64(q1, k1, v, causal), rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("shape", SHAPES)
def test_difference_of_two_library_attentions(oracle_mod, shape, causal):
    """Pre-norm output = SDPA(Q1,K1,V) - lambda_h SDPA(Q2_rep, K2_rep, V).

    Q2/K2 repeated r times along heads (repeat_interleave) is grouped-query
    sharing written out explicitly; this pins the group index g = h // r,
    the per-head lambda, the 1/sqrt(d) scale and the mask of both maps.
    """
    B, L, hs, hn, d, dv = shape
    q1, k1, q2, k2, v, lam = case(*shape, seed=3)
    r = hs // hn
    a = sdpa64(q1, k1, v, causal)
    b = sdpa64(q2.repeat_interleave(r, dim=2), k2.repeat_interleave(r, dim=2), v, causal)
    want = a - lam.double().numpy()[None, None, :, None] * b
    got = oracle_mod.prefill(q1, k1, q2, k2, v, lam, 0.8, causal=causal, norm=False)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


@pytest.mark.parametrize("eps", [1e-5, 1e-2])
def test_norm_is_library_rms_norm(oracle_mod, eps):
    """Epilogue = (1 - lambda_init) * rms_norm(o) with no gain, eps inside the root."""
    q1, k1, q2, k2, v, lam = case(2, 21, 6, 3, 16, 48, seed=5)
    lam_init = 0.37
    pre = oracle_mod.prefill(q1, k1, q2, k2, v, lam, lam_init, eps=eps, norm=False)
    got = oracle_mod.prefill(q1, k1, q2, k2, v, lam, lam_init, eps=eps, norm=True)
    want = (1 - lam_init) * F.rms_norm(torch.from_numpy(pre), (pre.shape[-1],), eps=eps)
    np.testing.assert_allclose(got, want.numpy(), rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("causal", [True, False])
def test_equal_maps_and_unit_lambda_cancel(oracle_mod, causal):
    """Q2 = Q1, K2 = K1, h_s = h_n and lambda = 1: the difference map is exactly 0."""
    q1, k1, _, _, v, lam = case(2, 30, 4, 4, 16, 32, seed=7)
    ones = torch.ones_like(lam)
    got = oracle_mod.prefill(q1, k1, q1, k1, v, ones, 0.8, causal=causal, norm=False)
    assert np.all(got == 0.0)
    # and a lambda != 1 leaves (1 - lambda) times plain attention
    got = oracle_mod.prefill(q1, k1, q1, k1, v, 0.25 * ones, 0.8, causal=causal, norm=False)
    np.testing.assert_allclose(got, 0.75 * sdpa64(q1, k1, v, causal), rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [True, False])
def test_rows_of_each_map_sum_to_one(oracle_mod, causal):
    """V = 1: every softmax row sums to 1, so the difference map rows sum to 1 - lambda_h.

    Pre-norm output is 1 - lambda_h everywhere; with the norm on it is the
    closed form (1 - lambda_init)(1 - lambda_h) / sqrt((1 - lambda_h)^2 + eps).
    """
    q1, k1, q2, k2, v, lam = case(1, 45, 6, 2, 16, 32, seed=9)
    v = torch.ones_like(v)
    lam_init, eps = 0.8, 1e-5
    pre = oracle_mod.prefill(q1, k1, q2, k2, v, lam, lam_init, causal=causal, norm=False)
    lam64 = lam.double().numpy()
    np.testing.assert_allclose(pre, np.broadcast_to((1 - lam64)[None, None, :, None], pre.shape),
                               rtol=0, atol=1e-14)
    post = oracle_mod.prefill(q1, k1, q2, k2, v, lam, lam_init, causal=causal, norm=True)
    closed = (1 - lam_init) * (1 - lam64) / np.sqrt((1 - lam64) ** 2 + eps)
    np.testing.assert_allclose(post, np.broadcast_to(closed[None, None, :, None], post.shape),
                               rtol=1e-14, atol=1e-14)



@pytest.mark.parametrize("causal", [True, False])
def test_lambda_outside_unit_interval(oracle_mod, causal):
    """lambda = -1 ... 2 (0 and 1 included): nothing in the definition clamps it.

    Pre-norm output = SDPA(Q1,K1,V) - lambda_h SDPA(Q2_rep,K2_rep,V) as above,
    and with V = 1 the norm's closed form holds for these lambda too.  At
    lambda = 1 the closed form is 0 while the pre-norm value is the float64
    residue of 1 - sum(p2) (a few ulp times L), which the norm scales by up
    to (1 - lambda_init) / sqrt(eps) ~ 63: hence the 1e-12 absolute slack."""
    hs, hn = 7, 1
    q1, k1, q2, k2, v, _ = case(2, 23, hs, hn, 16, 32, seed=19)
    lam = torch.linspace(-1.0, 2.0, hs)
    lam64 = lam.double().numpy()
    a = sdpa64(q1, k1, v, causal)
    b = sdpa64(q2.repeat_interleave(hs // hn, dim=2), k2.repeat_interleave(hs // hn, dim=2), v, causal)
    got = oracle_mod.prefill(q1, k1, q2, k2, v, lam, 0.8, causal=causal, norm=False)
    np.testing.assert_allclose(got, a - lam64[None, None, :, None] * b, rtol=0, atol=1e-12)
    post = oracle_mod.prefill(q1, k1, q2, k2, torch.ones_like(v), lam, 0.8, causal=causal)
    closed = 0.2 * (1 - lam64) / np.sqrt((1 - lam64) ** 2 + 1e-5)
    np.testing.assert_allclose(post, np.broadcast_to(closed[None, None, :, None], post.shape),
                               rtol=1e-14, atol=1e-12)


@pytest.mark.parametrize("causal", [True, False])
def test_magnitudes_are_library_attention_of_absolute_values(causal):
    """Pre-norm magnitudes = SDPA(Q1, K1, |V|) + |lambda_h| SDPA(Q2_rep, K2_rep, |V|):
    pins the maps, the group map and the absolute values of lambda and V."""
    hs, hn = 6, 2
    q1, k1, q2, k2, v, _ = case(2, 19, hs, hn, 16, 32, seed=25)
    lam = torch.linspace(-1.0, 2.0, hs)
    r = hs // hn
    want = (sdpa64(q1, k1, v.abs(), causal) + np.abs(lam.double().numpy())[None, None, :, None]
            * sdpa64(q2.repeat_interleave(r, dim=2), k2.repeat_interleave(r, dim=2), v.abs(), causal))
    got = ref_numpy.gda_magnitudes(q1, k1, q2, k2, v, lam, 0.8, causal=causal, norm=False)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def test_magnitudes_equal_the_output_when_terms_share_a_sign(oracle_mod):
    """lambda <= 0 and V >= 0: every term (a1 - lambda a2) v is >= 0, so the
    sum of absolute terms is the output itself, with and without the norm."""
    q1, k1, q2, k2, v, _ = case(1, 23, 4, 2, 16, 32, seed=27)
    v = v.abs()
    lam = torch.tensor([0.0, -0.3, -1.0, -2.5])
    for norm in (False, True):
        out = oracle_mod.prefill(q1, k1, q2, k2, v, lam, 0.8, norm=norm)
        mag = ref_numpy.gda_magnitudes(q1, k1, q2, k2, v, lam, 0.8, norm=norm)
        np.testing.assert_allclose(mag, out, rtol=1e-12, atol=1e-14)


def test_magnitudes_bound_the_output(oracle_mod):
    q1, k1, q2, k2, v, _ = case(2, 31, 7, 1, 16, 32, seed=29)
    lam = torch.linspace(-1.0, 2.0, 7)
    for norm in (False, True):
        out = oracle_mod.prefill(q1, k1, q2, k2, v, lam, 0.8, norm=norm)
        mag = ref_numpy.gda_magnitudes(q1, k1, q2, k2, v, lam, 0.8, norm=norm)
        assert np.all(np.abs(out) <= mag + 1e-12)

def test_first_row_under_causal_mask(oracle_mod):
    """Row 0 sees only key 0: y0 = (1-li)(1-lam) v0 / sqrt(mean(((1-lam) v0)^2) + eps)."""
    q1, k1, q2, k2, v, lam = case(2, 17, 6, 3, 16, 32, seed=11)
    lam_init, eps = 0.6, 1e-5
    got = oracle_mod.prefill(q1, k1, q2, k2, v, lam, lam_init, causal=True, eps=eps)[:, 0]
    v0 = v[:, 0].double().numpy()                            # [B, hs, dv]
    o0 = (1 - lam.double().numpy())[None, :, None] * v0
    want = (1 - lam_init) * o0 / np.sqrt(np.mean(o0 ** 2, axis=-1, keepdims=True) + eps)
    np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("norm", [True, False])
@pytest.mark.parametrize("hn", [1, 2])
@pytest.mark.parametrize("r", [1, 2, 3, 4])
@pytest.mark.parametrize("L", [1, 5, 16])
def test_loop_oracle_matches_dense_matrices(oracle_mod, L, r, hn, norm, causal):
    """The C loop oracle and the NumPy dense-matrix oracle agree to 1e-12."""
    hs = r * hn
    q1, k1, q2, k2, v, lam = case(2, L, hs, hn, 8, 16, seed=L * 100 + r * 10 + hn)
    got = oracle_mod.prefill(q1, k1, q2, k2, v, lam, 0.7, causal=causal, norm=norm)
    want = ref_numpy.gda_dense(q1.numpy(), k1.numpy(), q2.numpy(), k2.numpy(), v.numpy(),
                               lam.numpy(), 0.7, causal=causal, norm=norm)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_pins_notice_a_wrong_group_map(oracle_mod):
    """Interleaved groups (h % h_n) instead of contiguous ones fail the repetition pin."""
    B, L, hs, hn, d, dv = 1, 12, 6, 2, 8, 16
    q1, k1, q2, k2, v, lam = case(B, L, hs, hn, d, dv, seed=13)
    r = hs // hn
    want = sdpa64(q1, k1, v, True) - lam.double().numpy()[None, None, :, None] * sdpa64(
        q2.repeat_interleave(r, dim=2), k2.repeat_interleave(r, dim=2), v, True)
    good = ref_numpy.gda_dense(q1.numpy(), k1.numpy(), q2.numpy(), k2.numpy(), v.numpy(),
                               lam.numpy(), 0.8, norm=False)
    bad = ref_numpy.gda_dense(q1.numpy(), k1.numpy(), q2.numpy(), k2.numpy(), v.numpy(),
                              lam.numpy(), 0.8, norm=False, group_of=np.arange(hs) % hn)
    np.testing.assert_allclose(good, want, rtol=0, atol=1e-12)
    assert np.max(np.abs(bad - want)) > 1e-3


def test_bf16_inputs_are_used_exactly(oracle_mod):
    q1, k1, q2, k2, v, lam = case(1, 9, 4, 2, 16, 32, seed=15, dtype="bf16")
    a = oracle_mod.prefill(q1, k1, q2, k2, v, lam, 0.8)
    b = oracle_mod.prefill(q1.float(), k1.float(), q2.float(), k2.float(), v.float(), lam, 0.8)
    assert np.array_equal(a, b)


def test_sampled_rows_equal_full_rows(oracle_mod):
    q1, k1, q2, k2, v, lam = case(2, 50, 6, 2, 16, 32, seed=17)
    rows = [0, 1, 13, 49, 49, 7]
    full = oracle_mod.prefill(q1, k1, q2, k2, v, lam, 0.8)
    part = oracle_mod.prefill_rows(q1, k1, q2, k2, v, lam, 0.8, rows)
    assert np.array_equal(part, full[:, rows])


def _decode_case(B, Lcap, hs, hn, d, dv, seed):
    w = workloads.GDA3_DECODE_B64
    return workloads.make_decode_inputs(w, B=B, Lcap=Lcap, h_s=hs, h_n=hn, d=d, dv=dv,
                                        seed=seed, len_range=(1, Lcap))


@pytest.mark.parametrize("hs,hn", [(6, 2), (4, 4), (3, 1)])
def test_decode_is_last_causal_row(oracle_mod, hs, hn):
    """Decoding with the new token already in the cache equals prefill row len-1."""
    B, Lcap, d, dv = 5, 23, 16, 32
    q1, q2, k1c, k2c, vc, lens, lam = _decode_case(B, Lcap, hs, hn, d, dv, seed=hs * 7 + hn)
    lens[0], lens[1] = 1, Lcap
    got = oracle_mod.decode(q1, q2, k1c, k2c, vc, lens, lam, 0.8)
    for b in range(B):
        n = int(lens[b])
        # place the decode query at row n-1 of a prefill over the first n cache rows
        q1p = torch.zeros(1, n, hs, d, dtype=q1.dtype)
        q2p = torch.zeros(1, n, hn, d, dtype=q2.dtype)
        q1p[0, n - 1], q2p[0, n - 1] = q1[b], q2[b]
        want = oracle_mod.prefill_rows(q1p, k1c[b:b + 1, :n], q2p, k2c[b:b + 1, :n],
                                       vc[b:b + 1, :n], lam, 0.8, [n - 1])
        np.testing.assert_allclose(got[b], want[0, 0], rtol=0, atol=1e-13)


def test_decode_is_difference_of_library_attentions(oracle_mod):
    B, Lcap, hs, hn, d, dv = 3, 31, 6, 2, 16, 32
    q1, q2, k1c, k2c, vc, lens, lam = _decode_case(B, Lcap, hs, hn, d, dv, seed=21)
    r = hs // hn
    got = oracle_mod.decode(q1, q2, k1c, k2c, vc, lens, lam, 0.8, norm=False)
    for b in range(B):
        n = int(lens[b])
        a = sdpa64(q1[b:b + 1, None], k1c[b:b + 1, :n], vc[b:b + 1, :n], False)[0, 0]
        c = sdpa64(q2[b:b + 1, None].repeat_interleave(r, dim=2),
                   k2c[b:b + 1, :n].repeat_interleave(r, dim=2), vc[b:b + 1, :n], False)[0, 0]
        want = a - lam.double().numpy()[:, None] * c
        np.testing.assert_allclose(got[b], want, rtol=0, atol=1e-12)


def _golden_lambda_init():
    rows = []
    with open(os.path.join(HERE, "golden", "lambda_init_schedule.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                layer, value = line.split()
                rows.append((layer, float(value)))
    return rows


def test_lambda_init_schedule_matches_page(oracle_mod):
    for layer, value in _golden_lambda_init():
        if layer == "inf":
            assert abs(oracle_mod.lambda_init_schedule(10_000) - value) < 1e-12
        else:
            assert abs(oracle_mod.lambda_init_schedule(int(layer)) - value) < 1e-15
    # the layer-8 constant used by the 3:1 prefill workload
    assert abs(oracle_mod.lambda_init_schedule(8) - workloads.LAMBDA_INIT_LAYER8) < 1e-15
    assert abs(workloads.LAMBDA_INIT_LAYER8 - 0.8 + 0.6 * math.exp(-2.1)) < 1e-15


def test_oracle_rejects_bad_shapes(oracle_mod):
    q1, k1, q2, k2, v, lam = case(1, 4, 6, 4, 8, 16)   # 6 % 4 != 0
    with pytest.raises(ValueError):
        oracle_mod.prefill(q1, k1, q2, k2, v, lam, 0.8)


# ------------------------------------------------------------ lambda reparam
# "Differential Attention in Large Language Models ...", section "Learnable
# Lambda Re-parameterization": lambda = exp(lq1.lk1) - exp(lq2.lk2) + lambda_init.

def test_lambda_reparam_zero_vectors_give_lambda_init(oracle_mod):
    z = np.zeros((5, 64))
    got = oracle_mod.lambda_reparam(z, z, z, z, 0.37)
    assert np.all(got == 0.37)


def test_lambda_reparam_equal_branches_cancel_exactly(oracle_mod):
    g = np.random.default_rng(3)
    a, b = g.normal(size=(4, 32)), g.normal(size=(4, 32))
    got = oracle_mod.lambda_reparam(a, b, a, b, 0.8)
    assert np.all(got == 0.8)


def test_lambda_reparam_single_component_closed_form(oracle_mod):
    # one nonzero coordinate per vector: the dot products are plain products
    d = 16
    lq1, lk1, lq2, lk2 = (np.zeros((3, d)) for _ in range(4))
    vals = [(0.5, -0.25, 0.1, 0.3), (1.0, 1.0, 0.0, 2.0), (-0.2, 0.7, 0.4, -0.9)]
    for h, (a, b, c, e) in enumerate(vals):
        lq1[h, h] = a
        lk1[h, h] = b
        lq2[h, d - 1 - h] = c
        lk2[h, d - 1 - h] = e
    got = oracle_mod.lambda_reparam(lq1, lk1, lq2, lk2, 0.2)
    want = [math.exp(a * b) - math.exp(c * e) + 0.2 for (a, b, c, e) in vals]
    assert np.allclose(got, want, rtol=0, atol=1e-15)


def test_lambda_reparam_swapping_branches_mirrors_around_lambda_init(oracle_mod):
    g = np.random.default_rng(4)
    v = [g.normal(scale=0.3, size=(6, 64)) for _ in range(4)]
    fwd = oracle_mod.lambda_reparam(v[0], v[1], v[2], v[3], 0.5)
    rev = oracle_mod.lambda_reparam(v[2], v[3], v[0], v[1], 0.5)
    assert np.allclose((fwd - 0.5) + (rev - 0.5), 0.0, atol=1e-14)
    # one head through an explicit loop over the dimension
    h = 2
    a = sum(v[0][h, i] * v[1][h, i] for i in range(64))
    b = sum(v[2][h, i] * v[3][h, i] for i in range(64))
    assert abs(fwd[h] - (math.exp(a) - math.exp(b) + 0.5)) < 1e-13


# ------------------------------------------------------ dense float64 decode
def test_dense_decode_matches_c_oracle(oracle_mod):
    """The NumPy decode (used for scaled / quantised caches) agrees with the pinned C decode."""
    g = torch.Generator().manual_seed(21)
    B, Lcap, hs, hn, d, dv = 3, 40, 6, 2, 16, 32
    q1, q2 = torch.randn(B, hs, d, generator=g), torch.randn(B, hn, d, generator=g)
    k1, k2 = torch.randn(B, Lcap, hs, d, generator=g), torch.randn(B, Lcap, hn, d, generator=g)
    v = torch.randn(B, Lcap, hs, dv, generator=g)
    lens = torch.tensor([1, 17, 40], dtype=torch.int32)
    lam = torch.rand(hs, generator=g)
    ref = oracle_mod.decode(q1, q2, k1, k2, v, lens, lam, 0.8)
    got = ref_numpy.gda_decode_dense(q1, q2, k1, k2, v, lens, lam, 0.8)
    assert np.allclose(got, ref, rtol=0, atol=1e-12)


def test_dense_decode_scales_equal_prescaled_caches(oracle_mod):
    """Per-head scales multiply the cached values: same as scaling the caches first."""
    g = torch.Generator().manual_seed(22)
    B, Lcap, hs, hn, d, dv = 2, 24, 4, 2, 8, 16
    q1, q2 = torch.randn(B, hs, d, generator=g), torch.randn(B, hn, d, generator=g)
    k1, k2 = torch.randn(B, Lcap, hs, d, generator=g), torch.randn(B, Lcap, hn, d, generator=g)
    v = torch.randn(B, Lcap, hs, dv, generator=g)
    lens = torch.tensor([24, 9], dtype=torch.int32)
    lam = torch.rand(hs, generator=g)
    s1, s2, sv = torch.rand(hs, generator=g) + 0.5, torch.rand(hn, generator=g) + 0.5, torch.rand(hs, generator=g) + 0.5
    got = ref_numpy.gda_decode_dense(q1, q2, k1, k2, v, lens, lam, 0.8, k1_scale=s1, k2_scale=s2, v_scale=sv)
    k1s = k1.double() * s1.double()[None, None, :, None]
    k2s = k2.double() * s2.double()[None, None, :, None]
    vs = v.double() * sv.double()[None, None, :, None]
    want = ref_numpy.gda_decode_dense(q1, q2, k1s, k2s, vs, lens, lam, 0.8)
    assert np.allclose(got, want, rtol=0, atol=1e-13)
    # a V scale cancels in the headwise norm (up to eps): compare the pre-norm outputs instead
    pre = ref_numpy.gda_decode_dense(q1, q2, k1, k2, v, lens, lam, 0.8, norm=False, v_scale=sv)
    base = ref_numpy.gda_decode_dense(q1, q2, k1, k2, v, lens, lam, 0.8, norm=False)
    assert np.allclose(pre, base * sv.double().numpy()[None, :, None], rtol=1e-13, atol=1e-14)


# ------------------------------------------------------------- gradients
from oracle import ref_torch_grad


def _grad_case(seed, B=1, L=5, hs=4, hn=2, d=4, dv=6):
    g = torch.Generator().manual_seed(seed)
    t = lambda *shape: torch.randn(*shape, generator=g, dtype=torch.float64)
    return (t(B, L, hs, d), t(B, L, hs, d), t(B, L, hn, d), t(B, L, hn, d), t(B, L, hs, dv),
            torch.rand(hs, generator=g, dtype=torch.float64) * 0.6 + 0.2, t(B, L, hs, dv))


def test_torch_forward_matches_numpy_dense():
    q1, k1, q2, k2, v, lam, _ = _grad_case(31, B=2, L=7)
    for causal in (True, False):
        got = ref_torch_grad.gda_forward_torch(q1, k1, q2, k2, v, lam, 0.8, causal=causal).numpy()
        want = ref_numpy.gda_dense(q1, k1, q2, k2, v, lam, 0.8, causal=causal)
        assert np.allclose(got, want, rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal,norm,wide", [(True, True, False), (False, True, False), (True, False, False),
                                               (True, True, True)])
def test_backward_matches_central_finite_differences(causal, norm, wide):
    """d/dx sum(dy * y) against (f(x + h) - f(x - h)) / 2h, coordinate by coordinate.

    ``wide``: lambda = -1, -0.5, 1.5, 2 (outside [0, 1]; lambda = 1 is left out
    because its first causal row has o = 0, where the norm's curvature makes a
    central difference with this step inaccurate)."""
    inputs = _grad_case(32)
    if wide:
        inputs = inputs[:5] + (torch.tensor([-1.0, -0.5, 1.5, 2.0], dtype=torch.float64),) + inputs[6:]
    *fwd_in, dy = inputs
    grads = ref_torch_grad.gda_backward(*fwd_in, 0.8, dy, causal=causal, norm=norm)

    def f(args):
        y = ref_torch_grad.gda_forward_torch(*args, 0.8, causal=causal, norm=norm)
        return float((y * dy).sum())
    h = 1e-6
    for which in range(6):
        base = [t.clone() for t in fwd_in]
        flat = base[which].view(-1)
        for k in range(0, flat.numel(), max(1, flat.numel() // 7)):
            orig = float(flat[k])
            flat[k] = orig + h
            fp = f(base)
            flat[k] = orig - h
            fm = f(base)
            flat[k] = orig
            fd = (fp - fm) / (2 * h)
            an = float(grads[which].reshape(-1)[k])
            assert abs(fd - an) <= 1e-6 * (1 + abs(an)), (which, k, fd, an)


def test_noise_gradient_collects_the_whole_group():
    """dK2 of a noise head equals the sum over its signal heads of the per-head terms:
    with explicit repetition (h_n = h_s, K2 repeated) the repeated copies' gradients sum to it."""
    q1, k1, q2, k2, v, lam, dy = _grad_case(33, hs=4, hn=2)
    grads = ref_torch_grad.gda_backward(q1, k1, q2, k2, v, lam, 0.8, dy)
    q2r, k2r = q2.repeat_interleave(2, dim=2), k2.repeat_interleave(2, dim=2)
    rep = ref_torch_grad.gda_backward(q1, k1, q2r, k2r, v, lam, 0.8, dy)
    assert torch.allclose(grads[2], rep[2].view(1, 5, 2, 2, 4).sum(3), atol=1e-12)
    assert torch.allclose(grads[3], rep[3].view(1, 5, 2, 2, 4).sum(3), atol=1e-12)
    for i in (0, 1, 4, 5):
        assert torch.allclose(grads[i], rep[i], atol=1e-12)


@pytest.mark.parametrize("causal", [True, False])
def test_row_logsumexp_matches_library_and_normalises(causal):
    """The rows' log-sum-exp equals torch.logsumexp of the masked scaled
    logits (library routine), exp(s - lse) sums to 1 over the visible keys,
    and the first causal row (one visible key) has lse = its single logit."""
    from oracle.ref_numpy import row_logsumexp
    g = torch.Generator().manual_seed(71)
    q = torch.randn(2, 37, 3, 16, generator=g, dtype=torch.float64)
    k = torch.randn(2, 37, 3, 16, generator=g, dtype=torch.float64)
    got = row_logsumexp(q.numpy(), k.numpy(), causal=causal)
    s = torch.einsum("bihd,bjhd->bhij", q, k) / 4.0
    if causal:
        s = s.masked_fill(torch.triu(torch.ones(37, 37, dtype=torch.bool), diagonal=1), float("-inf"))
    np.testing.assert_allclose(got, torch.logsumexp(s, dim=-1).numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(np.exp(s.numpy() - got[..., None]).sum(-1), 1.0, rtol=0, atol=1e-12)
    if causal:
        np.testing.assert_allclose(got[:, :, 0], s[:, :, 0, 0].numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal,norm", [(True, True), (False, False)])
def test_gradient_magnitudes_bound_the_gradients(causal, norm):
    """Triangle inequality: every sum of absolute terms is at least the
    absolute value of the autograd gradient it belongs to."""
    from oracle.ref_torch_grad import gda_backward, gda_grad_magnitudes
    g = torch.Generator().manual_seed(81)
    B, L, hs, hn, d, dv = 1, 9, 4, 2, 8, 16
    args = [torch.randn(B, L, hs, d, generator=g, dtype=torch.float64),
            torch.randn(B, L, hs, d, generator=g, dtype=torch.float64),
            torch.randn(B, L, hn, d, generator=g, dtype=torch.float64),
            torch.randn(B, L, hn, d, generator=g, dtype=torch.float64),
            torch.randn(B, L, hs, dv, generator=g, dtype=torch.float64),
            torch.rand(hs, generator=g, dtype=torch.float64)]
    dy = torch.randn(B, L, hs, dv, generator=g, dtype=torch.float64)
    grads = gda_backward(*args, 0.7, dy, causal=causal, norm=norm)
    mags = gda_grad_magnitudes(*args, 0.7, dy, causal=causal, norm=norm)
    for gr, m in zip(grads, mags):
        assert gr.shape == m.shape
        assert torch.all(m >= gr.abs() - 1e-12)


def test_gradient_magnitudes_equal_gradients_when_terms_share_a_sign():
    """lambda = 0, no norm, dy >= 0: every term of dv is non-negative, so the
    magnitude equals dv itself; dlambda's magnitude is sum |do . O2|, equal to
    -dlambda when every do . O2 is non-negative (dy >= 0 and V >= 0)."""
    from oracle.ref_torch_grad import gda_backward, gda_grad_magnitudes
    g = torch.Generator().manual_seed(82)
    B, L, hs, hn, d, dv = 2, 7, 2, 1, 8, 16
    q1, k1 = torch.randn(B, L, hs, d, generator=g, dtype=torch.float64), torch.randn(B, L, hs, d, generator=g, dtype=torch.float64)
    q2, k2 = torch.randn(B, L, hn, d, generator=g, dtype=torch.float64), torch.randn(B, L, hn, d, generator=g, dtype=torch.float64)
    v = torch.rand(B, L, hs, dv, generator=g, dtype=torch.float64)
    dy = torch.rand(B, L, hs, dv, generator=g, dtype=torch.float64)
    lam = torch.zeros(hs, dtype=torch.float64)
    grads = gda_backward(q1, k1, q2, k2, v, lam, 0.5, dy, causal=True, norm=False)
    mags = gda_grad_magnitudes(q1, k1, q2, k2, v, lam, 0.5, dy, causal=True, norm=False)
    np.testing.assert_allclose(mags[4].numpy(), grads[4].numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(mags[5].numpy(), -grads[5].numpy(), rtol=0, atol=1e-12)


def _loop_grad_magnitudes(q1, k1, q2, k2, v, lam, lambda_init, dy, causal, norm, eps=1e-5):
    """The gradient magnitudes written out term by term with scalar loops.

    Independent of ``gda_grad_magnitudes``: both maps come from scalar
    max-shifted softmax loops, the accumulators O1, O2 from loops over keys,
    and the norm's input gradient from PyTorch autograd of the library
    ``rms_norm`` ("Headwise Normalization").  Every term of every gradient
    (the score gradients expanded down to the dot products over dv) enters as
    the product of the absolute values of its factors.
    """
    q1, k1, q2, k2, v, dy = (t.double().numpy() for t in (q1, k1, q2, k2, v, dy))
    lam = lam.double().numpy()
    B, L, hs, d = q1.shape
    hn = q2.shape[2]
    r = hs // hn
    dv = v.shape[3]
    sc = 1.0 / math.sqrt(d)

    def softmax_rows(q, k, hq, hk, b):
        a = np.zeros((L, L))
        for i in range(L):
            keys = range(i + 1) if causal else range(L)
            s = {j: sum(q[b, i, hq, c] * k[b, j, hk, c] for c in range(d)) * sc for j in keys}
            m = max(s.values())
            z = sum(math.exp(x - m) for x in s.values())
            for j, x in s.items():
                a[i, j] = math.exp(x - m) / z
        return a

    A1 = np.zeros((B, hs, L, L))
    A2 = np.zeros((B, hs, L, L))
    for b in range(B):
        for h in range(hs):
            A1[b, h] = softmax_rows(q1, k1, h, h, b)
            A2[b, h] = softmax_rows(q2, k2, h // r, h // r, b)
    O1 = np.zeros((B, L, hs, dv))
    O2 = np.zeros((B, L, hs, dv))
    for b in range(B):
        for h in range(hs):
            for i in range(L):
                for j in range(L):
                    O1[b, i, h] += A1[b, h, i, j] * v[b, j, h]
                    O2[b, i, h] += A2[b, h, i, j] * v[b, j, h]
    o = torch.tensor(O1 - lam[None, None, :, None] * O2, requires_grad=True)
    if norm:
        y = (1.0 - lambda_init) * F.rms_norm(o, (dv,), eps=eps)
        (do,) = torch.autograd.grad(y, o, grad_outputs=torch.tensor(dy))
        do = do.numpy()
    else:
        do = dy
    m = [np.zeros_like(q1), np.zeros_like(k1), np.zeros_like(q2), np.zeros_like(k2),
         np.zeros_like(v), np.zeros(hs)]
    for b in range(B):
        for h in range(hs):
            g = h // r
            for i in range(L):
                m[5][h] += abs(sum(do[b, i, h, e] * O2[b, i, h, e] for e in range(dv)))
                for j in range(L):
                    a1, a2 = A1[b, h, i, j], abs(lam[h]) * A2[b, h, i, j]
                    if a1 == 0.0 and a2 == 0.0:
                        continue
                    t1 = t2 = 0.0
                    for e in range(dv):
                        t1 += abs(do[b, i, h, e]) * abs(v[b, j, h, e]) + abs(do[b, i, h, e]) * abs(O1[b, i, h, e])
                        t2 += abs(do[b, i, h, e]) * abs(v[b, j, h, e]) + abs(do[b, i, h, e]) * abs(O2[b, i, h, e])
                        m[4][b, j, h, e] += (a1 + a2) * abs(do[b, i, h, e])
                    for c in range(d):
                        m[0][b, i, h, c] += a1 * t1 * abs(k1[b, j, h, c]) * sc
                        m[1][b, j, h, c] += a1 * t1 * abs(q1[b, i, h, c]) * sc
                        m[2][b, i, g, c] += a2 * t2 * abs(k2[b, j, g, c]) * sc
                        m[3][b, j, g, c] += a2 * t2 * abs(q2[b, i, g, c]) * sc
    return m


@pytest.mark.parametrize("r,hn,causal,norm", [(2, 1, True, True), (3, 1, False, True),
                                              (2, 2, False, False), (3, 2, True, False)])
def test_gradient_magnitudes_equal_the_term_by_term_sums(r, hn, causal, norm):
    """Pins gda_grad_magnitudes from above and below: each of its six outputs
    equals the same sums of absolute terms evaluated by scalar loops (a
    wrong factor, such as a dropped 1/sqrt(d) or terms scaled by a constant,
    fails here; the triangle-inequality pin only bounds them from below)."""
    from oracle.ref_torch_grad import gda_grad_magnitudes
    g = torch.Generator().manual_seed(90 + 10 * r + hn)
    B, L, d, dv = 1, 6, 4, 3
    hs = r * hn
    q1, k1 = (torch.randn(B, L, hs, d, generator=g, dtype=torch.float64) for _ in range(2))
    q2, k2 = (torch.randn(B, L, hn, d, generator=g, dtype=torch.float64) for _ in range(2))
    v = torch.randn(B, L, hs, dv, generator=g, dtype=torch.float64)
    lam = torch.rand(hs, generator=g, dtype=torch.float64) * 3.0 - 1.0   # includes negative lambda
    dy = torch.randn(B, L, hs, dv, generator=g, dtype=torch.float64)
    got = gda_grad_magnitudes(q1, k1, q2, k2, v, lam, 0.6, dy, causal=causal, norm=norm)
    want = _loop_grad_magnitudes(q1, k1, q2, k2, v, lam, 0.6, dy, causal, norm)
    for name, a, b in zip(("dq1", "dk1", "dq2", "dk2", "dv", "dlambda"), got, want):
        np.testing.assert_allclose(a.numpy(), b, rtol=1e-12, atol=1e-13, err_msg=name)
