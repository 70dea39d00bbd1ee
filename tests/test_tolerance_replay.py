"""Where the bf16 output bound with a magnitude term comes from (CPU only).

The tensor-core prefill rounds each map weight P = 2^(s - m) to bf16 before
the value product (m: the exact maximum of the row's first 64-key tile), and
normalises by the unrounded float32 sum of P.  This replays exactly that
rounding in float64 on the oracle's maps and checks two claims that
parity.assert_bf16_mag_close relies on:
- every output element stays within 2^-8 mag of the exact result, mag being
  oracle.ref_numpy.gda_magnitudes (the relative rounding of each weight
  moves a sum by at most 2^-8 times the sum of its absolute terms; the norm
  rescales both alike);
- with lambda near 1 the plain elementwise bound 3e-3 + 2e-2 |ref| does not
  hold for the replay itself, so a kernel that rounds P cannot meet it there.
"""
import numpy as np
import pytest
import torch

from grouped_differential_attention_gb300 import workloads as W
from oracle.ref_numpy import contiguous_groups, gda_dense, gda_magnitudes


def _bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x)).float().to(torch.bfloat16).double().numpy()


def _replay(q1, k1, q2, k2, v, lam, lambda_init, eps=1e-5):
    q1, k1, q2, k2, v = (t.double().numpy() for t in (q1, k1, q2, k2, v))
    lam = lam.double().numpy()
    B, L, hs, d = q1.shape
    hidden = np.triu(np.ones((L, L), dtype=bool), k=1)

    def weights(q, k):
        s = np.where(hidden, -np.inf, np.einsum("bihd,bjhd->bhij", q, k) / np.sqrt(d))
        m = np.max(s[..., :64], axis=-1, keepdims=True)
        p = np.exp(s - m)
        return _bf16(p) / p.sum(axis=-1, keepdims=True)

    w1 = weights(q1, k1)
    w2 = weights(q2, k2)[:, contiguous_groups(hs, q2.shape[2])]
    o = np.einsum("bhij,bjhe->bihe", w1 - lam[None, :, None, None] * w2, v)
    return (1.0 - lambda_init) * o / np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps)


@pytest.mark.parametrize("seed,d,dv,hs,hn,L", [(71, 64, 128, 7, 1, 259), (73, 128, 256, 7, 1, 200),
                                               (77, 64, 128, 4, 2, 300)])
def test_rounded_weights_stay_within_the_magnitude_term(seed, d, dv, hs, hn, L):
    q1, k1, q2, k2, v, _ = W.make_prefill_inputs(W.GDA3_PREFILL_L2048, B=2, L=L, h_s=hs, h_n=hn, d=d, dv=dv,
                                                 seed=seed)
    lam = torch.linspace(-1.0, 2.0, hs)
    got = _replay(q1, k1, q2, k2, v, lam, 0.8)
    f64 = [t.double() for t in (q1, k1, q2, k2, v, lam)]
    ref = gda_dense(*f64, 0.8)
    mag = gda_magnitudes(*f64, 0.8)
    err = np.abs(got - ref)
    assert np.all(err <= 2.0 ** -8 * mag)
    plain = err > 3e-3 + 2e-2 * np.abs(ref)
    assert plain.any()                                   # the plain bound alone is not enough ...
    lam_of_bad = lam.numpy()[np.nonzero(plain)[2]]
    assert np.all(np.abs(lam_of_bad - 1.0) < 0.75)      # ... and only near lambda = 1
