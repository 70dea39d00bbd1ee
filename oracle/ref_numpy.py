"""Dense-matrix NumPy formulation of grouped differential attention (float64).

TEST INFRASTRUCTURE ONLY (see the package docstring).  This is written
independently of ``gda_oracle.c``: it materialises the full attention maps as
matrices and applies the difference map to V with one contraction, whereas
the C oracle loops row by row.  It is meant for tiny inputs (L of a few
dozen) where the L x L maps are cheap.

Sources: "Differential Attention in Large Language Models ..." (sections
"Differential Attention Architecture" and "Headwise Normalization") and the
"Grouped Differential Attention" abstract (noise heads shared by groups of
signal heads, as in grouped-query attention).
"""
from __future__ import annotations

import numpy as np


def _softmax_last(x: np.ndarray) -> np.ndarray:
    m = np.max(x, axis=-1, keepdims=True)
    e = np.exp(x - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def contiguous_groups(h_s: int, h_n: int) -> np.ndarray:
    """Noise head index of every signal head: h -> h // (h_s / h_n)."""
    return np.arange(h_s) // (h_s // h_n)


def gda_dense(q1, k1, q2, k2, v, lam, lambda_init, causal=True, eps=1e-5, norm=True,
              group_of=None):
    """q1,k1: [B,L,hs,d]; q2,k2: [B,L,hn,d]; v: [B,L,hs,dv]; lam: [hs] -> [B,L,hs,dv].

    ``group_of`` maps each signal head to its noise head (default: contiguous
    groups); tests use it to check that the pins notice a wrong mapping.
    """
    q1, k1, q2, k2, v = (np.asarray(t, dtype=np.float64) for t in (q1, k1, q2, k2, v))
    lam = np.asarray(lam, dtype=np.float64).reshape(-1)
    B, L, hs, d = q1.shape
    hn = q2.shape[2]
    if group_of is None:
        group_of = contiguous_groups(hs, hn)
    group_of = np.asarray(group_of)

    # logits as [B, heads, L_q, L_k]
    s1 = np.einsum("bihd,bjhd->bhij", q1, k1) / np.sqrt(d)
    s2 = np.einsum("bigd,bjgd->bgij", q2, k2) / np.sqrt(d)
    if causal:
        hidden = np.triu(np.ones((L, L), dtype=bool), k=1)  # key j > query i
        s1 = np.where(hidden, -np.inf, s1)
        s2 = np.where(hidden, -np.inf, s2)
    a1 = _softmax_last(s1)                       # [B, hs, L, L]
    a2 = _softmax_last(s2)[:, group_of]          # noise map of each signal head
    diff = a1 - lam[None, :, None, None] * a2    # difference map
    o = np.einsum("bhij,bjhe->bihe", diff, v)    # [B, L, hs, dv]
    if norm:
        rms = np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps)
        o = (1.0 - lambda_init) * o / rms
    return o


def gda_decode_dense(q1, q2, k1c, k2c, vc, lens, lam, lambda_init, eps=1e-5, norm=True,
                     k1_scale=None, k2_scale=None, v_scale=None):
    """Decode of one query token per sequence over its cache, float64.

    q1: [B, hs, d]; q2: [B, hn, d]; k1c: [B, Lcap, hs, d]; k2c: [B, Lcap, hn, d];
    vc: [B, Lcap, hs, dv]; lens: [B] (rows 0 .. lens[b]-1 are attended);
    lam: [hs].  Optional per-head scales multiply the cached values first
    (k1_scale, v_scale: [hs]; k2_scale: [hn]), which is how a quantised cache
    (codes times a per-head scale) is dequantised.  The decode is the last
    row of the causal prefill over the first lens[b] cache rows.
    """
    q1, q2, k1c, k2c, vc = (np.asarray(t, dtype=np.float64) for t in (q1, q2, k1c, k2c, vc))
    lam = np.asarray(lam, dtype=np.float64).reshape(-1)
    B, hs, d = q1.shape
    hn = q2.shape[1]
    if k1_scale is not None:
        k1c = k1c * np.asarray(k1_scale, dtype=np.float64)[None, None, :, None]
    if k2_scale is not None:
        k2c = k2c * np.asarray(k2_scale, dtype=np.float64)[None, None, :, None]
    if v_scale is not None:
        vc = vc * np.asarray(v_scale, dtype=np.float64)[None, None, :, None]
    group_of = contiguous_groups(hs, hn)
    out = np.empty((B, hs, vc.shape[3]))
    for b in range(B):
        n = int(lens[b])
        s1 = np.einsum("hd,jhd->hj", q1[b], k1c[b, :n]) / np.sqrt(d)
        s2 = np.einsum("gd,jgd->gj", q2[b], k2c[b, :n]) / np.sqrt(d)
        a1 = _softmax_last(s1)
        a2 = _softmax_last(s2)[group_of]
        o = np.einsum("hj,jhe->he", a1 - lam[:, None] * a2, vc[b, :n])
        if norm:
            o = (1.0 - lambda_init) * o / np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps)
        out[b] = o
    return out


def row_logsumexp(q, k, causal=True):
    """Log-sum-exp (natural log) of every query row's scaled logits, float64.

    q, k: [B, L, heads, d] -> [B, heads, L]; entry (b, h, i) is
    log sum_{j visible} exp(q_i . k_j / sqrt d), the normaliser of that row's
    softmax map ("Differential Attention in Large Language Models ...",
    section "Differential Attention Architecture": each map is a softmax of
    the scaled logits).  Visible keys: j <= i when causal, all j otherwise.
    Written with the usual maximum shift: m + log sum exp(s - m).
    """
    q, k = (np.asarray(t, dtype=np.float64) for t in (q, k))
    B, L, H, d = q.shape
    s = np.einsum("bihd,bjhd->bhij", q, k) / np.sqrt(d)
    if causal:
        s = np.where(np.triu(np.ones((L, L), dtype=bool), k=1), -np.inf, s)
    m = np.max(s, axis=-1)
    return m + np.log(np.sum(np.exp(s - m[..., None]), axis=-1))


def gda_magnitudes(q1, k1, q2, k2, v, lam, lambda_init, causal=True, eps=1e-5, norm=True):
    """Size of the terms that make up each output element, float64, [B,L,hs,dv].

    The output is a sum over keys of (a1_ij - lambda_h a2_ij) v_jc with a1, a2
    the two softmax maps ("Differential Attention in Large Language Models
    ...", section "Differential Attention Architecture"; noise map of head
    h // (h_s / h_n) per the "Grouped Differential Attention" abstract).  This
    returns the same sum with every term replaced by its absolute value,
    sum_j (a1_ij + |lambda_h| a2_ij) |v_jc|, and with ``norm`` that sum scaled
    like the output, by |1 - lambda_init| / sqrt(mean_c(o_c^2) + eps)
    (section "Headwise Normalization").  It bounds |output| and measures how
    much a relative rounding of every map weight can move the output when
    the two maps nearly cancel (lambda near 1).
    """
    q1, k1, q2, k2, v = (np.asarray(t, dtype=np.float64) for t in (q1, k1, q2, k2, v))
    lam = np.asarray(lam, dtype=np.float64).reshape(-1)
    B, L, hs, d = q1.shape
    hn = q2.shape[2]
    s1 = np.einsum("bihd,bjhd->bhij", q1, k1) / np.sqrt(d)
    s2 = np.einsum("bigd,bjgd->bgij", q2, k2) / np.sqrt(d)
    if causal:
        hidden = np.triu(np.ones((L, L), dtype=bool), k=1)
        s1 = np.where(hidden, -np.inf, s1)
        s2 = np.where(hidden, -np.inf, s2)
    a1 = _softmax_last(s1)
    a2 = _softmax_last(s2)[:, contiguous_groups(hs, hn)]
    mag = np.einsum("bhij,bjhe->bihe", a1 + np.abs(lam)[None, :, None, None] * a2, np.abs(v))
    if norm:
        o = np.einsum("bhij,bjhe->bihe", a1 - lam[None, :, None, None] * a2, v)
        mag = abs(1.0 - lambda_init) * mag / np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps)
    return mag
