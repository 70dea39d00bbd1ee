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
