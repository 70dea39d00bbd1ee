"""Gradients of grouped differential attention in float64 (PyTorch autograd, CPU).

TEST INFRASTRUCTURE ONLY (see the package docstring).  The forward below is
the definition of ``gda_oracle.c`` written with dense PyTorch float64 ops;
``gda_backward`` differentiates it with autograd.  It is pinned by central
finite differences in ``tests/test_oracle_pins.py`` (an independent check:
no derivative formula is shared with it).

Sources: "Differential Attention in Large Language Models ...", sections
"Differential Attention Architecture" and "Headwise Normalization"; noise
heads shared by groups of signal heads per the "Grouped Differential
Attention" abstract (the noise head's gradient collects the contributions
of every signal head of its group).
"""
from __future__ import annotations

import math

import torch


def gda_forward_torch(q1, k1, q2, k2, v, lam, lambda_init: float, causal: bool = True,
                      eps: float = 1e-5, norm: bool = True):
    """q1,k1: [B,L,hs,d]; q2,k2: [B,L,hn,d]; v: [B,L,hs,dv]; lam: [hs] -> [B,L,hs,dv] (float64)."""
    B, L, hs, d = q1.shape
    hn = q2.shape[2]
    r = hs // hn
    s1 = torch.einsum("bihd,bjhd->bhij", q1, k1) / math.sqrt(d)
    s2 = torch.einsum("bigd,bjgd->bgij", q2, k2) / math.sqrt(d)
    if causal:
        hidden = torch.triu(torch.ones(L, L, dtype=torch.bool), diagonal=1)
        s1 = s1.masked_fill(hidden, float("-inf"))
        s2 = s2.masked_fill(hidden, float("-inf"))
    a1 = torch.softmax(s1, dim=-1)
    a2 = torch.softmax(s2, dim=-1).repeat_interleave(r, dim=1)    # noise map of each signal head
    o = torch.einsum("bhij,bjhe->bihe", a1 - lam.view(1, hs, 1, 1) * a2, v)
    if norm:
        o = (1.0 - lambda_init) * o / torch.sqrt((o * o).mean(dim=-1, keepdim=True) + eps)
    return o


def gda_backward(q1, k1, q2, k2, v, lam, lambda_init: float, dy, causal: bool = True,
                 eps: float = 1e-5, norm: bool = True):
    """Gradients (dq1, dk1, dq2, dk2, dv, dlam) of sum(dy * y), float64."""
    args = [torch.as_tensor(t).to(torch.float64).clone().requires_grad_(True)
            for t in (q1, k1, q2, k2, v, lam)]
    y = gda_forward_torch(*args, lambda_init, causal=causal, eps=eps, norm=norm)
    grads = torch.autograd.grad(y, args, grad_outputs=torch.as_tensor(dy).to(torch.float64))
    return tuple(g.detach() for g in grads)


def gda_grad_magnitudes(q1, k1, q2, k2, v, lam, lambda_init: float, dy, causal: bool = True,
                        eps: float = 1e-5, norm: bool = True):
    """Sums of the absolute values of the terms of each gradient (float64).

    Each gradient is a contraction of per-pair terms; this returns the same
    contractions with every factor replaced by its absolute value:
      dq1_i: sum_j A1_ij (|do_i| . |v_j| + |do_i| . |O1_i|) |k1_j| / sqrt d
      dk1_j: sum_i A1_ij (|do_i| . |v_j| + |do_i| . |O1_i|) |q1_i| / sqrt d
      dq2, dk2: the same with |lambda| A2 and O2, q2, k2, summed over the
                group's heads
      dv_j: sum_i (A1 + |lambda| A2)_ij |do_i|    dlambda_h: sum_{b,i} |do_i . O2_i|
    (the score gradients dS1 = A1 (dP - D1), dS2 = -lambda A2 (dP - D2) expanded
    into their terms down to the dot products over dv), dP_ij = do_i . v_j,
    D1 = do . O1, D2 = do . O2 and do the norm's input gradient (chain rule
    through "Headwise Normalization" of "Differential Attention in Large
    Language Models ...").  By the triangle inequality each is at least the
    absolute value of the gradient itself; rounding errors of a computation
    that forms these terms scale with them, which is what they are used for
    (sizing the tolerance of reduced-precision gradients).
    """
    q1, k1, q2, k2, v, dy = (torch.as_tensor(t).to(torch.float64) for t in (q1, k1, q2, k2, v, dy))
    lam = torch.as_tensor(lam).to(torch.float64)
    B, L, hs, d = q1.shape
    hn = q2.shape[2]
    r = hs // hn
    dv = v.shape[3]
    sc = 1.0 / math.sqrt(d)
    s1 = torch.einsum("bihd,bjhd->bhij", q1, k1) * sc
    s2 = torch.einsum("bigd,bjgd->bgij", q2, k2) * sc
    if causal:
        hidden = torch.triu(torch.ones(L, L, dtype=torch.bool), diagonal=1)
        s1 = s1.masked_fill(hidden, float("-inf"))
        s2 = s2.masked_fill(hidden, float("-inf"))
    a1 = torch.softmax(s1, dim=-1)
    a2 = torch.softmax(s2, dim=-1).repeat_interleave(r, dim=1)
    O1 = torch.einsum("bhij,bjhe->bihe", a1, v)
    O2 = torch.einsum("bhij,bjhe->bihe", a2, v)
    if norm:
        o = O1 - lam.view(1, 1, hs, 1) * O2
        r2 = (o * o).mean(dim=-1, keepdim=True) + eps
        c = (1.0 - lambda_init) / torch.sqrt(r2)
        do = c * (dy - o * (dy * o).sum(dim=-1, keepdim=True) / (dv * r2))
    else:
        do = dy
    dP = torch.einsum("bihe,bjhe->bhij", do, v)
    D1 = (do * O1).sum(-1).permute(0, 2, 1)[..., None]
    D2 = (do * O2).sum(-1).permute(0, 2, 1)[..., None]
    lam4 = lam.view(1, hs, 1, 1)
    # dS1 = A1 dP - A1 D1 and dS2 = -lambda A2 dP + lambda A2 D2, with dP and
    # D themselves dot products over dv: absolute values of every term
    dP_abs = torch.einsum("bihe,bjhe->bhij", do.abs(), v.abs())
    D1_abs = (do.abs() * O1.abs()).sum(-1).permute(0, 2, 1)[..., None]
    D2_abs = (do.abs() * O2.abs()).sum(-1).permute(0, 2, 1)[..., None]
    dS1 = a1 * (dP_abs + D1_abs)
    dS2 = lam4.abs() * a2 * (dP_abs + D2_abs)
    Wm = a1 + lam4.abs() * a2                 # the two terms of A1 - lambda A2
    m_dq1 = torch.einsum("bhij,bjhd->bihd", dS1, k1.abs()) * sc
    m_dk1 = torch.einsum("bhij,bihd->bjhd", dS1, q1.abs()) * sc
    dS2g = dS2.reshape(B, hn, r, L, L).sum(2)
    m_dq2 = torch.einsum("bgij,bjgd->bigd", dS2g, k2.abs()) * sc
    m_dk2 = torch.einsum("bgij,bigd->bjgd", dS2g, q2.abs()) * sc
    m_dv = torch.einsum("bhij,bihe->bjhe", Wm, do.abs())
    m_dlam = D2.abs().sum(dim=(0, 2, 3))
    return m_dq1, m_dk1, m_dq2, m_dk2, m_dv, m_dlam
