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
