"""Seeded synthetic inputs for grouped differential attention.

This module only draws random tensors with the shapes, distributions and
structure of the workloads below; it performs none of the attention
arithmetic, so the CUDA path and the float64 oracle can share it.

Every tensor is drawn on the CPU from ``torch.Generator().manual_seed(seed)``
in float32 and rounded once to the I/O dtype (bf16 round-to-nearest-even, or
kept as float32), so both sides see identical bytes.  Draw order: Q1, K1, Q2,
K2, V, lambda, then the boosted key positions (long-context workload); for
decode: Q1, Q2, then per sequence K1, K2, V cache rows, then lambda and the
cache lengths.

The pages measure whole language models on public corpora and benchmarks;
these standard-normal tensors at the same attention shapes stand in for them.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Tuple

import torch


@dataclasses.dataclass(frozen=True)
class PrefillWorkload:
    name: str
    B: int
    L: int
    h_s: int
    h_n: int
    d: int
    dv: int
    causal: bool
    dtype: str                 # "bf16" or "f32"
    lam_range: Tuple[float, float]
    lambda_init: float
    eps: float = 1e-5
    key_boost: Optional[Tuple[float, float]] = None   # (fraction of key positions, factor)
    seed: int = 0


@dataclasses.dataclass(frozen=True)
class DecodeWorkload:
    name: str
    B: int
    Lcap: int
    len_range: Tuple[int, int]   # inclusive
    h_s: int
    h_n: int
    d: int
    dv: int
    lam_range: Tuple[float, float]
    lambda_init: float
    eps: float = 1e-5
    seed: int = 0


# lambda_init of layer 8 under the depth schedule 0.8 - 0.6 exp(-0.3 (l - 1)),
# written out as a literal (this module does no method arithmetic).
LAMBDA_INIT_LAYER8 = 0.726526143048211

DIFF_F32_L128 = PrefillWorkload(
    name="diff_1to1_f32_B1_L128_h2+2_d64_dv128", B=1, L=128, h_s=2, h_n=2, d=64, dv=128,
    causal=True, dtype="f32", lam_range=(0.2, 0.8), lambda_init=0.8)

GDA3_PREFILL_L2048 = PrefillWorkload(
    name="gda_3to1_prefill_bf16_B4_L2048_h12+4_d64_dv128", B=4, L=2048, h_s=12, h_n=4,
    d=64, dv=128, causal=True, dtype="bf16", lam_range=(0.2, 0.8),
    lambda_init=LAMBDA_INIT_LAYER8)

GDA4_PREFILL_L8192 = PrefillWorkload(
    name="gda_4to1_prefill_bf16_B2_L8192_h16+4_d128_dv256", B=2, L=8192, h_s=16, h_n=4,
    d=128, dv=256, causal=True, dtype="bf16", lam_range=(0.1, 0.9), lambda_init=0.8)

GDA3_PREFILL_L32768 = PrefillWorkload(
    name="gda_3to1_longctx_prefill_bf16_B1_L32768_h24+8_d64_dv128", B=1, L=32768, h_s=24,
    h_n=8, d=64, dv=128, causal=True, dtype="bf16", lam_range=(0.2, 0.8), lambda_init=0.8,
    key_boost=(0.01, 4.0))

GDA3_DECODE_B64 = DecodeWorkload(
    name="gda_3to1_decode_bf16_B64_len4096-8192_h12+4_d64_dv128", B=64, Lcap=8192,
    len_range=(4096, 8192), h_s=12, h_n=4, d=64, dv=128, lam_range=(0.2, 0.8),
    lambda_init=0.8)

PREFILL_WORKLOADS = {w.name: w for w in (DIFF_F32_L128, GDA3_PREFILL_L2048,
                                         GDA4_PREFILL_L8192, GDA3_PREFILL_L32768)}


def _io_dtype(name: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "f32": torch.float32}[name]


def make_prefill_inputs(w: PrefillWorkload, **overrides):
    """Draw (q1, k1, q2, k2, v, lam) on the CPU for a prefill workload.

    ``overrides`` may replace B, L, h_s, h_n, d, dv, seed, dtype (small parity
    cases reuse a workload's recipe at other sizes).
    """
    return make_prefill_inputs_and_boosted(w, **overrides)[0]


def make_prefill_inputs_and_boosted(w: PrefillWorkload, **overrides):
    """``make_prefill_inputs`` plus the boosted key positions of each sequence.

    Returns ((q1, k1, q2, k2, v, lam), positions): positions[b] is the sorted
    list of key positions of sequence b whose K1 and K2 rows were scaled (an
    empty list for every b when the workload boosts none).
    """
    p = dataclasses.replace(w, **overrides) if overrides else w
    g = torch.Generator().manual_seed(p.seed)
    q1 = torch.randn(p.B, p.L, p.h_s, p.d, generator=g)
    k1 = torch.randn(p.B, p.L, p.h_s, p.d, generator=g)
    q2 = torch.randn(p.B, p.L, p.h_n, p.d, generator=g)
    k2 = torch.randn(p.B, p.L, p.h_n, p.d, generator=g)
    v = torch.randn(p.B, p.L, p.h_s, p.dv, generator=g)
    lo, hi = p.lam_range
    lam = torch.empty(p.h_s).uniform_(lo, hi, generator=g)
    positions = [[] for _ in range(p.B)]
    if p.key_boost is not None:
        frac, factor = p.key_boost
        n = int(math.floor(frac * p.L))
        for b in range(p.B):
            idx = torch.randperm(p.L, generator=g)[:n]
            k1[b, idx] *= factor
            k2[b, idx] *= factor
            positions[b] = sorted(int(i) for i in idx)
    dt = _io_dtype(p.dtype)
    return (q1.to(dt), k1.to(dt), q2.to(dt), k2.to(dt), v.to(dt), lam.to(torch.float32)), positions


def make_backward_inputs(w: PrefillWorkload, **overrides):
    """Draw (q1, k1, q2, k2, v, lam, dy) on the CPU: the prefill inputs of
    ``make_prefill_inputs`` plus an upstream gradient dy [B, L, h_s, dv]
    drawn from N(0, 1) with a generator seeded by seed + 1.
    """
    p = dataclasses.replace(w, **overrides) if overrides else w
    inputs = make_prefill_inputs(p)
    g = torch.Generator().manual_seed(p.seed + 1)
    dy = torch.randn(p.B, p.L, p.h_s, p.dv, generator=g).to(_io_dtype(p.dtype))
    return inputs + (dy,)


def make_decode_inputs(w: DecodeWorkload, **overrides):
    """Draw (q1, q2, k1_cache, k2_cache, v_cache, lens, lam) on the CPU (bf16 I/O).

    Cache rows at and beyond a sequence's length are drawn too (they are
    never read by a correct kernel); lens[b] is uniform on len_range.
    """
    p = dataclasses.replace(w, **overrides) if overrides else w
    g = torch.Generator().manual_seed(p.seed)
    bf = torch.bfloat16
    q1 = torch.randn(p.B, p.h_s, p.d, generator=g).to(bf)
    q2 = torch.randn(p.B, p.h_n, p.d, generator=g).to(bf)
    k1c = torch.empty(p.B, p.Lcap, p.h_s, p.d, dtype=bf)
    k2c = torch.empty(p.B, p.Lcap, p.h_n, p.d, dtype=bf)
    vc = torch.empty(p.B, p.Lcap, p.h_s, p.dv, dtype=bf)
    for b in range(p.B):
        k1c[b] = torch.randn(p.Lcap, p.h_s, p.d, generator=g).to(bf)
        k2c[b] = torch.randn(p.Lcap, p.h_n, p.d, generator=g).to(bf)
        vc[b] = torch.randn(p.Lcap, p.h_s, p.dv, generator=g).to(bf)
    lo, hi = p.lam_range
    lam = torch.empty(p.h_s).uniform_(lo, hi, generator=g).to(torch.float32)
    a, b_ = p.len_range
    lens = torch.randint(a, b_ + 1, (p.B,), generator=g, dtype=torch.int64).to(torch.int32)
    return q1, q2, k1c, k2c, vc, lens, lam


E4M3_MAX = 448.0   # largest finite float8 e4m3 value


def quantize_e4m3_per_head(x: torch.Tensor):
    """fp8 (e4m3) codes and per-head float32 scales of a cache [B, L, heads, dim].

    scale_h = amax_h / 448 over the head's values (1.0 for an all-zero head);
    codes = round-to-nearest e4m3 of x / scale_h.  The cached value a decode
    sees is codes * scale_h.
    """
    xf = x.float()
    amax = xf.abs().amax(dim=(0, 1, 3))
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax)).to(torch.float32)
    codes = (xf / scale[None, None, :, None]).to(torch.float8_e4m3fn)
    return codes, scale


def make_decode_inputs_fp8(w: DecodeWorkload, **overrides):
    """The decode inputs of make_decode_inputs with fp8 (e4m3) caches.

    Returns (q1, q2, k1_codes, k2_codes, v_codes, k1_scale, k2_scale, v_scale,
    lens, lam): the bf16 caches quantised per head by quantize_e4m3_per_head.
    """
    q1, q2, k1c, k2c, vc, lens, lam = make_decode_inputs(w, **overrides)
    k1q, k1s = quantize_e4m3_per_head(k1c)
    k2q, k2s = quantize_e4m3_per_head(k2c)
    vq, vs = quantize_e4m3_per_head(vc)
    return q1, q2, k1q, k2q, vq, k1s, k2s, vs, lens, lam


def page_caches(k1c, k2c, vc, page_size: int, seed: int = 0, spare_pages: int = 3):
    """Scatter contiguous caches [B, Lcap, heads, dim] into page pools.

    Lcap must be a multiple of page_size.  Returns (k1_pool, k2_pool, v_pool,
    block_table): the sequences' pages go to a seeded random permutation of
    the pool's pages (spare pages stay as noise), block_table[b, j] naming the
    page that holds cache rows j*page_size .. (j+1)*page_size - 1 of b.
    """
    B, Lcap = k1c.shape[0], k1c.shape[1]
    assert Lcap % page_size == 0
    max_pages = Lcap // page_size
    num_pages = B * max_pages + spare_pages
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(num_pages, generator=g)[:B * max_pages]
    table = perm.view(B, max_pages).to(torch.int32)

    def pool(c):
        out = torch.randn((num_pages, page_size) + tuple(c.shape[2:]), generator=g).to(c.dtype)
        out[perm] = c.reshape((B * max_pages, page_size) + tuple(c.shape[2:]))
        return out
    return pool(k1c), pool(k2c), pool(vc), table


def causal_pairs(L: int) -> int:
    """Number of (query, key <= query) pairs in one causal L x L map."""
    return L * (L + 1) // 2
