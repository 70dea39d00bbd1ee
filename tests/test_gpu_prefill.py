"""GPU parity of the prefill paths against the float64 oracle (same seeded inputs).

bf16 path (tcgen05/TMA kernels): |err| <= 3e-3 + 2e-2|ref| elementwise.
f32 path (CUDA-core kernel): |err| <= 1e-4 (|ref| + rms_row(ref)).
Small cases are compared on every element (several 128-row tiles, ragged
tails, L = 1, non-causal, d = 128 with dv split over a CTA pair); the
3:1 workload is compared on every element, the 4:1 and long-context workloads
on 1024 or more sampled rows (with the long-context workload's boosted key
positions among them), plus properties that hold at any size.
"""
import numpy as np
import pytest
import torch

import grouped_differential_attention_gb300 as gda
from grouped_differential_attention_gb300 import workloads as W
from parity import assert_bf16_close, assert_f32_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def device_error_word_stays_clear():
    from grouped_differential_attention_gb300 import build
    build.build()
    gda.gda_device_error(clear=True)
    yield
    assert gda.gda_device_error(clear=True) == 0


def to_cuda(ts):
    return [t.cuda() for t in ts]


def run_bf16(inputs, lam_init, causal=True, eps=1e-5, flags=0):
    out = gda.gda_attn_fwd(*to_cuda(inputs), lam_init, causal=causal, eps=eps, flags=flags)
    torch.cuda.synchronize()
    return out.cpu()


def run_f32(inputs, lam_init, causal=True, eps=1e-5, flags=0):
    out = gda.gda_attn_fwd_f32(*to_cuda(inputs), lam_init, causal=causal, eps=eps, flags=flags)
    torch.cuda.synchronize()
    return out.cpu()


SMALL_BF16 = [  # B, L, h_s, h_n, d, dv, causal
    (1, 1, 2, 2, 64, 128, True),
    (1, 128, 3, 1, 64, 128, True),
    (2, 300, 6, 2, 64, 128, True),
    (1, 129, 4, 4, 64, 128, False),
    (2, 257, 12, 4, 64, 128, True),
    (1, 520, 3, 1, 64, 128, True),
    (1, 200, 4, 1, 128, 256, True),
    (1, 131, 8, 2, 128, 128, False),
    (2, 64, 2, 1, 128, 256, False),
    (1, 390, 4, 2, 128, 128, True),
    (1, 200, 8, 2, 64, 128, True),       # groups of 4: two items of 2 signal heads per noise head
    (2, 150, 6, 1, 64, 128, False),      # groups of 6: two items of 3
    (1, 333, 4, 2, 64, 128, True),       # groups of 2
    (3, 70, 5, 1, 64, 128, True),        # groups of 5: items of one signal head
]


@pytest.mark.parametrize("shape", SMALL_BF16, ids=lambda s: "B%dL%dhs%dhn%dd%ddv%d%s" % (
    s[0], s[1], s[2], s[3], s[4], s[5], "c" if s[6] else "f"))
def test_prefill_bf16_matches_oracle(oracle_mod, shape):
    B, L, hs, hn, d, dv, causal = shape
    inp = W.make_prefill_inputs(W.GDA3_PREFILL_L2048, B=B, L=L, h_s=hs, h_n=hn, d=d, dv=dv,
                                seed=1000 + L + hs)
    got = run_bf16(inp, 0.8, causal)
    ref = oracle_mod.prefill(*inp, 0.8, causal=causal)
    assert_bf16_close(got, ref, str(shape))


@pytest.mark.parametrize("shape", SMALL_BF16[1:6], ids=lambda s: "B%dL%dhs%dhn%dd%ddv%d%s" % (
    s[0], s[1], s[2], s[3], s[4], s[5], "c" if s[6] else "f"))
def test_prefill_bf16_single_pass_flag(oracle_mod, shape):
    """GDA_FLAG_SINGLE_PASS runs the per-signal-head single-pass kernel
    whatever gda_attn_fwd would choose; it must match the oracle too."""
    B, L, hs, hn, d, dv, causal = shape
    inp = W.make_prefill_inputs(W.GDA3_PREFILL_L2048, B=B, L=L, h_s=hs, h_n=hn, d=d, dv=dv,
                                seed=1000 + L + hs)
    got = run_bf16(inp, 0.8, causal, flags=gda.GDA_FLAG_SINGLE_PASS)
    ref = oracle_mod.prefill(*inp, 0.8, causal=causal)
    assert_bf16_close(got, ref, str(shape))


def _sample_rows(L, n, seed, extra=()):
    """At least n distinct query rows of [0, L): the tile edges 0, 1, 127, 128,
    129, the middle and the last two rows, any ``extra`` rows, then seeded
    uniform draws."""
    g = np.random.default_rng(seed)
    rows = {r for r in [0, 1, 127, 128, 129, L // 2, L - 2, L - 1] + list(extra) if 0 <= r < L}
    rest = [int(r) for r in g.permutation(L) if int(r) not in rows]
    rows.update(rest[:max(0, n - len(rows))])
    return sorted(rows)


def test_prefill_3to1_workload_every_element(oracle_mod):
    """The 3:1 workload (B=4, L=2048, 12 + 4 heads) on every output element."""
    w = W.GDA3_PREFILL_L2048
    inp = W.make_prefill_inputs(w)
    got = run_bf16(inp, w.lambda_init, w.causal, w.eps)
    ref = oracle_mod.prefill(*inp, w.lambda_init, causal=w.causal, eps=w.eps)
    assert_bf16_close(got, ref, w.name)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("B,L,hs,hn", [(8, 1200, 3, 1), (4, 600, 8, 2)], ids=["three_heads", "two_heads"])
def test_prefill_whole_group_items_ragged_tail(oracle_mod, causal, B, L, hs, hn):
    """Short items of several signal heads (B=8, L=1200, a 3:1 group: 160 items of three
    heads; B=4, L=600, 4:1 groups: 160 items of two heads) with the output staged for TMA
    stores; the last query tile holds 48 or 88 rows, so one row quarter's store is clipped
    at L and the quarters past it have no rows at all."""
    inp = W.make_prefill_inputs(W.GDA3_PREFILL_L2048, B=B, L=L, h_s=hs, h_n=hn, seed=1201 + L)
    got = run_bf16(inp, 0.8, causal)
    ref = oracle_mod.prefill(*inp, 0.8, causal=causal)
    assert_bf16_close(got, ref, "short items of several heads, ragged tail")


@pytest.mark.parametrize("w", [W.GDA4_PREFILL_L8192, W.GDA3_PREFILL_L32768], ids=lambda x: x.name)
def test_prefill_full_size_sampled_rows(oracle_mod, w):
    """1024 or more seeded query rows (all sequences and heads) of the 4:1 and
    long-context workloads; for the long-context one every boosted key
    position is a sampled query row as well (its own key is then the peaked
    one), plus the row after each."""
    inp, boosted = W.make_prefill_inputs_and_boosted(w)
    got = run_bf16(inp, w.lambda_init, w.causal, w.eps)
    assert torch.isfinite(got.float()).all()
    extra = sorted({p + dp for pos in boosted for p in pos for dp in (0, 1)})
    rows = _sample_rows(w.L, 1024 + len(extra), seed=7, extra=extra)
    assert len(rows) >= 1024
    ref = oracle_mod.prefill_rows(*inp, w.lambda_init, rows, causal=w.causal, eps=w.eps)
    assert_bf16_close(got[:, rows], ref, w.name)


def test_prefill_bf16_unit_values_closed_form():
    """V = 1 at the full 3:1 size: every output element is (1-li)(1-lam)/sqrt((1-lam)^2+eps)."""
    w = W.GDA3_PREFILL_L2048
    q1, k1, q2, k2, v, lam = W.make_prefill_inputs(w)
    v = torch.ones_like(v)
    got = run_bf16((q1, k1, q2, k2, v, lam), w.lambda_init, True, w.eps).double()
    lam64 = lam.double()
    closed = (1 - w.lambda_init) * (1 - lam64) / torch.sqrt((1 - lam64) ** 2 + w.eps)
    assert_bf16_close(got, closed[None, None, :, None].expand_as(got).numpy(), "V=1 closed form")


@pytest.mark.parametrize("d,dv", [(64, 128), (128, 256)])
def test_prefill_bf16_equal_maps_cancel_exactly(d, dv):
    """Q2 = Q1, K2 = K1, h_s = h_n, lambda = 1: the pre-norm output is exactly 0."""
    q1, k1, _, _, v, lam = W.make_prefill_inputs(W.GDA3_PREFILL_L2048, B=2, L=333, h_s=4, h_n=4,
                                                 d=d, dv=dv, seed=5)
    got = run_bf16((q1, k1, q1, k1, v, torch.ones_like(lam)), 0.8, flags=gda.GDA_FLAG_NO_NORM)
    assert torch.count_nonzero(got) == 0


def test_prefill_bf16_no_norm_matches_oracle(oracle_mod):
    inp = W.make_prefill_inputs(W.GDA3_PREFILL_L2048, B=1, L=260, h_s=6, h_n=2, seed=9)
    got = run_bf16(inp, 0.8, flags=gda.GDA_FLAG_NO_NORM)
    ref = oracle_mod.prefill(*inp, 0.8, norm=False)
    assert_bf16_close(got, ref, "pre-norm")


def test_prefill_bf16_first_row_closed_form():
    q1, k1, q2, k2, v, lam = W.make_prefill_inputs(W.GDA3_PREFILL_L2048, B=2, L=150, h_s=6, h_n=3,
                                                   seed=13)
    got = run_bf16((q1, k1, q2, k2, v, lam), 0.6)[:, 0].double()
    o0 = (1 - lam.double())[None, :, None] * v[:, 0].double()
    want = 0.4 * o0 / torch.sqrt((o0 ** 2).mean(-1, keepdim=True) + 1e-5)
    assert_bf16_close(got, want.numpy(), "row 0")


def test_prefill_bf16_writes_nothing_outside_its_output():
    inp = W.make_prefill_inputs(W.GDA3_PREFILL_L2048, B=1, L=130, h_s=3, h_n=1, seed=17)
    q1, k1, q2, k2, v, lam = to_cuda(inp)
    n = v.numel()
    guard = torch.full((n + 2 * 4096,), 7.0, dtype=torch.bfloat16, device="cuda")
    out = guard[4096:4096 + n].view_as(v)
    gda.gda_attn_fwd(q1, k1, q2, k2, v, lam, 0.8, out=out)
    torch.cuda.synchronize()
    assert torch.all(guard[:4096] == 7.0) and torch.all(guard[4096 + n:] == 7.0)


def test_prefill_f32_diff_attention_workload(oracle_mod):
    """The float32 Diff-attention workload on every element; also the plain
    relative bound 1e-4 wherever it is well defined (|ref| at least the
    row's rms, away from the output's zero crossings)."""
    w = W.DIFF_F32_L128
    inp = W.make_prefill_inputs(w)
    got = run_f32(inp, w.lambda_init, w.causal, w.eps)
    ref = oracle_mod.prefill(*inp, w.lambda_init, causal=w.causal, eps=w.eps)
    assert_f32_close(got, ref, w.name)
    g64 = got.double().numpy()
    rms = np.sqrt(np.mean(ref * ref, axis=-1, keepdims=True))
    big = np.abs(ref) >= rms
    rel = np.abs(g64 - ref)[big] / np.abs(ref)[big]
    print(f"float32 prefill, {int(big.sum())} elements with |ref| >= rms_row: "
          f"largest relative error {rel.max():.3e}")
    assert rel.max() <= 1e-4


SMALL_F32 = [  # B, L, h_s, h_n, d, dv, causal
    (1, 1, 2, 2, 64, 128, True),
    (2, 37, 6, 2, 64, 128, True),
    (1, 129, 6, 3, 64, 128, False),
    (1, 70, 4, 1, 128, 256, True),
    (2, 45, 3, 3, 24, 96, True),
]


@pytest.mark.parametrize("shape", SMALL_F32)
def test_prefill_f32_matches_oracle(oracle_mod, shape):
    B, L, hs, hn, d, dv, causal = shape
    inp = W.make_prefill_inputs(W.DIFF_F32_L128, B=B, L=L, h_s=hs, h_n=hn, d=d, dv=dv, seed=L)
    got = run_f32(inp, 0.7, causal)
    ref = oracle_mod.prefill(*inp, 0.7, causal=causal)
    assert_f32_close(got, ref, str(shape))


def test_prefill_f32_equal_maps_cancel():
    q1, k1, _, _, v, lam = W.make_prefill_inputs(W.DIFF_F32_L128, B=1, L=77, h_s=2, h_n=2, seed=3)
    got = run_f32((q1, k1, q1, k1, v, torch.ones_like(lam)), 0.8, flags=gda.GDA_FLAG_NO_NORM)
    assert torch.count_nonzero(got) == 0


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("B,L", [(1, 600), (8, 1280)], ids=["one_head_items", "whole_group_items"])
def test_prefill_bf16_rising_and_falling_scores(oracle_mod, causal, B, L):
    """Scores that climb ~230 log2 units along the keys (2^230 overflows float32
    unless the kernel moves its reference maximum as the row goes on) for the
    signal map, and fall as steeply for the noise map (later keys underflow).
    B=1, L=600 gives the grouped kernel items of one signal head; B=8, L=1280
    (160 whole-group items) items of the whole 3-head group."""
    hs, hn, d, dv = 3, 1, 64, 128
    g = torch.Generator().manual_seed(23)
    t = torch.linspace(-1.0, 20.0, L)
    q1 = torch.ones(B, L, hs, d) + 0.05 * torch.randn(B, L, hs, d, generator=g)
    k1 = t[None, :, None, None] * torch.ones(B, L, hs, d)
    q2 = torch.ones(B, L, hn, d) + 0.05 * torch.randn(B, L, hn, d, generator=g)
    k2 = -t[None, :, None, None] * torch.ones(B, L, hn, d)
    v = torch.randn(B, L, hs, dv, generator=g)
    lam = torch.tensor([0.3, 0.5, 0.7])
    bf = torch.bfloat16
    inp = (q1.to(bf), k1.to(bf), q2.to(bf), k2.to(bf), v.to(bf), lam)
    got = run_bf16(inp, 0.8, causal)
    assert torch.isfinite(got.float()).all()
    ref = oracle_mod.prefill(*inp, 0.8, causal=causal)
    assert_bf16_close(got, ref, "rising/falling scores")
