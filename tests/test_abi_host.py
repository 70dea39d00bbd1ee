"""Host-side checks of the C ABI: the library builds for sm_103a, loads
without a GPU, exports every symbol of include/gda.h, and rejects bad
arguments with the documented status codes before touching CUDA."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gda.h")

OK, INVALID, UNSUPPORTED, MISALIGNED, WORKSPACE, CUDA = 0, -1, -2, -3, -4, -5


@pytest.fixture(scope="module")
def lib():
    from grouped_differential_attention_gb300 import build
    path = build.build()
    import grouped_differential_attention_gb300 as gda
    assert os.path.samefile(path, gda.library_path())
    return gda._load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gda_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("gda_attn_fwd", "gda_attn_fwd_f32", "gda_attn_decode",
              "gda_attn_decode_workspace_size", "gda_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_library_is_built_for_sm103a(lib):
    from grouped_differential_attention_gb300 import build
    flags = build.compile_flags()
    i = flags.index("-gencode")
    assert flags[i + 1] == "arch=compute_103a,code=sm_103a"
    assert flags.count("-gencode") == 1


def test_status_strings(lib):
    import grouped_differential_attention_gb300 as gda
    assert gda.gda_status_string(0) == "success"
    for code in (-1, -2, -3, -4, -5, -6):
        assert gda.gda_status_string(code) not in ("success", "unknown status")
    assert gda.gda_status_string(42) == "unknown status"


A = 0x10000  # fake, 16-byte aligned addresses: never dereferenced on these paths


def fwd(lib, entry="gda_attn_fwd", ptrs=None, B=1, L=128, hs=6, hn=2, d=64, dv=128, causal=1,
        eps=1e-5, lam_init=0.8):
    p = ptrs or [A, A + 16, A + 32, A + 48, A + 64, A + 80, A + 96]
    q1, k1, q2, k2, v, lam, out = (ctypes.c_void_p(x) if x is not None else None for x in p)
    return getattr(lib, entry)(q1, k1, q2, k2, v, lam, ctypes.c_float(lam_init), out, B, L, hs, hn,
                               d, dv, causal, ctypes.c_float(eps), None)


@pytest.mark.parametrize("entry", ["gda_attn_fwd", "gda_attn_fwd_f32"])
def test_prefill_rejects_bad_arguments(lib, entry):
    assert fwd(lib, entry, ptrs=[None, A, A, A, A, A, A]) == INVALID
    assert fwd(lib, entry, ptrs=[A, A, A, A, A, A, None]) == INVALID
    assert fwd(lib, entry, B=0) == INVALID
    assert fwd(lib, entry, L=0) == INVALID
    assert fwd(lib, entry, hs=6, hn=4) == INVALID
    assert fwd(lib, entry, causal=2) == INVALID
    assert fwd(lib, entry, eps=-1.0) == INVALID
    assert fwd(lib, entry, eps=float("nan")) == INVALID
    assert fwd(lib, entry, lam_init=float("inf")) == INVALID
    assert fwd(lib, entry, ptrs=[A, A, A + 8, A, A, A, A]) == MISALIGNED
    assert fwd(lib, entry, ptrs=[A, A, A, A, A, A + 4, A]) == MISALIGNED


def test_prefill_rejects_unsupported_dims(lib):
    assert fwd(lib, d=96) == UNSUPPORTED
    assert fwd(lib, dv=64) == UNSUPPORTED
    assert fwd(lib, "gda_attn_fwd_f32", dv=48) == UNSUPPORTED
    assert fwd(lib, "gda_attn_fwd_f32", d=512) == UNSUPPORTED


def test_ex_rejects_unknown_flags(lib):
    P = [ctypes.c_void_p(A)] * 5
    rc = lib.gda_attn_fwd_ex(*P, ctypes.c_void_p(A), ctypes.c_float(0.8), ctypes.c_void_p(A),
                             1, 128, 6, 2, 64, 128, 1, ctypes.c_float(1e-5), 0x80, None)
    assert rc == INVALID


def test_single_pass_flag_only_on_the_forward_entries(lib):
    P = [ctypes.c_void_p(A)] * 5
    F, U = ctypes.c_float, ctypes.c_uint
    # accepted by gda_attn_fwd_ex (validation passes; without a GPU the call then reports a CUDA error)
    rc = lib.gda_attn_fwd_ex(*P, ctypes.c_void_p(A), F(0.8), ctypes.c_void_p(A), 1, 128, 6, 2, 64, 256, 1,
                             F(1e-5), U(0x2), None)
    assert rc != INVALID
    # refused by the entries it does not apply to
    assert lib.gda_attn_fwd_f32_ex(*P, ctypes.c_void_p(A), F(0.8), ctypes.c_void_p(A), 1, 128, 6, 2, 64, 128, 1,
                                   F(1e-5), U(0x2), None) == INVALID
    assert lib.gda_attn_fwd_chunk(*P, ctypes.c_void_p(A), F(0.8), ctypes.c_void_p(A), 1, 128, 128, 6, 2, 64, 256,
                                  1, F(1e-5), U(0x2), None) != INVALID
    assert lib.gda_attn_fwd_chunk(*P, ctypes.c_void_p(A), F(0.8), ctypes.c_void_p(A), 1, 128, 128, 6, 2, 64, 256,
                                  1, F(1e-5), U(0x4), None) == INVALID
    assert lib.gda_attn_fwd_2pass(*P, ctypes.c_void_p(A), F(0.8), ctypes.c_void_p(A), 1, 128, 6, 2, 64, 256, 1,
                                  F(1e-5), U(0x2), ctypes.c_void_p(A), 1 << 20, None) == INVALID


def decode(lib, ws_bytes=None, ws=A, B=4, Lcap=256, hs=6, hn=2, d=64, dv=128, ptrs=None):
    need = lib.gda_attn_decode_workspace_size(B, Lcap, hs, hn, dv)
    p = ptrs or [A] * 8
    q1, q2, k1, k2, v, lens, lam, out = (ctypes.c_void_p(x) if x is not None else None for x in p)
    return lib.gda_attn_decode(q1, q2, k1, k2, v, lens, lam, ctypes.c_float(0.8), out, B, Lcap, hs,
                               hn, d, dv, ctypes.c_float(1e-5),
                               ctypes.c_void_p(ws) if ws is not None else None,
                               need if ws_bytes is None else ws_bytes, None)


def test_decode_workspace_size(lib):
    n = lib.gda_attn_decode_workspace_size(64, 8192, 12, 4, 128)
    # one slot per sequence at least: 12 heads x 2 accumulators x 128 floats,
    # plus (m, l) for 16 heads
    assert n >= 64 * (12 * 2 * 128 + 16 * 2) * 4
    # the slots do not depend on the cache length
    assert lib.gda_attn_decode_workspace_size(64, 128, 12, 4, 128) == n
    assert n % 16 == 0
    assert lib.gda_attn_decode_workspace_size(0, 8192, 12, 4, 128) == 0
    assert lib.gda_attn_decode_workspace_size(64, 8192, 12, 5, 128) == 0


def test_decode_rejects_bad_arguments(lib):
    assert decode(lib, ptrs=[A] * 5 + [None, A, A]) == INVALID
    assert decode(lib, hs=6, hn=4) == INVALID
    assert decode(lib, d=96) == UNSUPPORTED
    assert decode(lib, dv=96) == UNSUPPORTED
    assert decode(lib, ptrs=[A, A, A, A, A + 2, A, A, A]) == MISALIGNED
    assert decode(lib, ws=None) == WORKSPACE
    assert decode(lib, ws_bytes=16) == WORKSPACE
    assert decode(lib, ws=A + 8) == WORKSPACE


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_valid_call_without_a_gpu_reports_cuda_error(lib):
    assert fwd(lib) == CUDA
    assert decode(lib) == CUDA


def test_binding_checks_tensors_before_the_library():
    import grouped_differential_attention_gb300 as gda
    x = torch.zeros(1, 4, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        gda.gda_attn_fwd(x, x, x, x, torch.zeros(1, 4, 2, 128, dtype=torch.bfloat16),
                         torch.zeros(2), 0.8)


def test_lambda_reparam_rejects_bad_arguments(lib):
    # every call below fails validation before any device work
    F = ctypes.c_float
    P = [ctypes.c_void_p(A)] * 4
    out = ctypes.c_void_p(A)
    assert lib.gda_lambda_reparam(None, *P[1:], F(0.8), out, 12, 64, None) == INVALID
    assert lib.gda_lambda_reparam(*P, F(0.8), None, 12, 64, None) == INVALID
    assert lib.gda_lambda_reparam(*P, F(0.8), out, 0, 64, None) == INVALID
    assert lib.gda_lambda_reparam(*P, F(0.8), out, 12, 0, None) == INVALID
    assert lib.gda_lambda_reparam(*P, F(float("nan")), out, 12, 64, None) == INVALID
    assert lib.gda_lambda_reparam(ctypes.c_void_p(A + 2), *P[1:], F(0.8), out, 12, 64, None) == MISALIGNED


def test_decode_fp8_rejects_bad_arguments(lib):
    # every call below fails validation before any device work
    F, Z = ctypes.c_float, ctypes.c_size_t
    a = [ctypes.c_void_p(A)] * 10
    ws = ctypes.c_void_p(A)
    need = lib.gda_attn_decode_workspace_size(4, 256, 6, 2, 128)

    def call(ptrs=None, B=4, Lcap=256, hs=6, hn=2, d=64, dv=128, ws_ptr=ws, ws_bytes=None):
        p = ptrs or a
        return lib.gda_attn_decode_fp8(*p, F(0.8), ctypes.c_void_p(A), B, Lcap, hs, hn, d, dv, F(1e-5),
                                       ws_ptr, need if ws_bytes is None else ws_bytes, None)
    assert call(ptrs=[None] + a[1:]) == INVALID
    assert call(ptrs=a[:5] + [None] + a[6:]) == INVALID          # a missing scale array
    assert call(hs=6, hn=4) == INVALID
    assert call(d=96) == UNSUPPORTED
    assert call(ptrs=a[:2] + [ctypes.c_void_p(A + 8)] + a[3:]) == MISALIGNED
    assert call(ptrs=a[:6] + [ctypes.c_void_p(A + 2)] + a[7:]) == MISALIGNED   # scale not 4-byte aligned
    assert call(ws_ptr=None) == WORKSPACE
    assert call(ws_bytes=16) == WORKSPACE


def test_decode_paged_rejects_bad_arguments(lib):
    # every call below fails validation before any device work
    F = ctypes.c_float
    a = [ctypes.c_void_p(A)] * 8
    ws = ctypes.c_void_p(A)
    need = lib.gda_attn_decode_workspace_size(4, 256, 6, 2, 128)

    def call(ptrs=None, B=4, max_pages=8, page_size=32, num_pages=40, hs=6, hn=2, d=64, dv=128, ws_ptr=ws,
             ws_bytes=None):
        p = ptrs or a
        return lib.gda_attn_decode_paged(*p, F(0.8), ctypes.c_void_p(A), B, max_pages, page_size, num_pages,
                                         hs, hn, d, dv, F(1e-5), ws_ptr, need if ws_bytes is None else ws_bytes,
                                         None)
    assert call(ptrs=a[:5] + [None] + a[6:]) == INVALID           # no block table
    assert call(page_size=0) == INVALID
    assert call(num_pages=0) == INVALID
    assert call(hs=6, hn=4) == INVALID
    assert call(dv=96) == UNSUPPORTED
    assert call(ptrs=a[:5] + [ctypes.c_void_p(A + 2)] + a[6:]) == MISALIGNED
    assert call(ws_bytes=16) == WORKSPACE


def test_chunked_prefill_rejects_bad_arguments(lib):
    # every call below fails validation before any device work
    F, U = ctypes.c_float, ctypes.c_uint
    P = [ctypes.c_void_p(A)] * 6

    def call(L=128, Lk=512, causal=1, hs=6, hn=2, d=64, dv=128):
        return lib.gda_attn_fwd_chunk(*P, F(0.8), ctypes.c_void_p(A), 2, L, Lk, hs, hn, d, dv, causal,
                                      F(1e-5), U(0), None)
    assert call(Lk=0) == INVALID
    assert call(L=128, Lk=100) == INVALID            # causal chunk longer than its sequence
    assert call(hs=6, hn=4) == INVALID
    assert call(d=96) == UNSUPPORTED
    assert call(dv=64) == UNSUPPORTED


def test_chunked_two_pass_prefill_checks_arguments_and_workspace(lib):
    # every call below fails validation before any device work
    F, U, Z = ctypes.c_float, ctypes.c_uint, ctypes.c_size_t
    P = [ctypes.c_void_p(A)] * 6
    lib.gda_attn_fwd_chunk_2pass.argtypes = [ctypes.c_void_p] * 6 + [F, ctypes.c_void_p] + [ctypes.c_int] * 8 + [
        F, U, ctypes.c_void_p, Z, ctypes.c_void_p]

    def call(L=128, Lk=512, causal=1, hs=6, hn=2, d=64, dv=256, ws=A, ws_bytes=None, flags=0):
        need = lib.gda_attn_fwd_2pass_workspace_size(2, L, hs, hn)
        return lib.gda_attn_fwd_chunk_2pass(*P, F(0.8), ctypes.c_void_p(A), 2, L, Lk, hs, hn, d, dv, causal,
                                            F(1e-5), U(flags), ctypes.c_void_p(ws) if ws else None,
                                            need if ws_bytes is None else ws_bytes, None)
    assert call(Lk=0) == INVALID
    assert call(L=128, Lk=100) == INVALID
    assert call(hs=6, hn=4) == INVALID
    assert call(d=96) == UNSUPPORTED
    assert call(flags=0x2) == INVALID                 # the single-pass flag does not apply here
    assert call(ws=None) == WORKSPACE
    assert call(ws=A + 8) == WORKSPACE
    assert call(ws_bytes=lib.gda_attn_fwd_2pass_workspace_size(2, 128, 6, 2) - 4) == WORKSPACE


def test_backward_workspace_size(lib):
    assert lib.gda_attn_bwd_workspace_size(0, 128, 6, 64, 128) == 0
    assert lib.gda_attn_bwd_workspace_size(2, 128, 6, 64, -1) == 0
    small = lib.gda_attn_bwd_workspace_size(2, 128, 6, 64, 128)
    big = lib.gda_attn_bwd_workspace_size(2, 256, 6, 64, 128)
    # per (b, row, signal head): 6 statistics, dv of dL/do, 2 d of noise-gradient shares, 1 dlambda term
    assert small >= 4 * 2 * 128 * 6 * (6 + 128 + 2 * 64 + 1)
    assert big > small


def test_backward_rejects_bad_arguments(lib):
    # every call below fails validation before any device work
    F, U = ctypes.c_float, ctypes.c_uint
    P = [ctypes.c_void_p(A)] * 6

    def call(first=None, grads=None, L=128, hs=6, hn=2, d=64, dv=128, causal=1, eps=1e-5, flags=0,
             ws=ctypes.c_void_p(A), ws_bytes=1 << 30):
        ins = first if first is not None else P
        outs = grads if grads is not None else P
        return lib.gda_attn_bwd(*ins, F(0.8), ctypes.c_void_p(A), *outs, 2, L, hs, hn, d, dv, causal,
                                F(eps), U(flags), ws, ws_bytes, None)
    assert call(first=[None] + P[1:]) == INVALID
    assert call(grads=P[:5] + [None]) == INVALID
    assert call(L=0) == INVALID
    assert call(hs=6, hn=4) == INVALID
    assert call(causal=2) == INVALID
    assert call(eps=-1.0) == INVALID
    assert call(flags=0x10) == INVALID
    assert call(d=96) == UNSUPPORTED
    assert call(dv=96) == UNSUPPORTED
    assert call(grads=P[:4] + [ctypes.c_void_p(A + 4), P[5]]) == MISALIGNED
    assert call(ws=None) == WORKSPACE
    assert call(ws_bytes=16) == WORKSPACE


def test_two_pass_prefill_rejects_bad_arguments(lib):
    # every call below fails validation before any device work
    F, U = ctypes.c_float, ctypes.c_uint
    P = [ctypes.c_void_p(A)] * 6

    def call(L=128, hs=6, hn=2, d=64, dv=128, causal=1, ws=ctypes.c_void_p(A), ws_bytes=1 << 30, first=None):
        ins = first if first is not None else P
        return lib.gda_attn_fwd_2pass(*ins, F(0.8), ctypes.c_void_p(A), 2, L, hs, hn, d, dv, causal, F(1e-5),
                                      U(0), ws, ws_bytes, None)
    assert lib.gda_attn_fwd_2pass_workspace_size(2, 128, 6, 2) == 4 * 2 * 128 * 8
    assert lib.gda_attn_fwd_2pass_workspace_size(2, 0, 6, 2) == 0
    assert call(first=[None] + P[1:]) == INVALID
    assert call(L=0) == INVALID
    assert call(hs=6, hn=4) == INVALID
    assert call(causal=3) == INVALID
    assert call(d=96) == UNSUPPORTED
    assert call(dv=64) == UNSUPPORTED
    assert call(first=[ctypes.c_void_p(A + 8)] + P[1:]) == MISALIGNED
    assert call(ws=None) == WORKSPACE
    assert call(ws_bytes=4 * 2 * 128 * 8 - 4) == WORKSPACE
    assert call(ws=ctypes.c_void_p(A + 4)) == WORKSPACE


def test_decode_paged_fp8_rejects_bad_arguments(lib):
    # every call below fails validation before any device work
    F = ctypes.c_float

    def call(first=None, B=2, max_pages=4, page_size=16, num_pages=9, hs=6, hn=2, d=64, dv=128, scale_off=0,
             ws=ctypes.c_void_p(A), ws_bytes=1 << 30):
        ptrs = first if first is not None else [ctypes.c_void_p(A)] * 5
        scales = [ctypes.c_void_p(A + scale_off)] * 3
        return lib.gda_attn_decode_paged_fp8(*ptrs, *scales, ctypes.c_void_p(A), ctypes.c_void_p(A),
                                             ctypes.c_void_p(A), F(0.8), ctypes.c_void_p(A), B, max_pages, page_size,
                                             num_pages, hs, hn, d, dv, F(1e-5), ws, ws_bytes, None)
    assert call(first=[None] + [ctypes.c_void_p(A)] * 4) == INVALID
    assert call(page_size=0) == INVALID
    assert call(hs=6, hn=4) == INVALID
    assert call(d=96) == UNSUPPORTED
    assert call(scale_off=2) == MISALIGNED
    assert call(ws=None) == WORKSPACE
    assert call(ws_bytes=16) == WORKSPACE


def test_binding_refuses_host_tensors_for_every_entry():
    """Every binding refuses CPU tensors before calling the library (there is
    no CPU fallback)."""
    import grouped_differential_attention_gb300 as gda
    bf, f32 = torch.bfloat16, torch.float32
    q = torch.zeros(1, 4, 2, 64, dtype=bf)
    v = torch.zeros(1, 4, 2, 128, dtype=bf)
    lam = torch.zeros(2)
    qf, vf = q.float(), v.float()
    calls = [
        lambda: gda.gda_attn_fwd_2pass(q, q, q, q, v, lam, 0.8),
        lambda: gda.gda_attn_fwd_chunk(q, q, q, q, v, lam, 0.8),
        lambda: gda.gda_attn_fwd_f32(qf, qf, qf, qf, vf, lam, 0.8),
        lambda: gda.gda_attn_bwd(qf, qf, qf, qf, vf, lam, 0.8, vf),
        lambda: gda.gda_attn_bwd_bf16(q, q, q, q, v, lam, 0.8, v),
    ]
    qd = torch.zeros(1, 2, 64, dtype=bf)
    cache = torch.zeros(1, 16, 2, 64, dtype=torch.uint8)
    vcache = torch.zeros(1, 16, 2, 128, dtype=torch.uint8)
    lens = torch.ones(1, dtype=torch.int32)
    sc = torch.ones(2, dtype=f32)
    table = torch.zeros(1, 1, dtype=torch.int32)
    calls += [
        lambda: gda.gda_attn_decode_fp8(qd, qd, cache, cache, vcache, sc, sc, sc, lens, lam, 0.8),
        lambda: gda.gda_attn_decode_paged_fp8(qd, qd, cache, cache, vcache, sc, sc, sc, table, lens, lam, 0.8),
    ]
    for call in calls:
        with pytest.raises((ValueError, TypeError)):
            call()
