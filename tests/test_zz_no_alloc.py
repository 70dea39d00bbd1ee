"""The decode entry point that allocates nothing (gda_attn_decode_noalloc).

It serves callers that cannot allocate device memory (a plugin or serving
loop whose framework owns all device memory, or code that must not call
cudaMalloc/cudaFree because they can synchronise the device).  Its split
partials live in a fixed scratch array inside the library.  This file runs
last: it checks, through the C ABI, that two calls in a row match the regular
workspace-taking decode within the bf16 tolerance of the other tests, that a
call reads nothing an earlier, larger call left in the array, and that sizes
beyond the scratch array are refused.
"""
import ctypes
import dataclasses

import pytest
import torch

import grouped_differential_attention_gb300 as gda
from grouped_differential_attention_gb300 import workloads as W
from parity import assert_bf16_close

pytestmark = pytest.mark.gpu

GDA_ERR_WORKSPACE = -4
SCRATCH_BYTES = 32 << 20


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, q1, q2, k1c, k2c, vc, lens, lam, w, out):
    B, Lcap = k1c.shape[0], k1c.shape[1]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.gda_attn_decode_noalloc(_p(q1), _p(q2), _p(k1c), _p(k2c), _p(vc), _p(lens), _p(lam),
                                       ctypes.c_float(w.lambda_init), _p(out), B, Lcap, w.h_s, w.h_n,
                                       w.d, w.dv, ctypes.c_float(w.eps), stream)


@pytest.fixture(scope="module")
def lib():
    from grouped_differential_attention_gb300 import build
    build.build()
    return gda._load()


def test_no_alloc_decode_matches_workspace_decode(lib):
    gda.gda_device_error(clear=True)
    w = W.GDA3_DECODE_B64
    B, Lcap = 64, 8192
    # the 64-sequence decode workload's split partials: about 8.3 MB of the 32 MiB array
    need = gda.gda_attn_decode_workspace_size(B, Lcap, w.h_s, w.h_n, w.dv)
    assert 8_000_000 < need < 8_700_000
    assert need <= SCRATCH_BYTES
    q1, q2, k1c, k2c, vc, lens, lam = (t.cuda() for t in W.make_decode_inputs(w, seed=11))
    ref = gda.gda_attn_decode(q1, q2, k1c, k2c, vc, lens, lam, w.lambda_init, eps=w.eps)
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        rc = _noalloc(lib, q1, q2, k1c, k2c, vc, lens, lam, w, out)
        assert rc == 0, gda.gda_status_string(rc)
        torch.cuda.synchronize()
        assert_bf16_close(out.cpu(), ref.cpu().double().numpy(), f"no-alloc decode, call {call}")
    assert gda.gda_device_error(clear=True) == 0


def test_no_alloc_decode_reads_nothing_left_by_an_earlier_call(lib):
    """The scratch array keeps the previous call's partials.  A call with
    another batch size, other (short, ragged) lengths and other values must
    not read them: its result equals the workspace decode run on a fresh
    workspace filled with NaN bytes, so any value read before it was written
    would show up as NaN there or as a mismatch here."""
    gda.gda_device_error(clear=True)
    w = W.GDA3_DECODE_B64
    big = [t.cuda() for t in W.make_decode_inputs(w, seed=12)]
    out_big = torch.empty((w.B, w.h_s, w.dv), dtype=torch.bfloat16, device="cuda")
    assert _noalloc(lib, *big, w, out_big) == 0
    small = dataclasses.replace(w, B=5, Lcap=512, len_range=(1, 500), seed=13)
    q1, q2, k1c, k2c, vc, lens, lam = (t.cuda() for t in W.make_decode_inputs(small))
    need = gda.gda_attn_decode_workspace_size(small.B, small.Lcap, w.h_s, w.h_n, w.dv)
    fresh = torch.full((max(need, 16),), 0xFF, dtype=torch.uint8, device="cuda")
    ref = gda.gda_attn_decode(q1, q2, k1c, k2c, vc, lens, lam, w.lambda_init, eps=w.eps, workspace=fresh)
    out = torch.full_like(ref, float("nan"))
    assert _noalloc(lib, q1, q2, k1c, k2c, vc, lens, lam, small, out) == 0
    torch.cuda.synchronize()
    assert torch.isfinite(ref.float()).all()
    assert_bf16_close(out.cpu(), ref.cpu().double().numpy(), "no-alloc decode after a larger call")
    assert gda.gda_device_error(clear=True) == 0


def test_no_alloc_decode_refuses_sizes_beyond_its_scratch(lib):
    B, Lcap, hs, hn, dv = 4096, 16384, 12, 4, 128   # partials of ~4400 segment slots
    assert gda.gda_attn_decode_workspace_size(B, Lcap, hs, hn, dv) > SCRATCH_BYTES
    A = ctypes.c_void_p(0x10000)   # never dereferenced: the size check comes first
    rc = lib.gda_attn_decode_noalloc(A, A, A, A, A, A, A, ctypes.c_float(0.8), A, B, Lcap, hs, hn,
                                     64, dv, ctypes.c_float(1e-5), None)
    assert rc == GDA_ERR_WORKSPACE
