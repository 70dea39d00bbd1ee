"""The decode entry point that allocates nothing (gda_attn_decode_noalloc).

It serves callers that cannot allocate device memory (a plugin or serving
loop whose framework owns all device memory, or code that must not call
cudaMalloc/cudaFree because they can synchronise the device).  Its split
partials live in a fixed scratch array inside the library.  This file runs
last: it checks, through the C ABI, that two calls in a row match the regular
workspace-taking decode within the bf16 tolerance of the other tests, and
that sizes beyond the scratch array are refused.
"""
import ctypes

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


def test_no_alloc_decode_matches_workspace_decode():
    from grouped_differential_attention_gb300 import build
    build.build()
    lib = gda._load()
    gda.gda_device_error(clear=True)
    w = W.GDA3_DECODE_B64
    B, Lcap = 64, 8192            # the 64-sequence decode workload: ~25 MB of partials
    need = gda.gda_attn_decode_workspace_size(B, Lcap, w.h_s, w.h_n, w.dv)
    assert 0 < need <= SCRATCH_BYTES
    q1, q2, k1c, k2c, vc, lens, lam = (t.cuda() for t in W.make_decode_inputs(w, seed=11))
    ref = gda.gda_attn_decode(q1, q2, k1c, k2c, vc, lens, lam, w.lambda_init, eps=w.eps)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        rc = lib.gda_attn_decode_noalloc(_p(q1), _p(q2), _p(k1c), _p(k2c), _p(vc), _p(lens), _p(lam),
                                         ctypes.c_float(w.lambda_init), _p(out), B, Lcap, w.h_s, w.h_n,
                                         w.d, w.dv, ctypes.c_float(w.eps), stream)
        assert rc == 0, gda.gda_status_string(rc)
        torch.cuda.synchronize()
        assert_bf16_close(out.cpu(), ref.cpu().double().numpy(), f"no-alloc decode, call {call}")
    assert gda.gda_device_error(clear=True) == 0


def test_no_alloc_decode_refuses_sizes_beyond_its_scratch():
    lib = gda._load()
    B, Lcap, hs, hn, dv = 4096, 16384, 12, 4, 128   # partials of ~4400 segment slots
    assert gda.gda_attn_decode_workspace_size(B, Lcap, hs, hn, dv) > SCRATCH_BYTES
    A = ctypes.c_void_p(0x10000)   # never dereferenced: the size check comes first
    rc = lib.gda_attn_decode_noalloc(A, A, A, A, A, A, A, ctypes.c_float(0.8), A, B, Lcap, hs, hn,
                                     64, dv, ctypes.c_float(1e-5), None)
    assert rc == GDA_ERR_WORKSPACE
