"""Grouped differential attention on NVIDIA GB300 (sm_103a).

Python binding of ``libgda.so`` (C ABI in ``include/gda.h``).  The functions
below carry the C names and only marshal arguments: they check dtypes,
shapes, devices and contiguity on the PyTorch side, then pass raw device
pointers and the current CUDA stream to the library, whose kernels do every
step of the computation.  There is no CPU or PyTorch fallback: if the
library is missing, every call raises.

Operation (see ``include/gda.h``): for signal head h with noise head
g = h // (h_s // h_n),

    y_h = (1 - lambda_init) * RMSNorm( (softmax(Q1_h K1_h^T / sqrt d)
                                        - lambda_h softmax(Q2_g K2_g^T / sqrt d)) V_h )

Layouts: q_sig, k_sig [B, L, h_s, d]; q_noise, k_noise [B, L, h_n, d];
v and the output [B, L, h_s, dv]; lambda [h_s] float32.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = [
    "GDAError", "gda_attn_fwd", "gda_attn_fwd_f32", "gda_attn_decode",
    "gda_attn_decode_workspace_size", "gda_status_string", "gda_device_error",
    "library_path", "GDA_FLAG_NO_NORM", "GDA_FLAG_SINGLE_PASS",
    "gda_attn_decode_noalloc",
    "gda_attn_bwd", "gda_attn_bwd_workspace_size", "gda_attn_fwd_2pass",
    "gda_attn_fwd_2pass_workspace_size", "gda_attn_bwd_bf16", "gda_attn_bwd_bf16_workspace_size",
    "gda_attn_decode_paged_fp8", "gda_attn_fwd_chunk", "gda_attn_fwd_chunk_2pass",
]

GDA_OK = 0
GDA_ERR_INVALID_ARG = -1
GDA_ERR_UNSUPPORTED = -2
GDA_ERR_MISALIGNED = -3
GDA_ERR_WORKSPACE = -4
GDA_ERR_CUDA = -5
GDA_ERR_DEVICE_TIMEOUT = -6
GDA_FLAG_NO_NORM = 0x1
GDA_FLAG_SINGLE_PASS = 0x2
GDA_DEVERR_PREFILL_TIMEOUT = 0x1
GDA_DEVERR_BAD_LENGTH = 0x2
GDA_DEVERR_DECODE_TIMEOUT = 0x4
GDA_DEVERR_BAD_PAGE = 0x8

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "libgda.so")
_lock = threading.Lock()
_lib = None


class GDAError(RuntimeError):
    def __init__(self, status: int, what: str):
        extra = ""
        if status == GDA_ERR_CUDA:
            extra = f", cudaError {_load().gda_last_cuda_error()}"
        super().__init__(f"{what}: {gda_status_string(status)} (status {status}{extra})")
        self.status = status


def library_path() -> str:
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(
                    f"{_LIB_PATH} is missing: build it with "
                    "`python -m grouped_differential_attention_gb300.build`")
            lib = ctypes.CDLL(_LIB_PATH)
            P, I, F, U, Z = (ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_uint,
                             ctypes.c_size_t)
            fwd = [P, P, P, P, P, P, F, P, I, I, I, I, I, I, I, F]
            lib.gda_attn_fwd.argtypes = fwd + [P]
            lib.gda_attn_fwd_ex.argtypes = fwd + [U, P]
            lib.gda_attn_fwd_f32.argtypes = fwd + [P]
            lib.gda_attn_fwd_f32_ex.argtypes = fwd + [U, P]
            lib.gda_attn_decode_workspace_size.argtypes = [I, I, I, I, I]
            lib.gda_attn_decode_workspace_size.restype = Z
            lib.gda_attn_decode.argtypes = [P, P, P, P, P, P, P, F, P, I, I, I, I, I, I, F, P, Z, P]
            lib.gda_status_string.argtypes = [I]
            lib.gda_status_string.restype = ctypes.c_char_p
            lib.gda_attn_decode_noalloc.argtypes = [P, P, P, P, P, P, P, F, P, I, I, I, I, I, I, F, P]
            lib.gda_attn_decode_noalloc.restype = I
            lib.gda_attn_decode_fp8.argtypes = [P, P, P, P, P, P, P, P, P, P, F, P, I, I, I, I, I, I, F,
                                                P, Z, P]
            lib.gda_attn_decode_fp8.restype = I
            lib.gda_attn_decode_paged.argtypes = [P, P, P, P, P, P, P, P, F, P, I, I, I, I, I, I, I, I, F,
                                                  P, Z, P]
            lib.gda_attn_decode_paged.restype = I
            lib.gda_attn_fwd_chunk.argtypes = [P, P, P, P, P, P, F, P, I, I, I, I, I, I, I, I, F, U, P]
            lib.gda_attn_fwd_chunk.restype = I
            lib.gda_attn_fwd_chunk_2pass.argtypes = [P, P, P, P, P, P, F, P, I, I, I, I, I, I, I, I, F, U,
                                                     P, Z, P]
            lib.gda_attn_fwd_chunk_2pass.restype = I
            lib.gda_lambda_reparam.argtypes = [P, P, P, P, F, P, I, I, P]
            lib.gda_lambda_reparam.restype = I
            lib.gda_attn_decode_paged_fp8.argtypes = [P, P, P, P, P, P, P, P, P, P, P, F, P, I, I, I, I, I, I,
                                                      I, I, F, P, Z, P]
            lib.gda_attn_decode_paged_fp8.restype = I
            lib.gda_attn_fwd_2pass.argtypes = [P, P, P, P, P, P, F, P, I, I, I, I, I, I, I, F, U, P, Z, P]
            lib.gda_attn_fwd_2pass.restype = I
            lib.gda_attn_fwd_2pass_workspace_size.argtypes = [I, I, I, I]
            lib.gda_attn_fwd_2pass_workspace_size.restype = Z
            lib.gda_attn_bwd_bf16.argtypes = [P, P, P, P, P, P, F, P, P, P, P, P, P, P, I, I, I, I, I, I, I,
                                              F, U, P, Z, P]
            lib.gda_attn_bwd_bf16.restype = I
            lib.gda_attn_bwd_bf16_workspace_size.argtypes = [I, I, I, I, I]
            lib.gda_attn_bwd_bf16_workspace_size.restype = Z
            lib.gda_attn_bwd.argtypes = [P, P, P, P, P, P, F, P, P, P, P, P, P, P, I, I, I, I, I, I, I, F,
                                         U, P, Z, P]
            lib.gda_attn_bwd.restype = I
            lib.gda_attn_bwd_workspace_size.argtypes = [I, I, I, I, I]
            lib.gda_attn_bwd_workspace_size.restype = Z
            lib.gda_device_error.argtypes = [I]
            lib.gda_last_cuda_error.argtypes = []
            lib.gda_last_cuda_error.restype = I
            for name in ("gda_attn_fwd", "gda_attn_fwd_ex", "gda_attn_fwd_f32",
                         "gda_attn_fwd_f32_ex", "gda_attn_decode", "gda_device_error"):
                getattr(lib, name).restype = I
            _lib = lib
    return _lib


def gda_status_string(status: int) -> str:
    return _load().gda_status_string(int(status)).decode()


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check(rc: int, what: str):
    if rc != GDA_OK:
        raise GDAError(rc, what)


def _expect(t, name, dtype, shape, device):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _prefill(entry, dtype, q_sig, k_sig, q_noise, k_noise, v, lam, lambda_init, causal, eps,
             out, flags):
    dev = q_sig.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    if q_sig.dim() != 4 or q_noise.dim() != 4 or v.dim() != 4:
        raise ValueError("q_sig, q_noise and v must be 4-D [B, L, heads, dim]")
    B, L, hs, d = q_sig.shape
    hn = q_noise.shape[2]
    dv = v.shape[3]
    _expect(q_sig, "q_sig", dtype, (B, L, hs, d), dev)
    _expect(k_sig, "k_sig", dtype, (B, L, hs, d), dev)
    _expect(q_noise, "q_noise", dtype, (B, L, hn, d), dev)
    _expect(k_noise, "k_noise", dtype, (B, L, hn, d), dev)
    _expect(v, "v", dtype, (B, L, hs, dv), dev)
    _expect(lam, "lam", torch.float32, (hs,), dev)
    if out is None:
        out = torch.empty((B, L, hs, dv), dtype=dtype, device=dev)
    _expect(out, "out", dtype, (B, L, hs, dv), dev)
    with torch.cuda.device(dev):
        rc = entry(_ptr(q_sig), _ptr(k_sig), _ptr(q_noise), _ptr(k_noise), _ptr(v), _ptr(lam),
                   float(lambda_init), _ptr(out), B, L, hs, hn, d, dv, int(bool(causal)),
                   float(eps), int(flags), _stream(dev))
    _check(rc, "gda prefill")
    return out


def gda_attn_fwd(q_sig, k_sig, q_noise, k_noise, v, lam, lambda_init: float, *,
                 causal: bool = True, eps: float = 1e-5, out=None, flags: int = 0):
    """bf16 prefill on the tensor cores (tcgen05/TMEM, TMA); returns ``out``."""
    return _prefill(_load().gda_attn_fwd_ex, torch.bfloat16, q_sig, k_sig, q_noise, k_noise, v,
                    lam, lambda_init, causal, eps, out, flags)


def gda_attn_fwd_chunk(q_sig, k_sig, q_noise, k_noise, v, lam, lambda_init: float, *,
                       causal: bool = True, eps: float = 1e-5, out=None, flags: int = 0, workspace=None,
                       two_pass: bool = False):
    """Chunked bf16 prefill: L query rows at key positions Lk - L .. Lk - 1.

    q_sig [B, L, h_s, d], q_noise [B, L, h_n, d]; k_sig [B, Lk, h_s, d],
    k_noise [B, Lk, h_n, d], v [B, Lk, h_s, dv]; returns out [B, L, h_s, dv].
    ``two_pass`` calls gda_attn_fwd_chunk_2pass, whose statistics workspace
    (uint8 CUDA tensor of gda_attn_fwd_2pass_workspace_size(B, L, h_s, h_n)
    bytes) is ``workspace`` or allocated here.
    """
    dev = q_sig.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    B, L, hs, d = q_sig.shape
    hn = q_noise.shape[2]
    Lk = k_sig.shape[1]
    dv = v.shape[3]
    bf = torch.bfloat16
    _expect(q_sig, "q_sig", bf, (B, L, hs, d), dev)
    _expect(k_sig, "k_sig", bf, (B, Lk, hs, d), dev)
    _expect(q_noise, "q_noise", bf, (B, L, hn, d), dev)
    _expect(k_noise, "k_noise", bf, (B, Lk, hn, d), dev)
    _expect(v, "v", bf, (B, Lk, hs, dv), dev)
    _expect(lam, "lam", torch.float32, (hs,), dev)
    if out is None:
        out = torch.empty((B, L, hs, dv), dtype=bf, device=dev)
    _expect(out, "out", bf, (B, L, hs, dv), dev)
    args = (_ptr(q_sig), _ptr(k_sig), _ptr(q_noise), _ptr(k_noise), _ptr(v), _ptr(lam), float(lambda_init),
            _ptr(out), B, L, Lk, hs, hn, d, dv, int(bool(causal)), float(eps), int(flags))
    with torch.cuda.device(dev):
        if two_pass:
            need = gda_attn_fwd_2pass_workspace_size(B, L, hs, hn)
            if workspace is None:
                workspace = torch.empty((max(need, 16),), dtype=torch.uint8, device=dev)
            _expect(workspace, "workspace", torch.uint8, (workspace.numel(),), dev)
            rc = _load().gda_attn_fwd_chunk_2pass(*args, _ptr(workspace), workspace.numel(), _stream(dev))
        else:
            rc = _load().gda_attn_fwd_chunk(*args, _stream(dev))
    _check(rc, "gda chunked prefill")
    return out


def gda_attn_fwd_f32(q_sig, k_sig, q_noise, k_noise, v, lam, lambda_init: float, *,
                     causal: bool = True, eps: float = 1e-5, out=None, flags: int = 0):
    """float32 prefill on the CUDA cores; returns ``out``."""
    return _prefill(_load().gda_attn_fwd_f32_ex, torch.float32, q_sig, k_sig, q_noise, k_noise,
                    v, lam, lambda_init, causal, eps, out, flags)


def gda_attn_decode_fp8(q_sig, q_noise, k_sig_cache, k_noise_cache, v_cache, k_sig_scale,
                        k_noise_scale, v_scale, cache_lens, lam, lambda_init: float, *,
                        eps: float = 1e-5, out=None, workspace=None):
    """bf16 decode over fp8 (e4m3) caches: cached value = code * scale of its head.

    The caches are ``torch.float8_e4m3fn`` (or ``uint8`` holding the codes)
    CUDA tensors [B, Lcap, heads, dim]; scales are float32 [h_s], [h_n], [h_s].
    """
    dev = q_sig.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    B, hs, d = q_sig.shape
    hn = q_noise.shape[1]
    Lcap = k_sig_cache.shape[1]
    dv = v_cache.shape[3]
    bf = torch.bfloat16
    codes = []
    for t, name, shape in ((k_sig_cache, "k_sig_cache", (B, Lcap, hs, d)),
                           (k_noise_cache, "k_noise_cache", (B, Lcap, hn, d)),
                           (v_cache, "v_cache", (B, Lcap, hs, dv))):
        if t.dtype == torch.float8_e4m3fn:
            t = t.view(torch.uint8)
        _expect(t, name, torch.uint8, shape, dev)
        codes.append(t)
    _expect(q_sig, "q_sig", bf, (B, hs, d), dev)
    _expect(q_noise, "q_noise", bf, (B, hn, d), dev)
    _expect(k_sig_scale, "k_sig_scale", torch.float32, (hs,), dev)
    _expect(k_noise_scale, "k_noise_scale", torch.float32, (hn,), dev)
    _expect(v_scale, "v_scale", torch.float32, (hs,), dev)
    _expect(cache_lens, "cache_lens", torch.int32, (B,), dev)
    _expect(lam, "lam", torch.float32, (hs,), dev)
    if out is None:
        out = torch.empty((B, hs, dv), dtype=bf, device=dev)
    _expect(out, "out", bf, (B, hs, dv), dev)
    need = gda_attn_decode_workspace_size(B, Lcap, hs, hn, dv)
    if workspace is None:
        workspace = torch.empty((need,), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        rc = _load().gda_attn_decode_fp8(
            _ptr(q_sig), _ptr(q_noise), _ptr(codes[0]), _ptr(codes[1]), _ptr(codes[2]),
            _ptr(k_sig_scale), _ptr(k_noise_scale), _ptr(v_scale), _ptr(cache_lens), _ptr(lam),
            float(lambda_init), _ptr(out), B, Lcap, hs, hn, d, dv, float(eps), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _stream(dev))
    _check(rc, "gda decode (fp8 cache)")
    return out


def gda_attn_decode_paged(q_sig, q_noise, k_sig_pool, k_noise_pool, v_pool, block_table, cache_lens,
                          lam, lambda_init: float, *, eps: float = 1e-5, out=None, workspace=None):
    """bf16 decode over paged caches.

    Pools [num_pages, page_size, heads, dim] (bf16); block_table [B,
    max_pages] int32: position j of sequence b is row j % page_size of page
    block_table[b, j // page_size].
    """
    dev = q_sig.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    B, hs, d = q_sig.shape
    hn = q_noise.shape[1]
    num_pages, page_size = k_sig_pool.shape[0], k_sig_pool.shape[1]
    dv = v_pool.shape[3]
    max_pages = block_table.shape[1]
    bf = torch.bfloat16
    _expect(q_sig, "q_sig", bf, (B, hs, d), dev)
    _expect(q_noise, "q_noise", bf, (B, hn, d), dev)
    _expect(k_sig_pool, "k_sig_pool", bf, (num_pages, page_size, hs, d), dev)
    _expect(k_noise_pool, "k_noise_pool", bf, (num_pages, page_size, hn, d), dev)
    _expect(v_pool, "v_pool", bf, (num_pages, page_size, hs, dv), dev)
    _expect(block_table, "block_table", torch.int32, (B, max_pages), dev)
    _expect(cache_lens, "cache_lens", torch.int32, (B,), dev)
    _expect(lam, "lam", torch.float32, (hs,), dev)
    if out is None:
        out = torch.empty((B, hs, dv), dtype=bf, device=dev)
    _expect(out, "out", bf, (B, hs, dv), dev)
    need = gda_attn_decode_workspace_size(B, max_pages * page_size, hs, hn, dv)
    if workspace is None:
        workspace = torch.empty((need,), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        rc = _load().gda_attn_decode_paged(
            _ptr(q_sig), _ptr(q_noise), _ptr(k_sig_pool), _ptr(k_noise_pool), _ptr(v_pool),
            _ptr(block_table), _ptr(cache_lens), _ptr(lam), float(lambda_init), _ptr(out), B,
            max_pages, page_size, num_pages, hs, hn, d, dv, float(eps), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _stream(dev))
    _check(rc, "gda decode (paged caches)")
    return out


def gda_attn_decode_paged_fp8(q_sig, q_noise, k_sig_pool, k_noise_pool, v_pool, k_sig_scale, k_noise_scale,
                              v_scale, block_table, cache_lens, lam, lambda_init: float, *, eps: float = 1e-5,
                              out=None, workspace=None):
    """bf16 decode over paged fp8 (e4m3) caches: pools [num_pages, page_size,
    heads, dim] of float8_e4m3fn (or uint8 codes), per-head float32 scales,
    block_table [B, max_pages] int32."""
    dev = q_sig.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    B, hs, d = q_sig.shape
    hn = q_noise.shape[1]
    num_pages, page_size = k_sig_pool.shape[0], k_sig_pool.shape[1]
    dv = v_pool.shape[3]
    max_pages = block_table.shape[1]
    bf = torch.bfloat16
    pools = []
    for t, name, shape in ((k_sig_pool, "k_sig_pool", (num_pages, page_size, hs, d)),
                           (k_noise_pool, "k_noise_pool", (num_pages, page_size, hn, d)),
                           (v_pool, "v_pool", (num_pages, page_size, hs, dv))):
        if t.dtype == torch.float8_e4m3fn:
            t = t.view(torch.uint8)
        _expect(t, name, torch.uint8, shape, dev)
        pools.append(t)
    _expect(q_sig, "q_sig", bf, (B, hs, d), dev)
    _expect(q_noise, "q_noise", bf, (B, hn, d), dev)
    _expect(k_sig_scale, "k_sig_scale", torch.float32, (hs,), dev)
    _expect(k_noise_scale, "k_noise_scale", torch.float32, (hn,), dev)
    _expect(v_scale, "v_scale", torch.float32, (hs,), dev)
    _expect(block_table, "block_table", torch.int32, (B, max_pages), dev)
    _expect(cache_lens, "cache_lens", torch.int32, (B,), dev)
    _expect(lam, "lam", torch.float32, (hs,), dev)
    if out is None:
        out = torch.empty((B, hs, dv), dtype=bf, device=dev)
    _expect(out, "out", bf, (B, hs, dv), dev)
    need = gda_attn_decode_workspace_size(B, max_pages * page_size, hs, hn, dv)
    if workspace is None:
        workspace = torch.empty((need,), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        rc = _load().gda_attn_decode_paged_fp8(
            _ptr(q_sig), _ptr(q_noise), *[_ptr(t) for t in pools], _ptr(k_sig_scale), _ptr(k_noise_scale),
            _ptr(v_scale), _ptr(block_table), _ptr(cache_lens), _ptr(lam), float(lambda_init), _ptr(out), B,
            max_pages, page_size, num_pages, hs, hn, d, dv, float(eps), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _stream(dev))
    _check(rc, "gda decode (paged fp8 caches)")
    return out


def gda_attn_fwd_2pass_workspace_size(B: int, L: int, h_s: int, h_n: int) -> int:
    return int(_load().gda_attn_fwd_2pass_workspace_size(B, L, h_s, h_n))


def gda_attn_fwd_2pass(q_sig, k_sig, q_noise, k_noise, v, lam, lambda_init: float, *,
                       causal: bool = True, eps: float = 1e-5, out=None, flags: int = 0, workspace=None):
    """Two-pass bf16 prefill (difference map before the value product); returns ``out``.

    ``workspace`` (uint8 CUDA tensor) receives the rows' base-2 log-sum-exp
    values as float32 [B, h_s + h_n, L].
    """
    B, L, hs, _ = q_sig.shape
    hn = q_noise.shape[2]
    need = gda_attn_fwd_2pass_workspace_size(B, L, hs, hn)
    if workspace is None:
        workspace = torch.empty((max(need, 16),), dtype=torch.uint8, device=q_sig.device)
    _expect(workspace, "workspace", torch.uint8, (workspace.numel(),), q_sig.device)
    ws = workspace

    def entry(*args):
        *head, fl, stream = args
        return _load().gda_attn_fwd_2pass(*head, fl, _ptr(ws), ws.numel(), stream)
    return _prefill(entry, torch.bfloat16, q_sig, k_sig, q_noise, k_noise, v, lam, lambda_init, causal,
                    eps, out, flags)


def gda_attn_bwd_workspace_size(B: int, L: int, h_s: int, d: int, dv: int) -> int:
    return int(_load().gda_attn_bwd_workspace_size(B, L, h_s, d, dv))


def gda_attn_bwd(q_sig, k_sig, q_noise, k_noise, v, lam, lambda_init: float, dy, *,
                 causal: bool = True, eps: float = 1e-5, flags: int = 0, workspace=None, grads=None):
    """float32 gradients of the operation; returns (dq_sig, dk_sig, dq_noise, dk_noise, dv, dlambda).

    Inputs as for ``gda_attn_fwd_f32`` plus ``dy`` [B, L, h_s, dv] (the
    gradient of the loss with respect to the output).  ``grads`` may hold the
    six output tensors to overwrite.
    """
    dev = q_sig.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    if q_sig.dim() != 4 or q_noise.dim() != 4 or v.dim() != 4:
        raise ValueError("q_sig, q_noise and v must be 4-D [B, L, heads, dim]")
    f32 = torch.float32
    B, L, hs, d = q_sig.shape
    hn = q_noise.shape[2]
    dv = v.shape[3]
    shapes = ((B, L, hs, d), (B, L, hs, d), (B, L, hn, d), (B, L, hn, d), (B, L, hs, dv), (hs,))
    for t, name, shape in zip((q_sig, k_sig, q_noise, k_noise, v, lam), ("q_sig", "k_sig", "q_noise",
                              "k_noise", "v", "lam"), shapes):
        _expect(t, name, f32, shape, dev)
    _expect(dy, "dy", f32, (B, L, hs, dv), dev)
    if grads is None:
        grads = tuple(torch.empty(s, dtype=f32, device=dev) for s in shapes)
    for t, name, shape in zip(grads, ("dq_sig", "dk_sig", "dq_noise", "dk_noise", "dv", "dlambda"), shapes):
        _expect(t, name, f32, shape, dev)
    need = gda_attn_bwd_workspace_size(B, L, hs, d, dv)
    if workspace is None:
        workspace = torch.empty((max(need, 16),), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        rc = _load().gda_attn_bwd(
            _ptr(q_sig), _ptr(k_sig), _ptr(q_noise), _ptr(k_noise), _ptr(v), _ptr(lam),
            float(lambda_init), _ptr(dy), *[_ptr(t) for t in grads], B, L, hs, hn, d, dv,
            int(bool(causal)), float(eps), int(flags), _ptr(workspace), workspace.numel(), _stream(dev))
    _check(rc, "gda backward")
    return tuple(grads)


def gda_attn_bwd_bf16_workspace_size(B: int, L: int, h_s: int, h_n: int, dv: int) -> int:
    return int(_load().gda_attn_bwd_bf16_workspace_size(B, L, h_s, h_n, dv))


def gda_attn_bwd_bf16(q_sig, k_sig, q_noise, k_noise, v, lam, lambda_init: float, dy, *,
                      causal: bool = True, eps: float = 1e-5, flags: int = 0, workspace=None, grads=None):
    """Tensor-core gradients from bf16 inputs; returns float32
    (dq_sig, dk_sig, dq_noise, dk_noise, dv, dlambda)."""
    dev = q_sig.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    if q_sig.dim() != 4 or q_noise.dim() != 4 or v.dim() != 4:
        raise ValueError("q_sig, q_noise and v must be 4-D [B, L, heads, dim]")
    bf, f32 = torch.bfloat16, torch.float32
    B, L, hs, d = q_sig.shape
    hn = q_noise.shape[2]
    dv = v.shape[3]
    shapes = ((B, L, hs, d), (B, L, hs, d), (B, L, hn, d), (B, L, hn, d), (B, L, hs, dv), (hs,))
    for t, name, shape in zip((q_sig, k_sig, q_noise, k_noise, v), ("q_sig", "k_sig", "q_noise", "k_noise", "v"),
                              shapes):
        _expect(t, name, bf, shape, dev)
    _expect(lam, "lam", f32, (hs,), dev)
    _expect(dy, "dy", bf, (B, L, hs, dv), dev)
    if grads is None:
        grads = tuple(torch.empty(s, dtype=f32, device=dev) for s in shapes)
    for t, name, shape in zip(grads, ("dq_sig", "dk_sig", "dq_noise", "dk_noise", "dv", "dlambda"), shapes):
        _expect(t, name, f32, shape, dev)
    need = gda_attn_bwd_bf16_workspace_size(B, L, hs, hn, dv)
    if workspace is None:
        workspace = torch.empty((max(need, 16),), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        rc = _load().gda_attn_bwd_bf16(
            _ptr(q_sig), _ptr(k_sig), _ptr(q_noise), _ptr(k_noise), _ptr(v), _ptr(lam),
            float(lambda_init), _ptr(dy), *[_ptr(t) for t in grads], B, L, hs, hn, d, dv,
            int(bool(causal)), float(eps), int(flags), _ptr(workspace), workspace.numel(), _stream(dev))
    _check(rc, "gda backward (bf16)")
    return tuple(grads)


def gda_lambda_reparam(lambda_q1, lambda_k1, lambda_q2, lambda_k2, lambda_init: float, *, out=None):
    """lambda[h] = exp(lq1[h].lk1[h]) - exp(lq2[h].lk2[h]) + lambda_init on the device.

    The four vectors are float32 CUDA tensors [h_s, d]; returns ``out``
    (float32 [h_s]), ready to pass as ``lam`` to the attention calls.
    """
    dev = lambda_q1.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    if lambda_q1.dim() != 2:
        raise ValueError("lambda vectors must be 2-D [h_s, d]")
    hs, d = lambda_q1.shape
    for t, name in ((lambda_q1, "lambda_q1"), (lambda_k1, "lambda_k1"), (lambda_q2, "lambda_q2"),
                    (lambda_k2, "lambda_k2")):
        _expect(t, name, torch.float32, (hs, d), dev)
    if out is None:
        out = torch.empty((hs,), dtype=torch.float32, device=dev)
    _expect(out, "out", torch.float32, (hs,), dev)
    with torch.cuda.device(dev):
        rc = _load().gda_lambda_reparam(_ptr(lambda_q1), _ptr(lambda_k1), _ptr(lambda_q2),
                                        _ptr(lambda_k2), float(lambda_init), _ptr(out), hs, d,
                                        _stream(dev))
    _check(rc, "gda lambda re-parameterisation")
    return out


def gda_attn_decode_workspace_size(B: int, Lcap: int, h_s: int, h_n: int, dv: int) -> int:
    return int(_load().gda_attn_decode_workspace_size(B, Lcap, h_s, h_n, dv))


def gda_attn_decode(q_sig, q_noise, k_sig_cache, k_noise_cache, v_cache, cache_lens, lam,
                    lambda_init: float, *, eps: float = 1e-5, out=None, workspace=None):
    """bf16 decode of one query token per sequence over its KV cache; returns ``out``.

    ``workspace`` (a CUDA uint8 tensor of at least
    ``gda_attn_decode_workspace_size(...)`` bytes) is allocated here when not
    given.
    """
    dev = q_sig.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    if q_sig.dim() != 3 or k_sig_cache.dim() != 4 or v_cache.dim() != 4:
        raise ValueError("bad ranks: q [B, heads, d], caches [B, Lcap, heads, dim]")
    B, hs, d = q_sig.shape
    hn = q_noise.shape[1]
    Lcap = k_sig_cache.shape[1]
    dv = v_cache.shape[3]
    bf = torch.bfloat16
    _expect(q_sig, "q_sig", bf, (B, hs, d), dev)
    _expect(q_noise, "q_noise", bf, (B, hn, d), dev)
    _expect(k_sig_cache, "k_sig_cache", bf, (B, Lcap, hs, d), dev)
    _expect(k_noise_cache, "k_noise_cache", bf, (B, Lcap, hn, d), dev)
    _expect(v_cache, "v_cache", bf, (B, Lcap, hs, dv), dev)
    _expect(cache_lens, "cache_lens", torch.int32, (B,), dev)
    _expect(lam, "lam", torch.float32, (hs,), dev)
    if out is None:
        out = torch.empty((B, hs, dv), dtype=bf, device=dev)
    _expect(out, "out", bf, (B, hs, dv), dev)
    need = gda_attn_decode_workspace_size(B, Lcap, hs, hn, dv)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    if workspace.device != dev or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous tensor on the inputs' device")
    ws_bytes = workspace.numel() * workspace.element_size()
    with torch.cuda.device(dev):
        rc = _load().gda_attn_decode(
            _ptr(q_sig), _ptr(q_noise), _ptr(k_sig_cache), _ptr(k_noise_cache), _ptr(v_cache),
            _ptr(cache_lens), _ptr(lam), float(lambda_init), _ptr(out), B, Lcap, hs, hn, d, dv,
            float(eps), _ptr(workspace), ws_bytes, _stream(dev))
    _check(rc, "gda decode")
    return out


def gda_attn_decode_noalloc(q_sig, q_noise, k_sig_cache, k_noise_cache, v_cache, cache_lens,
                            lam, lambda_init: float, *, eps: float = 1e-5, out=None):
    """Decode without a workspace: the library's fixed scratch array holds the split partials.

    For callers that cannot allocate device memory.  Calls that overlap on
    the GPU race on the shared scratch array; see include/gda.h.
    """
    dev = q_sig.device
    B, hs, d = q_sig.shape
    hn = q_noise.shape[1]
    Lcap = k_sig_cache.shape[1]
    dv = v_cache.shape[3]
    bf = torch.bfloat16
    _expect(q_sig, "q_sig", bf, (B, hs, d), dev)
    _expect(q_noise, "q_noise", bf, (B, hn, d), dev)
    _expect(k_sig_cache, "k_sig_cache", bf, (B, Lcap, hs, d), dev)
    _expect(k_noise_cache, "k_noise_cache", bf, (B, Lcap, hn, d), dev)
    _expect(v_cache, "v_cache", bf, (B, Lcap, hs, dv), dev)
    _expect(cache_lens, "cache_lens", torch.int32, (B,), dev)
    _expect(lam, "lam", torch.float32, (hs,), dev)
    if out is None:
        out = torch.empty((B, hs, dv), dtype=bf, device=dev)
    _expect(out, "out", bf, (B, hs, dv), dev)
    with torch.cuda.device(dev):
        rc = _load().gda_attn_decode_noalloc(
            _ptr(q_sig), _ptr(q_noise), _ptr(k_sig_cache), _ptr(k_noise_cache), _ptr(v_cache),
            _ptr(cache_lens), _ptr(lam), float(lambda_init), _ptr(out), B, Lcap, hs, hn, d, dv,
            float(eps), _stream(dev))
    _check(rc, "gda decode (no allocation)")
    return out


def gda_device_error(clear: bool = True) -> int:
    """Device error word of the current device (synchronises it); see include/gda.h."""
    rc = _load().gda_device_error(int(bool(clear)))
    if rc < 0:
        raise GDAError(rc, "gda_device_error")
    return rc

