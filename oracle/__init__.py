"""Float64 CPU oracle for grouped differential attention.

TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
benchmark's CPU-baseline leg may import this package.  The product path (the
CUDA library and its Python binding) never imports it, and it imports nothing
from the product.

Two independent formulations of the same definition live here:

* ``gda_oracle.c`` -- a per-row loop in C, float64, OpenMP over
  (batch, signal head, query row).  ``prefill``, ``prefill_rows`` and
  ``decode`` wrap it.
* ``ref_numpy.py`` -- a dense-matrix NumPy formulation (full L x L maps),
  for brute-force cross-checks on tiny inputs.

Definition (see ``gda_oracle.c`` for the sources): with r = h_s / h_n and the
noise head of signal head h being g = h // r,

    o_h = (softmax(Q1_h K1_h^T / sqrt(d)) - lambda_h softmax(Q2_g K2_g^T / sqrt(d))) V_h
    y_h = (1 - lambda_init) * o_h / sqrt(mean(o_h^2) + eps)

Every function here is pinned by ``tests/test_oracle_pins.py`` against
library routines (PyTorch's float64 scaled-dot-product attention and
``rms_norm``), closed forms and the NumPy brute force.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gda_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libgda_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (-O2, OpenMP, IEEE arithmetic)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            D = ctypes.c_double
            I64 = ctypes.c_int64
            lib.gda_oracle_prefill.argtypes = [P, P, P, P, P, P, D, I, I, I, I, I, I, I,
                                               D, I, P, I64, P]
            lib.gda_oracle_prefill.restype = I
            lib.gda_oracle_decode.argtypes = [P, P, P, P, P, P, P, D, I, I, I, I, I, I,
                                              D, I, P]
            lib.gda_oracle_decode.restype = I
            lib.gda_oracle_max_threads.argtypes = []
            lib.gda_oracle_max_threads.restype = I
            lib.gda_oracle_set_threads.argtypes = [I]
            lib.gda_oracle_set_threads.restype = None
            _lib = lib
    return _lib


def _f32(x) -> np.ndarray:
    """Exact float32 copy of a tensor/array (bf16 widens exactly)."""
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().cpu()
        import torch
        if x.dtype != torch.float32:
            x = x.to(torch.float32)
        x = x.numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().cpu().to(dtype=__import__("torch").float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def max_threads() -> int:
    return _load().gda_oracle_max_threads()


def set_threads(n: int) -> None:
    _load().gda_oracle_set_threads(int(n))


def prefill(q1, k1, q2, k2, v, lam, lambda_init: float, causal: bool = True,
            eps: float = 1e-5, norm: bool = True, rows=None) -> np.ndarray:
    """Oracle prefill.

    q1, k1: [B, L, h_s, d]; q2, k2: [B, L, h_n, d]; v: [B, L, h_s, dv];
    lam: [h_s].  Returns float64 [B, L, h_s, dv], or [B, len(rows), h_s, dv]
    when ``rows`` lists query positions.
    """
    q1, k1, q2, k2, v = (_f32(t) for t in (q1, k1, q2, k2, v))
    lam = _f64(lam).reshape(-1)
    B, L, hs, d = q1.shape
    hn = q2.shape[2]
    dv = v.shape[3]
    assert k1.shape == (B, L, hs, d) and q2.shape == (B, L, hn, d)
    assert k2.shape == (B, L, hn, d) and v.shape == (B, L, hs, dv)
    assert lam.shape == (hs,)
    if rows is not None:
        rows_a = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
        out = np.empty((B, rows_a.size, hs, dv), dtype=np.float64)
        rows_p, nrows = _ptr(rows_a), rows_a.size
    else:
        out = np.empty((B, L, hs, dv), dtype=np.float64)
        rows_p, nrows = None, 0
    rc = _load().gda_oracle_prefill(_ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2), _ptr(v),
                                    _ptr(lam), float(lambda_init), B, L, hs, hn, d, dv,
                                    int(bool(causal)), float(eps), int(bool(norm)),
                                    rows_p, nrows, _ptr(out))
    if rc != 0:
        raise ValueError("gda_oracle_prefill rejected its arguments")
    return out


def prefill_rows(q1, k1, q2, k2, v, lam, lambda_init: float, rows, causal: bool = True,
                 eps: float = 1e-5, norm: bool = True) -> np.ndarray:
    """The prefill definition evaluated only at the listed query positions."""
    return prefill(q1, k1, q2, k2, v, lam, lambda_init, causal=causal, eps=eps,
                   norm=norm, rows=rows)


def decode(q1, q2, k1_cache, k2_cache, v_cache, lens, lam, lambda_init: float,
           eps: float = 1e-5, norm: bool = True) -> np.ndarray:
    """Oracle decode: one query token per sequence over its first lens[b] cache rows.

    q1: [B, h_s, d]; q2: [B, h_n, d]; k1_cache: [B, Lcap, h_s, d];
    k2_cache: [B, Lcap, h_n, d]; v_cache: [B, Lcap, h_s, dv]; lens: [B] int.
    Returns float64 [B, h_s, dv].
    """
    q1, q2, k1c, k2c, vc = (_f32(t) for t in (q1, q2, k1_cache, k2_cache, v_cache))
    lam = _f64(lam).reshape(-1)
    if hasattr(lens, "detach"):
        lens = lens.detach().cpu().numpy()
    lens_a = np.ascontiguousarray(np.asarray(lens, dtype=np.int32).reshape(-1))
    B, hs, d = q1.shape
    hn = q2.shape[1]
    Lcap = k1c.shape[1]
    dv = vc.shape[3]
    assert k1c.shape == (B, Lcap, hs, d) and k2c.shape == (B, Lcap, hn, d)
    assert vc.shape == (B, Lcap, hs, dv) and lens_a.shape == (B,)
    out = np.empty((B, hs, dv), dtype=np.float64)
    rc = _load().gda_oracle_decode(_ptr(q1), _ptr(q2), _ptr(k1c), _ptr(k2c), _ptr(vc),
                                   _ptr(lens_a), _ptr(lam), float(lambda_init), B, Lcap,
                                   hs, hn, d, dv, float(eps), int(bool(norm)), _ptr(out))
    if rc != 0:
        raise ValueError("gda_oracle_decode rejected its arguments")
    return out


def lambda_init_schedule(layer: int) -> float:
    """lambda_init for 1-based layer index ``layer``.

    "Differential Attention in Large Language Models ...", section "Learnable
    Lambda Re-parameterization": an exponential schedule over depth that
    starts at 0.2 in the first layer and approaches 0.8.
    """
    return 0.8 - 0.6 * math.exp(-0.3 * (layer - 1))


def lambda_reparam(lq1, lk1, lq2, lk2, lambda_init: float) -> np.ndarray:
    """lambda_h = exp(lq1_h . lk1_h) - exp(lq2_h . lk2_h) + lambda_init, float64.

    "Differential Attention in Large Language Models ...", section "Learnable
    Lambda Re-parameterization": four learnable vectors and the layer's
    initialisation constant.  One set of vectors per signal head (arrays
    [h_s, d]); a per-layer lambda is the case of identical rows.
    """
    a = np.sum(_f64(lq1) * _f64(lk1), axis=-1)
    b = np.sum(_f64(lq2) * _f64(lk2), axis=-1)
    return np.exp(a) - np.exp(b) + float(lambda_init)
