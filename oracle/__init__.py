"""KDA oracle -- TEST INFRASTRUCTURE ONLY.

Plain fp64 CPU statements of the Kimi Delta Attention forward pass, used to check the CUDA
library. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this package; the product package never does, and the two share no code.

* :func:`recurrent`, :func:`recurrent_varlen`, :func:`decode_step` call the C recurrence in
  ``kda_oracle.c`` (token by token, fp64; see that file for the definition followed).
* :mod:`oracle.chunkwise` restates the chunkwise (block) form in fp64 NumPy, to pin the
  algebra that the GPU path is built on against the recurrence.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``kda_oracle.c`` into ``oracle/_build/libkda_oracle.so`` with gcc."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"],
            check=True,
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            lib.kda_oracle_recurrent.argtypes = [P] * 8 + [I] * 6
            lib.kda_oracle_recurrent.restype = I
            lib.kda_oracle_recurrent_varlen.argtypes = [P] * 9 + [I] * 6
            lib.kda_oracle_recurrent_varlen.restype = I
            lib.kda_oracle_decode_step.argtypes = [P] * 7 + [I] * 4
            lib.kda_oracle_decode_step.restype = I
            _lib = lib
    return _lib


def _f64(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    return os.cpu_count() or 1


def recurrent(q, k, v, g, beta, S0=None, nthreads: int | None = None):
    """Token-by-token KDA over a dense batch.

    q, k, g: [B, T, H, d_k]; v: [B, T, H, d_v]; beta: [B, T, H]; S0: [B, H, d_k, d_v] or None
    (zeros). Returns (o [B, T, H, d_v], S_final [B, H, d_k, d_v]) in fp64.
    """
    q, k, v, g, beta = map(_f64, (q, k, v, g, beta))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    assert k.shape == q.shape and g.shape == q.shape and v.shape == (B, T, H, dv)
    assert beta.shape == (B, T, H)
    S0 = None if S0 is None else _f64(S0)
    if S0 is not None:
        assert S0.shape == (B, H, dk, dv)
    out = np.zeros((B, T, H, dv))
    Sf = np.zeros((B, H, dk, dv))
    rc = _load().kda_oracle_recurrent(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(S0), _ptr(out), _ptr(Sf),
        B, H, T, dk, dv, nthreads or default_threads())
    if rc != 0:
        raise ValueError("kda_oracle_recurrent rejected its arguments")
    return out, Sf


def recurrent_varlen(q, k, v, g, beta, cu_seqlens, S0=None, nthreads: int | None = None):
    """Token-by-token KDA over a packed batch (leading dimension 1).

    cu_seqlens: int32 [N+1], cu[0] = 0, cu[N] = T_total; S0: [N, H, d_k, d_v] or None.
    Returns (o [1, T_total, H, d_v], S_final [N, H, d_k, d_v]).
    """
    q, k, v, g, beta = map(_f64, (q, k, v, g, beta))
    _, T, H, dk = q.shape
    dv = v.shape[-1]
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    N = cu.shape[0] - 1
    S0 = None if S0 is None else _f64(S0)
    out = np.zeros((1, T, H, dv))
    Sf = np.zeros((N, H, dk, dv))
    rc = _load().kda_oracle_recurrent_varlen(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(S0), _ptr(out), _ptr(Sf), _ptr(cu),
        N, H, T, dk, dv, nthreads or default_threads())
    if rc != 0:
        raise ValueError("kda_oracle_recurrent_varlen rejected its arguments")
    return out, Sf


def decode_step(q, k, v, g, beta, S):
    """One token for N x H independent states. q, k, g [N, H, d_k]; v [N, H, d_v];
    beta [N, H]; S [N, H, d_k, d_v]. Returns (o [N, H, d_v], S_new) without touching S."""
    q, k, v, g, beta = map(_f64, (q, k, v, g, beta))
    N, H, dk = q.shape
    dv = v.shape[-1]
    Snew = _f64(S).copy()
    out = np.zeros((N, H, dv))
    rc = _load().kda_oracle_decode_step(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(Snew), _ptr(out), N, H, dk, dv)
    if rc != 0:
        raise ValueError("kda_oracle_decode_step rejected its arguments")
    return out, Snew
