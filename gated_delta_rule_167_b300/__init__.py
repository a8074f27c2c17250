"""KDA (Kimi Delta Attention) forward pass for NVIDIA B300 (sm_103a).

A thin ctypes binding over the C ABI declared in ``include/kda.h``. The functions here only
marshal arguments (shapes, dtypes, device pointers, the current CUDA stream); every step of the
computation runs in the CUDA kernels of ``libkda.so``. There is no CPU fallback: if the library
is missing, importing succeeds but every call raises :class:`KdaLibraryError`.

Tensors are PyTorch CUDA tensors in the layouts of ``include/kda.h``:
q, k, g ``[B, T, H, d_k]``; v, out ``[B, T, H, d_v]``; beta ``[B, T, H]`` (all the same
dtype: float32 or bfloat16); states fp32 ``[B, H, d_k, d_v]``.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "KdaError", "KdaLibraryError", "kda_chunk_fwd", "kda_chunk_fwd_varlen",
    "kda_recurrent_step", "kda_sync_status", "kda_status_string", "kda_version", "lib_path",
    "load_library", "chunk_fwd", "chunk_fwd_varlen", "recurrent_step", "chunk_fwd_host",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkda.so")

KDA_OK, KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED, KDA_ERR_CUDA, KDA_ERR_TIMEOUT = range(5)
KDA_DTYPE_F32, KDA_DTYPE_BF16 = 0, 1
_DTYPES = {torch.float32: KDA_DTYPE_F32, torch.bfloat16: KDA_DTYPE_BF16}

EXPORTED_SYMBOLS = (
    "kda_chunk_fwd", "kda_chunk_fwd_varlen", "kda_recurrent_step", "kda_sync_status",
    "kda_wait_selftest", "kda_status_string", "kda_last_error", "kda_version",
)


class KdaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


class KdaLibraryError(ImportError):
    pass


_lib = None


def lib_path() -> str:
    return LIB_PATH


def load_library(path: str | None = None):
    """Loads libkda.so (once) and declares the C signatures. Raises if it is missing."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise KdaLibraryError(
            f"{p} not found: build it with `python -m gated_delta_rule_167_b300.build` "
            "(or __graft_entry__.build())")
    lib = ctypes.CDLL(p)
    V, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_int
    lib.kda_chunk_fwd.argtypes = [V] * 8 + [I] * 7 + [V]
    lib.kda_chunk_fwd.restype = S
    lib.kda_chunk_fwd_varlen.argtypes = [V] * 9 + [I] * 6 + [I, V]
    lib.kda_chunk_fwd_varlen.restype = S
    lib.kda_recurrent_step.argtypes = [V] * 7 + [I] * 4 + [I, V]
    lib.kda_recurrent_step.restype = S
    lib.kda_sync_status.argtypes = [V]
    lib.kda_wait_selftest.argtypes = [ctypes.c_ulonglong, V]
    lib.kda_wait_selftest.restype = S
    lib.kda_sync_status.restype = S
    lib.kda_status_string.argtypes = [S]
    lib.kda_status_string.restype = ctypes.c_char_p
    lib.kda_last_error.argtypes = []
    lib.kda_last_error.restype = ctypes.c_char_p
    lib.kda_version.argtypes = []
    lib.kda_version.restype = I
    if path is None:
        _lib = lib
    return lib


def _check(status: int, what: str):
    if status != KDA_OK:
        lib = load_library()
        msg = lib.kda_last_error().decode() or lib.kda_status_string(status).decode()
        raise KdaError(status, f"{what}: {lib.kda_status_string(status).decode()}: {msg}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype not in _DTYPES:
        raise TypeError(f"unsupported dtype {t.dtype}; expected float32 or bfloat16")
    return _DTYPES[t.dtype]


def _require(cond: bool, msg: str):
    if not cond:
        raise ValueError(msg)


def _check_tensors(named, dtype, device):
    for name, t in named:
        if t is None:
            continue
        _require(t.is_cuda and t.device == device, f"{name} must be on {device}")
        _require(t.is_contiguous(), f"{name} must be contiguous")
        if dtype is not None:
            _require(t.dtype == dtype, f"{name} must be {dtype} (got {t.dtype})")


# ------------------------------------------------------------------------- C-ABI mirrors


def kda_chunk_fwd(q, k, v, g, beta, S0, out, S_final, C: int = 64, stream=None):
    """Chunkwise prefill (dense batch). Writes ``out`` and, if given, ``S_final``."""
    lib = load_library()
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    _check_tensors([("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("out", out)],
                   q.dtype, q.device)
    _check_tensors([("S0", S0), ("S_final", S_final)], torch.float32, q.device)
    _require(k.shape == q.shape and g.shape == q.shape, "q, k, g must share [B, T, H, d_k]")
    _require(v.shape == (B, T, H, dv) and out.shape == v.shape, "v/out must be [B, T, H, d_v]")
    _require(beta.shape == (B, T, H), "beta must be [B, T, H]")
    for name, s in (("S0", S0), ("S_final", S_final)):
        _require(s is None or s.shape == (B, H, dk, dv), f"{name} must be [B, H, d_k, d_v]")
    st = lib.kda_chunk_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(S0), _ptr(out),
                           _ptr(S_final), B, H, T, dk, dv, int(C), _dtype_code(q),
                           _stream_handle(stream))
    _check(st, "kda_chunk_fwd")


def kda_chunk_fwd_varlen(q, k, v, g, beta, S0, out, S_final, cu_seqlens, C: int = 64,
                         stream=None):
    """Chunkwise prefill over a packed batch ([1, T_total, H, d]; cu_seqlens int32 on device)."""
    lib = load_library()
    one, T, H, dk = q.shape
    dv = v.shape[-1]
    _require(one == 1, "packed batches have a leading dimension of 1")
    _check_tensors([("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("out", out)],
                   q.dtype, q.device)
    _check_tensors([("S0", S0), ("S_final", S_final)], torch.float32, q.device)
    _check_tensors([("cu_seqlens", cu_seqlens)], torch.int32, q.device)
    N = cu_seqlens.shape[0] - 1
    _require(N >= 0, "cu_seqlens needs at least one entry")
    for name, s in (("S0", S0), ("S_final", S_final)):
        _require(s is None or s.shape == (N, H, dk, dv), f"{name} must be [N, H, d_k, d_v]")
    st = lib.kda_chunk_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(S0),
                                  _ptr(out), _ptr(S_final), _ptr(cu_seqlens), N, H, T, dk, dv,
                                  int(C), _dtype_code(q), _stream_handle(stream))
    _check(st, "kda_chunk_fwd_varlen")


def kda_recurrent_step(q, k, v, g, beta, S, out, stream=None):
    """One decode token for [N, H] states; S (fp32 [N, H, d_k, d_v]) is updated in place."""
    lib = load_library()
    N, H, dk = q.shape
    dv = v.shape[-1]
    _check_tensors([("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("out", out)],
                   q.dtype, q.device)
    _check_tensors([("S", S)], torch.float32, q.device)
    _require(S.shape == (N, H, dk, dv), "S must be [N, H, d_k, d_v]")
    st = lib.kda_recurrent_step(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(S),
                                _ptr(out), N, H, dk, dv, _dtype_code(q), _stream_handle(stream))
    _check(st, "kda_recurrent_step")


def kda_sync_status(stream=None):
    """Synchronises the stream and raises if a kernel latched a device-side error."""
    _check(load_library().kda_sync_status(_stream_handle(stream)), "kda_sync_status")


def kda_wait_selftest(limit_ns: int, stream=None) -> int:
    """Launches the bounded-wait self-test (see include/kda.h); returns the launch status."""
    return load_library().kda_wait_selftest(int(limit_ns), _stream_handle(stream))


def kda_status_string(status: int) -> str:
    return load_library().kda_status_string(int(status)).decode()


def kda_version() -> int:
    return load_library().kda_version()


# ------------------------------------------------------------------------- conveniences


def chunk_fwd(q, k, v, g, beta, S0=None, C: int = 64, want_state: bool = True, stream=None):
    """Allocates the outputs with torch and calls :func:`kda_chunk_fwd`."""
    B, T, H, dk = q.shape
    out = torch.empty(B, T, H, v.shape[-1], dtype=q.dtype, device=q.device)
    Sf = (torch.empty(B, H, dk, v.shape[-1], dtype=torch.float32, device=q.device)
          if want_state else None)
    kda_chunk_fwd(q, k, v, g, beta, S0, out, Sf, C=C, stream=stream)
    return out, Sf


def chunk_fwd_varlen(q, k, v, g, beta, cu_seqlens, S0=None, C: int = 64, want_state=True,
                     stream=None):
    _, T, H, dk = q.shape
    N = cu_seqlens.shape[0] - 1
    out = torch.empty(1, T, H, v.shape[-1], dtype=q.dtype, device=q.device)
    Sf = (torch.empty(N, H, dk, v.shape[-1], dtype=torch.float32, device=q.device)
          if want_state else None)
    kda_chunk_fwd_varlen(q, k, v, g, beta, S0, out, Sf, cu_seqlens, C=C, stream=stream)
    return out, Sf


def recurrent_step(q, k, v, g, beta, S, stream=None):
    out = torch.empty(q.shape[0], q.shape[1], v.shape[-1], dtype=q.dtype, device=q.device)
    kda_recurrent_step(q, k, v, g, beta, S, out, stream=stream)
    return out


def chunk_fwd_host(q, k, v, g, beta, S0=None, C: int = 64, device=None, stream=None,
                   out_host=None, state_host=None):
    """End-to-end call on HOST tensors: copies the inputs to the device (pinned host memory
    gives asynchronous copies), runs :func:`kda_chunk_fwd`, and copies the output and final
    state back into ``out_host`` / ``state_host`` (allocated pinned if not given)."""
    device = device or torch.device("cuda", torch.cuda.current_device())
    nb = True
    dq, dk_, dv_, dg, db = (t.to(device, non_blocking=nb) for t in (q, k, v, g, beta))
    dS0 = None if S0 is None else S0.to(device, non_blocking=nb)
    out, Sf = chunk_fwd(dq, dk_, dv_, dg, db, dS0, C=C, stream=stream)
    if out_host is None:
        out_host = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    if state_host is None:
        state_host = torch.empty(Sf.shape, dtype=Sf.dtype, pin_memory=True)
    out_host.copy_(out, non_blocking=nb)
    state_host.copy_(Sf, non_blocking=nb)
    return out_host, state_host
