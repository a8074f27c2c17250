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

import contextlib
import ctypes
import os

import torch

__all__ = [
    "KdaError", "KdaLibraryError", "kda_chunk_fwd", "kda_chunk_fwd_varlen",
    "kda_recurrent_step", "kda_sync_status", "kda_status_string", "kda_version", "lib_path",
    "load_library", "chunk_fwd", "chunk_fwd_varlen", "recurrent_step", "chunk_fwd_host",
    "HostPipeline", "kda_segment_transitions", "kda_segment_scan", "kda_chunk_fwd_segmented",
    "chunk_fwd_segmented", "segmented_workspace_bytes", "segments_auto",
    "kda_chunk_fwd_segmented_noalloc", "NOALLOC_SCRATCH_BYTES", "kda_chunk_fwd_gated",
    "kda_output_gate", "kda_pre_core", "kda_chunk_fwd_fused", "kda_recurrent_steps",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkda.so")

KDA_OK, KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED, KDA_ERR_CUDA, KDA_ERR_TIMEOUT = range(5)
KDA_DTYPE_F32, KDA_DTYPE_BF16 = 0, 1
_DTYPES = {torch.float32: KDA_DTYPE_F32, torch.bfloat16: KDA_DTYPE_BF16}

EXPORTED_SYMBOLS = (
    "kda_chunk_fwd", "kda_chunk_fwd_varlen", "kda_recurrent_step", "kda_sync_status",
    "kda_wait_selftest", "kda_status_string", "kda_last_error", "kda_version",
    "kda_segment_transitions", "kda_segment_scan", "kda_chunk_fwd_segmented",
    "kda_chunk_fwd_segmented_workspace", "kda_segments_auto", "kda_chunk_fwd_segmented_noalloc",
    "kda_chunk_fwd_gated", "kda_output_gate", "kda_pre_core", "kda_chunk_fwd_fused",
    "kda_recurrent_steps",
)

# Bytes of the fixed device scratch behind kda_chunk_fwd_segmented_noalloc (include/kda.h).
NOALLOC_SCRATCH_BYTES = 32 << 20


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
    Z = ctypes.c_size_t
    lib.kda_segment_transitions.argtypes = [V] * 6 + [I] * 9 + [V]
    lib.kda_segment_transitions.restype = S
    lib.kda_segment_scan.argtypes = [V] * 4 + [I] * 5 + [V]
    lib.kda_segment_scan.restype = S
    lib.kda_chunk_fwd_segmented.argtypes = [V] * 8 + [I] * 7 + [V, Z, I, V]
    lib.kda_chunk_fwd_segmented.restype = S
    lib.kda_chunk_fwd_segmented_workspace.argtypes = [I] * 6
    lib.kda_chunk_fwd_segmented_workspace.restype = Z
    lib.kda_segments_auto.argtypes = [I] * 3
    lib.kda_segments_auto.restype = I
    lib.kda_chunk_fwd_segmented_noalloc.argtypes = [V] * 8 + [I] * 7 + [I, V]
    lib.kda_chunk_fwd_segmented_noalloc.restype = S
    F = ctypes.c_float
    lib.kda_chunk_fwd_gated.argtypes = [V] * 8 + [F, V, V, V] + [I] * 6 + [I, V]
    lib.kda_chunk_fwd_gated.restype = S
    lib.kda_output_gate.argtypes = [V, V, V, F, V, ctypes.c_longlong, I, I, V]
    lib.kda_output_gate.restype = S
    lib.kda_pre_core.argtypes = [V] * 14 + [I] * 4 + [I, V]
    lib.kda_pre_core.restype = S
    lib.kda_chunk_fwd_fused.argtypes = [V] * 13 + [F, V, V, V] + [I] * 6 + [I, V]
    lib.kda_chunk_fwd_fused.restype = S
    lib.kda_recurrent_steps.argtypes = [V] * 7 + [I] * 5 + [I, V]
    lib.kda_recurrent_steps.restype = S
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


def kda_segment_transitions(k, v, g, beta, M, S_tilde, seg_len: int, C: int = 64, stream=None):
    """(M, S~) of segments of ``seg_len`` tokens: M [n_seg, B, H, d_k, d_k] and S_tilde
    [n_seg, B, H, d_k, d_v] (fp32, written)."""
    lib = load_library()
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    n_seg = M.shape[0]
    _check_tensors([("k", k), ("v", v), ("g", g), ("beta", beta)], k.dtype, k.device)
    _check_tensors([("M", M), ("S_tilde", S_tilde)], torch.float32, k.device)
    _require(g.shape == k.shape and v.shape == (B, T, H, dv) and beta.shape == (B, T, H),
             "k, g [B, T, H, d_k]; v [B, T, H, d_v]; beta [B, T, H]")
    _require(M.shape == (n_seg, B, H, dk, dk), "M must be [n_seg, B, H, d_k, d_k]")
    _require(S_tilde.shape == (n_seg, B, H, dk, dv), "S_tilde must be [n_seg, B, H, d_k, d_v]")
    st = lib.kda_segment_transitions(_ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(M),
                                     _ptr(S_tilde), B, H, T, int(seg_len), n_seg, dk, dv, int(C),
                                     _dtype_code(k), _stream_handle(stream))
    _check(st, "kda_segment_transitions")


def kda_segment_scan(M, S_tilde, S0, S_in, stream=None):
    """S_in[0] = S0 (or zeros), S_in[s + 1] = M[s] S_in[s] + S_tilde[s]; S_in is
    [n_seg, B, H, d_k, d_v] fp32 (written)."""
    lib = load_library()
    n_seg, B, H, dk, dv = S_in.shape
    _check_tensors([("M", M), ("S_tilde", S_tilde), ("S0", S0), ("S_in", S_in)], torch.float32,
                   S_in.device)
    if n_seg > 1:
        _require(M is not None and M.shape == (n_seg - 1, B, H, dk, dk),
                 "M must be [n_seg - 1, B, H, d_k, d_k]")
        _require(S_tilde is not None and S_tilde.shape == (n_seg - 1, B, H, dk, dv),
                 "S_tilde must be [n_seg - 1, B, H, d_k, d_v]")
    _require(S0 is None or S0.shape == (B, H, dk, dv), "S0 must be [B, H, d_k, d_v]")
    st = lib.kda_segment_scan(_ptr(M), _ptr(S_tilde), _ptr(S0), _ptr(S_in), n_seg, B, H, dk, dv,
                              _stream_handle(stream))
    _check(st, "kda_segment_scan")


def segmented_workspace_bytes(B, H, T, d_k, d_v, n_seg) -> int:
    return int(load_library().kda_chunk_fwd_segmented_workspace(B, H, T, d_k, d_v, n_seg))


def segments_auto(B, H, T) -> int:
    return int(load_library().kda_segments_auto(B, H, T))


def kda_chunk_fwd_segmented(q, k, v, g, beta, S0, out, S_final, n_seg: int, workspace,
                            C: int = 64, stream=None):
    """Prefill parallel along T (see include/kda.h); ``workspace`` is a device tensor of at least
    :func:`segmented_workspace_bytes` bytes (or None when one segment suffices)."""
    lib = load_library()
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    _check_tensors([("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("out", out)],
                   q.dtype, q.device)
    _check_tensors([("S0", S0), ("S_final", S_final)], torch.float32, q.device)
    _check_tensors([("workspace", workspace)], None, q.device)
    _require(k.shape == q.shape and g.shape == q.shape, "q, k, g must share [B, T, H, d_k]")
    _require(v.shape == (B, T, H, dv) and out.shape == v.shape, "v/out must be [B, T, H, d_v]")
    _require(beta.shape == (B, T, H), "beta must be [B, T, H]")
    for name, s in (("S0", S0), ("S_final", S_final)):
        _require(s is None or s.shape == (B, H, dk, dv), f"{name} must be [B, H, d_k, d_v]")
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.kda_chunk_fwd_segmented(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(S0),
                                     _ptr(out), _ptr(S_final), B, H, T, dk, dv, int(C),
                                     int(n_seg), _ptr(workspace), nbytes, _dtype_code(q),
                                     _stream_handle(stream))
    _check(st, "kda_chunk_fwd_segmented")


def kda_chunk_fwd_segmented_noalloc(q, k, v, g, beta, S0, out, S_final, n_seg: int,
                                    C: int = 64, stream=None):
    """:func:`kda_chunk_fwd_segmented` without a workspace: the library's fixed device scratch
    (``NOALLOC_SCRATCH_BYTES``) serves instead, and nothing is allocated. For callers that cannot
    allocate device memory at the point of the call; calls that overlap on the GPU share that
    scratch and must be ordered on one stream (see include/kda.h)."""
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
    st = lib.kda_chunk_fwd_segmented_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                             _ptr(S0), _ptr(out), _ptr(S_final), B, H, T, dk, dv,
                                             int(C), int(n_seg), _dtype_code(q),
                                             _stream_handle(stream))
    _check(st, "kda_chunk_fwd_segmented_noalloc")


def kda_chunk_fwd_gated(q, k, v, g, beta, S0, gate_u, norm_w, out, S_final, cu_seqlens=None,
                        norm_eps: float = 1e-5, C: int = 64, stream=None):
    """Prefill plus the output side: ``out`` = RMSNorm(o~) * norm_w * sigma(gate_u) (see
    include/kda.h). Dense [B, T, H, d] tensors, or a packed batch with ``cu_seqlens``."""
    lib = load_library()
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    _check_tensors([("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("out", out),
                    ("gate_u", gate_u)], q.dtype, q.device)
    _check_tensors([("S0", S0), ("S_final", S_final), ("norm_w", norm_w)], torch.float32,
                   q.device)
    _require(k.shape == q.shape and g.shape == q.shape, "q, k, g must share [B, T, H, d_k]")
    _require(v.shape == (B, T, H, dv) and out.shape == v.shape and gate_u.shape == v.shape,
             "v, out, gate_u must be [B, T, H, d_v]")
    _require(beta.shape == (B, T, H), "beta must be [B, T, H]")
    _require(norm_w.shape == (dv,), "norm_w must be [d_v]")
    if cu_seqlens is not None:
        _check_tensors([("cu_seqlens", cu_seqlens)], torch.int32, q.device)
        _require(B == 1, "packed batches have a leading dimension of 1")
        n_seq = cu_seqlens.shape[0] - 1
    else:
        n_seq = B
    for name, s in (("S0", S0), ("S_final", S_final)):
        _require(s is None or s.shape == (n_seq, H, dk, dv), f"{name} must be [n_seq, H, d_k, d_v]")
    st = lib.kda_chunk_fwd_gated(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(S0),
                                 _ptr(gate_u), _ptr(norm_w), float(norm_eps), _ptr(out),
                                 _ptr(S_final), _ptr(cu_seqlens), n_seq, H, T, dk, dv, int(C),
                                 _dtype_code(q), _stream_handle(stream))
    _check(st, "kda_chunk_fwd_gated")


def kda_output_gate(o, gate_u, norm_w, y, norm_eps: float = 1e-5, stream=None):
    """y = RMSNorm(o) * norm_w * sigma(gate_u) over the last axis (d_v in {64, 128})."""
    lib = load_library()
    dv = o.shape[-1]
    _check_tensors([("o", o), ("gate_u", gate_u), ("y", y)], o.dtype, o.device)
    _check_tensors([("norm_w", norm_w)], torch.float32, o.device)
    _require(gate_u.shape == o.shape and y.shape == o.shape, "o, gate_u, y must share a shape")
    _require(norm_w.shape == (dv,), "norm_w must be [d_v]")
    st = lib.kda_output_gate(_ptr(o), _ptr(gate_u), _ptr(norm_w), float(norm_eps), _ptr(y),
                             o.numel() // dv, dv, _dtype_code(o), _stream_handle(stream))
    _check(st, "kda_output_gate")


def _layer_n_seq(q, cu_seqlens):
    if cu_seqlens is None:
        return q.shape[0]
    _check_tensors([("cu_seqlens", cu_seqlens)], torch.int32, q.device)
    _require(q.shape[0] == 1, "packed batches have a leading dimension of 1")
    return cu_seqlens.shape[0] - 1


def _check_pre_params(H, d, conv_q, conv_k, conv_v, A_log, b_decay, device):
    _check_tensors([("conv_q", conv_q), ("conv_k", conv_k), ("conv_v", conv_v),
                    ("A_log", A_log), ("b_decay", b_decay)], torch.float32, device)
    for name, c in (("conv_q", conv_q), ("conv_k", conv_k), ("conv_v", conv_v)):
        _require(c.shape == (H, 4, d), f"{name} must be tap-major [H, 4, d]")
    _require(A_log.shape == (H,) and b_decay.shape == (H, d), "A_log [H], b_decay [H, d]")


def kda_pre_core(q_raw, k_raw, v_raw, z, conv_q, conv_k, conv_v, A_log, b_decay, q, k, v, g,
                 cu_seqlens=None, stream=None):
    """The inputs of the recurrence from the raw projections (see include/kda.h)."""
    lib = load_library()
    B, T, H, d = q_raw.shape
    _check_tensors([(n, t) for n, t in (("q_raw", q_raw), ("k_raw", k_raw), ("v_raw", v_raw),
                                        ("z", z), ("q", q), ("k", k), ("v", v), ("g", g))],
                   q_raw.dtype, q_raw.device)
    for n, t in (("k_raw", k_raw), ("v_raw", v_raw), ("z", z), ("q", q), ("k", k), ("v", v),
                 ("g", g)):
        _require(t.shape == q_raw.shape, f"{n} must be [B, T, H, d] like q_raw")
    _check_pre_params(H, d, conv_q, conv_k, conv_v, A_log, b_decay, q_raw.device)
    n_seq = _layer_n_seq(q_raw, cu_seqlens)
    st = lib.kda_pre_core(*(_ptr(t) for t in (q_raw, k_raw, v_raw, z, conv_q, conv_k, conv_v,
                                              A_log, b_decay, q, k, v, g, cu_seqlens)),
                          n_seq, H, T, d, _dtype_code(q_raw), _stream_handle(stream))
    _check(st, "kda_pre_core")


def kda_chunk_fwd_fused(q_raw, k_raw, v_raw, z, beta, conv_q, conv_k, conv_v, A_log, b_decay,
                        S0, out, S_final, gate_u=None, norm_w=None, cu_seqlens=None,
                        norm_eps: float = 1e-5, C: int = 64, stream=None):
    """The layer from the raw projections in one kernel (input side fused; output side fused
    when ``gate_u`` is given). See include/kda.h."""
    lib = load_library()
    B, T, H, d = q_raw.shape
    _check_tensors([(n, t) for n, t in (("q_raw", q_raw), ("k_raw", k_raw), ("v_raw", v_raw),
                                        ("z", z), ("beta", beta), ("out", out),
                                        ("gate_u", gate_u))], q_raw.dtype, q_raw.device)
    for n, t in (("k_raw", k_raw), ("v_raw", v_raw), ("z", z), ("out", out)):
        _require(t.shape == q_raw.shape, f"{n} must be [B, T, H, d] like q_raw")
    _require(beta.shape == (B, T, H), "beta must be [B, T, H]")
    _require(gate_u is None or gate_u.shape == out.shape, "gate_u must be shaped like out")
    _check_pre_params(H, d, conv_q, conv_k, conv_v, A_log, b_decay, q_raw.device)
    _check_tensors([("S0", S0), ("S_final", S_final), ("norm_w", norm_w)], torch.float32,
                   q_raw.device)
    n_seq = _layer_n_seq(q_raw, cu_seqlens)
    st = lib.kda_chunk_fwd_fused(*(_ptr(t) for t in (q_raw, k_raw, v_raw, z, beta, conv_q, conv_k,
                                                     conv_v, A_log, b_decay, S0, gate_u, norm_w)),
                                 float(norm_eps), _ptr(out), _ptr(S_final), _ptr(cu_seqlens),
                                 n_seq, H, T, d, d, int(C), _dtype_code(q_raw),
                                 _stream_handle(stream))
    _check(st, "kda_chunk_fwd_fused")


def kda_recurrent_steps(q, k, v, g, beta, S, out, stream=None):
    """K decode tokens per (sequence, head): q, k, g [N, K, H, d_k]; v, out [N, K, H, d_v];
    beta [N, K, H]; S (fp32 [N, H, d_k, d_v]) updated in place."""
    lib = load_library()
    N, K, H, dk = q.shape
    dv = v.shape[-1]
    _check_tensors([("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("out", out)],
                   q.dtype, q.device)
    _check_tensors([("S", S)], torch.float32, q.device)
    _require(k.shape == q.shape and g.shape == q.shape, "q, k, g must share [N, K, H, d_k]")
    _require(v.shape == (N, K, H, dv) and out.shape == v.shape, "v/out must be [N, K, H, d_v]")
    _require(beta.shape == (N, K, H), "beta must be [N, K, H]")
    _require(S.shape == (N, H, dk, dv), "S must be [N, H, d_k, d_v]")
    st = lib.kda_recurrent_steps(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(S),
                                 _ptr(out), N, K, H, dk, dv, _dtype_code(q), _stream_handle(stream))
    _check(st, "kda_recurrent_steps")


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


def _on(stream):
    """Makes ``stream`` torch's current stream for the allocations and copies of a call, so
    that the caching allocator records them on the stream the kernel runs on."""
    return torch.cuda.stream(stream) if stream is not None else contextlib.nullcontext()


def chunk_fwd(q, k, v, g, beta, S0=None, C: int = 64, want_state: bool = True, stream=None):
    """Allocates the outputs with torch (on ``stream``) and calls :func:`kda_chunk_fwd`."""
    B, T, H, dk = q.shape
    with _on(stream):
        out = torch.empty(B, T, H, v.shape[-1], dtype=q.dtype, device=q.device)
        Sf = (torch.empty(B, H, dk, v.shape[-1], dtype=torch.float32, device=q.device)
              if want_state else None)
        kda_chunk_fwd(q, k, v, g, beta, S0, out, Sf, C=C, stream=stream)
    return out, Sf


def chunk_fwd_varlen(q, k, v, g, beta, cu_seqlens, S0=None, C: int = 64, want_state=True,
                     stream=None):
    _, T, H, dk = q.shape
    N = cu_seqlens.shape[0] - 1
    with _on(stream):
        out = torch.empty(1, T, H, v.shape[-1], dtype=q.dtype, device=q.device)
        Sf = (torch.empty(N, H, dk, v.shape[-1], dtype=torch.float32, device=q.device)
              if want_state else None)
        kda_chunk_fwd_varlen(q, k, v, g, beta, S0, out, Sf, cu_seqlens, C=C, stream=stream)
    return out, Sf


def chunk_fwd_segmented(q, k, v, g, beta, S0=None, C: int = 64, n_seg: int | None = None,
                        want_state: bool = True, workspace=None, stream=None):
    """Allocates the outputs (and the workspace, unless given) with torch on ``stream`` and
    calls :func:`kda_chunk_fwd_segmented`; ``n_seg=None`` takes :func:`segments_auto`."""
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if n_seg is None:
        n_seg = segments_auto(B, H, T)
    with _on(stream):
        out = torch.empty(B, T, H, dv, dtype=q.dtype, device=q.device)
        Sf = (torch.empty(B, H, dk, dv, dtype=torch.float32, device=q.device)
              if want_state else None)
        need = segmented_workspace_bytes(B, H, T, dk, dv, n_seg)
        if workspace is None and need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        kda_chunk_fwd_segmented(q, k, v, g, beta, S0, out, Sf, n_seg, workspace, C=C,
                                stream=stream)
    return out, Sf


def recurrent_step(q, k, v, g, beta, S, stream=None):
    with _on(stream):
        out = torch.empty(q.shape[0], q.shape[1], v.shape[-1], dtype=q.dtype, device=q.device)
        kda_recurrent_step(q, k, v, g, beta, S, out, stream=stream)
    return out


class HostPipeline:
    """Reusable device buffers and streams for :func:`chunk_fwd_host`.

    The batch is processed one sequence row at a time as a three-stage pipeline on three
    streams: every host-to-device copy on one stream, back to back; each row's kernel on a
    second stream once its inputs have landed; each row's device-to-host copies on a third once
    its kernel is done. The copies in the two directions use separate engines, so the input copy
    of row i + 1, the kernel of row i and the output copy of row i - 1 run at the same time; the
    caller's stream waits for all three before the call returns."""

    def __init__(self, device):
        self.device = torch.device(device)
        self.h2d = torch.cuda.Stream(device=self.device)
        self.compute = torch.cuda.Stream(device=self.device)
        self.d2h = torch.cuda.Stream(device=self.device)
        self.streams = [self.h2d, self.compute, self.d2h]
        self.bufs = {}

    def buffer(self, name, shape, dtype):
        t = self.bufs.get(name)
        if t is None or t.shape != torch.Size(shape) or t.dtype != dtype:
            t = torch.empty(shape, dtype=dtype, device=self.device)
            self.bufs[name] = t
        return t


def chunk_fwd_host(q, k, v, g, beta, S0=None, C: int = 64, device=None, stream=None,
                   out_host=None, state_host=None, pipeline: HostPipeline | None = None):
    """End-to-end call on HOST tensors: copies the inputs to the device, runs
    :func:`kda_chunk_fwd`, and copies the output and final state back into ``out_host`` /
    ``state_host`` (allocated pinned if not given).

    Rows of the batch are independent problems, so the work is split by batch row over the
    streams of ``pipeline`` (created if not given): the copies of one row overlap the kernel
    and the copies of its neighbours. Pinned host tensors make the copies asynchronous. The
    function returns once the results are in the host tensors."""
    device = torch.device(device or torch.device("cuda", torch.cuda.current_device()))
    pl = pipeline or HostPipeline(device)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    caller = stream if stream is not None else torch.cuda.current_stream(device)
    if out_host is None:
        out_host = torch.empty(B, T, H, dv, dtype=q.dtype, pin_memory=True)
    if state_host is None:
        state_host = torch.empty(B, H, dk, dv, dtype=torch.float32, pin_memory=True)
    dq = pl.buffer("q", q.shape, q.dtype)
    dk_ = pl.buffer("k", k.shape, k.dtype)
    dv_ = pl.buffer("v", v.shape, v.dtype)
    dg = pl.buffer("g", g.shape, g.dtype)
    db = pl.buffer("beta", beta.shape, beta.dtype)
    dS0 = None if S0 is None else pl.buffer("S0", S0.shape, torch.float32)
    dout = pl.buffer("out", (B, T, H, dv), q.dtype)
    dSf = pl.buffer("Sf", (B, H, dk, dv), torch.float32)
    for s in pl.streams:  # earlier work of the caller (e.g. on the buffers) comes first
        s.wait_stream(caller)
    for b in range(B):
        with torch.cuda.stream(pl.h2d):
            for src, dst in ((q, dq), (k, dk_), (v, dv_), (g, dg), (beta, db)):
                dst[b:b + 1].copy_(src[b:b + 1], non_blocking=True)
            if S0 is not None:
                dS0[b:b + 1].copy_(S0[b:b + 1], non_blocking=True)
            landed = torch.cuda.Event()
            landed.record(pl.h2d)
        pl.compute.wait_event(landed)
        kda_chunk_fwd(dq[b:b + 1], dk_[b:b + 1], dv_[b:b + 1], dg[b:b + 1], db[b:b + 1],
                      None if S0 is None else dS0[b:b + 1], dout[b:b + 1], dSf[b:b + 1],
                      C=C, stream=pl.compute)
        done = torch.cuda.Event()
        done.record(pl.compute)
        pl.d2h.wait_event(done)
        with torch.cuda.stream(pl.d2h):
            out_host[b:b + 1].copy_(dout[b:b + 1], non_blocking=True)
            state_host[b:b + 1].copy_(dSf[b:b + 1], non_blocking=True)
    for s in pl.streams:
        caller.wait_stream(s)
    caller.synchronize()
    return out_host, state_host
