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
    "kda_chunk_fwd_segmented_noalloc", "NOALLOC_SCRATCH_BYTES",
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

    The batch is processed one sequence row at a time on two alternating streams, so that the
    host-to-device copy of row i + 1, the kernel of row i and the device-to-host copy of row
    i - 1 can run at the same time (PCIe copies in the two directions use separate engines).
    Every row's copies and its kernel are ordered on that row's stream; the caller's stream
    waits for both streams before the call returns."""

    def __init__(self, device, n_streams: int = 2):
        self.device = torch.device(device)
        self.streams = [torch.cuda.Stream(device=self.device) for _ in range(n_streams)]
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
        s = pl.streams[b % len(pl.streams)]
        with torch.cuda.stream(s):
            for src, dst in ((q, dq), (k, dk_), (v, dv_), (g, dg), (beta, db)):
                dst[b:b + 1].copy_(src[b:b + 1], non_blocking=True)
            if S0 is not None:
                dS0[b:b + 1].copy_(S0[b:b + 1], non_blocking=True)
            kda_chunk_fwd(dq[b:b + 1], dk_[b:b + 1], dv_[b:b + 1], dg[b:b + 1], db[b:b + 1],
                          None if S0 is None else dS0[b:b + 1], dout[b:b + 1], dSf[b:b + 1],
                          C=C, stream=s)
            out_host[b:b + 1].copy_(dout[b:b + 1], non_blocking=True)
            state_host[b:b + 1].copy_(dSf[b:b + 1], non_blocking=True)
    for s in pl.streams:
        caller.wait_stream(s)
    caller.synchronize()
    return out_host, state_host
