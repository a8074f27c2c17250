"""The C-ABI library builds, loads and exports every entry point that include/kda.h declares.

These run without a GPU: they dlopen libkda.so and only call entry points (or argument
combinations) that return before touching the device.
"""
import ctypes
import os
import re
import subprocess

import pytest

from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "kda.h")


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z_0-9]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from gated_delta_rule_167_b300 import build as kbuild
    import gated_delta_rule_167_b300 as kda

    kbuild.build()
    return kda.load_library()


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("kda_chunk_fwd", "kda_chunk_fwd_varlen", "kda_recurrent_step"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    import gated_delta_rule_167_b300 as kda

    names = _declared_functions()
    for n in names:
        assert hasattr(lib, n), f"libkda.so does not export {n}"
    out = subprocess.run(["nm", "-D", "--defined-only", kda.lib_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(kda_\w+)", out))
    assert set(names) <= exported
    assert set(kda.EXPORTED_SYMBOLS) <= exported


def test_status_strings_and_version(lib):
    assert lib.kda_status_string(0) == b"KDA_OK"
    assert lib.kda_status_string(4) == b"KDA_ERR_TIMEOUT"
    assert lib.kda_status_string(99) == b"KDA_ERR_UNKNOWN"
    assert lib.kda_version() >= 100


def _fake(n=0x10000):
    return ctypes.c_void_p(n)  # never dereferenced: every call below fails validation first


@pytest.mark.parametrize(
    "args,status",
    [
        (dict(d_k=96, d_v=96), 2),          # unsupported head size
        (dict(d_k=128, d_v=64), 2),         # d_k != d_v
        (dict(C=48), 2),                    # unsupported block size
        (dict(H=0), 1),                     # no heads
        (dict(B=-1), 1),
        (dict(dtype=7), 1),
        (dict(q=None), 1),                  # missing input
        (dict(out=ctypes.c_void_p(0x10008)), 1),  # misaligned output
    ],
)
def test_chunk_fwd_rejects_bad_arguments_before_launch(lib, args, status):
    a = dict(q=_fake(), k=_fake(), v=_fake(), g=_fake(), beta=_fake(), S0=None, out=_fake(),
             S_final=None, B=1, H=1, T=8, d_k=128, d_v=128, C=64, dtype=1)
    a.update(args)
    st = lib.kda_chunk_fwd(a["q"], a["k"], a["v"], a["g"], a["beta"], a["S0"], a["out"],
                           a["S_final"], a["B"], a["H"], a["T"], a["d_k"], a["d_v"], a["C"],
                           a["dtype"], None)
    assert st == status
    assert lib.kda_last_error() != b""


def test_varlen_and_decode_reject_bad_arguments(lib):
    st = lib.kda_chunk_fwd_varlen(_fake(), _fake(), _fake(), _fake(), _fake(), None, _fake(),
                                  None, None, 2, 1, 16, 128, 128, 64, 1, None)
    assert st == 1  # cu_seqlens missing
    st = lib.kda_chunk_fwd_varlen(_fake(), _fake(), _fake(), _fake(), _fake(), None, _fake(),
                                  None, ctypes.c_void_p(0x10002), 2, 1, 16, 128, 128, 64, 1, None)
    assert st == 1  # misaligned cu_seqlens
    st = lib.kda_recurrent_step(_fake(), _fake(), _fake(), _fake(), _fake(), None, _fake(),
                                4, 2, 128, 128, 1, None)
    assert st == 1  # S missing
    st = lib.kda_recurrent_step(_fake(), _fake(), _fake(), _fake(), _fake(), _fake(), _fake(),
                                4, 2, 32, 32, 1, None)
    assert st == 2  # unsupported head size
    assert lib.kda_recurrent_step(None, None, None, None, None, None, None, 0, 2, 128, 128, 1,
                                  None) == 0  # N = 0 is a no-op


def test_segmented_workspace_size_and_validation(lib):
    # 4 segments of 64 tokens (T = 256), one (b, h): 3 x (M + S~) + 4 x S_in, 64 KiB each
    assert lib.kda_chunk_fwd_segmented_workspace(1, 1, 256, 128, 128, 4) == 4 * 128 * 128 * (3 * 2 + 4)
    assert lib.kda_chunk_fwd_segmented_workspace(2, 3, 256, 128, 128, 4) == 6 * 4 * 128 * 128 * 10
    assert lib.kda_chunk_fwd_segmented_workspace(1, 1, 256, 128, 128, 1) == 0
    # more segments than 64-token blocks: one segment per block
    assert lib.kda_chunk_fwd_segmented_workspace(1, 1, 130, 128, 128, 8) == 4 * 128 * 128 * (2 * 2 + 3)
    assert lib.kda_chunk_fwd_segmented_workspace(1, 1, 256, 128, 128, 0) == 0
    # workspace missing / too small: rejected before anything is launched
    a = [_fake()] * 5 + [None, _fake(), None]
    assert lib.kda_chunk_fwd_segmented(*a, 1, 1, 256, 128, 128, 64, 4, None, 0, 1, None) == 1
    assert lib.kda_chunk_fwd_segmented(*a, 1, 1, 256, 128, 128, 64, 4, _fake(), 100, 1, None) == 1
    assert b"workspace" in lib.kda_last_error()
    assert lib.kda_chunk_fwd_segmented(*a, 1, 1, 256, 128, 128, 64, 0, _fake(), 0, 1, None) == 1
    # transitions and scan: host validation
    assert lib.kda_segment_transitions(_fake(), _fake(), _fake(), _fake(), None, _fake(), 1, 1,
                                       256, 64, 4, 128, 128, 64, 1, None) == 1
    assert lib.kda_segment_transitions(_fake(), _fake(), _fake(), _fake(), _fake(), _fake(), 1, 1,
                                       256, 0, 4, 128, 128, 64, 1, None) == 1
    assert lib.kda_segment_scan(None, None, None, _fake(), 0, 1, 1, 128, 128, None) == 1
    assert lib.kda_segment_scan(None, None, None, _fake(), 3, 1, 1, 128, 128, None) == 1


def test_segments_auto_is_sane(lib):
    # a batch that fills the SMs stays whole; few problems over long T are split
    assert lib.kda_segments_auto(4, 96, 8192) == 1
    assert lib.kda_segments_auto(1, 8, 4096) > 1
    assert lib.kda_segments_auto(1, 1, 65536) > 8
    assert lib.kda_segments_auto(1, 1, 64) == 1
    assert lib.kda_segments_auto(0, 1, 64) == 1


def test_noalloc_entry_point_refuses_oversized_requests_on_the_host(lib):
    # 96 heads x 8192 tokens in 8 segments needs ~138 MB of scratch, beyond the fixed 32 MiB:
    # refused before the device is touched
    a = [_fake()] * 5 + [None, _fake(), None]
    assert lib.kda_chunk_fwd_segmented_noalloc(*a, 1, 96, 8192, 128, 128, 64, 8, 1, None) == 2
    assert b"scratch" in lib.kda_last_error()
    assert lib.kda_chunk_fwd_segmented_noalloc(*a, 1, 96, 8192, 128, 128, 64, 0, 1, None) == 1


def test_binding_refuses_host_tensors(lib):
    """No CPU fallback: the binding sends host tensors to no kernel and computes nothing itself;
    every mirror of a compute entry point raises before the call."""
    import torch
    import gated_delta_rule_167_b300 as kda

    B, T, H, d = 1, 8, 2, 64
    bf = torch.bfloat16
    q, k, v, g = (torch.zeros(B, T, H, d, dtype=bf) for _ in range(4))
    beta = torch.zeros(B, T, H, dtype=bf)
    out = torch.empty(B, T, H, d, dtype=bf)
    with pytest.raises(ValueError, match="must be on"):
        kda.kda_chunk_fwd(q, k, v, g, beta, None, out, None)
    S = torch.zeros(B, H, d, d)
    with pytest.raises(ValueError, match="must be on"):
        kda.kda_recurrent_step(q[:, 0], k[:, 0], v[:, 0], g[:, 0], beta[:, 0], S, out[:, 0])
    u, w = torch.zeros(T, d, dtype=bf), torch.ones(d)
    with pytest.raises(ValueError, match="must be on"):
        kda.kda_output_gate(out[0, :, 0], u, w, out[0, :, 0].clone())
