"""The allocation-free segmented prefill (kda_chunk_fwd_segmented_noalloc) against the
workspace entry point (kda_chunk_fwd_segmented), through the C ABI.

Some callers cannot allocate device memory where they call the library (their memory belongs
to a fixed arena, or their host gives them no allocator); this entry point serves them from a
fixed scratch array in the library's device image. Two calls in a row, on different inputs and
shapes, must each match the workspace entry point: the second call reuses the array the first
one left behind. A request larger than the fixed scratch is refused before any launch.

This file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import kda_synth

pytestmark = pytest.mark.gpu

BF16_REL = 1e-2
BF16_ABS = 5e-2
NAMES = ("q", "k", "v", "g", "beta")


@pytest.fixture(scope="module")
def kda():
    import gated_delta_rule_167_b300 as m
    from gated_delta_rule_167_b300 import build as kbuild

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    kbuild.build()
    m.load_library()
    torch.cuda.set_device(0)
    return m


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _close(got, ref, what):
    got = got.double().cpu().numpy()
    ref = ref.double().cpu().numpy()
    rel = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))
    mx = float(np.abs(got - ref).max())
    assert rel <= BF16_REL and mx <= BF16_ABS, f"{what}: rel-L2 {rel:.3e}, max-abs {mx:.3e}"


def _noalloc_call(kda, x, S0, out, Sf, n_seg, C=64):
    lib = kda.load_library()
    B, T, H, dk = x[0].shape
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.kda_chunk_fwd_segmented_noalloc(*(_ptr(t) for t in x), _ptr(S0), _ptr(out),
                                               _ptr(Sf), B, H, T, dk, dk, C, n_seg,
                                               kda.KDA_DTYPE_BF16, stream)


def test_noalloc_matches_workspace_entry_point_on_two_calls(kda):
    dev = torch.device("cuda", 0)
    cases = [  # (B, H, T, n_seg, seed, with S0)
        (1, 8, 4096, 10, 0, True),
        (2, 3, 3000, 7, 5, False),
    ]
    for B, H, T, n_seg, seed, with_S0 in cases:
        need = kda.segmented_workspace_bytes(B, H, T, 128, 128, n_seg)
        assert 0 < need <= kda.NOALLOC_SCRATCH_BYTES
        inp = kda_synth.make_prefill_inputs(B, T, H, 128, 128, "bf16", seed=seed,
                                            S0_std=0.02 if with_S0 else 0.0, device=dev)
        x = [inp[n] for n in NAMES]
        S0 = inp["S0"]
        ref_out, ref_S = kda.chunk_fwd_segmented(*x, S0, C=64, n_seg=n_seg)
        out = torch.full_like(ref_out, float("nan"))
        Sf = torch.full_like(ref_S, float("nan"))
        st = _noalloc_call(kda, x, S0, out, Sf, n_seg)
        assert st == kda.KDA_OK, kda.load_library().kda_last_error()
        kda.kda_sync_status()
        _close(out, ref_out, f"out (B={B}, H={H}, T={T}, n_seg={n_seg})")
        _close(Sf, ref_S, f"S_final (B={B}, H={H}, T={T}, n_seg={n_seg})")


def test_noalloc_refuses_requests_beyond_its_scratch(kda):
    B, H, T, n_seg = 1, 96, 8192, 8
    need = kda.segmented_workspace_bytes(B, H, T, 128, 128, n_seg)
    assert need > kda.NOALLOC_SCRATCH_BYTES
    dev = torch.device("cuda", 0)
    x = [torch.zeros(B, T, H, 128, dtype=torch.bfloat16, device=dev) for _ in range(4)]
    x.append(torch.zeros(B, T, H, dtype=torch.bfloat16, device=dev))
    out = torch.zeros(B, T, H, 128, dtype=torch.bfloat16, device=dev)
    st = _noalloc_call(kda, x, None, out, None, n_seg)
    assert st == kda.KDA_ERR_UNSUPPORTED
    assert b"scratch" in kda.load_library().kda_last_error()
    assert not out.any()  # nothing was launched
