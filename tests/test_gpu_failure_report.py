"""Device-side failure report, without a GPU fault.

A bounded wait that nothing answers gives up after its limit, latches KDA_ERR_TIMEOUT in the
library's device status word and returns; kda_sync_status reports the code once and clears it,
and the context keeps running kernels correctly. The wait is on an mbarrier that no thread or
copy ever completes, limited by the GPU global timer: nothing faults, traps or hangs.
"""
import time

import numpy as np
import pytest
import torch

import kda_synth
import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    import gated_delta_rule_167_b300 as m
    from gated_delta_rule_167_b300 import build as kbuild

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    kbuild.build()
    m.load_library()
    torch.cuda.set_device(0)
    return m


def _raw_status(kda):
    return kda.load_library().kda_sync_status(kda._stream_handle(None))


def test_unanswered_wait_reports_timeout_once(kda):
    torch.cuda.synchronize()
    assert _raw_status(kda) == kda.KDA_OK  # nothing latched before
    limit_ns = 20_000_000  # 20 ms
    t0 = time.perf_counter()
    assert kda.kda_wait_selftest(limit_ns) == kda.KDA_OK
    status = _raw_status(kda)  # synchronises the stream
    elapsed = time.perf_counter() - t0
    assert status == kda.KDA_ERR_TIMEOUT
    assert elapsed >= 0.9 * limit_ns * 1e-9  # the wait lasted its limit
    assert elapsed < 5.0
    assert _raw_status(kda) == kda.KDA_OK  # reported once, then cleared
    with pytest.raises(kda.KdaError):  # through the Python binding it raises
        kda.kda_wait_selftest(limit_ns)
        kda.kda_sync_status()


def test_invalid_limit_is_rejected_on_the_host(kda):
    assert kda.kda_wait_selftest(0) == kda.KDA_ERR_INVALID_ARG
    assert kda.kda_wait_selftest(2 * 10**10) == kda.KDA_ERR_INVALID_ARG
    assert _raw_status(kda) == kda.KDA_OK


def test_context_runs_the_prefill_after_a_timeout(kda):
    assert kda.kda_wait_selftest(1_000_000) == kda.KDA_OK
    assert _raw_status(kda) == kda.KDA_ERR_TIMEOUT
    inp = kda_synth.make_prefill_inputs(1, 200, 2, 128, 128, "bf16", seed=3)
    dev = torch.device("cuda", 0)
    x = [inp[n].to(dev) for n in ("q", "k", "v", "g", "beta")]
    out, s_final = kda.chunk_fwd(*x, None, C=64)
    kda.kda_sync_status()  # raises on any latched error
    f64 = kda_synth.to_f64_numpy
    o_ref, s_ref = oracle.recurrent(*(f64(inp[n]) for n in ("q", "k", "v", "g", "beta")))
    o = out.float().cpu().double().numpy()
    assert np.linalg.norm(o - o_ref) / np.linalg.norm(o_ref) <= 1e-2
    s = s_final.cpu().double().numpy()
    assert np.linalg.norm(s - s_ref) / np.linalg.norm(s_ref) <= 1e-2
