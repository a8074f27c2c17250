"""GPU parity of the tensor-core prefill at head size 64 (the nano-K3 shape: 8 heads, d_k = d_v
= 64; Kimi K3 wiki, "Tableau des spécifications", nano-K3 block) against the fp64 CPU oracle.

bf16 inputs with C = 64 or 128 take the tensor-core kernel, which runs a head of 64 channels in
its 128-channel tiles with the upper half zero; the bar is the bf16 one (rel-L2 <= 1e-2,
max-abs <= 5e-2) on outputs and final states.
"""
import numpy as np
import pytest
import torch

import kda_synth
import oracle

pytestmark = pytest.mark.gpu

BF16_REL = 1e-2
BF16_ABS = 5e-2
DEV = torch.device("cuda", 0)
f64 = kda_synth.to_f64_numpy
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


def check(got, ref, what):
    got = np.asarray(got, dtype=np.float64)
    e = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))
    m = float(np.abs(got - ref).max()) if got.size else 0.0
    assert e <= BF16_REL and m <= BF16_ABS, f"{what}: rel-L2 {e:.3e}, max-abs {m:.3e}"


def host(t):
    return t.float().cpu().double().numpy()


def test_nano_B64_H8_T2048_sampled(kda):
    """The nano-K3 layer shape at full size (512 problems, 3.5 waves); sampled problems."""
    inp = kda_synth.make_prefill_inputs(64, 2048, 8, 64, 64, "bf16", seed=3, g_bias=True,
                                        device=DEV)
    out, Sf = kda.chunk_fwd(*(inp[n] for n in NAMES), C=64)
    kda.kda_sync_status()
    for b, h in ((0, 0), (17, 5), (40, 2), (63, 7)):
        sub = [f64(inp[n][b:b + 1, :, h:h + 1].cpu()) for n in NAMES]
        o_ref, S_ref = oracle.recurrent(*sub)
        check(host(out[b:b + 1, :, h:h + 1]), o_ref, f"out[b={b},h={h}]")
        check(Sf[b:b + 1, h:h + 1].cpu().double().numpy(), S_ref, f"S_final[b={b},h={h}]")


@pytest.mark.parametrize("C", [64, 128])
@pytest.mark.parametrize("T", [1, 63, 64, 65, 200])
def test_lengths_with_initial_state(kda, C, T):
    inp = kda_synth.make_prefill_inputs(2, T, 3, 64, 64, "bf16", seed=T + C, S0_std=0.1)
    S0 = inp["S0"]
    out, Sf = kda.chunk_fwd(*(inp[n].to(DEV) for n in NAMES), S0.to(DEV), C=C)
    kda.kda_sync_status()
    o_ref, S_ref = oracle.recurrent(*(f64(inp[n]) for n in NAMES), f64(S0))
    check(host(out), o_ref, "out")
    check(Sf.cpu().double().numpy(), S_ref, "S_final")


def test_no_states_and_strong_decay(kda):
    """No initial state, no final state wanted, g at the floor on every channel."""
    inp = kda_synth.make_prefill_inputs(1, 150, 2, 64, 64, "bf16", seed=8)
    inp["g"] = torch.full_like(inp["g"], -5.0)
    out, Sf = kda.chunk_fwd(*(inp[n].to(DEV) for n in NAMES), C=64, want_state=False)
    kda.kda_sync_status()
    assert Sf is None
    o_ref, _ = oracle.recurrent(*(f64(inp[n]) for n in NAMES))
    check(host(out), o_ref, "out")


@pytest.mark.parametrize("C", [64, 128])
def test_varlen_edges(kda, C):
    cu = torch.tensor([0, 1, 1, 65, 66, 300, 429], dtype=torch.int32)  # lengths 1,0,64,1,234,129
    T = int(cu[-1])
    N = cu.numel() - 1
    inp = kda_synth.make_prefill_inputs(1, T, 2, 64, 64, "bf16", seed=C + 1, S0_std=0.05,
                                        n_state=N)
    out, Sf = kda.chunk_fwd_varlen(*(inp[n].to(DEV) for n in NAMES), cu.to(DEV),
                                   S0=inp["S0"].to(DEV), C=C)
    kda.kda_sync_status()
    o_ref, S_ref = oracle.recurrent_varlen(*(f64(inp[n]) for n in NAMES), cu.numpy(),
                                           f64(inp["S0"]))
    check(host(out), o_ref, "out")
    check(Sf.cpu().double().numpy(), S_ref, "S_final")


def test_segmented_matches_oracle(kda):
    """Parallel along T at head size 64: the transitions run in the same kernel from the
    identity (only the 64 x 64 block of it exists), then the scan and every segment."""
    inp = kda_synth.make_prefill_inputs(1, 4096, 2, 64, 64, "bf16", seed=12, S0_std=0.05)
    x = [inp[n].to(DEV) for n in NAMES]
    out, Sf = kda.chunk_fwd_segmented(*x, inp["S0"].to(DEV), C=64, n_seg=8)
    kda.kda_sync_status()
    o_ref, S_ref = oracle.recurrent(*(f64(inp[n]) for n in NAMES), f64(inp["S0"]))
    check(host(out), o_ref, "out")
    check(Sf.cpu().double().numpy(), S_ref, "S_final")
