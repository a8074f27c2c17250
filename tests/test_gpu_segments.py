"""GPU parity of the segment-parallel path (transitions, scan, segmented prefill) against the
fp64 oracle.

The transition of a stretch of tokens is defined by the pages as the product of its M_t, and S~
as the state reached from S = 0 (Kimi K3 wiki, "Notations mathématiques", rows M_t and S~;
"Glossaire", entry "KCP"). The oracle's recurrence gives both by definition: run from S0 = I
with v = 0 for M (then S_t = M_t S_{t-1}), from S0 = 0 with the real v for S~. The segmented
prefill must equal the plain recurrence over the whole sequence.
"""
import numpy as np
import pytest
import torch

import kda_synth
import oracle
from oracle import chunkwise
from tests.test_gpu_parity import BF16_ABS, BF16_REL, DEV, F32_REL, check, f64, kda, oracle_dense, to_dev  # noqa: F401

pytestmark = pytest.mark.gpu

NAMES = ("q", "k", "v", "g", "beta")


def oracle_transition(inp, b, h, a, e):
    """(M, S~) of tokens [a, e) of problem (b, h), by running the recurrence from I and 0."""
    sub = {n: f64(inp[n][b:b + 1, a:e, h:h + 1]) for n in NAMES}
    dk, dv = sub["k"].shape[-1], sub["v"].shape[-1]
    eye = np.eye(dk)[None, None]
    _, M = oracle.recurrent(sub["q"], sub["k"], np.zeros_like(sub["v"]), sub["g"], sub["beta"], eye)
    _, St = oracle.recurrent(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"], None)
    return M[0, 0], St[0, 0]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("seg_len,n_seg", [(128, 3), (100, 4), (64, 5)])
def test_transitions_match_definition(kda, dtype, seg_len, n_seg):
    """M and S~ entry by entry. The decay is scaled down (g x 0.005) so that M stays O(1): with
    the workload's decay a 128-token M is below 1e-100 and its relative error means nothing."""
    B, T, H = 2, 300, 3  # the last segment is partial (or empty for 64 x 5 = 320 > 300)
    inp = kda_synth.make_prefill_inputs(B, T, H, 128, 128, dtype, seed=seg_len + n_seg)
    inp["g"] = (inp["g"].float() * 0.005).to(inp["g"].dtype)
    q, k, v, g, b = to_dev(inp)
    M = torch.empty(n_seg, B, H, 128, 128, device=DEV)
    St = torch.empty_like(M)
    kda.kda_segment_transitions(k, v, g, b, M, St, seg_len, C=64)
    kda.kda_sync_status()
    Mh, Sh = M.cpu().double().numpy(), St.cpu().double().numpy()
    for s in range(n_seg):
        a, e = s * seg_len, min((s + 1) * seg_len, T)
        for bb, hh in ((0, 0), (1, 2)):
            if a >= e:  # empty segment: (I, 0)
                assert np.array_equal(Mh[s, bb, hh], np.eye(128))
                assert not Sh[s, bb, hh].any()
                continue
            Mr, Sr = oracle_transition(inp, bb, hh, a, e)
            check(Mh[s, bb, hh], Mr, dtype, f"M[seg {s}, b {bb}, h {hh}]")
            check(Sh[s, bb, hh], Sr, dtype, f"S~[seg {s}, b {bb}, h {hh}]")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_transitions_map_states_like_the_recurrence(kda, dtype):
    """With the workload's decay: M X + S~ for an arbitrary incoming state X equals the
    recurrence run over the segment from X (the property the scan relies on)."""
    B, T, H, seg_len, n_seg = 1, 256, 2, 96, 3
    inp = kda_synth.make_prefill_inputs(B, T, H, 128, 128, dtype, seed=7, S0_std=0.5)
    q, k, v, g, b = to_dev(inp)
    M = torch.empty(n_seg, B, H, 128, 128, device=DEV)
    St = torch.empty_like(M)
    kda.kda_segment_transitions(k, v, g, b, M, St, seg_len, C=64)
    kda.kda_sync_status()
    X = f64(inp["S0"])
    for s in range(n_seg):
        a, e = s * seg_len, min((s + 1) * seg_len, T)
        sub = {n: f64(inp[n][:, a:e]) for n in NAMES}
        _, ref = oracle.recurrent(*(sub[n] for n in NAMES), X)
        got = M[s].cpu().double().numpy() @ X + St[s].cpu().double().numpy()
        check(got, ref, dtype, f"M X + S~ [seg {s}]")


def test_scan_matches_composition(kda):
    """The scan against the composition rule of (M, S~) pairs, on random pairs with ||M|| <= 1
    (the composition itself is pinned against products of M_t on the CPU)."""
    gen = torch.Generator().manual_seed(3)
    n_seg, B, H, d = 7, 2, 3, 128
    M = torch.randn(n_seg - 1, B, H, d, d, generator=gen) / (2 * d ** 0.5)
    St = torch.randn(n_seg - 1, B, H, d, d, generator=gen) * 0.1
    S0 = torch.randn(B, H, d, d, generator=gen) * 0.1
    S_in = torch.empty(n_seg, B, H, d, d, device=DEV)
    kda.kda_segment_scan(M.to(DEV), St.to(DEV), S0.to(DEV), S_in)
    kda.kda_sync_status()
    got = S_in.cpu().double().numpy()
    for bb in range(B):
        for hh in range(H):
            state = (np.eye(d), f64(S0[bb, hh]))  # (identity transition, S0) as a pair
            ref = [state[1]]
            for s in range(n_seg - 1):
                Mc, Sc = chunkwise.compose((f64(M[s, bb, hh]), f64(St[s, bb, hh])), state)
                state = (Mc, Sc)
                ref.append(Mc @ np.zeros((d, d)) + Sc)
            for s in range(n_seg):
                check(got[s, bb, hh], ref[s], "f32", f"S_in[{s}, {bb}, {hh}]")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T,n_seg", [(300, 3), (513, 4), (1000, 16), (64, 2), (65, 2)])
def test_segmented_matches_recurrence(kda, dtype, T, n_seg):
    inp = kda_synth.make_prefill_inputs(2, T, 3, 128, 128, dtype, seed=T + n_seg, S0_std=0.05)
    q, k, v, g, b = to_dev(inp)
    out, Sf = kda.chunk_fwd_segmented(q, k, v, g, b, inp["S0"].to(DEV), C=64, n_seg=n_seg)
    kda.kda_sync_status()
    o_ref, S_ref = oracle_dense(inp)
    check(out.float().cpu().double().numpy(), o_ref, dtype, "out")
    check(Sf.cpu().double().numpy(), S_ref, dtype, "S_final")


@pytest.mark.parametrize("d", [64])
def test_segmented_small_head_size(kda, d):
    inp = kda_synth.make_prefill_inputs(1, 400, 2, d, d, "bf16", seed=d, S0_std=0.05)
    out, Sf = kda.chunk_fwd_segmented(*to_dev(inp), inp["S0"].to(DEV), C=64, n_seg=3)
    kda.kda_sync_status()
    o_ref, S_ref = oracle_dense(inp)
    check(out.float().cpu().double().numpy(), o_ref, "bf16", "out")
    check(Sf.cpu().double().numpy(), S_ref, "bf16", "S_final")


def test_segmented_B1_H8_T4096(kda):
    """The 8-head, 4096-token workload: too few (sequence, head) problems to fill the GPU, so it
    runs segmented (automatic segment count and a fixed 16)."""
    w = kda_synth.WORKLOADS[1]
    inp = kda_synth.make_prefill_inputs(w["B"], w["T"], w["H"], w["dk"], w["dv"], "bf16",
                                        w["seed"], S0_std=w["S0_std"])
    o_ref, S_ref = oracle_dense(inp)
    assert kda.segments_auto(w["B"], w["H"], w["T"]) > 1
    for n_seg in (None, 16):
        out, Sf = kda.chunk_fwd_segmented(*to_dev(inp), inp["S0"].to(DEV), C=w["C"], n_seg=n_seg)
        kda.kda_sync_status()
        check(out.float().cpu().double().numpy(), o_ref, "bf16", f"out (n_seg={n_seg})")
        check(Sf.cpu().double().numpy(), S_ref, "bf16", f"S_final (n_seg={n_seg})")


def test_segmented_long_single_sequence(kda):
    """One long sequence with two heads (T = 65536) against the recurrence over all of it."""
    inp = kda_synth.make_prefill_inputs(1, 65536, 2, 128, 128, "bf16", seed=12, S0_std=0.02)
    out, Sf = kda.chunk_fwd_segmented(*to_dev(inp), inp["S0"].to(DEV), C=64)
    kda.kda_sync_status()
    o_ref, S_ref = oracle_dense(inp)
    check(out.float().cpu().double().numpy(), o_ref, "bf16", "out")
    check(Sf.cpu().double().numpy(), S_ref, "bf16", "S_final")


def test_segmented_without_states_and_degenerate(kda):
    inp = kda_synth.make_prefill_inputs(1, 200, 2, 128, 128, "bf16", seed=2)
    x = to_dev(inp)
    out, Sf = kda.chunk_fwd_segmented(*x, None, C=64, n_seg=3, want_state=False)
    kda.kda_sync_status()
    assert Sf is None
    o_ref, _ = oracle_dense(inp, with_S0=False)
    check(out.float().cpu().double().numpy(), o_ref, "bf16", "out")
    # more segments than blocks, and T below one block: one segment per block / plain call
    for T in (130, 40):
        sub = {n: inp[n][:, :T].contiguous() for n in NAMES}
        out, Sf = kda.chunk_fwd_segmented(*to_dev(sub), None, C=64, n_seg=8)
        kda.kda_sync_status()
        o_ref, S_ref = oracle.recurrent(*(f64(sub[n]) for n in NAMES))
        check(out.float().cpu().double().numpy(), o_ref, "bf16", f"out T={T}")
        check(Sf.cpu().double().numpy(), S_ref, "bf16", f"S_final T={T}")


def test_segmented_rejects_small_workspace(kda):
    inp = kda_synth.make_prefill_inputs(1, 256, 1, 128, 128, "bf16", seed=1)
    x = to_dev(inp)
    out = torch.empty(1, 256, 1, 128, dtype=torch.bfloat16, device=DEV)
    need = kda.segmented_workspace_bytes(1, 1, 256, 128, 128, 4)
    ws = torch.empty(need - 16, dtype=torch.uint8, device=DEV)
    with pytest.raises(kda.KdaError) as ei:
        kda.kda_chunk_fwd_segmented(*x, None, out, None, 4, ws)
    assert ei.value.status == kda.KDA_ERR_INVALID_ARG


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("world", [2, 4])
def test_kcp_emulated_ranks_on_one_gpu(kda, dtype, world):
    """KCP with `world` ranks emulated as T-segments on one GPU (library transitions, exchange
    as a list, library scan, library forward per segment) equals the recurrence."""
    from gated_delta_rule_167_b300 import kcp

    inp = kda_synth.make_prefill_inputs(2, 512, 3, 128, 128, dtype, seed=world, S0_std=0.05)
    out, Sf = kcp.emulate(*to_dev(inp), world=world, S0=inp["S0"].to(DEV))
    kda.kda_sync_status()
    o_ref, S_ref = oracle_dense(inp)
    check(out.float().cpu().double().numpy(), o_ref, dtype, "out")
    check(Sf.cpu().double().numpy(), S_ref, dtype, "S_final")
