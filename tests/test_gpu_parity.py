"""GPU parity: the CUDA library (through its C ABI) against the fp64 CPU oracle.

Inputs are seeded and synthetic (kda_synth); the oracle reads exactly the values the GPU
reads. Tolerances: fp32 inputs rel-L2 <= 1e-5; bf16 inputs rel-L2 <= 1e-2 on outputs and final
states with max-abs <= 5e-2. Full-size workloads are compared on sampled (sequence, head)
problems that the oracle recomputes one by one.
"""
import numpy as np
import pytest
import torch

import kda_synth
import oracle

pytestmark = pytest.mark.gpu

F32_REL = 1e-5
BF16_REL = 1e-2
BF16_ABS = 5e-2


@pytest.fixture(scope="module")
def kda():
    import gated_delta_rule_167_b300 as m
    from gated_delta_rule_167_b300 import build as kbuild

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    kbuild.build()
    m.load_library()
    torch.cuda.set_device(0)
    return m


DEV = torch.device("cuda", 0)
f64 = kda_synth.to_f64_numpy


def rel_l2(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def check(got, ref, dtype, what):
    got = np.asarray(got, dtype=np.float64)
    e = rel_l2(got, ref)
    if dtype == "f32":
        assert e <= F32_REL, f"{what}: rel-L2 {e:.3e} > {F32_REL}"
    else:
        m = float(np.abs(got - ref).max()) if got.size else 0.0
        assert e <= BF16_REL and m <= BF16_ABS, f"{what}: rel-L2 {e:.3e}, max-abs {m:.3e}"
    return e


def to_dev(inp, names=("q", "k", "v", "g", "beta")):
    return [inp[n].to(DEV) for n in names]


def run_dense(kda, inp, C, want_state=True, with_S0=True):
    q, k, v, g, b = to_dev(inp)
    S0 = inp["S0"].to(DEV) if (with_S0 and inp["S0"] is not None) else None
    out, Sf = kda.chunk_fwd(q, k, v, g, b, S0, C=C, want_state=want_state)
    kda.kda_sync_status()
    return out.float().cpu().double().numpy(), (None if Sf is None else Sf.cpu().double().numpy())


def oracle_dense(inp, with_S0=True):
    S0 = f64(inp["S0"]) if with_S0 else None
    return oracle.recurrent(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["g"]),
                            f64(inp["beta"]), S0)


# ------------------------------------------------------------------ named workloads, full size


def test_fp32_B1_H1_T256(kda):
    w = kda_synth.WORKLOADS[0]
    inp = kda_synth.make_prefill_inputs(w["B"], w["T"], w["H"], w["dk"], w["dv"], "f32", w["seed"])
    out, Sf = run_dense(kda, inp, w["C"])
    o_ref, S_ref = oracle_dense(inp)
    check(out, o_ref, "f32", "out")
    check(Sf, S_ref, "f32", "S_final")


def test_bf16_B1_H8_T4096(kda):
    w = kda_synth.WORKLOADS[1]
    inp = kda_synth.make_prefill_inputs(w["B"], w["T"], w["H"], w["dk"], w["dv"], "bf16",
                                        w["seed"], S0_std=w["S0_std"])
    out, Sf = run_dense(kda, inp, w["C"])
    o_ref, S_ref = oracle_dense(inp)
    check(out, o_ref, "bf16", "out")
    check(Sf, S_ref, "bf16", "S_final")


def test_bf16_B4_H96_T8192_sampled(kda):
    """The K3 layer shape at full size; sampled (batch, head) problems against the oracle."""
    w = kda_synth.WORKLOADS[2]
    inp = kda_synth.make_prefill_inputs(w["B"], w["T"], w["H"], w["dk"], w["dv"], "bf16",
                                        w["seed"], g_bias=True)
    out, Sf = run_dense(kda, inp, w["C"])
    for b, h in ((0, 0), (1, 37), (2, 95), (3, 50)):
        sub = {n: inp[n][b:b + 1, :, h:h + 1] for n in ("q", "k", "v", "g", "beta")}
        o_ref, S_ref = oracle.recurrent(*(f64(sub[n]) for n in ("q", "k", "v", "g", "beta")))
        check(out[b:b + 1, :, h:h + 1], o_ref, "bf16", f"out[b={b},h={h}]")
        check(Sf[b:b + 1, h:h + 1], S_ref, "bf16", f"S_final[b={b},h={h}]")


def test_bf16_varlen8_H96_T131072_sampled(kda):
    """Packed long-context batch at full size; sampled (sequence, head) problems."""
    w = kda_synth.WORKLOADS[3]
    inp = kda_synth.make_varlen_inputs(w["T"], w["H"], w["dk"], w["dv"], w["n_seq"], "bf16",
                                       w["seed"], device=DEV)
    cu = inp["cu_seqlens"]
    q, k, v, g, b = (inp[n] for n in ("q", "k", "v", "g", "beta"))
    out, Sf = kda.chunk_fwd_varlen(q, k, v, g, b, cu.to(DEV), C=w["C"])
    kda.kda_sync_status()
    lens = (cu[1:] - cu[:-1]).tolist()
    shortest = int(np.argmin(lens))
    picks = [(shortest, 5), (0, 0), (len(lens) - 1, 95)]
    for s, h in picks:
        a, e = int(cu[s]), int(cu[s + 1])
        sub = {n: inp[n][:, a:e, h:h + 1].cpu() for n in ("q", "k", "v", "g", "beta")}
        o_ref, S_ref = oracle.recurrent(*(f64(sub[n]) for n in ("q", "k", "v", "g", "beta")))
        check(out[:, a:e, h:h + 1].float().cpu().double().numpy(), o_ref, "bf16",
              f"out[seq={s},h={h}]")
        check(Sf[s:s + 1, h:h + 1].cpu().double().numpy(), S_ref, "bf16",
              f"S_final[seq={s},h={h}]")


def test_decode_N256_H96_sampled(kda):
    """64 consecutive in-place decode steps on the full 256 x 96 state; sampled problems."""
    w = kda_synth.WORKLOADS[4]
    steps = 64
    dec = kda_synth.make_decode_inputs(w["N"], w["H"], w["dk"], w["dv"], "bf16", w["seed"],
                                       w["S0_std"], steps=steps, device=DEV)
    picks = [(0, 0), (17, 3), (128, 64), (255, 95)]
    S_host = {p: dec["S"][p[0], p[1]].cpu().double().numpy()[None, None] for p in picks}
    S = dec["S"]
    outs = []
    for st in dec["steps"]:
        outs.append(kda.recurrent_step(*(st[n] for n in ("q", "k", "v", "g", "beta")), S))
    kda.kda_sync_status()
    for (n, h) in picks:
        Sref = S_host[(n, h)]
        for t, st in enumerate(dec["steps"]):
            args = [f64(st[x][n:n + 1, h:h + 1].cpu()) for x in ("q", "k", "v", "g", "beta")]
            o_ref, Sref = oracle.decode_step(*args, Sref)
            if t in (0, steps - 1):
                check(outs[t][n:n + 1, h:h + 1].float().cpu().double().numpy(), o_ref, "bf16",
                      f"o[step {t}, n={n}, h={h}]")
        check(S[n:n + 1, h:h + 1].cpu().double().numpy(), Sref, "bf16", f"S[n={n},h={h}]")


# ------------------------------------------------------------------ small shapes and edges


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("C", [16, 32, 64, 128])
def test_small_shapes_all_block_sizes(kda, dtype, d, C):
    T = 2 * C + 7  # several blocks and a ragged tail
    inp = kda_synth.make_prefill_inputs(2, T, 3, d, d, dtype, seed=11 + C + d, S0_std=0.05)
    out, Sf = run_dense(kda, inp, C)
    o_ref, S_ref = oracle_dense(inp)
    check(out, o_ref, dtype, "out")
    check(Sf, S_ref, dtype, "S_final")


@pytest.mark.parametrize("T", [0, 1, 15, 63, 64, 65, 129])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_edge_lengths(kda, T, dtype):
    inp = kda_synth.make_prefill_inputs(1, T, 2, 128, 128, dtype, seed=T + 1, S0_std=0.1)
    out, Sf = run_dense(kda, inp, 64)
    o_ref, S_ref = oracle_dense(inp)
    if T > 0:
        check(out, o_ref, dtype, "out")
    check(Sf, S_ref, dtype, "S_final")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_no_initial_state_and_no_final_state(kda, dtype):
    inp = kda_synth.make_prefill_inputs(1, 100, 2, 128, 128, dtype, seed=5, S0_std=0.1)
    out, Sf = run_dense(kda, inp, 64, want_state=False, with_S0=False)
    assert Sf is None
    o_ref, _ = oracle_dense(inp, with_S0=False)
    check(out, o_ref, dtype, "out")


@pytest.mark.parametrize("C", [16, 64])
def test_beta_one_and_zero_edges(kda, C):
    """beta = 1 (full replacement along k) and beta = 0 (pure decay) are exact edges. The decay
    is scaled down so that the pure-decay state stays well inside the fp32 range."""
    inp = kda_synth.make_prefill_inputs(1, 130, 2, 128, 128, "f32", seed=9, S0_std=0.5)
    inp["g"] = inp["g"] * 0.05
    for val in (0.0, 1.0):
        inp["beta"] = torch.full_like(inp["beta"], val)
        out, Sf = run_dense(kda, inp, C)
        o_ref, S_ref = oracle_dense(inp)
        check(out, o_ref, "f32", f"out beta={val}")
        check(Sf, S_ref, "f32", f"S_final beta={val}")


def test_strong_decay_floor(kda):
    """g at the floor (-5 on every channel) drives every within-block factor to its range."""
    inp = kda_synth.make_prefill_inputs(1, 200, 2, 128, 128, "bf16", seed=21)
    inp["g"] = torch.full_like(inp["g"], -5.0)
    out, Sf = run_dense(kda, inp, 64)
    o_ref, S_ref = oracle_dense(inp)
    check(out, o_ref, "bf16", "out")
    check(Sf, S_ref, "bf16", "S_final")


@pytest.mark.parametrize("pattern", ["bursty", "gap"])
def test_uneven_decay(kda, pattern):
    """Decay concentrated on a few tokens: the within-block factors reach the ends of their
    range while some products across sub-blocks stay O(1). "gap" puts g = -5 on tokens 16..20
    and 34..47 of every block and 0 elsewhere; "bursty" draws g = -5 with probability 0.3 per
    token and channel, else 0."""
    inp = kda_synth.make_prefill_inputs(1, 256, 2, 128, 128, "bf16", seed=31, S0_std=0.05)
    g = torch.zeros_like(inp["g"], dtype=torch.float32)
    if pattern == "gap":
        pos = torch.arange(256) % 64
        mask = ((pos >= 16) & (pos <= 20)) | ((pos >= 34) & (pos <= 47))
        g[:, mask] = -5.0
    else:
        gen = torch.Generator().manual_seed(5)
        g = torch.where(torch.rand(g.shape, generator=gen) < 0.3, -5.0, 0.0)
    inp["g"] = g.to(inp["g"].dtype)
    out, Sf = run_dense(kda, inp, 64)
    o_ref, S_ref = oracle_dense(inp)
    check(out, o_ref, "bf16", "out")
    check(Sf, S_ref, "bf16", "S_final")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("C", [64, 128])
def test_varlen_small_edges(kda, dtype, C):
    cu = torch.tensor([0, 1, 1, 65, 66, 300, 429], dtype=torch.int32)  # lengths 1,0,64,1,234,129
    T = int(cu[-1])
    N = cu.numel() - 1
    inp = kda_synth.make_prefill_inputs(1, T, 2, 128, 128, dtype, seed=C, S0_std=0.05, n_state=N)
    q, k, v, g, b = to_dev(inp)
    out, Sf = kda.chunk_fwd_varlen(q, k, v, g, b, cu.to(DEV), S0=inp["S0"].to(DEV), C=C)
    kda.kda_sync_status()
    o_ref, S_ref = oracle.recurrent_varlen(*(f64(inp[n]) for n in ("q", "k", "v", "g", "beta")),
                                           cu.numpy(), f64(inp["S0"]))
    check(out.float().cpu().double().numpy(), o_ref, dtype, "out")
    check(Sf.cpu().double().numpy(), S_ref, dtype, "S_final")


@pytest.mark.parametrize("N", [200, 300])
def test_varlen_many_sequences_any_order(kda, N):
    """Packed batches are launched longest sequence first when they have at most 256 sequences
    (and in index order beyond): lengths 0..150 with many ties, every sequence against the
    oracle on its own tokens, per-sequence initial and final states."""
    gen = torch.Generator().manual_seed(N)
    lens = torch.randint(0, 151, (N,), generator=gen)
    lens[::7] = 64  # ties
    cu = torch.zeros(N + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(lens, 0).to(torch.int32)
    T = int(cu[-1])
    inp = kda_synth.make_prefill_inputs(1, T, 2, 128, 128, "bf16", seed=N, S0_std=0.05, n_state=N)
    q, k, v, g, b = to_dev(inp)
    out, Sf = kda.chunk_fwd_varlen(q, k, v, g, b, cu.to(DEV), S0=inp["S0"].to(DEV), C=64)
    kda.kda_sync_status()
    o_ref, S_ref = oracle.recurrent_varlen(*(f64(inp[n]) for n in ("q", "k", "v", "g", "beta")),
                                           cu.numpy(), f64(inp["S0"]))
    check(out.float().cpu().double().numpy(), o_ref, "bf16", "out")
    check(Sf.cpu().double().numpy(), S_ref, "bf16", "S_final")


def test_varlen_bad_offsets_are_reported_not_read(kda):
    """Inconsistent cu_seqlens are caught on the device and reported; nothing is read."""
    T = 64
    inp = kda_synth.make_prefill_inputs(1, T, 1, 128, 128, "bf16", seed=1)
    q, k, v, g, b = to_dev(inp)
    cu = torch.tensor([0, 40, 30, T], dtype=torch.int32, device=DEV)  # decreasing
    out = torch.zeros(1, T, 1, 128, dtype=torch.bfloat16, device=DEV)
    kda.kda_chunk_fwd_varlen(q, k, v, g, b, None, out, None, cu, C=64)
    with pytest.raises(kda.KdaError) as ei:
        kda.kda_sync_status()
    assert ei.value.status == kda.KDA_ERR_INVALID_ARG
    kda.kda_sync_status()  # cleared


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
def test_decode_small(kda, dtype, d):
    dec = kda_synth.make_decode_inputs(5, 3, d, d, dtype, seed=d, S0_std=0.3, steps=3)
    S = dec["S"].to(DEV)
    Sref = f64(dec["S"])
    for st in dec["steps"]:
        o = kda.recurrent_step(*(st[n].to(DEV) for n in ("q", "k", "v", "g", "beta")), S)
        o_ref, Sref = oracle.decode_step(*(f64(st[n]) for n in ("q", "k", "v", "g", "beta")), Sref)
        check(o.float().cpu().double().numpy(), o_ref, dtype, "o")
    kda.kda_sync_status()
    check(S.cpu().double().numpy(), Sref, dtype, "S")


def test_prefill_then_decode_continues_the_sequence(kda):
    """A decode step from the prefill's final state equals prefill over T + 1 tokens."""
    inp = kda_synth.make_prefill_inputs(2, 97, 3, 128, 128, "f32", seed=4, S0_std=0.1)
    q, k, v, g, b = to_dev(inp)
    S0 = inp["S0"].to(DEV)
    _, Sf = kda.chunk_fwd(q[:, :-1].contiguous(), k[:, :-1].contiguous(), v[:, :-1].contiguous(),
                          g[:, :-1].contiguous(), b[:, :-1].contiguous(), S0, C=64)
    o_last = kda.recurrent_step(q[:, -1].contiguous(), k[:, -1].contiguous(),
                                v[:, -1].contiguous(), g[:, -1].contiguous(),
                                b[:, -1].contiguous(), Sf)
    kda.kda_sync_status()
    o_ref, S_ref = oracle_dense(inp)
    check(o_last.cpu().double().numpy(), o_ref[:, -1], "f32", "o_last")
    check(Sf.cpu().double().numpy(), S_ref, "f32", "S")


@pytest.mark.parametrize("d,B,H", [(128, 2, 160), (64, 4, 80)])
def test_prefill_bits_repeat(kda, d, B, H):
    """The tensor-core prefill gives the same bits on every call: more problems than SMs (two
    waves, the second partial) and several blocks each, so that its warps and groups meet each
    hand-off at varying times. A race between the warps would show here as a few differing
    elements; the output is compared with the oracle on one sampled problem as well."""
    inp = kda_synth.make_prefill_inputs(B, 640, H, d, d, "bf16", seed=d + 5, S0_std=0.05,
                                        g_bias=True)
    x = to_dev(inp)
    S0 = inp["S0"].to(DEV)
    ref_out, ref_S = kda.chunk_fwd(*x, S0, C=64)
    for _ in range(6):
        out, Sf = kda.chunk_fwd(*x, S0, C=64)
        assert torch.equal(out, ref_out) and torch.equal(Sf, ref_S)
    kda.kda_sync_status()
    b, h = B - 1, H - 1
    sub = {n: inp[n][b:b + 1, :, h:h + 1] for n in ("q", "k", "v", "g", "beta")}
    o_ref, S_ref = oracle.recurrent(*(f64(sub[n]) for n in ("q", "k", "v", "g", "beta")),
                                    f64(inp["S0"][b:b + 1, h:h + 1]))
    check(ref_out[b:b + 1, :, h:h + 1].float().cpu().double().numpy(), o_ref, "bf16", "out")
    check(ref_S[b:b + 1, h:h + 1].cpu().double().numpy(), S_ref, "bf16", "S_final")


# ------------------------------------------------------------------ streams and host buffers


def test_nondefault_stream_matches_default(kda):
    """A call on a side stream allocates and writes on that stream; its result is bit-identical
    to the same call on the current stream, and both match the oracle."""
    inp = kda_synth.make_prefill_inputs(2, 300, 4, 128, 128, "bf16", seed=77, S0_std=0.05)
    x = to_dev(inp)
    S0 = inp["S0"].to(DEV)
    ref_out, ref_S = kda.chunk_fwd(*x, S0, C=64)
    side = torch.cuda.Stream(device=DEV)
    side.wait_stream(torch.cuda.current_stream(DEV))
    out, Sf = kda.chunk_fwd(*x, S0, C=64, stream=side)
    kda.kda_sync_status(side)
    torch.cuda.current_stream(DEV).wait_stream(side)
    assert torch.equal(out, ref_out) and torch.equal(Sf, ref_S)
    o_ref, S_ref = oracle_dense(inp)
    check(out.float().cpu().double().numpy(), o_ref, "bf16", "out")
    check(Sf.cpu().double().numpy(), S_ref, "bf16", "S_final")


def test_host_pipeline_matches_device_call(kda):
    """chunk_fwd_host splits the batch by row over two streams; its host results equal the
    device call's bits, including a caller stream that is not the current one."""
    inp = kda_synth.make_prefill_inputs(5, 200, 3, 128, 128, "bf16", seed=78, S0_std=0.05)
    hin = {n: inp[n].pin_memory() for n in ("q", "k", "v", "g", "beta")}
    S0h = inp["S0"].pin_memory()
    ref_out, ref_S = kda.chunk_fwd(*to_dev(inp), inp["S0"].to(DEV), C=64)
    torch.cuda.synchronize()
    side = torch.cuda.Stream(device=DEV)
    pl = kda.HostPipeline(DEV)
    for _ in range(2):  # the pipeline's buffers are reused on the second call
        oh, sh = kda.chunk_fwd_host(hin["q"], hin["k"], hin["v"], hin["g"], hin["beta"], S0h,
                                    C=64, device=DEV, stream=side, pipeline=pl)
        assert torch.equal(oh, ref_out.cpu()) and torch.equal(sh, ref_S.cpu())
    kda.kda_sync_status(side)


# ------------------------------------------------------------------ several decode tokens per call


def _decode_tokens_inputs(N, K, H, d, dtype, seed):
    dec = kda_synth.make_decode_inputs(N, H, d, d, dtype, seed=seed, S0_std=0.3, steps=K)
    stack = {n: torch.stack([st[n] for st in dec["steps"]], dim=1) for n in ("q", "k", "v", "g", "beta")}
    return dec, stack  # stack: [N, K, H, ...]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("K", [1, 3, 8, 11])
def test_decode_tokens_equal_single_steps_and_oracle(kda, dtype, d, K):
    """K tokens in one call agree with K single-token calls to fp32 rounding (the same arithmetic
    per token, the state kept in fp32 on chip instead of in HBM; the column sums over the key
    channel add the row groups' partial sums in another order) and match the oracle."""
    dec, stack = _decode_tokens_inputs(5, K, 3, d, dtype, seed=K + d)
    S1 = dec["S"].to(DEV)
    outs = [kda.recurrent_step(*(st[n].to(DEV) for n in ("q", "k", "v", "g", "beta")), S1)
            for st in dec["steps"]]
    S2 = dec["S"].to(DEV)
    out = torch.empty(5, K, 3, d, dtype=stack["q"].dtype, device=DEV)
    kda.kda_recurrent_steps(*(stack[n].to(DEV) for n in ("q", "k", "v", "g", "beta")), S2, out)
    kda.kda_sync_status()
    # fp32 state: a reassociated sum of eight partials; outputs may differ by one rounding of
    # the output type (bf16: 2^-8 relative)
    assert torch.allclose(S1, S2, rtol=1e-5, atol=1e-6)
    o_rtol = 1e-5 if dtype == "f32" else 2.0 ** -7
    for t in range(K):
        assert torch.allclose(out[:, t].float(), outs[t].float(), rtol=o_rtol, atol=1e-6)
    Sref = f64(dec["S"])
    for t, st in enumerate(dec["steps"]):
        o_ref, Sref = oracle.decode_step(*(f64(st[n]) for n in ("q", "k", "v", "g", "beta")), Sref)
        check(out[:, t].float().cpu().double().numpy(), o_ref, dtype, f"o[{t}]")
    check(S2.cpu().double().numpy(), Sref, dtype, "S")


def test_decode_tokens_N256_H96_K4_sampled(kda):
    """Four tokens for the full 256 x 96 state in one call; sampled problems against the oracle."""
    N, K, H, d = 256, 4, 96, 128
    dec = kda_synth.make_decode_inputs(N, H, d, d, "bf16", seed=7, S0_std=0.02, steps=K, device=DEV)
    stack = {n: torch.stack([st[n] for st in dec["steps"]], dim=1).contiguous()
             for n in ("q", "k", "v", "g", "beta")}
    picks = [(0, 0), (100, 50), (255, 95)]
    S_host = {p: dec["S"][p[0], p[1]].cpu().double().numpy()[None, None] for p in picks}
    S = dec["S"]
    out = torch.empty(N, K, H, d, dtype=torch.bfloat16, device=DEV)
    kda.kda_recurrent_steps(*(stack[n] for n in ("q", "k", "v", "g", "beta")), S, out)
    kda.kda_sync_status()
    for (n, h) in picks:
        Sref = S_host[(n, h)]
        for t in range(K):
            args = [f64(stack[x][n:n + 1, t, h:h + 1].cpu()) for x in ("q", "k", "v", "g", "beta")]
            o_ref, Sref = oracle.decode_step(*args, Sref)
            check(out[n:n + 1, t, h:h + 1].float().cpu().double().numpy(), o_ref, "bf16",
                  f"o[t={t}, n={n}, h={h}]")
        check(S[n:n + 1, h:h + 1].cpu().double().numpy(), Sref, "bf16", f"S[n={n},h={h}]")
