"""GPU parity of the layers around the recurrence against the fp64 oracle: the output side
(RMSNorm of the raw output times the sigmoid output gate: oracle.recurrent then
oracle.prepost.post_core) and the input side (ShortConv, L2Norm, the bounded decay gate:
oracle.prepost.pre_core then oracle.recurrent), standalone and fused into the prefill kernel.

Inputs are seeded and synthetic: raw projections ~ N(0, 1), decay logits z ~ N(0, 1), conv taps
~ N(0, 0.5^2), A_h ~ N(0, 0.1^2), b ~ U(-2, 2), gate pre-activation u ~ N(0, 1), norm weight
w ~ 1 + 0.1 N(0, 1). Tolerances: fp32 rel-L2 <= 1e-5; bf16 rel-L2 <= 1e-2 with max-abs <= 5e-2.
After RMSNorm each row has unit scale whatever the size of the raw output, so a row whose raw
output is small carries the core's absolute error magnified: end to end the gated outputs are
held to the rel-L2 bound, and the epilogue itself (the GPU's raw output through the oracle's
post_core) to max-abs <= 3e-2 (bf16 rounding of y <= 5 and of the staged raw output, plus the
tanh approximation of the sigmoid)."""
import numpy as np
import pytest
import torch

import kda_synth
import oracle
from oracle import prepost
from tests.test_gpu_parity import DEV, check, f64, kda, oracle_dense, to_dev  # noqa: F401

pytestmark = pytest.mark.gpu
NAMES = ("q", "k", "v", "g", "beta")


def _gate_inputs(shape, dtype, seed):
    gen = torch.Generator().manual_seed(seed)
    u = torch.randn(*shape, generator=gen).to(kda_synth.torch_dtype(dtype))
    w = 1.0 + 0.1 * torch.randn(shape[-1], generator=gen)
    return u, w


def rel_l2(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def check_gated(y, y_ref, dtype, what, y_epi=None):
    """End to end: rel-L2 against the oracle; bf16: the epilogue alone to max-abs <= 3e-2."""
    y = np.asarray(y, dtype=np.float64)
    e = rel_l2(y, y_ref)
    assert e <= (1e-5 if dtype == "f32" else 1e-2), f"{what}: rel-L2 {e:.3e}"
    if y_epi is not None:
        m = float(np.abs(y - y_epi).max())
        assert m <= 3e-2, f"{what}: epilogue max-abs {m:.3e}"


@pytest.mark.parametrize("dtype,d,C", [("bf16", 128, 64), ("bf16", 128, 128), ("f32", 128, 64),
                                       ("bf16", 64, 64), ("f32", 64, 32)])
def test_gated_prefill_dense(kda, dtype, d, C):
    B, T, H = 2, 200, 3  # several blocks and a ragged tail
    inp = kda_synth.make_prefill_inputs(B, T, H, d, d, dtype, seed=d + C, S0_std=0.05)
    u, w = _gate_inputs((B, T, H, d), dtype, seed=C)
    x = to_dev(inp)
    out = torch.empty(B, T, H, d, dtype=x[0].dtype, device=DEV)
    Sf = torch.empty(B, H, d, d, device=DEV)
    kda.kda_chunk_fwd_gated(*x, inp["S0"].to(DEV), u.to(DEV), w.to(DEV), out, Sf, C=C)
    raw, _ = kda.chunk_fwd(*x, inp["S0"].to(DEV), C=C, want_state=False)
    kda.kda_sync_status()
    o_ref, S_ref = oracle_dense(inp)
    y_ref = prepost.post_core(o_ref, f64(u), f64(w), eps=1e-5)
    y_epi = prepost.post_core(raw.float().cpu().double().numpy(), f64(u), f64(w), eps=1e-5)
    check_gated(out.float().cpu().double().numpy(), y_ref, dtype, "y", y_epi if dtype == "bf16" else None)
    check(Sf.cpu().double().numpy(), S_ref, dtype, "S_final")
    if dtype == "bf16" and d == 128:  # the epilogue and the standalone kernel: the same function
        y2 = torch.empty_like(raw)
        kda.kda_output_gate(raw, u.to(DEV), w.to(DEV), y2)
        kda.kda_sync_status()
        assert torch.equal(out, y2)


@pytest.mark.parametrize("C", [64, 128])
def test_gated_prefill_packed(kda, C):
    cu = torch.tensor([0, 1, 65, 66, 300, 429], dtype=torch.int32)
    T, N, H, d = int(cu[-1]), cu.numel() - 1, 2, 128
    inp = kda_synth.make_prefill_inputs(1, T, H, d, d, "bf16", seed=C + 1, S0_std=0.05, n_state=N)
    u, w = _gate_inputs((1, T, H, d), "bf16", seed=C + 2)
    x = to_dev(inp)
    out = torch.empty(1, T, H, d, dtype=torch.bfloat16, device=DEV)
    Sf = torch.empty(N, H, d, d, device=DEV)
    kda.kda_chunk_fwd_gated(*x, inp["S0"].to(DEV), u.to(DEV), w.to(DEV), out, Sf,
                            cu_seqlens=cu.to(DEV), C=C)
    raw, _ = kda.chunk_fwd_varlen(*x, cu.to(DEV), S0=inp["S0"].to(DEV), C=C, want_state=False)
    kda.kda_sync_status()
    o_ref, S_ref = oracle.recurrent_varlen(*(f64(inp[n]) for n in NAMES), cu.numpy(),
                                           f64(inp["S0"]))
    y_epi = prepost.post_core(raw.float().cpu().double().numpy(), f64(u), f64(w))
    check_gated(out.float().cpu().double().numpy(), prepost.post_core(o_ref, f64(u), f64(w)),
                "bf16", "y", y_epi)
    check(Sf.cpu().double().numpy(), S_ref, "bf16", "S_final")


def test_gated_prefill_B4_H96_T8192_sampled(kda):
    """The K3 layer shape at full size with the output side fused; sampled (batch, head)."""
    w_ = kda_synth.WORKLOADS[2]
    B, T, H, d = w_["B"], w_["T"], w_["H"], 128
    inp = kda_synth.make_prefill_inputs(B, T, H, d, d, "bf16", w_["seed"], g_bias=True)
    u, w = _gate_inputs((B, T, H, d), "bf16", seed=99)
    out = torch.empty(B, T, H, d, dtype=torch.bfloat16, device=DEV)
    x = to_dev(inp)
    kda.kda_chunk_fwd_gated(*x, None, u.to(DEV), w.to(DEV), out, None, C=64)
    raw, _ = kda.chunk_fwd(*x, None, C=64, want_state=False)
    kda.kda_sync_status()
    for b, h in ((0, 3), (3, 94)):
        sub = {n: inp[n][b:b + 1, :, h:h + 1] for n in NAMES}
        o_ref, _ = oracle.recurrent(*(f64(sub[n]) for n in NAMES))
        ub = f64(u[b:b + 1, :, h:h + 1])
        y_epi = prepost.post_core(raw[b:b + 1, :, h:h + 1].float().cpu().double().numpy(), ub, f64(w))
        check_gated(out[b:b + 1, :, h:h + 1].float().cpu().double().numpy(),
                    prepost.post_core(o_ref, ub, f64(w)), "bf16", f"y[b={b},h={h}]", y_epi)


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 128), ("bf16", 64)])
def test_output_gate_on_decode_outputs(kda, dtype, d):
    dec = kda_synth.make_decode_inputs(7, 5, d, d, dtype, seed=d, S0_std=0.3, steps=1)
    st = dec["steps"][0]
    S = dec["S"].to(DEV)
    o = kda.recurrent_step(*(st[n].to(DEV) for n in NAMES), S)
    u, w = _gate_inputs((7, 5, d), dtype, seed=3)
    y = torch.empty_like(o)
    kda.kda_output_gate(o, u.to(DEV), w.to(DEV), y)
    kda.kda_output_gate(o, u.to(DEV), w.to(DEV), o)  # in place
    kda.kda_sync_status()
    o_ref, _ = oracle.decode_step(*(f64(st[n]) for n in NAMES), f64(dec["S"]))
    y_ref = prepost.post_core(o_ref, f64(u), f64(w))
    raw = kda.recurrent_step(*(st[n].to(DEV) for n in NAMES), dec["S"].to(DEV))
    y_epi = prepost.post_core(raw.float().cpu().double().numpy(), f64(u), f64(w))
    check_gated(y.float().cpu().double().numpy(), y_ref, dtype, "y",
                y_epi if dtype == "bf16" else None)
    assert torch.equal(y, o)


# ------------------------------------------------------------------ the input side


def _raw_inputs(B, T, H, d, dtype, seed, n_state=None):
    gen = torch.Generator().manual_seed(seed)
    dt = kda_synth.torch_dtype(dtype)
    raw = {n: torch.randn(B, T, H, d, generator=gen).to(dt) for n in ("q_raw", "k_raw", "v_raw", "z")}
    raw["beta"] = torch.sigmoid(torch.randn(B, T, H, generator=gen)).to(dt)
    prm = {n: 0.5 * torch.randn(H, d, 4, generator=gen) for n in ("conv_q", "conv_k", "conv_v")}
    prm["A_log"] = 0.1 * torch.randn(H, generator=gen)
    prm["b_decay"] = torch.rand(H, d, generator=gen) * 4.0 - 2.0
    ns = B if n_state is None else n_state
    raw["S0"] = 0.05 * torch.randn(ns, H, d, d, generator=gen)
    return raw, prm


PRM = ("conv_q", "conv_k", "conv_v", "A_log", "b_decay")


def _dev_prm(prm):
    """The parameters as the library takes them: conv weights tap-major [H, 4, d] (the oracle
    keeps them [H, d, 4])."""
    return [(prm[n].permute(0, 2, 1).contiguous() if n.startswith("conv") else prm[n]).to(DEV)
            for n in PRM]


def _oracle_pre(raw, prm, cu=None):
    return prepost.pre_core(*(f64(raw[n]) for n in ("q_raw", "k_raw", "v_raw", "z")),
                            *(f64(prm[n]) for n in PRM), cu_seqlens=cu)


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 128), ("bf16", 64), ("f32", 64)])
@pytest.mark.parametrize("packed", [False, True])
def test_pre_core_standalone(kda, dtype, d, packed):
    cu = torch.tensor([0, 1, 5, 70, 133], dtype=torch.int32) if packed else None
    B, T, H = (1, 133, 3) if packed else (2, 70, 3)
    raw, prm = _raw_inputs(B, T, H, d, dtype, seed=d + packed)
    outs = {n: torch.empty(B, T, H, d, dtype=kda_synth.torch_dtype(dtype), device=DEV)
            for n in ("q", "k", "v", "g")}
    kda.kda_pre_core(*(raw[n].to(DEV) for n in ("q_raw", "k_raw", "v_raw", "z")),
                     *_dev_prm(prm), outs["q"], outs["k"], outs["v"], outs["g"],
                     cu_seqlens=None if cu is None else cu.to(DEV))
    kda.kda_sync_status()
    refs = _oracle_pre(raw, prm, None if cu is None else cu.numpy())
    for name, ref in zip(("q", "k", "v", "g"), refs):
        check(outs[name].float().cpu().double().numpy(), ref, dtype, name)


@pytest.mark.parametrize("C", [64, 128])
@pytest.mark.parametrize("gated", [False, True])
def test_fused_layer_dense(kda, C, gated):
    """Raw projections in, the layer's output out, in one kernel: the input side computed as
    each block lands (taps across block boundaries through the stash), the recurrence, and the
    output side. Against the oracle's pre_core, recurrence and post_core in fp64."""
    B, T, H, d = 2, 300, 3, 128
    raw, prm = _raw_inputs(B, T, H, d, "bf16", seed=C + gated)
    u, w = _gate_inputs((B, T, H, d), "bf16", seed=5)
    out = torch.empty(B, T, H, d, dtype=torch.bfloat16, device=DEV)
    Sf = torch.empty(B, H, d, d, device=DEV)
    kda.kda_chunk_fwd_fused(*(raw[n].to(DEV) for n in ("q_raw", "k_raw", "v_raw", "z", "beta")),
                            *_dev_prm(prm), raw["S0"].to(DEV), out, Sf,
                            gate_u=u.to(DEV) if gated else None,
                            norm_w=w.to(DEV) if gated else None, C=C)
    kda.kda_sync_status()
    q, k, v, g = _oracle_pre(raw, prm)
    o_ref, S_ref = oracle.recurrent(q, k, v, g, f64(raw["beta"]), f64(raw["S0"]))
    check(Sf.cpu().double().numpy(), S_ref, "bf16", "S_final")
    if gated:
        check_gated(out.float().cpu().double().numpy(), prepost.post_core(o_ref, f64(u), f64(w)),
                    "bf16", "y")
    else:
        check(out.float().cpu().double().numpy(), o_ref, "bf16", "out")


def test_fused_layer_packed(kda):
    cu = torch.tensor([0, 2, 66, 67, 300, 429], dtype=torch.int32)
    T, N, H, d = int(cu[-1]), cu.numel() - 1, 2, 128
    raw, prm = _raw_inputs(1, T, H, d, "bf16", seed=11, n_state=N)
    out = torch.empty(1, T, H, d, dtype=torch.bfloat16, device=DEV)
    Sf = torch.empty(N, H, d, d, device=DEV)
    kda.kda_chunk_fwd_fused(*(raw[n].to(DEV) for n in ("q_raw", "k_raw", "v_raw", "z", "beta")),
                            *_dev_prm(prm), raw["S0"].to(DEV), out, Sf,
                            cu_seqlens=cu.to(DEV), C=64)
    kda.kda_sync_status()
    q, k, v, g = _oracle_pre(raw, prm, cu.numpy())
    o_ref, S_ref = oracle.recurrent_varlen(q, k, v, g, f64(raw["beta"]), cu.numpy(), f64(raw["S0"]))
    check(out.float().cpu().double().numpy(), o_ref, "bf16", "out")
    check(Sf.cpu().double().numpy(), S_ref, "bf16", "S_final")


def test_fused_layer_equals_standalone_pre_core_then_core(kda):
    """The fused input side and the standalone kernel followed by the plain prefill agree."""
    B, T, H, d = 1, 500, 4, 128
    raw, prm = _raw_inputs(B, T, H, d, "bf16", seed=21)
    x = {n: raw[n].to(DEV) for n in ("q_raw", "k_raw", "v_raw", "z", "beta")}
    p = dict(zip(PRM, _dev_prm(prm)))
    out = torch.empty(B, T, H, d, dtype=torch.bfloat16, device=DEV)
    kda.kda_chunk_fwd_fused(*x.values(), *p.values(), None, out, None, C=64)
    qkvg = [torch.empty_like(x["q_raw"]) for _ in range(4)]
    kda.kda_pre_core(x["q_raw"], x["k_raw"], x["v_raw"], x["z"], *p.values(), *qkvg)
    ref, _ = kda.chunk_fwd(*qkvg, x["beta"], None, C=64, want_state=False)
    kda.kda_sync_status()
    check(out.float().cpu().double().numpy(), ref.float().cpu().double().numpy(), "bf16", "out")
