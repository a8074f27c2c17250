"""Seeded synthetic inputs for KDA, shared by the tests, the oracle side and the benchmark.

This module only draws random numbers in the shapes and distributions of the workloads; it
holds none of the KDA arithmetic. Everything is drawn with a CPU ``torch.Generator`` in fp32
and then cast, so a given (shape, seed) gives the same bits on every machine; the oracle reads
exactly the cast values.

Recipe (shapes of Kimi K3's KDA layers: 96 heads, d_k = d_v = 128; Kimi K3 wiki,
"Tableau des spécifications", table "Attention"):
  q, k  ~ N(0, 1) per element, then divided by their L2 norm per token and head
  v     ~ N(0, 1)
  g     = g_min * sigmoid(z), z ~ N(0, 1) per channel, g_min = -5; optionally z + b_h with a
          per-head, per-channel bias b_h ~ U(-2, 2) drawn once
  beta  = sigmoid(N(0, 1)) per token and head
  S0    = zeros, or N(0, s^2) fp32 when a standard deviation s is given
Packed batches cut T_total at n-1 distinct points drawn uniformly from [1, T_total - 1].
"""
from __future__ import annotations

import torch

G_MIN = -5.0

# Named workloads: (description, keyword arguments). The "cfg" index is the position in the
# list of workloads that the tests and the benchmark share.
WORKLOADS = [
    dict(name="kda_fp32_B1_H1_T256_d128_C64", kind="prefill", B=1, H=1, T=256, dk=128, dv=128,
         C=64, dtype="f32", seed=0, S0_std=0.0, g_bias=False),
    dict(name="kda_bf16_B1_H8_T4096_d128_C64", kind="prefill", B=1, H=8, T=4096, dk=128, dv=128,
         C=64, dtype="bf16", seed=0, S0_std=0.02, g_bias=False),
    dict(name="kda_bf16_B4_H96_T8192_d128_C64", kind="prefill", B=4, H=96, T=8192, dk=128,
         dv=128, C=64, dtype="bf16", seed=0, S0_std=0.0, g_bias=True),
    dict(name="kda_bf16_varlen8_H96_T131072_d128_C128", kind="varlen", B=1, H=96, T=131072,
         dk=128, dv=128, C=128, dtype="bf16", seed=0, S0_std=0.0, g_bias=False, n_seq=8),
    dict(name="kda_decode_bf16_N256_H96_d128_x64", kind="decode", N=256, H=96, dk=128, dv=128,
         dtype="bf16", seed=0, S0_std=0.02, steps=64),
]


def torch_dtype(name: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def _unit(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True)


def make_prefill_inputs(B, T, H, dk, dv, dtype="bf16", seed=0, S0_std=0.0, g_bias=False,
                        n_state=None, device="cpu"):
    """q, k, g [B, T, H, dk]; v [B, T, H, dv]; beta [B, T, H]; S0 [n_state or B, H, dk, dv]
    fp32 or None. With the default ``device="cpu"`` the bits are the same on every machine;
    a CUDA device draws the same distributions from torch's device generator (faster for the
    largest workloads, bit-identical only on the same torch build)."""
    gen = torch.Generator(device=device).manual_seed(int(seed))
    dt = torch_dtype(dtype)
    bias = None
    if g_bias:
        bias = torch.rand(H, dk, generator=gen, device=device) * 4.0 - 2.0
    out = {k_: [] for k_ in ("q", "k", "v", "g", "beta")}
    for _ in range(B):  # one batch row at a time bounds the fp32 scratch
        q = _unit(torch.randn(1, T, H, dk, generator=gen, device=device))
        k = _unit(torch.randn(1, T, H, dk, generator=gen, device=device))
        v = torch.randn(1, T, H, dv, generator=gen, device=device)
        z = torch.randn(1, T, H, dk, generator=gen, device=device)
        if bias is not None:
            z += bias
        g = G_MIN * torch.sigmoid(z)
        beta = torch.sigmoid(torch.randn(1, T, H, generator=gen, device=device))
        for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta)):
            out[name].append(t.to(dt))
    res = {name: torch.cat(ts, 0) if B > 0 else torch.empty(0) for name, ts in out.items()}
    ns = B if n_state is None else n_state
    res["S0"] = ((torch.randn(ns, H, dk, dv, generator=gen, device=device) * S0_std)
                 if S0_std > 0 else None)
    return res


def varlen_cu_seqlens(T_total: int, n_seq: int, seed: int = 0) -> torch.Tensor:
    """Uniform random composition of T_total into n_seq positive lengths (int32 [n_seq+1])."""
    gen = torch.Generator().manual_seed(int(seed) + 7919)
    if n_seq == 1:
        cuts = torch.empty(0, dtype=torch.int64)
    else:
        cuts = torch.randperm(T_total - 1, generator=gen)[: n_seq - 1] + 1
        cuts, _ = torch.sort(cuts)
    cu = torch.cat([torch.zeros(1, dtype=torch.int64), cuts,
                    torch.full((1,), T_total, dtype=torch.int64)])
    return cu.to(torch.int32)


def make_varlen_inputs(T, H, dk, dv, n_seq, dtype="bf16", seed=0, S0_std=0.0, device="cpu"):
    inp = make_prefill_inputs(1, T, H, dk, dv, dtype=dtype, seed=seed, S0_std=S0_std,
                              n_state=n_seq, device=device)
    inp["cu_seqlens"] = varlen_cu_seqlens(T, n_seq, seed)
    return inp


def make_decode_inputs(N, H, dk, dv, dtype="bf16", seed=0, S0_std=0.02, steps=1, device="cpu"):
    """Per step: q, k, g [N, H, dk]; v [N, H, dv]; beta [N, H]. Plus S [N, H, dk, dv] fp32."""
    gen = torch.Generator(device=device).manual_seed(int(seed))
    dt = torch_dtype(dtype)
    kw = dict(generator=gen, device=device)
    S = torch.randn(N, H, dk, dv, **kw) * S0_std
    seq = []
    for _ in range(steps):
        q = _unit(torch.randn(N, H, dk, **kw)).to(dt)
        k = _unit(torch.randn(N, H, dk, **kw)).to(dt)
        v = torch.randn(N, H, dv, **kw).to(dt)
        g = (G_MIN * torch.sigmoid(torch.randn(N, H, dk, **kw))).to(dt)
        beta = torch.sigmoid(torch.randn(N, H, **kw)).to(dt)
        seq.append(dict(q=q, k=k, v=v, g=g, beta=beta))
    return dict(S=S, steps=seq)


def to_f64_numpy(t):
    """Exact upcast of a (bf16/fp32) CPU tensor to an fp64 NumPy array."""
    return None if t is None else t.to(torch.float64).numpy()
