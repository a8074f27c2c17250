"""Runs one workload through the library a few times (for profilers such as ncu).

    python -m gated_delta_rule_167_b300.run_case prefill --B 1 --H 96 --T 8192 --C 64 --iters 2
    python -m gated_delta_rule_167_b300.run_case varlen --H 96 --T 16384 --nseq 4 --C 64
    python -m gated_delta_rule_167_b300.run_case decode --N 256 --H 96 --iters 3
    python -m gated_delta_rule_167_b300.run_case segmented --B 1 --H 8 --T 4096 --iters 3
    python -m gated_delta_rule_167_b300.run_case fused --B 1 --H 148 --T 2048 --iters 3
    python -m gated_delta_rule_167_b300.run_case decode_tokens --N 256 --H 96 --K 4 --iters 3

Inputs are drawn on the device with the seeded generators of `kda_synth`; nothing is checked
against a reference here (the test-suite does that). Exits non-zero if the library reports an
error.
"""
from __future__ import annotations

import argparse
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import gated_delta_rule_167_b300 as kda  # noqa: E402
import kda_synth  # noqa: E402


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("kind", choices=["prefill", "gated", "varlen", "decode", "segmented", "fused",
                                     "decode_tokens"])
    ap.add_argument("--K", type=int, default=4)
    ap.add_argument("--n_seg", type=int, default=0)
    ap.add_argument("--B", type=int, default=1)
    ap.add_argument("--N", type=int, default=256)
    ap.add_argument("--H", type=int, default=96)
    ap.add_argument("--T", type=int, default=8192)
    ap.add_argument("--d", type=int, default=128)
    ap.add_argument("--C", type=int, default=64)
    ap.add_argument("--nseq", type=int, default=8)
    ap.add_argument("--dtype", default="bf16", choices=["bf16", "f32"])
    ap.add_argument("--iters", type=int, default=2)
    a = ap.parse_args(argv)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    kda.load_library()
    if a.kind == "prefill":
        inp = kda_synth.make_prefill_inputs(a.B, a.T, a.H, a.d, a.d, a.dtype, seed=0,
                                            g_bias=True, device=dev)
        x = [inp[n] for n in ("q", "k", "v", "g", "beta")]
        out = torch.empty(a.B, a.T, a.H, a.d, dtype=x[0].dtype, device=dev)
        Sf = torch.empty(a.B, a.H, a.d, a.d, dtype=torch.float32, device=dev)
        for _ in range(a.iters):
            kda.kda_chunk_fwd(*x, None, out, Sf, C=a.C)
    elif a.kind == "gated":  # the prefill with the output side in its epilogue
        inp = kda_synth.make_prefill_inputs(a.B, a.T, a.H, a.d, a.d, a.dtype, seed=0,
                                            g_bias=True, device=dev)
        x = [inp[n] for n in ("q", "k", "v", "g", "beta")]
        gen = torch.Generator(device=dev).manual_seed(1)
        u = torch.randn(a.B, a.T, a.H, a.d, generator=gen, device=dev).to(x[0].dtype)
        w = 1.0 + 0.1 * torch.randn(a.d, generator=gen, device=dev)
        out = torch.empty(a.B, a.T, a.H, a.d, dtype=x[0].dtype, device=dev)
        Sf = torch.empty(a.B, a.H, a.d, a.d, dtype=torch.float32, device=dev)
        for _ in range(a.iters):
            kda.kda_chunk_fwd_gated(*x, None, u, w, out, Sf, C=a.C)
    elif a.kind == "varlen":
        inp = kda_synth.make_varlen_inputs(a.T, a.H, a.d, a.d, a.nseq, a.dtype, seed=0, device=dev)
        x = [inp[n] for n in ("q", "k", "v", "g", "beta")]
        cu = inp["cu_seqlens"].to(dev)
        out = torch.empty(1, a.T, a.H, a.d, dtype=x[0].dtype, device=dev)
        Sf = torch.empty(a.nseq, a.H, a.d, a.d, dtype=torch.float32, device=dev)
        for _ in range(a.iters):
            kda.kda_chunk_fwd_varlen(*x, None, out, Sf, cu, C=a.C)
    elif a.kind == "segmented":
        inp = kda_synth.make_prefill_inputs(a.B, a.T, a.H, a.d, a.d, a.dtype, seed=0,
                                            S0_std=0.02, device=dev)
        x = [inp[n] for n in ("q", "k", "v", "g", "beta")]
        n_seg = a.n_seg or kda.segments_auto(a.B, a.H, a.T)
        ws = torch.empty(max(1, kda.segmented_workspace_bytes(a.B, a.H, a.T, a.d, a.d, n_seg)),
                         dtype=torch.uint8, device=dev)
        out = torch.empty(a.B, a.T, a.H, a.d, dtype=x[0].dtype, device=dev)
        Sf = torch.empty(a.B, a.H, a.d, a.d, dtype=torch.float32, device=dev)
        for _ in range(a.iters):
            kda.kda_chunk_fwd_segmented(*x, inp["S0"], out, Sf, n_seg, ws, C=a.C)
    elif a.kind == "fused":
        gen = torch.Generator(device=dev).manual_seed(0)
        raw = [torch.randn(a.B, a.T, a.H, a.d, generator=gen, device=dev).to(torch.bfloat16)
               for _ in range(4)]
        beta = torch.sigmoid(torch.randn(a.B, a.T, a.H, generator=gen, device=dev)).to(torch.bfloat16)
        prm = [0.5 * torch.randn(a.H, 4, a.d, generator=gen, device=dev) for _ in range(3)]
        prm += [torch.zeros(a.H, device=dev), torch.zeros(a.H, a.d, device=dev)]
        out = torch.empty(a.B, a.T, a.H, a.d, dtype=torch.bfloat16, device=dev)
        for _ in range(a.iters):
            kda.kda_chunk_fwd_fused(*raw, beta, *prm, None, out, None, C=a.C)
    elif a.kind == "decode_tokens":
        dec = kda_synth.make_decode_inputs(a.N, a.H, a.d, a.d, a.dtype, seed=0, steps=a.K,
                                           device=dev)
        stack = [torch.stack([st[n] for st in dec["steps"]], dim=1).contiguous()
                 for n in ("q", "k", "v", "g", "beta")]
        out = torch.empty(a.N, a.K, a.H, a.d, dtype=stack[0].dtype, device=dev)
        for _ in range(a.iters):
            kda.kda_recurrent_steps(*stack, dec["S"], out)
    else:
        dec = kda_synth.make_decode_inputs(a.N, a.H, a.d, a.d, a.dtype, seed=0, steps=a.iters,
                                           device=dev)
        S = dec["S"]
        out = torch.empty(a.N, a.H, a.d, dtype=dec["steps"][0]["q"].dtype, device=dev)
        for st in dec["steps"]:
            kda.kda_recurrent_step(*(st[n] for n in ("q", "k", "v", "g", "beta")), S, out)
    kda.kda_sync_status()
    print(f"{a.kind} ok")
    return 0


if __name__ == "__main__":
    sys.exit(main())
