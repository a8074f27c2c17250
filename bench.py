#!/usr/bin/env python3
"""Benchmark of the KDA forward library on B300.

Headline: chunkwise prefill at the K3 layer shape (B=4, H=96, T=8192, d_k=d_v=128, C=64, bf16
inputs, fp32 state) -- tokens/s of one `kda_chunk_fwd` pass over the batch, inputs resident in
HBM. Secondary lines in the same JSON object: the one-token decode step (256 sequences x 96
heads, state resident and updated in place, 64 consecutive steps) as % of HBM bandwidth, and the
packed long-context prefill (8 sequences, T_total = 131072, C = 128).

`python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]`. Under torchrun each
rank runs its own batch (weak scaling, no data-path collective); rank 0 prints one JSON line.
`--impl reference` times the fp64 CPU oracle instead (the only other arm available).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import kda_synth  # noqa: E402

# Algorithmic bytes per token-head (bf16 q, k, g, v, beta in; o out) and useful FLOPs.
D = 128
BYTES_PER_TOKEN_HEAD = 3 * D * 2 + D * 2 + 2 + D * 2  # 1282
STATE_BYTES = D * D * 4


def useful_flops_per_token_head(C, dk=D, dv=D):
    return C * (3 * dk + 2 * dv) + 6 * dk * dv


def decode_bytes_per_head(dk=D, dv=D):
    return 2 * dk * dv * 4 + (3 * dk + dv) * 2 + 2 + dv * 2  # 132354


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sustained=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                    source="measured")
    except Exception:
        return dict(hbm=6400.0, bf16=1800.0, bf16_sustained=1400.0, source="fallback")


# The sources each timed kernel is compiled from (its DRAM counters stay valid while their code
# is unchanged).
PREFILL_SOURCES = ("kda_chunk_tc.cuh", "kda_chunk_simt.cuh", "kda_sm100.cuh", "kda_common.cuh",
                   "kda_pre.cuh", "kda_post.cuh")
DECODE_SOURCES = ("kda_decode.cuh", "kda_common.cuh", "kda_sm100.cuh")


def _code_lines(text):
    """The lines of a source file with `//` comments, trailing blanks and empty lines removed: an
    edit to the comments leaves the hash, like the compiled kernel, unchanged. A line holding a
    string literal is kept whole."""
    out = []
    for line in text.splitlines():
        if '"' not in line and "//" in line:
            line = line[:line.index("//")]
        line = line.rstrip()
        if line:
            out.append(line)
    return "\n".join(out)


def _kernel_source_hash(sources=PREFILL_SOURCES):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "gated_delta_rule_167_b300", "csrc")
    for name in sources:
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode() + b"\0" + _code_lines(f.read()).encode())
    return h.hexdigest()[:16]


def _recorded_traffic(kernel_key):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on this source."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)
        ent = rec.get(kernel_key)
        sources = DECODE_SOURCES if kernel_key.startswith("decode") else PREFILL_SOURCES
        if ent and ent.get("source_hash") == _kernel_source_hash(sources):
            return float(ent["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """Samples the SM clock and the clock-event (throttle) reasons while the timed region runs:
    through NVML when it initialises, else through `nvidia-smi -lms`."""

    REASONS = {
        0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
        0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
        0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting",
    }

    def __init__(self, device, period=0.02):
        self.index = _physical_gpu_id(device)
        self.period = period
        self.samples, self.reasons = [], set()
        self._stop = threading.Event()
        self._thread = None
        self._proc = None
        self.max_mhz = None
        self.source = None
        self.nv = None
        try:
            import pynvml

            pynvml.nvmlInit()
            if str(self.index).startswith("GPU-"):
                self.h = pynvml.nvmlDeviceGetHandleByUUID(self.index)
            else:
                self.h = pynvml.nvmlDeviceGetHandleByIndex(int(self.index))
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self.h, pynvml.NVML_CLOCK_SM)
            self.nv = pynvml
            self.source = "nvml"
        except Exception as e:  # fall back to nvidia-smi
            self.source = f"nvidia-smi (nvml unavailable: {type(e).__name__})"

    def _run_nvml(self):
        nv = self.nv
        while not self._stop.is_set():
            try:
                self.samples.append(nv.nvmlDeviceGetClockInfo(self.h, nv.NVML_CLOCK_SM))
                mask = nv.nvmlDeviceGetCurrentClocksEventReasons(self.h)
                for bit, name in self.REASONS.items():
                    if mask & bit:
                        self.reasons.add(name)
            except Exception:
                pass
            time.sleep(self.period)

    def __enter__(self):
        if self.nv is not None:
            self._thread = threading.Thread(target=self._run_nvml, daemon=True)
            self._thread.start()
        else:
            import subprocess

            try:
                self._proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(self.index), "--query-gpu=clocks.sm,clocks.max.sm,"
                     "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                     "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap",
                     "--format=csv,noheader,nounits", "-lms", "100"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
                time.sleep(0.3)  # let the first sample land before the timed region
            except Exception:
                self._proc = None
        return self

    def __exit__(self, *a):
        self._stop.set()
        if self._thread:
            self._thread.join()
        if self._proc is not None:
            time.sleep(0.25)
            self._proc.terminate()
            try:
                out, _ = self._proc.communicate(timeout=5)
            except Exception:
                out = ""
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for line in out.splitlines():
                f = [x.strip() for x in line.split(",")]
                if len(f) < 6:
                    continue
                try:
                    self.samples.append(float(f[0]))
                    self.max_mhz = float(f[1])
                except ValueError:
                    continue
                for name, val in zip(names, f[2:6]):
                    if val.lower() == "active":
                        self.reasons.add(name)

    def summary(self):
        med = statistics.median(self.samples) if self.samples else None
        return {"sm_mhz": med, "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
                "samples": len(self.samples), "source": self.source}


def _physical_gpu_id(device):
    """Identifier of the torch device for NVML / nvidia-smi: its UUID when torch exposes it,
    else the first CUDA_VISIBLE_DEVICES entry, else the index."""
    try:
        u = str(torch.cuda.get_device_properties(device).uuid)
        if u and u != "None":
            return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        pass
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    if vis:
        first = vis.split(",")[device.index or 0].strip()
        if first:
            return first
    return str(device.index or 0)


def _dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() and args.impl != "reference" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def _barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def _max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _hold_stream(stream, ms=50.0):
    """Queues a spin kernel of about `ms` on `stream` (outside any timed span), so that the
    launches that follow are all submitted while the GPU is still busy with it: the events then
    time the device work back to back, without gaps from the host's launch latency or from the
    clock sampler starting up."""
    if not hasattr(torch.cuda, "_sleep"):
        return
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(ms * 1e-3 * 2.0e9))


def _timed(fn, steps, warmup, world, device, stream, hold=True):
    """W untimed warm-up calls, then K timed calls bracketed by barrier + synchronize; the
    duration comes from CUDA events on the launching stream. `hold`: the timed calls are queued
    behind a spin kernel (see _hold_stream); not for calls that synchronize with the host.
    Returns (total_ms, clocks)."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize(device)
    _barrier(world)
    torch.cuda.synchronize(device)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(device) as cs:
        if hold:
            _hold_stream(stream)
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(device)
    _barrier(world)
    torch.cuda.synchronize(device)
    ms = e0.elapsed_time(e1)
    return _max_over_ranks(ms, world, device), cs.summary()


# ------------------------------------------------------------------------ CPU oracle arm


def _cpu_sample(T, n_heads, seed=0):
    inp = kda_synth.make_prefill_inputs(1, T, n_heads, D, D, "bf16", seed=seed, g_bias=True)
    return [kda_synth.to_f64_numpy(inp[n]) for n in ("q", "k", "v", "g", "beta")]


def cpu_baseline(T=8192, H=96, budget_s=15.0):
    """The oracle as it stands, on the host's cores, over a bounded sample of the headline
    workload: a number of complete (batch, head) sequences of T tokens."""
    import oracle

    cores = oracle.default_threads()
    n = max(1, min(cores, 8))
    x = _cpu_sample(T, n)
    t0 = time.perf_counter()
    oracle.recurrent(*x, nthreads=cores)
    dt = time.perf_counter() - t0
    reps = max(1, min(64, int(budget_s / max(dt, 1e-3))))
    n2 = n * reps
    if n2 > n:
        x = _cpu_sample(T, n2)
        t0 = time.perf_counter()
        oracle.recurrent(*x, nthreads=cores)
        dt = time.perf_counter() - t0
    else:
        n2 = n
    tokens = n2 * T / H  # token-heads -> tokens of the H-head layer
    return {"value": tokens / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{n2} complete (batch, head) sequences of T={T} tokens "
                      f"(fp64 token-by-token recurrence) in {dt:.2f} s; tokens = "
                      f"token-heads / H={H}"}


def run_reference(args):
    world, rank, _ = _dist_setup(args)
    if rank != 0:
        return 0
    import oracle

    T, H = 8192, 96
    cores = oracle.default_threads()
    n = max(1, min(cores, 16))
    x = _cpu_sample(T, n)
    for _ in range(args.warmup):
        oracle.recurrent(*x, nthreads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.recurrent(*x, nthreads=cores)
    dt = time.perf_counter() - t0
    tokens = args.steps * n * T / H
    value = tokens / dt
    line = {
        "impl": "reference", "metric": "KDA fwd tokens/s (B=4,H=96,T=8192,d=128,C=64)",
        "value": value, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "kda_bf16_B4_H96_T8192_d128_C64", "B": 4, "H": 96, "T": 8192,
                   "d_k": 128, "d_v": 128, "C": 64, "parallelism": "none"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step: {n} complete (batch, head) sequences of "
                                   f"T={T} tokens; tokens = token-heads / H={H}"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ------------------------------------------------------------------------ GPU arm


def bench_prefill(kda, args, world, rank, device, stream, peaks):
    w = kda_synth.WORKLOADS[2]
    B, T, H, C = w["B"], w["T"], w["H"], w["C"]
    inp = kda_synth.make_prefill_inputs(B, T, H, D, D, "bf16", seed=w["seed"] + rank,
                                        g_bias=True, device=device)
    q, k, v, g, b = (inp[n] for n in ("q", "k", "v", "g", "beta"))
    out = torch.empty(B, T, H, D, dtype=torch.bfloat16, device=device)
    Sf = torch.empty(B, H, D, D, dtype=torch.float32, device=device)

    def step():
        kda.kda_chunk_fwd(q, k, v, g, b, None, out, Sf, C=C, stream=stream)

    step()
    kda.kda_sync_status(stream)
    total_ms, clocks = _timed(step, args.steps, args.warmup, world, device, stream)
    kda.kda_sync_status(stream)
    ms = total_ms / args.steps
    token_heads = B * T * H
    alg_bytes = token_heads * BYTES_PER_TOKEN_HEAD + B * H * STATE_BYTES  # S0 = 0 is not read
    flops = token_heads * useful_flops_per_token_head(C)
    achieved_gbs = alg_bytes / (ms * 1e-3) / 1e9
    traffic = _recorded_traffic("prefill_bf16_B4_H96_T8192_C64")
    res = dict(ms=ms, clocks=clocks, tokens_per_s=world * B * T / (ms * 1e-3),
               roofline={"bound": "hbm", "achieved": achieved_gbs, "peak": peaks["hbm"],
                         "unit": "GB/s", "frac": achieved_gbs / peaks["hbm"],
                         "traffic": traffic, "peak_source": peaks["source"],
                         "algorithmic_bytes_per_launch": alg_bytes},
               tflops=flops / (ms * 1e-3) / 1e12)
    res["tensor_frac_of_bf16_peak"] = res["tflops"] / peaks["bf16"]

    # end to end through the public API with host buffers (copies inside the timed region)
    hin = {n: inp[n].cpu().pin_memory() for n in ("q", "k", "v", "g", "beta")}
    out_h = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    st_h = torch.empty(Sf.shape, dtype=Sf.dtype, pin_memory=True)

    pipe = kda.HostPipeline(device)

    def e2e_step():
        kda.chunk_fwd_host(hin["q"], hin["k"], hin["v"], hin["g"], hin["beta"], None, C=C,
                           device=device, stream=stream, out_host=out_h, state_host=st_h,
                           pipeline=pipe)

    e2e_steps = max(1, min(args.steps, 3))
    e2e_ms, _ = _timed(e2e_step, e2e_steps, 1, world, device, stream, hold=False)
    res["e2e"] = {"value": world * B * T / (e2e_ms / e2e_steps * 1e-3), "unit": "tokens/s",
                  "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in hin.values()),
                  "d2h_bytes_per_step": out_h.numel() * 2 + st_h.numel() * 4,
                  "steps": e2e_steps}
    del inp, q, k, v, g, b, out, hin, pipe
    torch.cuda.empty_cache()
    return res


def _timed_flushed(fn, steps, warmup, device, stream):
    """Per-iteration CUDA-event timing with the L2 flushed (a 256 MiB write, outside the timed
    span) before every iteration; for workloads smaller than L2. Returns (mean ms, clocks)."""
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize(device)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    with ClockSampler(device) as cs:
        _hold_stream(stream)
        for e0, e1 in ev:
            flush.fill_(1)
            e0.record(stream)
            fn()
            e1.record(stream)
        torch.cuda.synchronize(device)
    del flush
    return sum(e0.elapsed_time(e1) for e0, e1 in ev) / steps, cs.summary()


def _as_graph(fn, device):
    """Captures fn (which launches on torch's current stream) into a CUDA graph, so that a timed
    replay is one launch from the host; None if capture is not possible here."""
    try:
        side = torch.cuda.Stream(device)
        side.wait_stream(torch.cuda.current_stream(device))
        with torch.cuda.stream(side):
            fn()
        torch.cuda.current_stream(device).wait_stream(side)
        torch.cuda.synchronize(device)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            fn()
        torch.cuda.synchronize(device)
        return graph
    except Exception:  # capture refused: time the direct calls instead
        torch.cuda.synchronize(device)
        return None


def bench_small(kda, args, world, rank, device, stream, peaks, steps=20):
    """B=1, H=8, T=4096: eight (sequence, head) problems, far fewer than the SMs. Timed as the
    plain prefill (one CTA per problem) and segment-parallel along T (automatic segments)."""
    w = kda_synth.WORKLOADS[1]
    B, T, H, C = w["B"], w["T"], w["H"], w["C"]
    inp = kda_synth.make_prefill_inputs(B, T, H, D, D, "bf16", seed=w["seed"] + rank,
                                        S0_std=w["S0_std"], device=device)
    q, k, v, g, b, S0 = (inp[n] for n in ("q", "k", "v", "g", "beta", "S0"))
    out = torch.empty(B, T, H, D, dtype=torch.bfloat16, device=device)
    Sf = torch.empty(B, H, D, D, dtype=torch.float32, device=device)
    n_seg = kda.segments_auto(B, H, T)
    ws = torch.empty(max(1, kda.segmented_workspace_bytes(B, H, T, D, D, n_seg)),
                     dtype=torch.uint8, device=device)

    def plain():
        kda.kda_chunk_fwd(q, k, v, g, b, S0, out, Sf, C=C,
                          stream=torch.cuda.current_stream(device))

    def seg():
        kda.kda_chunk_fwd_segmented(q, k, v, g, b, S0, out, Sf, n_seg, ws, C=C,
                                    stream=torch.cuda.current_stream(device))

    # A call is 0.1-0.3 ms of device work: replayed from a CUDA graph, so that the host's
    # launch work (argument checks, tensor-map encodes) cannot leave gaps inside the timed span.
    graphs = {name: _as_graph(fn, device) for name, fn in (("plain", plain), ("seg", seg))}
    run = {name: (graphs[name].replay if graphs[name] is not None else fn)
           for name, fn in (("plain", plain), ("seg", seg))}
    ms_plain, _ = _timed_flushed(run["plain"], steps, 3, device, stream)
    ms_seg, clocks = _timed_flushed(run["seg"], steps, 3, device, stream)
    kda.kda_sync_status(stream)
    launch = ("CUDA graph replay" if all(gr is not None for gr in graphs.values())
              else "direct calls (graph capture unavailable)")
    token_heads = B * T * H
    alg = token_heads * BYTES_PER_TOKEN_HEAD + 2 * B * H * STATE_BYTES  # S0 read, S_final written
    gbs = alg / (ms_seg * 1e-3) / 1e9
    del inp, q, k, v, g, b, S0, out, ws, graphs, run
    torch.cuda.empty_cache()
    return {"workload": w["name"], "n_seg": n_seg, "ms_per_step": ms_seg,
            "ms_per_step_unsegmented": ms_plain, "tokens_per_s": world * B * T / (ms_seg * 1e-3),
            "tokens_per_s_unsegmented": world * B * T / (ms_plain * 1e-3),
            "tflops": token_heads * useful_flops_per_token_head(C) / (ms_seg * 1e-3) / 1e12,
            "l2": "flushed before every timed iteration (256 MiB write outside the timed span)",
            "launch": launch, "clocks": clocks,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm"], "traffic": None,
                         "algorithmic_bytes_per_launch": alg,
                         "note": "43 MB moved: far below the size at which HBM bandwidth can be "
                                 "reached; the fraction shows the latency floor"}}


def bench_decode(kda, args, world, rank, device, stream, peaks, steps=64):
    w = kda_synth.WORKLOADS[4]
    N, H = w["N"], w["H"]
    dec = kda_synth.make_decode_inputs(N, H, D, D, "bf16", seed=w["seed"] + rank,
                                       S0_std=w["S0_std"], steps=steps, device=device)
    S = dec["S"]
    outs = [torch.empty(N, H, D, dtype=torch.bfloat16, device=device) for _ in range(steps)]
    seq = [[st[n] for n in ("q", "k", "v", "g", "beta")] for st in dec["steps"]]

    def run64():
        for i in range(steps):
            kda.kda_recurrent_step(*seq[i], S, outs[i], stream=stream)

    total_ms, clocks = _timed(run64, 1, 1, world, device, stream)
    kda.kda_sync_status(stream)
    ms_step = total_ms / steps
    bytes_step = N * H * decode_bytes_per_head()
    gbs = bytes_step / (ms_step * 1e-3) / 1e9
    del dec, S, outs, seq
    torch.cuda.empty_cache()
    return {"workload": w["name"], "ms_per_step": ms_step, "steps_timed": steps,
            "tokens_per_s": world * N / (ms_step * 1e-3), "clocks": clocks,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm"],
                         "frac_of_8tbs": gbs / 8000.0,
                         "traffic": _recorded_traffic("decode_bf16_N256_H96"),
                         "traffic_note": "ncu DRAM bytes of a 32-sequence step scaled by "
                                         "sequences; writes still held in L2 when the kernel "
                                         "ends are not counted, so this is a lower bound",
                         "algorithmic_bytes_per_launch": bytes_step}}


def bench_varlen(kda, args, world, rank, device, stream, peaks, steps=3):
    w = kda_synth.WORKLOADS[3]
    T, H, C = w["T"], w["H"], w["C"]
    inp = kda_synth.make_varlen_inputs(T, H, D, D, w["n_seq"], "bf16", seed=w["seed"] + rank,
                                       device=device)
    cu = inp["cu_seqlens"].to(device)
    q, k, v, g, b = (inp[n] for n in ("q", "k", "v", "g", "beta"))
    N = cu.numel() - 1
    out = torch.empty(1, T, H, D, dtype=torch.bfloat16, device=device)
    Sf = torch.empty(N, H, D, D, dtype=torch.float32, device=device)

    def step():
        kda.kda_chunk_fwd_varlen(q, k, v, g, b, None, out, Sf, cu, C=C, stream=stream)

    total_ms, clocks = _timed(step, steps, 1, world, device, stream)
    kda.kda_sync_status(stream)
    ms = total_ms / steps
    alg = T * H * BYTES_PER_TOKEN_HEAD + N * H * STATE_BYTES
    gbs = alg / (ms * 1e-3) / 1e9
    lens = (inp["cu_seqlens"][1:] - inp["cu_seqlens"][:-1]).tolist()
    del inp, q, k, v, g, b, out
    torch.cuda.empty_cache()
    # the tensor-core kernel serves a 128-token chunk as two 64-token blocks: count that work
    block = 64 if C in (64, 128) else C
    return {"workload": w["name"], "ms_per_step": ms, "seq_lens": lens, "C": C,
            "block_tokens": block, "tokens_per_s": world * T / (ms * 1e-3),
            "tflops": T * H * useful_flops_per_token_head(block) / (ms * 1e-3) / 1e12,
            "clocks": clocks,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm"],
                         "traffic": _recorded_traffic("varlen_bf16_H96_T131072_C128"),
                         "algorithmic_bytes_per_launch": alg}}


def bench_layer_sides(kda, args, world, rank, device, stream, peaks, steps=5):
    """The layers around the core at the B=4, H=96, T=8192 shape: the output side (RMSNorm of the
    raw output times the sigmoid gate) fused into the prefill's epilogue vs the plain prefill
    plus the standalone gate pass; the input side (ShortConv, L2Norm, decay gate) fused into the
    prefill vs the standalone input pass plus the plain prefill."""
    w = kda_synth.WORKLOADS[2]
    B, T, H, C = w["B"], w["T"], w["H"], w["C"]
    inp = kda_synth.make_prefill_inputs(B, T, H, D, D, "bf16", seed=w["seed"] + rank,
                                        g_bias=True, device=device)
    x = [inp[n] for n in ("q", "k", "v", "g", "beta")]
    gen = torch.Generator(device=device).manual_seed(1234 + rank)
    u = torch.randn(B, T, H, D, generator=gen, device=device).to(torch.bfloat16)
    nw = 1.0 + 0.1 * torch.randn(D, generator=gen, device=device)
    conv = [0.5 * torch.randn(H, 4, D, generator=gen, device=device) for _ in range(3)]
    A_log = 0.1 * torch.randn(H, generator=gen, device=device)
    b_dec = torch.rand(H, D, generator=gen, device=device) * 4 - 2
    out = torch.empty(B, T, H, D, dtype=torch.bfloat16, device=device)
    Sf = torch.empty(B, H, D, D, dtype=torch.float32, device=device)
    qkvg = [torch.empty_like(x[0]) for _ in range(4)]
    prm = conv + [A_log, b_dec]

    def t(fn):
        ms, _ = _timed(fn, steps, 2, world, device, stream)
        return ms / steps

    core = t(lambda: kda.kda_chunk_fwd(*x, None, out, Sf, C=C, stream=stream))
    gated = t(lambda: kda.kda_chunk_fwd_gated(*x, None, u, nw, out, Sf, C=C, stream=stream))
    gate_alone = t(lambda: kda.kda_output_gate(out, u, nw, out, stream=stream))
    pre_alone = t(lambda: kda.kda_pre_core(x[0], x[1], x[2], x[3], *prm, *qkvg, stream=stream))
    fused_in = t(lambda: kda.kda_chunk_fwd_fused(x[0], x[1], x[2], x[3], x[4], *prm, None, out, Sf,
                                                 C=C, stream=stream))
    fused_both = t(lambda: kda.kda_chunk_fwd_fused(x[0], x[1], x[2], x[3], x[4], *prm, None, out,
                                                   Sf, gate_u=u, norm_w=nw, C=C, stream=stream))
    kda.kda_sync_status(stream)
    th = B * T * H
    gate_bytes = th * D * 2 * 3  # o~ and u in, y out
    pre_bytes = th * D * 2 * 8   # q~, k~, v~, z in; q, k, v, g out
    del inp, x, u, out, qkvg, conv
    torch.cuda.empty_cache()
    return {"workload": w["name"], "ms_core": core,
            "output_side": {"ms_fused_in_epilogue": gated, "ms_core_plus_standalone_gate": core + gate_alone,
                            "ms_standalone_gate": gate_alone,
                            "standalone_gate_gbs": gate_bytes / (gate_alone * 1e-3) / 1e9},
            "input_side": {"ms_fused_in_prefill": fused_in,
                           "ms_standalone_pass_plus_core": pre_alone + core,
                           "ms_standalone_pass": pre_alone,
                           "standalone_pass_gbs": pre_bytes / (pre_alone * 1e-3) / 1e9},
            "ms_fused_both_sides": fused_both,
            "tokens_per_s_fused_both_sides": world * B * T / (fused_both * 1e-3)}


def bench_decode_tokens(kda, args, world, rank, device, stream, peaks, K=4, calls=16):
    """K = 4 decode tokens per (sequence, head) per call for the 256 x 96 state: the state
    crosses HBM once per call whatever K is."""
    w = kda_synth.WORKLOADS[4]
    N, H = w["N"], w["H"]
    dec = kda_synth.make_decode_inputs(N, H, D, D, "bf16", seed=w["seed"] + rank,
                                       S0_std=w["S0_std"], steps=K, device=device)
    stack = [torch.stack([st[n] for st in dec["steps"]], dim=1).contiguous()
             for n in ("q", "k", "v", "g", "beta")]
    S = dec["S"]
    out = torch.empty(N, K, H, D, dtype=torch.bfloat16, device=device)

    def run():
        for _ in range(calls):
            kda.kda_recurrent_steps(*stack, S, out, stream=stream)

    total_ms, clocks = _timed(run, 1, 1, world, device, stream)
    kda.kda_sync_status(stream)
    ms = total_ms / calls
    bytes_call = N * H * (2 * D * D * 4 + K * ((3 * D + D) * 2 + 2 + D * 2))
    gbs = bytes_call / (ms * 1e-3) / 1e9
    del dec, stack, S, out
    torch.cuda.empty_cache()
    return {"workload": f"decode_bf16_N{N}_H{H}_K{K}", "K": K, "ms_per_call": ms,
            "tokens_per_s": world * N * K / (ms * 1e-3), "clocks": clocks,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm"],
                         "traffic": _recorded_traffic(f"decode_tokens_bf16_N{N}_H{H}_K{K}"),
                         "algorithmic_bytes_per_launch": bytes_call}}


def bench_nano(kda, args, world, rank, device, stream, peaks, steps=5):
    """The nano-K3 head shape (8 heads x 64 channels, context 2048), 64 sequences, bf16: the
    tensor-core kernel with 64-channel heads (run in its 128-channel tiles, upper half zero)."""
    B, T, H, d, C = 64, 2048, 8, 64, 64
    inp = kda_synth.make_prefill_inputs(B, T, H, d, d, "bf16", seed=rank, device=device)
    x = [inp[n] for n in ("q", "k", "v", "g", "beta")]
    out = torch.empty(B, T, H, d, dtype=torch.bfloat16, device=device)
    Sf = torch.empty(B, H, d, d, dtype=torch.float32, device=device)
    total_ms, clocks = _timed(lambda: kda.kda_chunk_fwd(*x, None, out, Sf, C=C, stream=stream),
                              steps, 2, world, device, stream)
    kda.kda_sync_status(stream)
    ms = total_ms / steps
    alg = B * T * H * (3 * d * 2 + d * 2 + 2 + d * 2) + B * H * d * d * 4
    gbs = alg / (ms * 1e-3) / 1e9
    del inp, x, out
    torch.cuda.empty_cache()
    return {"workload": f"kda_bf16_B{B}_H{H}_T{T}_d{d}_C{C}", "ms_per_step": ms,
            "tokens_per_s": world * B * T / (ms * 1e-3),
            "tflops": B * T * H * useful_flops_per_token_head(C, d, d) / (ms * 1e-3) / 1e12,
            "clocks": clocks,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm"],
                         "traffic": _recorded_traffic(f"nano_bf16_B{B}_H{H}_T{T}_d{d}"),
                         "algorithmic_bytes_per_launch": alg}}


def cpu_baseline_varlen(budget_s=8.0):
    """The oracle on a bounded sample of the packed workload: whole (sequence, head) problems of
    the shortest sequences, timed on all host cores; tokens = token-heads / H."""
    import oracle

    w = kda_synth.WORKLOADS[3]
    T, H = w["T"], w["H"]
    cu = kda_synth.varlen_cu_seqlens(T, w["n_seq"], w["seed"])
    lens = sorted((cu[1:] - cu[:-1]).tolist())
    cores = oracle.default_threads()
    Ls = lens[0]
    n = cores
    x = _cpu_sample(Ls, n, seed=1)
    t0 = time.perf_counter()
    oracle.recurrent(*x, nthreads=cores)
    dt = time.perf_counter() - t0
    return {"value": n * Ls / H / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} complete (sequence, head) problems of {Ls} tokens (the shortest "
                      f"packed sequence) in {dt:.2f} s; tokens = token-heads / H={H}"}


def cpu_baseline_decode(heads=2048, steps=8):
    """The oracle's decode step on a bounded sample: `heads` (sequence, head) states for `steps`
    steps, scaled to the 256 x 96 state; tokens/s = 256 sequences per step."""
    import oracle

    w = kda_synth.WORKLOADS[4]
    N, H = w["N"], w["H"]
    dec = kda_synth.make_decode_inputs(heads, 1, D, D, "bf16", seed=2, steps=steps)
    S = kda_synth.to_f64_numpy(dec["S"])
    xs = [[kda_synth.to_f64_numpy(st[n]) for n in ("q", "k", "v", "g", "beta")]
          for st in dec["steps"]]
    t0 = time.perf_counter()
    for x in xs:
        _, S = oracle.decode_step(*x, S)
    dt = time.perf_counter() - t0
    per_step = dt / steps * (N * H) / heads
    return {"value": N / per_step, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{heads} states x {steps} steps in {dt:.2f} s on one thread, scaled to "
                      f"{N} x {H} states ({per_step * 1e3:.1f} ms per step)"}


def run_gpu(args):
    import gated_delta_rule_167_b300 as kda

    world, rank, local = _dist_setup(args)
    device = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(device)
    kda.load_library()
    stream = torch.cuda.current_stream(device)
    peaks = _peaks()

    pre = bench_prefill(kda, args, world, rank, device, stream, peaks)
    secondary = {}
    if not args.headline_only:
        secondary["small"] = bench_small(kda, args, world, rank, device, stream, peaks)
        secondary["decode"] = bench_decode(kda, args, world, rank, device, stream, peaks)
        secondary["varlen"] = bench_varlen(kda, args, world, rank, device, stream, peaks)
        secondary["decode_tokens"] = bench_decode_tokens(kda, args, world, rank, device, stream, peaks)
        secondary["layer_sides"] = bench_layer_sides(kda, args, world, rank, device, stream, peaks)
        secondary["nano_d64"] = bench_nano(kda, args, world, rank, device, stream, peaks)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline()
        if not args.headline_only:
            secondary["decode"]["cpu_baseline"] = cpu_baseline_decode()
            secondary["varlen"]["cpu_baseline"] = cpu_baseline_varlen()

    if rank == 0:
        line = {
            "metric": "KDA fwd tokens/s (B=4,H=96,T=8192,d=128,C=64)",
            "value": pre["tokens_per_s"], "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": pre["ms"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": "kda_bf16_B4_H96_T8192_d128_C64", "B": 4, "H": 96,
                       "T": 8192, "d_k": 128, "d_v": 128, "C": 64, "state": "fp32",
                       "global_batch": 4 * world, "seq_len": 8192,
                       "parallelism": f"dp{world}" if world > 1 else "none",
                       "l2": "inputs larger than L2 (3.2 GB per step)"},
            "tflops": pre["tflops"], "tensor_frac_of_bf16_peak": pre["tensor_frac_of_bf16_peak"],
            "roofline": pre["roofline"], "clocks": pre["clocks"], "e2e": pre["e2e"],
            "gpu_launches": args.steps, "cpu_baseline": cpu,
        }
        line.update(secondary)
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--headline-only", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
