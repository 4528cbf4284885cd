#!/usr/bin/env python
"""Benchmark of exact attention forward + backward on GB300.

One step = the whole hot path over one batch of synthetic input: the forward
(O, L) and the backward (D pre-pass, dK/dV, dQ) of attention for the long-
context workload B=1, H=32, N=8192, d=128, bf16, causal.  Inputs are resident
in HBM before timing; the four inputs (256 MiB) and the per-kernel working sets
exceed the 126 MB L2, so no flush is needed between steps.  Smaller workloads
(--workload) whose inputs fit in L2 get a buffer of four times the L2 size
written between steps, outside the timed spans.

Prints one JSON line (rank 0).  FLOPs follow the usual convention: 4*B*H*N^2*d
forward, 2.5x that backward, halved when causal.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the fp64 CPU oracle on the host cores instead (one
(batch, head) pair of the same workload per step); it is the slow definition,
reported for scale, not a target.
Multi-GPU (torchrun): every rank runs its own full copy of the workload
(independent problems, no collective on the data path): weak scaling.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd/bwd TFLOP/s (N=8K,d=128,bf16,causal); % of GB300 tensor peak"
WORKLOADS = {
    # name: (B, H, N, d, dtype, causal[, Hkv[, window]]); Hkv < H: K/V heads shared by
    # groups of H/Hkv query heads (grouped-query attention), same FLOPs as H independent
    # heads; window > 0: causal sliding window of that many keys
    "n8k_causal_d128_bf16": (1, 32, 8192, 128, "bf16", True),
    "n16k_causal_d128_bf16": (1, 32, 16384, 128, "bf16", True),
    "n4k_causal_d128_bf16": (2, 16, 4096, 128, "bf16", True),
    "n4k_full_d128_bf16": (2, 16, 4096, 128, "bf16", False),
    "gpt2m_causal_d64_fp16": (8, 16, 1024, 64, "fp16", True),
    "ragged_causal_d32_fp16": (4, 8, 1000, 32, "fp16", True),
    "tiny_full_d64_fp16": (1, 1, 128, 64, "fp16", False),
    "gqa8_n8k_causal_d128_bf16": (1, 32, 8192, 128, "bf16", True, 8),
    "swa4k_gqa8_n16k_d128_bf16": (1, 32, 16384, 128, "bf16", True, 8, 4096),
}
# packed variable-length batches: name: (sequences, min len, max len, H, Hkv, d, dtype,
# causal); lengths uniform in [min, max] from a fixed seed
VARLEN_WORKLOADS = {
    "varlen64_gqa8_d128_bf16": (64, 256, 8192, 32, 8, 128, "bf16", True),
}
# split-KV decoding: name: (B, H, Hkv, Nmax, d, dtype); one query row per (batch, head)
# against K/V caches of lengths uniform in [Nmax/2, Nmax] from a fixed seed
DECODE_WORKLOADS = {
    "decode_b16_gqa8_kv32k_d128_bf16": (16, 32, 8, 32768, 128, "bf16"),
    # the same with E4M3 caches (per-tensor descale factors), bf16 q and O
    "decode_fp8cache_b16_gqa8_kv32k_d128": (16, 32, 8, 32768, 128, "bf16", "e4m3"),
}
DECODE_METRIC = "split-KV decode KV-cache read GB/s (B=16,H=32,Hkv=8,cache<=32K,d=128,bf16)"
DECODE8_METRIC = ("split-KV decode KV-cache read GB/s (B=16,H=32,Hkv=8,cache<=32K,d=128, "
                  "E4M3 caches)")


# forward on 8-bit E4M3 inputs: name: (B, H, Hkv, N, causal), d = 128
FP8_WORKLOADS = {
    "fp8_n8k_causal_d128": (1, 32, 32, 8192, True),
}
FP8_METRIC = "attention fwd TFLOP/s on E4M3 inputs (N=8K,d=128,causal); % of GB300 fp8 tensor peak"


def decode_workload(name):
    """(B, H, Hkv, Nmax, d, dtype, c8) of a decoding workload; c8: E4M3 caches."""
    w = DECODE_WORKLOADS[name]
    return (*w[:6], len(w) > 6 and w[6] == "e4m3")


def make_decode_x(name, seed):
    """Inputs of a decoding workload: q, k_cache, v_cache, cache_seqlens, and for E4M3
    caches the codes with k_scale, v_scale."""
    from exact_io_aware_22_gb300 import inputs
    B, H, Hkv, Nmax, d, dtype, c8 = decode_workload(name)
    lens = decode_lengths(name)
    if not c8:
        return inputs.make_decode_inputs(B, H, Hkv, Nmax, d, lens, dtype, seed=seed)
    x = inputs.make_decode_fp8_inputs(B, H, Hkv, Nmax, d, lens, dtype, seed=seed)
    return {"q": x["q"], "k_cache": x["k8"], "v_cache": x["v8"],
            "cache_seqlens": x["cache_seqlens"], "k_scale": x["k_scale"], "v_scale": x["v_scale"]}


def oracle_cache(x, name, sl, n):
    """fp64 cache rows [0, n) of batch entries sl, decoded from E4M3 codes if need be."""
    import oracle
    kc, vc = x["k_cache"][sl, :, :n], x["v_cache"][sl, :, :n]
    if "k_scale" in x:
        return (oracle.e4m3_values(kc.numpy()) * x["k_scale"],
                oracle.e4m3_values(vc.numpy()) * x["v_scale"])
    return kc.double().numpy(), vc.double().numpy()


def decode_lengths(name):
    import numpy as np
    B, _, _, Nmax = DECODE_WORKLOADS[name][:4]
    return [int(x) for x in np.random.default_rng(2027).integers(Nmax // 2, Nmax + 1, B)]


def varlen_lengths(name):
    import numpy as np
    n, lo, hi = VARLEN_WORKLOADS[name][:3]
    return [int(x) for x in np.random.default_rng(2026).integers(lo, hi + 1, n)]


def workload(name):
    """(B, H, Hkv, N, d, dtype, causal, window) of a named workload."""
    w = WORKLOADS[name]
    B, H, N, d, dtype, causal = w[:6]
    return (B, H, (w[6] if len(w) > 6 else H), N, d, dtype, causal,
            (w[7] if len(w) > 7 else 0))
DEFAULT_WORKLOAD = "n8k_causal_d128_bf16"
L2_BYTES = 129 * 1000 * 1000        # GB300 L2 (126 MiB)
# at head dims 32 and 64 the backward runs the persistent kernels of fa_bwd64.cu
SMALL_D_SOURCES = {
    "bwd_dkdv_kernel": "exact_io_aware_22_gb300/csrc/fa_bwd64.cu",
    "bwd_dq_kernel": "exact_io_aware_22_gb300/csrc/fa_bwd64.cu",
}
KERNEL_SOURCES = {
    "fwd_kernel": "exact_io_aware_22_gb300/csrc/fa_fwd.cu",
    "bwd_pre_kernel": "exact_io_aware_22_gb300/csrc/fa_bwd.cu",
    "bwd_dkdv_kernel": "exact_io_aware_22_gb300/csrc/fa_bwd128.cu",
    "bwd_dq_kernel": "exact_io_aware_22_gb300/csrc/fa_bwd128.cu",
    "decode_split_kernel": "exact_io_aware_22_gb300/csrc/fa_decode.cu",
    "fwd_fp8_kernel": "exact_io_aware_22_gb300/csrc/fa_fwd8.cu",
}


def attn_flops(B, H, N, d, causal, window=0):
    """(forward, backward) FLOPs: 4*d per (query, allowed key) pair forward, 2.5x that
    backward.  Causal counts N^2/2 pairs (the usual halving); a sliding window of W < N
    keys counts its exact pairs, W(W+1)/2 + (N-W)W."""
    if window and window < N:
        pairs = window * (window + 1) / 2 + (N - window) * window
    else:
        pairs = N * N * (0.5 if causal else 1.0)
    f = 4.0 * B * H * pairs * d
    return f, 2.5 * f


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest of every rank's value (the slowest rank's time)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_rank: float, world: int, ms_max: float) -> float:
    """Weak scaling: every rank runs its own copy of the workload; the job is done when the
    slowest rank is."""
    return world * flops_per_rank / (ms_max / 1e3) / 1e12


def e2e_measure(torch, h_in, dev_sets, h_out_sets, compute, steps, barrier):
    """Milliseconds per step, (pipelined, sequential), of whole steps through the public
    API with host buffers: every step copies its inputs from pinned host memory to the
    device, computes, and copies its results back to pinned host memory.

    Pipelined: step k's inputs go host -> device on one stream while step k-1 computes
    on a second and step k-2's results go device -> host on a third (full-duplex host
    link, copy engines beside the SMs), the device tensors double-buffered.  Sequential:
    copy in, compute, copy out, one step after another on one stream."""
    s_in, s_c, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_c = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    state = {"k": 0}

    def launch():
        k = state["k"]
        b = k % 2
        d, ho = dev_sets[b], h_out_sets[b]
        with torch.cuda.stream(s_in):
            if k >= 2:
                s_in.wait_event(ev_c[b])              # step k-2 has read set b's inputs
            for n, t in h_in.items():
                d[n].copy_(t, non_blocking=True)
            ev_in[b].record(s_in)
        with torch.cuda.stream(s_c):
            s_c.wait_event(ev_in[b])
            if k >= 2:
                s_c.wait_event(ev_out[b])             # step k-2's results have left set b
            compute(d)
            ev_c[b].record(s_c)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_c[b])
            for n, h in ho.items():
                h.copy_(d[n], non_blocking=True)
            ev_out[b].record(s_out)
        state["k"] = k + 1

    for _ in range(2):
        launch()
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for _ in range(steps):
        launch()
    e1.record(s_out)
    torch.cuda.synchronize()
    barrier()
    pipelined = e0.elapsed_time(e1) / steps

    d, ho = dev_sets[0], h_out_sets[0]
    st = torch.cuda.current_stream()

    def seq_step():
        for n, t in h_in.items():
            d[n].copy_(t, non_blocking=True)
        compute(d)
        for n, h in ho.items():
            h.copy_(d[n], non_blocking=True)

    seq_step()
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(steps):
        seq_step()
    e1.record(st)
    torch.cuda.synchronize()
    barrier()
    return pipelined, e0.elapsed_time(e1) / steps


# The end-to-end loop runs as many steps as the device loop (up to this many), so that
# filling and draining its three-stream pipeline (one step's copy in, one step's copy
# out) is spread over as many steps as the device timing's own start-up is.
E2E_MAX_STEPS = 100

E2E_NOTE = ("pipelined: step k's inputs copied host->device while step k-1 computes and step "
            "k-2's results are copied device->host (three streams, device tensors "
            "double-buffered); every step moves its own inputs and results")
E2E_SEQ_NOTE = "sequential: copy in, compute, copy out, one step after another on one stream"


def e2e_pick(pms, sms):
    """(ms per step, mode, other mode's ms) of the faster of the two end-to-end modes."""
    if pms <= sms:
        return pms, E2E_NOTE, ("sequential", sms)
    return sms, E2E_SEQ_NOTE, ("pipelined", pms)


def emit(out: dict, args) -> None:
    """Print the result as one JSON line; with --json-out also write it to that file."""
    line = json.dumps(out)
    print(line, flush=True)
    path = getattr(args, "json_out", None)
    if path:
        d = os.path.dirname(os.path.abspath(path))
        os.makedirs(d, exist_ok=True)
        with open(path, "w") as f:
            f.write(line + "\n")


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload",
                    choices=list(WORKLOADS) + list(VARLEN_WORKLOADS) + list(DECODE_WORKLOADS)
                    + list(FP8_WORKLOADS),
                    default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--json-out", default=None,
                    help="also write the JSON line to this file (rank 0)")
    return ap.parse_args(argv)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"bf16_tflops": d["bf16_tflops"], "bf16_tflops_sustained": d.get("bf16_tflops_sustained"),
                "hbm_gbs": d["hbm_gbs"], "source": "measured"}
    return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0,
            "source": "fallback"}


def kernel_source(kernel: str, workload: str) -> str:
    """Source file of the kernel that the trace kind `kernel` times on `workload`."""
    if workload in WORKLOADS and WORKLOADS[workload][3] <= 64 and kernel in SMALL_D_SOURCES:
        return SMALL_D_SOURCES[kernel]
    return KERNEL_SOURCES[kernel]


def profile_record(kernel: str, workload: str):
    """(dram bytes per launch, tensor-pipe active % of elapsed cycles) recorded by ncu in
    profiles/<kernel>__<workload>.txt; (None, None) when the file is missing or the
    kernel's source changed since the capture, and None for a figure it lacks."""
    path = os.path.join(ROOT, "profiles", f"{kernel}__{workload}.txt")
    src = os.path.join(ROOT, kernel_source(kernel, workload))
    if not os.path.exists(path) or not os.path.exists(src):
        return None, None
    text = open(path).read()
    m_sha = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
    if not m_sha or sha != m_sha.group(1):
        return None, None
    m_b = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    m_t = re.search(r"sm__pipe_tensor_cycles_active[^\n]*?([0-9.]+) %", text)
    return (float(m_b.group(1)) if m_b else None), (float(m_t.group(1)) if m_t else None)


def traffic_from_profiles(kernel: str, workload: str):
    """dram bytes per launch recorded in profiles/<kernel>__<workload>.txt, or None when
    the file is missing or the kernel's source changed since the capture."""
    return profile_record(kernel, workload)[0]


# Dense 16-bit tcgen05.mma rate of one SM per clock (M = 128, N >= 128, back-to-back
# MMAs on one SM: 64 cycles per 128 x 128 x 16 product); the 8-bit kind runs at twice it.
TENSOR_FLOP_PER_CLK_SM = 8192


def tensor_rate_at_clock(sm_count: int, sm_mhz: float, bits: int = 16) -> float:
    """TFLOP/s the tensor pipes of sm_count SMs deliver at sm_mhz when never idle."""
    return TENSOR_FLOP_PER_CLK_SM * (2 if bits == 8 else 1) * sm_count * sm_mhz * 1e6 / 1e12


def memory_report(lens, H, d, elem, device_bytes, peak_bytes):
    """The footprint arithmetic of the pages' calculator for sequences of the given
    lengths (B equal lengths N for a dense batch): the H*N*N score matrix per sequence
    that ordinary attention materialises against everything the tiled kernel keeps (Q,
    K, V, O in the input type plus L in fp32), their ratio, the N at which the score
    matrix of len(lens) sequences of N alone no longer fits the device, and the peak
    device bytes one step of this library held (inputs, outputs, workspace)."""
    score = sum(H * n * n * elem for n in lens)
    linear = sum(4 * H * n * d * elem + 4 * H * n for n in lens)
    oom_n = math.isqrt(device_bytes // (len(lens) * H * elem))
    return {"peak_device_bytes_step": peak_bytes, "score_matrix_bytes": score,
            "linear_footprint_bytes": linear, "score_over_linear": score / linear,
            "ordinary_attention_runs_out_at_N": oom_n, "device_bytes": device_bytes}


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str, period_ms: int = 20):
        self.lines = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", gpu_id, "-lms", str(period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def _head(flat, h, grp):
    """Query head h (flat b*H+h index) with its K/V head, as (1, 1, N, d) fp64 arrays."""
    return {n: flat[n][(h // grp if n in ("k", "v") else h):][:1].double().numpy()[None]
            for n in flat}


def cpu_baseline(x, B, H, N, d, causal, scale, budget_s=10.0, max_heads=8, window=0):
    """Time the fp64 oracle as it stands on the host cores over whole (batch, head) pairs
    of the workload until ``budget_s`` is spent (at least one pair)."""
    import numpy as np
    import oracle
    fwd_f, bwd_f = attn_flops(1, 1, N, d, causal, window)
    heads, t_fwd, t_bwd = 0, 0.0, 0.0
    flat = {n: x[n].reshape(-1, N, d) for n in ("q", "k", "v", "do")}
    grp = H * B // flat["k"].shape[0]
    while heads < min(max_heads, B * H) and (heads == 0 or t_fwd + t_bwd < budget_s):
        sel = _head(flat, heads, grp)
        t0 = time.perf_counter()
        oracle.fwd(sel["q"], sel["k"], sel["v"], causal, scale, window)
        t1 = time.perf_counter()
        oracle.bwd(sel["q"], sel["k"], sel["v"], sel["do"], causal, scale, window)
        t2 = time.perf_counter()
        t_fwd, t_bwd = t_fwd + (t1 - t0), t_bwd + (t2 - t1)
        heads += 1
    t_total = t_fwd + t_bwd
    value = heads * (fwd_f + bwd_f) / t_total / 1e12
    return {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
            "affinity_cores": len(os.sched_getaffinity(0)),
            "fwd_tflops": heads * fwd_f / t_fwd / 1e12, "bwd_tflops": heads * bwd_f / t_bwd / 1e12,
            "fwd_s_per_pair": t_fwd / heads, "bwd_s_per_pair": t_bwd / heads,
            "sample": f"{heads} of {B * H} (batch, head) pairs, full N={N}, fwd+bwd, "
                      f"{t_total:.1f} s on host cores"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    from exact_io_aware_22_gb300 import inputs
    B, H, Hkv, N, d, dtype, causal, window = workload(args.workload)
    scale = 1.0 / math.sqrt(d)
    x = inputs.make_inputs(B, H, N, d, dtype, seed=0, Hkv=Hkv)
    flat = {n: x[n].reshape(-1, N, d) for n in ("q", "k", "v", "do")}
    fwd_f, bwd_f = attn_flops(1, 1, N, d, causal, window)

    def step(i):
        sel = _head(flat, i % (B * H), H // Hkv)
        oracle.fwd(sel["q"], sel["k"], sel["v"], causal, scale, window)
        oracle.bwd(sel["q"], sel["k"], sel["v"], sel["do"], causal, scale, window)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    dt = time.perf_counter() - t0
    ms = dt / args.steps * 1e3
    value = (fwd_f + bwd_f) / (ms / 1e3) / 1e12
    sample = f"one (batch, head) pair per step, full N={N}, fwd+bwd, fp64 oracle"
    out = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "impl": "reference",
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic",
           "config": {"workload": args.workload, "B": B, "H": H, "Hkv": Hkv, "N": N, "d": d,
                      "causal": causal, "window": window, "step_unit": "one (batch, head) pair"},
           "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(),
                            "kind": "oracle", "sample": sample},
           "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    emit(out, args)


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import exact_io_aware_22_gb300 as fa
    from exact_io_aware_22_gb300 import inputs

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    varlen = args.workload in VARLEN_WORKLOADS
    if varlen:
        _, _, _, H, Hkv, d, dtype, causal = VARLEN_WORKLOADS[args.workload]
        lens = varlen_lengths(args.workload)
        B, N, window = len(lens), max(lens), 0
        fwd_f = bwd_f = 0.0
        for n_b in lens:
            f1, b1 = attn_flops(1, H, n_b, d, causal)
            fwd_f, bwd_f = fwd_f + f1, bwd_f + b1
        x = inputs.make_packed_inputs(lens, H, d, dtype, seed=rank, Hkv=Hkv)
        cu = x["cu_seqlens"].to(dev)
        lse_shape = (H, int(sum(lens)))
        ws_bytes = int(fa.load_library().fa_bwd_varlen_workspace_size(B, N, H, d))
    else:
        B, H, Hkv, N, d, dtype, causal, window = workload(args.workload)
        fwd_f, bwd_f = attn_flops(B, H, N, d, causal, window)
        x = inputs.make_inputs(B, H, N, d, dtype, seed=rank, Hkv=Hkv)
        lse_shape = (B, H, N)
        ws_bytes = fa.bwd_workspace_size(B, H, N, d, causal)
    scale = 1.0 / math.sqrt(d)
    torch.cuda.synchronize(dev)
    mem_base = torch.cuda.memory_allocated(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o = torch.empty_like(q)
    lse = torch.empty(lse_shape, dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        if varlen:
            fa.fwd_varlen(q, k, v, cu, N, causal=causal, scale=scale, out=o, lse=lse)
            fa.bwd_varlen(q, k, v, o, lse, do, cu, N, causal=causal, scale=scale, dq=dq, dk=dk,
                          dv=dv, workspace=ws)
            return
        fa.fwd(q, k, v, causal=causal, scale=scale, out=o, lse=lse, window=window)
        fa.bwd(q, k, v, o, lse, do, causal=causal, scale=scale, dq=dq, dk=dk, dv=dv, workspace=ws,
               window=window)

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if fa.device_status() != 0:
        raise RuntimeError("a kernel reported a bounded-wait timeout during warm-up")
    peak_step_bytes = torch.cuda.max_memory_allocated(dev) - mem_base

    try:   # the UUID names this process's GPU whatever CUDA_VISIBLE_DEVICES says
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = str(local_rank)
    # Q, K, V, dO larger than L2: nothing survives in L2 from one step to the next.
    # Otherwise write a buffer larger than L2 between steps and time each step alone.
    in_bytes = sum(t.numel() * t.element_size() for t in (q, k, v, do))
    flush = None
    if in_bytes < L2_BYTES:
        flush = torch.empty(4 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    l2_note = (f"inputs larger than L2 ({in_bytes >> 20} MiB of Q,K,V,dO), no flush" if flush is None
               else f"inputs fit in L2 ({in_bytes >> 20} MiB of Q,K,V,dO): "
                    f"{flush.numel() * 4 >> 20} MiB written between steps, outside the timed spans")
    sampler = ClockSampler(gpu_id)
    time.sleep(0.2)
    barrier()
    torch.cuda.synchronize()

    def timed_steps():
        if flush is None:
            # one event per step boundary: back-to-back steps, per-step times for the median
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
            evs[0].record(stream)
            for i in range(args.steps):
                step()
                evs[i + 1].record(stream)
            sp = list(zip(evs[:-1], evs[1:]))
        else:
            sp = []
            for _ in range(args.steps):
                flush.zero_()
                t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                t0.record(stream)
                step()
                t1.record(stream)
                sp.append((t0, t1))
        torch.cuda.synchronize()
        barrier()
        return sp

    # The step time comes from a pass without per-kernel events: an event recorded
    # between two kernels stops the second from starting while the first drains (the
    # kernels are launched as programmatic dependents).  A second pass of the same
    # steps records an event pair around every kernel for the per-kernel times.
    spans = timed_steps()
    fa.trace_enable(True)
    timed_steps()
    fa.trace_enable(False)
    clocks = sampler.stop()
    if fa.device_status() != 0:
        raise RuntimeError("a kernel reported a bounded-wait timeout in the timed region")
    step_ms = [a.elapsed_time(b) for a, b in spans]
    ms = sum(step_ms) / args.steps
    ms_median = statistics.median(step_ms)
    traced = fa.trace_read()
    ms = max_over_ranks(ms, world, dev)
    value = whole_job_tflops(fwd_f + bwd_f, world, ms)
    launches = sum(n for _, n in traced.values())

    traced = {kname: v for kname, v in traced.items() if v[1] > 0}
    per = {kname: (tot / n, n) for kname, (tot, n) in traced.items()}
    fwd_ms = per["fwd_kernel"][0]
    bwd_ms = sum(t for kname, (t, _) in per.items() if kname.startswith("bwd_"))
    peaks = load_peaks()
    # algorithmic bytes of the forward (Q, K, V read, O and L written) and backward (Q, K, V,
    # O, dO, L read; D written and read; dQ, dK, dV written)
    qb, kvb = q.numel() * 2, k.numel() * 2
    fwd_bytes = 2 * qb + 2 * kvb + lse.numel() * 4
    bwd_bytes = 3 * qb + 2 * kvb + 2 * kvb + qb + 3 * lse.numel() * 4
    # algorithmic work of one launch of each kernel
    elem = 2
    n_bytes = q.numel() * elem
    Np = (N + 127) // 128 * 128
    alg = {
        "fwd_kernel": ("tensor", fwd_f),
        "bwd_dkdv_kernel": ("tensor", 0.8 * bwd_f),     # S, dP recompute, dV, dK: 4 of 5 products
        "bwd_dq_kernel": ("tensor", 0.2 * bwd_f),       # dQ: 1 of 5 products (S, dP recomputed)
        # reads O, dO, L; writes D and L*log2e
        "bwd_pre_kernel": ("hbm", 2 * n_bytes + 4 * lse.numel() + 2 * 4 * B * H * Np),
    }
    top = max(traced, key=lambda kk: traced[kk][0])
    bound, work = alg[top]
    if bound == "tensor":
        achieved = work / (per[top][0] / 1e3) / 1e12
        peak, unit = peaks["bf16_tflops"], "TFLOP/s"
    else:
        achieved = work / (per[top][0] / 1e3) / 1e9
        peak, unit = peaks["hbm_gbs"], "GB/s"
    traffic, tensor_active = profile_record(top, args.workload)
    roofline = {"bound": bound, "kernel": top, "achieved": achieved, "peak": peak, "unit": unit,
                "frac": achieved / peak, "traffic": traffic,
                "peak_source": f"{peaks['source']} (burst)",
                "algorithmic_work_per_launch": work,
                "avg_launch_ms": per[top][0]}
    sm_count = torch.cuda.get_device_properties(dev).multi_processor_count
    if bound == "tensor":
        # the measured peak is cuBLAS at the clock it ran at (power-capped, below this
        # run's); beside it, the fraction of the tensor pipes' rate at this run's median
        # SM clock, and the tensor-pipe activity ncu recorded for this kernel
        run_mhz = clocks["sm_mhz"] if clocks else None
        roofline["ncu_tensor_active_pct"] = tensor_active
        if run_mhz:
            at_clock = tensor_rate_at_clock(sm_count, run_mhz)
            roofline["tensor_rate_at_run_clock"] = at_clock
            roofline["frac_of_tensor_rate_at_run_clock"] = achieved / at_clock

    e2e = None
    if not args.no_e2e:
        h_in = {n: x[n].pin_memory() for n in ("q", "k", "v", "do")}
        outs = {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}
        dev_sets = [{"q": q, "k": k, "v": v, "do": do, **outs},
                    {**{n: torch.empty_like(t) for n, t in (("q", q), ("k", k), ("v", v),
                                                          ("do", do))},
                     **{n: torch.empty_like(t) for n, t in outs.items()}}]
        h_out_sets = [{n: torch.empty(t.shape, dtype=t.dtype).pin_memory() for n, t in outs.items()}
                      for _ in range(2)]

        def compute(dset):
            if varlen:
                fa.fwd_varlen(dset["q"], dset["k"], dset["v"], cu, N, causal=causal, scale=scale,
                              out=dset["o"], lse=dset["lse"])
                fa.bwd_varlen(dset["q"], dset["k"], dset["v"], dset["o"], dset["lse"], dset["do"],
                              cu, N, causal=causal, scale=scale, dq=dset["dq"], dk=dset["dk"],
                              dv=dset["dv"], workspace=ws)
                return
            fa.fwd(dset["q"], dset["k"], dset["v"], causal=causal, scale=scale, out=dset["o"],
                   lse=dset["lse"], window=window)
            fa.bwd(dset["q"], dset["k"], dset["v"], dset["o"], dset["lse"], dset["do"],
                   causal=causal, scale=scale, dq=dset["dq"], dk=dset["dk"], dv=dset["dv"],
                   workspace=ws, window=window)

        ke = max(1, min(args.steps, E2E_MAX_STEPS))
        pms, sms = e2e_measure(torch, h_in, dev_sets, h_out_sets, compute, ke, barrier)
        pms, sms = max_over_ranks(pms, world, dev), max_over_ranks(sms, world, dev)
        ems, mode, (other, oms) = e2e_pick(pms, sms)
        e2e = {"value": whole_job_tflops(fwd_f + bwd_f, world, ems), "unit": "TFLOP/s",
               "h2d_bytes_per_step": in_bytes,
               "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in outs.values()),
               "ms_per_step": ems, "steps": ke, "mode": mode,
               other: {"value": whole_job_tflops(fwd_f + bwd_f, world, oms), "ms_per_step": oms}}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = None if varlen else cpu_baseline(x, B, H, N, d, causal, scale, window=window)

    if rank == 0:
        out = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
               "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
               "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": dtype,
               "data": "synthetic",
               "config": {"workload": args.workload, "B": B, "H": H, "N": N, "d": d,
                          "causal": causal, "Hkv": Hkv, "window": window,
                          "parallelism": f"replicas x{world}",
                          "l2": l2_note,
                          **({"packed_tokens": int(q.shape[0]), "max_seqlen": N,
                              "lengths": "uniform 256..8192, 64 sequences, seed 2026"}
                             if varlen else {})},
               "fwd_ms": fwd_ms, "bwd_ms": bwd_ms, "ms_per_step_median": ms_median,
               "fwd_gbs": fwd_bytes / (fwd_ms / 1e3) / 1e9 if fwd_ms else None,
               "bwd_gbs": bwd_bytes / (bwd_ms / 1e3) / 1e9 if bwd_ms else None,
               "frac_of_hbm_peak": {"fwd": fwd_bytes / (fwd_ms / 1e3) / 1e9 / peaks["hbm_gbs"],
                                    "bwd": bwd_bytes / (bwd_ms / 1e3) / 1e9 / peaks["hbm_gbs"]},
               "fwd_tflops": fwd_f / (fwd_ms / 1e3) / 1e12 if fwd_ms else None,
               "bwd_tflops": bwd_f / (bwd_ms / 1e3) / 1e12 if bwd_ms else None,
               "frac_of_peak": value / world / peaks["bf16_tflops"],
               "frac_of_peak_basis": "measured cuBLAS bf16 burst rate (MEASURED_PEAKS.json "
                                     "bf16_tflops) at the clock it ran at",
               "frac_of_tensor_rate_at_run_clock": (
                   value / world / tensor_rate_at_clock(sm_count, clocks["sm_mhz"])
                   if clocks else None),
               "memory": memory_report(
                   lens if varlen else [N] * B, H, d, 2,
                   torch.cuda.get_device_properties(dev).total_memory, peak_step_bytes),
               "kernels_ms": {kk: per[kk][0] for kk in per},
               "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
               "gpu_launches": launches, "clocks": clocks}
        emit(out, args)


def decode_bytes(lens, H, Hkv, d, elem=2):
    """Algorithmic HBM bytes of one decoding step: every cached K and V row in use read
    once (elem bytes per value), q read, O written (16-bit), L written."""
    return sum(lens) * Hkv * d * elem * 2 + len(lens) * H * (d * 2 * 2 + 4)


def decode_cpu_sample(x, name, lens, H, Hkv, d, scale, budget_s=10.0):
    """Time the fp64 oracle's decode as it stands on the host cores, whole batch entries
    (all heads) at a time until ``budget_s`` is spent (at least one)."""
    import oracle
    elem = 1 if "k_scale" in x else 2
    done, t_total, nbytes = 0, 0.0, 0
    B = len(lens)
    while done < B and (done == 0 or t_total < budget_s):
        sl = slice(done, done + 1)
        q = x["q"][sl].double().numpy()
        kc, vc = oracle_cache(x, name, sl, lens[done])
        t0 = time.perf_counter()
        oracle.decode(q, kc, vc, [lens[done]], scale)
        t_total += time.perf_counter() - t0
        nbytes += decode_bytes([lens[done]], H, Hkv, d, elem)
        done += 1
    return nbytes / t_total / 1e9, done, t_total


def run_decode_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    B, H, Hkv, Nmax, d, dtype, c8 = decode_workload(args.workload)
    lens = decode_lengths(args.workload)
    scale = 1.0 / math.sqrt(d)
    x = make_decode_x(args.workload, 0)
    elem = 1 if c8 else 2

    def step(i):
        b = i % B
        kc, vc = oracle_cache(x, args.workload, slice(b, b + 1), lens[b])
        oracle.decode(x["q"][b:b + 1].double().numpy(), kc, vc, [lens[b]], scale)
        return decode_bytes([lens[b]], H, Hkv, d, elem)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    nbytes = sum(step(args.warmup + i) for i in range(args.steps))
    dt = time.perf_counter() - t0
    value = nbytes / dt / 1e9
    sample = f"one batch entry (all {H} heads, its whole cache) per step, fp64 oracle"
    out = {"metric": DECODE8_METRIC if c8 else DECODE_METRIC, "value": value, "unit": "GB/s",
           "impl": "reference",
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": args.workload, "B": B, "H": H, "Hkv": Hkv, "Nmax": Nmax,
                      "d": d, "cache": "e4m3" if c8 else dtype, "step_unit": "one batch entry"},
           "cpu_baseline": {"value": value, "unit": "GB/s", "cores": oracle.num_threads(),
                            "kind": "oracle", "sample": sample},
           "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    emit(out, args)


def run_decode(args, rank, world, local_rank):
    """One step = one decoding call over the whole batch (split kernel + merge kernel)."""
    import torch
    import torch.distributed as dist

    import exact_io_aware_22_gb300 as fa
    from exact_io_aware_22_gb300 import inputs

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    B, H, Hkv, Nmax, d, dtype, c8 = decode_workload(args.workload)
    lens = decode_lengths(args.workload)
    scale = 1.0 / math.sqrt(d)
    x = make_decode_x(args.workload, rank)
    q, kc, vc, cl = (x[n].to(dev) for n in ("q", "k_cache", "v_cache", "cache_seqlens"))
    o = torch.empty_like(q)
    lse = torch.empty((B, H), dtype=torch.float32, device=dev)
    ws = torch.empty(fa.decode_workspace_size(B, H, Hkv, Nmax, d), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    alg_bytes = decode_bytes(lens, H, Hkv, d, 1 if c8 else 2)
    flops = 4.0 * sum(lens) * H * d

    def run(qq, kk, vv, ll, oo, lo):
        if c8:
            fa.decode_fp8(qq, kk, vv, ll, x["k_scale"], x["v_scale"], scale=scale, out=oo, lse=lo,
                          workspace=ws)
        else:
            fa.decode(qq, kk, vv, ll, scale=scale, out=oo, lse=lo, workspace=ws)

    def step():
        run(q, kc, vc, cl, o, lse)

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if fa.device_status() != 0:
        raise RuntimeError("a kernel reported a bounded-wait timeout during warm-up")
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = str(local_rank)
    sampler = ClockSampler(gpu_id)
    time.sleep(0.2)
    barrier()
    torch.cuda.synchronize()

    def timed_steps():
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(args.steps):
            step()
        t1.record(stream)
        torch.cuda.synchronize()
        barrier()
        return t0, t1

    # step time without per-kernel events (they would stand between the split kernel and
    # the merge kernel, its programmatic dependent); per-kernel times from a second pass
    t0, t1 = timed_steps()
    fa.trace_enable(True)
    timed_steps()
    fa.trace_enable(False)
    clocks = sampler.stop()
    if fa.device_status() != 0:
        raise RuntimeError("a kernel reported a bounded-wait timeout in the timed region")
    ms = max_over_ranks(t0.elapsed_time(t1) / args.steps, world, dev)
    value = world * alg_bytes / (ms / 1e3) / 1e9
    traced = {kk: v for kk, v in fa.trace_read().items() if v[1] > 0}
    launches = sum(n for _, n in traced.values())
    per = {kk: tot / n for kk, (tot, n) in traced.items()}
    peaks = load_peaks()
    split_ms = per["decode_split_kernel"]
    achieved = alg_bytes / (split_ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "kernel": "decode_split_kernel", "achieved": achieved,
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                "traffic": traffic_from_profiles("decode_split_kernel", args.workload),
                "peak_source": f"{peaks['source']} (burst)",
                "algorithmic_work_per_launch": alg_bytes, "avg_launch_ms": split_ms}

    e2e = None
    if not args.no_e2e:
        names = ("q", "k_cache", "v_cache", "cache_seqlens")
        h_in = {n: x[n].pin_memory() for n in names}
        dev_sets = [{"q": q, "k_cache": kc, "v_cache": vc, "cache_seqlens": cl, "o": o, "lse": lse},
                    {**{n: torch.empty_like(t) for n, t in zip(names, (q, kc, vc, cl))},
                     "o": torch.empty_like(o), "lse": torch.empty_like(lse)}]
        h_out_sets = [{"o": torch.empty(o.shape, dtype=o.dtype).pin_memory(),
                       "lse": torch.empty(lse.shape, dtype=lse.dtype).pin_memory()}
                      for _ in range(2)]

        def compute(dset):
            run(dset["q"], dset["k_cache"], dset["v_cache"], dset["cache_seqlens"], dset["o"],
                dset["lse"])

        ke = max(1, min(args.steps, 10))
        pms, sms = e2e_measure(torch, h_in, dev_sets, h_out_sets, compute, ke, barrier)
        pms, sms = max_over_ranks(pms, world, dev), max_over_ranks(sms, world, dev)
        ems, mode, (other, oms) = e2e_pick(pms, sms)
        e2e = {"value": world * alg_bytes / (ems / 1e3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in h_in.values()),
               "d2h_bytes_per_step": o.numel() * o.element_size() + lse.numel() * 4,
               "ms_per_step": ems, "steps": ke, "mode": mode,
               other: {"value": world * alg_bytes / (oms / 1e3) / 1e9, "ms_per_step": oms},
               "note": "the whole K/V cache is copied host to device every step"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        v_cpu, done, t_cpu = decode_cpu_sample(x, args.workload, lens, H, Hkv, d, scale)
        cpu = {"value": v_cpu, "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
               "sample": f"{done} of {B} batch entries (all heads, whole caches), "
                         f"{t_cpu:.1f} s on host cores"}
    if rank == 0:
        out = {"metric": DECODE8_METRIC if c8 else DECODE_METRIC, "value": value, "unit": "GB/s",
               "n_gpus": world,
               "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
               "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": dtype,
               "data": "synthetic",
               "config": {"workload": args.workload, "B": B, "H": H, "Hkv": Hkv, "Nmax": Nmax,
                          "d": d, "cache": "e4m3" if c8 else dtype, "cached_keys": sum(lens),
                          "lengths": f"uniform {Nmax // 2}..{Nmax}, seed 2027",
                          "parallelism": f"replicas x{world}",
                          "l2": f"inputs larger than L2 ({alg_bytes >> 20} MiB of K/V rows "
                                "read per step), no flush"},
               "tflops": world * flops / (ms / 1e3) / 1e12,
               "cached_rows_per_s": world * sum(lens) * Hkv / (ms / 1e3),
               "kernels_ms": per, "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
               "gpu_launches": launches, "clocks": clocks}
        emit(out, args)


def run_fp8_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    from exact_io_aware_22_gb300 import inputs
    B, H, Hkv, N, causal = FP8_WORKLOADS[args.workload]
    d = 128
    scale = 1.0 / math.sqrt(d)
    x = inputs.make_fp8_inputs(B, H, N, d, seed=0, Hkv=Hkv)
    q8, k8, v8 = (x[n].numpy().reshape(-1, N, d) for n in ("q8", "k8", "v8"))
    fwd_f, _ = attn_flops(1, 1, N, d, causal)

    def step(i):
        h = i % (B * H)
        hk = (h // H) * Hkv + (h % H) // (H // Hkv)
        oracle.fwd_fp8(q8[h][None, None], k8[hk][None, None], v8[hk][None, None], x["q_scale"],
                       x["k_scale"], x["v_scale"], causal, scale)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    dt = time.perf_counter() - t0
    value = fwd_f * args.steps / dt / 1e12
    sample = f"one (batch, head) pair per step, full N={N}, forward, fp64 oracle on the E4M3 codes"
    out = {"metric": FP8_METRIC, "value": value, "unit": "TFLOP/s", "impl": "reference",
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": args.workload, "B": B, "H": H, "Hkv": Hkv, "N": N, "d": d,
                      "causal": causal, "step_unit": "one (batch, head) pair"},
           "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(),
                            "kind": "oracle", "sample": sample},
           "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    emit(out, args)


def run_fp8(args, rank, world, local_rank):
    """One step = one forward on the E4M3 inputs (already quantised, in HBM)."""
    import torch
    import torch.distributed as dist

    import exact_io_aware_22_gb300 as fa
    from exact_io_aware_22_gb300 import inputs

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    B, H, Hkv, N, causal = FP8_WORKLOADS[args.workload]
    d = 128
    scale = 1.0 / math.sqrt(d)
    x = inputs.make_fp8_inputs(B, H, N, d, seed=rank, Hkv=Hkv)
    qs, ks, vs = x["q_scale"], x["k_scale"], x["v_scale"]
    q8, k8, vt8 = (x[n].to(dev) for n in ("q8", "k8", "vt8"))
    o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    fwd_f, _ = attn_flops(B, H, N, d, causal)
    stream = torch.cuda.current_stream()

    def step():
        fa.fwd_fp8(q8, k8, vt8, qs, ks, vs, causal=causal, scale=scale, out=o, lse=lse)

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if fa.device_status() != 0:
        raise RuntimeError("a kernel reported a bounded-wait timeout during warm-up")
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = str(local_rank)
    # inputs (96 MiB) fit in L2: a buffer four times L2 is written between steps
    flush = torch.empty(4 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    sampler = ClockSampler(gpu_id)
    time.sleep(0.2)
    barrier()
    torch.cuda.synchronize()
    fa.trace_enable(True)
    spans = []
    for _ in range(args.steps):
        flush.zero_()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        step()
        t1.record(stream)
        spans.append((t0, t1))
    torch.cuda.synchronize()
    barrier()
    fa.trace_enable(False)
    clocks = sampler.stop()
    if fa.device_status() != 0:
        raise RuntimeError("a kernel reported a bounded-wait timeout in the timed region")
    ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in spans) / args.steps, world, dev)
    value = world * fwd_f / (ms / 1e3) / 1e12
    traced = {kk: v for kk, v in fa.trace_read().items() if v[1] > 0}
    launches = sum(n for _, n in traced.values())
    k_ms = traced["fwd_fp8_kernel"][0] / traced["fwd_fp8_kernel"][1]
    peaks = load_peaks()
    peak8 = 2.0 * peaks["bf16_tflops"]          # fp8 dense rate = 2 x bf16 (4.5 vs 2.25 PF nominal)
    achieved = fwd_f / (k_ms / 1e3) / 1e12
    roofline = {"bound": "tensor", "kernel": "fwd_fp8_kernel", "achieved": achieved,
                "peak": peak8, "unit": "TFLOP/s", "frac": achieved / peak8,
                "traffic": traffic_from_profiles("fwd_fp8_kernel", args.workload),
                "peak_source": f"{peaks['source']} bf16 (burst) x 2, the nominal fp8/bf16 ratio",
                "algorithmic_work_per_launch": fwd_f, "avg_launch_ms": k_ms}
    e2e = None
    if not args.no_e2e:
        h_in = {n: x[n].pin_memory() for n in ("q8", "k8", "vt8")}
        dev_sets = [{"q8": q8, "k8": k8, "vt8": vt8, "o": o, "lse": lse},
                    {"q8": torch.empty_like(q8), "k8": torch.empty_like(k8),
                     "vt8": torch.empty_like(vt8), "o": torch.empty_like(o),
                     "lse": torch.empty_like(lse)}]
        h_out_sets = [{"o": torch.empty(o.shape, dtype=o.dtype).pin_memory(),
                       "lse": torch.empty(lse.shape, dtype=lse.dtype).pin_memory()}
                      for _ in range(2)]

        def compute(dset):
            fa.fwd_fp8(dset["q8"], dset["k8"], dset["vt8"], qs, ks, vs, causal=causal, scale=scale,
                       out=dset["o"], lse=dset["lse"])

        ke = max(1, min(args.steps, E2E_MAX_STEPS))
        pms, sms = e2e_measure(torch, h_in, dev_sets, h_out_sets, compute, ke, barrier)
        pms, sms = max_over_ranks(pms, world, dev), max_over_ranks(sms, world, dev)
        ems, mode, (other, oms) = e2e_pick(pms, sms)
        e2e = {"value": world * fwd_f / (ems / 1e3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": sum(t.numel() for t in h_in.values()),
               "d2h_bytes_per_step": o.numel() * 2 + lse.numel() * 4,
               "ms_per_step": ems, "steps": ke, "mode": mode,
               other: {"value": world * fwd_f / (oms / 1e3) / 1e12, "ms_per_step": oms}}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        fwd1, _ = attn_flops(1, 1, N, d, causal)
        heads, t_cpu = 0, 0.0
        q8c, k8c, v8c = (x[n].numpy().reshape(-1, N, d) for n in ("q8", "k8", "v8"))
        while heads < B * H and (heads == 0 or t_cpu < 10.0):
            hk = (heads // H) * Hkv + (heads % H) // (H // Hkv)
            t0c = time.perf_counter()
            oracle.fwd_fp8(q8c[heads][None, None], k8c[hk][None, None], v8c[hk][None, None],
                           qs, ks, vs, causal, scale)
            t_cpu += time.perf_counter() - t0c
            heads += 1
        cpu = {"value": heads * fwd1 / t_cpu / 1e12, "unit": "TFLOP/s",
               "cores": oracle.num_threads(), "kind": "oracle",
               "sample": f"{heads} of {B * H} (batch, head) pairs, full N={N}, forward, "
                         f"{t_cpu:.1f} s on host cores"}
    if rank == 0:
        out = {"metric": FP8_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
               "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
               "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
               "data": "synthetic",
               "config": {"workload": args.workload, "B": B, "H": H, "Hkv": Hkv, "N": N, "d": d,
                          "causal": causal, "output": "bf16",
                          "parallelism": f"replicas x{world}",
                          "l2": "inputs fit in L2 (96 MiB of E4M3 Q, K, V^T): "
                                f"{flush.numel() * 4 >> 20} MiB written between steps, "
                                "outside the timed spans"},
               "kernels_ms": {kk: v[0] / v[1] for kk, v in traced.items()},
               "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
               "gpu_launches": launches, "clocks": clocks}
        emit(out, args)


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    decode = args.workload in DECODE_WORKLOADS
    fp8 = args.workload in FP8_WORKLOADS
    if args.impl == "reference":
        (run_decode_reference if decode else run_fp8_reference if fp8 else run_reference)(
            args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        (run_decode if decode else run_fp8 if fp8 else run_ours)(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
