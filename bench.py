#!/usr/bin/env python
"""Benchmark of the block-sparse top-k GQA attention hot path on GB300.

One step = one pass of the prefill hot path over the 32K causal 'sink'
workload (B=1, Sq=Skv=32768, Hkv=4, qhead_per_kv=16, topk=16, D=128): k->q CSR
build + work plan, attention tiles, LSE combine, inputs resident in HBM.
The metric is effective TFLOP/s = 4 * D * sum over (query, head) of visible
keys / step time.  Reported alongside, each with its own roofline fraction:
the other prefill workloads (tiny non-causal 1K, 48K uniform with one KV
head, 384K sink with qhead_per_kv 2 in bf16 and with NVFP4 K/V) and the
paged-decode sweep (B=32, Sq=8, Hkv=4, qpk=16, topk=16, L = 1K..128K,
seqused = L-17) in GB/s of algorithmic bytes.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference]

Multi-GPU runs (torchrun) process one independent problem per rank (weak
scaling, no collective on the data path); rank 0 prints one JSON line.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import msa_synth as synth  # noqa: E402

METRIC = "sparse-attn fwd effective TFLOP/s & % bf16 peak; paged decode GB/s & % HBM"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# hist, column scan, row scan, scatter, tail fill, plan count, plan scan, plan
# write (plus one cudaMemset2DAsync of the row_ptr heads, not counted)
KERNELS_PER_CSR = 8
KERNELS_PER_PARTIAL = 1  # attention tiles
KERNELS_PER_COMBINE = 1  # LSE combine

# DRAM traffic (read + write bytes per launch) of the attention-tile kernel on
# the 32K causal sink workload from one single-pass ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum), keyed by the hash of the
# source it was measured on (stale -> reported as null).
PROFILED_TRAFFIC: dict = {
    "b5ee4a9835e4ca32": 1.101e10,  # 2.47 GB read + 8.54 GB written
    "b02f23509976d36b": 1.087e10,  # 2.33 GB read + 8.54 GB written
    "5b5733e4b8e18d14": 1.0749e10,  # 2.21 GB read + 8.54 GB written
    "7cb41653a1839e32": 1.0781e10,  # 2.24 GB read + 8.54 GB written
    "3b71fc819f216446": 1.0738e10,  # 2.20 GB read + 8.54 GB written
    "cc01a715c29fdf13": 1.0761e10,  # 2.22 GB read + 8.54 GB written
    "6f386edfcd051062": 1.0790e10,  # 2.25 GB read + 8.54 GB written
    "a80da73977f45668": 1.0778e10,  # 2.24 GB read + 8.54 GB written
    "362d894189bb3b67": 1.0715e10,  # 2.18 GB read + 8.54 GB written
    "c932c9210ba72cff": 1.0688e10,  # 2.15 GB read + 8.54 GB written
    "d7e317ae04c8bfe8": 1.0686e10,  # 2.15 GB read + 8.54 GB written
    "c328ed59c4f503f0": 1.0655e10,  # 2.12 GB read + 8.54 GB written
}


# ---------------------------------------------------------------------------
# workload arithmetic (measurement only)
# ---------------------------------------------------------------------------

def visible_keys(q2k: torch.Tensor, Sq: int, kv_len: torch.Tensor, causal: bool, blk: int = 128,
                 positions: torch.Tensor | None = None) -> torch.Tensor:
    """Visible keys per (b, h, s): union of the distinct valid blocks, below kv_len, causal limit."""
    B, Hkv, S, topk = q2k.shape
    kv = kv_len.to(torch.int64).view(B, 1, 1, 1)
    ids = q2k.to(torch.int64)
    nvalid = (kv + blk - 1) // blk
    valid = (ids >= 0) & (ids < nvalid)
    srt, _ = torch.sort(torch.where(valid, ids, torch.full_like(ids, -1)), dim=-1)
    dup = torch.zeros_like(valid)
    dup[..., 1:] = srt[..., 1:] == srt[..., :-1]
    keep = (srt >= 0) & ~dup
    s = torch.arange(S, dtype=torch.int64, device=q2k.device).view(1, 1, S, 1) if positions is None \
        else positions.to(torch.int64).view(1, 1, S, 1)
    limit = kv - 1
    if causal:
        limit = torch.minimum(limit, s + (kv - Sq))
    n = torch.clamp(limit - srt * blk + 1, 0, blk)
    return torch.where(keep, n, torch.zeros_like(n)).sum(-1)


def prefill_flops(spec: synth.PrefillSpec, q2k: torch.Tensor) -> float:
    kv = torch.full((spec.B,), spec.Skv, dtype=torch.int64, device=q2k.device)
    vis = visible_keys(q2k, spec.Sq, kv, spec.causal)
    return 4.0 * spec.D * spec.qpk * float(vis.sum())


def decode_bytes(spec: synth.DecodeSpec, q2k: torch.Tensor, seqused: torch.Tensor) -> float:
    """Unique K+V bytes of the union of selected blocks per (b, h), tokens < seqused, plus
    Q, O, LSE, q2k and the page-table entries of the union."""
    B, Hkv, Sq, topk = q2k.shape
    ids = q2k.to(torch.int64).cpu()
    su = seqused.to(torch.int64).cpu()
    kv_bytes = 0
    entries = 0
    for b in range(B):
        nvalid = (int(su[b]) + 127) // 128
        for h in range(Hkv):
            blocks = {int(j) for j in ids[b, h].flatten().tolist() if 0 <= j < nvalid}
            entries += len(blocks)
            for j in blocks:
                kv_bytes += min(128, int(su[b]) - 128 * j) * spec.D * 2 * 2
    q_o = 2 * B * Sq * spec.Hq * spec.D * 2
    return float(kv_bytes + q_o + B * Sq * spec.Hq * 4 + q2k.numel() * 4 + entries * 4)


def decode_gathered_bytes(spec: synth.DecodeSpec, q2k: torch.Tensor, seqused: torch.Tensor) -> float:
    """K+V bytes a per-query gather would read (no dedup across the queries of a
    (b, h)): each query's distinct valid blocks, tokens < seqused."""
    B, Hkv, Sq, topk = q2k.shape
    ids = q2k.to(torch.int64).cpu()
    su = seqused.to(torch.int64).cpu()
    tokens = 0
    for b in range(B):
        nvalid = (int(su[b]) + 127) // 128
        for h in range(Hkv):
            for s in range(Sq):
                for j in {int(j) for j in ids[b, h, s].tolist() if 0 <= j < nvalid}:
                    tokens += min(128, int(su[b]) - 128 * j)
    return float(tokens * spec.D * 2 * 2)


# ---------------------------------------------------------------------------
# environment helpers
# ---------------------------------------------------------------------------

def load_peaks() -> tuple[dict, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle sampling during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        power = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(power) if power else None}


def source_hash(*names) -> str:
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "block_sparse_top_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def workload_config(spec: synth.PrefillSpec) -> dict:
    """The JSON `config` of a prefill workload (both arms print the same one)."""
    q_mib = spec.B * spec.Sq * spec.Hq * spec.D * 2 / 2 ** 20
    part_gb = spec.B * spec.Sq * spec.topk * spec.Hq * (spec.D * 2 + 8) / 1e9
    return {"workload": spec.name, "B": spec.B, "Sq": spec.Sq, "Skv": spec.Skv, "Hkv": spec.Hkv,
            "qhead_per_kv": spec.qpk, "topk": spec.topk, "D": spec.D, "blk_kv": 128, "causal": spec.causal,
            "pattern": spec.pattern, "kv_format": spec.kv_format, "per_rank_problem": "independent (seed + rank)",
            "l2": f"inputs larger than L2 (Q {q_mib:.0f} MiB; split partials {part_gb:.1f} GB per step); "
                  "no flush"}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------------------
# CPU oracle baseline
# ---------------------------------------------------------------------------

def oracle_rate(spec: synth.PrefillSpec, x_cpu: dict, budget_s: float, seed: int = 7) -> dict:
    """Times the float64 oracle on a sample of query rows; returns effective TFLOP/s."""
    import oracle
    total_q = spec.B * spec.Sq
    kv = torch.full((spec.B,), spec.Skv, dtype=torch.int64)

    def rows_flops(rows):
        r = torch.tensor(rows, dtype=torch.int64)
        b, s = r // spec.Sq, r % spec.Sq
        sub = x_cpu["q2k"][b, :, s, :].permute(1, 0, 2).unsqueeze(0)  # [1,Hkv,n,topk]
        vis = visible_keys(sub, spec.Sq, kv[:1], spec.causal, positions=s)
        return 4.0 * spec.D * spec.qpk * float(vis.sum())

    n = 16
    while True:
        rows = synth.sample_query_rows(total_q, n, seed=seed)
        t0 = time.perf_counter()
        _, _, threads = oracle.sparse_attn(x_cpu["q"], x_cpu["k"], x_cpu["v"], x_cpu["q2k"], causal=spec.causal,
                                           rows=rows, return_threads=True)
        dt = time.perf_counter() - t0
        if dt >= budget_s or n >= total_q:
            break
        n = min(total_q, max(n * 2, int(n * budget_s / max(dt, 1e-3) * 1.05)))
    fl = rows_flops(rows)
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "cpu_model": cpu_model(),
            "kind": "oracle",
            "sample": f"{len(rows)} of {total_q} query rows (all {spec.Hq} heads), float64, {dt:.1f} s"}


# ---------------------------------------------------------------------------
# main GPU benchmark
# ---------------------------------------------------------------------------

WORKLOADS = {
    "causal_sink_32k": synth.CAUSAL_SINK_32K,
    # smaller case of the same kernel for ncu captures (partials ~1.1 GB on the device)
    "causal_sink_16k_1kv": synth.PrefillSpec("causal_sink_16k_1kv", B=1, Sq=16384, Skv=16384, Hkv=1, qpk=16,
                                             topk=16, causal=True, pattern="sink"),
    # smaller case of the NVFP4 instance (qhead_per_kv 2, as the 384K NVFP4 workload) for ncu captures
    "causal_sink_64k_qpk2_nvfp4": synth.PrefillSpec("causal_sink_64k_qpk2_nvfp4", B=1, Sq=65536, Skv=65536, Hkv=1,
                                                    qpk=2, topk=16, causal=True, pattern="sink", kv_format="nvfp4"),
}


def run_ours(args, world, rank):
    import block_sparse_top_gb300 as msa

    dev = torch.device("cuda", torch.cuda.current_device())
    spec = WORKLOADS[args.workload]
    spec_r = synth.PrefillSpec(**{**spec.__dict__, "seed": spec.seed + rank})
    x = synth.make_prefill_inputs(spec_r, device=dev)
    flops = prefill_flops(spec_r, x["q2k"])
    kvkw = {}
    kv_bf16 = {"k": x["k"], "v": x["v"]}  # the oracle's timing sample runs on bf16 K/V
    if spec.kv_format == "nvfp4":
        # NVFP4 workloads: K/V (and their scales) stored as the library's encoder writes them
        x["k"], x["k_scales"] = msa.nvfp4_quantize(x["k"])
        x["v"], x["v_scales"] = msa.nvfp4_quantize(x["v"])
        kvkw = {"kv_format": "nvfp4"}
    nominal = 4.0 * spec.D * spec.Hq * spec.Sq * spec.B * spec.topk * 128
    csr, csr_ws = msa.csr_buffers(spec.B, spec.Hkv, spec.Sq, spec.Skv, spec.topk, spec.qpk, dev)
    fwd_ws = msa.fwd_workspace(spec.B, spec.Sq, spec.Hq, spec.topk, dev)
    out = torch.empty_like(x["q"])
    lse = torch.empty((spec.B, spec.Sq, spec.Hq), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        msa.build_k2q_csr(x["q2k"], spec.Skv, spec.qpk, out=csr, workspace=csr_ws)
        if ev is not None:
            ev[1].record(stream)
        msa.sparse_attn_fwd_partial(x["q"], x["k"], x["v"], csr, causal=True, workspace=fwd_ws,
                                    k_scales=x.get("k_scales"), v_scales=x.get("v_scales"), **kvkw)
        if ev is not None:
            ev[2].record(stream)
        msa.sparse_attn_combine(csr, spec.Hq, out, lse, fwd_ws)
        if ev is not None:
            ev[3].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(dev.index)
    barrier(world)
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)  # let the sampler take its first reading
    start.record(stream)
    for i in range(K):
        step(evs[i])
    stop.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    barrier(world)
    total_ms = start.elapsed_time(stop)
    csr_ms = sum(e[0].elapsed_time(e[1]) for e in evs) / K
    attn_ms = sum(e[1].elapsed_time(e[2]) for e in evs) / K
    comb_ms = sum(e[2].elapsed_time(e[3]) for e in evs) / K
    step_ms = total_ms / K
    step_ms_max = reduce_max(step_ms, world)
    flops_all = reduce_sum(flops, world)
    value = flops_all / (step_ms_max * 1e-3) / 1e12

    # End to end through the public API with host buffers: every step uploads
    # its inputs from pinned host memory, runs the CSR build and the forward,
    # and downloads O and LSE.  Steps are software-pipelined on three streams
    # (upload, compute, download) with double-buffered device inputs and
    # outputs, so step i+1's upload and step i-1's download overlap step i's
    # compute; every step's copies are inside the timed region.
    host = {k_: v_.cpu().pin_memory() for k_, v_ in x.items()}
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    lse_h = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    dev_in = [{k_: torch.empty_like(v_) for k_, v_ in x.items()} for _ in range(2)]
    dev_out = [(torch.empty_like(out), torch.empty_like(lse)) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_h.numel() * 2 + lse_h.numel() * 4
    up, comp, down = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_up = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_down = [torch.cuda.Event() for _ in range(2)]

    def e2e_step(i):
        s = i % 2
        up.wait_event(ev_comp[s])  # step i-2 has finished reading input buffer s
        with torch.cuda.stream(up):
            for k_ in host:
                dev_in[s][k_].copy_(host[k_], non_blocking=True)
            ev_up[s].record(up)
        comp.wait_event(ev_up[s])
        comp.wait_event(ev_down[s])  # step i-2's outputs in buffer s are downloaded
        with torch.cuda.stream(comp):
            msa.build_k2q_csr(dev_in[s]["q2k"], spec.Skv, spec.qpk, out=csr, workspace=csr_ws)
            msa.sparse_attn_fwd(dev_in[s]["q"], dev_in[s]["k"], dev_in[s]["v"], csr, causal=True, out=dev_out[s][0],
                                lse=dev_out[s][1], workspace=fwd_ws, k_scales=dev_in[s].get("k_scales"),
                                v_scales=dev_in[s].get("v_scales"), **kvkw)
            ev_comp[s].record(comp)
        down.wait_event(ev_comp[s])
        with torch.cuda.stream(down):
            out_h.copy_(dev_out[s][0], non_blocking=True)
            lse_h.copy_(dev_out[s][1], non_blocking=True)
            ev_down[s].record(down)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    Ke = max(3, min(K, 20))
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(up)
    for i in range(Ke):
        e2e_step(i)
    stream.wait_stream(down)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = reduce_max(e0.elapsed_time(e1) / Ke, world)
    e2e_val = flops_all / (e2e_ms * 1e-3) / 1e12

    peaks, peak_src = load_peaks()
    long_region = total_ms > 2000
    peak = peaks["bf16_tflops_sustained"] if long_region else peaks["bf16_tflops"]
    achieved = flops / (attn_ms * 1e-3) / 1e12
    khash = source_hash("attn.cu", "attn_tc.cuh", "attn_mma.cuh", "tc.cuh", "common.cuh", "combine.cuh")
    traffic = PROFILED_TRAFFIC.get(khash)
    result = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(step_ms_max, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(spec),
        "breakdown_ms": {"csr_build_and_plan": round(csr_ms, 4), "attention_tiles": round(attn_ms, 4),
                         "lse_combine": round(comb_ms, 4)},
        "effective_flop_per_step": flops, "nominal_tflops": round(nominal / (step_ms_max * 1e-3) / 1e12, 3),
        "clocks": clocks,
        "e2e": {"value": round(e2e_val, 3), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
                "pipelining": "upload of step i+1 and download of step i-1 overlap step i (three streams, "
                              "double-buffered device inputs and outputs)"},
        "gpu_launches": K * (KERNELS_PER_CSR + KERNELS_PER_PARTIAL + KERNELS_PER_COMBINE),
        "roofline": {"bound": "tensor", "kernel": "attention tiles (msa_sparse_attn_fwd_partial)",
                     "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "peak_source": f"{peak_src} bf16 {'sustained' if long_region else 'burst'}",
                     "kernel_source_hash": khash},
    }
    x_cpu = {k_: v_.cpu() for k_, v_ in {**x, **kv_bf16}.items() if k_ in ("q", "k", "v", "q2k")}
    del x, csr, csr_ws, fwd_ws, out, lse, host, out_h, lse_h, dev_in, dev_out
    torch.cuda.empty_cache()
    if not args.no_configs:
        result["configs"] = {c.name: measure_config(c, dev, args.config_steps, args.warmup, peaks, peak_src)
                             for c in OTHER_CONFIGS}
    if not args.no_decode:
        result["decode"] = decode_sweep(args, dev, peaks, peak_src)
    if not args.no_variants:
        result["variants"] = measure_variants(dev, args.config_steps, args.warmup, peaks, peak_src)
    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = oracle_rate(spec, x_cpu, args.cpu_budget)
    return result


OTHER_CONFIGS = [synth.TINY_NONCAUSAL_1K, synth.CAUSAL_UNIFORM_48K, synth.CAUSAL_SINK_384K,
                 synth.CAUSAL_SINK_384K_NVFP4]


def measure_config(spec, dev, steps, warmup, peaks, peak_src):
    """One prefill workload: CSR + plan, tiles and combine timed per step with
    CUDA events; effective TFLOP/s of the step and of the tile kernel alone.
    Workloads whose inputs and partials fit in L2 get an L2 flush (a 256 MiB
    write) before every step, outside the events."""
    import block_sparse_top_gb300 as msa
    x = synth.make_prefill_inputs(spec, device=dev)
    flops = prefill_flops(spec, x["q2k"])
    k, v, kw = x["k"], x["v"], {}
    if spec.kv_format == "nvfp4":
        k, ks = msa.nvfp4_quantize(x["k"])
        v, vs = msa.nvfp4_quantize(x["v"])
        kw = {"kv_format": "nvfp4", "k_scales": ks, "v_scales": vs}
    csr, csr_ws = msa.csr_buffers(spec.B, spec.Hkv, spec.Sq, spec.Skv, spec.topk, spec.qpk, dev)
    fwd_ws = msa.fwd_workspace(spec.B, spec.Sq, spec.Hq, spec.topk, dev)
    out = torch.empty_like(x["q"])
    lse = torch.empty((spec.B, spec.Sq, spec.Hq), dtype=torch.float32, device=dev)
    small = x["q"].numel() * 2 + fwd_ws.numel() < 256 * 2 ** 20
    flush = torch.empty(256 * 2 ** 20, dtype=torch.uint8, device=dev) if small else None
    stream = torch.cuda.current_stream()

    def step(ev=None):
        if flush is not None:
            flush.fill_(1)
        if ev is not None:
            ev[0].record(stream)
        msa.build_k2q_csr(x["q2k"], spec.Skv, spec.qpk, out=csr, workspace=csr_ws)
        if ev is not None:
            ev[1].record(stream)
        msa.sparse_attn_fwd_partial(x["q"], k, v, csr, causal=spec.causal, workspace=fwd_ws, **kw)
        if ev is not None:
            ev[2].record(stream)
        msa.sparse_attn_combine(csr, spec.Hq, out, lse, fwd_ws)
        if ev is not None:
            ev[3].record(stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    for i in range(steps):
        step(evs[i])
    torch.cuda.synchronize()
    csr_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    attn_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    comb_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in evs)
    step_ms = statistics.mean(e[0].elapsed_time(e[3]) for e in evs)
    peak = peaks["bf16_tflops"]
    tiles = flops / (attn_ms * 1e-3) / 1e12
    res = {"config": {**workload_config(spec), "kv_format": spec.kv_format,
                      "l2": "L2 flushed (256 MiB write) before every step, outside the events" if small
                      else workload_config(spec)["l2"]},
           "effective_flop_per_step": flops, "steps": steps, "ms_per_step": round(step_ms, 4),
           "TFLOP/s": round(flops / (step_ms * 1e-3) / 1e12, 3),
           "breakdown_ms": {"csr_build_and_plan": round(csr_ms, 4), "attention_tiles": round(attn_ms, 4),
                            "lse_combine": round(comb_ms, 4)},
           "roofline": {"bound": "tensor", "kernel": "attention tiles", "achieved": round(tiles, 2), "peak": peak,
                        "unit": "TFLOP/s", "frac": round(tiles / peak, 4),
                        "peak_source": f"{peak_src} bf16 burst"},
           "step_frac_of_peak": round(flops / (step_ms * 1e-3) / 1e12 / peak, 4)}
    del x, k, v, csr, csr_ws, fwd_ws, out, lse, flush
    torch.cuda.empty_cache()
    return res


RAGGED_32K = synth.VarlenSpec("ragged_sink_32k", q_lens=(16384, 8192, 4096, 4096), k_lens=(16384, 8192, 4096, 4096),
                              Hkv=4, qpk=16, topk=16, causal=True, pattern="sink")


def measure_variants(dev, steps, warmup, peaks, peak_src):
    """The other forward paths on the 32K causal sink workload (the same
    inputs, so the same effective FLOP): ragged-batch entry point, e4m3 K/V,
    e4m3 Q and K, fp16 / fp32 partials, temperature LSE; plus a ragged batch of
    four sequences and the dense paged decode.  Each step is the CSR build and
    one forward call, timed with CUDA events over `steps` back-to-back steps
    (outputs of the ragged entry point come from PyTorch's caching allocator
    inside the timed region; the CSR row count is passed in, as a caller that
    knows its batch would, so no call reads cu_seqlens back)."""
    import block_sparse_top_gb300 as msa
    spec = synth.CAUSAL_SINK_32K
    x = synth.make_prefill_inputs(spec, device=dev)
    flops = prefill_flops(spec, x["q2k"])
    peak = peaks["bf16_tflops"]
    B, Sq, Hq, D = x["q"].shape
    Skv, Hkv, qpk = spec.Skv, spec.Hkv, spec.qpk
    q_v, k_v, v_v = x["q"].view(B * Sq, Hq, D), x["k"].view(B * Skv, Hkv, D), x["v"].view(B * Skv, Hkv, D)
    q2k_v = x["q2k"][0].contiguous()  # [Hkv, Sq, topk]: one sequence
    cu_q = torch.tensor([0, Sq], dtype=torch.int32, device=dev)
    cu_k = torch.tensor([0, Skv], dtype=torch.int32, device=dev)
    k8 = k_v.float().to(torch.float8_e4m3fn).view(torch.uint8).contiguous()
    v8 = v_v.float().to(torch.float8_e4m3fn).view(torch.uint8).contiguous()
    q8 = q_v.float().to(torch.float8_e4m3fn).contiguous()
    csr, csr_ws = msa.csr_buffers(B, Hkv, Sq, Skv, spec.topk, qpk, dev)
    fwd_ws = msa.fwd_workspace(B, Sq, Hq, spec.topk, dev)
    out = torch.empty_like(x["q"])
    lse = torch.empty((B, Sq, Hq), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def time_steps(fn):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    rows_1 = (Skv + 127) // 128  # the row count, known on the host (no read-back of cu_seqlens per call)

    def varlen(q, k, v, **kw):
        c = msa.build_k2q_csr_varlen(q2k_v, cu_q, cu_k, Sq, Skv, qpk, total_rows=rows_1)
        msa.sparse_attn_fwd_varlen(q, k, v, c, causal=True, **kw)

    def uniform_fp8():
        msa.build_k2q_csr(x["q2k"], Skv, qpk, out=csr, workspace=csr_ws)
        msa.sparse_attn_fwd(x["q"], k8.view(B, Skv, Hkv, D), v8.view(B, Skv, Hkv, D), csr, causal=True,
                            kv_format="fp8", workspace=fwd_ws, out=out, lse=lse)

    res = {"workload": "causal_sink_32k (C2) unless named otherwise", "steps": steps, "warmup": warmup,
           "peak": peak, "peak_source": f"{peak_src} bf16 burst"}

    def rec(name, ms, fl=flops, note=None):
        tf = fl / (ms * 1e-3) / 1e12
        res[name] = {"ms_per_step": round(ms, 4), "TFLOP/s": round(tf, 3), "step_frac_of_peak": round(tf / peak, 4)}
        if note:
            res[name]["path"] = note

    rec("varlen_entry_bf16", time_steps(lambda: varlen(q_v, k_v, v_v)), note="msa_build_k2q_csr_varlen + msa_sparse_attn_fwd_varlen, one sequence")
    rec("e4m3_kv", time_steps(uniform_fp8), note="K/V as e4m3 bytes, staged to bf16 in the tile kernel")
    rec("e4m3_qk", time_steps(lambda: varlen(q8, k8, v8, kv_format="fp8")), note="S = Q K^T as an e4m3 MMA, PV in bf16")
    rec("partials_fp16", time_steps(lambda: varlen(q_v, k_v, v_v, partial_dtype=msa.MSA_PARTIAL_FP16)))
    rec("partials_fp32", time_steps(lambda: varlen(q_v, k_v, v_v, partial_dtype=msa.MSA_PARTIAL_FP32)))
    rec("temperature_lse", time_steps(lambda: varlen(q_v, k_v, v_v, lse_temperature_scale=2.0)), note="lse_temperature_scale 2")
    del x, q_v, k_v, v_v, k8, v8, q8, csr, csr_ws, fwd_ws, out, lse
    torch.cuda.empty_cache()
    # a ragged batch: four causal sink sequences, 32K queries in all
    r = RAGGED_32K
    xr = synth.make_varlen_inputs(r, device=dev)
    fl_r, q0 = 0.0, 0
    for n_q, n_k in zip(r.q_lens, r.k_lens):
        q2k_s = xr["q2k"][:, q0:q0 + n_q].unsqueeze(0)
        vis = visible_keys(q2k_s, n_q, torch.tensor([n_k], device=dev), r.causal)
        fl_r += 4.0 * r.D * r.qpk * float(vis.sum())
        q0 += n_q

    rows_r = sum((n + 127) // 128 for n in r.k_lens)

    def ragged():
        c = msa.build_k2q_csr_varlen(xr["q2k"], xr["cu_seqlens_q"], xr["cu_seqlens_k"], max(r.q_lens), max(r.k_lens),
                                     r.qpk, total_rows=rows_r)
        msa.sparse_attn_fwd_varlen(xr["q"], xr["k"], xr["v"], c, causal=True)

    rec("ragged_sink_32k", time_steps(ragged), fl=fl_r,
        note=f"{r.B} sequences of {'/'.join(str(n) for n in r.q_lens)} queries and keys, Hkv {r.Hkv}, qhead_per_kv {r.qpk}, topk {r.topk}")
    del xr
    torch.cuda.empty_cache()
    # the dense paged decode (no selection: every block of each sequence)
    ds = synth.paged_decode_spec(32768)
    d = synth.make_decode_inputs(ds, device=dev)
    su = d["seqused"].to(torch.int64).cpu()
    kv_bytes = sum(int(su[b]) * ds.Hkv * ds.D * 2 * 2 for b in range(ds.B))
    dbytes = float(kv_bytes + 2 * ds.B * ds.Sq * ds.Hq * ds.D * 2 + ds.B * ds.Sq * ds.Hq * 4)
    ms_d = time_steps(lambda: msa.paged_attn_fwd(d["q"], d["k_pool"], d["v_pool"], d["page_table"], d["seqused"], None))
    gbs = dbytes / (ms_d * 1e-3) / 1e9
    res["dense_decode_32k"] = {"us_per_call": round(ms_d * 1e3, 2), "GB/s": round(gbs, 1),
                               "frac_hbm": round(gbs / peaks["hbm_gbs"], 4), "bytes": dbytes,
                               "path": "msa_paged_attn_fwd with q2k NULL: B 32, Sq 8, Hkv 4, qhead_per_kv 16, 32K keys"}
    del d
    torch.cuda.empty_cache()
    return res


def decode_kernels_per_call(spec) -> int:
    """Kernels one paged-decode call launches, as the library reports it for
    this shape on the current device (1: the decode kernel plans each group
    itself; 2: plan kernel + decode)."""
    import block_sparse_top_gb300 as msa
    return msa.paged_fwd_launches(spec.B, spec.Sq, spec.Hq, spec.Hkv, spec.topk, spec.pages_per_seq)


def decode_sweep(args, dev, peaks, peak_src):
    """Paged decode GB/s per KV length.

    Calls are captured back to back in a CUDA graph (so host launch overhead
    is not timed), cycling through enough independent input sets that the
    data one call touches (>= 600 MB per cycle) is not left in L2 by the
    previous call on the same set.
    """
    import block_sparse_top_gb300 as msa
    out = []
    for L in args.decode_L:
        spec = synth.paged_decode_spec(L)
        first = synth.make_decode_inputs(spec, device=dev)
        nbytes = decode_bytes(spec, first["q2k"], first["seqused"])
        gathered = decode_gathered_bytes(spec, first["q2k"], first["seqused"])
        nsets = max(1, math.ceil(600e6 / nbytes))
        sets = [first] + [synth.make_decode_inputs(
            synth.DecodeSpec(**{**spec.__dict__, "seed": spec.seed + 1000 + i}), device=dev) for i in range(1, nsets)]
        outs = [(torch.empty_like(d["q"]), torch.empty(d["q"].shape[:2], dtype=torch.float32, device=dev))
                for d in sets]
        ws = msa.paged_workspace(spec.B, spec.Sq, spec.Hq, spec.Hkv, spec.topk, spec.pages_per_seq, dev)

        def call(i):
            d, (o, lse) = sets[i % nsets], outs[i % nsets]
            msa.sparse_attn_paged_fwd(d["q"], d["k_pool"], d["v_pool"], d["page_table"], d["seqused"], d["q2k"],
                                      out=o, lse=lse, workspace=ws)

        n_calls = max(nsets, 24)
        for i in range(nsets):
            call(i)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph):
                for i in range(n_calls):
                    call(i)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        reps = 3
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            graph.replay()
        b.record()
        torch.cuda.synchronize()
        us = a.elapsed_time(b) * 1e3 / (reps * n_calls)
        gbs = nbytes / (us * 1e-6) / 1e9
        out.append({"L": L, "us": round(us, 2), "GB/s": round(gbs, 1), "frac_hbm": round(gbs / peaks["hbm_gbs"], 4),
                    "bytes": nbytes, "gathered_kv_bytes_no_dedup": gathered, "input_sets": nsets,
                    "kernels": decode_kernels_per_call(spec)})
        del sets, outs, first, graph
        torch.cuda.empty_cache()
    return {"unit": "GB/s", "peak_gbs": peaks["hbm_gbs"], "peak_source": peak_src,
            "timing": "CUDA-graph replay of back-to-back calls cycling input sets (>= 600 MB per cycle)",
            "kernels_per_call": "per L in the sweep (1: each CTA plans its own group; 2: plan kernel + decode)",
            "sweep": out}


# ---------------------------------------------------------------------------
# reference arm: the float64 oracle on the host cores
# ---------------------------------------------------------------------------

def run_reference(args, world, rank):
    spec = WORKLOADS[args.workload]  # the same workload as the library's arm
    x_cpu = synth.make_prefill_inputs(spec, device="cuda" if torch.cuda.is_available() else "cpu")
    x_cpu = {k_: v_.cpu() for k_, v_ in x_cpu.items()}
    per_step = max(0.2, args.ref_budget / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_rate(spec, x_cpu, per_step)
    vals = []
    last = None
    t0 = time.perf_counter()
    for i in range(args.steps):
        last = oracle_rate(spec, x_cpu, per_step, seed=100 + i)
        vals.append(last["value"])
    wall = time.perf_counter() - t0
    value = statistics.mean(vals)
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(wall / args.steps * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(spec),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": last["cores"], "cpu_model": last["cpu_model"],
                         "kind": "oracle", "sample": f"per step: {last['sample']}"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="causal_sink_32k", choices=sorted(WORKLOADS))
    ap.add_argument("--decode-L", type=int, nargs="*", default=list(synth.DECODE_SWEEP_L))
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the other prefill workloads")
    ap.add_argument("--no-variants", action="store_true",
                    help="skip the other forward paths (ragged batches, e4m3, partial types, temperature LSE, dense decode)")
    ap.add_argument("--decode-only", action="store_true",
                    help="run only the paged-decode sweep (for profiling its kernels); prints its JSON")
    ap.add_argument("--config-steps", type=int, default=10)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--ref-budget", type=float, default=150.0, help="seconds for the whole reference arm")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    world, rank, _ = dist_setup()
    if args.impl == "reference":
        if rank != 0:
            return
        res = run_reference(args, world, rank)
        print(json.dumps(res), flush=True)
        return
    if args.decode_only:
        dev = torch.device("cuda", torch.cuda.current_device())
        peaks, peak_src = load_peaks()
        if rank == 0:
            print(json.dumps({"decode": decode_sweep(args, dev, peaks, peak_src)}), flush=True)
        return
    res = run_ours(args, world, rank)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
