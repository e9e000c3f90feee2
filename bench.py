#!/usr/bin/env python3
"""Benchmark of the LTX-2.5 Stage-2 attention hot path on GB300.

One step = the attention of one Stage-2 transformer block on synthetic data:
  1. Sol-Attn routing of the 65664-token video+audio sequence (pool + route),
  2. block-sparse self-attention with the Taylor term (H=32, d=128, block 128, beta=1),
  3. audio->video cross attention: 128 audio queries against 65536 video keys
     as 8 split-KV partial answers,
  4. the exact log-sum-exp merge of those partials.
Metric: executed attention TFLOP/s of the whole step (dense-equivalent
TFLOP/s and the fraction of the measured bf16 tensor peak are reported too).

Usage: python bench.py [--gpus N --steps K --warmup W] [--impl reference]
Under torchrun every rank runs its own copy of the step (weak scaling, no
data-path collective); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from workloads import LINEAR_WORKLOADS, WORKLOADS, Workload, make_linear, make_qkv, to_f64  # noqa: E402

METRIC = "attention TFLOP/s (executed & dense-equiv) and % bf16 tensor peak, S=64K, d=128"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
CROSS_N_SPLIT = 8
CROSS_SKV = 65536
CROSS_SQ = 128


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_fingerprint() -> str:
    """Hash of the profiled kernels' source with comments and layout removed, so that counters
    taken on a kernel stay attached to it across edits of its comments only."""
    h = hashlib.sha256()
    for name in ("attn_fwd.cuh", "ptx.cuh", "attn_fwd_d128.cu", "na_persist.cuh"):
        with open(os.path.join(ROOT, "video_diffusion_transformer_block_gb300", "csrc", name)) as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def profiled_counters(workload: str):
    """Per-launch DRAM bytes and tensor-pipe activity of a workload's dominant kernel (sparse64k:
    the sparse forward; na3d: the neighbourhood kernel) from the committed ncu summary, if they
    were taken on the current kernel source (else None for both)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None, None
    with open(path) as f:
        t = json.load(f)
    ent = t.get(workload)
    if not ent or ent.get("kernel_fingerprint") != kernel_fingerprint():
        return None, None
    return ent.get("dram_bytes_per_launch"), ent.get("tensor_pipe_active_pct")


def cpu_model() -> str:
    """The host CPU's model name (lscpu), with the machine architecture."""
    import platform
    name = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.lower().startswith("model name"):
                name = ln.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    return f"{name or 'unknown'} ({platform.machine()})"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.15)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": smax, "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def executed_sparse_flops(sel_idx: torch.Tensor, sel_cnt: torch.Tensor, S: int, block: int, d: int) -> float:
    """sum over (b, h, query block i, selected j) of 4 * m_i * n_j * d."""
    idx = sel_idx.cpu().numpy()
    cnt = sel_cnt.cpu().numpy()
    nb = idx.shape[-1]
    sizes = np.array([min(block, S - j * block) for j in range(nb)], dtype=np.float64)
    total = 0.0
    flat_idx = idx.reshape(-1, nb)
    flat_cnt = cnt.reshape(-1)
    for r in range(flat_cnt.size):
        i = r % nb
        keys = sizes[flat_idx[r, :flat_cnt[r]]].sum()
        total += sizes[i] * keys
    return 4.0 * d * total


# ============================================================ native arm

def make_inputs(rank: int, beta: float, heads: int):
    w = WORKLOADS["sparse64k"]
    wr = Workload(w.name, B=w.B, H=heads, Sq=w.Sq, Skv=w.Skv, d=w.d, seed=w.seed + 1000 * rank, q_std=w.q_std,
                  k_std=w.k_std, grid=w.grid, audio_per_frame=w.audio_per_frame, pe=True, block=w.block, beta=beta)
    q, k, v = make_qkv(wr, device="cuda")
    wc = Workload("cross_stage2", B=1, H=heads, Sq=CROSS_SQ, Skv=CROSS_SKV, d=w.d, seed=3 + 1000 * rank)
    qa, kx, vx = make_qkv(wc, device="cuda")
    return wr, (q, k, v), (qa, kx, vx)


def run_native(args, world, rank, local):
    import video_diffusion_transformer_block_gb300 as vd
    from video_diffusion_transformer_block_gb300 import build as vbuild

    vbuild.build()
    vd.load_library()
    peaks, peaks_src = load_peaks()
    w, (q, k, v), (qa, kx, vx) = make_inputs(rank, args.beta, args.heads)
    B, H, S, d, block = w.B, w.H, w.Sq, w.d, w.block
    dev = q.device
    ws = torch.empty(vd.attn_sparse_workspace_bytes(B, H, S, d, block, block), dtype=torch.uint8, device=dev)
    rt = vd.sparse_route_buffers(B, H, S, d, block, dev, order=True)
    out = torch.empty_like(q)
    lse = torch.empty((B, H, S), dtype=torch.float32, device=dev)
    op = torch.empty((CROSS_N_SPLIT, B, H, CROSS_SQ, d), dtype=torch.float32, device=dev)
    lp = torch.empty((CROSS_N_SPLIT, B, H, CROSS_SQ), dtype=torch.float32, device=dev)
    oa = torch.empty((B, H, CROSS_SQ, d), dtype=torch.bfloat16, device=dev)
    la = torch.empty((B, H, CROSS_SQ), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    # the audio->video cross attention needs none of the self-attention's results: it runs on a
    # second stream, beside pool/route (HBM- and shared-memory-bound) and the sparse forward
    xstream = stream if args.serial_cross else torch.cuda.Stream()
    # pool, routing (the tensor-core tiles and, for 513 query blocks a head, the last block's
    # tail kernel), the query-block order, sparse forward, split-KV forward, merge
    kernels_per_step = 7

    def step(ev=None, xev=None):
        start = ev[0] if ev is not None else torch.cuda.Event()
        start.record(stream)
        if xstream is not stream:
            xstream.wait_event(start)
        with torch.cuda.stream(xstream):
            if xev is not None:
                xev[0].record(xstream)
            vd.attn_cross_splitkv_fwd(qa, kx, vx, CROSS_N_SPLIT, out_part=op, lse_part=lp, stream=xstream)
            vd.attn_lse_merge(op, lp, out=oa, lse=la, stream=xstream)
            xdone = xev[1] if xev is not None else torch.cuda.Event()
            xdone.record(xstream)
        vd.attn_sparse_route(q, k, v, args.beta, block=block, route=rt, workspace=ws)
        if ev is not None:
            ev[1].record(stream)
        vd.attn_sparse_fwd(q, k, v, rt, block=block, out=out, lse=lse)
        if ev is not None:
            ev[2].record(stream)
        stream.wait_event(xdone)
        if ev is not None:
            ev[3].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    status = vd.attn_last_device_status()
    if status != 0:
        raise RuntimeError(f"device status after warm-up: {vd.attn_status_string(status)}")
    sparse_flops = executed_sparse_flops(rt["sel_idx"], rt["sel_cnt"], S, block, d)
    dense_eq = 4.0 * B * H * S * S * d
    cross_flops = 4.0 * B * H * CROSS_SQ * CROSS_SKV * d
    density = sparse_flops / dense_eq

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    xevs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        for i in range(args.steps):
            step(evs[i], xevs[i])
        torch.cuda.synchronize()
    barrier(world)
    status = vd.attn_last_device_status()
    if status != 0:
        raise RuntimeError(f"device status after timed region: {vd.attn_status_string(status)}")
    total_ms = evs[0][0].elapsed_time(evs[-1][3])
    route_ms = sum(e[0].elapsed_time(e[1]) for e in evs) / args.steps
    fwd_ms = sum(e[1].elapsed_time(e[2]) for e in evs) / args.steps
    cross_ms = sum(e[0].elapsed_time(e[1]) for e in xevs) / args.steps
    total_ms = max_over_ranks(total_ms, world)
    ms_per_step = total_ms / args.steps
    step_flops = sparse_flops + cross_flops
    value = world * step_flops * args.steps / (total_ms * 1e-3) / 1e12
    dense_equiv = world * (dense_eq + cross_flops) * args.steps / (total_ms * 1e-3) / 1e12

    peak_sus = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    peak_burst = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    fwd_tflops = sparse_flops / (fwd_ms * 1e-3) / 1e12
    traffic, tensor_pipe = profiled_counters("sparse64k")
    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded noise + 3D sinusoidal position code)",
        "config": {"workload": f"sparse64k: Stage-2 block-sparse self-attention B=1 H={H} S=65664 (16x64x64 video + "
                               "8 audio tokens per frame) d=128 block 128 beta=1.0, plus audio->video cross "
                               "attention 128 x 65536 split into 8 KV chunks and LSE-merged",
                   "global_batch": world, "seq_len": S, "parallelism": f"replicas x{world} (heads/batches shard "
                   "with no exchange)", "l2": "inputs (3.2 GB per step) larger than L2; no flush"},
        "dense_equiv_tflops": round(dense_equiv, 2),
        "density": round(density, 5),
        "pct_bf16_peak_executed": round(100 * value / world / peak_burst, 2),
        "breakdown_ms": {"pool_route": round(route_ms, 4), "sparse_fwd": round(fwd_ms, 4),
                         "cross_splitkv_merge": round(cross_ms, 4)},
        "schedule": ("one stream" if args.serial_cross else
                     "cross attention on a second stream, concurrent with pool/route and the sparse forward "
                     "(breakdown times overlap)"),
        "roofline": {"bound": "tensor", "kernel": "attn_fwd_kernel (sparse, d=128, block 128)",
                     "achieved": round(fwd_tflops, 2), "peak": peak_burst, "unit": "TFLOP/s",
                     "frac": round(fwd_tflops / peak_burst, 4),
                     "frac_of_sustained_peak": round(fwd_tflops / peak_sus, 4),
                     "peak_source": f"{peaks_src} bf16_tflops (burst: the timed region is {total_ms:.0f} ms, "
                                    "far from the seconds-long loop the sustained figure was measured in)",
                     "traffic": traffic,
                     "tensor_pipe_active_pct_ncu": tensor_pipe},
        "gpu_launches": kernels_per_step * args.steps,
        "clocks": clocks.summary(),
    }
    if not args.no_e2e:
        result["e2e"] = run_e2e(args, vd, w, (q, k, v), (qa, kx, vx), rt, ws, step_flops, world)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"], result["routing"] = cpu_baseline(q, k, v, w, rt, budget_s=args.cpu_seconds)
    return result


def run_fp8_projection(args, world, rank, local):
    """The block's attention output projection in FP8: per-row quantisation of the
    activations (fp8_quantize_rows) + the scaled FP8 GEMM (fp8_scaled_gemm), x [65664, 4096]
    against W [4096, 4096].  The weights ship in FP8, so W is quantised once before timing."""
    import video_diffusion_transformer_block_gb300 as vd
    from video_diffusion_transformer_block_gb300 import build as vbuild

    vbuild.build()
    vd.load_library()
    peaks, peaks_src = load_peaks()
    lw = LINEAR_WORKLOADS["fp8_proj"]
    M = lw.M if args.tokens is None else args.tokens
    x, W = make_linear(lw, device="cuda", M=M)
    wq, sw = vd.fp8_quantize_rows(W)
    K, N = lw.K, lw.N
    aq = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    sa = torch.empty(M, dtype=torch.float32, device=x.device)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    stream = torch.cuda.current_stream()
    flops = 2.0 * M * N * K
    q_bytes = M * K * 2 + M * K + M * 4                    # read x, write codes and scales
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]

    def step(e=None):
        if e is not None:
            e[0].record(stream)
        vd.fp8_quantize_rows(x, q=aq, scale=sa)
        if e is not None:
            e[1].record(stream)
        vd.fp8_scaled_gemm(aq, sa, wq, sw, y=y)
        if e is not None:
            e[2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        for e in ev:
            step(e)
        torch.cuda.synchronize()
    barrier(world)
    status = vd.attn_last_device_status()
    if status != 0:
        raise RuntimeError(f"device status after timed region: {vd.attn_status_string(status)}")
    ms = max_over_ranks(sum(e[0].elapsed_time(e[2]) for e in ev) / args.steps, world)
    ms_q = sum(e[0].elapsed_time(e[1]) for e in ev) / args.steps
    ms_g = sum(e[1].elapsed_time(e[2]) for e in ev) / args.steps
    value = world * flops / (ms * 1e-3) / 1e12
    peak_bf16 = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    peak = 2.0 * peak_bf16                                  # fp8 = 2 x bf16 (nominal 4.5 / 2.25 PFLOP/s)
    ach = flops / (ms_g * 1e-3) / 1e12
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    q_gbs = q_bytes / (ms_q * 1e-3) / 1e9
    return {"metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "fp8 (e4m3) x fp8, fp32 accumulate, bf16 out", "data": "synthetic",
            "config": {"workload": f"fp8_proj: y = x W^T, x [{M}, {K}] quantised per row, W [{N}, {K}] in FP8",
                       "seq_len": M, "l2": "inputs (538 MB of activations per step) larger than L2; no flush"},
            "breakdown_ms": {"quantize": round(ms_q, 4), "gemm": round(ms_g, 4)},
            "roofline": {"bound": "tensor", "kernel": "fp8_gemm_kernel (tcgen05 kind::f8f6f4, 128x256 tiles)",
                         "achieved": round(ach, 2), "peak": round(peak, 1), "unit": "TFLOP/s",
                         "frac": round(ach / peak, 4),
                         "peak_source": f"{peaks_src} bf16_tflops x 2 (the nominal fp8 / bf16 ratio), burst",
                         "traffic": None},
            "quantize_roofline": {"bound": "hbm", "kernel": "fp8_quantize_rows_reg_kernel", "achieved": round(q_gbs, 1),
                                  "peak": hbm, "unit": "GB/s", "frac": round(q_gbs / hbm, 4), "traffic": None},
            "gpu_launches": 2 * args.steps, "clocks": clocks.summary()}


def run_merge64(args, world, rank, local):
    """The exact LSE merge on its own: 64 back-to-back attn_lse_merge calls per step, each on its
    own partials (8 chunks of the cross-attention shape, [8, 1, 32, 128, 128] fp32 + lse), 1.15 GB
    in all, so that neither launch latency nor L2 residency decides the figure.  The 64 launches
    are captured once in a CUDA graph and the graph is replayed, so the host's launch rate does
    not decide it either."""
    import video_diffusion_transformer_block_gb300 as vd
    from video_diffusion_transformer_block_gb300 import build as vbuild

    vbuild.build()
    vd.load_library()
    peaks, peaks_src = load_peaks()
    n, B, H, Sq, d, inst = CROSS_N_SPLIT, 1, 32, CROSS_SQ, 128, 64
    g = torch.Generator(device="cuda")
    g.manual_seed(9 + rank)
    ops = [torch.randn((n, B, H, Sq, d), generator=g, device="cuda") for _ in range(inst)]
    lps = [torch.randn((n, B, H, Sq), generator=g, device="cuda") * 3 for _ in range(inst)]
    outs = [torch.empty((B, H, Sq, d), dtype=torch.bfloat16, device="cuda") for _ in range(inst)]
    lses = [torch.empty((B, H, Sq), dtype=torch.float32, device="cuda") for _ in range(inst)]
    per = n * B * H * Sq * (d + 1) * 4 + B * H * Sq * (d * 2 + 4)   # partials read, out + lse written
    stream = torch.cuda.current_stream()

    def launches():
        for i in range(inst):
            vd.attn_lse_merge(ops[i], lps[i], out=outs[i], lse=lses[i])

    launches()                                   # warm the library (descriptor setup, module load)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        launches()
    torch.cuda.synchronize()

    def step():
        graph.replay()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        for e0, e1 in evs:
            e0.record(stream)
            step()
            e1.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in evs) / args.steps, world)
    gbs = inst * per / (ms * 1e-3) / 1e9
    peak = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    return {"metric": "LSE merge GB/s (64 instances per step)", "value": round(world * gbs, 1), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32 partials, bf16 out",
            "data": "synthetic",
            "config": {"workload": f"merge64: 64 x attn_lse_merge of {n} partials [1, 32, 128, 128], one CUDA graph",
                       "l2": "64 distinct buffer sets, 1.15 GB per step (> L2)"},
            "roofline": {"bound": "hbm", "kernel": "lse_merge_kernel", "achieved": round(gbs, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(gbs / peak, 4), "peak_source": f"{peaks_src} hbm_gbs",
                         "traffic": None},
            "gpu_launches": inst * args.steps, "clocks": clocks.summary()}


def run_sweep(args, world, rank, local):
    """The beta sweep workload at S = 131072 (32x64x64 grid, H32 d128, block 128) for one beta
    (--beta): pool + route (attn_sparse_route) and the block-sparse forward (attn_sparse_fwd) per
    step, timed separately with CUDA events; inputs (3.2 GB) are larger than L2."""
    import video_diffusion_transformer_block_gb300 as vd
    from video_diffusion_transformer_block_gb300 import build as vbuild

    vbuild.build()
    vd.load_library()
    peaks, peaks_src = load_peaks()
    w0 = WORKLOADS["sweep128k"]
    w = Workload(w0.name, B=w0.B, H=args.heads, Sq=w0.Sq, Skv=w0.Skv, d=w0.d, seed=w0.seed + 1000 * rank,
                 q_std=w0.q_std, k_std=w0.k_std, grid=w0.grid, pe=True, block=w0.block, beta=args.beta)
    q, k, v = make_qkv(w, device="cuda")
    B, H, S, d, block = w.B, w.H, w.Sq, w.d, w.block
    ws = torch.empty(vd.attn_sparse_workspace_bytes(B, H, S, d, block, block), dtype=torch.uint8, device=q.device)
    rt = vd.sparse_route_buffers(B, H, S, d, block, q.device, order=True)
    out = torch.empty_like(q)
    lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
    stream = torch.cuda.current_stream()

    def step(e=None):
        if e is not None:
            e[0].record(stream)
        vd.attn_sparse_route(q, k, v, args.beta, block=block, route=rt, workspace=ws)
        if e is not None:
            e[1].record(stream)
        vd.attn_sparse_fwd(q, k, v, rt, block=block, out=out, lse=lse)
        if e is not None:
            e[2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    flops = executed_sparse_flops(rt["sel_idx"], rt["sel_cnt"], S, block, d)
    dense_eq = 4.0 * B * H * S * S * d
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        for e in evs:
            step(e)
        torch.cuda.synchronize()
    barrier(world)
    status = vd.attn_last_device_status()
    if status != 0:
        raise RuntimeError(f"device status after timed region: {vd.attn_status_string(status)}")
    ms = max_over_ranks(sum(e[0].elapsed_time(e[2]) for e in evs) / args.steps, world)
    ms_route = sum(e[0].elapsed_time(e[1]) for e in evs) / args.steps
    ms_fwd = sum(e[1].elapsed_time(e[2]) for e in evs) / args.steps
    value = world * flops / (ms * 1e-3) / 1e12
    peak = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    fwd = flops / (ms_fwd * 1e-3) / 1e12
    return {"metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"sweep128k: B1 H{H} S{S} (32x64x64) d128 block 128 beta {args.beta}",
                       "seq_len": S, "l2": "inputs (3.2 GB) larger than L2; no flush"},
            "density": round(flops / dense_eq, 5),
            "dense_equiv_tflops": round(world * dense_eq / (ms * 1e-3) / 1e12, 2),
            "breakdown_ms": {"pool_route": round(ms_route, 4), "sparse_fwd": round(ms_fwd, 4)},
            "roofline": {"bound": "tensor", "kernel": "attn_fwd_kernel (sparse, d=128, block 128)",
                         "achieved": round(fwd, 2), "peak": peak, "unit": "TFLOP/s", "frac": round(fwd / peak, 4),
                         "peak_source": f"{peaks_src} bf16_tflops (burst)", "traffic": None},
            # pool, routing (1024 query blocks a head: tensor-core tiles only), query-block order, forward
            "gpu_launches": 4 * args.steps, "clocks": clocks.summary()}


def run_native_kernel(args, world, rank, local):
    """Secondary workloads (not the benchmark line): one kernel path per step.
      dense16k: attn_dense_fwd on B1 H32 S16384 d128 (tensor-bound)
      cross:    attn_cross_splitkv_fwd + attn_lse_merge, 128 x 32768, 8 chunks (HBM-bound)
      na3d:     attn_na3d_fwd, 3D neighbourhood attention, 4x128x128 volume, window 3x7x7 (tensor-bound on
                the executed key boxes; the value counts only the window's FLOPs)"""
    import video_diffusion_transformer_block_gb300 as vd
    from video_diffusion_transformer_block_gb300 import build as vbuild

    vbuild.build()
    vd.load_library()
    peaks, peaks_src = load_peaks()
    w0 = WORKLOADS[args.workload]
    w = Workload(w0.name, B=w0.B, H=args.heads, Sq=w0.Sq, Skv=w0.Skv, d=w0.d, seed=w0.seed + 1000 * rank,
                 q_std=w0.q_std, k_std=w0.k_std, grid=w0.grid, audio_per_frame=w0.audio_per_frame, pe=w0.pe,
                 n_split=w0.n_split)
    q, k, v = make_qkv(w, device="cuda")
    B, H, Sq, Skv, d = w.B, w.H, w.Sq, w.Skv, w.d
    stream = torch.cuda.current_stream()
    out = torch.empty_like(q)
    lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)
    if args.workload == "dense16k":
        launches = 1
        flops = 4.0 * B * H * Sq * Skv * d

        def step():
            vd.attn_dense_fwd(q, k, v, out=out, lse=lse)
    elif args.workload == "na3d":
        launches = 1
        kern = w0.extra["kernel"]
        brick, pair, boxes = vd.attn_na3d_plan(w.grid, kern, 0, args.na_plan)
        flops = 4.0 * B * H * Sq * math.prod(kern) * d                 # the windows' own work
        # what the tensor cores run: per key box S = Q K^T and O += P V, and on the
        # persistent plans one (plan 4, 4x4x8 bricks) or two K = 16 steps that add the window;
        # plan 6's one K = 32 step of E5M2 operands takes the tensor pipe as long as one bf16
        # K = 16 step, and is counted as one
        window_k = (16 if (brick == 3 and pair == 4) or pair == 6 else 32) if pair in (4, 5, 6) else 0
        exec_flops = 2.0 * B * H * boxes * 128 * 128 * (2 * d + window_k)

        def step():
            vd.attn_na3d_fwd(q, k, v, w.grid, kern, brick=brick, pair_axis=pair, out=out, lse=lse)
    else:
        n = w.n_split
        op = torch.empty((n, B, H, Sq, d), dtype=torch.float32, device=q.device)
        lp = torch.empty((n, B, H, Sq), dtype=torch.float32, device=q.device)
        launches = 2
        flops = 4.0 * B * H * Sq * Skv * d
        kv_bytes = 2.0 * B * H * Skv * d * 2 + B * H * Sq * d * 2 + n * B * H * Sq * (d + 1) * 4

        def step():
            vd.attn_cross_splitkv_fwd(q, k, v, n, out_part=op, lse_part=lp)
            vd.attn_lse_merge(op, lp, out=out, lse=lse)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=q.device)   # 256 MB > L2, written between steps
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        for e0, e1 in evs:
            flush.fill_(1)
            e0.record(stream)
            step()
            e1.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    status = vd.attn_last_device_status()
    if status != 0:
        raise RuntimeError(f"device status after timed region: {vd.attn_status_string(status)}")
    ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in evs) / args.steps, world)
    value = world * flops / (ms * 1e-3) / 1e12
    extra = {}
    if args.workload == "na3d":
        peak = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
        ach = exec_flops / (ms * 1e-3) / 1e12
        kname = (f"attn_na_persist_kernel (3D neighbourhood, persistent one-brick tiles, brick {brick}"
                 f"{', key boxes 4x2x16' if pair in (5, 6) else ''}{', E5M2 window operands' if pair == 6 else ''}"
                 f", d={d})"
                 if pair in (4, 5, 6) else f"attn_fwd_kernel (3D neighbourhood, brick {brick}, pair {pair}, d={d})")
        # counters of the library's own plan under "na3d", of an explicit plan under "na3d_plan<n>"
        traffic, tpipe = (profiled_counters("na3d" if args.na_plan == -1 else f"na3d_plan{args.na_plan}")
                          if H == 32 else (None, None))
        roof = {"bound": "tensor", "kernel": kname,
                "achieved": round(ach, 2), "peak": peak, "unit": "TFLOP/s", "frac": round(ach / peak, 4),
                "peak_source": f"{peaks_src} bf16_tflops (burst: one kernel per timed step, L2 flushed between)",
                "traffic": traffic, "tensor_pipe_active_pct_ncu": tpipe}
        extra = {"executed_tflops": round(world * ach, 2), "window_fraction_of_executed": round(flops / exec_flops, 4)}
    elif args.workload == "dense16k":
        peak = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
        roof = {"bound": "tensor", "kernel": "attn_fwd_kernel (dense, d=128)", "achieved": round(value / world, 2),
                "peak": peak, "unit": "TFLOP/s", "frac": round(value / world / peak, 4),
                "peak_source": f"{peaks_src} bf16_tflops (burst: one kernel per timed step, L2 flushed between)",
                "traffic": None}
    else:
        peak = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
        gbs = kv_bytes / (ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "kernel": "attn_fwd_kernel (split-KV) + lse_merge_kernel", "achieved": round(gbs, 1),
                "peak": peak, "unit": "GB/s", "frac": round(gbs / peak, 4), "peak_source": f"{peaks_src} hbm_gbs",
                "traffic": None}
    return {"metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"{args.workload}: B={B} H={H} Sq={Sq} Skv={Skv} d={d}"
                       + (f" volume {w.grid} window {w0.extra['kernel']} plan {pair}" if args.workload == "na3d"
                          else ""),
                       "seq_len": Skv, "l2": "256 MB buffer written between timed steps (L2 flush)"},
            **extra, "roofline": roof, "gpu_launches": launches * args.steps, "clocks": clocks.summary()}


def run_e2e(args, vd, w, qkv, cross, rt, ws, step_flops, world):
    """Same step through the public API with the inputs in pinned host memory.

    Every step copies its inputs host->device (q, k, v and the cross-attention
    inputs) and reads its outputs (out, lse and the cross-attention out, lse)
    back to pinned host memory, inside the timed region.  Like a serving loop,
    the copies are double-buffered: step i+1's inputs are uploaded (one copy
    stream) and step i-1's outputs downloaded (another copy stream, so the two
    directions of the host link run concurrently) while step i computes."""
    q, k, v = qkv
    qa, kx, vx = cross
    B, H, S, d, block = w.B, w.H, w.Sq, w.d, w.block
    hin = [t.cpu().pin_memory() for t in (q, k, v, qa, kx, vx)]
    din = [[torch.empty_like(t) for t in (q, k, v, qa, kx, vx)] for _ in range(2)]

    def outputs():
        return [torch.empty_like(q), torch.empty((B, H, S), dtype=torch.float32, device=q.device),
                torch.empty((B, H, CROSS_SQ, d), dtype=torch.bfloat16, device=q.device),
                torch.empty((B, H, CROSS_SQ), dtype=torch.float32, device=q.device)]
    dout = [outputs(), outputs()]
    op = torch.empty((CROSS_N_SPLIT, B, H, CROSS_SQ, d), dtype=torch.float32, device=q.device)
    lp = torch.empty((CROSS_N_SPLIT, B, H, CROSS_SQ), dtype=torch.float32, device=q.device)
    hout = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in dout[0]]
    h2d = sum(t.numel() * t.element_size() for t in hin)
    d2h = sum(t.numel() * t.element_size() for t in hout)
    comp = torch.cuda.current_stream()
    xcomp = comp if args.serial_cross else torch.cuda.Stream()   # the cross attention, as in the device-timed step
    upload, download = torch.cuda.Stream(), torch.cuda.Stream()

    def run(steps):
        up = [torch.cuda.Event() for _ in range(steps + 1)]
        done = [torch.cuda.Event() for _ in range(steps)]
        down = [torch.cuda.Event() for _ in range(steps)]
        with torch.cuda.stream(upload):
            for dst, src in zip(din[0], hin):
                dst.copy_(src, non_blocking=True)
            up[0].record(upload)
        for i in range(steps):
            buf, ob = din[i % 2], dout[i % 2]
            for st in {comp, xcomp}:
                st.wait_event(up[i])
                if i >= 2:
                    st.wait_event(down[i - 2])            # this output buffer has been read back
            vd.attn_cross_splitkv_fwd(buf[3], buf[4], buf[5], CROSS_N_SPLIT, out_part=op, lse_part=lp, stream=xcomp)
            vd.attn_lse_merge(op, lp, out=ob[2], lse=ob[3], stream=xcomp)
            xdone = torch.cuda.Event()
            xdone.record(xcomp)
            vd.attn_sparse_route(buf[0], buf[1], buf[2], args.beta, block=block, route=rt, workspace=ws, stream=comp)
            vd.attn_sparse_fwd(buf[0], buf[1], buf[2], rt, block=block, out=ob[0], lse=ob[1], stream=comp)
            comp.wait_event(xdone)
            done[i].record(comp)
            if i + 1 < steps:
                with torch.cuda.stream(upload):
                    if i >= 1:
                        upload.wait_event(done[i - 1])    # the other input buffer is free again
                    for dst, src in zip(din[(i + 1) % 2], hin):
                        dst.copy_(src, non_blocking=True)
                    up[i + 1].record(upload)
            with torch.cuda.stream(download):
                download.wait_event(done[i])
                for dst, src in zip(hout, ob):
                    dst.copy_(src, non_blocking=True)
                down[i].record(download)
        comp.wait_stream(upload)
        comp.wait_stream(download)

    run(2)
    torch.cuda.synchronize()
    # the host link's own rate in this run (the step is bound by it): one upload of q from pinned
    # memory and one download into pinned memory, timed with CUDA events on the copy streams
    def link_gbs(dst, src, st):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(st):
            e0.record(st)
            dst.copy_(src, non_blocking=True)
            e1.record(st)
        e1.synchronize()
        return src.numel() * src.element_size() / (e0.elapsed_time(e1) * 1e-3) / 1e9
    link = {"h2d_gbs": round(link_gbs(din[0][0], hin[0], upload), 1),
            "d2h_gbs": round(link_gbs(hin[0], din[0][0], download), 1)}
    steps = max(3, args.steps // 2)
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    run(steps)
    e1.record(comp)
    torch.cuda.synchronize()
    barrier(world)
    ms = max_over_ranks(e0.elapsed_time(e1), world) / steps
    return {"value": round(world * step_flops / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "ms_per_step": round(ms, 4),
            "steps": steps, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "host_link_measured": link,
            "pipelining": "double-buffered: uploads and downloads on two copy streams overlap each other and the "
                          "previous/next step's compute; the cross attention on its own compute stream"}


# ============================================================ oracle (CPU baseline / reference arm)

def oracle_sample(qh, kh, vh, w, n_rows, rng):
    """Oracle work on a bounded sample of the Stage-2 workload: pool + route of one head and
    block-sparse attention of n_rows sampled query rows of it.  Returns (seconds, executed FLOPs)."""
    import oracle
    S, d, block = w.Sq, w.d, w.block
    rows = np.sort(rng.choice(S, size=n_rows, replace=False)).astype(np.int64)
    t0 = time.perf_counter()
    qp, kp, vp = oracle.block_pool(qh, block), oracle.block_pool(kh, block), oracle.block_pool(vh, block)
    rt = oracle.route(qp, kp, vp, S, block, w.scale, w.beta)
    oracle.sparse_attention(qh, kh, vh, block, block, rt["sel"], rt["mu"], rt["W"], rt["T"], w.scale, rows=rows)
    dt = time.perf_counter() - t0
    nb = rt["sel"].shape[-1]
    sizes = np.array([min(block, S - j * block) for j in range(nb)], dtype=np.float64)
    keys_per_block = rt["sel"][0, 0].astype(np.float64) @ sizes
    flops = 4.0 * d * keys_per_block[rows // block].sum()
    return dt, flops


def host_head(q, k, v, h=0):
    return [to_f64(x[:, h:h + 1].contiguous()) for x in (q, k, v)]


def routing_report(q, k, v, w, rt):
    """The oracle's routing of every head (pool + route in fp64) against the GPU routing of the timed
    steps: selection flips (each must lie in the 1e-4 band around tau or the row max), the number of
    clamped Taylor weights on the GPU's selection, and both densities.  Returns (seconds, report)."""
    import oracle
    S, block = w.Sq, w.block
    idx, cnt = rt["sel_idx"].cpu().numpy(), rt["sel_cnt"].cpu().numpy()
    nb = idx.shape[-1]
    flips = outside = clamped = sel_gpu = sel_oracle = 0
    dt = 0.0
    for h in range(w.H):
        qh, kh, vh = host_head(q, k, v, h)
        gsel = np.zeros((1, 1, nb, nb), dtype=bool)
        for i in range(nb):
            gsel[0, 0, i, idx[0, h, i, :cnt[0, h, i]]] = True
        t0 = time.perf_counter()
        qp, kp, vp = oracle.block_pool(qh, block), oracle.block_pool(kh, block), oracle.block_pool(vh, block)
        ort = oracle.route(qp, kp, vp, S, block, w.scale, w.beta)
        forced = oracle.route(qp, kp, vp, S, block, w.scale, w.beta, force_sel=gsel)
        dt += time.perf_counter() - t0
        proxy, tau = ort["proxy"], ort["tau"][..., None]
        near = (np.abs(proxy - tau) < 1e-4) | (np.abs(proxy - proxy.max(-1, keepdims=True)) < 1e-4)
        diff = gsel != ort["sel"]
        flips += int(diff.sum())
        outside += int((diff & ~near).sum())
        clamped += forced["n_clamped"]
        sel_gpu += int(gsel.sum())
        sel_oracle += int(ort["sel"].sum())
    pairs = w.H * nb * nb
    return dt, {"near_tau_flips": flips, "flips_outside_1e-4_band": outside, "clamped_taylor_weights": clamped,
                "selected_blocks_gpu": sel_gpu, "selected_blocks_oracle": sel_oracle,
                "block_density_gpu": round(sel_gpu / pairs, 6), "block_density_oracle": round(sel_oracle / pairs, 6),
                "source": "fp64 oracle pool + route of every head against the GPU's routing of the timed steps"}


def single_core_oracle():
    """The oracle on one core for the tiny block-sparse config (the whole config: pool, route and every
    row of the sparse attention, beta 0.5) and the cross-attention config (split partials + merge;
    head 0 timed, extrapolated to the 32 heads).  Returns a dict of seconds and GFLOP/s."""
    import ctypes
    import oracle
    try:
        gomp = ctypes.CDLL("libgomp.so.1")
    except OSError:
        return {"unavailable": "libgomp not found"}
    prev = gomp.omp_get_max_threads()
    gomp.omp_set_num_threads(1)
    try:
        wt = WORKLOADS["tiny"]
        q, k, v = make_qkv(wt, device="cpu")
        qh, kh, vh = to_f64(q), to_f64(k), to_f64(v)
        t0 = time.perf_counter()
        out, lse, rt, _ = oracle.sparse_route_attention(qh, kh, vh, wt.block, wt.block, wt.scale, wt.beta)
        t_tiny = time.perf_counter() - t0
        nb = rt["sel"].shape[-1]
        sizes = np.array([min(wt.block, wt.Sq - j * wt.block) for j in range(nb)], dtype=np.float64)
        f_tiny = 4.0 * wt.d * float(((rt["sel"] @ sizes) * sizes[None, None, :]).sum())
        wc = WORKLOADS["cross"]
        q, k, v = make_qkv(Workload(wc.name, B=1, H=1, Sq=wc.Sq, Skv=wc.Skv, d=wc.d, seed=wc.seed), device="cpu")
        qh, kh, vh = to_f64(q), to_f64(k), to_f64(v)
        t0 = time.perf_counter()
        op, lp = oracle.split_partials(qh, kh, vh, wc.scale, wc.n_split)
        oracle.lse_merge(op, lp)
        t_head = time.perf_counter() - t0
        f_head = 4.0 * wc.Sq * wc.Skv * wc.d
    finally:
        gomp.omp_set_num_threads(prev)
    return {"cores": 1,
            "tiny": {"seconds": round(t_tiny, 4), "gflops": round(f_tiny / t_tiny / 1e9, 3),
                     "sample": "whole config: B1 H2 S1024 d64 block 64 beta 0.5, pool + route + all rows"},
            "cross": {"seconds": round(t_head * wc.H, 3), "gflops": round(f_head / t_head / 1e9, 3),
                      "sample": f"head 0 of 32 timed ({t_head:.3f} s), extrapolated x32: split partials (8 chunks) "
                                "+ LSE merge, 128 x 32768 d128"}}


def cpu_baseline(q, k, v, w, rt=None, budget_s=15.0):
    """The oracle on the host cores over heads 0, 1, ... of the same inputs until about budget_s
    seconds of work: each head's pool + route, then its block-sparse attention on sampled rows
    (all rows while the budget lasts).  With the GPU routing ``rt``, the oracle also routes every
    head (routing_report).  Returns (cpu_baseline dict, routing report or None)."""
    import oracle
    oracle.build()
    rng = np.random.default_rng(0)
    qh, kh, vh = host_head(q, k, v, 0)
    dt0, _ = oracle_sample(qh, kh, vh, w, 64, rng)                     # calibration
    per_row = max(dt0 / 64, 1e-6)
    dt = flops = 0.0
    heads, rows_done = 0, 0
    while heads < w.H and (heads == 0 or dt < budget_s * 0.8):
        if heads > 0:
            qh, kh, vh = host_head(q, k, v, heads)
        n_rows = int(min(w.Sq, max(256, (budget_s - dt) / per_row)))
        t, f = oracle_sample(qh, kh, vh, w, n_rows, rng)
        dt, flops, heads, rows_done = dt + t, flops + f, heads + 1, rows_done + n_rows
    cores = len(os.sched_getaffinity(0))
    base = {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": cores, "cpu_model": cpu_model(),
            "kind": "oracle", "seconds": round(dt, 3),
            "sample": f"heads 0-{heads - 1} of the sparse64k workload: per head, block pool + route and block-sparse "
                      f"attention of seeded sampled query rows ({rows_done} rows in all; fp64 C oracle, OpenMP on "
                      f"{cores} threads)",
            "single_core": single_core_oracle()}
    report = None
    if rt is not None:
        t_route, report = routing_report(q, k, v, w, rt)
        base["route_all_heads_seconds"] = round(t_route, 3)
    return base, report


def run_reference(args, world, rank):
    """Reference arm: the fp64 CPU oracle timed on bounded samples of the same workload."""
    if rank != 0:
        return None
    import oracle
    oracle.build()
    w = WORKLOADS["sparse64k"]
    q, k, v = make_qkv(Workload(w.name, B=1, H=1, Sq=w.Sq, Skv=w.Skv, d=w.d, seed=w.seed, q_std=w.q_std,
                                k_std=w.k_std, grid=w.grid, audio_per_frame=w.audio_per_frame, pe=True,
                                block=w.block, beta=args.beta), device="cpu")
    w = Workload(w.name, B=1, H=1, Sq=w.Sq, Skv=w.Skv, d=w.d, seed=w.seed, block=w.block, beta=args.beta)
    qh, kh, vh = to_f64(q), to_f64(k), to_f64(v)
    rng = np.random.default_rng(1)
    dt0, _ = oracle_sample(qh, kh, vh, w, 32, rng)
    per_row = max(dt0 / 32, 1e-6)
    budget = max(2.0, args.cpu_seconds * 4 / max(1, args.steps + args.warmup))
    n_rows = int(min(w.Sq, max(64, budget / per_row)))
    for _ in range(args.warmup):
        oracle_sample(qh, kh, vh, w, n_rows, rng)
    tot_t, tot_f = 0.0, 0.0
    for _ in range(args.steps):
        dt, fl = oracle_sample(qh, kh, vh, w, n_rows, rng)
        tot_t += dt
        tot_f += fl
    val = tot_f / tot_t / 1e12
    cores = len(os.sched_getaffinity(0))
    sample = (f"per step: head 0 of the sparse64k workload, block pool + route of the head and block-sparse "
              f"attention of {n_rows} seeded sampled query rows (fp64 C oracle, {cores} threads)")
    return {"metric": METRIC, "value": round(val, 6), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(1e3 * tot_t / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "sparse64k (bounded sample, see cpu_baseline.sample)", "seq_len": w.Sq},
            "impl": "reference",
            "cpu_baseline": {"value": round(val, 6), "unit": "TFLOP/s", "cores": cores, "cpu_model": cpu_model(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(val, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--beta", type=float, default=1.0)
    ap.add_argument("--heads", type=int, default=32, help="heads (32 = the benchmark; fewer only for profiling)")
    ap.add_argument("--workload", choices=["sparse64k", "dense16k", "cross", "na3d", "fp8_proj", "merge64",
                                           "sweep128k"],
                    default="sparse64k",
                    help="sparse64k = the benchmark step; dense16k / cross / na3d / fp8_proj time one path each")
    ap.add_argument("--na-plan", type=int, default=-1, choices=[-1, 3, 4, 5, 6],
                    help="na3d only: the pair axis / plan (-1 = the library's choice; 6 = E5M2 window operands, "
                         "exact for raw scores |q.k| < 2^30)")
    ap.add_argument("--tokens", type=int, default=None,
                    help="fp8_proj only: activation rows (default 65664; fewer only for profiling)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--serial-cross", action="store_true",
                    help="run the cross attention after the self-attention on one stream (no overlap)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup()
    if args.impl == "reference":
        res = run_reference(args, world, rank)
    elif args.workload == "fp8_proj":
        res = run_fp8_projection(args, world, rank, local)
    elif args.workload == "merge64":
        res = run_merge64(args, world, rank, local)
    elif args.workload == "sweep128k":
        res = run_sweep(args, world, rank, local)
    elif args.workload != "sparse64k":
        res = run_native_kernel(args, world, rank, local)
    else:
        res = run_native(args, world, rank, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
