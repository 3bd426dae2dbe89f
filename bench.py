#!/usr/bin/env python3
"""Benchmark: HCA attention forward + backward on GB300.

One step = hca_attn_fwd + hca_attn_bwd on one batch of the headline
workload (B=1, H=64, S=65536, D=128, W=128, m=128, one document, bf16,
q/kv/ckv/dO ~ N(0,1)).  Throughput counts FLOPs over visible (query, key)
pairs only: 4*D per pair and head for the forward, 10*D for the backward.

Prints ONE JSON line (rank 0).  With torchrun (N > 1) every rank runs its own
batch (weak scaling, no collective on the data path); timing is the max over
ranks of the device-timed region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

``--impl reference`` times the fp64 CPU oracle on the host cores on a bounded
sample of the same workload (the only other place this file runs the oracle
is the cpu_baseline leg of the default arm).
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
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "HCA attn fwd+bwd TFLOP/s (visible pairs) and % bf16 TC peak at S=65536"
UNIT = "TFLOP/s"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
PROFILES = os.path.join(ROOT, "profiles")
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}

# algorithmic GEMM FLOPs per visible (query, key) pair per head, per kernel
# (D multiplies each): forward QK^T + PV; dq kernel S + dP + dQ; dkv kernel
# dK + dV.  The S^T and dP^T that the key-major dkv kernel recomputes are not
# algorithmic work: the backward as a whole counts 10*D (S, dP, dQ, dK, dV).
KERNEL_FLOP_PER_PAIR_D = {"hca_fwd_tc": 4, "hca_bwd_dq": 6, "hca_bwd_dkv": 4}
KERNEL_SOURCES = {"hca_fwd_tc": "hca_fwd_tc.cu", "hca_bwd_dq": "hca_bwd_tc.cu", "hca_bwd_dkv": "hca_bwd_tc.cu"}
# headers every tensor-core kernel is built from (part of a kernel's digest)
KERNEL_HEADERS = ("hca_common.cuh", "tc_ptx.cuh", "tc_tiles.cuh")
# secondary roof: exponentials.  ex2.approx.f32 issues at 32 per clock per SM
# on GB300 (measured with 1024 threads x 8 independent chains per SM); the
# path needs one exp per visible pair and head in the forward and one in each
# backward kernel (dq and dkv both form P).
EX2_PER_CLK_PER_SM = 32
EXP_PER_PAIR = {"fwd": 1, "bwd": 2}


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing leg")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="target CPU time of the oracle sample")
    ap.add_argument("--mode", choices=("hca", "local", "compress", "indexer", "csa"), default="hca",
                    help="local: the local sliding-window entry points (no compressed set) on the same shape; "
                         "compress: the HCA compressor (m=128) and its backward; indexer: the Lightning Indexer "
                         "scores + top-k on the CSA shape (m=4); csa: compressed sparse attention fwd+bwd "
                         "(m=4, k=256 selected entries per query)")
    ap.add_argument("--ncu-case", type=int, default=0, metavar="S",
                    help="profiling case: run --warmup + 1 untimed fwd+bwd steps of the headline shape at sequence "
                         "length S and exit (for ncu captures; prints nothing to time)")
    return ap.parse_args(argv)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world, backend):
    if world <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group(backend=backend)
    return dist


def max_over_ranks(value: float, dist, device=None) -> float:
    """Max of a float over all ranks (identity without a process group)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def workload():
    from block_sparse_compressed_gb300 import inputs as I
    return I.LONG_S65536


def visible_pairs_closed_form(S, W, m):
    """Per-head visible pairs of one unpadded document of length S."""
    raw = S * (S + 1) // 2 if S <= W else W * S - W * (W - 1) // 2
    q, r = divmod(S, m)
    comp = m * q * (q - 1) // 2 + q * (r + 1)
    return raw, comp


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        # raw samples go to $HCA_BENCH_CLOCKS_DIR when set (to keep them), else a temporary directory
        out_dir = os.environ.get("HCA_BENCH_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(out_dir, f"hca_bench_clocks_rank{gpu_index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sms, maxs, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sms.append(float(parts[1]))
                    maxs.append(float(parts[2]))
                except ValueError:
                    continue
                for nm, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(nm)
        if not sms:
            return None
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxs), "samples": len(sms),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# profiles: DRAM traffic of the dominant kernel from a committed ncu summary
# ---------------------------------------------------------------------------
def source_digest(kernel: str) -> str:
    csrc = os.path.join(ROOT, "block_sparse_compressed_gb300", "csrc")
    if kernel not in KERNEL_SOURCES:
        return ""
    h = hashlib.sha256()
    try:
        for name in (KERNEL_SOURCES[kernel],) + KERNEL_HEADERS:
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(f.read())
    except OSError:
        return ""
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, work_key: str):
    """traffic bytes per launch recorded for `kernel` on this workload, or
    None when there is no summary or the kernel source changed since."""
    if not os.path.isdir(PROFILES):
        return None
    digest = source_digest(kernel)
    for name in sorted(os.listdir(PROFILES)):
        if not name.startswith(kernel) or not name.endswith((".md", ".txt")):
            continue
        text = open(os.path.join(PROFILES, name)).read()
        m_w = re.search(r"^workload:\s*(.+)$", text, re.M)
        m_t = re.search(r"^traffic_bytes_per_launch:\s*([0-9.eE+]+)", text, re.M)
        m_h = re.search(r"^source_sha256_16:\s*([0-9a-f]+)", text, re.M)
        if not (m_w and m_t and m_h) or m_w.group(1).strip() != work_key:
            continue
        if m_h.group(1) != digest:
            return None
        return float(m_t.group(1))
    return None


# ---------------------------------------------------------------------------
# CPU baseline (oracle) on a bounded sample
# ---------------------------------------------------------------------------
def cpu_baseline(w, q, kv, ckv, dout, target_s: float):
    """Time the fp64 oracle forward+backward on the last R query positions of
    the workload (the rows with the most keys), R sized to ~target_s."""
    import oracle
    S = w.S
    qc, kvc, ckvc, dc = q.cpu(), kv.cpu(), ckv.cpu(), dout.cpu()

    def pairs_in(lo, hi):
        raw = sum(min(i + 1, w.W) for i in range(lo, hi))
        comp = sum((i + 1) // w.m for i in range(lo, hi))
        return (raw + comp) * w.H

    def run(R):
        lo = S - R
        t0 = time.perf_counter()
        oracle.fwd(qc, kvc, ckvc, None, w.W, w.m, w.scale, rows=(lo, S))
        oracle.bwd(qc, kvc, ckvc, None, dc, w.W, w.m, w.scale, rows=(lo, S))
        return time.perf_counter() - t0, pairs_in(lo, S)

    # grow the sample until it takes about target_s (the fixed cost of a call
    # makes the first small samples a poor predictor)
    R = 16
    dt, pairs = run(R)
    while dt < 0.6 * target_s and R < S:
        R = int(min(S, R * min(8.0, max(1.5, 0.9 * target_s / max(dt, 1e-3)))))
        dt, pairs = run(R)
    flops = 14 * w.D * pairs
    return {"value": flops / dt / 1e12, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"fp64 oracle fwd+bwd over query rows [{S - R},{S}) of the workload "
                      f"({pairs} visible pair-heads, {dt:.1f} s)", "seconds": dt}


# ---------------------------------------------------------------------------
# reference arm: the oracle as the reference implementation
# ---------------------------------------------------------------------------
def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import torch
    from block_sparse_compressed_gb300 import inputs as I
    w = workload()
    q, kv, ckv, seg, dout = I.tensors(w, device="cpu")
    import oracle
    # each step: a bounded sample of the workload sized so the run stays short
    per_step = max(2.0, 60.0 / max(1, args.steps + args.warmup))
    probe = cpu_baseline(w, q, kv, ckv, dout, per_step)
    R_rows = int(re.search(r"\[(\d+),", probe["sample"]).group(1))
    lo = R_rows
    times, pairs = [], None
    for k in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.fwd(q, kv, ckv, None, w.W, w.m, w.scale, rows=(lo, w.S))
        oracle.bwd(q, kv, ckv, None, dout, w.W, w.m, w.scale, rows=(lo, w.S))
        dt = time.perf_counter() - t0
        if k >= args.warmup:
            times.append(dt)
    raw = sum(min(i + 1, w.W) for i in range(lo, w.S))
    comp = sum((i + 1) // w.m for i in range(lo, w.S))
    pairs = (raw + comp) * w.H
    total = sum(times)
    value = 14 * w.D * pairs * len(times) / total / 1e12
    cb = {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
          "sample": f"fp64 oracle fwd+bwd over query rows [{lo},{w.S}) per step"}
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * total / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_dict(w), "cpu_baseline": cb,
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def config_dict(w):
    return {"workload": w.name, "B": w.B, "H": w.H, "S": w.S, "D": w.D, "W": w.W, "m": w.m, "segments": "one",
            "l2": "no flush: q/dO/out/dq are 1.07 GB each, far above the 129 MB L2",
            "parallelism": "replicas (one independent batch per GPU)"}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def run_ours(args):
    import torch
    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        print(json.dumps({"metric": METRIC, "error": "no CUDA device"}), flush=True)
        return 1
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    from block_sparse_compressed_gb300 import hca
    from block_sparse_compressed_gb300 import inputs as I
    w = workload()
    hca.load()
    q, kv, ckv, seg, dout = I.tensors(w, device=dev, seed=I.SEED + 100 * rank)
    raw, comp = visible_pairs_closed_form(w.S, w.W, w.m)
    pairs = (raw + comp) * w.H * w.B
    gr, gc = hca.hca_visible_pairs(seg, w.B, w.S, w.W, w.m, device=dev)
    assert int((gr + gc).sum().item()) * w.H == pairs, "visible-pair count mismatch"
    flop_fwd, flop_bwd = 4 * w.D * pairs, 10 * w.D * pairs
    out = torch.empty_like(q)
    lse = torch.empty(w.B, w.H, w.S, dtype=torch.float32, device=dev)
    dq, dkv, dckv = torch.empty_like(q), torch.empty_like(kv), torch.empty_like(ckv)
    wsf = hca.workspace(w.B, w.H, w.S, w.D, w.W, w.m, w.dtype, False, dev)
    wsb = hca.workspace(w.B, w.H, w.S, w.D, w.W, w.m, w.dtype, True, dev)

    def step():
        hca.hca_attn_fwd(q, kv, ckv, seg, w.W, w.m, w.scale, out=out, lse=lse, ws=wsf)
        hca.hca_attn_bwd(q, kv, ckv, seg, out, lse, dout, w.W, w.m, w.scale, dq=dq, dkv=dkv, dckv=dckv, ws=wsb)

    step()
    if hca.hca_workspace_status(wsf) != 0 or hca.hca_workspace_status(wsb) != 0:
        raise RuntimeError("device reported an error status")
    for _ in range(max(0, args.warmup - 1)):
        step()
    # no hidden allocation in a step: peak memory before/after one more step
    torch.cuda.synchronize(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    base_alloc = torch.cuda.memory_allocated(dev)
    step()
    torch.cuda.synchronize(dev)
    memory = {"workspace_fwd_bytes": wsf.numel(), "workspace_bwd_bytes": wsb.numel(),
              "step_peak_delta_bytes": torch.cuda.max_memory_allocated(dev) - base_alloc,
              "mask_bytes": 0, "note": "workspace is O(B*S + B*H*S + slots*Sc*D); no (query, key) mask in memory"}
    stream = torch.cuda.current_stream(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local) if rank == 0 else None
    torch.cuda.synchronize(dev)
    barrier(dist)
    if clocks:
        clocks.start()
        time.sleep(0.3)
    hca.hca_profile_enable(True)
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    prof = hca.hca_profile_read()
    hca.hca_profile_enable(False)
    barrier(dist)
    ms_total = ev0.elapsed_time(ev1)
    clk = clocks.stop() if clocks else None
    ms_total = max_over_ranks(ms_total, dist, dev)
    ms_step = ms_total / args.steps
    value = (flop_fwd + flop_bwd) * world / (ms_step * 1e-3) / 1e12

    # per-kernel share and the dominant kernel's roofline
    launches = sum(n for n, _ in prof.values())
    tot_ms = sum(ms for _, ms in prof.values()) or 1.0
    kernels = {k: {"launches": n, "ms_total": round(ms, 4), "share": round(ms / tot_ms, 4)}
               for k, (n, ms) in prof.items() if n}
    dom = max((k for k in kernels if k in KERNEL_FLOP_PER_PAIR_D), key=lambda k: kernels[k]["ms_total"])
    n_dom, ms_dom = prof[dom]
    avg_ms = ms_dom / n_dom
    alg_flops = KERNEL_FLOP_PER_PAIR_D[dom] * w.D * pairs
    peaks, peak_src = load_peaks()
    # the timed region is ~0.1 s of few-ms steps at unthrottled clocks: the
    # burst GEMM figure is the matching denominator (the sustained one was
    # taken over seconds under the power cap)
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    achieved = alg_flops / (avg_ms * 1e-3) / 1e12
    roofline = {"bound": "tensor", "kernel": dom, "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4), "traffic": profiled_traffic(dom, w.name),
                "peak_source": f"{peak_src} bf16_tflops (burst)",
                "algorithmic": f"{KERNEL_FLOP_PER_PAIR_D[dom]}*D FLOP per visible pair-head x {pairs} pair-heads"}
    per_kernel_roof = {}
    for k, fpd in KERNEL_FLOP_PER_PAIR_D.items():
        n_k, ms_k = prof.get(k, (0, 0.0))
        if n_k:
            ach = fpd * w.D * pairs / (ms_k / n_k * 1e-3) / 1e12
            per_kernel_roof[k] = {"ms_per_launch": round(ms_k / n_k, 4), "achieved": round(ach, 2),
                                  "frac": round(ach / peak, 4), "flop_per_pair_head": f"{fpd}*D"}
    roofline["per_kernel"] = per_kernel_roof
    per_phase = {}
    fwd_ms = prof.get("hca_fwd_tc", (0, 0.0))[1] / args.steps
    bwd_ms = sum(prof.get(k, (0, 0.0))[1] for k in ("hca_bwd_dq", "hca_bwd_dkv", "hca_bwd_reduce")) / args.steps
    burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    if fwd_ms > 0:
        per_phase["fwd"] = {"ms": round(fwd_ms, 4), "tflops": round(flop_fwd / fwd_ms / 1e9, 2),
                            "pct_bf16_peak": round(100 * flop_fwd / fwd_ms / 1e9 / burst, 2)}
    if bwd_ms > 0:
        per_phase["bwd"] = {"ms": round(bwd_ms, 4), "tflops": round(flop_bwd / bwd_ms / 1e9, 2),
                            "pct_bf16_peak": round(100 * flop_bwd / bwd_ms / 1e9 / burst, 2)}

    # end to end: host buffers in, results back to host, through the API
    e2e = run_e2e(args, w, q, kv, ckv, dout, dev, dist, flop_fwd + flop_bwd, world)

    sm_mhz = (clk or {}).get("sm_mhz") or 2070.0
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    ex2_rate = EX2_PER_CLK_PER_SM * n_sm * sm_mhz * 1e6
    mufu = {"unit": "exp/s", "peak": ex2_rate, "peak_source": "32 ex2.approx per clock per SM (probe) x SMs x sm_mhz"}
    for ph, ph_ms in (("fwd", fwd_ms), ("bwd", bwd_ms)):
        n_exp = EXP_PER_PAIR[ph] * pairs
        mufu[ph] = {"exp": n_exp, "floor_ms": round(n_exp / ex2_rate * 1e3, 4),
                    "tensor_floor_ms": round((flop_fwd if ph == "fwd" else flop_bwd) / (burst * 1e12) * 1e3, 4),
                    "frac": round(n_exp / (ph_ms * 1e-3) / ex2_rate, 4) if ph_ms > 0 else None}
    line = {"metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": config_dict(w),
            "pct_bf16_peak": round(100 * value / world / burst, 2), "peak_tflops": burst,
            "phases": per_phase, "kernels": kernels, "gpu_launches": launches, "roofline": roofline,
            "secondary_roof_exp": mufu, "memory": memory,
            "clocks": clk, "e2e": e2e}
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, q, kv, ckv, dout, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def run_e2e(args, w, q, kv, ckv, dout, dev, dist, flops_step, world):
    """The same fwd+bwd step end to end through the public API: every step
    copies its inputs from pinned host memory to the device and every output
    back.  Steps are pipelined over three streams with two device buffer sets
    (inputs of step k+1 go up and outputs of step k-1 come down while step k
    computes), as a training loop that feeds the op from the host would."""
    import torch
    from block_sparse_compressed_gb300 import hca
    hin = [x.cpu().pin_memory() for x in (q, kv, ckv, dout)]
    hout = [torch.empty(q.shape, dtype=q.dtype).pin_memory(), torch.empty(w.B, w.H, w.S).pin_memory(),
            torch.empty(q.shape, dtype=q.dtype).pin_memory(), torch.empty(kv.shape, dtype=kv.dtype).pin_memory(),
            torch.empty(ckv.shape, dtype=ckv.dtype).pin_memory()]
    gin = [[torch.empty_like(x) for x in (q, kv, ckv, dout)] for _ in range(2)]
    gout = [[torch.empty_like(q), torch.empty(w.B, w.H, w.S, dtype=torch.float32, device=dev), torch.empty_like(q),
             torch.empty_like(kv), torch.empty_like(ckv)] for _ in range(2)]
    wsf = hca.workspace(w.B, w.H, w.S, w.D, w.W, w.m, w.dtype, False, dev)
    wsb = hca.workspace(w.B, w.H, w.S, w.D, w.W, w.m, w.dtype, True, dev)
    h2d = sum(x.numel() * x.element_size() for x in hin)
    d2h = sum(x.numel() * x.element_size() for x in hout)
    s_in, s_comp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    in_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]

    def step(k):
        b = k & 1
        gq, gkv, gckv, gdo = gin[b]
        out, lse, dq_, dkv_, dckv_ = gout[b]
        with torch.cuda.stream(s_in):
            if k >= 2:
                s_in.wait_event(comp_done[b])  # step k-2 has finished reading these inputs
            for g, h in zip(gin[b], hin):
                g.copy_(h, non_blocking=True)
            in_done[b].record(s_in)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(in_done[b])
            if k >= 2:
                s_comp.wait_event(out_done[b])  # step k-2's outputs have been copied out
            hca.hca_attn_fwd(gq, gkv, gckv, None, w.W, w.m, w.scale, out=out, lse=lse, ws=wsf)
            hca.hca_attn_bwd(gq, gkv, gckv, None, out, lse, gdo, w.W, w.m, w.scale, dq=dq_, dkv=dkv_, dckv=dckv_,
                             ws=wsb)
            comp_done[b].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[b])
            for h, g in zip(hout, gout[b]):
                h.copy_(g, non_blocking=True)
            out_done[b].record(s_out)

    for k in range(2):
        step(k)
    torch.cuda.synchronize(dev)
    steps = max(4, args.steps)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist)
    e0.record(s_in)
    for k in range(steps):
        step(k)
    s_out.wait_event(out_done[(steps - 1) & 1])
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(e0.elapsed_time(e1), dist, dev) / steps
    return {"value": round(flops_step * world / (ms * 1e-3) / 1e12, 3), "unit": UNIT, "ms_per_step": round(ms, 3),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "path": "pinned host tensors -> hca_attn_fwd/hca_attn_bwd (C ABI) -> pinned host tensors, "
                    "copies of neighbouring steps overlapped with compute on three streams"}


def run_local(args):
    """Local sliding-window attention (no compressed set) on the headline
    shape: same timing rules, FLOPs over the raw visible pairs."""
    import torch
    from block_sparse_compressed_gb300 import hca
    from block_sparse_compressed_gb300 import inputs as I
    w = workload()
    dev = torch.device("cuda", 0)
    q, kv, _, seg, dout = I.tensors(w, device=dev)
    raw, _ = visible_pairs_closed_form(w.S, w.W, w.S + 1)
    pairs = raw * w.H * w.B
    out = torch.empty_like(q)
    lse = torch.empty(w.B, w.H, w.S, dtype=torch.float32, device=dev)
    dq, dkv = torch.empty_like(q), torch.empty_like(kv)
    wsf = hca.local_workspace(w.B, w.H, w.S, w.D, w.W, w.dtype, False, dev)
    wsb = hca.local_workspace(w.B, w.H, w.S, w.D, w.W, w.dtype, True, dev)

    def step():
        hca.hca_local_attn_fwd(q, kv, seg, w.W, w.scale, out=out, lse=lse, ws=wsf)
        hca.hca_local_attn_bwd(q, kv, seg, out, lse, dout, w.W, w.scale, dq=dq, dkv=dkv, ws=wsb)

    for _ in range(max(1, args.warmup)):
        step()
    if hca.hca_workspace_status(wsf) != 0 or hca.hca_workspace_status(wsb) != 0:
        raise RuntimeError("device reported an error status")
    stream = torch.cuda.current_stream(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    hca.hca_profile_enable(True)
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    prof = hca.hca_profile_read()
    hca.hca_profile_enable(False)
    ms = ev0.elapsed_time(ev1) / args.steps
    flops = 14 * w.D * pairs
    fwd_ms = prof.get("hca_fwd_tc", (0, 0.0))[1] / args.steps
    bwd_ms = sum(prof.get(k, (0, 0.0))[1] for k in ("hca_bwd_dq", "hca_bwd_dkv", "hca_bwd_reduce")) / args.steps
    line = {"metric": "LOCAL_SLIDING attn fwd+bwd TFLOP/s (visible pairs) at S=65536", "value": round(
        flops / (ms * 1e-3) / 1e12, 3), "unit": UNIT, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 4), "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"local fwd+bwd bf16 B{w.B} H{w.H} S{w.S} D{w.D} W{w.W}", "pairs_per_head": raw},
        "phases": {"fwd": {"ms": round(fwd_ms, 4), "tflops": round(4 * w.D * pairs / fwd_ms / 1e9, 2)},
                   "bwd": {"ms": round(bwd_ms, 4), "tflops": round(10 * w.D * pairs / bwd_ms / 1e9, 2)}},
        "kernels": {k: {"launches": n, "ms_total": round(t, 4)} for k, (n, t) in prof.items() if n}}
    print(json.dumps(line), flush=True)
    return 0


def _time_cuda(fn, steps, warmup):
    import torch
    for _ in range(max(3, warmup)):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def run_compress(args):
    """HCA compressor forward and backward on 16 sequences of the headline
    length (kv [16, 65536, 128] bf16, 268 MB: above L2, so no flush needed);
    HBM-bound, reported against the measured copy bandwidth."""
    import torch
    from block_sparse_compressed_gb300 import hca
    from block_sparse_compressed_gb300 import inputs as I
    B, S, D, m = 16, 65536, 128, 128
    dev = torch.device("cuda", 0)
    x = I.normal((B, S, D), 1, torch.bfloat16, dev)
    g = I.normal((B, S), 2, torch.float32, dev)
    bias = I.normal((m,), 3, torch.float32, dev)
    Sc = S // m
    dck = I.normal((B, Sc, D), 4, torch.bfloat16, dev)
    ckv = torch.empty(B, Sc, D, dtype=torch.bfloat16, device=dev)
    dx, dg, db = torch.empty_like(x), torch.empty_like(g), torch.empty_like(bias)
    ws = torch.empty(hca.load().hca_compress_workspace_size(B, S, m), dtype=torch.uint8, device=dev)
    f_ms = _time_cuda(lambda: hca.hca_compress_fwd(x, g, bias, None, m, ckv=ckv), args.steps, args.warmup)
    b_ms = _time_cuda(lambda: hca.hca_compress_bwd(x, g, bias, None, m, dck, dx=dx, dg=dg, dbias=db, ws=ws),
                      args.steps, args.warmup)
    fwd_bytes = x.numel() * 2 + g.numel() * 4 + ckv.numel() * 2
    # backward: x and g read, dckv read, dx and dg written, per-window logit grads written + read
    bwd_bytes = x.numel() * 2 + g.numel() * 4 + dck.numel() * 2 + dx.numel() * 2 + dg.numel() * 4 + 2 * 4 * B * S
    peaks, src = load_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    line = {"metric": "HCA compressor GB/s (algorithmic bytes) fwd and bwd", "unit": "GB/s",
            "value": round(fwd_bytes / f_ms / 1e6, 1), "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"compressor B{B} S{S} D{D} m{m}"},
            "fwd": {"ms": round(f_ms, 4), "bytes": fwd_bytes, "gbs": round(fwd_bytes / f_ms / 1e6, 1),
                    "frac_hbm": round(fwd_bytes / f_ms / 1e6 / hbm, 4)},
            "bwd": {"ms": round(b_ms, 4), "bytes": bwd_bytes, "gbs": round(bwd_bytes / b_ms / 1e6, 1),
                    "frac_hbm": round(bwd_bytes / b_ms / 1e6 / hbm, 4)},
            "peak_hbm_gbs": hbm, "peak_source": f"{src} hbm_gbs"}
    print(json.dumps(line), flush=True)
    return 0


def run_indexer(args):
    """Lightning Indexer scores + top-k on the CSA shape: S = 65536, m = 4
    (16384 compressed entries), 64 index heads of dim 128, k = 512."""
    import torch
    from block_sparse_compressed_gb300 import hca
    from block_sparse_compressed_gb300 import inputs as I
    B, S, Hi, m, k = 1, 65536, 64, 4, 512
    dev = torch.device("cuda", 0)
    Sc = S // m
    qi = I.normal((B, S, Hi, 128), 1, torch.bfloat16, dev)
    ki = I.normal((B, Sc, 128), 2, torch.bfloat16, dev)
    w = I.normal((B, S, Hi), 3, torch.float32, dev)
    ws = torch.empty(hca.load().hca_indexer_workspace_size(B, S, m), dtype=torch.uint8, device=dev)
    hca.hca_profile_enable(True)
    ms = _time_cuda(lambda: hca.hca_indexer_topk(qi, ki, w, None, m, k, ws=ws), args.steps, args.warmup)
    prof = hca.hca_profile_read()
    hca.hca_profile_enable(False)
    # visible (query, entry) pairs: entry j is complete at query (j+1)m-1
    q_, r_ = divmod(S, m)
    pairs = m * q_ * (q_ - 1) // 2 + q_ * (r_ + 1)
    flops_def = 2 * Hi * 128 * pairs   # the per-head definition
    flops_gemm = 2 * 128 * pairs       # after collapsing the heads (what the GEMM executes on visible pairs)
    line = {"metric": "Lightning Indexer scores + top-k, ms per call", "unit": "ms", "value": round(ms, 4),
            "higher_is_better": False, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"indexer B{B} S{S} Hi{Hi} Di128 m{m} k{k}"},
            "visible_pairs": pairs, "definition_tflops": round(flops_def / ms / 1e9, 2),
            "collapsed_gemm_tflops": round(flops_gemm / ms / 1e9, 2),
            "kernels": {kk: {"launches": n, "ms_total": round(t, 4)} for kk, (n, t) in prof.items() if n}}
    print(json.dumps(line), flush=True)
    return 0


def run_csa(args):
    """Compressed sparse attention forward + backward: B=1, H=64, S=65536,
    D=128, W=128, m=4 (16384 compressed entries), k=256 selected entries per
    query (uniform random among the completed ones, with repeats and
    padding: the indexer's output on random inputs has no locality either).
    FLOPs over visible pairs as the HCA metric (4*D fwd, 10*D bwd per pair
    and head)."""
    import torch
    from block_sparse_compressed_gb300 import hca
    from block_sparse_compressed_gb300 import inputs as I
    B, H, S, D, W, m, k = 1, 64, 65536, 128, 128, 4, 256
    dev = torch.device("cuda", 0)
    w = I.Workload(f"csa fwd+bwd bf16 B{B} H{H} S{S} D{D} W{W} m{m} k{k}", B, H, S, D, W, m, torch.bfloat16)
    q, kv, ckv, seg, dout = I.tensors(w, device=dev)
    sel = I.random_selection(B, S, m, k, 77, extra=0).to(dev)
    # visible pairs per head: raw window + distinct selected entries that are complete
    i = torch.arange(S, device=dev)
    srt = torch.sort(sel[0].long(), dim=1).values
    valid = (srt >= 0) & (srt <= ((i + 1) // m - 1)[:, None])
    first = torch.ones_like(valid)
    first[:, 1:] = srt[:, 1:] != srt[:, :-1]
    comp_pairs = int((valid & first).sum().item())
    raw_pairs, _ = visible_pairs_closed_form(S, W, m)
    pairs = (raw_pairs + comp_pairs) * H
    out = torch.empty_like(q)
    lse = torch.empty(B, H, S, dtype=torch.float32, device=dev)
    dq, dkv, dckv = torch.empty_like(q), torch.empty_like(kv), torch.empty_like(ckv)
    wsf = hca.csa_workspace(B, H, S, D, W, m, k, torch.bfloat16, False, dev)
    wsb = hca.csa_workspace(B, H, S, D, W, m, k, torch.bfloat16, True, dev)

    def fwd():
        hca.hca_csa_attn_fwd(q, kv, ckv, None, sel, W, m, w.scale, out=out, lse=lse, ws=wsf)

    def bwd():
        hca.hca_csa_attn_bwd(q, kv, ckv, None, sel, out, lse, dout, W, m, w.scale, dq=dq, dkv=dkv, dckv=dckv, ws=wsb)

    fwd()
    bwd()
    if hca.hca_workspace_status(wsf) != 0 or hca.hca_workspace_status(wsb) != 0:
        raise RuntimeError("device reported an error status")
    hca.hca_profile_enable(True)
    f_ms = _time_cuda(fwd, args.steps, args.warmup)
    b_ms = _time_cuda(bwd, args.steps, args.warmup)
    prof = hca.hca_profile_read()
    hca.hca_profile_enable(False)
    peaks, src = load_peaks()
    burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    ff, fb = 4 * D * pairs, 10 * D * pairs
    line = {"metric": "CSA attn fwd+bwd TFLOP/s (visible pairs) at S=65536", "unit": "TFLOP/s",
            "value": round((ff + fb) / ((f_ms + b_ms) * 1e-3) / 1e12, 3), "higher_is_better": True, "dtype": "bf16",
            "data": "synthetic", "config": {"workload": w.name, "selected_pairs_per_head": comp_pairs,
                                            "raw_pairs_per_head": raw_pairs},
            "fwd": {"ms": round(f_ms, 4), "tflops": round(ff / f_ms / 1e9, 2),
                    "pct_bf16_peak": round(100 * ff / f_ms / 1e9 / burst, 2)},
            "bwd": {"ms": round(b_ms, 4), "tflops": round(fb / b_ms / 1e9, 2),
                    "pct_bf16_peak": round(100 * fb / b_ms / 1e9 / burst, 2)},
            "kernels": {kk: {"launches": n, "ms_total": round(t, 4)} for kk, (n, t) in prof.items() if n}}
    print(json.dumps(line), flush=True)
    return 0


def run_ncu_case(args):
    """One small run of a path for a profiler capture (S = --ncu-case): the
    HCA fwd+bwd by default, else the path --mode names."""
    import torch
    from block_sparse_compressed_gb300 import hca
    from block_sparse_compressed_gb300 import inputs as I
    S = args.ncu_case
    dev = torch.device("cuda", 0)
    if args.mode == "compress":
        B, D, m = 4, 128, 128
        x = I.normal((B, S, D), 1, torch.bfloat16, dev)
        g = I.normal((B, S), 2, torch.float32, dev)
        bias = I.normal((m,), 3, torch.float32, dev)
        for _ in range(args.warmup + 1):
            ckv = hca.hca_compress_fwd(x, g, bias, None, m)
            hca.hca_compress_bwd(x, g, bias, None, m, ckv)
        torch.cuda.synchronize()
        print(json.dumps({"ncu_case": f"compressor B{B} S{S} D{D} m{m}", "ok": True}))
        return 0
    if args.mode == "indexer":
        Hi, m, k = 64, 4, 512
        qi = I.normal((1, S, Hi, 128), 1, torch.bfloat16, dev)
        ki = I.normal((1, (S + m - 1) // m, 128), 2, torch.bfloat16, dev)
        wt = I.normal((1, S, Hi), 3, torch.float32, dev)
        for _ in range(args.warmup + 1):
            hca.hca_indexer_topk(qi, ki, wt, None, m, k)
        torch.cuda.synchronize()
        print(json.dumps({"ncu_case": f"indexer B1 S{S} Hi{Hi} Di128 m{m} k{k}", "ok": True}))
        return 0
    if args.mode == "csa":
        H, D, W, m, k = 64, 128, 128, 4, 256
        w = I.Workload(f"csa fwd+bwd bf16 B1 H{H} S{S} D{D} W{W} m{m} k{k}", 1, H, S, D, W, m, torch.bfloat16)
        q, kv, ckv, _, dout = I.tensors(w, device=dev)
        sel = I.random_selection(1, S, m, k, 77, extra=0).to(dev)
        for _ in range(args.warmup + 1):
            out, lse = hca.hca_csa_attn_fwd(q, kv, ckv, None, sel, W, m, w.scale)
            hca.hca_csa_attn_bwd(q, kv, ckv, None, sel, out, lse, dout, W, m, w.scale)
        torch.cuda.synchronize()
        print(json.dumps({"ncu_case": w.name, "ok": True}))
        return 0
    base = workload()
    w = I.Workload(f"fwd+bwd bf16 B1 H64 S{args.ncu_case} D128 W128 m128", base.B, base.H, args.ncu_case, base.D,
                   base.W, base.m, base.dtype)
    q, kv, ckv, seg, dout = I.tensors(w, device="cuda")
    for _ in range(args.warmup + 1):
        out, lse = hca.hca_attn_fwd(q, kv, ckv, seg, w.W, w.m, w.scale)
        hca.hca_attn_bwd(q, kv, ckv, seg, out, lse, dout, w.W, w.m, w.scale)
    torch.cuda.synchronize()
    print(json.dumps({"ncu_case": w.name, "ok": True}))
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.ncu_case:
        return run_ncu_case(args)
    if args.impl == "reference":
        return run_reference(args)
    if args.mode == "local":
        return run_local(args)
    if args.mode == "compress":
        return run_compress(args)
    if args.mode == "indexer":
        return run_indexer(args)
    if args.mode == "csa":
        return run_csa(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
