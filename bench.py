"""Benchmark of the EXL3 trellis linear hot path on one GB300 (or N replicas).

Workload: the decode-shaped merged gate/up projection, hidden 5120 -> 2 x 17408,
gate coded at K=2 and up at K=3, written into two column slices of one bf16
out[M, 34816], M = 8 tokens (seeded synthetic data, uniform int16 code words).
A step = both shards through the C ABI (pre-transform, fused trellis GEMM,
output transform into the slice).  Metric: tokens/s (M per step); the roofline
object reports the decode GEMM kernel's HBM bandwidth on code bytes.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--m M] [--impl ours|reference]

Under torchrun each rank runs an independent replica on its own GPU (the path
shards without a data-path collective); value = all ranks' tokens / max time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

IC, OC, KS = 5120, 17408, (2, 3)
METRIC = "EXL3 linear tokens/s (decode-shaped gate_up, M<=8)"
L2_BYTES = 129 * 2 ** 20


def code_bytes(K, ic=IC, oc=OC):
    return ic * oc * K // 8


def algorithmic_bytes(M, K, ic=IC, oc=OC):
    """Bytes one decode GEMM launch must move: code words, activations in, bf16 out, scales."""
    return code_bytes(K, ic, oc) + 2 * M * ic + 2 * M * oc + 2 * 2 * oc


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


# ------------------------------------------------------------------ dist
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ ours
def run_ours(args):
    import torch
    import moe_gemm_exl3_gb300 as m
    from moe_gemm_exl3_gb300 import build as b
    import synthetic as syn

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    b.build()
    M = args.m

    x, shards = syn.gate_up(1, M=M)
    # rotate through enough copies of the code words that every step streams from HBM
    per_step_code = sum(code_bytes(K) for K in KS)
    R = max(4, int(np.ceil(4 * L2_BYTES / per_step_code)))
    codes = [[torch.from_numpy(s.code).to(dev) for s in shards]]
    for _ in range(R - 1):
        codes.append([c.clone() for c in codes[0]])
    scal = [[torch.from_numpy(v.view(np.int16)).to(dev).view(torch.float16)
             for v in (s.s_in, s.rin, s.rout, s.s_out)] for s in shards]
    xd = torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16)
    out = torch.empty((M, 2 * OC), dtype=torch.bfloat16, device=dev)

    # one merged-layer call per step: both shards, each with its own K and scales
    shard_sets = [[(codes[r][i], sh.K, *scal[i], i * OC) for i, sh in enumerate(shards)] for r in range(R)]
    ws = m.workspace(m.exl3_linear_shards_workspace_bytes(M, IC, shard_sets[0]), dev)

    def step(r, xin=None, o=None):
        xin = xd if xin is None else xin
        o = out if o is None else o
        m.exl3_linear_into_shards(xin, shard_sets[r], o, ws)

    # pre-transform + one grouped GEMM per 32 rows
    launches_per_step = 1 + (M + 31) // 32

    # capture R steps (one per code copy) in one CUDA graph
    stream = torch.cuda.Stream(dev)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for r in range(R):
            step(r)                          # eager warm-up of every path
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for r in range(R):
                step(r)
    torch.cuda.synchronize()

    steps = max(R, (args.steps // R) * R)
    reps = steps // R
    warm = max(1, -(-args.warmup // R))
    with torch.cuda.stream(stream):
        for _ in range(warm):
            g.replay()
    torch.cuda.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with Clocks(local) as clk:
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    ms = e0.elapsed_time(e1)
    if world > 1:
        t = torch.tensor([ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    ms_step = ms / steps
    value = world * M * steps / (ms / 1e3)

    # ---- roofline: the step's grouped trellis GEMM kernel alone (exl3_gemm_into_shards is
    # that one launch for M <= 32), timed with events on its stream; the stream is kept
    # busy so no launch gap is measured
    u = torch.empty((len(shards), M, IC), dtype=torch.float16, device=dev)
    for i in range(len(shards)):
        m.exl3_pretransform(xd, *scal[i][:2], u=u[i])
    n_k = 4 * R
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_k)]
    with torch.cuda.stream(stream):
        torch.cuda._sleep(50_000_000)
        for j in range(n_k):
            evs[j][0].record(stream)
            m.exl3_gemm_into_shards(u, shard_sets[j % R], out, ws)
            evs[j][1].record(stream)
    torch.cuda.synchronize()
    dur_ms = statistics.mean(a.elapsed_time(b2) for a, b2 in evs[n_k // 4:])
    hbm_peak, bf16_peak, peak_src = peaks()
    alg = sum(algorithmic_bytes(M, K) for K in KS)
    achieved = alg / (dur_ms * 1e-3) / 1e9
    roof = {"bound": "hbm", "kernel": "group_gemm_kernel (gate K=2 + up K=3 in one launch)",
            "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
            "frac": round(achieved / hbm_peak, 4), "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)",
            "traffic": traffic_from_profile(), "per_launch_us": round(dur_ms * 1e3, 2),
            "algorithmic_bytes_per_launch": alg,
            "code_GBps": round(sum(code_bytes(K) for K in KS) / (dur_ms * 1e-3) / 1e9, 1)}

    # ---- end to end through the public API with host buffers
    xh = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory()
    oh = torch.empty((M, 2 * OC), dtype=torch.bfloat16).pin_memory()
    xdev = torch.empty_like(xd)
    e2e_steps = max(R, min(steps, 20 * R))
    with torch.cuda.stream(stream):
        for r in range(R):
            xdev.copy_(xh, non_blocking=True)
            step(r, xdev)
            oh.copy_(out, non_blocking=True)
        torch.cuda.synchronize()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for i in range(e2e_steps):
            xdev.copy_(xh, non_blocking=True)
            step(i % R, xdev)
            oh.copy_(out, non_blocking=True)
        a1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = a0.elapsed_time(a1)
    e2e_val = M * e2e_steps / (e2e_ms / 1e3)
    if world > 1:
        t = torch.tensor([e2e_ms / e2e_steps], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_val = world * M / (float(t.item()) / 1e3)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
            "steps": steps, "warmup": warm * R, "ms_per_step": round(ms_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f16",
            "data": "synthetic (seeded; uniform int16 code words, x ~ N(0,1))",
            "config": {"workload": "gate_up 5120->2x17408, K=2|K=3, M=%d, out[M,34816]" % M,
                       "M": M, "IC": IC, "OC_per_shard": OC, "K": list(KS),
                       "l2": f"inputs larger than L2: {R} rotating code copies "
                             f"({R * per_step_code / 1e6:.0f} MB)",
                       "timing": "CUDA graph of %d steps, replayed; CUDA events" % R,
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "gpu_launches": launches_per_step * steps,
            "roofline": roof,
            "e2e": {"value": round(e2e_val, 1), "unit": "tokens/s",
                    "h2d_bytes_per_step": int(xh.numel() * 2), "d2h_bytes_per_step": int(oh.numel() * 2),
                    "note": "exl3_linear_into_shards (one call for both shards), x copied from pinned host "
                            "memory and out read back every step, eager launches"},
            "clocks": clk.summary(),
        }
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = cpu_baseline(M, budget_s=args.cpu_budget)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def traffic_from_profile():
    """DRAM bytes per launch from the committed ncu summary, if it matches the current kernel."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "decode_gemm_gate_up_m8.json")
    src = os.path.join(ROOT, "moe_gemm_exl3_gb300", "csrc", "linear.cu")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    with open(src, "rb") as f:
        h = hashlib.sha256(f.read()).hexdigest()[:16]
    if d.get("source_sha256_16") != h:
        return None
    return d.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ oracle
def cpu_baseline(M, budget_s=15.0, seed=1):
    """The CPU oracle on a bounded sample of the workload, scaled to tokens/s."""
    import oracle
    import synthetic as syn
    x, shards = syn.gate_up(seed, M=M)
    nblk_total = OC // 128
    oracle.lib()
    # time one block per shard, then size the sample to the budget
    t0 = time.perf_counter()
    for sh in shards:
        oracle.linear_f64(x, sh.code, sh.K, sh.s_in, sh.rin, sh.rout, sh.s_out, blk0=0, nblk=1)
    per_blk = (time.perf_counter() - t0) / 2
    nblk = int(min(nblk_total, max(1, budget_s / max(per_blk, 1e-6) / 2)))
    t0 = time.perf_counter()
    for sh in shards:
        oracle.linear_f64(x, sh.code, sh.K, sh.s_in, sh.rin, sh.rout, sh.s_out, blk0=0, nblk=nblk)
    t = time.perf_counter() - t0
    full = t * nblk_total / nblk
    return {"value": round(M / full, 3), "unit": "tokens/s", "cores": _omp_threads(),
            "kind": "oracle",
            "sample": f"M={M}, output blocks 0..{nblk - 1} of {nblk_total} (128 columns each) of both "
                      f"shards in {t:.1f} s, scaled linearly to all {nblk_total} blocks"}


def _omp_threads():
    n = os.environ.get("OMP_NUM_THREADS")
    return int(n) if n else os.cpu_count()


def run_reference(args):
    """The oracle as the reference arm: same metric and workload, each step a bounded
    sample (whole 128-column output blocks of both shards), scaled to the full step."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    M = args.m
    import oracle
    import synthetic as syn
    x, shards = syn.gate_up(1, M=M)
    nblk_total = OC // 128
    oracle.lib()

    def one(nblk):
        for sh in shards:
            oracle.linear_f64(x, sh.code, sh.K, sh.s_in, sh.rin, sh.rout, sh.s_out, blk0=0, nblk=nblk)

    t0 = time.perf_counter()
    one(1)
    per_blk = time.perf_counter() - t0
    K, W = args.steps, args.warmup
    budget = args.ref_budget
    # blocks per step so that W + K steps fit the budget; at least one block per step,
    # and if even that does not fit, fewer steps are executed (reported as such)
    nblk = int(max(1, min(nblk_total, budget / max(1, K + W) / per_blk)))
    run_steps = int(max(1, min(K, budget / (nblk * per_blk) - min(W, 1))))
    for _ in range(min(W, 1)):
        one(nblk)
    t0 = time.perf_counter()
    for _ in range(run_steps):
        one(nblk)
    t = (time.perf_counter() - t0) / run_steps * nblk_total / nblk
    v = M / t
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 3), "unit": "tokens/s",
            "n_gpus": 1, "steps": run_steps, "steps_requested": K, "warmup": min(W, 1),
            "ms_per_step": round(t * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": {"workload": "gate_up 5120->2x17408, K=2|K=3, M=%d, out[M,34816]" % M, "M": M},
            "cpu_baseline": {"value": round(v, 3), "unit": "tokens/s", "cores": _omp_threads(),
                             "kind": "oracle",
                             "sample": f"each step: output blocks 0..{nblk - 1} of {nblk_total} (128 columns) "
                                       f"of both shards, scaled linearly to the full step"},
            "e2e": {"value": round(v, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--m", type=int, default=8)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--ref-budget", type=float, default=90.0, help="seconds of oracle work")
    args = ap.parse_args()
    if args.steps is None:
        args.steps = 50000
    if args.warmup is None:
        args.warmup = 200
    args.warmup = max(3, args.warmup)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
