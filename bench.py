"""Benchmark of the EXL3 trellis hot path on one GB300 (or N replicas).

Default workload (the headline): the decode-shaped merged gate/up projection,
hidden 5120 -> 2 x 17408, gate coded at K=2 and up at K=3, written into two
column slices of one bf16 out[M, 34816], M = 8 tokens, seeded synthetic data.
A step = one merged-layer call through the C ABI (pre-transform, grouped fused
trellis GEMM, output transform into the slices).  Metric: tokens/s.

Other workloads (--workload): prefill (5120 -> 17408 at M = 8192, K per
--k), moe (128 experts, H 2048, I 768, top-8, T tokens per --t), gather
(8192 ids from a 248,320 x 5120 int8 table), layer (the five projections of a
hidden-5120 decoder layer at --m rows), lm_head (that int8 table as the output
projection at --m rows).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload W] [--impl ours|reference]

Under torchrun each rank runs an independent replica on its own GPU (the path
shards without a data-path collective); value = all ranks' units / max time.
"""
from __future__ import annotations

import argparse
import hashlib
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

L2_BYTES = 129 * 2 ** 20


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def sustained_tflops():
    """Dense bf16 TFLOP/s held for seconds under the power cap (the denominator for a
    tensor-bound kernel timed inside a long run of steps)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        if "bf16_tflops_sustained" in d:
            return float(d["bf16_tflops_sustained"]), "measured"
    return 1700.0, "fallback"


def dist_env():
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def omp_threads():
    n = os.environ.get("OMP_NUM_THREADS")
    return int(n) if n else os.cpu_count()


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index, self.proc, self.lines = index, None, []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
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


def kernel_time_ms(torch, stream, fn, n, reps=4):
    """Mean duration of fn(j) (the launches of one call), j = 0..n-1, in the launch
    configuration of the timed steps: the n calls are captured in one CUDA graph,
    which is replayed `reps` times between two CUDA events on `stream`."""
    with torch.cuda.stream(stream):
        for j in range(n):
            fn(j)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for j in range(n):
            fn(j)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        g.replay()
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / (reps * n)


def profile_traffic(name):
    """DRAM bytes per launch from a committed ncu record, if the source files it lists
    (the kernel's own) still hash to what they were when it was captured."""
    p = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if not d.get("source_files"):
        return None
    h = hashlib.sha256()
    for s in d["source_files"]:
        with open(os.path.join(ROOT, "moe_gemm_exl3_gb300", "csrc", s), "rb") as f:
            h.update(f.read())
    if d.get("source_sha256_16") != h.hexdigest()[:16]:
        return None
    return d.get("dram_bytes_per_launch")


def max_over_ranks(torch, dist, value, device):
    """The largest value over all ranks (every rank gets it); the value itself without a group."""
    if dist is None:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world, units_per_step, steps, max_ms):
    """Whole-job throughput: the units all ranks processed over the slowest rank's time."""
    return world * units_per_step * steps / (max_ms / 1e3)


def t16(torch, a, dev, dtype):
    a = np.ascontiguousarray(a)
    if dtype in (torch.bfloat16, torch.float16):
        a = a.view(np.int16)
    return torch.from_numpy(a).to(dev).view(dtype)


# ------------------------------------------------------------------ workloads
def gemm_path(M):
    """The GEMM path the library takes for M rows (the C-ABI's default choice)."""
    return "decode" if M <= 16 else ("fused" if M <= 128 else "prefill")


def decode_kernel(torch, M, OCs):
    """The decode-mode kernel of a merged call: the paired one (a 16-warp CTA per
    column group of each of two equal shards) at up to 16 rows, when each shard
    has more column groups than half the SMs and no more than the SMs."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    g = OCs[0] // 128
    if M <= 16 and len(OCs) == 2 and OCs[0] == OCs[1] and sms < 2 * g and g <= sms:
        return "group_pair_kernel"
    return "group_gemm_kernel"


def linear_launches(M, n_shards):
    """Kernel launches of one linear call: the pre-transform plus the GEMM path's."""
    return 1 + (2 * n_shards if gemm_path(M) == "prefill" else 1)


class GateUp:
    """Decode-shaped merged gate (K=2) / up (K=3) projection, 5120 -> 2 x 17408."""
    IC, OC, KS = 5120, 17408, (2, 3)

    def __init__(self, args):
        self.M = args.m
        self.metric = "EXL3 linear tokens/s (decode-shaped gate_up, M<=8)"
        self.unit = "tokens/s"
        self.units_per_step = self.M

    def config(self):
        return {"workload": f"gate_up 5120->2x17408, K=2|K=3, M={self.M}, out[M,34816]", "M": self.M,
                "IC": self.IC, "OC_per_shard": self.OC, "K": list(self.KS)}

    def code_bytes(self, K):
        return self.IC * self.OC * K // 8

    _codes = {}   # device code copies, shared by every M of one run

    def setup(self, torch, m, syn, dev):
        M, IC, OC = self.M, self.IC, self.OC
        self.x, shards = syn.gate_up(1, M=M)
        per_step = sum(self.code_bytes(K) for K in self.KS)
        self.R = R = max(4, int(np.ceil(4 * L2_BYTES / per_step)))
        codes = GateUp._codes.get(R)
        if codes is None:
            codes = [[t16(torch, s.code, dev, torch.int16) for s in shards]]
            for _ in range(R - 1):
                codes.append([c.clone() for c in codes[0]])
            GateUp._codes[R] = codes
        scal = [[t16(torch, v, dev, torch.float16) for v in (s.s_in, s.rin, s.rout, s.s_out)] for s in shards]
        self.sets = [[(codes[r][i], s.K, *scal[i], i * OC) for i, s in enumerate(shards)] for r in range(R)]
        self.xd = t16(torch, self.x, dev, torch.bfloat16)
        self.out = torch.empty((M, 2 * OC), dtype=torch.bfloat16, device=dev)
        self.ws = m.workspace(m.exl3_linear_shards_workspace_bytes(M, IC, self.sets[0]), dev)
        self.u = torch.empty((len(shards), M, IC), dtype=torch.float16, device=dev)
        for i in range(len(shards)):
            m.exl3_pretransform(self.xd, *scal[i][:2], u=self.u[i])
        self.m = m
        self.l2 = f"inputs larger than L2: {R} rotating code copies ({R * per_step / 1e6:.0f} MB)"
        self.launches_per_step = linear_launches(M, 2)

    def step(self, r, x=None):
        self.m.exl3_linear_into_shards(self.xd if x is None else x, self.sets[r], self.out, self.ws)

    def roofline(self, torch, stream):
        R, m = self.R, self.m
        ms = kernel_time_ms(torch, stream,
                            lambda j: m.exl3_gemm_into_shards(self.u, self.sets[j % R], self.out, self.ws), 4 * R)
        hbm, _, src = peaks()
        alg = sum(self.code_bytes(K) + 2 * self.M * self.IC + 2 * self.M * self.OC + 2 * 2 * self.OC
                  for K in self.KS)
        a = alg / (ms * 1e-3) / 1e9
        kernel = {"decode": decode_kernel(torch, self.M, (self.OC, self.OC)), "fused": "fused_tc_kernel",
                  "prefill": "reconstruct + prefill_gemm_kernel"}[gemm_path(self.M)]
        return {"bound": "hbm", "kernel": kernel + " (gate K=2 + up K=3 in one call)",
                "achieved": round(a, 1), "peak": hbm, "unit": "GB/s", "frac": round(a / hbm, 4),
                "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs)",
                "traffic": {"decode": lambda: profile_traffic(f"decode_gemm_gate_up_m{self.M}.json"),
                            "fused": lambda: profile_traffic(f"fused_gemm_gate_up_m{self.M}.json"),
                            "prefill": lambda: None}[gemm_path(self.M)](),
                "per_launch_us": round(ms * 1e3, 2), "algorithmic_bytes_per_launch": alg,
                "code_GBps": round(sum(self.code_bytes(K) for K in self.KS) / (ms * 1e-3) / 1e9, 1)}

    def e2e_io(self, torch, dev):
        xh = torch.from_numpy(self.x.view(np.int16)).view(torch.bfloat16).pin_memory()
        oh = torch.empty(self.out.shape, dtype=torch.bfloat16).pin_memory()
        return xh, torch.empty_like(self.xd), oh, self.out

    def e2e_step(self, r, xh, oh):
        """One step on host buffers through the host-buffer entry point: the kernels
        read x from, and write out to, pinned host memory (no staging copies)."""
        self.m.exl3_linear_into_shards_host(xh, self.sets[r], oh, self.ws)

    def cpu_sample(self, budget):
        import oracle
        import synthetic as syn
        x, shards = syn.gate_up(1, M=self.M)
        nblk_total = self.OC // 128
        oracle.lib()
        t0 = time.perf_counter()
        for sh in shards:
            oracle.linear_f64(x, sh.code, sh.K, sh.s_in, sh.rin, sh.rout, sh.s_out, blk0=0, nblk=1)
        per_blk = (time.perf_counter() - t0) / 2
        nblk = int(min(nblk_total, max(1, budget / max(per_blk, 1e-6) / 2)))
        t0 = time.perf_counter()
        for sh in shards:
            oracle.linear_f64(x, sh.code, sh.K, sh.s_in, sh.rin, sh.rout, sh.s_out, blk0=0, nblk=nblk)
        t = (time.perf_counter() - t0) * nblk_total / nblk
        return self.M / t, (f"M={self.M}, output blocks 0..{nblk - 1} of {nblk_total} (128 columns each) of both "
                            f"shards, scaled linearly to all {nblk_total} blocks")


class GateUpA8(GateUp):
    """The gate/up projection with 8-bit activations: each shard's activations
    are quantized per row (uint8 codes + fp32 row scale), then one grouped GEMM
    launch multiplies the codes of both shards."""
    e2e_step = None   # the device-buffer call with copies (no 8-bit host-buffer entry point)

    def __init__(self, args):
        super().__init__(args)
        self.metric = "EXL3 linear tokens/s (decode-shaped gate_up, 8-bit activations)"

    def config(self):
        c = super().config()
        c["workload"] = c["workload"].replace("gate_up", "gate_up a8", 1)
        c["activations"] = "uint8 codes + fp32 row scale"
        return c

    def setup(self, torch, m, syn, dev):
        super().setup(torch, m, syn, dev)
        self.ws8 = m.workspace(m.exl3_linear_shards_a8_workspace_bytes(self.M, self.IC, self.sets[0]), dev)
        self.A = torch.empty((2, self.M, self.IC), dtype=torch.uint8, device=dev)
        self.As = torch.empty((2, self.M), dtype=torch.float32, device=dev)
        for i, st in enumerate(self.sets[0]):
            m.exl3_quantize_a8(self.xd, *st[2:4], A=self.A[i], As=self.As[i])
        self.launches_per_step = linear_launches(self.M, 2)

    def step(self, r, x=None):
        self.m.exl3_linear_into_shards_a8(self.xd if x is None else x, self.sets[r], self.out, self.ws8)

    def roofline(self, torch, stream):
        R, m = self.R, self.m
        ms = kernel_time_ms(torch, stream,
                            lambda j: m.exl3_gemm_a8_into_shards(self.A, self.As, self.sets[j % R], self.out,
                                                                 self.ws8), 4 * R)
        hbm, _, src = peaks()
        alg = sum(self.code_bytes(K) + self.M * self.IC + 4 * self.M + 2 * self.M * self.OC + 2 * 2 * self.OC
                  for K in self.KS)
        a = alg / (ms * 1e-3) / 1e9
        kernel = {"decode": decode_kernel(torch, self.M, (self.OC, self.OC)) + (" (8-bit codes)" if self.M <= 8 else ""),
                  "fused": "codes_to_f16 + fused_tc_kernel",
                  "prefill": "codes_to_f16 + reconstruct + prefill_gemm_kernel"}[gemm_path(self.M)]
        return {"bound": "hbm", "kernel": kernel + " (gate K=2 + up K=3 in one call)",
                "achieved": round(a, 1), "peak": hbm, "unit": "GB/s", "frac": round(a / hbm, 4),
                "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs)", "traffic": None,
                "per_launch_us": round(ms * 1e3, 2), "algorithmic_bytes_per_launch": alg}

    def cpu_sample(self, budget):
        import oracle
        import synthetic as syn
        x, shards = syn.gate_up(1, M=self.M)
        nblk_total = self.OC // 128
        oracle.lib()
        t0 = time.perf_counter()
        for sh in shards:
            oracle.linear_a8_f64(x, sh.code, sh.K, sh.s_in, sh.rin, sh.rout, sh.s_out, blk0=0, nblk=1)
        per_blk = (time.perf_counter() - t0) / 2
        nblk = int(min(nblk_total, max(1, budget / max(per_blk, 1e-6) / 2)))
        t0 = time.perf_counter()
        for sh in shards:
            oracle.linear_a8_f64(x, sh.code, sh.K, sh.s_in, sh.rin, sh.rout, sh.s_out, blk0=0, nblk=nblk)
        t = (time.perf_counter() - t0) * nblk_total / nblk
        return self.M / t, (f"M={self.M}, output blocks 0..{nblk - 1} of {nblk_total} (128 columns each) of both "
                            f"shards, scaled linearly to all {nblk_total} blocks")


class Prefill:
    """Prefill-shaped linear 5120 -> 17408 at M = 8192 (1 % outlier channels)."""
    IC, OC = 5120, 17408

    def __init__(self, args):
        self.M, self.K = (args.m if args.m > 32 else 8192), args.k
        self.metric = f"EXL3 linear TFLOP/s (prefill-shaped, M={self.M})"
        self.unit = "TFLOP/s"
        self.units_per_step = 2.0 * self.M * self.IC * self.OC / 1e12

    def config(self):
        return {"workload": f"prefill 5120->17408, K={self.K}, M={self.M}, 1% outlier channels", "M": self.M,
                "IC": self.IC, "OC": self.OC, "K": self.K}

    def setup(self, torch, m, syn, dev):
        self.x, sh = syn.prefill(2, M=self.M, K=self.K)
        self.code = t16(torch, sh.code, dev, torch.int16)
        self.sc = [t16(torch, v, dev, torch.float16) for v in (sh.s_in, sh.rin, sh.rout, sh.s_out)]
        self.xd = t16(torch, self.x, dev, torch.bfloat16)
        self.out = torch.empty((self.M, self.OC), dtype=torch.bfloat16, device=dev)
        self.ws = m.workspace(m.exl3_linear_workspace_bytes(self.M, self.IC, self.OC), dev)
        self.u = m.exl3_pretransform(self.xd, self.sc[0], self.sc[1])
        self.m, self.R = m, 1
        self.l2 = "inputs larger than L2 (decoded weights 178 MB, activations and output M x 10 KB / 34 KB)"
        self.launches_per_step = 3      # pre-transform, reconstruct, tcgen05 GEMM

    def step(self, r, x=None):
        self.m.exl3_linear_into(self.xd if x is None else x, self.code, self.K, *self.sc, self.out, 0, self.ws)

    def roofline(self, torch, stream):
        m = self.m
        W = torch.empty((self.IC, self.OC), dtype=torch.float16, device=self.out.device)
        ms_all = kernel_time_ms(torch, stream, lambda j: m.exl3_gemm_into(self.u, self.code, self.K, *self.sc[2:],
                                                                           self.out, 0, self.ws), 8)
        ms_rec = kernel_time_ms(torch, stream, lambda j: m.exl3_reconstruct(self.code, self.K, W), 8)
        ms = ms_all - ms_rec
        _, burst, src = peaks()
        ts, _ = sustained_tflops()
        fl = 2.0 * self.M * self.IC * self.OC
        a = fl / (ms * 1e-3) / 1e12
        # timed alone (a few graph replays, tens of ms): the burst peak
        return {"bound": "tensor", "kernel": "prefill_gemm_kernel (tcgen05 128x256 tiles)",
                "achieved": round(a, 1), "peak": burst, "unit": "TFLOP/s", "frac": round(a / burst, 4),
                "peak_source": f"{src} (MEASURED_PEAKS.json bf16_tflops burst: the kernel timed alone; fp16 has "
                               f"the same dense rate)",
                "frac_of_sustained": round(a / ts, 4),
                "traffic": profile_traffic(f"prefill_gemm_m{self.M}.json"),
                "per_launch_us": round(ms * 1e3, 1), "reconstruct_us": round(ms_rec * 1e3, 1),
                "algorithmic_flops_per_launch": fl}

    def e2e_io(self, torch, dev):
        xh = torch.from_numpy(self.x.view(np.int16)).view(torch.bfloat16).pin_memory()
        oh = torch.empty(self.out.shape, dtype=torch.bfloat16).pin_memory()
        return xh, torch.empty_like(self.xd), oh, self.out

    def cpu_sample(self, budget):
        import oracle
        import synthetic as syn
        x, sh = syn.prefill(2, M=self.M, K=self.K)
        rows = 8
        self_M = self.M
        t0 = time.perf_counter()
        oracle.linear_f64(np.ascontiguousarray(x[:rows]), sh.code, self.K, sh.s_in, sh.rin, sh.rout, sh.s_out)
        t = time.perf_counter() - t0
        flops = 2.0 * rows * self.IC * self.OC
        return flops / t / 1e12, (f"{rows} of {self_M} rows, all 17408 columns (the weights decoded once), "
                                  f"TFLOP/s of the sample")


class Moe:
    """Grouped MoE: 128 experts, H 2048, I 768, top-8, per-expert K in {2, 3, 4}."""
    H, I, E, TOPK = 2048, 768, 128, 8

    def __init__(self, args):
        self.T = args.t
        self.metric = f"EXL3 grouped MoE tokens/s (T={self.T})"
        self.unit = "tokens/s"
        self.units_per_step = self.T

    def config(self):
        return {"workload": f"moe E=128 H=2048 I=768 top-8, T={self.T}, K per expert in {{2,3,4}}", "T": self.T}

    def setup(self, torch, m, syn, dev):
        self.bank_np = syn.moe_bank(3)
        dt = dict(w13=torch.int16, w2=torch.int16, off_w1=torch.int64, off_w3=torch.int64, off_w2=torch.int64,
                  perm=torch.int32, k_gu=torch.int32, k_d=torch.int32, w13_suh=torch.float16,
                  w13_svh=torch.float16, w2_suh=torch.float16, w2_svh=torch.float16)
        self.bank = {k: t16(torch, v, dev, dt[k]) for k, v in self.bank_np.items()}
        # rotating token batches route to different experts every step (defeats L2 reuse)
        self.R = R = 8
        self.xs, self.ls = [], []
        for r in range(R):
            x, logits = syn.moe_tokens(100 + r, self.T)
            self.xs.append(t16(torch, x, dev, torch.bfloat16))
            self.ls.append(torch.from_numpy(logits).to(dev))
            if r == 0:
                self.x0 = x
        self.ids = torch.empty((self.T, self.TOPK), dtype=torch.int32, device=dev)
        self.w = torch.empty((self.T, self.TOPK), dtype=torch.float32, device=dev)
        self.y = torch.empty((self.T, self.H), dtype=torch.bfloat16, device=dev)
        self.ws = m.workspace(m.exl3_moe_workspace_bytes(self.T, self.H, self.I, self.E, self.TOPK), dev)
        self.m = m
        kk = self.bank_np["k_gu"].astype(np.int64)
        per_slot = 3 * self.H * self.I * kk // 8
        self.touched = []
        for r in range(R):
            # experts a batch touches (bookkeeping for the byte count: the largest
            # logits, ties to the lower expert id)
            ids = np.argsort(-self.ls[r].cpu().numpy(), axis=1, kind="stable")[:, :self.TOPK]
            slots = np.unique(self.bank_np["perm"][ids.ravel()])
            self.touched.append(int(per_slot[slots].sum()))
        bank_mb = (self.bank["w13"].numel() + self.bank["w2"].numel()) * 2 / 1e6
        self.l2 = f"{R} rotating token batches (different experts per step; bank {bank_mb:.0f} MB)"
        # one 8-row block per entry: top-k (inside the routing launch up to 8 tokens),
        # routing + rotation, FC1 with the activation in its epilogue, FC2 with the
        # combine; otherwise top-k, route, rotate, FC1, act, FC2, combine
        chain = self.T * self.TOPK <= 4 * self.E
        self.launches_per_step = (3 if self.T <= 8 else 4) if chain else 7

    def step(self, r, x=None):
        # the layer from router logits in one call (top-k, routing, FC1, FC2, combine)
        self.m.exl3_moe_forward(self.xs[r] if x is None else x, self.ls[r], self.TOPK, self.bank, self.ws, y=self.y,
                                ids=self.ids, w=self.w)

    def roofline(self, torch, stream):
        # the layer's launch chain: code bytes of the touched experts / layer time
        ms = kernel_time_ms(torch, stream, lambda j: self.step(j % self.R), 4 * self.R)
        hbm, _, src = peaks()
        code = statistics.mean(self.touched)
        a = code / (ms * 1e-3) / 1e9
        return {"bound": "hbm", "kernel": "grouped MoE launch chain (top-k .. combine)",
                "achieved": round(a, 1), "peak": hbm, "unit": "GB/s", "frac": round(a / hbm, 4),
                "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs)", "traffic": None,
                "per_layer_us": round(ms * 1e3, 2), "touched_code_bytes": int(code)}

    def e2e_io(self, torch, dev):
        xh = torch.from_numpy(self.x0.view(np.int16)).view(torch.bfloat16).pin_memory()
        oh = torch.empty(self.y.shape, dtype=torch.bfloat16).pin_memory()
        return xh, torch.empty_like(self.xs[0]), oh, self.y

    def cpu_sample(self, budget):
        import oracle
        import synthetic as syn
        x, logits = syn.moe_tokens(100, self.T)
        ids, w = oracle.topk_softmax(logits, self.TOPK)
        n = min(self.T, 4)
        t0 = time.perf_counter()
        oracle.moe_f64(np.ascontiguousarray(x[:n]), np.ascontiguousarray(ids[:n]), np.ascontiguousarray(w[:n]),
                       self.bank_np)
        t = time.perf_counter() - t0
        return n / t, f"{n} of {self.T} tokens (their experts decoded), tokens/s of the sample"


class Gather:
    """int8 embedding gather: 8192 ids from a 248,320 x 5120 int8 table."""
    V, H, N = 248320, 5120, 8192

    def __init__(self, args):
        self.metric = "int8 embedding gather tokens/s (8192 ids, 248320 x 5120)"
        self.unit = "tokens/s"
        self.units_per_step = self.N

    def config(self):
        return {"workload": "gather 8192 ids from int8 [248320, 5120] + fp16 row scale -> bf16"}

    def setup(self, torch, m, syn, dev):
        q, s, _ = syn.embedding(5)
        self.q = t16(torch, q, dev, torch.int8)
        self.s = t16(torch, s, dev, torch.float16)
        self.R = R = 8
        g = syn.rng(77)
        self.idss = [torch.from_numpy(g.integers(0, self.V, self.N, dtype=np.int32)).to(dev) for _ in range(R)]
        self.ids0 = self.idss[0].cpu().numpy()
        self.out = torch.empty((self.N, self.H), dtype=torch.bfloat16, device=dev)
        self.m = m
        self.l2 = "table 1.27 GB >> L2; 8 rotating id sets"
        self.launches_per_step = 1

    def step(self, r, ids=None):
        self.m.exl3_embed_int8_gather(self.q, self.s, self.idss[r] if ids is None else ids, out=self.out)

    def roofline(self, torch, stream):
        ms = kernel_time_ms(torch, stream, lambda j: self.step(j % self.R), 4 * self.R)
        hbm, _, src = peaks()
        alg = self.N * self.H + 2 * self.N + 4 * self.N + 2 * self.N * self.H
        a = alg / (ms * 1e-3) / 1e9
        return {"bound": "hbm", "kernel": "gather_kernel", "achieved": round(a, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(a / hbm, 4), "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs)",
                "traffic": profile_traffic("gather_8192.json"), "per_launch_us": round(ms * 1e3, 2),
                "algorithmic_bytes_per_launch": alg}

    def e2e_io(self, torch, dev):
        xh = torch.from_numpy(self.ids0).pin_memory()
        oh = torch.empty(self.out.shape, dtype=torch.bfloat16).pin_memory()
        return xh, torch.empty_like(self.idss[0]), oh, self.out

    def cpu_sample(self, budget):
        import oracle
        import synthetic as syn
        q, s, ids = syn.embedding(5)
        t0 = time.perf_counter()
        oracle.gather(q, s, ids)
        t = time.perf_counter() - t0
        return self.N / t, "all 8192 ids"


class Layer:
    """The five projections of a hidden-5120 decoder layer (qkv K4, o K3, gate K2 + up K3, down K3)."""

    def __init__(self, args):
        self.M = args.m
        self.metric = f"EXL3 decoder-layer projections tokens/s (M={self.M})"
        self.unit = "tokens/s"
        self.units_per_step = self.M

    def config(self):
        return {"workload": f"layer qkv 5120->7168 K4, o 5120->5120 K3, gate|up 5120->2x17408 K2|K3, "
                            f"down 17408->5120 K3; M={self.M}", "M": self.M}

    def setup(self, torch, m, syn, dev):
        projs = syn.decoder_layer(4, M=self.M)
        self.projs = projs
        self.m = m
        self.code_bytes = sum(sh.IC * sh.OC * sh.K // 8 for _, _, sh in projs)
        self.R = R = max(2, int(np.ceil(4 * L2_BYTES / self.code_bytes))) if self.M <= 128 else 1
        self.xs = {n: t16(torch, x, dev, torch.bfloat16) for n, x, _ in projs}
        self.x0 = self.xs["qkv"]
        self.dsh = {}
        for n, _, sh in projs:
            c = [t16(torch, sh.code, dev, torch.int16)]
            for _ in range(R - 1):
                c.append(c[0].clone())
            self.dsh[n] = (c, sh.K, [t16(torch, v, dev, torch.float16) for v in (sh.s_in, sh.rin, sh.rout, sh.s_out)])
        self.outs = {"qkv": torch.empty((self.M, 7168), dtype=torch.bfloat16, device=dev),
                     "o": torch.empty((self.M, 5120), dtype=torch.bfloat16, device=dev),
                     "gu": torch.empty((self.M, 34816), dtype=torch.bfloat16, device=dev),
                     "down": torch.empty((self.M, 5120), dtype=torch.bfloat16, device=dev)}
        self.ws = m.workspace(m.exl3_projections_workspace_bytes(self.M, self._projs(0)), dev)
        self.l2 = (f"{R} rotating code copies ({R * self.code_bytes / 1e6:.0f} MB)" if R > 1
                   else "inputs larger than L2")
        self.launches_per_step = sum(linear_launches(self.M, n) for n in (1, 1, 2, 1))

    def _sh(self, n, r, col0=None):
        c, K, sc = self.dsh[n]
        t = (c[r], K, *sc)
        return t + ((col0,) if col0 is not None else ())

    def _projs(self, r, x=None):
        return [(self.x0 if x is None else x, [self._sh("qkv", r, 0)], self.outs["qkv"]),
                (self.xs["o"], [self._sh("o", r, 0)], self.outs["o"]),
                (self.xs["gate"], [self._sh("gate", r, 0), self._sh("up", r, 17408)], self.outs["gu"]),
                (self.xs["down"], [self._sh("down", r, 0)], self.outs["down"])]

    def step(self, r, x=None):
        # the layer's projections in one library call on one workspace
        self.m.exl3_linear_projections(self._projs(r, x), self.ws)

    def roofline(self, torch, stream):
        ms = kernel_time_ms(torch, stream, lambda j: self.step(j % self.R), 4 * self.R)
        hbm, tf, src = peaks()
        if gemm_path(self.M) != "prefill":
            a = self.code_bytes / (ms * 1e-3) / 1e9
            return {"bound": "hbm", "kernel": "the layer's launches (code bytes / layer time)",
                    "achieved": round(a, 1), "peak": hbm, "unit": "GB/s", "frac": round(a / hbm, 4),
                    "peak_source": src, "traffic": None, "per_layer_us": round(ms * 1e3, 2),
                    "code_bytes": self.code_bytes}
        fl = sum(2.0 * self.M * sh.IC * sh.OC for _, _, sh in self.projs)
        a = fl / (ms * 1e-3) / 1e12
        ts, _ = sustained_tflops()
        # timed alone (a few graph replays, tens of ms): the burst peak
        return {"bound": "tensor", "kernel": "the layer's launches (flops / layer time)", "achieved": round(a, 1),
                "peak": tf, "unit": "TFLOP/s", "frac": round(a / tf, 4),
                "peak_source": f"{src} (MEASURED_PEAKS.json bf16_tflops burst: the layer timed alone)",
                "frac_of_sustained": round(a / ts, 4), "traffic": None, "per_layer_us": round(ms * 1e3, 1)}

    def e2e_io(self, torch, dev):
        xh = torch.from_numpy(np.ascontiguousarray(self.projs[0][1]).view(np.int16)).view(torch.bfloat16).pin_memory()
        oh = torch.empty(self.outs["down"].shape, dtype=torch.bfloat16).pin_memory()
        return xh, torch.empty_like(self.x0), oh, self.outs["down"]

    def cpu_sample(self, budget):
        import oracle
        t = 0.0
        for _, x, sh in self.projs:
            nb, rows = 2, min(self.M, 8)
            t0 = time.perf_counter()
            oracle.linear_f64(np.ascontiguousarray(x[:rows]), sh.code, sh.K, sh.s_in, sh.rin, sh.rout,
                              sh.s_out, blk0=0, nblk=nb)
            t += (time.perf_counter() - t0) * (sh.OC // 128) / nb * (self.M / rows)
        return self.M / t, "2 output blocks of each projection (<= 8 rows), scaled to all blocks and rows"


class LmHead:
    """int8 output head: the 248,320 x 5120 int8 table (fp16 row scale) as the output projection."""
    V, H = 248320, 5120

    def __init__(self, args):
        self.M = args.m
        self.metric = f"int8 output head tokens/s (M={self.M}, 248320 x 5120)"
        self.unit = "tokens/s"
        self.units_per_step = self.M

    def config(self):
        return {"workload": f"lm_head int8 [248320, 5120] + fp16 row scale, M={self.M} -> bf16 logits", "M": self.M}

    def setup(self, torch, m, syn, dev):
        q, s, _ = syn.embedding(5)
        self.q = t16(torch, q, dev, torch.int8)
        self.s = t16(torch, s, dev, torch.float16)
        self.R = R = 4
        g = syn.rng(78)
        self.xnp = [syn.normal_bf16(g, self.M, self.H) for _ in range(R)]
        self.xs = [t16(torch, x, dev, torch.bfloat16) for x in self.xnp]
        self.out = torch.empty((self.M, self.V), dtype=torch.bfloat16, device=dev)
        self.ws = m.workspace(m.exl3_lm_head_workspace_bytes(self.M, self.H, self.V), dev)
        self.m = m
        self.l2 = "table 1.27 GB >> L2"
        # the activations to fp16, then one streaming pass (M <= 32) or a conversion
        # and a tensor-core GEMM per 16384-row chunk of the table
        self.launches_per_step = 2 if self.M <= 32 else 1 + 2 * -(-self.V // 16384)

    def step(self, r, x=None):
        self.m.exl3_lm_head_int8(self.xs[r] if x is None else x, self.q, self.s, self.ws, out=self.out)

    def roofline(self, torch, stream):
        ms = kernel_time_ms(torch, stream, lambda j: self.step(j % self.R), 4 * self.R)
        hbm, tf, src = peaks()
        if self.M <= 32:
            alg = self.V * self.H + 2 * self.V + 2 * self.M * self.H + 2 * self.M * self.V
            a = alg / (ms * 1e-3) / 1e9
            return {"bound": "hbm", "kernel": "lm_head_decode_kernel (int8 table streamed, mma.sync)",
                    "achieved": round(a, 1), "peak": hbm, "unit": "GB/s", "frac": round(a / hbm, 4),
                    "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs)",
                    "traffic": profile_traffic(f"lm_head_decode_m{self.M}.json"),
                    "per_launch_us": round(ms * 1e3, 2), "algorithmic_bytes_per_launch": alg}
        fl = 2.0 * self.M * self.H * self.V
        a = fl / (ms * 1e-3) / 1e12
        ts, _ = sustained_tflops()
        # timed alone (a few graph replays, tens of ms): the burst peak
        return {"bound": "tensor", "kernel": "int8->fp16 chunks + prefill_gemm_kernel (row-scale epilogue)",
                "achieved": round(a, 1), "peak": tf, "unit": "TFLOP/s", "frac": round(a / tf, 4),
                "peak_source": f"{src} (MEASURED_PEAKS.json bf16_tflops burst: the call timed alone)",
                "frac_of_sustained": round(a / ts, 4), "traffic": None, "per_call_us": round(ms * 1e3, 1)}

    def e2e_io(self, torch, dev):
        xh = torch.from_numpy(self.xnp[0].view(np.int16)).view(torch.bfloat16).pin_memory()
        oh = torch.empty(self.out.shape, dtype=torch.bfloat16).pin_memory()
        return xh, torch.empty_like(self.xs[0]), oh, self.out

    def cpu_sample(self, budget):
        import oracle
        import synthetic as syn
        q, s, _ = syn.embedding(5)
        x = self.xnp[0]
        nv = 2048
        t0 = time.perf_counter()
        oracle.lm_head_f64(x, q, s, v0=0, nv=nv)
        t = (time.perf_counter() - t0) * self.V / nv
        return self.M / t, f"vocabulary rows 0..{nv - 1} of {self.V}, scaled linearly to the whole table"


WORKLOADS = {"gate_up": GateUp, "gate_up_a8": GateUpA8, "prefill": Prefill, "moe": Moe, "gather": Gather, "layer": Layer, "lm_head": LmHead}


# ------------------------------------------------------------------ our arm
def capture(torch, stream, fn):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


def timed_steps(torch, stream, wl, K, W, dist, min_seconds, min_trials=5):
    """Time exactly K steps per trial (CUDA events on `stream`, a barrier and a
    device synchronize on both sides), after at least W warm-up steps; trials repeat
    until they add up to min_seconds.  Returns the trial durations in ms."""
    R = wl.R
    with torch.cuda.stream(stream):
        for r in range(R):
            wl.step(r)                       # eager warm-up of every path
    torch.cuda.synchronize()
    g_full = capture(torch, stream, lambda: [wl.step(r) for r in range(R)])
    rem = K % R
    g_rem = capture(torch, stream, lambda: [wl.step(r) for r in range(rem)]) if rem else None
    torch.cuda.synchronize()

    def k_steps():
        for _ in range(K // R):
            g_full.replay()
        if g_rem is not None:
            g_rem.replay()

    with torch.cuda.stream(stream):
        for _ in range(-(-W // R)):
            g_full.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    trials, total = [], 0.0
    while len(trials) < min_trials or total < min_seconds:
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            e0.record(stream)
            k_steps()
            e1.record(stream)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        t = e0.elapsed_time(e1)
        trials.append(t)
        total += t / 1e3
        if len(trials) >= 200000:
            break
    return trials


def secondary_workloads():
    """The other configurations timed beside the headline (one GPU): each line
    carries its own throughput and the roofline of its dominant kernel."""
    ns = argparse.Namespace
    return [("gate_up", ns(m=1)), ("gate_up", ns(m=64)), ("prefill", ns(m=8192, k=2)),
            ("moe", ns(t=1)), ("moe", ns(t=16)), ("moe", ns(t=512)), ("gather", ns()),
            ("layer", ns(m=8)), ("layer", ns(m=8192)), ("lm_head", ns(m=1)), ("lm_head", ns(m=8)),
            ("gate_up_a8", ns(m=8)), ("gate_up_a8", ns(m=64))]


def run_secondary(torch, m, syn, dev, stream, local, K, W, min_seconds):
    out = []
    for name, a in secondary_workloads():
        wl = WORKLOADS[name](a)
        wl.setup(torch, m, syn, dev)
        k = K if getattr(wl, "M", 0) <= 128 and name != "prefill" else max(wl.R, min(K, 20))
        with Clocks(local) as clk:
            trials = timed_steps(torch, stream, wl, k, W, None, min_seconds)
        ms = statistics.median(trials)
        value = job_throughput(1, wl.units_per_step, k, ms)
        out.append({"workload": wl.config()["workload"], "metric": wl.metric, "value": round(value, 3),
                    "unit": wl.unit, "steps": k, "trials": len(trials), "ms_per_step": round(ms / k, 5),
                    "roofline": wl.roofline(torch, stream), "clocks": clk.summary()})
        del wl
        GateUp._codes.clear() if name.startswith("gate_up") and a.m == 64 else None
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return out


def run_ours(args):
    import torch
    import moe_gemm_exl3_gb300 as m
    from moe_gemm_exl3_gb300 import build as b
    import synthetic as syn

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    b.build()
    wl = WORKLOADS[args.workload](args)
    wl.setup(torch, m, syn, dev)
    R = wl.R
    stream = torch.cuda.Stream(dev)
    K, W = args.steps, args.warmup
    with Clocks(local) as clk:
        trials = timed_steps(torch, stream, wl, K, W, dist, args.min_seconds)
    ms = max_over_ranks(torch, dist, statistics.median(trials), dev)
    value = job_throughput(world, wl.units_per_step, K, ms)

    roof = wl.roofline(torch, stream)

    # ---- end to end through the public API with host buffers (pinned), eager launches
    xh, xdev, oh, out = wl.e2e_io(torch, dev)
    e2e_steps = max(R, min(K, 20 * R))
    host_step = getattr(wl, "e2e_step", None)

    def e2e_one(r):
        if host_step is not None:
            host_step(r, xh, oh)   # the kernels move x in and out back themselves
        else:
            xdev.copy_(xh, non_blocking=True)
            wl.step(r, xdev)
            oh.copy_(out, non_blocking=True)

    with torch.cuda.stream(stream):
        for r in range(R):
            e2e_one(r)
        torch.cuda.synchronize()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for i in range(e2e_steps):
            e2e_one(i % R)
        a1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(torch, dist, a0.elapsed_time(a1) / e2e_steps, dev)
    e2e_val = job_throughput(world, wl.units_per_step, 1, e2e_ms)

    line = {
        "metric": wl.metric, "value": round(value, 3), "unit": wl.unit, "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": round(ms / K, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic (seeded; uniform int16 code words, N(0,1) activations)",
        "config": dict(wl.config(), l2=wl.l2,
                       timing=(f"median of {len(trials)} timed trials of exactly {K} steps each "
                               f"({sum(trials) / 1e3:.2f} s timed); each trial replays CUDA graphs of the "
                               f"steps between CUDA events, barrier + synchronize on both sides"),
                       parallelism="replicas" if world > 1 else "single GPU"),
        "gpu_launches": wl.launches_per_step * K,
        "roofline": roof,
        "e2e": {"value": round(e2e_val, 3), "unit": wl.unit,
                "h2d_bytes_per_step": int(xh.numel() * xh.element_size()),
                "d2h_bytes_per_step": int(oh.numel() * oh.element_size()),
                "note": ("exl3_linear_into_shards_host: the kernels read the pinned host input and write the "
                         "result to pinned host memory every step, eager launches" if host_step is not None else
                         "public API with pinned host input copied in and the result read back every step, "
                         "eager launches")},
        "clocks": clk.summary(),
    }
    del xh, xdev, oh, out
    if world == 1 and not args.no_secondary and args.workload == "gate_up" and args.m == 8:
        del wl
        torch.cuda.empty_cache()
        line["secondary"] = run_secondary(torch, m, syn, dev, stream, local, K, W, args.secondary_seconds)
    if rank == 0:
        if not args.no_cpu_baseline and world == 1:
            wl0 = WORKLOADS[args.workload](args)
            v, sample = wl0.cpu_sample(args.cpu_budget)
            line["cpu_baseline"] = {"value": round(v, 4), "unit": wl0.unit, "cores": omp_threads(),
                                    "kind": "oracle", "sample": sample}
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


# ------------------------------------------------------------------ reference arm
def run_reference(args):
    """The CPU oracle as the reference arm: same metric and workload, each step a bounded
    sample (whole 128-column output blocks of both shards), scaled to the full step."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    if args.workload != "gate_up":
        print(json.dumps({"impl": "reference", "unavailable": "the reference arm covers the headline workload only"}))
        return
    M, OC = args.m, GateUp.OC
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
    run_steps = int(max(1, min(K, budget / (nblk * per_blk) - W)))
    for _ in range(W):
        one(nblk)
    t0 = time.perf_counter()
    for _ in range(run_steps):
        one(nblk)
    t = (time.perf_counter() - t0) / run_steps * nblk_total / nblk
    v = M / t
    wl = GateUp(args)
    line = {"impl": "reference", "metric": wl.metric, "value": round(v, 3), "unit": "tokens/s",
            "n_gpus": 1, "steps": run_steps, "steps_requested": K, "warmup": W,
            "ms_per_step": round(t * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)", "config": wl.config(),
            "cpu_baseline": {"value": round(v, 3), "unit": "tokens/s", "cores": omp_threads(), "kind": "oracle",
                             "sample": f"each step: output blocks 0..{nblk - 1} of {nblk_total} (128 columns) "
                                       f"of both shards, scaled linearly to the full step"},
            "e2e": {"value": round(v, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--workload", default="gate_up", choices=sorted(WORKLOADS))
    ap.add_argument("--m", type=int, default=8, help="rows (gate_up, layer)")
    ap.add_argument("--k", type=int, default=2, help="bits per weight (prefill)")
    ap.add_argument("--t", type=int, default=16, help="tokens (moe)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true", help="skip the other configurations")
    ap.add_argument("--min-seconds", type=float, default=1.5, help="timed seconds of the headline trials")
    ap.add_argument("--secondary-seconds", type=float, default=0.3, help="timed seconds per secondary line")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--ref-budget", type=float, default=90.0, help="seconds of oracle work (reference arm)")
    args = ap.parse_args()
    if args.steps is None:
        args.steps = 200 if args.workload != "prefill" and not (args.workload == "layer" and args.m > 128) else 20
    if args.warmup is None:
        args.warmup = 20
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
