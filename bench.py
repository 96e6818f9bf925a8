"""Benchmark of the batched dense product on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one call of the product over the workload's whole batch, through
the C ABI (bmm_run) with inputs resident in HBM.  The default workload is the
square GEMM the headline metric is quoted on: batch 1, M = N = K = 4096,
A row-major, B column-major (transB), bf16 normal(0,1) inputs, fp32
accumulation, bf16 output, alpha = 1, beta = 0.  Its working set (96 MB) fits
in the 129 MB L2, so a 512 MB buffer is written between timed steps to
evict L2; the flush is outside the timed interval.

Prints one JSON line (rank 0).  ``roofline`` compares the dominant kernel's
algorithmic FLOP/s (2*M*N*K per launch over its CUDA-event duration) with the
measured dense bf16 peak (``MEASURED_PEAKS.json``: cuBLAS bf16 burst), with
ncu's tensor-pipe activity of the same kernel source beside it (null once the
sources change) and the median and best launch times beside the mean;
``e2e`` repeats the metric with host buffers (H2D of
A and B from pinned memory, the call, D2H of C inside each timed step);
``cpu_baseline`` times the fp64 oracle on the host cores on a bounded sample
of the same workload.  ``other_workloads`` reports the remaining specified
shapes (ragged, attention pair, skinny, small) measured the same way; a shape
with a staged operand also reports ``row_loader``, the same product with the
kernels' row loader reading that operand in place.

With ``--impl reference`` the reference arm runs instead: the fp64 CPU
oracle, timed on this host's cores on a bounded sample of each step.
Multi-GPU (torchrun): every rank runs its own copy of the workload
(independent problems, no collective on the data path); value = all ranks'
FLOPs over the slowest rank's time.
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

# Denominators measured on the GB300s (copy of MEASURED_PEAKS.json,
# 2026-12-02): read live when the file is present.
MEASURED_FALLBACK = {"hbm_gbs": 6676.5, "bf16_tflops": 1932.9, "bf16_tflops_sustained": 1743.9,
                     "sm_max_mhz": 2070.0}
RECIPE_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM traffic per launch of the dominant kernel from one ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum; profiles/ has the summary),
# keyed by a hash of that kernel's sources and the workload: reported only
# while those sources are unchanged.
NCU_TRAFFIC = {
    ("74de60fa447a3efe", "gemm_4096x4096x4096_tn_bf16"): 86637824 + 17863936,
    # captured at batch 64 and scaled by 2 to the batch-128 launch (every query
    # tile does the same work); most of O's write-back happens after the kernel
    ("d0000e4da038c4a4", "attn_fused_b128_2048x2048x128_bf16"): 2 * (100719104 + 6902784),
}
# Tensor-pipe activity of the same captures (sm__pipe_tensor_cycles_active,
# % of elapsed cycles): the hardware's own measure of how busy the tensor
# cores were, reported beside the fraction of the measured cuBLAS peak.
NCU_TENSOR_ACTIVE_PCT = {
    ("74de60fa447a3efe", "gemm_4096x4096x4096_tn_bf16"): 71.44,
    ("d0000e4da038c4a4", "attn_fused_b128_2048x2048x128_bf16"): 40.76,
}

# the sources each kernel family is built from
GEMM_SOURCES = ("bmm_api.cu", "bmm_kernel.cuh", "ptx.cuh")
ATTN_SOURCES = ("attn_api.cu", "attn_kernel.cuh", "bmm_kernel.cuh", "ptx.cuh")

FLUSH_BYTES = 512 << 20

# the headline metric (both arms print it; the reference arm is the fp64 oracle)
METRIC = "BMM TFLOP/s & % of GB300 bf16 tensor peak; GB/s & % HBM for skinny shapes"


def kernel_source_hash(files=GEMM_SOURCES) -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "dense_matmul_tensor_gb300", "csrc")
    for f in files:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, \
                "measured"
        except Exception:
            pass
    return dict(MEASURED_FALLBACK), "measured (copied from this pool's MEASURED_PEAKS.json)"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="gemm_4096x4096x4096_tn_bf16")
    ap.add_argument("--no-other", action="store_true", help="skip the other workloads")
    ap.add_argument("--no-cpu", action="store_true", help="skip the cpu_baseline leg")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch count (small cases for profiling)")
    ap.add_argument("--attn-only", type=int, default=None, metavar="BATCH",
                    help="time only the fused attention kernel (L = 2048, D = 128) at this batch "
                         "and print its entry (profiling)")
    ap.add_argument("--grouped-only", action="store_true",
                    help="time only the grouped launch of 1000 small problems (no one-call-per-problem "
                         "comparison) and print its entry (profiling)")
    return ap.parse_args()


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons (every 100 ms)."""

    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str):
        self.uuid = uuid.lower()
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu=timestamp,{self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except FileNotFoundError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def samples(self):
        out = []
        if not self.path or not os.path.exists(self.path):
            return out
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            ts, uuid = parts[0], parts[1].lower()
            if self.uuid and self.uuid not in uuid:
                continue
            try:
                t = time.mktime(time.strptime(ts.split(".")[0], "%Y/%m/%d %H:%M:%S")) + \
                    float("0." + ts.split(".")[1]) if "." in ts else 0.0
            except Exception:
                t = 0.0
            out.append(dict(t=t, sm=float(parts[2]), sm_max=float(parts[3]),
                            power=float(parts[4]) if parts[4].replace(".", "").isdigit() else None,
                            hw_slowdown=parts[6], hw_thermal=parts[7], sw_thermal=parts[8],
                            sw_power_cap=parts[9]))
        return out

    def summary(self, t0, t1):
        s = self.samples()
        window = [x for x in s if t0 - 0.15 <= x["t"] <= t1 + 0.15]
        used = window or ([min(s, key=lambda x: abs(x["t"] - (t0 + t1) / 2))] if s else [])
        if not used:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        reasons = set()
        for x in used:
            for k, name in (("hw_slowdown", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                            ("sw_thermal", "sw_thermal_slowdown"), ("sw_power_cap", "sw_power_cap")):
                if x[k].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(x["sm"] for x in used),
                "sm_max_mhz": max(x["sm_max"] for x in used), "reasons": sorted(reasons),
                "samples": len(window), "nearest_only": not window}


# ---------------------------------------------------------- our GPU arm

def gpu_inputs(p, dev, seed):
    """Seeded synthetic inputs drawn on the device (same distributions as the
    host generator; used only where values do not enter a parity check)."""
    import torch
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    dt = torch.bfloat16 if p.type_ab == "bf16" else torch.float16
    na, nb, nc = p.storage_elems()

    def draw(n, dist):
        if dist == "uniform":
            return (torch.rand(n, generator=g, device=dev, dtype=torch.float32) * 2 - 1).to(dt)
        return torch.randn(n, generator=g, device=dev, dtype=torch.float32).to(dt)

    A, B = draw(na, p.dist_ab), draw(nb, p.dist_ab)
    if p.name.startswith("attn_pv"):
        # P rows are softmax rows of N(0,1) scores, as in the attention pair
        A = torch.softmax(torch.randn(p.batch * p.M, p.K, generator=g, device=dev), dim=1).to(dt)
        A = A.reshape(-1)
    cdt = torch.float32 if p.type_c == "f32" else torch.bfloat16
    if p.beta != 0.0:
        C = draw(nc, p.dist_c).to(cdt)
    else:
        C = torch.empty(nc, dtype=cdt, device=dev)
    return A, B, C


def host_inputs(p):
    """Seeded inputs from the shared generator module, as torch CPU tensors."""
    import torch
    from dense_matmul_tensor_gb300 import workloads as wl
    x = wl.make_inputs(p)
    A = wl.as_torch16(x.A, p.type_ab)
    B = wl.as_torch16(x.B, p.type_ab)
    nc = p.storage_elems()[2]
    if x.C_in is not None:
        C = torch.from_numpy(x.C_in) if p.type_c == "f32" else wl.as_torch16(x.C_in, "bf16")
    else:
        C = torch.zeros(nc, dtype=torch.float32 if p.type_c == "f32" else torch.bfloat16)
    return A, B, C


def desc_of(p):
    from dense_matmul_tensor_gb300 import bmm
    s = p.strides()
    return bmm.make_desc(batch=p.batch, M=p.M, N=p.N, K=p.K, lda=s["lda"], ldb=s["ldb"],
                         ldc=s["ldc"], strideA=s["sA"], strideB=s["sB"], strideC=s["sC"],
                         transA=p.transA, transB=p.transB, typeA=p.type_ab, typeC=p.type_c)


def time_device(p, A, B, C, steps, warmup, flush, stream, barrier):
    """Per-step CUDA-event times (ms) of bmm_run with resident inputs."""
    import torch
    from dense_matmul_tensor_gb300 import bmm
    plan = bmm.Plan(desc_of(p))
    info = plan.info()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(warmup):
            flush.fill_(i & 0xFF)
            plan.run(A, B, C, p.alpha, p.beta, stream)
    torch.cuda.synchronize()
    st, word = plan.device_error()
    if st != bmm.BMM_OK:
        raise RuntimeError(f"device error {word:#x} during warm-up")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    with torch.cuda.stream(stream):
        for i in range(steps):
            flush.fill_(i & 0xFF)
            ev[i][0].record(stream)
            plan.run(A, B, C, p.alpha, p.beta, stream)
            ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier()
    t1 = time.time()
    st, word = plan.device_error()
    plan.close()
    if st != bmm.BMM_OK:
        raise RuntimeError(f"device error {word:#x} in the timed region")
    ms = [a.elapsed_time(b) for a, b in ev]
    launches = 1 + int(info.pack_a) + int(info.pack_b)
    return ms, info, launches, (t0, t1)


def time_e2e(p, steps, warmup, stream, dev):
    """The metric through the host-buffer C ABI (bmm_host_run), the call a
    user with operands in host memory makes: per step A and B (and C_in when
    beta != 0) go in from pinned host memory and C comes back, inside the
    call, which overlaps those transfers with the computation in chunks.
    CUDA events around the steps on the caller's stream."""
    import torch
    from dense_matmul_tensor_gb300 import bmm
    hA, hB, hC = host_inputs(p)
    hA, hB, hC = hA.pin_memory(), hB.pin_memory(), hC.pin_memory()
    plan = bmm.HostPlan(desc_of(p))

    def step():
        plan.run(hA, hB, hC, p.alpha, p.beta, stream)

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
    torch.cuda.synchronize()
    st, word = plan.device_error()
    chunks = plan.chunks()
    plan.close()
    if st != bmm.BMM_OK:
        raise RuntimeError(f"device error {word:#x} in the end-to-end leg")
    ms = e0.elapsed_time(e1) / steps
    h2d = hA.numel() * hA.element_size() + hB.numel() * hB.element_size() + \
        (hC.numel() * hC.element_size() if p.beta != 0.0 else 0)
    d2h = hC.numel() * hC.element_size()
    return ms, h2d, d2h, chunks


def grouped_measure(dev, stream, steps, peaks, count=1000, seed=7, compare_singles=True):
    """Many small independent products (M, N, K drawn from 64..256, bf16 in,
    fp32 out): one grouped launch against one bmm_run per problem.  Both
    are timed with CUDA events around the whole set on the same stream (back
    to back: the set's operands, ~205 MB, exceed L2).  The set's arithmetic
    intensity (~41 FLOP/byte) is far below the ridge, so the grouped launch
    is also reported as GB/s of algorithmic bytes (A and B read, C written
    once per problem) against the measured HBM copy bandwidth."""
    import torch
    from dense_matmul_tensor_gb300 import bmm
    rng = np.random.default_rng(seed)
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    items, plans, flops, nbytes = [], [], 0, 0
    for _ in range(count):
        M, N, K = (int(rng.choice([64, 128, 192, 256])) for _ in range(3))
        A = torch.randn(M * K, generator=g, device=dev).to(torch.bfloat16)
        B = torch.randn(K * N, generator=g, device=dev).to(torch.bfloat16)
        C = torch.empty(M * N, dtype=torch.float32, device=dev)
        items.append(dict(M=M, N=N, K=K, lda=K, ldb=N, ldc=N, A=A, B=B, C=C, alpha=1.0, beta=0.0))
        if compare_singles:
            plans.append(bmm.Plan(bmm.make_desc(batch=1, M=M, N=N, K=K, lda=K, ldb=N, ldc=N, strideA=0,
                                                strideB=0, strideC=0, typeA="bf16", typeC="f32")))
        flops += 2 * M * N * K
        nbytes += 2 * M * K + 2 * K * N + 4 * M * N
    arr, n = bmm.make_problems(items)
    gplan = bmm.bmm_grouped_create(arr, n, 0, 0, "bf16", "f32")
    torch.cuda.synchronize()

    def grouped():
        bmm.bmm_grouped_run(gplan, arr, stream)

    def singles():
        for it, pl in zip(items, plans):
            pl.run(it["A"], it["B"], it["C"], 1.0, 0.0, stream)

    out = {}
    legs = (("grouped", grouped), ("one_call_per_problem", singles)) if compare_singles else (("grouped", grouped),)
    for name, fn in legs:
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = max(3, min(steps, 20))
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        out[name] = {"ms": ms, "TFLOP/s": flops / (ms * 1e-3) / 1e12, "GB/s": nbytes / (ms * 1e-3) / 1e9}
    info = bmm.bmm_grouped_get_info(gplan)
    bmm.bmm_grouped_destroy(gplan)
    for pl in plans:
        pl.close()
    out.update({"workload": f"grouped_{count}_problems_64_to_256_bf16_f32", "problems": count,
                "tiles": info["tiles"], "tile_n": info["tile_n"], "algorithmic_bytes": nbytes,
                "frac_hbm": out["grouped"]["GB/s"] / peaks["hbm_gbs"]})
    if compare_singles:
        out["speedup_vs_one_call_per_problem"] = out["one_call_per_problem"]["ms"] / out["grouped"]["ms"]
    return out


def fused_attention_measure(dev, stream, steps, flush, peaks, pair_ms=None, batch=128, L=2048,
                            D=128):
    """O = softmax(alpha Q K^T) V in one launch (bf16 in and out, fp32
    accumulate), on the attention pair's shape: CUDA events per step with the
    L2 flushed before each.  ``pair_ms`` (the two products of the unfused pair,
    timed separately) is reported beside it."""
    import torch
    from dense_matmul_tensor_gb300 import bmm
    from dense_matmul_tensor_gb300 import workloads as wl
    alpha = float(np.float32(1.0 / np.sqrt(D)))
    g = torch.Generator(device=dev)
    g.manual_seed(4000)
    q, k, v = (torch.randn(batch * L * D, generator=g, device=dev).to(torch.bfloat16)
               for _ in range(3))
    o = torch.empty_like(q)
    plan = bmm.AttnPlan(bmm.make_attn_desc(batch=batch, Lq=L, Lk=L, D=D, alpha=alpha))
    for i in range(3):
        flush.fill_(i & 0xFF)
        plan.run(q, k, v, o, stream)
    torch.cuda.synchronize()
    reps = max(3, min(steps, 20))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(reps)]
    with torch.cuda.stream(stream):
        for i in range(reps):
            flush.fill_(i & 0xFF)
            ev[i][0].record(stream)
            plan.run(q, k, v, o, stream)
            ev[i][1].record(stream)
    torch.cuda.synchronize()
    st, word = plan.device_error()
    plan.close()
    if st != bmm.BMM_OK:
        raise RuntimeError(f"device error {word:#x} in the fused attention")
    ms = statistics.fmean(a.elapsed_time(b) for a, b in ev)
    flops = 4.0 * batch * L * L * D
    nbytes = 4.0 * batch * L * D * 2
    name = f"attn_fused_b{batch}_{L}x{L}x{D}_bf16"
    tf = flops / (ms * 1e-3) / 1e12
    # two products of 2 L^2 D flops per batch item against Q, K, V and O once
    # each: about 1000 flops per byte, far right of the ridge: tensor bound
    out = {"workload": name, "ms": ms, "TFLOP/s": tf, "GB/s": nbytes / (ms * 1e-3) / 1e9,
           "exp2_per_s": batch * L * L / (ms * 1e-3),
           "roofline": {"bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops"],
                        "unit": "TFLOP/s", "frac": tf / peaks["bf16_tflops"],
                        "traffic": NCU_TRAFFIC.get((kernel_source_hash(ATTN_SOURCES), name)),
                        "ncu_tensor_pipe_active_pct": NCU_TENSOR_ACTIVE_PCT.get(
                            (kernel_source_hash(ATTN_SOURCES), name)),
                        "algorithmic_flops_per_launch": flops,
                        "algorithmic_bytes_per_launch": nbytes},
           "kernel": "attn_fwd_kernel", "launches_per_step": 1}
    if pair_ms is not None:
        out["pair_qk_plus_pv_ms"] = pair_ms
        out["speedup_vs_pair"] = pair_ms / ms
    return out


def metric_value(p, ms):
    return p.flops() / (ms * 1e-3) / 1e12  # TFLOP/s


# ------------------------------------------------------------ CPU oracle

class OracleSample:
    """The fp64 oracle on the first ``rows`` rows of C (batch item 0, full N
    and K).  ``calibrate`` picks ``rows`` from a short probe so that one run
    takes about ``target_s`` seconds."""

    def __init__(self, p, threads=None):
        import oracle
        from dense_matmul_tensor_gb300 import workloads as wl
        self.oracle = oracle
        self.p = p
        self.x = wl.make_inputs(wl.Problem(**{**p.__dict__, "batch": 1}))
        self.cores = threads or oracle.host_threads()
        self.kw = dict(p.oracle_kwargs(), batch=1)
        self.rows = max(1, min(p.M, 32))

    def run(self, rows=None):
        rows = rows or self.rows
        k = dict(self.kw, M=rows)
        A = self.x.A if self.p.transA else self.x.A[: rows * self.kw["lda"]]
        t = time.perf_counter()
        self.oracle.bmm(A, self.x.B, self.x.C_in, threads=self.cores, **k)
        dt = time.perf_counter() - t
        return 2.0 * rows * self.p.N * self.p.K / dt / 1e12, dt

    def calibrate(self, target_s):
        probe = max(1, min(self.p.M, 32))
        _, dt = self.run(probe)
        self.rows = int(max(1, min(self.p.M, round(probe / max(dt, 1e-6) * target_s))))
        return self.rows


# ------------------------------------------------------------------ main

def reduce_max(x: float, world: int, device=None) -> float:
    """Max of ``x`` over all ranks (the slowest rank sets the job's time)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_rank: float, world: int, ms_slowest: float) -> float:
    """Weak scaling: every rank does ``flops_per_rank``; the job takes as long
    as its slowest rank."""
    return world * flops_per_rank / (ms_slowest * 1e-3) / 1e12


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def main():
    args = parse()
    world, rank, local = dist_env()
    import dataclasses
    from dense_matmul_tensor_gb300 import workloads as wl
    p = wl.WORKLOADS[args.workload]
    if args.batch is not None:
        p = dataclasses.replace(p, batch=args.batch, name=f"{p.name}@batch{args.batch}")

    if args.impl == "reference":
        if rank != 0:
            return
        total = args.steps + args.warmup
        sampler = OracleSample(p)
        rows = sampler.calibrate(max(0.02, min(10.0, 120.0 / max(total, 1))))
        cores = sampler.cores
        vals = []
        for i in range(total):
            v, dt = sampler.run()
            if i >= args.warmup:
                vals.append((v, dt))
        value = statistics.median(v for v, _ in vals)
        ms = statistics.median(dt for _, dt in vals) * 1e3
        line = {"impl": "reference", "metric": METRIC,
                "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": p.name, "batch": p.batch, "M": p.M, "N": p.N, "K": p.K,
                           "transA": p.transA, "transB": p.transB, "inputs": p.type_ab,
                           "output": p.type_c},
                "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                                 "sample": f"first {rows} of {p.M} rows of C per step (fp64 oracle, "
                                           f"{cores} threads)"},
                "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    import torch
    import torch.distributed as dist
    from dense_matmul_tensor_gb300 import bmm

    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    bmm.load_library()

    def barrier():
        if world > 1:
            dist.barrier()

    if args.grouped_only:
        peaks_now, _ = load_peaks()
        entry = grouped_measure(dev, torch.cuda.current_stream(), args.steps, peaks_now, compare_singles=False)
        if rank == 0:
            print(json.dumps(entry), flush=True)
        return
    if args.attn_only is not None:
        flush_buf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
        peaks_now, _ = load_peaks()
        entry = fused_attention_measure(dev, torch.cuda.current_stream(), args.steps, flush_buf,
                                        peaks_now, batch=args.attn_only)
        if rank == 0:
            print(json.dumps(entry), flush=True)
        return

    def max_over_ranks(x):
        return reduce_max(x, world, dev)

    peaks, peak_src = load_peaks()
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    A, B, C = (t.to(dev) for t in host_inputs(p))

    props = torch.cuda.get_device_properties(dev)
    clocks = ClockSampler(str(getattr(props, "uuid", "")))
    clocks.start()
    ms_list, info, launches, (t0, t1) = time_device(p, A, B, C, args.steps, max(args.warmup, 3),
                                                     flush, stream, barrier)
    clocks.stop()
    ms_mean = statistics.fmean(ms_list)
    ms_step = max_over_ranks(ms_mean)
    value = whole_job_tflops(p.flops(), world, ms_step)

    # The bound follows the workload's arithmetic intensity against the ridge
    # of the measured peaks (about 290 FLOP/byte): the square GEMM is tensor
    # bound, the skinny and attention shapes HBM bound.
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    tensor_bound = p.flops() / p.algorithmic_bytes() >= ridge
    if tensor_bound:
        achieved = p.flops() / (ms_mean * 1e-3) / 1e12
        peak, unit, per_launch = peaks["bf16_tflops"], "TFLOP/s", {"algorithmic_flops_per_launch": p.flops()}
    else:
        achieved = p.algorithmic_bytes() / (ms_mean * 1e-3) / 1e9
        peak, unit, per_launch = peaks["hbm_gbs"], "GB/s", {"algorithmic_bytes_per_launch": p.algorithmic_bytes()}
    roof = {"bound": "tensor" if tensor_bound else "hbm", "achieved": achieved, "peak": peak,
            "unit": unit, "frac": achieved / peak,
            "traffic": NCU_TRAFFIC.get((kernel_source_hash(), p.name)),
            "kernel": (f"bmm_tc2_kernel<{info.tile_n}> (CTA pairs)" if info.cta_pair
                       else f"bmm_tc_kernel<{info.tile_n}>"),
            "peak_source": f"{peak_src} " + ("bf16 burst" if tensor_bound else "HBM copy"),
            **per_launch,
            "ncu_tensor_pipe_active_pct": NCU_TENSOR_ACTIVE_PCT.get((kernel_source_hash(), p.name)),
            "ms_per_launch_median": statistics.median(ms_list),
            "ms_per_launch_best": min(ms_list)}

    line = {"metric": METRIC,
            "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": p.name, "batch": p.batch, "M": p.M, "N": p.N, "K": p.K,
                       "transA": p.transA, "transB": p.transB, "inputs": f"{p.type_ab} {p.dist_ab}",
                       "output": p.type_c, "alpha": p.alpha, "beta": p.beta,
                       "l2": f"flushed: {FLUSH_BYTES >> 20} MB write between timed steps",
                       "tile": [info.tile_m, info.tile_n, info.tile_k],
                       # ring depth of this launch: pair launches writing bf16 C by box stores take the deeper ring
                       "stages": (info.stages_bf16_box if (info.cta_pair and p.type_c == "bf16" and p.beta == 0.0)
                                  else info.stages),
                       "cta_pair": bool(info.cta_pair),
                       "parallelism": f"{world} independent replicas" if world > 1 else "1 GPU"},
            "roofline": roof,
            "gpu_launches": launches * args.steps,
            "clocks": clocks.summary(t0, t1)}

    if not args.no_e2e:
        e2e_steps = max(5, min(args.steps, 50))
        ms_e, h2d, d2h, chunks = time_e2e(p, e2e_steps, 3, stream, dev)
        ms_e = max_over_ranks(ms_e)
        line["e2e"] = {"value": whole_job_tflops(p.flops(), world, ms_e), "unit": "TFLOP/s",
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                       "ms_per_step": ms_e, "api": "bmm_host_run",
                       "chunks": chunks[0], "chunked_by": "rows" if chunks[1] else "batch items"}

    if not args.no_other:
        other = []
        for name, q in wl.WORKLOADS.items():
            if name == p.name:
                continue
            qa, qb, qc = gpu_inputs(q, dev, 1000 * q.seed)
            torch.cuda.synchronize()
            qs = min(args.steps, 20)
            mq, qinfo, _, _ = time_device(q, qa, qb, qc, qs, 3, flush, stream, lambda: None)
            mqm = statistics.fmean(mq)
            gbs = q.algorithmic_bytes() / (mqm * 1e-3) / 1e9
            tf = q.flops() / (mqm * 1e-3) / 1e12
            entry = {"workload": name, "ms": mqm, "TFLOP/s": tf,
                     "frac_bf16_peak": tf / peaks["bf16_tflops"], "GB/s": gbs,
                     "frac_hbm": gbs / peaks["hbm_gbs"],
                     "intensity_flop_per_byte": q.flops() / q.algorithmic_bytes(),
                     "tile_n": qinfo.tile_n, "swap_ab": qinfo.swap_ab,
                     "cta_pair": qinfo.cta_pair,
                     "pack": [qinfo.pack_a, qinfo.pack_b]}
            if qinfo.pack_a == 1 or qinfo.pack_b == 1:
                # the same product with the kernels' row loader instead of the
                # staging copy (pack 2: read in place, no workspace)
                os.environ["DMT_BMM_LDG"] = "1"
                try:
                    ml, linfo, _, _ = time_device(q, qa, qb, qc, qs, 3, flush, stream, lambda: None)
                finally:
                    del os.environ["DMT_BMM_LDG"]
                entry["row_loader"] = {"ms": statistics.fmean(ml), "pack": [linfo.pack_a, linfo.pack_b]}
            other.append(entry)
            del qa, qb, qc
            torch.cuda.empty_cache()
        line["other_workloads"] = other
        # a GEMM whose tile count is no multiple of the CTA pairs, against the
        # headline's rate
        q = wl.UNEVEN_GEMM
        qa, qb, qc = gpu_inputs(q, dev, 1000 * q.seed)
        torch.cuda.synchronize()
        mq, qinfo, _, _ = time_device(q, qa, qb, qc, min(args.steps, 50), 3, flush, stream, lambda: None)
        mqm = statistics.fmean(mq)
        tf = q.flops() / (mqm * 1e-3) / 1e12
        line["uneven_gemm"] = {"workload": q.name, "ms": mqm, "TFLOP/s": tf, "frac_bf16_peak": tf / peaks["bf16_tflops"],
                               "vs_headline": tf / value, "tile_n": qinfo.tile_n, "tiles": qinfo.tiles,
                               "stream_k_tiles": qinfo.sk_tiles}
        del qa, qb, qc
        torch.cuda.empty_cache()
        pair = {e["workload"]: e["ms"] for e in other}
        qk, pv = wl.ATTN_QK.name, wl.ATTN_PV.name
        pair_ms = pair[qk] + pair[pv] if qk in pair and pv in pair else None
        line["fused_attention"] = fused_attention_measure(dev, stream, args.steps, flush, peaks,
                                                          pair_ms)
        line["grouped"] = grouped_measure(dev, stream, args.steps, peaks)

    if rank == 0 and not args.no_cpu:
        sampler = OracleSample(p)
        rows = sampler.calibrate(15.0)
        v, dt = sampler.run()
        cores = sampler.cores
        line["cpu_baseline"] = {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                                "sample": f"first {rows} of {p.M} rows of C, full N and K "
                                          f"({2 * rows * p.N * p.K / 1e9:.1f} GFLOP in {dt:.1f} s)"}
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
