#!/usr/bin/env python3
"""Benchmark: GEMM TFLOPS (2MNK / device-timed median) and fraction of the GB300 roofline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one gemm_run of the workload (plan cached, inputs resident in HBM).
Each timed step has its own CUDA-event pair on the launching stream; between
steps a 512 MiB buffer is written to flush L2 (outside the event pair).  The
reported time is the median step (the pages time the median of 100 runs:
"SGEMM ... 83% of cuBLAS", sec. 4.1).  Default workload: FP32 SGEMM
4096^3 on the CUDA-core path (that page's headline size).

Multi-GPU: the GEMM does not need a collective; each rank runs an independent
replica on its own GPU (weak scaling) and the per-step times are max-reduced
over ranks.  Prints one JSON line on rank 0.

--impl reference times the FP64 CPU oracle (the only comparison arm this
project has) on a bounded sample of the same workload on the host cores.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FP32_LANES_PER_SM = 128          # FP32 FMA lanes per SM (4 partitions x 32)
L2_FLUSH_BYTES = 512 << 20       # > 129 MB L2
TF32_PER_BF16 = 1.1 / 2.25         # nominal dense TF32 / BF16 tensor rates


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="sgemm_4096")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-extra", action="store_true", help="skip the secondary workloads")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-sweep", action="store_true", help="skip the ragged-sweep bucket summary")
    return ap.parse_args()


# ----------------------------------------------------------------- distributed
def dist_setup(n: int):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
        return rank, ws, local, dist
    return 0, 1, 0, None


def max_over_ranks(values: list[float], dist, device) -> list[float]:
    """Element-wise max of a per-step time list over all ranks."""
    if dist is None:
        return values
    import torch
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.cpu().tolist()


def barrier(dist):
    if dist is not None:
        dist.barrier()


# ----------------------------------------------------------------- helpers
def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "sm_max_mhz": 2070.0}, "fallback"


KERNEL_SOURCES = {"tc": ("tc_kernel.cuh", "tc_sm103.cu", "tc_any_kn.cu", "tc_any_nk.cu",
                         "tc_spec_kn.cu", "tc_spec_nk.cu", "tc_sk_kn.cu", "tc_sk_nk.cu"),
                  "ffma": ("sgemm_ffma.cu",),
                  "skinny": ("aux_kernels.cu", "skinny_tma.cu"),
                  "tf32x3": ("tc_kernel.cuh", "tc_any_nk.cu")}


def source_hash(kernel: str) -> str:
    """Hash of the files that make up one kernel family (its .cu files and the shared headers)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "dense_gemm_13_gb300", "csrc")
    for f in (*KERNEL_SOURCES[kernel], "epilogue.cuh", "ptx.cuh", "internal.h"):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str, root: str = ROOT):
    """DRAM bytes per launch recorded from an ncu capture (profiles/traffic.json), if the
    kernel's sources still hash the same as when the counters were taken, else None."""
    path = os.path.join(root, "profiles", "traffic.json")
    if not os.path.exists(path) or kernel not in KERNEL_SOURCES:
        return None
    with open(path) as f:
        rec = json.load(f).get(f"{kernel}/{workload}")
    if not rec or rec.get("source_hash") != source_hash(kernel):
        return None
    return float(rec["dram_bytes_per_launch"])


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sms, maxs, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sms.append(float(f[1]))
                maxs.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sms:
            return None
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxs), "samples": len(sms),
                "reasons": sorted(reasons)}


# ----------------------------------------------------------------- GPU arm
def workload_by_name(name: str):
    """A named workload, or one triple of the ragged sweep as "sweep:M,N,K"."""
    from dense_gemm_13_gb300.inputs import WORKLOADS, sweep_workload
    if name.startswith("sweep:"):
        M, N, K = (int(x) for x in name[len("sweep:"):].split(","))
        return sweep_workload(M, N, K)
    return WORKLOADS[name]


def make_device_inputs(w, seed, device):
    t = w.make(seed)
    dev = {k: (v.to(device) if v is not None else None) for k, v in t.items()}
    return t, dev


def make_plan(g13, w, flags=0):
    bt = w.batch
    ep = g13.Epilogue(b_layout=w.b_layout, out_dtype=w.out_dtype, bias=w.bias, act=w.act,
                      residual=w.residual, beta=w.beta, batch=bt,
                      stride_a=w.M * w.K if bt > 1 else 0, stride_b=w.N * w.K if bt > 1 else 0,
                      stride_c=w.M * w.N if bt > 1 else 0, stride_r=w.M * w.N if (bt > 1 and w.residual) else 0,
                      flags=flags)
    ldb = w.N if w.b_layout == "kn" else w.K
    return g13.gemm_plan(w.dtype, w.M, w.N, w.K, w.K, ldb, w.N, ep)


def time_device(g13, torch, w, plan, dev, steps, warmup, dist, device, C):
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    sp = stream.cuda_stream
    args = (dev["A"].data_ptr(), dev["B"].data_ptr(), C.data_ptr(),
            dev["bias"].data_ptr() if dev["bias"] is not None else None,
            dev["R"].data_ptr() if dev["R"] is not None else None, float(w.alpha), sp)
    L = g13.lib()
    for _ in range(warmup):
        flush.fill_(1.0)
        rc = L.gemm_run(plan.handle, *args)
        assert rc == 0, rc
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    torch.cuda.synchronize()
    barrier(dist)
    torch.cuda.synchronize()
    region0 = torch.cuda.Event(enable_timing=True)
    region1 = torch.cuda.Event(enable_timing=True)
    region0.record(stream)
    for i in range(steps):
        flush.fill_(float(i))
        starts[i].record(stream)
        rc = L.gemm_run(plan.handle, *args)
        ends[i].record(stream)
        assert rc == 0, rc
    region1.record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    torch.cuda.synchronize()
    times = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    st = g13.gemm_plan_status(plan)
    assert st == 0, f"device status {st}"
    return times, region0.elapsed_time(region1)


def time_e2e(g13, torch, w, plan, host, steps, warmup, device):
    """Same GEMM with host buffers: pinned H2D of the inputs, gemm_run, D2H of C, every step.

    Two measurements.  Serial: one stream, each step's copies and GEMM back to back, the
    median step.  Pipelined (the reported value): two sets of device buffers, a copy-in,
    a compute and a copy-out stream ordered by events, so step i's copies overlap the
    GEMMs of steps i - 1 and i + 1; whole-job time from the first copy-in to the last
    copy-out, divided by the steps.  Every step still copies its own inputs in and its
    result out inside the timed region.
    """
    stream = torch.cuda.current_stream()
    hp = {k: (v.pin_memory() if v is not None else None) for k, v in host.items()}
    odt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[w.out_dtype]
    shape = (w.M, w.N) if w.batch == 1 else (w.batch, w.M, w.N)
    slots = []
    for _ in range(2):
        dv = {k: (torch.empty_like(v, device=device) if v is not None else None)
              for k, v in host.items()}
        slots.append((dv, torch.empty(shape, dtype=odt, device=device),
                      torch.empty(shape, dtype=odt).pin_memory()))
    h2d = sum(v.numel() * v.element_size() for v in hp.values() if v is not None)
    d2h = slots[0][2].numel() * slots[0][2].element_size()

    def step(slot, s_in, s_run, s_out, ev):
        dv, C, Ch = slots[slot]
        with torch.cuda.stream(s_in):
            if ev is not None:
                s_in.wait_event(ev["ran"][slot])      # the slot's inputs were consumed
            for k, v in hp.items():
                if v is not None:
                    dv[k].copy_(v, non_blocking=True)
            if ev is not None:
                ev["in"][slot].record(s_in)
        with torch.cuda.stream(s_run):
            if ev is not None:
                s_run.wait_event(ev["in"][slot])
                s_run.wait_event(ev["out"][slot])     # the slot's C was read out
            g13.gemm_run(plan, dv["A"], dv["B"], C, dv["bias"], dv["R"], w.alpha,
                         stream=s_run.cuda_stream)
            if ev is not None:
                ev["ran"][slot].record(s_run)
        with torch.cuda.stream(s_out):
            if ev is not None:
                s_out.wait_event(ev["ran"][slot])
            Ch.copy_(C, non_blocking=True)
            if ev is not None:
                ev["out"][slot].record(s_out)

    # serial: everything on the current stream
    for i in range(warmup):
        step(i % 2, stream, stream, stream, None)
    torch.cuda.synchronize()
    times = []
    for i in range(steps):
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        step(i % 2, stream, stream, stream, None)
        s1.record(stream)
        s1.synchronize()
        times.append(s0.elapsed_time(s1))
    serial_ms = statistics.median(times)

    # pipelined: copy-in, compute and copy-out streams
    s_in, s_run, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "ran", "out")}
    for e_list in ev.values():
        for e in e_list:
            e.record(stream)
    torch.cuda.synchronize()
    for i in range(warmup):
        step(i % 2, s_in, s_run, s_out, ev)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(s_in)
    for i in range(steps):
        step(i % 2, s_in, s_run, s_out, ev)
    t1.record(s_out)
    torch.cuda.synchronize()
    pipe_ms = t0.elapsed_time(t1) / steps
    return pipe_ms, serial_ms, h2d, d2h


def roofline_for(w, kernel, ms, pk, pk_kind, num_sms=152):
    """Roofline object for the workload's main kernel (achieved from the median launch).
    num_sms: the SMs of the plan's device (the FP32 FMA peak scales with it)."""
    flops = w.flops
    if kernel == "ffma":
        sm_count = num_sms
        peak = sm_count * FP32_LANES_PER_SM * 2 * pk.get("sm_max_mhz", 2070.0) * 1e6 / 1e12
        return {"bound": "alu", "achieved": flops / (ms * 1e-3) / 1e12, "peak": round(peak, 2),
                "unit": "TFLOP/s", "peak_source": f"derived: {sm_count} SMs x {FP32_LANES_PER_SM} FP32 "
                f"FMA lanes x 2 x {pk.get('sm_max_mhz', 2070.0):.0f} MHz"}
    if kernel == "tf32x3":
        # three TF32 MMAs per product on the tensor cores; TF32 runs at the nominal
        # 1.1 / 2.25 of the BF16 rate, applied to the measured BF16 peak
        peak = pk["bf16_tflops"] * TF32_PER_BF16
        return {"bound": "tensor", "achieved": 3 * flops / (ms * 1e-3) / 1e12,
                "peak": round(peak, 1), "unit": "TFLOP/s (TF32 MMA work, 3 x 2MNK)",
                "peak_source": f"{pk_kind} bf16_tflops x {TF32_PER_BF16:.3f} (nominal TF32/BF16)",
                "frac_basis": "against a nominal ratio: no TF32 peak is measured on this GPU"}
    byts = w.algorithmic_bytes()
    ai = flops / byts
    bw = pk["hbm_gbs"] * 1e9
    tens = pk["bf16_tflops"] * 1e12
    if ai * bw < tens:
        return {"bound": "hbm", "achieved": byts / (ms * 1e-3) / 1e9, "peak": pk["hbm_gbs"],
                "unit": "GB/s", "peak_source": f"{pk_kind} hbm_gbs"}
    return {"bound": "tensor", "achieved": flops / (ms * 1e-3) / 1e12, "peak": pk["bf16_tflops"],
            "unit": "TFLOP/s", "peak_source": f"{pk_kind} bf16_tflops (burst; fp16 nominal rate = bf16)"}


def sweep_summary(g13, torch, device, pk, pk_kind, reps=8):
    """Times all 343 ragged sweep triples (BF16, C = 0.5 AB + R) and summarises per bucket.

    Buckets by the dispatcher's kernel and regime: skinny (M or N <= 4), tensor-core
    problems that are HBM-bound by their arithmetic intensity, and compute-bound ones.
    Each triple: 2 warm-up runs, then `reps` runs each between an L2 flush and a CUDA
    event pair; median time.  Roofline fraction as in the main line.  Besides the
    medians (which the many launch-latency-bound tiny triples dominate), each bucket
    and the whole sweep report aggregate_frac = sum of the triples' roofline times /
    sum of their measured times: the fraction for running the bucket as one job.
    """
    from dense_gemm_13_gb300.inputs import SWEEP_SIZES, sweep_workload
    big = max(SWEEP_SIZES)
    gen = torch.Generator(device=device)
    gen.manual_seed(0)
    Ab = (torch.rand((big, big), generator=gen, device=device) * 2 - 1).to(torch.bfloat16)
    Bb = (torch.rand((big, big), generator=gen, device=device) * 2 - 1).to(torch.bfloat16)
    Rb = torch.rand((big, big), generator=gen, device=device) * 2 - 1
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream()
    rows = []
    for M in SWEEP_SIZES:
        for N in SWEEP_SIZES:
            for K in SWEEP_SIZES:
                w = sweep_workload(M, N, K)
                A = Ab[:M, :K].contiguous()
                B = Bb[:K, :N].contiguous()
                R = Rb[:M, :N].contiguous()
                C = torch.empty((M, N), dtype=torch.float32, device=device)
                plan = make_plan(g13, w)
                kern = plan.info()["config"].kernel
                ts = []
                for i in range(2 + reps):
                    flush.fill_(float(i))
                    s0 = torch.cuda.Event(enable_timing=True)
                    s1 = torch.cuda.Event(enable_timing=True)
                    s0.record(stream)
                    g13.gemm_run(plan, A, B, C, None, R, w.alpha)
                    s1.record(stream)
                    if i >= 2:
                        ts.append((s0, s1))
                torch.cuda.synchronize()
                ms = statistics.median(a.elapsed_time(b) for a, b in ts)
                r = roofline_for(w, kern, ms, pk, pk_kind, plan.info()["num_sms"])
                if kern == "skinny" or min(M, N) <= 16:
                    bucket = "skinny"
                elif r["bound"] == "hbm":
                    bucket = "tc_hbm_bound"
                else:
                    bucket = "tc_compute_bound"
                rows.append((bucket, w.flops / (ms * 1e-3) / 1e12, r["achieved"] / r["peak"], ms))
                del plan, A, B, R, C
    out = {}
    for bucket in ("skinny", "tc_hbm_bound", "tc_compute_bound"):
        sel = [x for x in rows if x[0] == bucket]
        if not sel:
            continue
        out[bucket] = {"triples": len(sel),
                       "median_tflops": round(statistics.median(x[1] for x in sel), 3),
                       "median_frac": round(statistics.median(x[2] for x in sel), 4),
                       "min_frac": round(min(x[2] for x in sel), 4),
                       "max_frac": round(max(x[2] for x in sel), 4),
                       # the bucket as one job: sum of roofline times / sum of measured times
                       "aggregate_frac": round(sum(x[2] * x[3] for x in sel) /
                                               sum(x[3] for x in sel), 4),
                       "ms": round(sum(x[3] for x in sel), 3)}
    out["total_ms"] = round(sum(x[3] for x in rows), 3)
    out["aggregate_frac"] = round(sum(x[2] * x[3] for x in rows) / sum(x[3] for x in rows), 4)
    return out


def cpu_baseline(w, host, budget_s=12.0):
    """The FP64 oracle, as it stands, on sampled rows of the workload (host cores)."""
    import numpy as np
    import oracle
    from dense_gemm_13_gb300.inputs import host_view
    A, B = host_view(host["A"]), host_view(host["B"])
    bias = host["bias"].numpy() if host["bias"] is not None else None
    R = host["R"].numpy() if host["R"] is not None else None
    kw = dict(b_layout=w.b_layout, dtype=w.dtype, alpha=w.alpha, bias=bias, act=w.act, R=R,
              beta=w.beta, out_dtype=w.out_dtype)
    threads = oracle.max_threads()
    # calibrate on a few rows, then size the sample for ~budget_s
    r0 = max(1, min(w.M, threads))
    t0 = time.perf_counter()
    oracle.gemm(A, B, rows=np.arange(r0), **kw)
    t1 = time.perf_counter() - t0
    rows = int(min(w.M, max(r0, r0 * budget_s / max(t1, 1e-6))))
    rows = max(threads, rows // threads * threads) if rows >= threads else rows
    t0 = time.perf_counter()
    oracle.gemm(A, B, rows=np.arange(rows), **kw)
    dt = time.perf_counter() - t0
    flops = 2.0 * rows * w.N * w.K * w.batch
    return {"value": flops / dt / 1e12, "unit": "TFLOPS", "cores": threads, "kind": "oracle",
            "seconds": round(dt, 3),
            "sample": f"rows 0..{rows - 1} of {w.M} (all {w.N} columns, K={w.K}"
                      f"{', ' + str(w.batch) + ' batches' if w.batch > 1 else ''}), FP64 triple loop"}


def run_ours(args):
    import torch
    import dense_gemm_13_gb300 as g13
    from dense_gemm_13_gb300 import _build
    from dense_gemm_13_gb300.inputs import WORKLOADS

    rank, ws, local, dist = dist_setup(args.gpus)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if rank == 0 or not os.path.exists(_build.LIB):
        _build.build()
    barrier(dist)
    g13.load()
    pk, pk_kind = peaks()

    # "<workload>+3xtf32": the same FP32 workload with GEMM_FLAG_FP32_TENSOR
    base, _, mode = args.workload.partition("+")
    w = workload_by_name(base)
    host, dev = make_device_inputs(w, 0, device)
    plan = make_plan(g13, w, g13.FLAG_FP32_TENSOR if mode == "3xtf32" else 0)
    info = plan.info()
    kernel = info["config"].kernel
    odt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[w.out_dtype]
    C = torch.empty((w.M, w.N) if w.batch == 1 else (w.batch, w.M, w.N), dtype=odt, device=device)

    with ClockSampler(local) as clk:
        times, region_ms = time_device(g13, torch, w, plan, dev, args.steps, args.warmup, dist, device, C)
    times = max_over_ranks(times, dist, device)
    med = statistics.median(times)
    mean = statistics.fmean(times)
    value = w.flops * ws / (med * 1e-3) / 1e12

    result = {
        "metric": "GEMM TFLOPS (2MNK/s, device-timed median) and % of GB300 dtype roofline",
        "value": round(value, 3), "unit": "TFLOPS", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(med, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": args.workload, "M": w.M, "N": w.N, "K": w.K, "batch": w.batch,
                   "b_layout": w.b_layout, "out_dtype": w.out_dtype, "epilogue": {
                       "alpha": w.alpha, "bias": w.bias, "act": w.act, "residual": w.residual,
                       "beta": w.beta},
                   "kernel": info["config"].as_dict(), "l2": "flushed between steps (512 MiB write)",
                   "timing": "per-step CUDA events, median", "parallelism": f"replicas x{ws}"},
    }
    rf = roofline_for(w, kernel, mean, pk, pk_kind, info["num_sms"])
    rf["achieved"] = round(rf["achieved"], 3)
    rf["frac"] = round(rf["achieved"] / rf["peak"], 4)
    rf["timed_on"] = "mean launch duration over the timed steps"
    rf["traffic"] = recorded_traffic(kernel, w.name)
    result["roofline"] = rf
    result["gpu_launches"] = info["kernels_per_run"] * args.steps
    cs = clk.summary()
    if cs:
        result["clocks"] = cs
    if not args.no_e2e:
        e2e_ms, serial_ms, h2d, d2h = time_e2e(g13, torch, w, plan, host, max(10, args.steps // 5),
                                               3, device)
        result["e2e"] = {"value": round(w.flops * ws / (e2e_ms * 1e-3) / 1e12, 3), "unit": "TFLOPS",
                         "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                         "ms_per_step": round(e2e_ms, 4),
                         "serial_ms_per_step": round(serial_ms, 4),
                         "serial_value": round(w.flops * ws / (serial_ms * 1e-3) / 1e12, 3),
                         "how": "every step copies its pinned host inputs in, runs gemm_run and "
                                "copies C out; value: two buffer sets on copy-in / compute / "
                                "copy-out streams, whole-job time / steps; serial: one stream, "
                                "median step"}
    if not args.no_extra:
        extra = []
        for name in ("bf16_8192", "bf16_4096", "ffn1_bf16", "ffn1_f16", "ffn2_bf16", "qkt_bf16",
                     "qkt_softmax_bf16", "sgemm_256", "sgemm_4096+3xtf32"):
            if name == w.name:
                continue
            base, _, mode = name.partition("+")
            wx = WORKLOADS[base]
            hx, dx = make_device_inputs(wx, 0, device)
            px = make_plan(g13, wx, g13.FLAG_FP32_TENSOR if mode == "3xtf32" else 0)
            ox = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[wx.out_dtype]
            Cx = torch.empty((wx.M, wx.N) if wx.batch == 1 else (wx.batch, wx.M, wx.N), dtype=ox,
                             device=device)
            tx, _ = time_device(g13, torch, wx, px, dx, max(20, args.steps // 2), 5, dist, device, Cx)
            tx = max_over_ranks(tx, dist, device)
            mx = statistics.median(tx)
            kx = px.info()["config"].kernel
            r = roofline_for(wx, kx, statistics.fmean(tx), pk, pk_kind, px.info()["num_sms"])
            entry = {"workload": name, "tflops": round(wx.flops / (mx * 1e-3) / 1e12, 2),
                     "ms": round(mx, 4), "kernel": kx, "bn": px.info()["config"].bn,
                     "bound": r["bound"], "frac": round(r["achieved"] / r["peak"], 4)}
            if "frac_basis" in r:
                entry["frac_basis"] = r["frac_basis"]
            extra.append(entry)
            del dx, Cx, px
            torch.cuda.empty_cache()
        result["secondary"] = extra
    if not args.no_sweep and ws == 1:
        result["sweep"] = sweep_summary(g13, torch, device, pk, pk_kind)
    if rank == 0 and ws == 1 and not args.no_cpu:
        result["cpu_baseline"] = cpu_baseline(w, host)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_reference(args):
    """The FP64 oracle timed on host cores, K steps of a bounded row sample each."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import numpy as np
    import oracle
    from dense_gemm_13_gb300.inputs import host_view
    w = workload_by_name(args.workload.partition("+")[0])
    host = w.make(0)
    A, B = host_view(host["A"]), host_view(host["B"])
    bias = host["bias"].numpy() if host["bias"] is not None else None
    R = host["R"].numpy() if host["R"] is not None else None
    kw = dict(b_layout=w.b_layout, dtype=w.dtype, alpha=w.alpha, bias=bias, act=w.act, R=R,
              beta=w.beta, out_dtype=w.out_dtype)
    threads = oracle.max_threads()
    rows = max(1, min(w.M, threads))
    # size each step so the whole run stays within ~2 minutes
    t0 = time.perf_counter()
    oracle.gemm(A, B, rows=np.arange(rows), **kw)
    t1 = time.perf_counter() - t0
    per_step_budget = 120.0 / max(1, args.steps + args.warmup)
    scale = max(1, int(per_step_budget / max(t1, 1e-6)))
    rows = min(w.M, rows * scale)
    for i in range(args.warmup):
        oracle.gemm(A, B, rows=np.arange(rows), **kw)
    times = []
    for i in range(args.steps):
        t0 = time.perf_counter()
        oracle.gemm(A, B, rows=np.arange(rows), **kw)
        times.append(time.perf_counter() - t0)
    med = statistics.median(times)
    flops = 2.0 * rows * w.N * w.K * w.batch
    val = flops / med / 1e12
    out = {"impl": "reference", "metric": "GEMM TFLOPS (2MNK/s, device-timed median) and % of GB300 "
           "dtype roofline", "value": round(val, 6), "unit": "TFLOPS", "n_gpus": args.gpus,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(med * 1e3, 3),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic", "config": {"workload": args.workload, "M": w.M, "N": w.N, "K": w.K,
                                           "batch": w.batch},
           "cpu_baseline": {"value": round(val, 6), "unit": "TFLOPS", "cores": threads,
                            "kind": "oracle",
                            "sample": f"rows 0..{rows - 1} of {w.M} per step (all {w.N} columns, "
                                      f"K={w.K}), FP64 triple loop, wall clock"},
           "e2e": {"value": round(val, 6), "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
