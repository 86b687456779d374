#!/usr/bin/env python3
"""Benchmark of the GB300 FP32 SGEMM: GFLOP/s on the 2048^3 workload.

One step is one sgemm_run call (C = A*B, row-major FP32, 2*M*N*K flops) on
inputs already resident in HBM.  L2 is flushed before every step (a 256 MiB
write, read back so that the lines left are clean) and each GEMM is timed with CUDA events on the stream it runs on; steps
are queued in batches behind a short hold kernel, so that the host has
submitted a GEMM before the device reaches its start event.  The line printed
also carries:
  roofline      the GEMM kernel against the FP32 FFMA peak (alu bound), with
                the same-run FFMA probe beside it;
  e2e           the same metric through sgemm_run_host: host->device copies of
                A and B, the GEMM and the device->host copy of C, per step;
  cpu_baseline  the CPU oracle timed on this host's cores on a bounded sample
                of the same workload;
  secondary     the 4092^3 (alpha=0.5, beta=2) workload, timed the same way;
  cublas_context  the same products through cuBLAS FP32 with TF32 off (context);
  tensor_core_3xtf32  the separate 3xTF32 entry point (sgemm_run_3xtf32) on
                the 2048^3 and 4092^3 workloads: FP32 GFLOP/s, and its MMA
                kernel against the TF32 tensor peak (3 TF32 products per FP32
                product); reported apart from the FP32 metric;
  sets          the value over the first and the second half of the timed steps;
  clocks        SM clocks sampled with nvidia-smi during the timed region.

--impl reference times the CPU oracle instead (rank 0 only).
Several GPUs (torchrun) run independent replicas: no data exchange.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import datagen  # noqa: E402

WORKLOADS = {
    "s2_2048": "sgemm 2048x2048x2048 fp32 row-major alpha=1 beta=0 A,B U[-1,1)",
    "s3_4092": "sgemm 4092x4092x4092 fp32 row-major alpha=0.5 beta=2 A,B,C U[-1,1)",
    "s4_rect": "sgemm 8192x6144x2048 fp32 row-major alpha=1 beta=0 A,B N(0,1)",
    "s5_odd": "sgemm 1023x1025x513 fp32 row-major alpha=1 beta=0 A,B N(0,1)",
    "s6_skinny": "sgemm 16x8192x8192 fp32 row-major alpha=1 beta=0 A,B U[-1,1)",
    "s1_128": "sgemm 128x128x128 fp32 row-major alpha=1 beta=0 A,B U[-1,1)",
    "s7_gemv": "sgemm 1x8192x8192 fp32 row-major alpha=1 beta=0 A,B U[-1,1) (GEMV)",
    "s8_2049": "sgemm 2049x2049x2049 fp32 row-major alpha=1 beta=0 A,B U[-1,1)",
    "s9_ax": "sgemm 8192x1x8192 fp32 row-major alpha=1 beta=0 A,B U[-1,1) (A x)",
}
METRIC = "SGEMM GFLOP/s at 4092^3 and 2048^3 FP32; % of GB300 FP32 FFMA peak"
FP32_LANES_PER_SM = 128
SM_MAX_MHZ = 2070.0  # GB300's maximum SM clock, used when nvidia-smi reports none
L2_FLUSH_BYTES = 256 << 20
HOLD_BATCH = 32
REFERENCE_SECONDS = 120.0


def nominal_fp32_tflops(sms, mhz=SM_MAX_MHZ):
    return sms * FP32_LANES_PER_SM * 2 * mhz * 1e6 / 1e12


# GB300's L2 (nominal 129 MB); a workload whose operands are larger is timed
# back to back, without a flush.
L2_BYTES_GB300 = 129 * 10**6


def streams_past_l2(cfg, l2_bytes=L2_BYTES_GB300):
    """True when the operands of one step are larger than L2, so that back-to-back
    steps already start with a cold cache (the timing rules' alternative to a
    flush): HBM-bound streaming workloads (s6, the GEMV, A x) and the largest
    compute-bound ones."""
    return algorithmic_bytes(cfg) > l2_bytes


def l2_note(name):
    if streams_past_l2(datagen.CONFIGS[name]):
        return ("GPU arm: operands larger than L2, so steps run back to back without a "
                "flush and one CUDA event pair brackets the K launches; the per-call time "
                "(flush, then one event pair per launch) is reported beside it; CPU "
                "reference arm: not applicable")
    return ("GPU arm: L2 flushed before every timed step (256 MiB write, then a read "
            "of it so no dirty lines remain); CPU reference arm: not applicable")


def workload_config(name):
    """The `config` object of a bench line: the workload alone (the same for
    the GPU arm and the reference arm), plus how L2 is handled."""
    cfg = datagen.CONFIGS[name]
    return {"workload": WORKLOADS[name], "M": cfg["M"], "N": cfg["N"], "K": cfg["K"],
            "alpha": cfg["alpha"], "beta": cfg["beta"], "seed": datagen.CONFIG_SEEDS[name],
            "l2": l2_note(name)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x, ws, device=None):
    """The largest value of x over all ranks (the slowest rank's time)."""
    if ws <= 1:
        return float(x)
    import torch
    import torch.distributed as tdist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(ws, steps, flops_per_step, slowest_total_s):
    """Whole-job GFLOP/s: every rank ran `steps` steps; the job took as long
    as its slowest rank's summed step time."""
    return ws * steps * flops_per_step / slowest_total_s / 1e9


def flops_of(cfg):
    return 2.0 * cfg["M"] * cfg["N"] * cfg["K"]


def algorithmic_bytes(cfg):
    """Read A and B once, read C if beta != 0, write C once (FP32)."""
    M, N, K = cfg["M"], cfg["N"], cfg["K"]
    return 4 * (M * K + K * N + M * N * (2 if cfg["beta"] != 0 else 1))


# Nominal dense tensor rates (PFLOP/s) on GB300: TF32 1.1, BF16 2.25.  The
# TF32 denominator is the measured BF16 rate scaled by their ratio.
TF32_PER_BF16 = 1.1 / 2.25


def measured_tf32_peak():
    """TF32 tensor peak (TFLOP/s): measured BF16 x nominal TF32/BF16, else the
    fallback BF16 figure x the same ratio."""
    try:
        pk = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        return (round(float(pk["bf16_tflops"]) * TF32_PER_BF16, 1),
                round(float(pk["bf16_tflops_sustained"]) * TF32_PER_BF16, 1),
                "MEASURED_PEAKS.json bf16_tflops x 1.1/2.25 (nominal TF32/BF16), of measured")
    except (OSError, KeyError, ValueError):
        return (round(1900.0 * TF32_PER_BF16, 1), round(1700.0 * TF32_PER_BF16, 1),
                "fallback 1.9 PFLOP/s bf16 x 1.1/2.25, of fallback")


def measured_hbm_peak():
    """Copy bandwidth measured by the pool's driver on GB300, else the fallback."""
    try:
        v = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))["hbm_gbs"]
        return float(v), "MEASURED_PEAKS.json hbm_gbs (copy, of measured)"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback 6.8 TB/s (of fallback)"


# --------------------------------------------------------------------------
# CPU oracle timing (the reference arm and the cpu_baseline object)
# --------------------------------------------------------------------------

def time_oracle(name, budget_s=12.0, threads=0):
    """Time the oracle on consecutive row blocks of workload `name` (wrapping
    around the matrix) until about budget_s of wall time is spent."""
    import oracle

    cfg, A, B, C = datagen.config_inputs(name)
    M, N, K = cfg["M"], cfg["N"], cfg["K"]
    nthreads = threads or oracle.default_threads()
    rows = min(M, max(nthreads, 1))
    total_rows = 0
    elapsed = 0.0
    start_row = 0
    while elapsed < budget_s:
        take = min(rows, M - start_row)
        idx = np.arange(start_row, start_row + take)
        t0 = time.perf_counter()
        oracle.sgemm_ref_flat(M, N, K, cfg["alpha"], A, K, B, N, cfg["beta"], C, N,
                              rows=idx, threads=nthreads, want_absprod=False)
        dt = time.perf_counter() - t0
        elapsed += dt
        total_rows += take
        start_row = (start_row + take) % M
        if dt < budget_s / 8:
            rows = min(M, rows * 2)
    gflops = 2.0 * total_rows * N * K / elapsed / 1e9
    return {
        "value": round(gflops, 3), "unit": "GFLOP/s", "cores": int(nthreads), "kind": "oracle",
        "sample": f"{total_rows} rows ({total_rows / M:.2f} x the {M} rows) of {name} "
                  f"({M}x{N}x{K}), fp64 triple loop, {elapsed:.1f} s wall on {nthreads} threads",
    }


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel's sources changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        rec = json.load(open(path))[kernel]
    except (OSError, KeyError, ValueError):
        return None
    if rec.get("workload") != workload:
        return None
    import hashlib
    h = hashlib.sha256()
    for f in rec.get("sources", []):
        try:
            h.update(open(os.path.join(ROOT, f), "rb").read())
        except OSError:
            return None
    if h.hexdigest() != rec.get("sources_sha256"):
        return None
    return rec.get("dram_bytes_per_launch")


# --------------------------------------------------------------------------
# Clock sampling
# --------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.out = None
        self.gpu_index = gpu_index

    def __enter__(self):
        try:
            import tempfile
            self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.out is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.out.flush()
        self.out.seek(0)
        lines = [l.strip() for l in self.out.read().splitlines() if l.strip()]
        path = self.out.name
        self.out.close()
        try:
            os.remove(path)
        except OSError:
            pass
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in lines:
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        busy = sorted(sm)[len(sm) // 2:] or sm  # upper half: the samples under load
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(smax),
                "power_w_max": max(power), "samples": len(sm), "reasons": sorted(reasons)}


# --------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------

def gpu_arm(args, ws, rank, local):
    import torch

    import dense_fp32_sgemm_gb300 as sg

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    sg.build()
    sg.library()
    num_sms = torch.cuda.get_device_properties(dev).multi_processor_count

    def device_inputs(name):
        cfg, A, B, C = datagen.config_inputs(name)
        M, N, K = cfg["M"], cfg["N"], cfg["K"]
        dA = torch.from_numpy(A).to(dev)
        dB = torch.from_numpy(B).to(dev)
        dC = torch.from_numpy(C).to(dev) if C is not None else torch.zeros(M * N, device=dev)
        return cfg, A, B, C, dA, dB, dC

    flush = torch.empty(L2_FLUSH_BYTES // 4, device=dev)
    flush_sink = torch.empty(1, device=dev)
    stream = torch.cuda.current_stream(dev)

    def flush_l2():
        # Evict A, B and C from L2 between steps: write a buffer twice the
        # size of L2, then read it back, so the lines left in L2 are clean and
        # the timed GEMM does not pay for writing the flush's dirty lines.
        flush.fill_(1.0)
        torch.sum(flush, dim=0, keepdim=True, out=flush_sink)

    def step(cfg, dA, dB, dC, entry=None):
        fn = getattr(sg, entry or args.entry)
        st = fn(cfg["M"], cfg["N"], cfg["K"], cfg["alpha"], dA.data_ptr(), cfg["K"],
                dB.data_ptr(), cfg["N"], cfg["beta"], dC.data_ptr(), cfg["N"], stream.cuda_stream)
        if st != 0:
            raise RuntimeError(f"{entry or args.entry}: " + sg.status_string(st))

    def timed(cfg, dA, dB, dC, steps, warmup, entry=None):
        for _ in range(warmup):
            step(cfg, dA, dB, dC, entry)
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        hold_ns = 2_000_000
        for b in range(0, len(evs), HOLD_BATCH):
            # The batch is queued behind a hold kernel that outlasts the host's
            # queueing of it, so no event pair brackets time the device spent
            # waiting for the host to submit the GEMM.
            sg.probe_hold(hold_ns, stream)
            h0 = time.perf_counter()
            for e0, e1 in evs[b:b + HOLD_BATCH]:
                flush_l2()
                e0.record(stream)
                step(cfg, dA, dB, dC, entry)
                e1.record(stream)
            host_ns = (time.perf_counter() - h0) * 1e9
            hold_ns = int(min(1e9, max(hold_ns, 2 * host_ns)))
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        if ws > 1:
            torch.distributed.barrier()
        st = sg.device_status(stream)
        if st != 0:
            raise RuntimeError("device status: " + sg.status_string(st))
        durs = [e0.elapsed_time(e1) / 1e3 for e0, e1 in evs]
        return durs, wall

    def timed_streamed(cfg, dA, dB, dC, steps, warmup, entry=None):
        """Steps back to back without a flush, for operands larger than L2: one
        event pair brackets each batch of up to HOLD_BATCH launches, queued
        behind a hold kernel; each step of a batch is given the batch's mean."""
        for _ in range(warmup):
            step(cfg, dA, dB, dC, entry)
        torch.cuda.synchronize()
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        hold_ns = 2_000_000
        batches = []
        for b in range(0, steps, HOLD_BATCH):
            n = min(HOLD_BATCH, steps - b)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            sg.probe_hold(hold_ns, stream)
            h0 = time.perf_counter()
            e0.record(stream)
            for _ in range(n):
                step(cfg, dA, dB, dC, entry)
            e1.record(stream)
            host_ns = (time.perf_counter() - h0) * 1e9
            hold_ns = int(min(1e9, max(hold_ns, 2 * host_ns)))
            batches.append((e0, e1, n))
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        if ws > 1:
            torch.distributed.barrier()
        st = sg.device_status(stream)
        if st != 0:
            raise RuntimeError("device status: " + sg.status_string(st))
        durs = []
        for e0, e1, n in batches:
            durs += [e0.elapsed_time(e1) / 1e3 / n] * n
        return durs, wall

    def timed_cublas(cfg, dA, dB, dC, steps, warmup):
        """The same product through cuBLAS FP32 (torch.mm / addmm with TF32
        off), timed like the GEMM: context for the reader, not a baseline."""
        M, N, K = cfg["M"], cfg["N"], cfg["K"]
        a, b = dA.view(M, K), dB.view(K, N)
        c_in = dC.view(M, N)
        out = torch.empty(M, N, device=dev)

        def one():
            if cfg["beta"] != 0:
                torch.addmm(c_in, a, b, beta=cfg["beta"], alpha=cfg["alpha"], out=out)
            elif cfg["alpha"] != 1:
                torch.mm(a, b, out=out).mul_(cfg["alpha"])
            else:
                torch.mm(a, b, out=out)

        for _ in range(warmup):
            one()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        for b0 in range(0, steps, HOLD_BATCH):
            sg.probe_hold(20_000_000, stream)
            for e0, e1 in evs[b0:b0 + HOLD_BATCH]:
                flush_l2()
                e0.record(stream)
                one()
                e1.record(stream)
        torch.cuda.synchronize()
        return [e0.elapsed_time(e1) / 1e3 for e0, e1 in evs]

    def ffma_probe(seconds_target, paired):
        sink = torch.zeros(4096, device=dev)
        blocks = num_sms * 4
        iters = 200
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        # calibrate
        sg.probe_ffma(paired, iters, blocks, sink.data_ptr(), stream)
        torch.cuda.synchronize()
        e0.record(stream)
        fl = sg.probe_ffma(paired, iters, blocks, sink.data_ptr(), stream)
        e1.record(stream)
        torch.cuda.synchronize()
        dt = e0.elapsed_time(e1) / 1e3
        iters = max(200, int(iters * min(seconds_target, 2.0) / max(dt, 1e-6)))
        best = 0.0
        rates = []
        t_end = time.perf_counter() + seconds_target
        while True:
            e0.record(stream)
            fl = sg.probe_ffma(paired, iters, blocks, sink.data_ptr(), stream)
            e1.record(stream)
            torch.cuda.synchronize()
            r = fl / (e0.elapsed_time(e1) / 1e3) / 1e12
            rates.append(r)
            best = max(best, r)
            if time.perf_counter() > t_end:
                break
        return {"burst": round(best, 3), "sustained": round(statistics.median(rates), 3)}

    def tf32_probe(seconds_target):
        """tcgen05 TF32 MMA rate (TFLOP/s) over all SMs: best and median of
        launches of about 10 ms each, for about seconds_target."""
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        iters = 2000
        sg.probe_tf32(iters, num_sms, stream)
        torch.cuda.synchronize()
        e0.record(stream)
        sg.probe_tf32(iters, num_sms, stream)
        e1.record(stream)
        torch.cuda.synchronize()
        dt = e0.elapsed_time(e1) / 1e3
        iters = int(min(1 << 18, max(2000, iters * 0.01 / max(dt, 1e-6))))
        rates = []
        t_end = time.perf_counter() + seconds_target
        while True:
            e0.record(stream)
            fl = sg.probe_tf32(iters, num_sms, stream)
            e1.record(stream)
            torch.cuda.synchronize()
            rates.append(fl / (e0.elapsed_time(e1) / 1e3) / 1e12)
            if time.perf_counter() > t_end:
                break
        if sg.device_status(stream) != 0:
            raise RuntimeError("TF32 probe: a bounded wait gave up")
        return {"burst": round(max(rates), 1), "sustained": round(statistics.median(rates), 1),
                "launches": len(rates), "iters": iters}

    def read_probe():
        sink = torch.zeros(4096, device=dev)
        buf = torch.ones(1 << 28, device=dev)  # 1 GiB, 8x the L2
        best = 0.0
        for _ in range(5):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            nb = sg.probe_read(buf.data_ptr(), buf.numel(), sink.data_ptr(), num_sms * 4, stream)
            e1.record(stream)
            torch.cuda.synchronize()
            best = max(best, nb / (e0.elapsed_time(e1) / 1e3) / 1e9)
        del buf
        return round(best, 1)

    gpu_index = 0
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    if vis and vis.split(",")[local].strip().isdigit():
        gpu_index = int(vis.split(",")[local])

    # ---- primary workload ----
    name = args.workload
    cfg, A, B, C, dA, dB, dC = device_inputs(name)
    flops = flops_of(cfg)
    streamed = streams_past_l2(cfg)
    with ClockSampler(gpu_index) as clk:
        durs, wall = (timed_streamed if streamed else timed)(cfg, dA, dB, dC, args.steps,
                                                              args.warmup)
    clocks = clk.summary()
    mean_s = sum(durs) / len(durs)
    # max over ranks of the summed GEMM time
    value = job_throughput(ws, args.steps, flops, max_over_ranks(sum(durs), ws, dev))

    half = len(durs) // 2
    drift = {"first_half": round(half * flops / sum(durs[:half]) / 1e9, 2),
             "second_half": round((len(durs) - half) * flops / sum(durs[half:]) / 1e9, 2),
             "unit": "GFLOP/s"} if half > 0 else None

    plan = sg.plan_describe(cfg["M"], cfg["N"], cfg["K"], a_addr=dA.data_ptr(),
                            b_addr=dB.data_ptr(), c_addr=dC.data_ptr(), beta=cfg["beta"])

    # sgemm_run: one kernel per step; sgemm_run_3xtf32: two split kernels and
    # the MMA kernel
    per_step = 3 if args.entry == "sgemm_run_3xtf32" else 1
    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "GFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(mean_s * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_config(name),
        "method": {"timing": ("GEMM steps back to back (operands larger than L2, no "
                              "flush), one CUDA event pair per batch of 32 launches on its "
                              "stream" if streamed else
                              "GEMM timed per step with CUDA events on its stream") +
                             "; batches queued behind a hold kernel so the device never "
                             "waits for the host",
                   "parallelism": "replicas" if ws > 1 else "single GPU",
                   "plan": plan.get("variant") if args.entry == "sgemm_run" else "3xtf32",
                   "grid": int(plan.get("grid", 0)) if args.entry == "sgemm_run" else None,
                   "entry": args.entry, "sms": num_sms},
        "sets": drift,
        "gpu_launches": per_step * args.steps + -(-args.steps // HOLD_BATCH),
        "gpu_launches_detail": {"sgemm (inside the event pairs)": per_step * args.steps,
                                "hold (between batches)": -(-args.steps // HOLD_BATCH)},
        "clocks": clocks,
    }
    if args.quick:
        return result, rank

    # ---- probes: same process, run as long as the timed GEMMs ----
    probe_s = max(2.0, min(10.0, 2.0 * wall))
    read_probe_gbs = read_probe()
    ffma = ffma_probe(probe_s, False)
    ffma2 = ffma_probe(probe_s, True)
    probe_peak = max(ffma["sustained"], ffma2["sustained"])
    achieved = flops / mean_s / 1e12
    sm_mhz_max = clocks.get("sm_max_mhz") or SM_MAX_MHZ
    peak = nominal_fp32_tflops(num_sms, sm_mhz_max)
    hbm_peak, hbm_src = measured_hbm_peak()
    kernel = {"tile": "sgemm_tile_kernel", "streamk": "sgemm_tile_kernel",
              "skinny": "sgemm_skinny_kernel", "generic": "sgemm_generic_kernel"}.get(
                  plan.get("variant"), plan.get("variant"))
    if plan.get("variant") == "skinny":
        nbytes = algorithmic_bytes(cfg)
        result["roofline"] = {
            "bound": "hbm", "achieved": round(nbytes / mean_s / 1e9, 1), "peak": hbm_peak,
            "unit": "GB/s", "frac": round(nbytes / mean_s / 1e9 / hbm_peak, 4),
            "traffic": recorded_traffic(kernel, name), "peak_source": hbm_src,
            "bytes_per_launch": nbytes, "read_probe_gbs": read_probe_gbs, "kernel": kernel,
            "fp32": {"achieved_tflops": round(achieved, 3),
                     "frac_of_probe": round(achieved / probe_peak, 4)},
        }
    else:
        result["roofline"] = {
            "bound": "alu", "achieved": round(achieved, 3), "peak": round(peak, 3),
            "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
            "traffic": recorded_traffic(kernel, name),
            "peak_source": f"{num_sms} SMs x 128 FP32 lanes x 2 flop x {sm_mhz_max:.0f} MHz "
                           "(max SM clock)",
            "probe": {"ffma_tflops": ffma, "ffma2_tflops": ffma2,
                      "frac_of_probe": round(achieved / probe_peak, 4)},
            "kernel": kernel,
        }

    # ---- the other workloads, timed the same way (fewer steps) ----
    if not args.no_secondary:
        others = []
        for other in ("s3_4092", "s4_rect", "s5_odd", "s6_skinny", "s7_gemv", "s1_128", "s8_2049",
                      "s9_ax"):
            if other == name:
                continue
            cfgo, _, _, _, dAo, dBo, dCo = device_inputs(other)
            durso, _ = timed(cfgo, dAo, dBo, dCo, max(5, args.steps // 10), args.warmup)
            mo = statistics.median(durso)
            per_call = None
            if streams_past_l2(cfgo):
                # back to back (the rate); the per-call time above is kept beside it
                per_call = mo
                durss, _ = timed_streamed(cfgo, dAo, dBo, dCo, max(HOLD_BATCH, args.steps // 10),
                                          args.warmup)
                mo = statistics.median(durss)
            po = sg.plan_describe(cfgo["M"], cfgo["N"], cfgo["K"], a_addr=dAo.data_ptr(),
                                  b_addr=dBo.data_ptr(), c_addr=dCo.data_ptr(),
                                  beta=cfgo["beta"])
            ent = {"workload": WORKLOADS[other], "plan": po.get("variant"),
                   "value": round(flops_of(cfgo) / mo / 1e9, 2), "unit": "GFLOP/s",
                   "ms_per_step": round(mo * 1e3, 4),
                   "timing": "back to back, no flush (operands larger than L2)"
                             if per_call is not None else "flush + one event pair per step"}
            if per_call is not None:
                ent["per_call_ms"] = round(per_call * 1e3, 4)
            ao = flops_of(cfgo) / mo / 1e12
            if other in ("s6_skinny", "s7_gemv", "s9_ax"):
                nbytes = algorithmic_bytes(cfgo)
                ent["roofline"] = {"bound": "hbm", "achieved": round(nbytes / mo / 1e9, 1),
                                   "peak": hbm_peak, "unit": "GB/s",
                                   "frac": round(nbytes / mo / 1e9 / hbm_peak, 4),
                                   "peak_source": hbm_src, "bytes_per_launch": nbytes,
                                   "read_probe_gbs": read_probe_gbs}
                if per_call is not None:
                    ent["roofline"]["frac_per_call"] = round(nbytes / per_call / 1e9 / hbm_peak, 4)
            else:
                ent["frac_of_peak"] = round(ao / peak, 4)
                ent["frac_of_probe"] = round(ao / probe_peak, 4)
                if per_call is not None:
                    ent["frac_of_peak_per_call"] = round(flops_of(cfgo) / per_call / 1e12 / peak, 4)
            if other == "s3_4092":
                result["secondary"] = dict(ent, note="the second size the metric is quoted at")
            else:
                others.append(ent)
            del dAo, dBo, dCo
        result["other_workloads"] = others

    # ---- cuBLAS FP32 on the same products (context, TF32 off) ----
    if not args.no_cublas:
        torch.backends.cuda.matmul.allow_tf32 = False
        ctx = []
        for cname in (name, "s3_4092", "s6_skinny"):
            if any(e["workload"] == WORKLOADS[cname] for e in ctx):
                continue
            cfgc, _, _, _, dAc, dBc, dCc = device_inputs(cname)
            steps_c = max(5, min(200, args.steps // 10))
            dc = statistics.median(timed_cublas(cfgc, dAc, dBc, dCc, steps_c, 3))
            ctx.append({"workload": WORKLOADS[cname], "api": "torch.mm/addmm, cuBLAS FP32, TF32 off",
                        "value": round(flops_of(cfgc) / dc / 1e9, 2), "unit": "GFLOP/s",
                        "ms_per_step": round(dc * 1e3, 4), "steps": steps_c})
            del dAc, dBc, dCc
        result["cublas_context"] = ctx

    # ---- the 3xTF32 tensor-core entry point (reported apart) ----
    if not args.no_secondary and args.entry == "sgemm_run":
        derived_burst, derived_sust, derived_src = measured_tf32_peak()
        tf32 = tf32_probe(2.0)
        tf32_burst, tf32_sust = tf32["burst"], tf32["sustained"]
        tf32_src = ("same-run tcgen05.mma kind::tf32 probe (M 128, N 256, K 8, all SMs), "
                    f"best of {tf32['launches']} launches; derived from MEASURED_PEAKS.json: "
                    f"{derived_burst} ({derived_src})")
        x3 = []
        for xname in ("s2_2048", "s3_4092"):
            cfgx, _, _, _, dAx, dBx, dCx = device_inputs(xname)
            steps_x = max(5, min(200, args.steps // 10))
            dx = statistics.median(timed(cfgx, dAx, dBx, dCx, steps_x, args.warmup,
                                         entry="sgemm_run_3xtf32")[0])
            fl = flops_of(cfgx)
            xplan = sg.plan_describe_3xtf32(cfgx["M"], cfgx["N"], cfgx["K"], lda=cfgx["K"],
                                            a_addr=dAx.data_ptr())
            x3.append({"workload": WORKLOADS[xname], "api": "sgemm_run_3xtf32", "plan": xplan,
                       "value": round(fl / dx / 1e9, 2), "unit": "GFLOP/s (FP32 products)",
                       "ms_per_step": round(dx * 1e3, 4), "steps": steps_x,
                       "vs_ffma_path": round(fl / dx / 1e12 / achieved, 3)
                       if xname == name else None,
                       "roofline": {"bound": "tensor",
                                    "achieved": round(3 * fl / dx / 1e12, 1),
                                    "peak": tf32_burst, "unit": "TFLOP/s",
                                    "frac": round(3 * fl / dx / 1e12 / tf32_burst, 4),
                                    "note": "3 TF32 products per FP32 product; step time "
                                            "includes the split pass",
                                    "peak_source": tf32_src, "sustained_peak": tf32_sust,
                                    "traffic": recorded_traffic("sgemm_3xtf32_kernel", xname),
                                    "kernel": "sgemm_3xtf32_kernel"}})
            del dAx, dBx, dCx
        result["tensor_core_3xtf32"] = x3

    # ---- end to end through the host entry point ----
    pA = torch.from_numpy(A.reshape(cfg["M"], cfg["K"])).pin_memory()
    pB = torch.from_numpy(B.reshape(cfg["K"], cfg["N"])).pin_memory()
    pC = torch.zeros(cfg["M"], cfg["N"]).pin_memory()
    for _ in range(2):
        sg.run_host(pA, pB, pC, cfg["alpha"], cfg["beta"])
    e2e_steps = max(3, min(args.steps, 20))
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        sg.run_host(pA, pB, pC, cfg["alpha"], cfg["beta"])
    e2e_wall = time.perf_counter() - t0
    h2d = 4 * (cfg["M"] * cfg["K"] + cfg["K"] * cfg["N"]
               + (cfg["M"] * cfg["N"] if cfg["beta"] != 0 else 0))
    result["e2e"] = {"value": round(e2e_steps * flops / e2e_wall / 1e9, 2), "unit": "GFLOP/s",
                     "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": 4 * cfg["M"] * cfg["N"],
                     "steps": e2e_steps, "api": "sgemm_run_host (pinned host buffers)"}

    # ---- CPU baseline (rank 0 only) ----
    if rank == 0 and not args.no_cpu:
        result["cpu_baseline"] = time_oracle(name, budget_s=args.cpu_seconds)
        result["cpu_baseline"]["s1_128_one_thread_gflops"] = time_oracle("s1_128", budget_s=1.0,
                                                                 threads=1)["value"]
    return with_summary_last(result, name), rank


def with_summary_last(result, name):
    """The line with its long per-workload sections moved to the end and a
    compact summary of every workload after them, so that a reader who keeps
    only the tail of the line still sees each workload's rate and fraction."""
    short = {"s1_128": "s1 128^3", "s2_2048": "s2 2048^3", "s3_4092": "s3 4092^3",
             "s4_rect": "s4 8192x6144x2048", "s5_odd": "s5 1023x1025x513",
             "s6_skinny": "s6 16x8192x8192", "s7_gemv": "gemv 1x8192x8192",
             "s8_2049": "2049^3", "s9_ax": "Ax 8192x1x8192"}
    by_text = {v: k for k, v in WORKLOADS.items()}
    summary = {}

    def put(key, ent, frac, of):
        summary[key] = {"GFLOP/s": ent.get("value"), "us": round(ent["ms_per_step"] * 1e3, 1),
                        "frac": frac, "of": of}
        if "per_call_ms" in ent:
            summary[key]["us_per_call"] = round(ent["per_call_ms"] * 1e3, 1)

    rl = result.get("roofline", {})
    if rl.get("bound") == "hbm":
        put(short[name], result, rl.get("frac"), "HBM copy peak")
    elif rl:
        put(short[name], result, rl.get("frac"), "FP32 nominal")
    for ent in ([result["secondary"]] if "secondary" in result else []) + \
            result.get("other_workloads", []):
        key = short.get(by_text.get(ent["workload"], ""), ent["workload"])
        if "roofline" in ent:
            put(key, ent, ent["roofline"]["frac"], "HBM copy peak")
        else:
            put(key, ent, ent.get("frac_of_peak"), "FP32 nominal")
    for ent in result.get("tensor_core_3xtf32", []):
        key = "3xTF32 " + short.get(by_text.get(ent["workload"], ""), ent["workload"])
        put(key, ent, ent["roofline"]["frac"], "TF32 tensor peak")
    out = {k: v for k, v in result.items()
           if k not in ("cublas_context", "tensor_core_3xtf32", "other_workloads", "secondary")}
    for k in ("cublas_context", "tensor_core_3xtf32", "other_workloads", "secondary"):
        if k in result:
            out[k] = result[k]
    if summary:
        out["summary"] = summary
    return out


def reference_arm(args, ws, rank):
    if rank != 0:
        return None
    name = args.workload
    cfg = datagen.CONFIGS[name]
    samples = []
    info = None
    # The whole run stays within about REFERENCE_SECONDS of CPU work, however
    # many steps are asked for: each step times a bounded row sample.
    per_step = max(0.05, min(1.0, REFERENCE_SECONDS / (args.warmup + args.steps)))
    for i in range(args.warmup + args.steps):
        info = time_oracle(name, budget_s=per_step)
        if i >= args.warmup:
            samples.append(info["value"])
    value = statistics.mean(samples)
    flops = flops_of(cfg)
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GFLOP/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(flops / (value * 1e9) * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(name),
        "method": {"timing": "each step times a bounded row sample of the workload on the "
                             "host cores; ms_per_step is extrapolated to the whole product"},
        "cpu_baseline": {"value": round(value, 3), "unit": "GFLOP/s", "cores": info["cores"],
                         "kind": "oracle", "sample": info["sample"]},
        "e2e": {"value": round(value, 3), "unit": "GFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="s2_2048")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU baseline")
    ap.add_argument("--no-secondary", action="store_true", help="skip the 4092^3 line")
    ap.add_argument("--no-cublas", action="store_true", help="skip the cuBLAS context timings")
    ap.add_argument("--entry", choices=["sgemm_run", "sgemm_run_3xtf32"], default="sgemm_run",
                    help="entry point of the timed steps (the metric is sgemm_run's; "
                         "sgemm_run_3xtf32 is for profiler runs of that variant)")
    ap.add_argument("--quick", action="store_true",
                    help="only the timed GEMM steps (for profiler runs)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    ws, rank, local = dist_env()
    if ws > 1:
        import torch
        import torch.distributed as tdist
        if args.impl == "reference":
            if rank != 0:
                return 0
        else:
            torch.cuda.set_device(local)
            tdist.init_process_group("nccl")

    if args.impl == "reference":
        out = reference_arm(args, ws, rank)
        if out is not None:
            print(json.dumps(out), flush=True)
        return 0

    result, rank = gpu_arm(args, ws, rank, local)
    if ws > 1:
        import torch.distributed as tdist
        tdist.barrier()
        tdist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
