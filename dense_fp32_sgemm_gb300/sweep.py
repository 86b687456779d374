"""Planner check over a sweep of shapes: for each shape, time the plan the
library picks and the alternatives it could have picked (the tiled kernel
with whole tiles only or with a stream-K tail, the mid-size kernel with 128-
or 64-row tiles, the split-K kernel, the 64 x 64 kernel), and report how far the automatic choice
is from the fastest, and how far each plan's time estimate is from its time.

    python -m dense_fp32_sgemm_gb300.sweep [--sizes 511,512,513,...] [--reps 30]

Square M = N = K by default, with sizes around the powers of two where tile
quantisation changes ("Optimizing Matrix Multiply on CUDA, Part 1", section
"Small and Odd Sizes"; "Part 2", section "Selecting Among Three Kernels").
Each timing is the median of CUDA-event times of single launches, each
after an L2 flush, queued behind a hold kernel so the device never waits for
the host.  Prints one line per shape and a JSON summary at the end.
"""
from __future__ import annotations

import argparse
import json
import statistics

import dense_fp32_sgemm_gb300 as sg

DEFAULT_SIZES = [256, 511, 512, 513, 1023, 1024, 1025, 1535, 1536, 2047, 2048, 2049,
                 3071, 3072, 3073, 4095, 4096, 4097]

CANDIDATES = [("auto", sg.VARIANT_AUTO), ("tile", sg.VARIANT_TILE),
              ("streamk", sg.VARIANT_STREAMK), ("mid", sg.VARIANT_MID),
              ("mid64", sg.VARIANT_MID64), ("ksplit", sg.VARIANT_KSPLIT),
              ("ksplit64", sg.VARIANT_KSPLIT64), ("small", sg.VARIANT_SMALL),
              ("generic", sg.VARIANT_GENERIC)]


def time_launches(torch, fn, reps, flush, sink, stream):
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps)]
    sg.probe_hold(20_000_000, stream)
    for e0, e1 in evs:
        flush.fill_(1.0)
        torch.sum(flush, dim=0, keepdim=True, out=sink)
        e0.record(stream)
        fn()
        e1.record(stream)
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) * 1e-3 for a, b in evs)


def main():
    import torch

    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--sizes", default=",".join(map(str, DEFAULT_SIZES)),
                    help="square sizes n (M = N = K = n)")
    ap.add_argument("--shapes", default="",
                    help="extra shapes MxNxK, comma separated (leading dimensions K and N)")
    ap.add_argument("--reps", type=int, default=30)
    ap.add_argument("--variants", default=",".join(n for n, _ in CANDIDATES),
                    help="candidates to time (auto is always timed)")
    args = ap.parse_args()
    chosen = set(args.variants.split(",")) | {"auto"}
    shapes = [(int(x),) * 3 for x in args.sizes.split(",") if x]
    shapes += [tuple(int(v) for v in x.split("x")) for x in args.shapes.split(",") if x]

    sg.build()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(64 << 20, device=dev)
    sink = torch.empty(1, device=dev)
    # A first timing on an idle GPU reads several times too long (the clocks
    # are still rising); 50 ms of device work first.
    sg.probe_hold(50_000_000, stream)
    torch.cuda.synchronize()
    rows = []
    for M, N, K in shapes:
        A = torch.rand(M, K, device=dev) - 0.5
        B = torch.rand(K, N, device=dev) - 0.5
        C = torch.empty(M, N, device=dev)
        times = {}
        plans = {}
        for name, variant in CANDIDATES:
            if name not in chosen:
                continue
            sg.set_plan_override(variant, 0)
            try:
                plans[name] = sg.plan_describe(M, N, K, a_addr=A.data_ptr(), b_addr=B.data_ptr(),
                                               c_addr=C.data_ptr())
                st = sg.sgemm_run(M, N, K, 1.0, A.data_ptr(), K, B.data_ptr(), N, 0.0,
                                  C.data_ptr(), N, stream.cuda_stream)
                if st != 0:
                    continue

                def one():
                    sg.sgemm_run(M, N, K, 1.0, A.data_ptr(), K, B.data_ptr(), N, 0.0,
                                 C.data_ptr(), N, stream.cuda_stream)

                times[name] = time_launches(torch, one, args.reps, flush, sink, stream)
            finally:
                sg.set_plan_override(-1, 0)
        if sg.device_status(stream) != 0:
            raise RuntimeError("device reported a timeout")
        flops = 2.0 * M * N * K
        best = min(times, key=times.get)
        row = {"M": M, "N": N, "K": K, "auto": plans["auto"]["variant"],
               "auto_us": round(times["auto"] * 1e6, 2),
               "best": best, "best_us": round(times[best] * 1e6, 2),
               "auto_over_best": round(times["auto"] / times[best], 3),
               "auto_tflops": round(flops / times["auto"] / 1e12, 2),
               "us": {k: round(v * 1e6, 2) for k, v in times.items()},
               "est_us": {k: float(plans[k].get("est_us", 0)) for k in times},
               "plans": {k: {f: plans[k].get(f) for f in ("variant", "bm", "grid", "dp_tiles",
                                                           "sk_tiles", "sk_share", "kt", "edge_m",
                                                           "edge_n")}
                         for k in times}}
        rows.append(row)
        print(f"{M:5d}x{N:5d}x{K:5d} auto={row['auto']:8s} {row['auto_us']:9.2f} us "
              f"({row['auto_tflops']:6.2f} TFLOP/s)  best={best:8s} {row['best_us']:9.2f} us  "
              f"auto/best={row['auto_over_best']:.3f}", flush=True)
    print(json.dumps({"sweep": rows}))


if __name__ == "__main__":
    main()
