"""Runs one operation of one seeded workload through the C ABI and prints its time.

    python -m moe_ragged_bf16_grouped_b300.run_case --workload mixtral --op wgrad \
        [--experts 2] [--iters 20] [--warmup 3] [--split-rows 0]

``--experts`` keeps only the first E groups of the workload's routing (a smaller
case of the same shapes, e.g. for profiler captures).  Times are CUDA-event
medians on the launching stream with a 512 MiB L2 flush before each launch.

The JSON line also carries the op's roofline: algorithmic FLOPs 2 M N K and bytes
(fwd / dgrad: 2 (M K + E_ne N K + M N) with E_ne the non-empty groups; wgrad:
2 (M K + M N) + E N K s_out, plus E N K s_out read when accumulating),
t_roof = max(FLOPs / P, bytes / BW) against the measured burst bf16 GEMM rate P
and copy bandwidth BW of MEASURED_PEAKS.json (when present), and t_roof / t.
"""
from __future__ import annotations

import argparse
import json
import os
import sys

import numpy as np
import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import moe_ragged_bf16_grouped_b300 as gdg  # noqa: E402
import workloads as wl  # noqa: E402


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="mixtral", choices=sorted(wl.WORKLOADS))
    ap.add_argument("--op", default="fwd", choices=("fwd", "dgrad", "wgrad"))
    ap.add_argument("--experts", type=int, default=0)
    ap.add_argument("--iters", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--split-rows", type=int, default=0)
    ap.add_argument("--out-dtype", default=None, choices=(None, "bf16", "fp32"))
    ap.add_argument("--accumulate", action="store_true")
    ap.add_argument("--nondet", action="store_true",
                    help="wgrad: the non-deterministic entry (unordered adds of the split form)")
    ap.add_argument("--shape", default=None,
                    help="E,N,K,rows: equal groups of a synthetic shape instead of a workload")
    args = ap.parse_args()

    w = wl.WORKLOADS[args.workload]
    sizes = wl.SIZES[w.name](0)
    if args.shape:
        E, N, K, rows = (int(v) for v in args.shape.split(","))
        sizes = np.full(E, rows // E, dtype=np.int64)
        w = wl.Workload(f"shape_{E}x{N}x{K}x{rows}", E=E, N=N, K=K, ops=(), main_grad_std=0.01)
    if args.experts:
        sizes = sizes[:args.experts]
        w = wl.Workload(w.name, E=len(sizes), N=w.N, K=w.K, ops=w.ops,
                        main_grad_std=w.main_grad_std)
    dev = torch.device("cuda", 0)
    d = wl.make_inputs(w, seed=0, device=dev, sizes=sizes,
                       need=("X", "G") if args.op == "wgrad" else ("X", "W", "G"))
    rows, M = d["rows"], int(np.sum(sizes))
    flops = 2.0 * M * w.N * w.K
    ops_in_cfg = " ".join(w.ops)
    fp32 = args.out_dtype == "fp32" or (args.out_dtype is None and "fp32" in ops_in_cfg)
    acc = args.op == "wgrad" and (args.accumulate or (args.out_dtype is None and "acc" in ops_in_cfg))
    if args.op == "fwd":
        out = torch.empty((rows, w.N), dtype=torch.bfloat16, device=dev)
        fn = lambda: gdg.grouped_det_gemm_fwd(d["X"], d["W"], d["offs"], out=out)  # noqa: E731
    elif args.op == "dgrad":
        out = torch.empty((rows, w.K), dtype=torch.bfloat16, device=dev)
        fn = lambda: gdg.grouped_det_gemm_dgrad(d["G"], d["W"], d["offs"], out=out)  # noqa: E731
    else:
        out = torch.zeros((w.E, w.N, w.K), dtype=torch.float32 if fp32 else torch.bfloat16,
                          device=dev)
        if args.nondet:
            need = gdg.grouped_gemm_wgrad_workspace_bytes(rows, w.E, w.N, w.K, out.dtype, acc,
                                                          args.split_rows)
            ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
            fn = lambda: gdg.grouped_gemm_wgrad(d["G"], d["X"], d["offs"], out=out,  # noqa: E731
                                                accumulate=acc, split_rows=args.split_rows,
                                                workspace=ws, deterministic=False)
        else:
            need = gdg.grouped_det_gemm_workspace_bytes(gdg.GDG_OP_WGRAD, rows, w.E, w.N, w.K,
                                                        out.dtype, acc, args.split_rows)
            ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
            fn = lambda: gdg.grouped_det_gemm_wgrad(d["G"], d["X"], d["offs"], out=out,  # noqa: E731
                                                    accumulate=acc, split_rows=args.split_rows,
                                                    workspace=ws)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(args.iters):
        flush.fill_(1)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    if gdg.gdg_device_error() != 0:
        raise RuntimeError("device error word set")
    med = float(np.median(ts)) if ts else float("nan")
    line = {"workload": w.name, "op": args.op, "E": w.E, "N": w.N, "K": w.K,
            "rows": M, "ms_median": med, "ms_min": float(np.min(ts)) if ts else None,
            "tflops": flops / med / 1e9 if ts else None,
            "out_dtype": str(out.dtype), "accumulate": acc, "split_rows": args.split_rows,
            "nondet": bool(args.nondet)}
    e_ne = int(np.count_nonzero(sizes))
    if args.op == "wgrad":
        s_out = out.element_size()
        nbytes = 2 * (M * w.K + M * w.N) + w.E * w.N * w.K * s_out * (2 if acc else 1)
    else:
        nbytes = 2 * (M * w.K + e_ne * w.N * w.K + M * w.N)   # fwd and dgrad alike
    line["bytes"] = nbytes
    line["gbs"] = nbytes / med / 1e6 if ts else None
    peaks_path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                              "MEASURED_PEAKS.json")
    if os.path.exists(peaks_path):
        with open(peaks_path) as f:
            pk = json.load(f)
        t_f = flops / (pk["bf16_tflops"] * 1e12) * 1e3
        t_b = nbytes / (pk["hbm_gbs"] * 1e9) * 1e3
        line["t_roof_ms"] = max(t_f, t_b)
        line["roof_bound"] = "tensor" if t_f >= t_b else "hbm"
        line["frac_of_roof"] = max(t_f, t_b) / med if ts else None
    print(json.dumps(line))


if __name__ == "__main__":
    main()
