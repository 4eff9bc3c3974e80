"""Benchmark of the ragged BF16 grouped GEMM step on B300.

One step = fwd + dgrad + wgrad (bf16 dW) of the Mixtral-style expert projection
(E=8, K=4096, N=14336, 8192 tokens routed top-2 -> 16384 packed rows), the
grouped GEMM hot path end to end.  Prints ONE JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the fp64 CPU oracle (test infrastructure, the only
reference this path has) on the host cores, on a bounded sample per step.
With N > 1 (torchrun) every rank runs an independent replica of the step
("replicas only": the grouped GEMM has no exchange step of its own).

Besides the headline step, the line carries "per_config": every workload the
path is specified on (tiny, Mixtral-style, fine-grained, wgrad-heavy fused
accumulate, decode-sized), each op timed alone (CUDA events, L2 flushed before
each launch) against its combined roofline, with the fp64 oracle timed on a
bounded sample of the same workload beside it.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402
from moe_ragged_bf16_grouped_b300 import roofline as rl  # noqa: E402

WORKLOAD = wl.MIXTRAL
METRIC = "grouped GEMM fwd/dgrad/wgrad TFLOP/s and % of B300 BF16 tensor peak"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
KERNEL_NAMES = {"fwd": "grouped_gemm_kernel<fwd>", "dgrad": "grouped_gemm_kernel<dgrad>",
                "wgrad": "grouped_gemm_kernel<wgrad>"}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ------------------------------------------------------------------ distributed

def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ peaks, clocks, traffic

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured (MEASURED_PEAKS.json)"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
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
            return None
        try:
            sm = [float(r[1]) for r in rows]
            smax = max(float(r[2]) for r in rows)
        except ValueError:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": reasons,
                "samples": len(rows), "sm_mhz_min": min(sm)}


def kernel_source_hash() -> str:
    csrc = os.path.join(ROOT, "moe_ragged_bf16_grouped_b300", "csrc")
    h = hashlib.sha256()
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str):
    """DRAM bytes per launch from a committed ncu summary, valid only while the kernel
    sources are unchanged since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    e = rec.get(WORKLOAD.name, {}).get(kernel)
    if not e or e.get("source_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ workload

def step_flops(sizes, w=WORKLOAD):
    M = int(np.sum(sizes))
    per_op = 2.0 * M * w.N * w.K
    return {"fwd": per_op, "dgrad": per_op, "wgrad": per_op}


def make_device_inputs(device, seed=0):
    d = wl.make_inputs(WORKLOAD, seed=seed, device=device, need=("X", "W", "G"))
    return d


# ------------------------------------------------------------------ CPU oracle timing

def oracle_sample_time(h, n_fwd, n_dgrad, n_wgrad):
    """Times the oracle's sampled forms on host copies of the inputs; returns
    (seconds, flops, description)."""
    import oracle
    w = WORKLOAD
    sizes, offs = h["sizes"], h["offs_np"]
    rows = int(np.sum(sizes))
    rng = np.random.default_rng(1234)
    fr = np.sort(rng.choice(rows, n_fwd, replace=False)).astype(np.int64)
    dr = np.sort(rng.choice(rows, n_dgrad, replace=False)).astype(np.int64)
    nonempty = np.nonzero(sizes)[0]
    pe = rng.choice(nonempty, n_wgrad)
    pn = rng.integers(0, w.N, n_wgrad)
    pairs = np.stack([pe, pn], 1)
    t0 = time.perf_counter()
    oracle.fwd_rows(h["Xb"], h["Wb"], offs, fr)
    oracle.dgrad_rows(h["Gb"], h["Wb"], offs, dr)
    oracle.wgrad_rows(h["Gb"], h["Xb"], offs, w.E, w.N, w.K, pairs)
    dt = time.perf_counter() - t0
    flops = 2.0 * w.N * w.K * (n_fwd + n_dgrad) + 2.0 * w.K * float(np.sum(sizes[pe]))
    desc = (f"{n_fwd} Y rows + {n_dgrad} dX rows + {n_wgrad} dW rows (e, n, all k) of the "
            f"{w.name} workload, fp64 C oracle")
    return dt, flops, desc


def host_bits(h):
    import oracle
    return {"Xb": oracle._bits(h["X"]), "Gb": oracle._bits(h["G"]), "Wb": oracle._bits(h["W"]),
            "sizes": h["sizes"], "offs_np": h["offs_np"]}


def scaled_sample(h, target_s):
    """Pilot runs, then a sample of equal FLOPs per op sized to about target_s seconds.
    The pilot grows until it takes a measurable time with every core busy."""
    import oracle
    w = WORKLOAD
    mean_rows = float(np.mean(h["sizes"][np.nonzero(h["sizes"])[0]]))
    wg_per_row = max(1, int(round(w.N / mean_rows)))     # dW rows per Y row of equal FLOPs
    n = max(4, oracle.num_threads())
    while True:
        dt, fl, _ = oracle_sample_time(h, n, n, n * wg_per_row)
        if dt >= min(2.0, target_s / 4) or n >= 1 << 14:
            break
        n *= 2
    n = max(1, int(n * target_s / max(dt, 1e-3)))
    return n, n, n * wg_per_row


def cpu_baseline(h, target_s=15.0):
    import oracle
    n_f, n_d, n_w = scaled_sample(h, target_s)
    dt, fl, desc = oracle_sample_time(h, n_f, n_d, n_w)
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle", "sample": desc + f"; {dt:.1f} s"}


def pick_peak(clocks, timed_ms, burst, sustained):
    """The bf16 peak that applies to kernels timed in this run.  The burst figure is a GEMM
    timed alone at full clocks; the sustained one a GEMM looped for seconds under the power
    cap.  A timed region shorter than a second, or one whose median SM clock stayed within
    10 % of the maximum, ran at burst clocks."""
    if clocks and clocks.get("sm_mhz") and clocks.get("sm_max_mhz"):
        ratio = clocks["sm_mhz"] / clocks["sm_max_mhz"]
        if ratio >= 0.9 or timed_ms < 1000.0:
            return burst, (f"burst bf16 (timed region {timed_ms:.0f} ms, median SM clock "
                           f"{clocks['sm_mhz']:.0f} of {clocks['sm_max_mhz']:.0f} MHz)")
        return sustained, (f"sustained bf16 (timed region {timed_ms:.0f} ms, median SM clock "
                           f"{clocks['sm_mhz']:.0f} of {clocks['sm_max_mhz']:.0f} MHz: "
                           f"power-capped)")
    if timed_ms < 1000.0:
        return burst, f"burst bf16 (timed region {timed_ms:.0f} ms, no clock record)"
    return sustained, f"sustained bf16 (timed region {timed_ms:.0f} ms, no clock record)"


# ------------------------------------------------------------------ every workload, op by op

def _oracle_probe(w, d, ops, target_s, rng):
    """Times the fp64 oracle on a bounded sample of the workload: rows of Y / dX and rows
    (e, n, all k) of dW of up to four non-empty groups, each as a one-group problem copied to
    the host.  Returns (GFLOP/s over the sample, GFLOP/s per op kind, cores, description)."""
    import oracle
    sizes = d["sizes"]
    st = np.concatenate([[0], np.cumsum(sizes)[:-1]])
    nz = np.nonzero(sizes)[0]
    groups = sorted(rng.choice(nz, size=min(4, len(nz)), replace=False).tolist())
    host = []
    for e in groups:
        s, m = int(st[e]), int(sizes[e])
        g = {"m": m, "one": np.array([m], dtype=np.int32)}
        g["X"] = oracle._bits(d["X"][s:s + m])
        g["G"] = oracle._bits(d["G"][s:s + m])
        if "W" in d:
            g["W"] = oracle._bits(d["W"][e:e + 1])
        host.append(g)

    def run(n):
        """Seconds and FLOPs of each op kind over the sample."""
        t, fl = {k: 0.0 for k in ops}, {k: 0.0 for k in ops}
        for g in host:
            ids = rng.integers(0, g["m"], n).astype(np.int64)
            for kind in ops:
                t0 = time.perf_counter()
                if kind == "fwd":
                    oracle.fwd_rows(g["X"], g["W"], g["one"], ids)
                    fl[kind] += 2.0 * w.N * w.K * n
                elif kind == "dgrad":
                    oracle.dgrad_rows(g["G"], g["W"], g["one"], ids)
                    fl[kind] += 2.0 * w.N * w.K * n
                else:
                    ns = rng.integers(0, w.N, n)
                    oracle.wgrad_rows(g["G"], g["X"], g["one"], 1, w.N, w.K,
                                      np.stack([np.zeros_like(ns), ns], 1))
                    fl[kind] += 2.0 * g["m"] * w.K * n
                t[kind] += time.perf_counter() - t0
        return t, fl

    n = max(1, oracle.num_threads() // len(host))
    while True:
        t, fl = run(n)
        dt = sum(t.values())
        if dt >= target_s / 4 or n >= 1 << 12:
            break
        n *= 2
    n = max(1, int(n * target_s / max(dt, 1e-3)))
    t, fl = run(n)
    dt = sum(t.values())
    desc = (f"{n} sampled outputs per op ({', '.join(ops)}) in each of groups {groups}, "
            f"one-group fp64 C oracle problems; {dt:.1f} s")
    per_op = {k: fl[k] / max(t[k], 1e-9) / 1e9 for k in ops}
    return sum(fl.values()) / dt / 1e9, per_op, oracle.num_threads(), desc


def time_configs(dev, peaks, iters, oracle_s, with_oracle, pause):
    """Every workload of the path, each op timed alone: median of `iters` launches, CUDA events on
    the launching stream.  Before each timed launch: `pause` seconds of idle GPU, two untimed
    launches of the same op and a 512 MiB L2 flush (ops shorter than 0.2 ms: the flush only).  The pause lets the power controller bring
    the SM clock back (back to back, the heavier ops run at power-capped clocks), the two
    launches bring the clocks up from idle, so that each timed launch runs as a kernel timed
    alone does: the condition of the burst peak that the fractions use."""
    import moe_ragged_bf16_grouped_b300 as gdg
    P = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    BW = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    rng = np.random.default_rng(5)
    result = {}
    for name in ("tiny", "mixtral", "fine_grained", "wgrad_heavy", "decode"):
        w = wl.WORKLOADS[name]
        d = wl.make_inputs(w, seed=0, device=dev)
        sizes, rows = d["sizes"], d["rows"]
        calls = {}
        if "fwd" in w.ops:
            Y = torch.empty((rows, w.N), dtype=torch.bfloat16, device=dev)
            dX = torch.empty((rows, w.K), dtype=torch.bfloat16, device=dev)
            calls["fwd"] = (lambda: gdg.grouped_det_gemm_fwd(d["X"], d["W"], d["offs"], out=Y),
                            2, False)
            calls["dgrad"] = (lambda: gdg.grouped_det_gemm_dgrad(d["G"], d["W"], d["offs"],
                                                                 out=dX), 2, False)
        for op in w.ops:
            if not op.startswith("wgrad"):
                continue
            dt = torch.float32 if "fp32" in op else torch.bfloat16
            acc = op.endswith("_acc")
            out = d["main_grad"].clone() if acc else torch.empty((w.E, w.N, w.K), dtype=dt,
                                                                 device=dev)
            need = gdg.grouped_det_gemm_workspace_bytes(gdg.GDG_OP_WGRAD, rows, w.E, w.N, w.K,
                                                        dt, acc)
            ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
            calls[op] = ((lambda out=out, acc=acc, ws=ws: gdg.grouped_det_gemm_wgrad(
                d["G"], d["X"], d["offs"], out=out, accumulate=acc, workspace=ws)),
                out.element_size(), acc)
        ops = {}
        for op, (fn, esz, acc) in calls.items():
            for _ in range(2):
                fn()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize(dev)
            # A launch far shorter than the power controller's reaction time is not slowed by
            # it, and the pause would only leave its clocks at idle: no pause for those.
            op_pause = pause if a.elapsed_time(b) > 0.2 else 0.0
            ts = []
            for _ in range(iters):
                if op_pause > 0:
                    torch.cuda.synchronize(dev)
                    time.sleep(op_pause)
                    fn()
                    fn()
                flush.fill_(1)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                b.record(stream)
                torch.cuda.synchronize(dev)
                ts.append(a.elapsed_time(b))
            ms = float(np.median(ts))
            kind = "wgrad" if op.startswith("wgrad") else op
            flops, nbytes, wbytes = rl.op_cost(kind, sizes, w.N, w.K, esz, acc)
            r = {"ms": round(ms, 4), "ms_min": round(float(np.min(ts)), 4), "pause_s": op_pause,
                 "tflops": round(flops / ms / 1e9, 1), "gbs": round(nbytes / ms / 1e6, 1),
                 "algorithmic_bytes": nbytes}
            roof = rl.roofline(ms, flops, nbytes, P, BW)
            r.update({"t_roof_ms": round(roof["t_roof_ms"], 4), "bound": roof["bound"],
                      "frac_of_roof": round(roof["frac_of_roof"], 4),
                      "frac_of_nominal_roof": round(rl.roofline(
                          ms, flops, nbytes, rl.NOMINAL_BF16_TFLOPS,
                          rl.NOMINAL_HBM_GBS)["frac_of_roof"], 4),
                      "frac_of_bf16_peak": round(flops / ms / 1e9 / P, 4),
                      "frac_of_nominal_bf16_peak": round(flops / ms / 1e9
                                                         / rl.NOMINAL_BF16_TFLOPS, 4)})
            if name == "decode":
                r["weight_gbs"] = round(wbytes / ms / 1e6, 1)
                r["weight_frac_of_hbm"] = round(wbytes / ms / 1e6 / BW, 4)
                r["weight_frac_of_nominal_hbm"] = round(wbytes / ms / 1e6
                                                        / rl.NOMINAL_HBM_GBS, 4)
            ops[op] = r
        entry = {"E": w.E, "N": w.N, "K": w.K, "rows": int(rows),
                 "nonempty_groups": int(np.count_nonzero(sizes)), "ops": ops}
        if with_oracle:
            kinds = [("wgrad" if o.startswith("wgrad") else o) for o in calls]
            kinds_u = list(dict.fromkeys(kinds))
            gf, per_op, cores, desc = _oracle_probe(w, d, kinds_u, oracle_s, rng)
            entry["oracle"] = {"gflops": round(gf, 2), "cores": cores, "sample": desc,
                               "gflops_per_op": {k: round(v, 2) for k, v in per_op.items()},
                               "full_op_s_extrapolated": {
                                   o: round(rl.op_cost(k, sizes, w.N, w.K)[0] / (per_op[k] * 1e9), 1)
                                   for o, k in zip(calls, kinds)}}
        if gdg.gdg_device_error() != 0:
            raise RuntimeError(f"device error word set during the {name} timings")
        result[name] = entry
        del d, calls
        torch.cuda.empty_cache()
    return {"timing": f"median of {iters} launches per op, each after {pause} s of idle GPU, two "
                      f"untimed launches and a 512 MiB L2 flush (ops under 0.2 ms: the flush "
                      f"only); "
                      f"roofline against the measured burst bf16 rate {P} TFLOP/s and copy "
                      f"bandwidth {BW} GB/s, and against the nominal 2250 TFLOP/s, 8000 GB/s",
            "configs": result}


# ------------------------------------------------------------------ our arm

def run_ours(args, world, rank, local):
    import moe_ragged_bf16_grouped_b300 as gdg
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = WORKLOAD
    d = make_device_inputs(dev)
    sizes = d["sizes"]
    rows = d["rows"]
    X, G, W, offs = d["X"], d["G"], d["W"], d["offs"]
    Y = torch.empty((rows, w.N), dtype=torch.bfloat16, device=dev)
    dX = torch.empty((rows, w.K), dtype=torch.bfloat16, device=dev)
    dW = torch.empty((w.E, w.N, w.K), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    flops = step_flops(sizes)
    split = gdg.grouped_det_gemm_auto_split_rows(rows, w.E, w.N, w.K)
    ws_bytes = gdg.grouped_det_gemm_workspace_bytes(gdg.GDG_OP_WGRAD, rows, w.E, w.N, w.K)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    launches_per_step = 3 + (1 if split > 0 else 0)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        gdg.grouped_det_gemm_fwd(X, W, offs, out=Y, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        gdg.grouped_det_gemm_dgrad(G, W, offs, out=dX, stream=stream)
        if ev is not None:
            ev[2].record(stream)
        gdg.grouped_det_gemm_wgrad(G, X, offs, out=dW, workspace=ws, stream=stream)
        if ev is not None:
            ev[3].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if gdg.gdg_device_error() != 0:
        raise RuntimeError("device error word set during warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    sampler = ClockSampler(local)
    sampler.start()
    barrier(world)
    torch.cuda.synchronize(dev)
    for i in range(args.steps):
        step(evs[i])
    torch.cuda.synchronize(dev)
    barrier(world)
    clocks = sampler.stop()
    total_ms = evs[0][0].elapsed_time(evs[-1][3])
    per = {"fwd": [], "dgrad": [], "wgrad": []}
    for e in evs:
        per["fwd"].append(e[0].elapsed_time(e[1]))
        per["dgrad"].append(e[1].elapsed_time(e[2]))
        per["wgrad"].append(e[2].elapsed_time(e[3]))
    total_ms = max_over_ranks(total_ms, world)
    if gdg.gdg_device_error() != 0:
        raise RuntimeError("device error word set during the timed region")

    step_f = sum(flops.values())
    ms_per_step = total_ms / args.steps
    value = world * step_f * args.steps / (total_ms * 1e-3) / 1e12

    # ---- end to end through the public API: pinned host inputs -> device -> host results.
    # Every step copies its inputs (X, G, W, offs) in from pinned host memory and its results
    # (Y, dX, dW) out, all inside the timed region.  Copies run on their own streams with two
    # sets of device buffers, so step i's kernels overlap the copy-in of step i + 1 and the
    # copy-out of step i - 1 (what a training loop feeding the GPU from the host would do).
    hX, hG, hW = (t.cpu().pin_memory() for t in (X, G, W))
    hoffs = offs.cpu().pin_memory()
    hY = torch.empty(Y.shape, dtype=Y.dtype).pin_memory()
    hdX = torch.empty(dX.shape, dtype=dX.dtype).pin_memory()
    hdW = torch.empty(dW.shape, dtype=dW.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (hX, hG, hW, hoffs))
    d2h = sum(t.numel() * t.element_size() for t in (hY, hdX, hdW))
    bufs = [dict(X=torch.empty_like(X), G=torch.empty_like(G), W=torch.empty_like(W),
                 offs=torch.empty_like(offs), Y=torch.empty_like(Y), dX=torch.empty_like(dX),
                 dW=torch.empty_like(dW)) for _ in range(2)]
    del Y, dX, dW
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    inputs_ready = [ev(), ev()]       # copy-in of buffer set b done
    inputs_free = [ev(), ev()]        # kernels of buffer set b done reading it (and writing)
    outputs_free = [ev(), ev()]       # copy-out of buffer set b done
    for b in range(2):
        inputs_free[b].record(stream)
        outputs_free[b].record(stream)
    e2e_steps = max(2, min(args.steps, 8))

    def e2e_step(i):
        b = bufs[i % 2]
        with torch.cuda.stream(s_in):
            s_in.wait_event(inputs_free[i % 2])
            b["X"].copy_(hX, non_blocking=True)
            b["G"].copy_(hG, non_blocking=True)
            b["W"].copy_(hW, non_blocking=True)
            b["offs"].copy_(hoffs, non_blocking=True)
            inputs_ready[i % 2].record(s_in)
        stream.wait_event(inputs_ready[i % 2])
        stream.wait_event(outputs_free[i % 2])
        gdg.grouped_det_gemm_fwd(b["X"], b["W"], b["offs"], out=b["Y"], stream=stream)
        gdg.grouped_det_gemm_dgrad(b["G"], b["W"], b["offs"], out=b["dX"], stream=stream)
        gdg.grouped_det_gemm_wgrad(b["G"], b["X"], b["offs"], out=b["dW"], workspace=ws,
                                   stream=stream)
        inputs_free[i % 2].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(inputs_free[i % 2])
            hY.copy_(b["Y"], non_blocking=True)
            hdX.copy_(b["dX"], non_blocking=True)
            hdW.copy_(b["dW"], non_blocking=True)
            outputs_free[i % 2].record(s_out)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_stream(stream)
    s_out.wait_stream(stream)
    for i in range(e2e_steps):
        e2e_step(i)
    stream.wait_stream(s_out)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    e2e_value = world * step_f * e2e_steps / (e2e_ms * 1e-3) / 1e12
    if gdg.gdg_device_error() != 0:
        raise RuntimeError("device error word set during the end-to-end steps")

    # ---- roofline of the dominant kernel (largest share of the timed region)
    peaks, peak_src = load_peaks()
    means = {k: float(np.mean(v)) for k, v in per.items()}
    dom = max(means, key=lambda k: means[k] * len(per[k]))
    achieved = flops[dom] / (means[dom] * 1e-3) / 1e12
    burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    sustained = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    peak, why = pick_peak(clocks, total_ms, burst, sustained)
    roofline = {"bound": "tensor", "kernel": KERNEL_NAMES[dom], "achieved": achieved,
                "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": recorded_traffic(KERNEL_NAMES[dom]),
                "peak_source": f"{peak_src}: {why}",
                "per_kernel_ms": {k: round(v, 4) for k, v in means.items()},
                "per_kernel_tflops": {k: round(flops[k] / (means[k] * 1e-3) / 1e12, 1)
                                      for k in means},
                "frac_of_burst": round(achieved / burst, 4),
                "frac_of_sustained": round(achieved / sustained, 4),
                "frac_of_nominal_2250": round(achieved / rl.NOMINAL_BF16_TFLOPS, 4),
                "step_frac_of_nominal_2250": round(step_f / (ms_per_step * 1e-3) / 1e12
                                                   / rl.NOMINAL_BF16_TFLOPS, 4)}
    # The error word once more, read without a host synchronisation of its own.
    err_word = torch.zeros(1, dtype=torch.int32).pin_memory()
    gdg.gdg_device_error_async(err_word, stream=stream)
    stream.synchronize()
    if int(err_word.item()) != 0:
        raise RuntimeError("device error word set after the end-to-end steps")

    out = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
           "data": "synthetic (seeded routing simulation and N(0, std) bf16 operands)",
           "config": {"workload": f"{w.name}: E={w.E} K={w.K} N={w.N}, 8192 tokens top-2 "
                                  f"(sum_m={rows}), fwd + dgrad + wgrad (bf16 dW)",
                      "group_sizes": [int(s) for s in sizes],
                      "flops_per_step": step_f,
                      "l2": "inputs larger than L2 (W 0.94 GB, G 0.47 GB per step; no flush)",
                      "parallelism": "replicas" if world > 1 else "single GPU",
                      "wgrad_form": "split" if split > 0 else "unsplit"},
           "clocks": clocks, "gpu_launches": launches_per_step * args.steps,
           "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                   "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                   "overlap": "copy-in, kernels and copy-out on three streams, two buffer sets"},
           "roofline": roofline}
    if rank == 0 and not args.no_per_config:
        out["per_config"] = time_configs(dev, peaks, args.config_iters, args.config_oracle_s,
                                         not args.no_cpu_baseline, args.config_pause)
    if rank == 0:
        if not args.no_cpu_baseline:
            h = {"X": X, "G": G, "W": W}
            hb = host_bits({"X": hX, "G": hG, "W": hW, "sizes": sizes, "offs_np": d["offs_np"]})
            del h
            out["cpu_baseline"] = cpu_baseline(hb, target_s=args.cpu_seconds)
        else:
            out["cpu_baseline"] = None
        print(json.dumps(out), flush=True)


# ------------------------------------------------------------------ reference arm (oracle)

def run_reference(args, world, rank):
    if rank != 0:
        return
    import oracle
    w = WORKLOAD
    t0 = time.perf_counter()
    d = wl.make_inputs(w, seed=0, device="cpu", need=("X", "W", "G"))
    hb = host_bits(d)
    log(f"reference arm: inputs generated in {time.perf_counter() - t0:.1f} s")
    budget = args.ref_seconds / max(1, args.steps + args.warmup)   # whole run within a few minutes
    n_f, n_d, n_w = scaled_sample(hb, budget)
    for _ in range(args.warmup):
        oracle_sample_time(hb, n_f, n_d, n_w)
    tot_t, tot_f, desc = 0.0, 0.0, ""
    for _ in range(args.steps):
        dt, fl, desc = oracle_sample_time(hb, n_f, n_d, n_w)
        tot_t += dt
        tot_f += fl
    value = tot_f / tot_t / 1e12
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": tot_t / args.steps * 1e3, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (seeded routing simulation and N(0, std) bf16 operands)",
           "config": {"workload": f"{w.name}: E={w.E} K={w.K} N={w.N}, 8192 tokens top-2 "
                                  f"(sum_m={int(np.sum(d['sizes']))}), fwd + dgrad + wgrad",
                      "sample_per_step": desc},
           "cpu_baseline": {"kind": "oracle", "cores": oracle.num_threads(), "sample": desc,
                            "value": value, "unit": "TFLOP/s"},
           "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-workload op timings (the headline step only)")
    ap.add_argument("--config-iters", type=int, default=10)
    ap.add_argument("--config-pause", type=float, default=0.1,
                    help="idle seconds before each per-config launch (power controller recovery)")
    ap.add_argument("--config-oracle-s", type=float, default=3.0,
                    help="oracle seconds per workload in the per-config timings")
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="reference arm: oracle seconds for the whole run (warm-up + timed steps)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_init()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
