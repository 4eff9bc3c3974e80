"""Host-side logic of bench.py and of the roofline helpers (no GPU): which bf16 peak a timed
region is judged against, and the algorithmic FLOPs / bytes of each workload's ops."""
import importlib.util
import os

import numpy as np

import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _load(name, rel):
    spec = importlib.util.spec_from_file_location(name, os.path.join(ROOT, rel))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


rl = _load("gdg_roofline", "moe_ragged_bf16_grouped_b300/roofline.py")


def test_peak_follows_the_clock_record():
    bench = _load("gdg_bench_host", "bench.py")
    full = {"sm_mhz": 2032.0, "sm_max_mhz": 2032.0}
    capped = {"sm_mhz": 1190.0, "sm_max_mhz": 2032.0}
    assert bench.pick_peak(full, 5000.0, 1747.0, 1378.6)[0] == 1747.0     # long, full clocks
    assert bench.pick_peak(capped, 73.0, 1747.0, 1378.6)[0] == 1747.0     # short region
    assert bench.pick_peak(capped, 5000.0, 1747.0, 1378.6)[0] == 1378.6   # long, power-capped
    assert bench.pick_peak(None, 73.0, 1747.0, 1378.6)[0] == 1747.0
    assert bench.pick_peak(None, 9000.0, 1747.0, 1378.6)[0] == 1378.6


def test_algorithmic_costs_of_the_workloads():
    sizes = wl.sizes_mixtral(0)
    f, b, wb = rl.op_cost("fwd", sizes, 14336, 4096)
    assert f == 2.0 * 16384 * 14336 * 4096                     # 1.924 TFLOP
    assert b == 2 * (16384 * 4096 + 8 * 14336 * 4096 + 16384 * 14336)
    assert wb == 2 * 8 * 14336 * 4096
    assert rl.op_cost("dgrad", sizes, 14336, 4096) == (f, b, wb)   # reads G [M, N], writes dX [M, K]
    dec = wl.sizes_decode(0)
    e_ne = int(np.count_nonzero(dec))
    f, b, wb = rl.op_cost("fwd", dec, 2048, 7168)
    assert wb == 2 * e_ne * 2048 * 7168
    f, b, _ = rl.op_cost("wgrad", wl.sizes_wgrad_heavy(0), 1536, 2048, out_esize=4,
                         accumulate=True)
    assert b == 2 * 65536 * (2048 + 1536) + 2 * 64 * 1536 * 2048 * 4    # about 2.08 GB
    r = rl.roofline(2.0, 2.0e12, 1.0e9, 2000.0, 8000.0)
    assert r["bound"] == "tensor" and abs(r["t_roof_ms"] - 1.0) < 1e-12
    assert abs(r["frac_of_roof"] - 0.5) < 1e-12
