"""The team schedule of the weight gradient (groups walked by size; a group's tiles fewer than
the launch's CTA pairs): full teams run a group's tiles side by side, the remainder team in
rounds whose idle slots rotate.  Every tile must still be computed exactly once, with the
same arithmetic as in the unit-by-unit schedule, for any pair count: results against the fp64
oracle and bitwise equal across grid sizes that give full teams only, a one-pair remainder
team (many rounds), several teams, and no teams at all."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import assert_bf16_close, assert_bitwise, assert_fp32_close, inputs_on

pytestmark = pytest.mark.gpu


def test_team_schedule_against_oracle_and_across_grid_sizes(cuda_lib):
    # E = 6 groups, 768 x 1024 outputs: 3 x 4 = 12 tiles per group; rows >= 512 E walks the
    # groups by size.  One group empty, one a single row.
    sizes = [1500, 0, 1, 900, 700, 2300]
    w = wl.Workload("teams", E=6, N=768, K=1024, ops=(), main_grad_std=0.01)
    h, d = inputs_on(w, "cuda", seed=15, sizes=sizes)
    assert h["rows"] >= 512 * w.E
    ref = oracle.wgrad(h["G"], h["X"], h["offs_np"], w.E)
    setcap = cuda_lib._lib.gdg_test_set_max_pairs
    setcap.restype = None
    setcap.argtypes = [ctypes.c_int]
    empty = torch.from_numpy(np.array(sizes) == 0).to("cuda")

    def run():
        acc = d["main_grad"].clone()
        cuda_lib.grouped_det_gemm_wgrad(d["G"], d["X"], d["offs"], out=acc, accumulate=True,
                                        split_rows=-1)
        return {
            "fp32": cuda_lib.grouped_det_gemm_wgrad(d["G"], d["X"], d["offs"],
                                                    out_dtype=torch.float32, split_rows=-1),
            "bf16": cuda_lib.grouped_det_gemm_wgrad(d["G"], d["X"], d["offs"], split_rows=-1),
            "acc": acc,
        }

    results = {}
    try:
        # 0: the full grid (6 full teams of 12 + a remainder team); 24: two full teams;
        # 13: one full team and a one-pair remainder team (12 rounds); 17: remainder of 5;
        # 3: fewer pairs than tiles (no teams)
        for cap in (0, 24, 13, 17, 3):
            setcap(cap)
            results[cap] = run()
    finally:
        setcap(0)
    torch.cuda.synchronize()
    assert cuda_lib.gdg_device_error() == 0
    for cap, r in results.items():
        assert_fp32_close(r["fp32"], ref, f"fp32, cap {cap}")
        assert_bf16_close(r["bf16"], ref, f"bf16, cap {cap}")
        assert_fp32_close(r["acc"], h["main_grad"].double().numpy() + ref, f"acc, cap {cap}")
        assert torch.all(r["fp32"][empty].view(torch.int32) == 0)
        for k in r:
            assert_bitwise(r[k], results[0][k], f"{k}: cap {cap} vs full grid")
