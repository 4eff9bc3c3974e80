"""Offsets that are not valid cumulative row counts are memory-safe.

The offsets live on the device and the host never reads them (docs page intro paragraph), so
the library cannot refuse decreasing, negative or too-large values.  Its own contract (the C ABI
header) is that such input gives unspecified values but never touches memory outside the given
buffers: every group range is clamped to [0, rows], a reversed range is empty, and every unit
index is capped by the bound the host derives from the buffer sizes.

Each output (and the split form's workspace) lives in a larger buffer whose bytes before and
after it are a sentinel; after every call the sentinels must be intact, no in-kernel wait may
have run out, and the context must still give oracle-exact results on valid offsets.  Output
values are not checked.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import assert_bf16_close, inputs_on

DEV = "cuda"
PAD = 4096          # sentinel elements on each side (keeps 16-byte alignment for 2- and 4-byte types)
I32_MAX = 2**31 - 1

# (name, kind, offsets) for E = 4 groups over rows = 600 (offs_kind ends: 4 values; m_indptr: 5)
CASES = [
    ("decreasing", wl.OFFS_ENDS, [500, 100, 600, 300]),
    ("negative", wl.OFFS_ENDS, [-5, 200, -100, 600]),
    ("past_rows", wl.OFFS_ENDS, [200, 700, 5000, I32_MAX]),
    ("all_max", wl.OFFS_ENDS, [I32_MAX] * 4),
    ("all_min", wl.OFFS_ENDS, [-2**31] * 4),
    ("overlapping_full", wl.OFFS_ENDS, [600, 0, 600, 0]),
    ("indptr_decreasing", wl.OFFS_INDPTR, [300, 100, 700, 50, 599]),
    ("indptr_negative_lead", wl.OFFS_INDPTR, [-1000, 10, 10, 600, 600]),
    ("indptr_past_rows", wl.OFFS_INDPTR, [0, 601, I32_MAX, -7, 1 << 30]),
]

E, N, K, ROWS = 4, 264, 136, 600


def fenced(n, dtype, fill):
    flat = torch.full((n + 2 * PAD,), fill, dtype=dtype, device=DEV)
    return flat, flat[PAD:PAD + n]


def intact(flat, fill, what):
    iv = torch.int16 if flat.element_size() == 2 else torch.int32
    ref = torch.full((PAD,), fill, dtype=flat.dtype, device=DEV).view(iv)
    assert torch.equal(flat[:PAD].view(iv), ref), f"{what}: wrote before its buffer"
    assert torch.equal(flat[-PAD:].view(iv), ref), f"{what}: wrote past its buffer"


@pytest.mark.gpu
@pytest.mark.parametrize("name,kind,offs", CASES, ids=[c[0] for c in CASES])
def test_invalid_offsets_stay_inside_buffers(cuda_lib, name, kind, offs):
    w = wl.Workload("bad_offs", E=E, N=N, K=K, ops=(), main_grad_std=1.0)
    _, d = inputs_on(w, DEV, seed=9, sizes=[150, 150, 150, 150], kind=kind)
    assert d["rows"] == ROWS
    bad = torch.tensor(offs, dtype=torch.int32, device=DEV)

    flat, Y = fenced(ROWS * N, torch.bfloat16, -3.0)
    cuda_lib.grouped_det_gemm_fwd(d["X"], d["W"], bad, out=Y.view(ROWS, N), offs_kind=kind)
    torch.cuda.synchronize()
    intact(flat, -3.0, f"{name} fwd")

    flat, dX = fenced(ROWS * K, torch.bfloat16, -3.0)
    cuda_lib.grouped_det_gemm_dgrad(d["G"], d["W"], bad, out=dX.view(ROWS, K), offs_kind=kind)
    torch.cuda.synchronize()
    intact(flat, -3.0, f"{name} dgrad")

    for dtype, acc, split in ((torch.bfloat16, False, -1), (torch.float32, True, -1),
                              (torch.float32, False, 64), (torch.bfloat16, True, 128)):
        flat, dW = fenced(E * N * K, dtype, -5.0)
        need = cuda_lib.grouped_det_gemm_workspace_bytes(cuda_lib.GDG_OP_WGRAD, ROWS, E, N, K,
                                                         dtype, acc, split)
        wflat, ws = fenced(max(need, 16) // 4, torch.float32, -9.0)
        cuda_lib.grouped_det_gemm_wgrad(d["G"], d["X"], bad, out=dW.view(E, N, K),
                                        accumulate=acc, split_rows=split,
                                        workspace=ws.view(torch.uint8), offs_kind=kind)
        torch.cuda.synchronize()
        what = f"{name} wgrad {dtype} accumulate={acc} split_rows={split}"
        intact(flat, -5.0, what)
        intact(wflat, -9.0, what + " workspace")

    assert cuda_lib.gdg_device_error() == 0, f"{name}: an in-kernel wait ran out"
    # The context is still usable and exact on valid offsets.
    Y = cuda_lib.grouped_det_gemm_fwd(d["X"], d["W"], d["offs"], offs_kind=kind)
    h = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    assert_bf16_close(Y, oracle.fwd(h["X"], h["W"], h["offs_np"], kind), f"{name}: valid call after")


def test_oracle_rejects_the_same_offsets():
    """The oracle refuses every invalid case above (it is only defined on valid offsets)."""
    for name, kind, offs in CASES:
        with pytest.raises(oracle.OracleError):
            oracle.bounds(np.array(offs, dtype=np.int64).astype(np.int32), kind, E, ROWS)
