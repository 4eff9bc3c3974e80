"""The autograd wrapper's contract on the CPU: the three library calls are replaced by plain
torch stand-ins (test-only), so the routing and the Megatron main_grad convention are checked
without a GPU: gradients routed to x and w, the fused accumulation into w.main_grad, the
placeholder and zero_out_wgrad, repeated backwards adding again, autograd.grad without w, a
frozen w, activation checkpoints (reentrant refused with the fused accumulation, non-reentrant
and nested adding once), and the refusals (create_graph, tracing or compiling, bad flag, bad
main_grad)."""
import pytest
import torch

import moe_ragged_bf16_grouped_b300 as gdg

E, N, K = 3, 8, 6
SIZES = [4, 0, 3]


def _bounds(offs):
    ends = offs.tolist()
    return [(ends[e - 1] if e else 0, ends[e]) for e in range(len(ends))]


def _fwd(x, w, offs, out=None, **_):
    y = torch.zeros(x.shape[0], w.shape[1], dtype=torch.float32)
    for e, (s, t) in enumerate(_bounds(offs)):
        y[s:t] = x[s:t].float() @ w[e].float().T
    return y.to(torch.bfloat16)


def _dgrad(g, w, offs, out=None, **_):
    dx = torch.zeros(g.shape[0], w.shape[2], dtype=torch.float32)
    for e, (s, t) in enumerate(_bounds(offs)):
        dx[s:t] = g[s:t].float() @ w[e].float()
    return dx.to(torch.bfloat16)


def _wgrad(g, x, offs, out=None, out_dtype=None, accumulate=False, **_):
    dw = torch.zeros(len(offs), g.shape[1], x.shape[1], dtype=torch.float32)
    for e, (s, t) in enumerate(_bounds(offs)):
        dw[e] = g[s:t].float().T @ x[s:t].float()
    if accumulate:
        out.add_(dw.to(out.dtype))
        return out
    return dw.to(out_dtype or torch.bfloat16)


@pytest.fixture
def standins(monkeypatch):
    monkeypatch.setattr(gdg, "grouped_det_gemm_fwd", _fwd)
    monkeypatch.setattr(gdg, "grouped_det_gemm_dgrad", _dgrad)
    monkeypatch.setattr(gdg, "grouped_det_gemm_wgrad", _wgrad)


def _inputs(seed=0):
    gen = torch.Generator().manual_seed(seed)
    rows = sum(SIZES)
    x = torch.randn(rows, K, generator=gen).to(torch.bfloat16).requires_grad_()
    w = torch.randn(E, N, K, generator=gen).to(torch.bfloat16).requires_grad_()
    offs = torch.tensor([4, 4, 7], dtype=torch.int32)
    dy = torch.randn(rows, N, generator=gen).to(torch.bfloat16)
    return x, w, offs, dy


def test_plain_gradients(standins):
    x, w, offs, dy = _inputs()
    gdg.grouped_det_mm(x, w, offs).backward(dy)
    assert torch.equal(x.grad, _dgrad(dy, w.detach(), offs))
    assert w.grad.dtype == torch.bfloat16
    assert torch.equal(w.grad, _wgrad(dy, x.detach(), offs))


def test_fused_accumulation_and_placeholder(standins):
    x, w, offs, dy = _inputs()
    w.main_grad = torch.ones(E, N, K)
    y = gdg.grouped_det_mm(x, w, offs, fuse_wgrad_accumulation=True)
    y.backward(dy, retain_graph=True)
    dw = _wgrad(dy, x.detach(), offs, out_dtype=torch.float32)
    assert torch.equal(w.main_grad, torch.ones(E, N, K) + dw)
    assert w.grad is None                      # no grad_added_to_main_grad attribute
    y.backward(dy)                             # every backward adds again
    assert torch.equal(w.main_grad, torch.ones(E, N, K) + dw + dw)

    x2, w2, _, _ = _inputs(1)
    w2.main_grad = torch.zeros(E, N, K)
    w2.grad_added_to_main_grad = False
    w2.zero_out_wgrad = True
    gdg.grouped_det_mm(x2, w2, offs, fuse_wgrad_accumulation=True).backward(dy)
    assert w2.grad_added_to_main_grad is True
    assert w2.grad is not None and torch.all(w2.grad == 0) and w2.grad.shape == w2.shape


def test_autograd_grad_without_w_still_accumulates(standins):
    x, w, offs, dy = _inputs()
    w.main_grad = torch.zeros(E, N, K)
    y = gdg.grouped_det_mm(x, w, offs, fuse_wgrad_accumulation=True)
    (gx,) = torch.autograd.grad(y, x, dy)
    assert torch.equal(gx, _dgrad(dy, w.detach(), offs))
    assert torch.equal(w.main_grad, _wgrad(dy, x.detach(), offs, out_dtype=torch.float32))


def test_frozen_w_does_not_accumulate(standins):
    x, w, offs, dy = _inputs()
    w = w.detach()
    w.main_grad = torch.zeros(E, N, K)
    gdg.grouped_det_mm(x, w, offs, fuse_wgrad_accumulation=True).backward(dy)
    assert torch.all(w.main_grad == 0)
    assert x.grad is not None


def test_refusals(standins):
    x, w, offs, dy = _inputs()
    with pytest.raises(ValueError):
        gdg.GroupedDetMm.apply(x, w, offs, 1)          # the flag must be a bool
    with pytest.raises(ValueError):
        gdg.grouped_det_mm(x, w, offs, fuse_wgrad_accumulation=True)   # no main_grad
    w.main_grad = torch.zeros(E, N, K + 1)
    with pytest.raises(ValueError):
        gdg.grouped_det_mm(x, w, offs, fuse_wgrad_accumulation=True)   # wrong shape
    w.main_grad = torch.zeros(E, N, K, dtype=torch.float16)
    with pytest.raises(TypeError):
        gdg.grouped_det_mm(x, w, offs, fuse_wgrad_accumulation=True)   # wrong dtype
    y = gdg.grouped_det_mm(x, w, offs)
    with pytest.raises(NotImplementedError):
        torch.autograd.grad(y, x, dy, create_graph=True)


def test_tracing_and_compiling_refused(standins, monkeypatch):
    x, w, offs, _ = _inputs()
    monkeypatch.setattr(torch.jit, "is_tracing", lambda: True)
    with pytest.raises(NotImplementedError):
        gdg.grouped_det_mm(x, w, offs)
    monkeypatch.setattr(torch.jit, "is_tracing", lambda: False)
    monkeypatch.setattr(torch.compiler, "is_compiling", lambda: True)
    with pytest.raises(NotImplementedError):
        gdg.grouped_det_mm(x, w, offs)


def test_reentrant_checkpoint_refused_with_fusion(standins):
    from torch.utils.checkpoint import checkpoint
    x, w, offs, dy = _inputs()
    w.main_grad = torch.zeros(E, N, K)
    with pytest.raises(ValueError, match="reentrant"):
        checkpoint(lambda a, b: gdg.grouped_det_mm(a, b, offs, fuse_wgrad_accumulation=True),
                   x, w, use_reentrant=True)
    assert torch.equal(w.main_grad, torch.zeros(E, N, K))
    # without fusion a reentrant checkpoint is an ordinary recomputation
    y = checkpoint(lambda a, b: gdg.grouped_det_mm(a, b, offs), x, w, use_reentrant=True)
    y.backward(dy)
    assert torch.equal(x.grad, _dgrad(dy, w.detach(), offs))
    assert torch.equal(w.grad, _wgrad(dy, x.detach(), offs))


@pytest.mark.parametrize("nested", [False, True])
def test_non_reentrant_checkpoint_adds_once(standins, nested):
    from torch.utils.checkpoint import checkpoint
    x, w, offs, dy = _inputs()
    w.main_grad = torch.ones(E, N, K)

    def inner(a, b):
        return gdg.grouped_det_mm(a, b, offs, fuse_wgrad_accumulation=True)

    def outer(a, b):
        return checkpoint(inner, a, b, use_reentrant=False) if nested else inner(a, b)

    y = checkpoint(outer, x, w, use_reentrant=False)
    y.backward(dy)
    dw = _wgrad(dy, x.detach(), offs, out_dtype=torch.float32)
    assert torch.equal(w.main_grad, torch.ones(E, N, K) + dw)
    assert torch.equal(x.grad, _dgrad(dy, w.detach(), offs))
    assert w.grad is None


def test_missing_main_grad_refused_in_checkpointed_forward(standins):
    """The recomputation exemption does not reach the first forward of a checkpoint."""
    from torch.utils.checkpoint import checkpoint
    x, w, offs, _ = _inputs()
    with pytest.raises(ValueError, match="main_grad"):
        checkpoint(lambda a, b: gdg.grouped_det_mm(a, b, offs, fuse_wgrad_accumulation=True),
                   x, w, use_reentrant=False)
