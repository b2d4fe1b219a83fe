"""Pins for the oracle's router GEMM (logits = X Wr^T) and its backward.

Independent checks:
* brute-force loops on a tiny case;
* closed forms: Wr = 0 gives zero logits; a one-hot token row picks out one
  column of Wr; the backward of an all-ones upstream gradient is a row or
  column sum;
* the whole routed layer (router GEMM -> top-k/softmax -> SwiGLU experts ->
  combine) rebuilt from torch float64 library routines, with torch autograd
  for dX (through both the experts and the router) and dWr, against the
  oracle's layer backward chained into its router backward;
* central finite differences of that chained oracle for dWr.
"""
import numpy as np
import pytest
import torch

from mixture_experts_layer_19_gb300.workload import LayerShape, make_inputs, to_f64
from oracle import moe_ref


def _router_inputs(T, d, F, E, k, seed):
    inp = make_inputs(LayerShape(T, d, F, E, k), seed=seed, router=True)
    return (to_f64(inp.X), to_f64(inp.Wr), to_f64(inp.Wg), to_f64(inp.Wu), to_f64(inp.Wd), to_f64(inp.dY))


def test_router_logits_brute_force():
    rng = np.random.default_rng(3)
    X, Wr = rng.standard_normal((3, 5)), rng.standard_normal((4, 5))
    L = moe_ref.router_logits(X, Wr)
    for t in range(3):
        for e in range(4):
            acc = 0.0
            for i in range(5):
                acc += X[t, i] * Wr[e, i]
            assert abs(L[t, e] - acc) <= 1e-12
    G = rng.standard_normal((3, 4))
    g = moe_ref.router_backward(X, Wr, G)
    for t in range(3):
        for i in range(5):
            assert abs(g["dX"][t, i] - sum(G[t, e] * Wr[e, i] for e in range(4))) <= 1e-12
    for e in range(4):
        for i in range(5):
            assert abs(g["dWr"][e, i] - sum(G[t, e] * X[t, i] for t in range(3))) <= 1e-12


def test_router_closed_forms():
    rng = np.random.default_rng(4)
    X, Wr = rng.standard_normal((6, 8)), rng.standard_normal((5, 8))
    assert np.array_equal(moe_ref.router_logits(X, np.zeros_like(Wr)), np.zeros((6, 5)))
    onehot = np.zeros((8, 8))
    onehot[np.arange(8), np.arange(8)] = 1.0
    assert np.array_equal(moe_ref.router_logits(onehot, Wr), Wr.T)
    g = moe_ref.router_backward(X, Wr, np.ones((6, 5)))
    assert np.allclose(g["dX"], np.tile(Wr.sum(0), (6, 1)), rtol=0, atol=1e-12)
    assert np.allclose(g["dWr"], np.tile(X.sum(0), (5, 1)), rtol=0, atol=1e-12)


def _chained_oracle(X, Wr, Wg, Wu, Wd, dY, k):
    L = moe_ref.router_logits(X, Wr)
    Y, ctx = moe_ref.forward(X, L, Wg, Wu, Wd, k)
    g = moe_ref.backward(dY, X, L, Wg, Wu, Wd, ctx)
    r = moe_ref.router_backward(X, Wr, g["dlogits"])
    return Y, g["dX"] + r["dX"], r["dWr"], ctx


@pytest.mark.parametrize("T,d,F,E,k", [(12, 32, 32, 6, 2), (9, 16, 32, 4, 3)])
def test_routed_layer_matches_torch_autograd(T, d, F, E, k):
    X, Wr, Wg, Wu, Wd, dY = _router_inputs(T, d, F, E, k, seed=11)
    Y, dX, dWr, _ = _chained_oracle(X, Wr, Wg, Wu, Wd, dY, k)
    tX, tWr = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (X, Wr))
    tWg, tWu, tWd = (torch.tensor(a, dtype=torch.float64) for a in (Wg, Wu, Wd))
    logits = tX @ tWr.T
    vals, ids = torch.topk(logits, k, dim=1)
    w = torch.softmax(vals, dim=1)
    tY = torch.zeros_like(tX)
    for j in range(k):
        e = ids[:, j]
        a = torch.einsum("td,tfd->tf", tX, tWg[e])
        b = torch.einsum("td,tfd->tf", tX, tWu[e])
        y = torch.einsum("tf,tdf->td", torch.nn.functional.silu(a) * b, tWd[e])
        tY = tY + w[:, j:j + 1] * y
    (tY * torch.tensor(dY)).sum().backward()
    assert np.abs(Y - tY.detach().numpy()).max() <= 1e-12 * max(1.0, np.abs(Y).max())
    assert np.abs(dX - tX.grad.numpy()).max() <= 1e-10 * max(1.0, np.abs(dX).max())
    assert np.abs(dWr - tWr.grad.numpy()).max() <= 1e-10 * max(1.0, np.abs(dWr).max())


def test_router_weight_gradient_finite_differences():
    T, d, F, E, k = 6, 8, 16, 4, 2
    X, Wr, Wg, Wu, Wd, dY = _router_inputs(T, d, F, E, k, seed=13)
    _, _, dWr, ctx = _chained_oracle(X, Wr, Wg, Wu, Wd, dY, k)
    eps = 1e-6
    rng = np.random.default_rng(0)
    for _ in range(8):
        e, i = int(rng.integers(E)), int(rng.integers(d))
        Wp, Wm = Wr.copy(), Wr.copy()
        Wp[e, i] += eps
        Wm[e, i] -= eps
        Yp, _ = moe_ref.forward(X, moe_ref.router_logits(X, Wp), Wg, Wu, Wd, k)
        Ym, _ = moe_ref.forward(X, moe_ref.router_logits(X, Wm), Wg, Wu, Wd, k)
        # the top-k choice must not flip inside the stencil
        assert np.array_equal(moe_ref.route(moe_ref.router_logits(X, Wp), k)[0], ctx["idx"])
        assert np.array_equal(moe_ref.route(moe_ref.router_logits(X, Wm), k)[0], ctx["idx"])
        fd = ((Yp - Ym) * dY).sum() / (2 * eps)
        assert abs(fd - dWr[e, i]) <= 1e-6 * max(1.0, abs(dWr[e, i]))
