"""GPU checks of the router GEMM (logits = X Wr^T) and its backward against
the fp64 oracle, through the C ABI.

* logits: fp32 accumulation of exact bf16 products, so they match the oracle
  to ~1e-5 relative; routing on the GPU's own logits is bit-exact with the
  oracle's route() of the same logits;
* backward: dX += dlogits Wr and dWr = dlogits^T X within the bf16 tolerance
  (dlogits is rounded to bf16 for the tensor cores), bitwise repeatable;
* the routed layer end to end (router GEMM -> layer -> layer backward ->
  router backward) against the oracle chain, through both dX paths;
* ragged T, E below one tile (E = 8) and above one N tile (E = 264), T = 0,
  and the E % 8 rule.
"""
import numpy as np
import pytest
import torch

from mixture_experts_layer_19_gb300 import moe
from mixture_experts_layer_19_gb300.workload import LayerShape, make_inputs, to_f64
from oracle import moe_ref
from tests.util import BF16_TOL, rel_err

pytestmark = pytest.mark.gpu
LOGIT_TOL = 1e-4


def _plan(T, d, F, E, k):
    return moe.Plan(moe.Config(T_max=T, d=d, F=F, E=E, k=k))


def _inputs(T, d, F, E, k, seed, weights=True):
    inp = make_inputs(LayerShape(T, d, F, E, k), seed=seed, alpha=1.1, weights=weights, router=True)
    gpu = {n: getattr(inp, n).cuda() for n in ("X", "Wr", "dY") + (("Wg", "Wu", "Wd") if weights else ())}
    cpu = {n: to_f64(getattr(inp, n)) for n in gpu}
    return gpu, cpu


@pytest.mark.parametrize("T,d,E", [(300, 512, 16), (129, 256, 8), (700, 1024, 264), (1, 256, 8)])
def test_router_forward_and_backward_parity(T, d, E):
    k = 2
    g, h = _inputs(T, d, 256, E, k, seed=T + E, weights=False)
    plan = _plan(T, d, 256, E, k)
    logits = plan.router_forward(g["X"], g["Wr"])
    torch.cuda.synchronize()
    L = logits.cpu().double().numpy()
    Lr = moe_ref.router_logits(h["X"], h["Wr"])
    assert np.abs(L - Lr).max() <= LOGIT_TOL * np.abs(Lr).max()
    # backward with a given upstream dlogits and a non-zero incoming dX
    gen = torch.Generator().manual_seed(7)
    dlog = torch.randn((T, E), generator=gen).cuda()
    dX0 = torch.randn((T, d), generator=gen).to(torch.bfloat16).cuda()
    dX = dX0.clone()
    dWr = plan.router_backward(g["X"], g["Wr"], dlog, dX)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    r = moe_ref.router_backward(h["X"], h["Wr"], dlog.cpu().double().numpy())
    assert rel_err(dX, to_f64(dX0) + r["dX"]) <= BF16_TOL
    assert rel_err(dWr, r["dWr"]) <= BF16_TOL
    # bitwise repeatable
    dX2 = dX0.clone()
    dWr2 = plan.router_backward(g["X"], g["Wr"], dlog, dX2)
    torch.cuda.synchronize()
    assert torch.equal(dX, dX2) and torch.equal(dWr, dWr2)


def test_routing_of_router_logits_is_bit_exact():
    T, d, F, E, k = 512, 512, 256, 32, 4
    g, _ = _inputs(T, d, F, E, k, seed=3)
    plan = _plan(T, d, F, E, k)
    logits = plan.router_forward(g["X"], g["Wr"])
    Y, saved = plan.forward(g["X"], logits, g["Wg"], g["Wu"], g["Wd"])
    r = plan.routing(saved, T)
    torch.cuda.synchronize()
    idx_ref, w_ref = moe_ref.route(logits.cpu().double().numpy(), k)
    assert np.array_equal(r["idx"].cpu().numpy(), idx_ref)
    assert np.abs(r["w"].cpu().double().numpy() - w_ref).max() <= 1e-6


def test_routed_layer_end_to_end():
    """Router GEMM, layer, layer backward and router backward (the
    RoutedMoELayer autograd path) against the oracle chain."""
    T, d, F, E, k = 256, 512, 512, 16, 2
    g, h = _inputs(T, d, F, E, k, seed=21)
    layer = moe.RoutedMoELayer(d, F, E, k, T_max=T)
    with torch.no_grad():
        for n in ("Wr", "Wg", "Wu", "Wd"):
            getattr(layer, n).copy_(g[n])
    X = g["X"].clone().requires_grad_(True)
    Y = layer(X)
    Y.backward(g["dY"])
    torch.cuda.synchronize()
    assert layer.plan.device_status() == 0
    L = moe_ref.router_logits(h["X"], h["Wr"])
    # the oracle routes on its own fp64 logits: check that the choice agrees
    idx_gpu = layer.plan.routing(*_saved_of(layer, g, T), T)["idx"].cpu().numpy()
    assert np.array_equal(idx_gpu, moe_ref.route(L, k)[0])
    Yr, ctx = moe_ref.forward(h["X"], L, h["Wg"], h["Wu"], h["Wd"], k)
    gr = moe_ref.backward(h["dY"], h["X"], L, h["Wg"], h["Wu"], h["Wd"], ctx)
    rr = moe_ref.router_backward(h["X"], h["Wr"], gr["dlogits"])
    assert rel_err(Y, Yr) <= BF16_TOL
    assert rel_err(X.grad, gr["dX"] + rr["dX"]) <= BF16_TOL
    assert rel_err(layer.Wr.grad, rr["dWr"]) <= BF16_TOL
    for n in ("Wg", "Wu", "Wd"):
        assert rel_err(getattr(layer, n).grad, gr["d" + n]) <= BF16_TOL, n


def _saved_of(layer, g, T):
    logits = layer.plan.router_forward(g["X"], layer.Wr.detach())
    _, saved = layer.plan.forward(g["X"], logits, g["Wg"], g["Wu"], g["Wd"])
    return (saved,)


def test_router_edge_cases():
    T, d, F, E, k = 64, 256, 256, 8, 2
    g, _ = _inputs(T, d, F, E, k, seed=5, weights=False)
    plan = _plan(T, d, F, E, k)
    dWr = torch.full((E, d), 3.0, dtype=torch.bfloat16, device="cuda")
    dX = torch.ones((0, d), dtype=torch.bfloat16, device="cuda")
    plan.router_forward(g["X"][:0], g["Wr"], torch.empty((0, E), device="cuda"))
    plan.router_backward(g["X"][:0], g["Wr"], torch.empty((0, E), device="cuda"), dX, dWr)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dWr).item() == 0      # no tokens: zero router-weight gradient
    odd = _plan(T, d, F, 12, k)                        # E % 8 != 0 is refused, synchronously
    with pytest.raises(moe.MoEError) as ei:
        odd.router_forward(g["X"], torch.zeros((12, d), dtype=torch.bfloat16, device="cuda"))
    assert ei.value.status == 2


def test_routed_layer_initialises_its_weights():
    """A freshly built layer holds N(0, 1/fan_in) weights (fan_in = d for Wr,
    Wg, Wu and F for Wd), not uninitialised memory, and runs a step."""
    T, d, F, E, k = 64, 256, 512, 8, 2
    layer = moe.RoutedMoELayer(d, F, E, k, T_max=T)
    for n, fan_in in (("Wr", d), ("Wg", d), ("Wu", d), ("Wd", F)):
        w = getattr(layer, n).detach().float()
        assert torch.isfinite(w).all(), n
        assert abs(w.std().item() * fan_in ** 0.5 - 1.0) < 0.1, n
        assert abs(w.mean().item()) < 0.1 * fan_in ** -0.5, n
    X = torch.randn((T, d), device="cuda").to(torch.bfloat16).requires_grad_(True)
    Y = layer(X)
    Y.float().sum().backward()
    torch.cuda.synchronize()
    assert torch.isfinite(Y.float()).all() and torch.isfinite(X.grad.float()).all()
    assert layer.plan.device_status() == 0
