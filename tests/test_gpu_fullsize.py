"""Parity at the benchmark's full size, in the launch configuration the
benchmark times: T = 4096 tokens, d = 7168, F = 2048, E = 256 experts, top-8,
Zipf 1.1 skew, inputs drawn on the device by the benchmark's recipe (seed 0),
the default schedule, for the BF16,
MXFP8 and NVFP4 plans.

The fp64 oracle cannot run the whole layer in seconds, so it computes
sampled outputs one by one:

* routing of all 4096 tokens, bit-exact (ids, counts, offsets, permutation);
* the Y, dX, dg and dlogits rows of a few tokens (forward_backward_tokens:
  each token's outputs depend on that token alone);
* the full dWg, dWu, dWd of sampled experts (expert_weight_grads, over every
  row of the expert), and zeros for an expert that received no row.

Block-scaled plans compare with the oracle's emulation of their quantisation
points, the backward reading a|b as the saved context stores them (bf16).
"""
import numpy as np
import pytest
import torch

from mixture_experts_layer_19_gb300 import moe
from mixture_experts_layer_19_gb300.workload import LayerShape, make_inputs
from oracle import moe_ref, nvfp4
from tests.util import BF16_TOL, rel_err

pytestmark = pytest.mark.gpu
T, D, F, E, K = 4096, 7168, 2048, 256, 8
ALPHA, SEED = 1.1, 0


class _HostExperts:
    """fp64 host copy of one expert of a device weight tensor at a time."""

    def __init__(self, W):
        self.W = W

    def __len__(self):
        return self.W.shape[0]

    def __getitem__(self, e):
        return self.W[e].float().cpu().numpy().astype(np.float64)


def _host(t):
    return t.float().cpu().numpy().astype(np.float64)


def _amax(W):
    return max(float(W[e].cpu().abs().max()) for e in range(W.shape[0]))


@pytest.fixture(scope="module")
def layer():
    inp = make_inputs(LayerShape(T, D, F, E, K), seed=SEED, alpha=ALPHA, device=torch.device("cuda", 0))
    host = {"X": _host(inp.X), "logits": inp.logits.cpu().numpy().astype(np.float64), "dY": _host(inp.dY)}
    yield inp, host
    del inp
    torch.cuda.empty_cache()


# (precision, oracle recipe, tolerance, sampled tokens); every case also
# checks the full weight gradients of the lightest and the heaviest expert
CASES = [(moe.MOE_BF16, False, BF16_TOL, 6), (moe.MOE_MXFP8, "mxfp8", 4e-2, 6),
         (moe.MOE_NVFP4, "nvfp4", 4e-2, 6)]


@pytest.mark.parametrize("case", CASES, ids=["bf16", "mxfp8", "nvfp4"])
def test_full_size_sampled_parity(layer, case):
    prec, fmt, tol, ntok = case
    inp, host = layer
    plan = moe.Plan(moe.Config(T_max=T, d=D, F=F, E=E, k=K, prec=prec))
    if prec != moe.MOE_BF16:
        plan.quantize_weights(inp.Wg, inp.Wu, inp.Wd)
    Y, saved = plan.forward(inp.X, inp.logits, inp.Wg, inp.Wu, inp.Wd)
    out = plan.backward(inp.dY, inp.X, inp.Wg, inp.Wu, inp.Wd, saved)
    r = plan.routing(saved, T)
    torch.cuda.synchronize()
    assert plan.device_status() == 0

    # routing of every token, bit-exact
    idx_ref, w_ref = moe_ref.route(host["logits"], K)
    lay = moe_ref.layout(idx_ref, E)
    assert np.array_equal(r["idx"].cpu().numpy(), idx_ref)
    assert np.abs(r["w"].cpu().numpy() - w_ref).max() <= 1e-6
    for key in ("counts", "offsets", "perm_src"):
        assert np.array_equal(r[key].cpu().numpy(), lay[key]), key

    Wg, Wu, Wd = _HostExperts(inp.Wg), _HostExperts(inp.Wu), _HostExperts(inp.Wd)
    ws = None
    if fmt == "nvfp4":
        ws = (nvfp4.tensor_scale(max(_amax(inp.Wg), _amax(inp.Wu))), nvfp4.tensor_scale(_amax(inp.Wd)))
    toks = np.linspace(0, T - 1, ntok).astype(np.int64)
    s = moe_ref.forward_backward_tokens(host["X"], host["logits"], Wg, Wu, Wd, host["dY"], K, toks, mx=fmt,
                                        wscales=ws, stored=fmt is not False)
    ti = torch.from_numpy(toks).cuda()
    for key, full in (("Y", Y), ("dX", out["dX"]), ("dg", out["dg"]), ("dlogits", out["dlogits"])):
        err = rel_err(full[ti], s[key])
        assert err <= tol, (key, err)

    counts = lay["counts"]
    live = np.nonzero(counts)[0]
    experts = [int(live[np.argmin(counts[live])]), int(np.argmax(counts))]
    for e in experts:
        dwg, dwu, dwd = moe_ref.expert_weight_grads(host["X"], host["logits"], Wg, Wu, Wd, host["dY"], K, e,
                                                    mx=fmt, wscales=ws, stored=fmt is not False)
        for name, ref in (("dWg", dwg), ("dWu", dwu), ("dWd", dwd)):
            err = rel_err(out[name][e], ref)
            assert err <= tol, (e, int(counts[e]), name, err)
    for e in np.nonzero(counts == 0)[0][:1]:
        for name in ("dWg", "dWu", "dWd"):
            assert torch.count_nonzero(out[name][int(e)]).item() == 0
    del plan, Y, saved, out
    torch.cuda.empty_cache()
