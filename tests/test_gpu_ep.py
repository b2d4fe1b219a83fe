"""Expert parallelism over virtual ranks on one GPU (pull dispatch, push
combine, pull reverse-combine, push reverse-dispatch with flag signalling).

Rank r owns a contiguous slice of the tokens and of the experts; each rank
lays out and pulls its own experts' rows, so the sorted layout, every GEMM
tile and every reduction order equal the single-GPU path.  The whole layer --
routing, Y, dX, dW, dg, dlogits -- must therefore match it bit for bit, for
several rank counts, ragged token counts (ranks without tokens), and repeated
calls (the flags reset themselves).  Block-scaled plans (MXFP8, NVFP4) run
the same exchanges on bf16 rows and quantise the pulled rows along d, which
gives the bytes of the single-GPU path's dispatch quantisation, so they
too match their single-GPU path bit for bit."""
import numpy as np
import pytest
import torch

from mixture_experts_layer_19_gb300 import moe
from oracle import moe_ref
from tests.util import BF16_TOL, cpu_and_gpu_inputs, rel_err

pytestmark = pytest.mark.gpu


def _run(plan, g, T):
    Y, saved = plan.forward(g["X"], g["logits"], g["Wg"], g["Wu"], g["Wd"])
    out = plan.backward(g["dY"], g["X"], g["Wg"], g["Wu"], g["Wd"], saved)
    r = plan.routing(saved, T)
    return Y, out, r


@pytest.mark.parametrize("case", [(700, 512, 512, 24, 4, 1.1, 2), (700, 512, 512, 24, 4, 1.1, 8),
                                  (1000, 256, 256, 64, 8, 1.5, 4), (33, 256, 512, 8, 2, 0.0, 4)],
                         ids=lambda c: "T%d_d%d_F%d_E%d_k%d_a%g_R%d" % c)
def test_virtual_rank_ep_matches_single_gpu_bitwise(case):
    T, d, F, E, k, alpha, R = case
    g, h = cpu_and_gpu_inputs(T, d, F, E, k, seed=51, alpha=alpha)
    ep = moe.Plan(moe.Config(T_max=T, d=d, F=F, E=E, k=k, ep_ranks=R))
    one = moe.Plan(moe.Config(T_max=T, d=d, F=F, E=E, k=k))
    runs = [_run(ep, g, T) for _ in range(3)]
    Yb, outb, rb = _run(one, g, T)
    torch.cuda.synchronize()
    assert ep.device_status() == 0 and one.device_status() == 0
    for Y, out, r in runs:
        assert torch.equal(Y, Yb)
        for key in ("dX", "dWg", "dWu", "dWd", "dg", "dlogits"):
            assert torch.equal(out[key], outb[key]), key
        for key in ("idx", "w", "counts", "offsets", "perm_src", "dest"):
            assert torch.equal(r[key], rb[key]), key
    Yr, ctx = moe_ref.forward(h["X"], h["logits"], h["Wg"], h["Wu"], h["Wd"], k)
    assert rel_err(runs[0][0], Yr) <= BF16_TOL
    assert np.array_equal(runs[0][2]["idx"].cpu().numpy(), moe_ref.route(h["logits"], k)[0])


@pytest.mark.parametrize("prec", [moe.MOE_MXFP8, moe.MOE_NVFP4], ids=["mxfp8", "nvfp4"])
@pytest.mark.parametrize("case", [(700, 512, 512, 24, 4, 1.1, 4), (33, 256, 512, 8, 2, 0.0, 2)],
                         ids=lambda c: "T%d_d%d_F%d_E%d_k%d_a%g_R%d" % c)
def test_virtual_rank_ep_block_scaled_matches_single_gpu_bitwise(prec, case):
    T, d, F, E, k, alpha, R = case
    g, h = cpu_and_gpu_inputs(T, d, F, E, k, seed=52, alpha=alpha)
    ep = moe.Plan(moe.Config(T_max=T, d=d, F=F, E=E, k=k, ep_ranks=R, prec=prec))
    one = moe.Plan(moe.Config(T_max=T, d=d, F=F, E=E, k=k, prec=prec))
    for p in (ep, one):
        p.quantize_weights(g["Wg"], g["Wu"], g["Wd"])
    runs = [_run(ep, g, T) for _ in range(2)]
    Yb, outb, rb = _run(one, g, T)
    torch.cuda.synchronize()
    assert ep.device_status() == 0 and one.device_status() == 0
    for Y, out, r in runs:
        assert torch.equal(Y, Yb)
        for key in ("dX", "dWg", "dWu", "dWd", "dg", "dlogits"):
            assert torch.equal(out[key], outb[key]), key
        for key in ("idx", "w", "counts", "offsets", "perm_src", "dest"):
            assert torch.equal(r[key], rb[key]), key
    fmt = "nvfp4" if prec == moe.MOE_NVFP4 else "mxfp8"
    ws = None
    if fmt == "nvfp4":
        from oracle import nvfp4
        ws = nvfp4.weight_scales(h["Wg"], h["Wu"], h["Wd"])
    Yr, _ = moe_ref.forward(h["X"], h["logits"], h["Wg"], h["Wu"], h["Wd"], k, mx=fmt, wscales=ws)
    assert rel_err(runs[0][0], Yr) <= 4e-2


def test_virtual_rank_ep_config_is_validated():
    with pytest.raises(moe.MoEError) as ei:
        moe.Plan(moe.Config(T_max=64, d=256, F=256, E=12, k=2, ep_ranks=5))   # 5 does not divide 12
    assert ei.value.status == 2
    with pytest.raises(moe.MoEError) as ei:   # identity experts have no EP form
        moe.Plan(moe.Config(T_max=64, d=256, F=256, E=8, k=2, ep_ranks=2,
                            debug_flags=moe.MOE_DEBUG_IDENTITY_EXPERTS))
    assert ei.value.status == 2


@pytest.mark.parametrize("prec", [moe.MOE_BF16, moe.MOE_MXFP8], ids=["bf16", "mxfp8"])
def test_virtual_rank_ep_step_replays_from_a_cuda_graph(prec):
    """A virtual-rank EP forward + backward captured once and replayed: the
    exchange flags reset at the end of every launch, so each replay equals
    the eager step bitwise."""
    T, d, F, E, k, R = 300, 256, 512, 16, 4, 4
    g, _ = cpu_and_gpu_inputs(T, d, F, E, k, seed=63, alpha=1.1)
    plan = moe.Plan(moe.Config(T_max=T, d=d, F=F, E=E, k=k, prec=prec, ep_ranks=R))
    if prec != moe.MOE_BF16:
        plan.quantize_weights(g["Wg"], g["Wu"], g["Wd"])
    saved = plan.new_saved(T)
    Y = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    out = {"dX": torch.empty((T, d), dtype=torch.bfloat16, device="cuda"),
           "dWg": torch.empty((E, F, d), dtype=torch.bfloat16, device="cuda"),
           "dWu": torch.empty((E, F, d), dtype=torch.bfloat16, device="cuda"),
           "dWd": torch.empty((E, d, F), dtype=torch.bfloat16, device="cuda"),
           "dg": torch.empty((T, k), dtype=torch.float32, device="cuda"),
           "dlogits": torch.empty((T, E), dtype=torch.float32, device="cuda")}
    stream = torch.cuda.Stream()

    def step():
        plan.forward(g["X"], g["logits"], g["Wg"], g["Wu"], g["Wd"], Y=Y, saved=saved, stream=stream)
        plan.backward(g["dY"], g["X"], g["Wg"], g["Wu"], g["Wd"], saved, out=out, stream=stream)

    with torch.cuda.stream(stream):
        step()
    stream.synchronize()
    assert plan.device_status() == 0
    bufs = {"Y": Y, **out}
    ref = {n: v.clone() for n, v in bufs.items()}
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    for _ in range(2):
        for v in bufs.values():
            v.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert plan.device_status() == 0
        for n, v in bufs.items():
            assert torch.equal(v, ref[n]), n
