"""GPU parity of the fused MoE layer against the fp64 CPU oracle, through
the C ABI.  Routing, histograms and the permutation are compared bit for
bit; floating-point outputs within max|err| / max|ref| <= 2e-2 (bf16)."""
import gc

import numpy as np
import pytest
import torch

from mixture_experts_layer_19_gb300 import moe
from oracle import moe_ref
from tests.util import BF16_TOL, cpu_and_gpu_inputs, rel_err

pytestmark = pytest.mark.gpu

# (T, d, F, E, k, alpha): tiny config, a mid config spanning several tiles in
# every dimension with ragged expert segments, and skewed routing.
CASES = [
    (128, 256, 512, 8, 2, 0.0),
    (512, 1024, 512, 32, 4, 1.1),
    (300, 512, 768, 16, 3, 1.5),
]


def _plan(T, d, F, E, k, flags=0):
    return moe.Plan(moe.Config(T_max=T, d=d, F=F, E=E, k=k, debug_flags=flags))


def _check_routing(plan, saved, T, k, E, L):
    r = plan.routing(saved, T)
    torch.cuda.synchronize()
    idx_ref, w_ref = moe_ref.route(L, k)
    lay = moe_ref.layout(idx_ref, E)
    assert np.array_equal(r["idx"].cpu().numpy(), idx_ref)
    assert np.array_equal(r["counts"].cpu().numpy(), lay["counts"])
    assert np.array_equal(r["offsets"].cpu().numpy(), lay["offsets"])
    assert np.array_equal(r["perm_src"].cpu().numpy(), lay["perm_src"])
    assert np.array_equal(r["dest"].cpu().numpy(), lay["dest"])
    w = r["w"].cpu().double().numpy()
    assert np.abs(w - w_ref).max() <= 1e-6
    assert np.abs(w.sum(1) - 1.0).max() <= 4 * 2.0 ** -23 * k


@pytest.mark.parametrize("case", CASES, ids=lambda c: "T%d_d%d_F%d_E%d_k%d_a%g" % c)
def test_forward_backward_parity(case):
    T, d, F, E, k, alpha = case
    g, h = cpu_and_gpu_inputs(T, d, F, E, k, seed=1, alpha=alpha)
    plan = _plan(T, d, F, E, k)
    Y, saved = plan.forward(g["X"], g["logits"], g["Wg"], g["Wu"], g["Wd"])
    out = plan.backward(g["dY"], g["X"], g["Wg"], g["Wu"], g["Wd"], saved)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    _check_routing(plan, saved, T, k, E, h["logits"])
    Yr, ctx = moe_ref.forward(h["X"], h["logits"], h["Wg"], h["Wu"], h["Wd"], k)
    gr = moe_ref.backward(h["dY"], h["X"], h["logits"], h["Wg"], h["Wu"], h["Wd"], ctx)
    errs = {"Y": rel_err(Y, Yr)}
    for key in ("dX", "dWg", "dWu", "dWd", "dg", "dlogits"):
        errs[key] = rel_err(out[key], gr[key])
    assert all(v <= BF16_TOL for v in errs.values()), errs


def test_identity_experts_top1_returns_input_bitwise():
    T, d, F, E, k = 257, 512, 256, 16, 1
    g, _ = cpu_and_gpu_inputs(T, d, F, E, k, seed=4, alpha=1.5)
    plan = _plan(T, d, F, E, k, flags=moe.MOE_DEBUG_IDENTITY_EXPERTS)
    Y, _ = plan.forward(g["X"], g["logits"], None, None, None)
    torch.cuda.synchronize()
    assert torch.equal(Y, g["X"])
    plan3 = _plan(T, d, F, E, 3, flags=moe.MOE_DEBUG_IDENTITY_EXPERTS)
    Y3, _ = plan3.forward(g["X"], g["logits"], None, None, None)
    torch.cuda.synchronize()
    assert rel_err(Y3, g["X"].double().cpu().numpy()) <= 2 ** -8


@pytest.mark.parametrize("T", [1, 3, 127, 129])
def test_ragged_token_counts(T):
    d, F, E, k = 256, 256, 8, 2
    g, h = cpu_and_gpu_inputs(T, d, F, E, k, seed=T)
    plan = _plan(256, d, F, E, k)
    Y, saved = plan.forward(g["X"], g["logits"], g["Wg"], g["Wu"], g["Wd"])
    out = plan.backward(g["dY"], g["X"], g["Wg"], g["Wu"], g["Wd"], saved)
    torch.cuda.synchronize()
    _check_routing(plan, saved, T, k, E, h["logits"])
    Yr, ctx = moe_ref.forward(h["X"], h["logits"], h["Wg"], h["Wu"], h["Wd"], k)
    gr = moe_ref.backward(h["dY"], h["X"], h["logits"], h["Wg"], h["Wu"], h["Wd"], ctx)
    assert rel_err(Y, Yr) <= BF16_TOL
    for key in ("dX", "dWg", "dWu", "dWd", "dg", "dlogits"):
        assert rel_err(out[key], gr[key]) <= BF16_TOL, key


def test_all_tokens_to_same_experts_and_empty_experts():
    T, d, F, E, k = 300, 256, 256, 12, 2
    bias = torch.zeros(E)
    bias[5], bias[9] = 40.0, 30.0  # every token picks experts 5 then 9; the other ten get nothing

    g, h = cpu_and_gpu_inputs(T, d, F, E, k, seed=8, logits_fn=lambda L: L + bias[None, :])
    plan = _plan(T, d, F, E, k)
    Y, saved = plan.forward(g["X"], g["logits"], g["Wg"], g["Wu"], g["Wd"])
    out = plan.backward(g["dY"], g["X"], g["Wg"], g["Wu"], g["Wd"], saved)
    torch.cuda.synchronize()
    _check_routing(plan, saved, T, k, E, h["logits"])
    Yr, ctx = moe_ref.forward(h["X"], h["logits"], h["Wg"], h["Wu"], h["Wd"], k)
    gr = moe_ref.backward(h["dY"], h["X"], h["logits"], h["Wg"], h["Wu"], h["Wd"], ctx)
    assert rel_err(Y, Yr) <= BF16_TOL
    for key in ("dX", "dWg", "dWu", "dWd", "dg", "dlogits"):
        assert rel_err(out[key], gr[key]) <= BF16_TOL, key
    empty = [e for e in range(E) if e not in (5, 9)]
    for key in ("dWg", "dWu", "dWd"):
        assert torch.count_nonzero(out[key][empty]).item() == 0


def test_k_equals_E():
    T, d, F, E, k = 64, 256, 256, 4, 4
    g, h = cpu_and_gpu_inputs(T, d, F, E, k, seed=9)
    plan = _plan(T, d, F, E, k)
    Y, saved = plan.forward(g["X"], g["logits"], g["Wg"], g["Wu"], g["Wd"])
    out = plan.backward(g["dY"], g["X"], g["Wg"], g["Wu"], g["Wd"], saved)
    torch.cuda.synchronize()
    _check_routing(plan, saved, T, k, E, h["logits"])
    Yr, ctx = moe_ref.forward(h["X"], h["logits"], h["Wg"], h["Wu"], h["Wd"], k)
    gr = moe_ref.backward(h["dY"], h["X"], h["logits"], h["Wg"], h["Wu"], h["Wd"], ctx)
    assert rel_err(Y, Yr) <= BF16_TOL
    for key in ("dX", "dWg", "dWu", "dWd", "dg", "dlogits"):
        assert rel_err(out[key], gr[key]) <= BF16_TOL, key


@pytest.mark.parametrize("flags", [0, moe.MOE_DEBUG_RING_MEGAKERNEL], ids=["separate", "ring_one_launch"])
def test_bitwise_deterministic_over_10_runs(flags):
    T, d, F, E, k = 512, 512, 512, 16, 4
    for alpha in (0.0, 1.1, 1.5):
        g, _ = cpu_and_gpu_inputs(T, d, F, E, k, seed=12, alpha=alpha)
        plan = _plan(T, d, F, E, k, flags=flags)
        ref = None
        for _ in range(10):
            Y, saved = plan.forward(g["X"], g["logits"], g["Wg"], g["Wu"], g["Wd"])
            out = plan.backward(g["dY"], g["X"], g["Wg"], g["Wu"], g["Wd"], saved)
            r = plan.routing(saved, T)
            cur = [Y.clone()] + [out[n].clone() for n in ("dX", "dWg", "dWu", "dWd", "dg", "dlogits")] + \
                  [r[n].clone() for n in ("idx", "w", "perm_src", "dest")]
            if ref is None:
                ref = cur
            else:
                for a, b in zip(ref, cur):
                    assert torch.equal(a, b)


@pytest.mark.parametrize("mb_rows,slots,movers", [(0, 0, 0), (128, 2, 1), (256, 3, 5), (1024, 2, 2)])
def test_ring_megakernel_matches_separate_kernels_bitwise(mb_rows, slots, movers):
    """The ring-buffer megakernel (movers, minibatches, GPU-local counters) must
    give exactly the separate-kernel results: same tiles, same K order.  Small
    minibatches and few slots force many minibatches and ring wrap-around."""
    T, d, F, E, k = 700, 512, 512, 24, 4
    g, h = cpu_and_gpu_inputs(T, d, F, E, k, seed=31, alpha=1.1)
    ring = moe.Plan(moe.Config(T_max=T, d=d, F=F, E=E, k=k, minibatch_rows=mb_rows, ring_slots=slots,
                               mover_ctas=movers, debug_flags=moe.MOE_DEBUG_RING_MEGAKERNEL))
    sep = _plan(T, d, F, E, k, flags=moe.MOE_DEBUG_SEPARATE_KERNELS)
    Ya, sa = ring.forward(g["X"], g["logits"], g["Wg"], g["Wu"], g["Wd"])
    Yb, sb = sep.forward(g["X"], g["logits"], g["Wg"], g["Wu"], g["Wd"])
    ga = ring.backward(g["dY"], g["X"], g["Wg"], g["Wu"], g["Wd"], sa)
    gb = sep.backward(g["dY"], g["X"], g["Wg"], g["Wu"], g["Wd"], sb)
    torch.cuda.synchronize()
    assert ring.device_status() == 0 and sep.device_status() == 0
    assert torch.equal(Ya, Yb)
    for key in ("dX", "dWg", "dWu", "dWd", "dg", "dlogits"):
        assert torch.equal(ga[key], gb[key]), key
    Yr, _ = moe_ref.forward(h["X"], h["logits"], h["Wg"], h["Wu"], h["Wd"], k)
    assert rel_err(Ya, Yr) <= BF16_TOL


@pytest.mark.parametrize("case", [(700, 512, 512, 24, 4, 1.1), (300, 768, 768, 16, 3, 1.5), (64, 256, 512, 8, 2, 0.0)],
                         ids=lambda c: "T%d_d%d_F%d_E%d_k%d_a%g" % c)
def test_schedules_match_bitwise_fwd_bwd(case):
    """The default schedule, the separate kernels and the ring megakernel
    compute every tile in the same fixed K order, so the whole forward and
    backward agree bit for bit.  d=768 / F=768 give odd N-tile counts."""
    T, d, F, E, k, alpha = case
    g, h = cpu_and_gpu_inputs(T, d, F, E, k, seed=43, alpha=alpha)
    dflt = _plan(T, d, F, E, k)
    sep = _plan(T, d, F, E, k, flags=moe.MOE_DEBUG_SEPARATE_KERNELS)
    ring = _plan(T, d, F, E, k, flags=moe.MOE_DEBUG_RING_MEGAKERNEL)
    outs = []
    for p in (dflt, sep, ring):
        Y, s = p.forward(g["X"], g["logits"], g["Wg"], g["Wu"], g["Wd"])
        gr = p.backward(g["dY"], g["X"], g["Wg"], g["Wu"], g["Wd"], s)
        outs.append((Y, gr))
    torch.cuda.synchronize()
    assert all(p.device_status() == 0 for p in (dflt, sep, ring))
    for Y, gr in outs[1:]:
        assert torch.equal(outs[0][0], Y)
        for key in ("dX", "dWg", "dWu", "dWd", "dg", "dlogits"):
            assert torch.equal(outs[0][1][key], gr[key]), key
    Yr, ctx = moe_ref.forward(h["X"], h["logits"], h["Wg"], h["Wu"], h["Wd"], k)
    gref = moe_ref.backward(h["dY"], h["X"], h["logits"], h["Wg"], h["Wu"], h["Wd"], ctx)
    assert rel_err(outs[0][0], Yr) <= BF16_TOL
    for key in ("dX", "dWg", "dWu", "dWd"):
        assert rel_err(outs[0][1][key], gref[key]) <= BF16_TOL, key


@pytest.mark.parametrize("case", [(700, 512, 512, 24, 4, 1.1), (1000, 256, 256, 64, 8, 1.5), (33, 256, 512, 8, 2, 0.0)],
                         ids=lambda c: "T%d_d%d_F%d_E%d_k%d_a%g" % c)
def test_one_launch_forward_matches_multi_launch_and_separate_bitwise(case):
    """The BF16 ring schedule's one-launch forward routes, lays out, plans
    minibatches and combines inside the persistent kernel (the combine is done
    by the last of a token's k down tiles to arrive).  Routing, saved context
    and Y must equal the multi-launch ring schedule and the separate kernels."""
    T, d, F, E, k, alpha = case
    g, h = cpu_and_gpu_inputs(T, d, F, E, k, seed=47, alpha=alpha)
    ring = moe.MOE_DEBUG_RING_MEGAKERNEL
    plans = [_plan(T, d, F, E, k, flags=ring), _plan(T, d, F, E, k, flags=ring | moe.MOE_DEBUG_MULTI_LAUNCH),
             _plan(T, d, F, E, k)]
    outs = []
    for p in plans:
        Y, s = p.forward(g["X"], g["logits"], g["Wg"], g["Wu"], g["Wd"])
        outs.append((Y, s, p.routing(s, T)))
    torch.cuda.synchronize()
    assert all(p.device_status() == 0 for p in plans)
    for Y, s, r in outs[1:]:
        assert torch.equal(outs[0][0], Y)
        for key in ("idx", "w", "counts", "offsets", "perm_src", "dest"):
            assert torch.equal(outs[0][2][key], r[key]), key
    idx_ref, _ = moe_ref.route(h["logits"], k)
    assert np.array_equal(outs[0][2]["idx"].cpu().numpy(), idx_ref)
    Yr, _ = moe_ref.forward(h["X"], h["logits"], h["Wg"], h["Wu"], h["Wd"], k)
    assert rel_err(outs[0][0], Yr) <= BF16_TOL


@pytest.mark.parametrize("flags", [0, moe.MOE_DEBUG_RING_MEGAKERNEL], ids=["separate", "ring_one_launch"])
def test_forward_replays_from_a_cuda_graph(flags):
    """A captured forward can be replayed: the enqueued work needs no host
    state, and the one-launch forward's grid barriers reset themselves at the
    end of every launch."""
    T, d, F, E, k = 300, 256, 512, 16, 4
    g, _ = cpu_and_gpu_inputs(T, d, F, E, k, seed=48, alpha=1.1)
    plan = _plan(T, d, F, E, k, flags=flags)
    saved = plan.new_saved(T)
    Y = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        plan.forward(g["X"], g["logits"], g["Wg"], g["Wu"], g["Wd"], Y=Y, saved=saved, stream=stream)
    stream.synchronize()
    ref = Y.clone()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        plan.forward(g["X"], g["logits"], g["Wg"], g["Wu"], g["Wd"], Y=Y, saved=saved, stream=stream)
    for _ in range(3):
        Y.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert plan.device_status() == 0
        assert torch.equal(Y, ref)


@pytest.mark.parametrize("prec", [moe.MOE_BF16, moe.MOE_MXFP8, moe.MOE_NVFP4], ids=["bf16", "mxfp8", "nvfp4"])
def test_training_step_with_router_replays_from_a_cuda_graph(prec):
    """A whole training step of the layer -- router GEMM (split over K), layer
    forward, layer backward, router backward into dX -- captured once and
    replayed: every output bitwise equal to the eager step's, for each
    precision's default schedule."""
    T, d, F, E, k = 300, 256, 512, 16, 4
    g, _ = cpu_and_gpu_inputs(T, d, F, E, k, seed=50, alpha=1.1)
    gen = torch.Generator().manual_seed(51)
    Wr = (torch.randn((E, d), generator=gen) / d ** 0.5).to(torch.bfloat16).cuda()
    plan = moe.Plan(moe.Config(T_max=T, d=d, F=F, E=E, k=k, prec=prec))
    if prec != moe.MOE_BF16:
        plan.quantize_weights(g["Wg"], g["Wu"], g["Wd"])
    saved = plan.new_saved(T)
    logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
    Y = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    dWr = torch.empty((E, d), dtype=torch.bfloat16, device="cuda")
    out = {"dX": torch.empty((T, d), dtype=torch.bfloat16, device="cuda"),
           "dWg": torch.empty((E, F, d), dtype=torch.bfloat16, device="cuda"),
           "dWu": torch.empty((E, F, d), dtype=torch.bfloat16, device="cuda"),
           "dWd": torch.empty((E, d, F), dtype=torch.bfloat16, device="cuda"),
           "dg": torch.empty((T, k), dtype=torch.float32, device="cuda"),
           "dlogits": torch.empty((T, E), dtype=torch.float32, device="cuda")}
    stream = torch.cuda.Stream()

    def step():
        plan.router_forward(g["X"], Wr, logits=logits, stream=stream)
        plan.forward(g["X"], logits, g["Wg"], g["Wu"], g["Wd"], Y=Y, saved=saved, stream=stream)
        plan.backward(g["dY"], g["X"], g["Wg"], g["Wu"], g["Wd"], saved, out=out, stream=stream)
        plan.router_backward(g["X"], Wr, out["dlogits"], out["dX"], dWr=dWr, stream=stream)

    with torch.cuda.stream(stream):
        step()
    stream.synchronize()
    assert plan.device_status() == 0
    bufs = {"logits": logits, "Y": Y, "dWr": dWr, **out}
    ref = {n: v.clone() for n, v in bufs.items()}
    assert torch.count_nonzero(ref["dWr"]).item() > 0
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


def test_plan_collected_during_a_capture_is_destroyed_afterwards():
    """The garbage collector may reach an unreferenced plan while a CUDA graph
    is being captured.  Destroying it then (device synchronise, frees) would
    invalidate the capture, so the binding defers it: the capture and its
    replays succeed, and the next plan creation destroys the deferred one."""
    T, d, F, E, k = 300, 256, 512, 16, 4
    g, _ = cpu_and_gpu_inputs(T, d, F, E, k, seed=49, alpha=1.1)
    plan = _plan(T, d, F, E, k, flags=moe.MOE_DEBUG_RING_MEGAKERNEL)
    saved = plan.new_saved(T)
    Y = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        plan.forward(g["X"], g["logits"], g["Wg"], g["Wu"], g["Wd"], Y=Y, saved=saved, stream=stream)
    stream.synchronize()
    ref = Y.clone()
    gc.collect()                      # earlier garbage goes outside the capture
    gc.disable()
    try:
        doomed = [_plan(64, 256, 256, 4, 2)]
        doomed.append(doomed)         # reachable only through a reference cycle
        del doomed
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            gc.collect()              # the collector runs inside the capture
            plan.forward(g["X"], g["logits"], g["Wg"], g["Wu"], g["Wd"], Y=Y, saved=saved, stream=stream)
    finally:
        gc.enable()
    assert len(moe._deferred_destroy) == 1
    Y.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    assert torch.equal(Y, ref)
    _plan(64, 256, 256, 4, 2).close()
    assert len(moe._deferred_destroy) == 0


def test_ring_config_is_validated():
    with pytest.raises(moe.MoEError):
        moe.Plan(moe.Config(T_max=64, d=256, F=256, E=4, k=2, ring_slots=1))
    with pytest.raises(moe.MoEError):
        moe.Plan(moe.Config(T_max=64, d=256, F=256, E=4, k=2, mover_ctas=100000))


def test_zero_tokens_is_noop_and_zero_weight_grads():
    d, F, E, k = 256, 256, 4, 2
    plan = _plan(16, d, F, E, k)
    dev = torch.device("cuda", 0)
    X = torch.empty((0, d), dtype=torch.bfloat16, device=dev)
    L = torch.empty((0, E), dtype=torch.float32, device=dev)
    W = torch.randn((E, F, d), device=dev).to(torch.bfloat16)
    Wd = torch.randn((E, d, F), device=dev).to(torch.bfloat16)
    Y, saved = plan.forward(X, L, W, W, Wd)
    out = plan.backward(X, X, W, W, Wd, saved)
    torch.cuda.synchronize()
    assert Y.shape == (0, d)
    for key in ("dWg", "dWu", "dWd"):
        assert torch.count_nonzero(out[key]).item() == 0


def test_argument_errors_are_synchronous():
    T, d, F, E, k = 32, 256, 256, 4, 2
    g, _ = cpu_and_gpu_inputs(T, d, F, E, k, seed=2)
    plan = _plan(T, d, F, E, k)
    with pytest.raises(moe.MoEError) as ei:
        plan.forward(torch.cat([g["X"], g["X"]]), torch.cat([g["logits"], g["logits"]]), g["Wg"], g["Wu"], g["Wd"])
    assert ei.value.status == 1  # T > T_max
    bad = torch.empty(g["X"].numel() * 2 + 8, dtype=torch.uint8, device=g["X"].device)[8:].view(torch.bfloat16)
    Xmis = bad[: g["X"].numel()].view(T, d)
    with pytest.raises(moe.MoEError):
        plan.forward(Xmis, g["logits"], g["Wg"], g["Wu"], g["Wd"])
    small = torch.empty(plan.saved_bytes(T) - 1, dtype=torch.uint8, device=g["X"].device)
    with pytest.raises(ValueError):   # a context too small for T is refused before any launch
        plan.forward(g["X"], g["logits"], g["Wg"], g["Wu"], g["Wd"], saved=small)
    assert plan.device_status() == 0


@pytest.mark.parametrize("prec", [moe.MOE_BF16, moe.MOE_NVFP4], ids=["bf16", "nvfp4"])
def test_maximum_experts_and_top_k(prec):
    """The largest supported routing: E = 1024 experts and k = 32 slots per
    token (most experts get one or two rows, each padded to a 128-row tile),
    plus the ring and one-launch schedules on the BF16 plan."""
    T, d, F, E, k = 64, 256, 256, 1024, 32
    g, h = cpu_and_gpu_inputs(T, d, F, E, k, seed=13, alpha=1.1)
    plan = moe.Plan(moe.Config(T_max=T, d=d, F=F, E=E, k=k, prec=prec))
    if prec != moe.MOE_BF16:
        plan.quantize_weights(g["Wg"], g["Wu"], g["Wd"])
    Y, saved = plan.forward(g["X"], g["logits"], g["Wg"], g["Wu"], g["Wd"])
    out = plan.backward(g["dY"], g["X"], g["Wg"], g["Wu"], g["Wd"], saved)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    _check_routing(plan, saved, T, k, E, h["logits"])
    fmt = "nvfp4" if prec == moe.MOE_NVFP4 else False
    tol = 4e-2 if fmt else BF16_TOL
    Yr, ctx = moe_ref.forward(h["X"], h["logits"], h["Wg"], h["Wu"], h["Wd"], k, mx=fmt)
    gr = moe_ref.backward(h["dY"], h["X"], h["logits"], h["Wg"], h["Wu"], h["Wd"],
                          moe_ref.stored_context(ctx) if fmt else ctx)
    errs = {"Y": rel_err(Y, Yr)}
    for key in ("dX", "dWg", "dWu", "dWd", "dg", "dlogits"):
        errs[key] = rel_err(out[key], gr[key])
    assert all(v <= tol for v in errs.values()), errs
    if prec == moe.MOE_BF16:
        for flags in (moe.MOE_DEBUG_RING_MEGAKERNEL, moe.MOE_DEBUG_RING_MEGAKERNEL | moe.MOE_DEBUG_MULTI_LAUNCH):
            other = _plan(T, d, F, E, k, flags)
            Y2, s2 = other.forward(g["X"], g["logits"], g["Wg"], g["Wu"], g["Wd"])
            out2 = other.backward(g["dY"], g["X"], g["Wg"], g["Wu"], g["Wd"], s2)
            torch.cuda.synchronize()
            assert other.device_status() == 0
            assert torch.equal(Y2, Y), flags
            for key in ("dX", "dWg", "dWu", "dWd", "dg", "dlogits"):
                assert torch.equal(out2[key], out[key]), (flags, key)


def test_backward_reuses_sorted_x_only_for_its_own_forward():
    """The backward of the plan's last (separate-schedule) forward reads X's
    sorted rows left by that forward; after another forward on the plan it
    gathers them again.  Both must give the same gradients bit for bit."""
    T, d, F, E, k = 300, 512, 512, 16, 4
    gA, _ = cpu_and_gpu_inputs(T, d, F, E, k, seed=41, alpha=1.1)
    gB, _ = cpu_and_gpu_inputs(T, d, F, E, k, seed=42, alpha=0.0)
    W = (gA["Wg"], gA["Wu"], gA["Wd"])
    plan = _plan(T, d, F, E, k, moe.MOE_DEBUG_SEPARATE_KERNELS)
    _, sA = plan.forward(gA["X"], gA["logits"], *W)
    reused = plan.backward(gA["dY"], gA["X"], *W, sA)
    _, sA2 = plan.forward(gA["X"], gA["logits"], *W)
    plan.forward(gB["X"], gB["logits"], *W)             # another forward: its rows replace A's
    regathered = plan.backward(gA["dY"], gA["X"], *W, sA2)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    for key in ("dX", "dWg", "dWu", "dWd", "dg", "dlogits"):
        assert torch.equal(reused[key], regathered[key]), key


@pytest.mark.parametrize("prec", [moe.MOE_BF16, moe.MOE_MXFP8, moe.MOE_NVFP4], ids=["bf16", "mxfp8", "nvfp4"])
def test_idle_experts_get_zero_weight_gradients_over_poisoned_buffers(prec):
    """Experts that receive no row get exactly zero dWg, dWu and dWd, written
    over whatever the output buffers held (here NaN), and the experts that
    do receive rows still match the oracle.  Every token is routed among
    experts 0-5 of 16, so experts 6-15 are idle."""
    T, d, F, E, k = 96, 256, 512, 16, 2

    def first_six(logits):
        out = logits.clone()
        out[:, 6:] -= 30.0
        return out

    g, h = cpu_and_gpu_inputs(T, d, F, E, k, seed=5, logits_fn=first_six)
    plan = moe.Plan(moe.Config(T_max=T, d=d, F=F, E=E, k=k, prec=prec))
    fmt = {moe.MOE_BF16: False, moe.MOE_MXFP8: "mxfp8", moe.MOE_NVFP4: "nvfp4"}[prec]
    if fmt:
        plan.quantize_weights(g["Wg"], g["Wu"], g["Wd"])
    Y, saved = plan.forward(g["X"], g["logits"], g["Wg"], g["Wu"], g["Wd"])
    nan = float("nan")
    out = {
        "dX": torch.full((T, d), nan, dtype=torch.bfloat16, device="cuda"),
        "dWg": torch.full((E, F, d), nan, dtype=torch.bfloat16, device="cuda"),
        "dWu": torch.full((E, F, d), nan, dtype=torch.bfloat16, device="cuda"),
        "dWd": torch.full((E, d, F), nan, dtype=torch.bfloat16, device="cuda"),
        "dg": torch.full((T, k), nan, dtype=torch.float32, device="cuda"),
        "dlogits": torch.full((T, E), nan, dtype=torch.float32, device="cuda"),
    }
    plan.backward(g["dY"], g["X"], g["Wg"], g["Wu"], g["Wd"], saved, out=out)
    counts = plan.routing(saved, T)["counts"].cpu().numpy()
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    assert (counts[6:] == 0).all() and (counts[:6] > 0).all()
    for name in ("dWg", "dWu", "dWd"):
        assert torch.count_nonzero(out[name][6:]).item() == 0, name     # NaN counts as nonzero
        assert not torch.isnan(out[name][:6]).any().item(), name
    Yr, ctx = moe_ref.forward(h["X"], h["logits"], h["Wg"], h["Wu"], h["Wd"], k, mx=fmt)
    gref = moe_ref.backward(h["dY"], h["X"], h["logits"], h["Wg"], h["Wu"], h["Wd"],
                            moe_ref.stored_context(ctx) if fmt else ctx)
    tol = 4e-2 if fmt else BF16_TOL
    for name in ("dX", "dWg", "dWu", "dWd"):
        assert rel_err(out[name], gref[name]) <= tol, name


def _ring_vs_separate(T, d, F, E, k, g, h, dlogits=True):
    """Forward + backward of the one-launch ring schedule (both megakernels)
    against the separate kernels, bit for bit, and the oracle."""
    ring = _plan(T, d, F, E, k, moe.MOE_DEBUG_RING_MEGAKERNEL)
    sep = _plan(T, d, F, E, k, moe.MOE_DEBUG_SEPARATE_KERNELS)
    res = []
    for p in (ring, sep):
        Y, s = p.forward(g["X"], g["logits"], g["Wg"], g["Wu"], g["Wd"])
        out = {
            "dX": torch.empty((T, d), dtype=torch.bfloat16, device="cuda"),
            "dWg": torch.empty((E, F, d), dtype=torch.bfloat16, device="cuda"),
            "dWu": torch.empty((E, F, d), dtype=torch.bfloat16, device="cuda"),
            "dWd": torch.empty((E, d, F), dtype=torch.bfloat16, device="cuda"),
            "dg": torch.empty((T, k), dtype=torch.float32, device="cuda"),
            "dlogits": torch.empty((T, E), dtype=torch.float32, device="cuda") if dlogits else None,
        }
        p.backward(g["dY"], g["X"], g["Wg"], g["Wu"], g["Wd"], s, out=out)
        res.append((Y, out))
    torch.cuda.synchronize()
    assert ring.device_status() == 0 and sep.device_status() == 0
    assert torch.equal(res[0][0], res[1][0])
    keys = ("dX", "dWg", "dWu", "dWd", "dg") + (("dlogits",) if dlogits else ())
    for key in keys:
        assert torch.equal(res[0][1][key], res[1][1][key]), key
    Yr, ctx = moe_ref.forward(h["X"], h["logits"], h["Wg"], h["Wu"], h["Wd"], k)
    gr = moe_ref.backward(h["dY"], h["X"], h["logits"], h["Wg"], h["Wu"], h["Wd"], ctx)
    assert rel_err(res[0][0], Yr) <= BF16_TOL
    for key in keys:
        assert rel_err(res[0][1][key], gr[key]) <= BF16_TOL, key


@pytest.mark.parametrize("case", [(1, 256, 256, 8, 2), (3, 256, 512, 4, 4), (129, 512, 256, 16, 3),
                                  (200, 256, 256, 1024, 32)],
                         ids=lambda c: "T%d_d%d_F%d_E%d_k%d" % c)
def test_ring_backward_megakernel_edge_cases(case):
    """The one-launch forward and backward megakernels at the edges: a single
    token, k = E, a ragged token count, and the largest routing (E = 1024,
    k = 32, most experts with one row each, padded to a 128-row tile)."""
    T, d, F, E, k = case
    g, h = cpu_and_gpu_inputs(T, d, F, E, k, seed=70 + T, alpha=1.1)
    _ring_vs_separate(T, d, F, E, k, g, h)


def test_ring_backward_megakernel_degenerate_routing_without_dlogits():
    """Every token routed to the same two experts (all others idle), and a
    backward that skips dlogits: the in-kernel router gradient writes dg alone."""
    T, d, F, E, k = 300, 256, 256, 12, 2
    bias = torch.zeros(E)
    bias[5], bias[9] = 40.0, 30.0
    g, h = cpu_and_gpu_inputs(T, d, F, E, k, seed=71, logits_fn=lambda L: L + bias[None, :])
    _ring_vs_separate(T, d, F, E, k, g, h, dlogits=False)


def test_ring_forward_and_backward_replay_from_a_cuda_graph():
    """A captured one-launch forward and backward replay correctly: both
    megakernels reset their grid barrier and zero their own counters."""
    T, d, F, E, k = 300, 256, 512, 16, 4
    g, _ = cpu_and_gpu_inputs(T, d, F, E, k, seed=49, alpha=1.1)
    plan = _plan(T, d, F, E, k, flags=moe.MOE_DEBUG_RING_MEGAKERNEL)
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
    ref = {"Y": Y.clone(), **{n: v.clone() for n, v in out.items()}}
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    for _ in range(3):
        Y.zero_()
        for v in out.values():
            v.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert plan.device_status() == 0
        assert torch.equal(Y, ref["Y"])
        for n, v in out.items():
            assert torch.equal(v, ref[n]), n


def test_module_autograd_matches_the_plan_calls():
    """MoELayer through autograd gives, bitwise, the gradients of the plan's
    own forward + backward -- dlogits included when the logits require a
    gradient, and not computed (None) when they do not."""
    T, d, F, E, k = 200, 256, 512, 8, 2
    g, _ = cpu_and_gpu_inputs(T, d, F, E, k, seed=52, alpha=1.1)
    layer = moe.MoELayer(d, F, E, k, T_max=T)
    with torch.no_grad():
        for n in ("Wg", "Wu", "Wd"):
            getattr(layer, n).copy_(g[n])
    Y, saved = layer.plan.forward(g["X"], g["logits"], g["Wg"], g["Wu"], g["Wd"])
    ref = layer.plan.backward(g["dY"], g["X"], g["Wg"], g["Wu"], g["Wd"], saved)
    for logits_grad in (True, False):
        layer.zero_grad(set_to_none=True)
        X = g["X"].clone().requires_grad_(True)
        L = g["logits"].clone().requires_grad_(logits_grad)
        Ym = layer(X, L)
        Ym.backward(g["dY"])
        torch.cuda.synchronize()
        assert torch.equal(Ym, Y)
        assert torch.equal(X.grad, ref["dX"])
        for n in ("Wg", "Wu", "Wd"):
            assert torch.equal(getattr(layer, n).grad, ref["d" + n]), n
        if logits_grad:
            assert torch.equal(L.grad, ref["dlogits"])
        else:
            assert L.grad is None
    assert layer.plan.device_status() == 0
