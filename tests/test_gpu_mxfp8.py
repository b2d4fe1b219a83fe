"""GPU checks of the MXFP8 path against the fp64 oracle.

* The quantiser (moe_mx_quantize, which also quantises the weights) is
  compared byte for byte with the oracle's OCP MX codec: every E4M3 element and
  every E8M0 scale, including zero blocks, saturation, subnormals and -0.
* The MXFP8 forward (E4M3 gather, block-scaled [a|b] GEMM + SwiGLU with h
  re-quantised in its epilogue, block-scaled down GEMM, combine) is compared
  with the oracle's MXFP8 emulation: max|err| / max|ref| <= 4e-2, routing
  bit-exact, bitwise identical over repeated runs.
"""
import numpy as np
import pytest
import torch

from mixture_experts_layer_19_gb300 import moe
from oracle import moe_ref, mxfp8
from tests.util import cpu_and_gpu_inputs, rel_err, rel_err_norm

pytestmark = pytest.mark.gpu
MX_TOL = 4e-2


def _atom_offsets(rows, K):
    # scale byte of (row r, block b): atom (r // 128) * (K // 128) + b // 4, byte
    # (r % 32) * 16 + ((r // 32) % 4) * 4 + b % 4 inside the 512-byte atom
    out = np.empty((rows, K // 32), dtype=np.int64)
    for r in range(rows):
        for b in range(K // 32):
            atom = (r // 128) * (K // 128) + b // 4
            out[r, b] = atom * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + b % 4
    return out


def _special_matrix(rows, K, seed):
    g = torch.Generator().manual_seed(seed)
    v = torch.randn((rows, K), generator=g) * torch.exp2(torch.randint(-20, 20, (rows, 1), generator=g).float())
    v[0, :32] = 0.0                                   # all-zero block
    v[1, :32] = -0.0
    v[1, 5] = 1e-30                                    # tiny amax -> clamped scale
    v[2, :32] = torch.linspace(-600, 600, 32)          # includes values that saturate
    v[3, 0:32] = 1.0
    v[3, 1] = 1.9375                                   # saturates at 448 after scaling
    v[4, :32] = 2.0 ** -133                            # bf16 subnormals
    v[5, 7] = -1e-3                                    # rounds to -0 in a block with a large amax
    v[5, 8] = 1000.0
    return v.to(torch.bfloat16)


@pytest.mark.parametrize("rows,K", [(128, 128), (200, 512), (384, 7168 // 4)])
def test_mx_quantize_bit_exact(rows, K):
    src = _special_matrix(rows, K, seed=rows + K)
    q, sf = moe.mx_quantize(src.cuda())
    torch.cuda.synchronize()
    codes, scales = mxfp8.mx_quantize(src.to(torch.float64).numpy(), axis=1)
    assert np.array_equal(q.cpu().numpy(), codes)
    got_scales = sf.cpu().numpy()[_atom_offsets(rows, K)]
    assert np.array_equal(got_scales, scales)


def _mx_plan(T, d, F, E, k):
    return moe.Plan(moe.Config(T_max=T, d=d, F=F, E=E, k=k, prec=moe.MOE_MXFP8))


@pytest.mark.parametrize("case", [(128, 256, 512, 8, 2, 0.0), (512, 1024, 512, 32, 4, 1.1), (300, 512, 768, 16, 3, 1.5)],
                         ids=lambda c: "T%d_d%d_F%d_E%d_k%d_a%g" % c)
def test_mxfp8_forward_parity(case):
    T, d, F, E, k, alpha = case
    g, h = cpu_and_gpu_inputs(T, d, F, E, k, seed=21, alpha=alpha)
    plan = _mx_plan(T, d, F, E, k)
    plan.quantize_weights(g["Wg"], g["Wu"], g["Wd"])
    Y, saved = plan.forward(g["X"], g["logits"], g["Wg"], g["Wu"], g["Wd"])
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    r = plan.routing(saved, T)
    idx_ref, _ = moe_ref.route(h["logits"], k)
    assert np.array_equal(r["idx"].cpu().numpy(), idx_ref)
    Yr, _ = moe_ref.forward(h["X"], h["logits"], h["Wg"], h["Wu"], h["Wd"], k, mx=True)
    Yb, _ = moe_ref.forward(h["X"], h["logits"], h["Wg"], h["Wu"], h["Wd"], k)
    err = rel_err(Y, Yr)
    assert err <= MX_TOL, (err, rel_err(Y, Yb))


@pytest.mark.parametrize("case", [(128, 256, 512, 8, 2, 0.0), (512, 1024, 512, 32, 4, 1.1), (300, 512, 768, 16, 3, 1.5)],
                         ids=lambda c: "T%d_d%d_F%d_E%d_k%d_a%g" % c)
def test_mxfp8_backward_parity(case):
    """MXFP8 dgrad GEMMs (dY along d with Wd^T along d; dA/dB along F with
    Wg^T/Wu^T along F), bf16 weight gradients, against the oracle's emulation
    (the backward on the saved context as stored: a|b in bf16)."""
    T, d, F, E, k, alpha = case
    g, h = cpu_and_gpu_inputs(T, d, F, E, k, seed=22, alpha=alpha)
    plan = _mx_plan(T, d, F, E, k)
    plan.quantize_weights(g["Wg"], g["Wu"], g["Wd"])
    Y, saved = plan.forward(g["X"], g["logits"], g["Wg"], g["Wu"], g["Wd"])
    out = plan.backward(g["dY"], g["X"], g["Wg"], g["Wu"], g["Wd"], saved)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    Yr, ctx = moe_ref.forward(h["X"], h["logits"], h["Wg"], h["Wu"], h["Wd"], k, mx=True)
    # the backward reads a|b as the forward stored them (bf16); the E4M3 codes
    # of dA|dB are decided from those values on the GPU
    gr = moe_ref.backward(h["dY"], h["X"], h["logits"], h["Wg"], h["Wu"], h["Wd"], moe_ref.stored_context(ctx))
    errs = {key: rel_err(out[key], gr[key]) for key in ("dX", "dWg", "dWu", "dWd", "dg", "dlogits")}
    assert all(v <= MX_TOL for v in errs.values()), errs
    # the gradient of the plain quantised layer (a|b never rounded to bf16):
    # storing a|b in bf16 must not move any gradient by more than the bound
    # as a whole, nor dX, dg, dlogits at any element.  Element-wise, a weight
    # gradient can differ by one E4M3 code step of an operand whose code flips
    # between the two contexts, so dW is bounded normwise only.
    gu = moe_ref.backward(h["dY"], h["X"], h["logits"], h["Wg"], h["Wu"], h["Wd"], ctx)
    errs_u = {key: rel_err_norm(out[key], gu[key]) for key in ("dX", "dWg", "dWu", "dWd", "dg", "dlogits")}
    errs_u.update({key + "_max": rel_err(out[key], gu[key]) for key in ("dX", "dg", "dlogits")})
    assert all(v <= MX_TOL for v in errs_u.values()), errs_u


@pytest.mark.parametrize("multi", [False, True], ids=["one_launch", "multi_launch"])
@pytest.mark.parametrize("mb_rows,slots,movers", [(0, 0, 0), (128, 2, 1), (512, 3, 4)])
def test_mxfp8_ring_megakernel_matches_separate_kernels_bitwise(mb_rows, slots, movers, multi):
    """The MXFP8 ring megakernel (movers copy the once-quantised token rows
    into the slot; h is re-quantised into the ring slot) must equal the
    separate-kernel MXFP8 schedule bit for bit, forward and backward -- as one
    launch that also quantises, routes and combines, and between separate
    routing / quantisation / combine launches."""
    T, d, F, E, k = 700, 512, 512, 24, 4
    g, h = cpu_and_gpu_inputs(T, d, F, E, k, seed=41, alpha=1.1)
    flags = moe.MOE_DEBUG_RING_MEGAKERNEL | (moe.MOE_DEBUG_MULTI_LAUNCH if multi else 0)
    ring = moe.Plan(moe.Config(T_max=T, d=d, F=F, E=E, k=k, prec=moe.MOE_MXFP8, minibatch_rows=mb_rows,
                               ring_slots=slots, mover_ctas=movers, debug_flags=flags))
    sep = moe.Plan(moe.Config(T_max=T, d=d, F=F, E=E, k=k, prec=moe.MOE_MXFP8,
                              debug_flags=moe.MOE_DEBUG_SEPARATE_KERNELS))
    for p in (ring, sep):
        p.quantize_weights(g["Wg"], g["Wu"], g["Wd"])
    Ya, sa = ring.forward(g["X"], g["logits"], g["Wg"], g["Wu"], g["Wd"])
    Yb, sb = sep.forward(g["X"], g["logits"], g["Wg"], g["Wu"], g["Wd"])
    ga = ring.backward(g["dY"], g["X"], g["Wg"], g["Wu"], g["Wd"], sa)
    gb = sep.backward(g["dY"], g["X"], g["Wg"], g["Wu"], g["Wd"], sb)
    torch.cuda.synchronize()
    assert ring.device_status() == 0 and sep.device_status() == 0
    assert torch.equal(Ya, Yb)
    for key in ("dX", "dWg", "dWu", "dWd", "dg", "dlogits"):
        assert torch.equal(ga[key], gb[key]), key
    ra, rb = ring.routing(sa, T), sep.routing(sb, T)
    for key in ("idx", "w", "counts", "offsets", "perm_src", "dest"):
        assert torch.equal(ra[key], rb[key]), key
    Yr, _ = moe_ref.forward(h["X"], h["logits"], h["Wg"], h["Wu"], h["Wd"], k, mx=True)
    assert rel_err(Ya, Yr) <= MX_TOL


@pytest.mark.parametrize("flags", [0, moe.MOE_DEBUG_RING_MEGAKERNEL], ids=["default", "ring"])
@pytest.mark.parametrize("alpha", [0.0, 1.1, 1.5])
def test_mxfp8_bitwise_deterministic_over_10_runs(flags, alpha):
    """Ten forward + backward runs give bitwise identical outputs, gradients
    and routing buffers, for each routing skew and schedule."""
    T, d, F, E, k = 512, 512, 512, 16, 4
    g, _ = cpu_and_gpu_inputs(T, d, F, E, k, seed=5, alpha=alpha)
    plan = moe.Plan(moe.Config(T_max=T, d=d, F=F, E=E, k=k, prec=moe.MOE_MXFP8, debug_flags=flags))
    plan.quantize_weights(g["Wg"], g["Wu"], g["Wd"])
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
    torch.cuda.synchronize()
    assert plan.device_status() == 0


def test_mxfp8_forward_needs_quantized_weights():
    T, d, F, E, k = 64, 256, 256, 4, 2
    g, _ = cpu_and_gpu_inputs(T, d, F, E, k, seed=6)
    plan = _mx_plan(T, d, F, E, k)
    with pytest.raises(moe.MoEError) as ei:
        plan.forward(g["X"], g["logits"], g["Wg"], g["Wu"], g["Wd"])
    assert ei.value.status == 1


@pytest.mark.parametrize("E,A,B", [(2, 128, 64), (3, 256, 192), (1, 7168 // 4, 128)])
def test_mx_quantize_transposed_bit_exact(E, A, B):
    """The transposed weight quantiser (the dgrad GEMMs' copies) against the
    oracle's codec applied to each transposed matrix, byte for byte."""
    src = torch.stack([_special_matrix(A, B, seed=E * 100 + i + A) for i in range(E)])
    q, sf = moe.mx_quantize_transposed(src.cuda())
    torch.cuda.synchronize()
    T = src.to(torch.float64).transpose(1, 2).reshape(E * B, A).numpy()
    codes, scales = mxfp8.mx_quantize(T, axis=1)
    assert np.array_equal(q.cpu().numpy().reshape(E * B, A), codes)
    assert np.array_equal(sf.cpu().numpy()[_atom_offsets(E * B, A)], scales)


@pytest.mark.parametrize("prec", [moe.MOE_MXFP8, moe.MOE_NVFP4], ids=["mxfp8", "nvfp4"])
def test_block_scaled_module_requantises_after_an_update(prec):
    """MoELayer(prec=...) quantises its weights before its first forward and
    again after an in-place update (what an optimiser step does): each forward
    equals, bitwise, a plan given the current weights' quantisation."""
    T, d, F, E, k = 128, 256, 512, 8, 2
    g, _ = cpu_and_gpu_inputs(T, d, F, E, k, seed=61, alpha=1.1)
    layer = moe.MoELayer(d, F, E, k, T_max=T, prec=prec)
    with torch.no_grad():
        for n in ("Wg", "Wu", "Wd"):
            getattr(layer, n).copy_(g[n])
    ref = moe.Plan(moe.Config(T_max=T, d=d, F=F, E=E, k=k, prec=prec))

    def expected():
        W = [getattr(layer, n).detach() for n in ("Wg", "Wu", "Wd")]
        ref.quantize_weights(*W)
        Y, _ = ref.forward(g["X"], g["logits"], *W)
        return Y

    X = g["X"].clone().requires_grad_(True)
    Y1 = layer(X, g["logits"])
    assert torch.equal(Y1, expected())
    Y1.backward(g["dY"])
    assert X.grad is not None and all(getattr(layer, n).grad is not None for n in ("Wg", "Wu", "Wd"))
    torch.optim.SGD(layer.parameters(), lr=0.5).step()   # in-place: the layer must quantise again
    Y2 = layer(g["X"], g["logits"])
    assert not torch.equal(Y2, Y1)
    assert torch.equal(Y2, expected())
    torch.cuda.synchronize()
    assert layer.plan.device_status() == 0 and ref.device_status() == 0


def test_mxfp8_one_launch_ring_forward_replays_from_a_cuda_graph():
    """The MXFP8 one-launch forward (token quantisation, routing, layout, ring
    pipeline and combine in one cooperative kernel) captured once and
    replayed: its grid barriers and hand-off counters reset themselves, so
    every replay equals the eager forward bitwise."""
    T, d, F, E, k = 300, 256, 512, 16, 4
    g, _ = cpu_and_gpu_inputs(T, d, F, E, k, seed=62, alpha=1.1)
    plan = moe.Plan(moe.Config(T_max=T, d=d, F=F, E=E, k=k, prec=moe.MOE_MXFP8,
                               debug_flags=moe.MOE_DEBUG_RING_MEGAKERNEL))
    plan.quantize_weights(g["Wg"], g["Wu"], g["Wd"])
    saved = plan.new_saved(T)
    Y = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        plan.forward(g["X"], g["logits"], g["Wg"], g["Wu"], g["Wd"], Y=Y, saved=saved, stream=stream)
    stream.synchronize()
    assert plan.device_status() == 0
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
