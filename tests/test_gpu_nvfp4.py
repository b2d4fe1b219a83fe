"""GPU checks of the NVFP4 path against the fp64 oracle.

* The quantisers (moe_nv_quantize, moe_nv_quantize_transposed, which also
  quantise the weights) and the tensor scale (moe_nv_tensor_scale) are
  compared byte for byte with the oracle's codec: every packed E2M1 element,
  every E4M3 scale, zero blocks, -0, saturation, subnormal and vanishing
  scales, with tensor scale 1 and with a weight-style tensor scale.
* The NVFP4 layer (E2M1 gather, kind::mxf4nvf4 [a|b] GEMM + SwiGLU with h
  re-quantised in its epilogue, down GEMM, combine; dgrad GEMMs with dA|dB
  re-quantised; bf16 weight gradients) against the oracle's NVFP4 emulation:
  max|err| / max|ref| <= 4e-2, routing bit-exact, bitwise repeatable.  The
  backward's oracle receives the saved context as the forward stored it
  (a|b rounded to bf16): it is an input of the backward, and the E2M1 codes
  of dA|dB are decided from it on the GPU.
"""
import numpy as np
import pytest
import torch

from mixture_experts_layer_19_gb300 import moe
from oracle import moe_ref, mxfp8, nvfp4
from tests.util import cpu_and_gpu_inputs, rel_err, rel_err_norm

pytestmark = pytest.mark.gpu
NV_TOL = 4e-2


def _atom_offsets(rows, K):
    # scale byte of (row r, 16-block b): atom (r // 128) * (K // 64) + b // 4,
    # byte (r % 32) * 16 + ((r // 32) % 4) * 4 + b % 4 inside the 512-byte atom
    r = np.arange(rows)[:, None]
    b = np.arange(K // 16)[None, :]
    atom = (r // 128) * (K // 64) + b // 4
    return atom * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + b % 4


def _special_matrix(rows, K, seed):
    g = torch.Generator().manual_seed(seed)
    v = torch.randn((rows, K), generator=g) * torch.exp2(torch.randint(-8, 8, (rows, 1), generator=g).float())
    v[0, :16] = 0.0                                    # all-zero block
    v[1, :16] = -0.0
    v[1, 16:32] = 2.0 ** -14                           # scale rounds to zero: zero codes
    v[2, :16] = torch.linspace(-3000, 3000, 16)        # block scale saturates at 448
    v[3, :16] = 1.0                                    # scale 0x23, elements 6
    v[4, :16] = torch.tensor([6, 5, 0.25, 0.75, -1.25, 2.5, 3.5, -0.1, 1.5, 3, 0, 0, 0, 0, 0, 0.0])  # ties
    v[5, :16] = 0.01                                   # subnormal E4M3 scale
    v[5, 3] = -0.001
    v[6, 16:32] = -1e-4                                # negative values that round to -0
    v[6, 20] = 1.0
    return v.to(torch.bfloat16)


def _unpack(q):
    return nvfp4.nv_unpack(q.cpu().numpy())


@pytest.mark.parametrize("rows,K,tensor_scale", [(128, 64, False), (200, 512, False), (384, 7168 // 4, True),
                                                 (130, 256, True)])
def test_nv_quantize_bit_exact(rows, K, tensor_scale):
    src = _special_matrix(rows, K, seed=rows + K)
    srcd = src.cuda()
    g = moe.nv_tensor_scale(srcd) if tensor_scale else None
    q, sf = moe.nv_quantize(srcd, g)
    torch.cuda.synchronize()
    gv = 1.0
    if tensor_scale:
        gv = nvfp4.tensor_scale(float(src.abs().max()))
        assert g.cpu().numpy()[0] == gv                # the tensor scale itself is bit-exact
    codes, scales = nvfp4.nv_quantize(src.to(torch.float64).numpy(), axis=1, g=gv)
    assert np.array_equal(_unpack(q), codes)
    assert np.array_equal(sf.cpu().numpy()[_atom_offsets(rows, K)], scales)


def test_nv_tensor_scale_of_two_tensors_and_zero():
    a = torch.randn((300, 64)).to(torch.bfloat16)
    b = (torch.randn((77,)) * 40).to(torch.bfloat16)
    g = moe.nv_tensor_scale(a.cuda(), b.cuda())
    z = moe.nv_tensor_scale(torch.zeros((64,), dtype=torch.bfloat16, device="cuda"))
    torch.cuda.synchronize()
    amax = max(float(a.abs().max()), float(b.abs().max()))
    assert g.cpu().numpy()[0] == nvfp4.tensor_scale(amax)
    assert z.cpu().numpy()[0] == 1.0


@pytest.mark.parametrize("E,A,B", [(2, 128, 64), (3, 256, 192), (1, 7168 // 4, 128)])
def test_nv_quantize_transposed_bit_exact(E, A, B):
    src = torch.stack([_special_matrix(A, B, seed=E * 100 + i + A) for i in range(E)])
    srcd = src.cuda()
    g = moe.nv_tensor_scale(srcd)
    q, sf = moe.nv_quantize_transposed(srcd, g)
    torch.cuda.synchronize()
    gv = nvfp4.tensor_scale(float(src.abs().max()))
    codes = _unpack(q).reshape(E * B, A)
    offs = _atom_offsets(E * B, A)
    sfn = sf.cpu().numpy()
    for e in range(E):
        c_ref, s_ref = nvfp4.nv_quantize(src[e].to(torch.float64).numpy().T, axis=1, g=gv)
        assert np.array_equal(codes[e * B:(e + 1) * B], c_ref), e
        assert np.array_equal(sfn[offs[e * B:(e + 1) * B]], s_ref), e


def _nv_plan(T, d, F, E, k):
    return moe.Plan(moe.Config(T_max=T, d=d, F=F, E=E, k=k, prec=moe.MOE_NVFP4))


def _weight_scales(h):
    return nvfp4.weight_scales(h["Wg"], h["Wu"], h["Wd"])


CASES = [(128, 256, 512, 8, 2, 0.0), (512, 1024, 512, 32, 4, 1.1), (300, 512, 768, 16, 3, 1.5)]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "T%d_d%d_F%d_E%d_k%d_a%g" % c)
def test_nvfp4_forward_parity(case):
    T, d, F, E, k, alpha = case
    g, h = cpu_and_gpu_inputs(T, d, F, E, k, seed=21, alpha=alpha)
    plan = _nv_plan(T, d, F, E, k)
    plan.quantize_weights(g["Wg"], g["Wu"], g["Wd"])
    Y, saved = plan.forward(g["X"], g["logits"], g["Wg"], g["Wu"], g["Wd"])
    scales = plan.nv_weight_scales()
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    ws = _weight_scales(h)
    assert np.array_equal(scales.cpu().numpy(), np.array(ws, dtype=np.float32))
    r = plan.routing(saved, T)
    idx_ref, _ = moe_ref.route(h["logits"], k)
    assert np.array_equal(r["idx"].cpu().numpy(), idx_ref)
    Yr, _ = moe_ref.forward(h["X"], h["logits"], h["Wg"], h["Wu"], h["Wd"], k, mx="nvfp4", wscales=ws)
    Yb, _ = moe_ref.forward(h["X"], h["logits"], h["Wg"], h["Wu"], h["Wd"], k)
    err = rel_err(Y, Yr)
    assert err <= NV_TOL, (err, rel_err(Y, Yb))
    assert rel_err(Y, Yb) > 0.05                       # the quantisation really happened


@pytest.mark.parametrize("case", CASES, ids=lambda c: "T%d_d%d_F%d_E%d_k%d_a%g" % c)
def test_nvfp4_backward_parity(case):
    T, d, F, E, k, alpha = case
    g, h = cpu_and_gpu_inputs(T, d, F, E, k, seed=22, alpha=alpha)
    plan = _nv_plan(T, d, F, E, k)
    plan.quantize_weights(g["Wg"], g["Wu"], g["Wd"])
    Y, saved = plan.forward(g["X"], g["logits"], g["Wg"], g["Wu"], g["Wd"])
    out = plan.backward(g["dY"], g["X"], g["Wg"], g["Wu"], g["Wd"], saved)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    ws = _weight_scales(h)
    _, ctx = moe_ref.forward(h["X"], h["logits"], h["Wg"], h["Wu"], h["Wd"], k, mx="nvfp4", wscales=ws)
    gr = moe_ref.backward(h["dY"], h["X"], h["logits"], h["Wg"], h["Wu"], h["Wd"], moe_ref.stored_context(ctx))
    errs = {key: rel_err(out[key], gr[key]) for key in ("dX", "dWg", "dWu", "dWd", "dg", "dlogits")}
    assert all(v <= NV_TOL for v in errs.values()), errs
    # the gradient of the plain quantised layer (a|b never rounded to bf16),
    # normwise: E2M1 has one mantissa bit, so a code that flips between the two
    # contexts moves single elements of dX and dW by a large step
    gu = moe_ref.backward(h["dY"], h["X"], h["logits"], h["Wg"], h["Wu"], h["Wd"], ctx)
    errs_u = {key: rel_err_norm(out[key], gu[key]) for key in ("dX", "dWg", "dWu", "dWd", "dg", "dlogits")}
    assert all(v <= NV_TOL for v in errs_u.values()), errs_u


@pytest.mark.parametrize("alpha", [0.0, 1.1, 1.5])
def test_nvfp4_bitwise_deterministic_over_10_runs(alpha):
    """Ten forward + backward runs give bitwise identical outputs, gradients
    and routing buffers, for each routing skew."""
    T, d, F, E, k = 512, 512, 512, 16, 4
    g, _ = cpu_and_gpu_inputs(T, d, F, E, k, seed=5, alpha=alpha)
    plan = _nv_plan(T, d, F, E, k)
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


def test_nvfp4_bitwise_deterministic_and_empty_experts():
    T, d, F, E, k = 256, 512, 512, 16, 4
    # every token prefers experts 0..3: the other 12 experts receive no rows
    g, _ = cpu_and_gpu_inputs(T, d, F, E, k, seed=5,
                              logits_fn=lambda L: L + torch.tensor([20.0] * 4 + [0.0] * 12))
    plan = _nv_plan(T, d, F, E, k)
    plan.quantize_weights(g["Wg"], g["Wu"], g["Wd"])
    ref = None
    for _ in range(5):
        Y, saved = plan.forward(g["X"], g["logits"], g["Wg"], g["Wu"], g["Wd"])
        out = plan.backward(g["dY"], g["X"], g["Wg"], g["Wu"], g["Wd"], saved)
        cur = [Y.clone()] + [out[n].clone() for n in ("dX", "dWg", "dWu", "dWd", "dg", "dlogits")]
        if ref is None:
            ref = cur
        else:
            for a, b in zip(ref, cur):
                assert torch.equal(a, b)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    assert torch.count_nonzero(ref[2][4:]).item() == 0 and torch.count_nonzero(ref[4][4:]).item() == 0


def test_nvfp4_needs_quantized_weights_and_validates():
    T, d, F, E, k = 64, 256, 256, 4, 2
    g, _ = cpu_and_gpu_inputs(T, d, F, E, k, seed=6)
    plan = _nv_plan(T, d, F, E, k)
    with pytest.raises(moe.MoEError) as ei:
        plan.forward(g["X"], g["logits"], g["Wg"], g["Wu"], g["Wd"])
    assert ei.value.status == 1
    with pytest.raises(moe.MoEError) as ei:   # bf16 plans hold no tensor scales
        moe.Plan(moe.Config(T_max=T, d=d, F=F, E=E, k=k)).nv_weight_scales()
    assert ei.value.status == 1
    with pytest.raises(moe.MoEError) as ei:
        moe.nv_quantize(torch.zeros((4, 48), dtype=torch.bfloat16, device="cuda"))   # K % 64 != 0
    assert ei.value.status == 1


def _block_scaled_parity(prec, plan, g, h, k, T):
    """Forward + backward of a block-scaled plan against the oracle's emulation
    of its quantisation points (backward on the saved context as stored)."""
    fmt = "nvfp4" if prec == moe.MOE_NVFP4 else "mxfp8"
    Y, saved = plan.forward(g["X"], g["logits"], g["Wg"], g["Wu"], g["Wd"])
    out = plan.backward(g["dY"], g["X"], g["Wg"], g["Wu"], g["Wd"], saved)
    r = plan.routing(saved, T)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    assert np.array_equal(r["idx"].cpu().numpy(), moe_ref.route(h["logits"], k)[0])
    ws = _weight_scales(h) if fmt == "nvfp4" else None
    Yr, ctx = moe_ref.forward(h["X"], h["logits"], h["Wg"], h["Wu"], h["Wd"], k, mx=fmt, wscales=ws)
    gr = moe_ref.backward(h["dY"], h["X"], h["logits"], h["Wg"], h["Wu"], h["Wd"], moe_ref.stored_context(ctx))
    errs = {"Y": rel_err(Y, Yr)}
    errs.update({key: rel_err(out[key], gr[key]) for key in ("dX", "dWg", "dWu", "dWd", "dg", "dlogits")})
    assert all(v <= NV_TOL for v in errs.values()), errs
    return out


@pytest.mark.parametrize("prec", [moe.MOE_MXFP8, moe.MOE_NVFP4], ids=["mxfp8", "nvfp4"])
@pytest.mark.parametrize("T", [1, 3, 129])
def test_block_scaled_ragged_token_counts(prec, T):
    d, F, E, k = 256, 256, 8, 2
    g, h = cpu_and_gpu_inputs(T, d, F, E, k, seed=100 + T)
    plan = moe.Plan(moe.Config(T_max=256, d=d, F=F, E=E, k=k, prec=prec))
    plan.quantize_weights(g["Wg"], g["Wu"], g["Wd"])
    _block_scaled_parity(prec, plan, g, h, k, T)


@pytest.mark.parametrize("prec", [moe.MOE_MXFP8, moe.MOE_NVFP4], ids=["mxfp8", "nvfp4"])
def test_block_scaled_degenerate_routing_and_zero_tokens(prec):
    # every token picks experts 5 then 9; the other ten get nothing
    T, d, F, E, k = 300, 256, 256, 12, 2
    bias = torch.zeros(E)
    bias[5], bias[9] = 40.0, 30.0
    g, h = cpu_and_gpu_inputs(T, d, F, E, k, seed=8, logits_fn=lambda L: L + bias[None, :])
    plan = moe.Plan(moe.Config(T_max=T, d=d, F=F, E=E, k=k, prec=prec))
    plan.quantize_weights(g["Wg"], g["Wu"], g["Wd"])
    out = _block_scaled_parity(prec, plan, g, h, k, T)
    empty = [e for e in range(E) if e not in (5, 9)]
    for key in ("dWg", "dWu", "dWd"):
        assert torch.count_nonzero(out[key][empty]).item() == 0
    # no tokens: a no-op forward and zero weight gradients
    X0 = g["X"][:0].contiguous()
    Y0, s0 = plan.forward(X0, g["logits"][:0].contiguous(), g["Wg"], g["Wu"], g["Wd"])
    out0 = plan.backward(X0, X0, g["Wg"], g["Wu"], g["Wd"], s0)
    torch.cuda.synchronize()
    assert Y0.shape == (0, d)
    for key in ("dWg", "dWu", "dWd"):
        assert torch.count_nonzero(out0[key]).item() == 0
