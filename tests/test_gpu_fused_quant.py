"""The quantisers fused into the block-scaled GEMM epilogues, bit for bit.

With MOE_DEBUG_DUMP_QUANT the plan keeps the fp32 values its epilogues
quantise -- h in the forward's up GEMM (along F), dA|dB in the backward's u
GEMM (along 2F) -- next to the bytes they wrote.  Re-quantising the GPU's own
fp32 values with the oracle's codec (OCP MX for MXFP8; E2M1 with E4M3 scales
per 16 and tensor scale 1 for NVFP4) must reproduce every element byte and
every scale byte, padding rows included.  The same holds for the operands
quantised outside the GEMMs (the dispatch's sorted rows, the weight
gradients' transposed operands), checked against the oracle's quantisation of
rows built here from the inputs and the routing.
"""
import numpy as np
import pytest
import torch

from mixture_experts_layer_19_gb300 import moe
from oracle import mxfp8, nvfp4
from tests.util import cpu_and_gpu_inputs

pytestmark = pytest.mark.gpu


def _atom_offsets(rows, K, blk):
    # scale byte of (row r, block b): atom (r // 128) * (K // (4 blk)) + b // 4,
    # byte (r % 32) * 16 + ((r // 32) % 4) * 4 + b % 4 inside the 512-byte atom
    r = np.arange(rows)[:, None]
    b = np.arange(K // blk)[None, :]
    atom = (r // 128) * (K // (4 * blk)) + b // 4
    return atom * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + b % 4


@pytest.mark.parametrize("prec", [moe.MOE_MXFP8, moe.MOE_NVFP4], ids=["mxfp8", "nvfp4"])
@pytest.mark.parametrize("case", [(300, 512, 768, 16, 3, 1.5), (128, 256, 512, 8, 2, 0.0)],
                         ids=lambda c: "T%d_d%d_F%d_E%d_k%d_a%g" % c)
def test_fused_epilogue_quantisation_bit_exact(prec, case):
    T, d, F, E, k, alpha = case
    g, _ = cpu_and_gpu_inputs(T, d, F, E, k, seed=17, alpha=alpha)
    plan = moe.Plan(moe.Config(T_max=T, d=d, F=F, E=E, k=k, prec=prec, debug_flags=moe.MOE_DEBUG_DUMP_QUANT))
    plan.quantize_weights(g["Wg"], g["Wu"], g["Wd"])
    Y, saved = plan.forward(g["X"], g["logits"], g["Wg"], g["Wu"], g["Wd"])
    plan.backward(g["dY"], g["X"], g["Wg"], g["Wu"], g["Wd"], saved)
    counts = plan.routing(saved, T)["counts"].cpu().numpy()
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    rows = int(sum((c + 127) // 128 * 128 for c in counts))   # padded sorted rows in use
    nv = prec == moe.MOE_NVFP4
    blk = 16 if nv else 32
    for which, C in ((0, F), (1, 2 * F)):
        vals, q, sf = plan.debug_quant_dump(which)
        torch.cuda.synchronize()
        v = vals[:rows].cpu().double().numpy()
        assert np.isfinite(v).all() and np.abs(v).max() > 0
        if nv:
            codes, scales = nvfp4.nv_quantize(v, axis=1, g=1.0)
            got = nvfp4.nv_unpack(q[:rows].cpu().numpy())
        else:
            codes, scales = mxfp8.mx_quantize(v, axis=1)
            got = q[:rows].cpu().numpy()
        bad = np.argwhere(got != codes)
        assert bad.size == 0, (which, bad[:5].tolist(), v[tuple(bad[0])] if bad.size else None)
        assert np.array_equal(sf.cpu().numpy()[_atom_offsets(rows, C, blk)], scales), which


def _sorted_rows(src, perm, counts, k):
    """The padded sorted rows of a token tensor: expert segments padded to 128
    rows, row j of expert e's segment = token perm[offsets[e] + j] // k, the
    padding rows zero."""
    rows = int(sum((c + 127) // 128 * 128 for c in counts))
    out = np.zeros((rows, src.shape[1]))
    r0 = o = 0
    for c in counts:
        out[r0:r0 + c] = src[perm[o:o + c] // k]
        r0 += (c + 127) // 128 * 128
        o += c
    return out


@pytest.mark.parametrize("prec", [moe.MOE_MXFP8, moe.MOE_NVFP4], ids=["mxfp8", "nvfp4"])
@pytest.mark.parametrize("case", [(300, 512, 768, 16, 3, 1.5), (200, 256, 512, 8, 2, 0.0),
                                  # one token, k = 1 (the plain-division row lookup); k = 8 over 32
                                  # experts, most of them empty, 12 column blocks
                                  (1, 256, 512, 4, 1, 0.0), (64, 768, 512, 32, 8, 1.1)],
                         ids=lambda c: "T%d_d%d_F%d_E%d_k%d_a%g" % c)
def test_weight_gradient_operands_bit_exact(prec, case):
    """The block-scaled weight gradients' operands, transposed and quantised
    along the sorted rows: dY^T and X^T (gathered from the token tensors in
    one pass) against the oracle's quantisation of the sorted rows built here
    from the inputs and the routing; [dA|dB]^T and (w h)^T against the
    oracle's quantisation of the bf16 rows they were made from.  Every element
    byte and scale byte of the rows in use, padding rows included."""
    T, d, F, E, k, alpha = case
    g, h = cpu_and_gpu_inputs(T, d, F, E, k, seed=29, alpha=alpha)
    plan = moe.Plan(moe.Config(T_max=T, d=d, F=F, E=E, k=k, prec=prec, debug_flags=moe.MOE_DEBUG_DUMP_QUANT))
    plan.quantize_weights(g["Wg"], g["Wu"], g["Wd"])
    Y, saved = plan.forward(g["X"], g["logits"], g["Wg"], g["Wu"], g["Wd"])
    plan.backward(g["dY"], g["X"], g["Wg"], g["Wu"], g["Wd"], saved)
    r = plan.routing(saved, T)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    counts = r["counts"].cpu().numpy()
    perm = r["perm_src"].cpu().numpy().astype(np.int64)
    rows = int(sum((c + 127) // 128 * 128 for c in counts))
    P = plan.padded_rows()
    nv = prec == moe.MOE_NVFP4
    blk = 16 if nv else 32
    for which, name in ((2, "dY"), (3, "X"), (4, "dAB"), (5, "wH")):
        vals, q, sf = plan.debug_quant_dump(which)
        torch.cuda.synchronize()
        if which in (2, 3):
            assert vals is None
            src = _sorted_rows(h[name], perm, counts, k)
        else:
            src = vals[:rows].cpu().double().numpy()
            assert np.abs(src).max() > 0
        op = src.T                                   # [C, rows]: quantised along the sorted rows
        C = op.shape[0]
        if nv:
            codes, scales = nvfp4.nv_quantize(op, axis=1, g=1.0)
            got = nvfp4.nv_unpack(q.cpu().numpy()[:, :rows // 2])
        else:
            codes, scales = mxfp8.mx_quantize(op, axis=1)
            got = q.cpu().numpy()[:, :rows]
        bad = np.argwhere(got != codes)
        assert bad.size == 0, (name, bad[:5].tolist())
        atoms = _atom_offsets(C, P, blk)[:, :rows // blk]
        assert np.array_equal(sf.cpu().numpy()[atoms], scales), name


@pytest.mark.parametrize("prec", [moe.MOE_MXFP8, moe.MOE_NVFP4], ids=["mxfp8", "nvfp4"])
@pytest.mark.parametrize("case", [(300, 512, 768, 16, 3, 1.5), (200, 256, 512, 8, 2, 0.0),
                                  (1, 256, 512, 4, 1, 0.0), (64, 768, 512, 32, 8, 1.1)],
                         ids=lambda c: "T%d_d%d_F%d_E%d_k%d_a%g" % c)
def test_dispatched_rows_bit_exact(prec, case):
    """The dispatch's quantised sorted rows (each token quantised along d once
    and stored into its k sorted rows): X after the forward, dY after the
    backward, against the oracle's quantisation of the sorted rows built here
    from the inputs and the routing.  Every element byte and scale byte of the
    rows in use, padding rows (zero codes, zero scales) included."""
    T, d, F, E, k, alpha = case
    g, h = cpu_and_gpu_inputs(T, d, F, E, k, seed=31, alpha=alpha)
    plan = moe.Plan(moe.Config(T_max=T, d=d, F=F, E=E, k=k, prec=prec, debug_flags=moe.MOE_DEBUG_DUMP_QUANT))
    plan.quantize_weights(g["Wg"], g["Wu"], g["Wd"])
    nv = prec == moe.MOE_NVFP4
    blk = 16 if nv else 32
    Y, saved = plan.forward(g["X"], g["logits"], g["Wg"], g["Wu"], g["Wd"])
    r = plan.routing(saved, T)
    counts = r["counts"].cpu().numpy()
    perm = r["perm_src"].cpu().numpy().astype(np.int64)
    rows = int(sum((c + 127) // 128 * 128 for c in counts))
    for name in ("X", "dY"):
        if name == "dY":
            plan.backward(g["dY"], g["X"], g["Wg"], g["Wu"], g["Wd"], saved)
        vals, q, sf = plan.debug_quant_dump(6)
        torch.cuda.synchronize()
        assert plan.device_status() == 0
        assert vals is None
        src = _sorted_rows(h[name], perm, counts, k)
        if nv:
            codes, scales = nvfp4.nv_quantize(src, axis=1, g=1.0)
            got = nvfp4.nv_unpack(q[:rows].cpu().numpy())
        else:
            codes, scales = mxfp8.mx_quantize(src, axis=1)
            got = q[:rows].cpu().numpy()
        bad = np.argwhere(got != codes)
        assert bad.size == 0, (name, bad[:5].tolist())
        assert np.array_equal(sf.cpu().numpy()[_atom_offsets(rows, d, blk)], scales), name


def test_dump_needs_the_flag():
    plan = moe.Plan(moe.Config(T_max=64, d=256, F=256, E=4, k=2, prec=moe.MOE_NVFP4))
    with pytest.raises(moe.MoEError) as ei:
        plan.debug_quant_dump(0)
    assert ei.value.status == 1


def test_dump_rejects_bad_operand_arguments():
    """which outside 0..6, and source values asked of dY^T, X^T or the
    dispatched rows (which keep none), are argument errors that copy
    nothing."""
    plan = moe.Plan(moe.Config(T_max=64, d=256, F=256, E=4, k=2, prec=moe.MOE_MXFP8,
                               debug_flags=moe.MOE_DEBUG_DUMP_QUANT))
    buf = torch.zeros(plan.padded_rows() * 256, dtype=torch.float32, device="cuda")
    for which, vals in ((7, None), (-1, None), (2, buf), (3, buf), (6, buf)):
        st = moe.lib().moe_debug_quant_dump(plan.handle, which, moe._ptr(vals), None, None, None)
        assert st == moe.MOE_ERR_INVALID_ARG, which
    assert torch.count_nonzero(buf).item() == 0
