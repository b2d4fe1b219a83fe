"""Pins for the oracle's layer forward/backward (BF16 arithmetic and MXFP8
quantisation points).

Independent checks:
* the whole layer rebuilt from torch float64 library routines (topk, softmax,
  silu, matmul) with torch autograd for every gradient;
* E=1, k=1 reduces to a dense SwiGLU FFN;
* central finite differences of the oracle's own forward for its backward;
* identity experts: top-1 returns X exactly, top-k returns X;
* closed forms (Wu = 0 gives Y = 0 and zero gate/up gradients);
* MXFP8 inputs that are exactly representable along every axis, where only
  the re-quantised intermediates (h, dA/dB, w*h) can add error.
"""
import numpy as np
import pytest
import torch

from mixture_experts_layer_19_gb300.workload import LayerShape, make_inputs, to_f64
from oracle import moe_ref, mxfp8


def _inputs(T, d, F, E, k, seed=0, alpha=0.0):
    inp = make_inputs(LayerShape(T, d, F, E, k), seed=seed, alpha=alpha)
    return (to_f64(inp.X), to_f64(inp.logits), to_f64(inp.Wg), to_f64(inp.Wu),
            to_f64(inp.Wd), to_f64(inp.dY))


def _torch_layer(X, logits, Wg, Wu, Wd, dY, k):
    X, logits, Wg, Wu, Wd = [torch.tensor(a, dtype=torch.float64, requires_grad=True)
                             for a in (X, logits, Wg, Wu, Wd)]
    vals, ids = torch.topk(logits, k, dim=1)
    w = torch.softmax(vals, dim=1)
    Y = torch.zeros_like(X)
    for j in range(k):
        e = ids[:, j]
        a = torch.einsum("td,tfd->tf", X, Wg[e])
        b = torch.einsum("td,tfd->tf", X, Wu[e])
        h = torch.nn.functional.silu(a) * b
        y = torch.einsum("tf,tdf->td", h, Wd[e])
        Y = Y + w[:, j:j + 1] * y
    (Y * torch.tensor(dY)).sum().backward()
    return {"Y": Y.detach().numpy(), "dX": X.grad.numpy(), "dWg": Wg.grad.numpy(),
            "dWu": Wu.grad.numpy(), "dWd": Wd.grad.numpy(), "dlogits": logits.grad.numpy(),
            "ids": ids.numpy()}


@pytest.mark.parametrize("T,d,F,E,k,alpha", [(16, 32, 64, 4, 2, 0.0), (24, 64, 32, 8, 3, 1.1), (9, 32, 32, 3, 1, 0.0)])
def test_layer_matches_torch_autograd(T, d, F, E, k, alpha):
    X, L, Wg, Wu, Wd, dY = _inputs(T, d, F, E, k, seed=5, alpha=alpha)
    Y, ctx = moe_ref.forward(X, L, Wg, Wu, Wd, k)
    g = moe_ref.backward(dY, X, L, Wg, Wu, Wd, ctx)
    ref = _torch_layer(X, L, Wg, Wu, Wd, dY, k)
    assert np.array_equal(ctx["idx"], ref["ids"])
    rel = lambda a, b: np.abs(a - b).max() / max(np.abs(b).max(), 1e-300)
    assert rel(Y, ref["Y"]) < 1e-12
    for key in ("dX", "dWg", "dWu", "dWd", "dlogits"):
        assert rel(g[key], ref[key]) < 1e-12, key


def test_single_expert_top1_is_dense_swiglu():
    X, L, Wg, Wu, Wd, dY = _inputs(12, 32, 64, 1, 1, seed=7)
    Y, ctx = moe_ref.forward(X, L, Wg, Wu, Wd, 1)
    x = torch.tensor(X)
    ref = (torch.nn.functional.silu(x @ torch.tensor(Wg[0]).T) * (x @ torch.tensor(Wu[0]).T)) @ torch.tensor(Wd[0]).T
    assert np.abs(Y - ref.numpy()).max() <= 1e-13 * np.abs(ref.numpy()).max()
    assert np.all(ctx["w"] == 1.0)


def test_finite_differences():
    T, d, F, E, k = 4, 8, 16, 4, 2
    X, L, Wg, Wu, Wd, dY = _inputs(T, d, F, E, k, seed=11)
    # spread logits so every top-k choice has a margin >> eps
    L = L + np.arange(E)[None, :] * 0.7
    Y, ctx = moe_ref.forward(X, L, Wg, Wu, Wd, k)
    g = moe_ref.backward(dY, X, L, Wg, Wu, Wd, ctx)
    eps = 1e-6

    def loss(X_, L_, Wg_, Wu_, Wd_):
        return float(np.sum(dY * moe_ref.forward(X_, L_, Wg_, Wu_, Wd_, k)[0]))

    args = {"X": X, "L": L, "Wg": Wg, "Wu": Wu, "Wd": Wd}
    grads = {"X": g["dX"], "L": g["dlogits"], "Wg": g["dWg"], "Wu": g["dWu"], "Wd": g["dWd"]}
    rng = np.random.default_rng(0)
    for name, arr in args.items():
        flat_idx = rng.choice(arr.size, size=min(arr.size, 12), replace=False)
        for fi in flat_idx:
            pos = np.unravel_index(fi, arr.shape)
            plus = {n: a.copy() for n, a in args.items()}
            minus = {n: a.copy() for n, a in args.items()}
            plus[name][pos] += eps
            minus[name][pos] -= eps
            fd = (loss(*plus.values()) - loss(*minus.values())) / (2 * eps)
            an = grads[name][pos]
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, pos, fd, an)


def test_identity_experts_return_input():
    X, L, Wg, Wu, Wd, _ = _inputs(20, 32, 32, 5, 1, seed=3)
    Y, _ = moe_ref.forward(X, L, None, None, None, 1, identity=True)
    assert np.array_equal(Y, X)
    Y3, _ = moe_ref.forward(X, L, None, None, None, 3, identity=True)
    assert np.abs(Y3 - X).max() <= 1e-15 * np.abs(X).max() * 4


def test_zero_up_projection_closed_form():
    X, L, Wg, Wu, Wd, dY = _inputs(16, 32, 32, 4, 2, seed=4)
    Wu = np.zeros_like(Wu)
    Y, ctx = moe_ref.forward(X, L, Wg, Wu, Wd, 2)
    g = moe_ref.backward(dY, X, L, Wg, Wu, Wd, ctx)
    assert np.all(Y == 0) and np.all(g["dWg"] == 0) and np.all(g["dWd"] == 0)
    assert np.all(g["dg"] == 0) and np.all(g["dlogits"] == 0)


def _mx_exact(shape, rng, scale_pow):
    """Values +-(1 + m/8) * 2^scale_pow, m in 0..6: exact MXFP8 along any axis."""
    m = rng.integers(0, 7, shape)
    s = rng.choice([-1.0, 1.0], shape)
    return s * (1.0 + m / 8.0) * 2.0 ** scale_pow


def test_mx_exact_inputs_only_intermediates_add_error():
    rng = np.random.default_rng(9)
    T, d, F, E, k = 32, 64, 64, 4, 2
    X = _mx_exact((T, d), rng, 0)
    Wg = _mx_exact((E, F, d), rng, -4)
    Wu = _mx_exact((E, F, d), rng, -4)
    Wd = _mx_exact((E, d, F), rng, -4)
    dY = _mx_exact((T, d), rng, 0)
    L = rng.standard_normal((T, E))
    for a in (X, Wg[0], Wd[0], dY):
        assert np.array_equal(mxfp8.mx_fake_quant(a, 0), a)
        assert np.array_equal(mxfp8.mx_fake_quant(a, -1), a)
    Y0, c0 = moe_ref.forward(X, L, Wg, Wu, Wd, k)
    Y1, c1 = moe_ref.forward(X, L, Wg, Wu, Wd, k, mx=True)
    # a and b come from exact operands: identical
    assert np.array_equal(c0["a"], c1["a"]) and np.array_equal(c0["b"], c1["b"])
    # y differs only through h's quantisation along F
    hq = mxfp8.mx_fake_quant(c0["h"], 1)
    y_expect = np.zeros_like(c0["y"])
    for e in range(E):
        rows = c0["layout"]["perm_src"][c0["layout"]["offsets"][e]:c0["layout"]["offsets"][e + 1]]
        y_expect[rows] = hq[rows] @ Wd[e].T
    assert np.abs(c1["y"] - y_expect).max() <= 1e-12 * np.abs(y_expect).max()
    rel = np.abs(Y1 - Y0).max() / np.abs(Y0).max()
    assert 0 < rel < 2 ** -4
    g0 = moe_ref.backward(dY, X, L, Wg, Wu, Wd, c0)
    g1 = moe_ref.backward(dY, X, L, Wg, Wu, Wd, c1)
    # dX differs only through dA/dB re-quantised along F
    r = np.abs(g1["dX"] - g0["dX"]).max() / np.abs(g0["dX"]).max()
    assert 0 < r < 2 ** -3, r
    # weight gradients: every operand quantised along the expert's tokens;
    # dY and X are exact along any axis, so only w*h, dA and dB (quantised from
    # their bf16 values) change
    qt = lambda v: mxfp8.mx_fake_quant(v, 0)
    lay = c0["layout"]
    for e in range(E):
        rows = lay["perm_src"][lay["offsets"][e]:lay["offsets"][e + 1]]
        if rows.size == 0:
            continue
        tok = rows // k
        wr = c0["w"].reshape(-1)[rows][:, None]
        a, b, h = c0["a"][rows], c0["b"][rows], c0["h"][rows]
        u = dY[tok] @ Wd[e]
        sa = moe_ref.sigmoid(a)
        da = wr * u * b * sa * (1 + a * (1 - sa))
        db = wr * u * moe_ref.silu(a)
        assert np.array_equal(qt(dY[tok]), dY[tok]) and np.array_equal(qt(X[tok]), X[tok])
        assert np.allclose(g1["dWd"][e], dY[tok].T @ qt(moe_ref.bf16_round(wr * h)), rtol=1e-12, atol=1e-12)
        assert np.allclose(g1["dWg"][e], qt(moe_ref.bf16_round(da)).T @ X[tok], rtol=1e-12, atol=1e-12)
        assert np.allclose(g1["dWu"][e], qt(moe_ref.bf16_round(db)).T @ X[tok], rtol=1e-12, atol=1e-12)
    rel_w = np.abs(g1["dWg"] - g0["dWg"]).max() / np.abs(g0["dWg"]).max()
    assert 0 < rel_w < 2 ** -3, rel_w
    # dg uses u (exact operands) and the unquantised h: identical
    assert np.array_equal(g0["dg"], g1["dg"])


def test_sampled_forms_equal_full_forms():
    T, d, F, E, k = 40, 64, 64, 6, 3
    X, L, Wg, Wu, Wd, dY = _inputs(T, d, F, E, k, seed=2, alpha=1.1)
    for mx in (False, True):
        Y, ctx = moe_ref.forward(X, L, Wg, Wu, Wd, k, mx=mx)
        g = moe_ref.backward(dY, X, L, Wg, Wu, Wd, ctx)
        toks = np.array([0, 5, 17, 39])
        s = moe_ref.forward_backward_tokens(X, L, Wg, Wu, Wd, dY, k, toks, mx=mx)
        for key, full in (("Y", Y), ("dX", g["dX"]), ("dg", g["dg"]), ("dlogits", g["dlogits"])):
            assert np.allclose(s[key], full[toks], rtol=1e-12, atol=1e-12), (mx, key)
        for e in (0, int(np.argmax(ctx["layout"]["counts"]))):
            dwg, dwu, dwd = moe_ref.expert_weight_grads(X, L, Wg, Wu, Wd, dY, k, e, mx=mx)
            assert np.allclose(dwg, g["dWg"][e], rtol=1e-12, atol=1e-12)
            assert np.allclose(dwu, g["dWu"][e], rtol=1e-12, atol=1e-12)
            assert np.allclose(dwd, g["dWd"][e], rtol=1e-12, atol=1e-12)


def test_bf16_round_matches_torch_and_ties():
    import torch
    rng = np.random.default_rng(4)
    v = np.concatenate([rng.standard_normal(20000) * np.exp2(rng.integers(-60, 60, 20000)),
                        [0.0, -0.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 65504.0]])
    want = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).double().numpy()
    assert np.array_equal(moe_ref.bf16_round(v), want)
    # ties go to the even significand: 1 + 2^-8 -> 1, 1 + 3 * 2^-8 -> 1 + 2^-6
    assert moe_ref.bf16_round(1.0 + 2.0 ** -8) == 1.0
    assert moe_ref.bf16_round(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6


def test_stored_context_sampled_form_matches_full_form():
    T, d, F, E, k = 24, 64, 64, 5, 2
    X, L, Wg, Wu, Wd, dY = _inputs(T, d, F, E, k, seed=8, alpha=0.5)
    for mx in (False, "mxfp8", "nvfp4"):
        Y, ctx = moe_ref.forward(X, L, Wg, Wu, Wd, k, mx=mx)
        st = moe_ref.stored_context(ctx)
        assert np.array_equal(st["a"], moe_ref.bf16_round(ctx["a"])) and not np.array_equal(st["a"], ctx["a"])
        g = moe_ref.backward(dY, X, L, Wg, Wu, Wd, st)
        toks = np.array([1, 9, 23])
        s = moe_ref.forward_backward_tokens(X, L, Wg, Wu, Wd, dY, k, toks, mx=mx, stored=True)
        for key, full in (("Y", Y), ("dX", g["dX"]), ("dg", g["dg"]), ("dlogits", g["dlogits"])):
            assert np.allclose(s[key], full[toks], rtol=1e-12, atol=1e-12), (mx, key)
        e = int(np.argmax(ctx["layout"]["counts"]))
        dwg, dwu, dwd = moe_ref.expert_weight_grads(X, L, Wg, Wu, Wd, dY, k, e, mx=mx, stored=True)
        for name, got in (("dWg", dwg), ("dWu", dwu), ("dWd", dwd)):
            assert np.allclose(got, g[name][e], rtol=1e-12, atol=1e-12), (mx, name)


def test_weight_gradient_quantisation_axis_hand_pins():
    """The block-scaled weight gradients quantise every operand along the
    expert's rows (the tokens), and dA, dB, w h from their bf16 values.  The
    expected sums below are worked out by hand from the formats' definitions
    (OCP MX: E8M0 scale 2^(floor(log2 amax) - 8) for E4M3, round to nearest
    even; NVFP4: E4M3 scale of amax / 6, E2M1 elements {0, 0.5, 1, 1.5, 2, 3,
    4, 6}), not from the oracle's code; quantising along the features, or
    skipping the bf16 step, gives different numbers."""
    # MXFP8, one 32-row block.  dy column 0: 448 then 31 x 2^-10.  Along the
    # rows amax = 448 = 1.75 * 2^8 sets scale 2^0, and 2^-10 is exactly half of
    # E4M3's smallest subnormal 2^-9: the tie goes to the even code, 0.  Column
    # 1 (32 x 2^-10) has scale 2^-18 and is exact.  Along the features each of
    # rows 1..31 would keep its 2^-10 (column 0 would sum to 448 + 31 * 2^-10).
    n = 32
    dy = np.full((n, 2), 2.0 ** -10)
    dy[0, 0] = 448.0
    ones = np.ones((n, 1))
    # da column 0: 448, then 1.0625 + 2^-12, then zeros.  bf16 rounds
    # 1.0625 + 2^-12 to 1.0625 (its spacing at 1 is 2^-7), the E4M3 midpoint
    # of 1 and 1.125, which ties to the even code, 1.0; without the bf16 step
    # the value lies above the midpoint and becomes 1.125.
    da = np.zeros((n, 1))
    da[0, 0] = 448.0
    da[1, 0] = 1.0625 + 2.0 ** -12
    dWd, dWg, dWu = moe_ref._weight_grads(dy, ones, ones, da, da, "mxfp8")
    assert dWd.shape == (2, 1) and dWg.shape == (1, 1)
    assert dWd[0, 0] == 448.0
    assert dWd[1, 0] == 32 * 2.0 ** -10
    assert dWg[0, 0] == 449.0 and dWu[0, 0] == 449.0
    # w h takes the same bf16 step (dy = ones)
    dWd2, _, _ = moe_ref._weight_grads(ones, ones, da, da, da, "mxfp8")
    assert dWd2[0, 0] == 449.0
    # NVFP4 (activations: tensor scale 1), one 16-row block.  Column 0: 6, then
    # 15 x 0.25: the scale is E4M3(6 / 6) = 1, and 0.25 is the midpoint of the
    # E2M1 codes 0 and 0.5, so it ties to 0.  Column 1 (16 x 0.25): amax / 6 =
    # 0.041666... lies between the E4M3 values 1.25 * 2^-5 and 1.375 * 2^-5 and
    # rounds to the nearer, 0.04296875; 0.25 / 0.04296875 = 5.818... rounds to
    # the code 6, so each row dequantises to 6 * 0.04296875 = 0.2578125.
    # The other operand is 16 x 6, exact with scale E4M3(6 / 6) = 1 (a column
    # of ones is not: its scale E4M3(1 / 6) = 0.171875 makes each 1 read
    # 6 * 0.171875 = 1.03125).
    m = 16
    dy4 = np.full((m, 2), 0.25)
    dy4[0, 0] = 6.0
    six = np.full((m, 1), 6.0)
    dWd4, _, _ = moe_ref._weight_grads(dy4, six, six, six, six, "nvfp4")
    assert dWd4[0, 0] == 6.0 * 6.0
    assert dWd4[1, 0] == 16 * 0.2578125 * 6.0
