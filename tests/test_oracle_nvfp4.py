"""Pins for the oracle's NVFP4 codec (E2M1 elements, E4M3 block scale per 16,
fp32 tensor scale) and for the layer oracle's NVFP4 quantisation points.

Independent checks: hand-derived examples (tests/golden), an exhaustive
comparison of the element path over every bf16 bit pattern against a
nearest-value table search, round trips over all 16 codes, the scale rule's
range invariant and error bound, exact power-of-two scaling of the tensor
scale, and a layer whose inputs are exactly representable, where only the
re-quantised intermediates (h, dA, dB) may change the result.
"""
import os

import numpy as np
import pytest

from oracle import moe_ref, mxfp8, nvfp4

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "nvfp4_spec_examples.txt")


def _golden_cases():
    cases = []
    with open(GOLDEN, encoding="utf-8") as fh:
        golden_lines = fh.read().splitlines(keepends=True)
    for line in golden_lines:
        if line.startswith("#") or not line.strip():
            continue
        name, g, vals, scale, elems = [f.strip() for f in line.split("|")]
        block = np.zeros(16)
        pos = 0
        for tok in [v.strip() for v in vals.split(",")]:
            if tok.startswith("fill"):
                block[pos:] = float(tok.split()[1])
                break
            block[pos] = float(tok)
            pos += 1
        expect = {}
        for pair in elems.split():
            v, c = pair.split(":")
            expect[float(v)] = int(c, 16)
        cases.append((name, float(g), block, int(scale, 16), expect))
    return cases


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c[0])
def test_hand_derived_examples(case):
    _, g, block, scale, expect = case
    codes, scales = nvfp4.nv_quantize(block[None, :], axis=1, g=g)
    assert int(scales[0, 0]) == scale, hex(int(scales[0, 0]))
    for v, c in expect.items():
        i = int(np.nonzero(block == v)[0][0])
        assert int(codes[0, i]) == c, (v, hex(int(codes[0, i])), hex(c))


def _nearest_e2m1_by_table(x):
    """Independent element path: nearest of the 15 distinct E2M1 values by
    search, ties to the even mantissa (code bit 0), saturation at 6, sign kept."""
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    a = abs(x)
    if a >= 6.0:
        m = 7
    else:
        dist = [abs(a - v) for v in mags]
        best = min(dist)
        cand = [i for i, dd in enumerate(dist) if dd == best]
        if len(cand) > 1:
            cand = [i for i in cand if i % 2 == 0]
        m = cand[0]
    return (8 if np.signbit(x) else 0) | m


def test_exhaustive_bf16_element_path():
    bits = np.arange(1 << 16, dtype=np.uint32)
    f = (bits << 16).view(np.float32)
    v = f[np.isfinite(f)].astype(np.float64)
    got = nvfp4.e2m1_encode(v)
    want = np.array([_nearest_e2m1_by_table(x) for x in v], dtype=np.uint8)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(v[i], int(got[i]), int(want[i])) for i in bad[:10]]


def test_all_codes_round_trip():
    codes = np.arange(16, dtype=np.uint8)
    vals = nvfp4.e2m1_decode(codes)
    assert np.array_equal(nvfp4.e2m1_encode(vals), codes)      # -0.0 (code 8) included
    assert vals[7] == 6.0 and vals[15] == -6.0 and vals[1] == 0.5
    assert sorted(set(np.abs(vals))) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_tensor_scale_and_top_block():
    assert nvfp4.tensor_scale(10.5) == np.float32(2.0 ** -8)
    assert nvfp4.tensor_scale(0.0) == 1.0
    rng = np.random.default_rng(3)
    for _ in range(20):
        W = (rng.standard_normal((8, 64)) * rng.uniform(1e-3, 1e2)).astype(np.float32).astype(np.float64)
        g = nvfp4.tensor_scale(np.abs(W).max())
        codes, scales = nvfp4.nv_quantize(W, axis=1, g=g)
        r, b = np.unravel_index(np.argmax(np.abs(W)), W.shape)
        assert scales[r, b // 16] == 0x7E                      # the tensor's amax block uses E4M3's top value
        assert (codes[r, b] & 7) == 7                          # and its amax element E2M1's top value


def test_scale_rule_range_and_error_bound():
    rng = np.random.default_rng(0)
    v = rng.standard_normal((64, 16 * 8)) * np.exp2(rng.integers(-4, 8, (64, 1)))
    v = v.astype(np.float32).astype(np.float64)
    g = 1.0
    codes, scales = nvfp4.nv_quantize(v, axis=1, g=g)
    s = mxfp8.e4m3_decode(scales)
    amax = np.abs(v).reshape(64, 8, 16).max(axis=2)
    normal = (s >= 2.0 ** -6) & (s < 448)
    ratio = amax[normal] / s[normal]
    assert np.all((ratio >= 6 / (1 + 2 ** -4) * (1 - 1e-6)) & (ratio <= 6 / (1 - 2 ** -4) * (1 + 1e-6)))
    dq = nvfp4.nv_dequantize(codes, scales, axis=1, g=g)
    sc = np.repeat(s, 16, axis=1)
    x = np.abs(v) / sc
    quantum = np.where(x < 2, 0.5, np.where(x < 4, 1.0, 2.0))
    sat = x > 6
    err = np.abs(dq - v)
    assert np.all(err[~sat] <= 0.5 * quantum[~sat] * sc[~sat] * (1 + 1e-6) + 1e-6 * np.abs(v[~sat]))
    assert np.all(np.abs(dq[sat]) == 6 * sc[sat])


def test_tensor_scale_commutes_with_powers_of_two():
    rng = np.random.default_rng(5)
    v = (rng.standard_normal((16, 64)) * 0.02).astype(np.float32).astype(np.float64)
    g = nvfp4.tensor_scale(np.abs(v).max())
    c0, s0 = nvfp4.nv_quantize(v, axis=1, g=g)
    for j in (-6, -1, 1, 7):
        c1, s1 = nvfp4.nv_quantize(v * 2.0 ** j, axis=1, g=np.float32(g * 2.0 ** j))
        assert np.array_equal(c0, c1) and np.array_equal(s0, s1), j
    # the tensor scale changes codes when it is not a power-of-two multiple
    c2, s2 = nvfp4.nv_quantize(v, axis=1, g=np.float32(g * 1.3))
    assert not np.array_equal(s0, s2)


def test_axis_packing_and_padding():
    rng = np.random.default_rng(1)
    v = rng.standard_normal((32, 48))
    c0, s0 = nvfp4.nv_quantize(v, axis=0)
    c1, s1 = nvfp4.nv_quantize(v.T.copy(), axis=1)
    assert np.array_equal(c0, c1.T) and np.array_equal(s0, s1.T)
    assert nvfp4.nv_pack(np.array([[1, 2, 15, 8]], dtype=np.uint8)).tolist() == [[0x21, 0x8F]]
    assert np.array_equal(nvfp4.nv_unpack(nvfp4.nv_pack(c1)), c1)
    fq = nvfp4.nv_fake_quant(v[:, :40], axis=1)                # padded to 48 inside
    assert fq.shape == (32, 40)
    assert np.array_equal(fq, nvfp4.nv_fake_quant(np.pad(v[:, :40], ((0, 0), (0, 8))), axis=1)[:, :40])


def _nv_exact(shape, rng, g, top):
    """Values exactly representable in NVFP4 along the last axis with tensor
    scale g: each 16-block is e2m1 * s * g for one E4M3 scale s, and holds a
    +-6 (so the block's scale is exactly s).  `top` forces s = 448 in the first
    block (the tensor's amax is then 2688 g, which makes g its tensor scale)."""
    mags = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    n = shape[-1] // 16
    blocks = mags[rng.integers(0, 8, shape[:-1] + (n, 16))] * rng.choice([-1.0, 1.0], shape[:-1] + (n, 16))
    blocks[..., 0] = 6.0 * rng.choice([-1.0, 1.0], shape[:-1] + (n,))
    s_codes = rng.integers(0x30, 0x58, shape[:-1] + (n,))       # E4M3 scales 0.5 .. 6.5 (below 448)
    s = mxfp8.e4m3_decode(s_codes)
    if top:
        s.reshape(-1)[0] = 448.0
    return (blocks * s[..., None] * g).reshape(shape)


def test_nvfp4_exact_inputs_only_intermediates_add_error():
    rng = np.random.default_rng(11)
    T, d, F, E, k = 32, 64, 64, 4, 2
    g_gu, g_d = 2.0 ** -12, 2.0 ** -11
    X = _nv_exact((T, d), rng, 1.0, False)
    dY = _nv_exact((T, d), rng, 1.0, False)
    Wg = _nv_exact((E, F, d), rng, g_gu, True)
    Wu = _nv_exact((E, F, d), rng, g_gu, False)
    Wd = _nv_exact((E, d, F), rng, g_d, True)
    L = rng.standard_normal((T, E))
    assert nvfp4.weight_scales(Wg, Wu, Wd) == (np.float32(g_gu), np.float32(g_d))
    for a, g in ((X, 1.0), (dY, 1.0), (Wg[0], g_gu), (Wd[1], g_d)):
        assert np.array_equal(nvfp4.nv_fake_quant(a, -1, g), a)
    Y0, c0 = moe_ref.forward(X, L, Wg, Wu, Wd, k)
    Y1, c1 = moe_ref.forward(X, L, Wg, Wu, Wd, k, mx="nvfp4")
    # a and b come from exact operands: identical
    assert np.array_equal(c0["a"], c1["a"]) and np.array_equal(c0["b"], c1["b"])
    # y differs only through h's quantisation along F (tensor scale 1)
    hq = nvfp4.nv_fake_quant(c0["h"], 1)
    y_expect = np.zeros_like(c0["y"])
    lay = c0["layout"]
    for e in range(E):
        rows = lay["perm_src"][lay["offsets"][e]:lay["offsets"][e + 1]]
        y_expect[rows] = hq[rows] @ Wd[e].T
    assert np.abs(c1["y"] - y_expect).max() <= 1e-12 * np.abs(y_expect).max()
    rel = np.abs(Y1 - Y0).max() / np.abs(Y0).max()
    assert 0 < rel < 0.25
    # backward: the weights' other orientation is not exact, so compare with
    # an explicit emulation: dY (exact), dA/dB and the re-oriented weights are
    # quantised for dX; dg uses the unquantised u and h; the weight gradients
    # quantise their operands along the tokens (below)
    g0 = moe_ref.backward(dY, X, L, Wg, Wu, Wd, c0)
    g1 = moe_ref.backward(dY, X, L, Wg, Wu, Wd, c1)
    dX = np.zeros_like(X)
    for e in range(E):
        rows = lay["perm_src"][lay["offsets"][e]:lay["offsets"][e + 1]]
        tok = rows // k
        u = dY[tok] @ nvfp4.nv_fake_quant(Wd[e], 0, g_d)
        wr = c0["w"].reshape(-1)[rows][:, None]
        a, b = c0["a"][rows], c0["b"][rows]
        sa = moe_ref.sigmoid(a)
        da = wr * u * b * sa * (1 + a * (1 - sa))
        db = wr * u * moe_ref.silu(a)
        dx = (nvfp4.nv_fake_quant(da, 1) @ nvfp4.nv_fake_quant(Wg[e], 0, g_gu)
              + nvfp4.nv_fake_quant(db, 1) @ nvfp4.nv_fake_quant(Wu[e], 0, g_gu))
        np.add.at(dX, tok, dx)
        assert np.allclose(g1["dg"].reshape(-1)[rows], np.sum(u * c0["h"][rows], axis=1), rtol=1e-12, atol=1e-12)
        # weight gradients: every operand quantised along the expert's tokens
        # (tensor scale 1), dA, dB and w*h from their bf16 values
        qt = lambda v: nvfp4.nv_fake_quant(v, 0)
        xq = qt(X[tok])
        assert np.allclose(g1["dWg"][e], qt(moe_ref.bf16_round(da)).T @ xq, rtol=1e-12, atol=1e-12)
        assert np.allclose(g1["dWu"][e], qt(moe_ref.bf16_round(db)).T @ xq, rtol=1e-12, atol=1e-12)
        assert np.allclose(g1["dWd"][e], qt(dY[tok]).T @ qt(moe_ref.bf16_round(wr * c0["h"][rows])),
                           rtol=1e-12, atol=1e-12)
    assert np.abs(g1["dX"] - dX).max() <= 1e-12 * np.abs(dX).max()
    assert not np.array_equal(g1["dWd"], g0["dWd"])


def test_nvfp4_sampled_forms_equal_full_forms():
    rng = np.random.default_rng(2)
    T, d, F, E, k = 24, 64, 32, 5, 2
    X = rng.standard_normal((T, d))
    L = rng.standard_normal((T, E))
    Wg = rng.standard_normal((E, F, d)) / 8
    Wu = rng.standard_normal((E, F, d)) / 8
    Wd = rng.standard_normal((E, d, F)) / 6
    dY = rng.standard_normal((T, d))
    Y, ctx = moe_ref.forward(X, L, Wg, Wu, Wd, k, mx="nvfp4")
    g = moe_ref.backward(dY, X, L, Wg, Wu, Wd, ctx)
    toks = np.array([0, 7, 23])
    s = moe_ref.forward_backward_tokens(X, L, Wg, Wu, Wd, dY, k, toks, mx="nvfp4")
    for key, full in (("Y", Y), ("dX", g["dX"]), ("dg", g["dg"]), ("dlogits", g["dlogits"])):
        assert np.allclose(s[key], full[toks], rtol=1e-12, atol=1e-12), key
    e = int(np.argmax(ctx["layout"]["counts"]))
    dwg, dwu, dwd = moe_ref.expert_weight_grads(X, L, Wg, Wu, Wd, dY, k, e, mx="nvfp4")
    assert np.allclose(dwg, g["dWg"][e], rtol=1e-12, atol=1e-12)
    assert np.allclose(dwd, g["dWd"][e], rtol=1e-12, atol=1e-12)
    # NVFP4 noise against the unquantised layer: present, and bounded
    Yb, _ = moe_ref.forward(X, L, Wg, Wu, Wd, k)
    rel = np.abs(Y - Yb).max() / np.abs(Yb).max()
    assert 0.01 < rel < 0.4, rel
