"""Pins for the oracle's MXFP8 codec (E4M3 elements + E8M0 block scale).

Independent checks: hand-derived spec examples (tests/golden), an exhaustive
comparison over every bf16 bit pattern against a nearest-value table search,
decode/encode round trips over all finite codes, and the scale rule's range
invariant.
"""
import os

import numpy as np
import pytest
import torch

from oracle import mxfp8

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "mx_spec_examples.txt")


def _golden_cases():
    cases = []
    with open(GOLDEN, encoding="utf-8") as fh:
        golden_lines = fh.read().splitlines(keepends=True)
    for line in golden_lines:
        if line.startswith("#") or not line.strip():
            continue
        name, vals, scale, elems = [f.strip() for f in line.split("|")]
        block = np.zeros(32)
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
        cases.append((name, block, int(scale, 16), expect))
    return cases


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c[0])
def test_hand_derived_spec_examples(case):
    _, block, scale, expect = case
    codes, scales = mxfp8.mx_quantize(block[None, :], axis=1)
    assert int(scales[0, 0]) == scale
    for v, c in expect.items():
        i = int(np.nonzero(block == v)[0][0])
        assert int(codes[0, i]) == c, (v, hex(int(codes[0, i])), hex(c))


def _finite_table():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)])
    return codes, mxfp8.e4m3_decode(codes)


def _nearest_by_table(v):
    """Independent element path: nearest finite E4M3 by search; ties -> even mantissa."""
    codes, vals = _finite_table()
    out = np.empty(v.shape, dtype=np.uint8)
    for i, x in enumerate(v):
        if abs(x) >= 448.0:
            c = 0x7E if x > 0 else 0xFE
        else:
            dist = np.abs(vals - x)
            best = dist.min()
            cand = codes[dist == best]
            # same-sign candidates only (+0 / -0 both have distance |x|)
            sgn = 0x80 if np.signbit(x) else 0
            cand = [int(cc) for cc in cand if (int(cc) & 0x80) == sgn or (int(cc) & 0x7F) != 0]
            if len(cand) > 1:
                cand = [cc for cc in cand if (cc & 1) == 0] or cand
            c = cand[0]
            if (c & 0x7F) == 0:
                c = sgn
        out[i] = c
    return out


def test_exhaustive_bf16_element_path():
    bits = np.arange(1 << 16, dtype=np.uint32)
    with np.errstate(invalid="ignore"):          # the NaN patterns widen to NaN, then are dropped
        f32 = (bits << 16).view(np.float32).astype(np.float64)
    finite = np.isfinite(f32)
    v = f32[finite]
    got = mxfp8.e4m3_encode(v)
    want = _nearest_by_table(v)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(v[i], hex(got[i]), hex(want[i])) for i in bad[:10]]


def test_decode_encode_round_trip_all_finite_codes():
    codes, vals = _finite_table()
    assert np.array_equal(mxfp8.e4m3_encode(vals), codes.astype(np.uint8))
    assert vals.max() == 448.0 and vals.min() == -448.0
    # spec facts: smallest subnormal 2^-9, smallest normal 2^-6
    assert mxfp8.e4m3_decode(0x01) == 2.0 ** -9
    assert mxfp8.e4m3_decode(0x08) == 2.0 ** -6
    assert np.isnan(mxfp8.e4m3_decode(0x7F))


def test_scale_rule_range_invariant():
    rng = np.random.default_rng(0)
    v = rng.standard_normal((64, 32 * 8)) * np.exp2(rng.integers(-40, 40, (64, 1)))
    codes, scales = mxfp8.mx_quantize(v, axis=1)
    blocks = np.abs(v).reshape(64, 8, 32).max(axis=2)
    scaled = blocks / np.exp2(scales.astype(np.int64) - 127)
    assert np.all((scaled >= 256) & (scaled < 512))      # amax lands in E4M3's top binade
    dq = mxfp8.mx_dequantize(codes, scales, axis=1)
    err = np.abs(dq - v)
    # element error: half a quantum of the element's binade, or saturation at 448 * 2^X
    sc = np.repeat(np.exp2(scales.astype(np.int64) - 127), 32, axis=1)
    sat = np.abs(v) >= 448 * sc
    assert np.all(err[~sat] <= np.maximum(np.abs(v[~sat]) * 2.0 ** -4, sc[~sat] * 2.0 ** -10))
    assert np.all(np.abs(dq[sat]) == 448 * sc[sat])


def test_quantise_axis_and_padding():
    rng = np.random.default_rng(1)
    v = rng.standard_normal((64, 96))
    c0, s0 = mxfp8.mx_quantize(v, axis=0)
    c1, s1 = mxfp8.mx_quantize(v.T.copy(), axis=1)
    assert np.array_equal(c0, c1.T) and np.array_equal(s0, s1.T)
    assert s0.shape == (2, 96)
    # padding with zeros does not change any block's amax
    w = rng.standard_normal((40, 8))
    fq = mxfp8.mx_fake_quant(w, axis=0)
    full = mxfp8.mx_fake_quant(np.vstack([w, np.zeros((24, 8))]), axis=0)[:40]
    assert np.array_equal(fq, full)


def test_device_independent_of_torch_bf16_rounding():
    # values from bf16 tensors (the layer's inputs) widen exactly to fp64
    t = torch.randn(1000).to(torch.bfloat16)
    v = t.to(torch.float64).numpy()
    assert np.array_equal(v.astype(np.float32).astype(np.float64), v)
