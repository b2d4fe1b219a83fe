"""Pins for the oracle's router (top-k + softmax weights) and layout (histogram,
offsets, stable permutation).  Independent checks: brute force over all
k-subsets, hand-written tie cases, SciPy's softmax, and pure-Python loops for
the stable counting sort."""
import itertools
import os

import numpy as np
import pytest
import scipy.special

from oracle import moe_ref

GOLDEN_FLOOR = os.path.join(os.path.dirname(__file__), "golden", "minibatch_floor.txt")


def test_topk_brute_force_subsets():
    rng = np.random.default_rng(0)
    T, E, k = 40, 7, 3
    logits = rng.standard_normal((T, E)).astype(np.float32).astype(np.float64)
    idx, w = moe_ref.route(logits, k)
    for t in range(T):
        best = max(itertools.combinations(range(E), k), key=lambda s: sum(logits[t, list(s)]))
        assert set(idx[t]) == set(best)
        assert list(idx[t]) == sorted(best, key=lambda e: -logits[t, e])


def test_ties_go_to_lower_id():
    logits = np.array([[1.0, 3.0, 3.0, 0.0, 3.0],
                       [2.0, 2.0, 2.0, 2.0, 2.0],
                       [0.0, -1.0, 5.0, 5.0, -1.0]])
    idx, w = moe_ref.route(logits, 2)
    assert idx.tolist() == [[1, 2], [0, 1], [2, 3]]
    assert np.allclose(w, 0.5, rtol=0, atol=0)
    idx3, w3 = moe_ref.route(logits, 5)
    assert idx3[1].tolist() == [0, 1, 2, 3, 4]
    assert np.all(w3[1] == 0.2)


def test_weights_softmax_over_selected():
    rng = np.random.default_rng(2)
    logits = rng.standard_normal((100, 16)) * 3
    for k in (1, 2, 4, 8):
        idx, w = moe_ref.route(logits, k)
        assert np.all(np.abs(w.sum(1) - 1.0) <= 1e-15)
        sel = np.take_along_axis(logits, idx, 1)
        assert np.allclose(w, scipy.special.softmax(sel, axis=1), rtol=1e-14, atol=0)
        # closed form: w_i / w_j = exp(l_i - l_j)
        assert np.allclose(w[:, 0] / w[:, -1], np.exp(sel[:, 0] - sel[:, -1]), rtol=1e-13)
        # equals a full softmax renormalised over the selected experts
        full = scipy.special.softmax(logits, axis=1)
        fs = np.take_along_axis(full, idx, 1)
        assert np.allclose(w, fs / fs.sum(1, keepdims=True), rtol=1e-13)
        if k == 1:
            assert np.all(w == 1.0)


def test_nonfinite_rejected():
    with pytest.raises(ValueError):
        moe_ref.route(np.array([[0.0, np.inf]]), 1)


def _brute_layout(idx, E):
    T, k = idx.shape
    flat = [int(v) for v in idx.reshape(-1)]
    counts = [sum(1 for v in flat if v == e) for e in range(E)]
    perm = []
    for e in range(E):
        for p in range(len(flat)):
            if flat[p] == e:
                perm.append(p)
    return counts, perm


@pytest.mark.parametrize("alpha,T,E,k", [(0.0, 50, 8, 2), (1.5, 64, 16, 4), (3.0, 33, 5, 5), (0.0, 1, 4, 1)])
def test_layout_matches_brute_force(alpha, T, E, k):
    rng = np.random.default_rng(3)
    bias = -alpha * np.log(rng.permutation(E) + 1.0)
    logits = rng.standard_normal((T, E)) + bias
    idx, _ = moe_ref.route(logits, k)
    lay = moe_ref.layout(idx, E)
    counts, perm = _brute_layout(idx, E)
    assert lay["counts"].tolist() == counts
    assert lay["perm_src"].tolist() == perm
    R = T * k
    assert lay["counts"].sum() == R and lay["offsets"][-1] == R
    assert sorted(lay["perm_src"].tolist()) == list(range(R))          # bijection
    assert np.array_equal(lay["perm_src"][lay["dest"].reshape(-1)], np.arange(R))  # round trip
    flat = idx.reshape(-1)
    for e in range(E):
        seg = lay["perm_src"][lay["offsets"][e]:lay["offsets"][e + 1]]
        assert np.all(flat[seg] == e)                                   # contiguous
        assert np.all(np.diff(seg) > 0)                                 # stable


def test_layout_degenerate_cases():
    # every token to the same k experts; some experts empty
    T, E, k = 10, 6, 2
    logits = np.tile(np.array([0.0, 5.0, 0.0, 4.0, 0.0, 0.0]), (T, 1))
    idx, w = moe_ref.route(logits, k)
    lay = moe_ref.layout(idx, E)
    assert lay["counts"].tolist() == [0, T, 0, T, 0, 0]
    assert lay["perm_src"][:T].tolist() == list(range(0, 2 * T, 2))
    assert lay["perm_src"][T:].tolist() == list(range(1, 2 * T, 2))


def test_minibatch_floor_golden():
    with open(GOLDEN_FLOOR, encoding="utf-8") as fh:
        golden_lines = fh.read().splitlines(keepends=True)
    for line in golden_lines:
        if line.startswith("#") or not line.strip():
            continue
        hidden, ffn, waves, sms, tm, tn, expect = map(int, line.split())
        assert moe_ref.minibatch_floor(sms, tm, tn, ffn, waves) == expect
