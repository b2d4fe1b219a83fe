"""Plain fp64 oracle of the fused MoE layer (TEST INFRASTRUCTURE ONLY).

What the layer computes, step by step, in the order the Mixture-of-Kittens
pages describe it: the router picks experts per token, the layout step counts
tokens per expert and places each expert's tokens contiguously, the experts
(SwiGLU FFNs) run, results return to their token, and a final weighted fusion
sums them; backward runs the same chain in reverse.

Sources (page title, section):
* kucoin page "Cursor's MoK réalise une amélioration des performances de
  2,37x sur NVIDIA GB300 NVL72", section 01 (router re-decides per step; count
  tokens per expert, then place them contiguously for a grouped GEMM;
  dispatch, combine, and two reverse steps in backward), section 02 (SwiGLU
  with fused MXFP8; pull dispatch / push combine and their reverses),
  section 03 (benchmarked layer = scheduler, routing, expert FFNs, combine,
  final weighted fusion);
* laura-martel.com blog on Mixture-of-Kittens, section "Le déterminisme est
  la partie sous-estimée" (same inputs, same result).

The pages never print the layer's formulas.  Readings used here (each one is
listed with its reason in the design notes):
* gate weights: softmax over the k selected logits (max-subtracted), which
  equals a full softmax renormalised over the top-k; weights sum to 1;
* top-k order: logit descending, ties to the lower expert id; slot j of a
  token is its j-th choice;
* layout: stable counting sort of the flat pair index t*k+j by expert;
* expert: h = silu(x Wg^T) * (x Wu^T), y = h Wd^T, no biases;
* combine: Y_t = sum_j w_tj y_tj;
* backward: ordinary calculus of the above; the router-weight gradient is
  dg_tj = <dY_t, y_tj> and dlogits is the softmax Jacobian applied to dg,
  zero on experts that were not selected.

Weights may be numpy arrays or any object whose ``[e]`` returns something
``np.asarray`` turns into float64 (the tests pass a lazy per-expert converter
for full-size layers, so one expert at a time is widened to fp64).
"""
from __future__ import annotations

import numpy as np

from . import mxfp8, nvfp4


def _expert(W, e):
    return np.asarray(W[e], dtype=np.float64)


def sigmoid(a):
    return 1.0 / (1.0 + np.exp(-a))


def silu(a):
    return a * sigmoid(a)


# ----------------------------------------------------------------------------
# 0. Router GEMM, the step before the layer: logits = X Wr^T.
# ----------------------------------------------------------------------------
def router_logits(X, Wr):
    """logits[t, e] = sum_i X[t, i] Wr[e, i], in fp64.

    The pages say the router re-decides each token's experts at every step
    (kucoin page, section 01) but print no router.  The plain reading: one
    linear map from the token to one logit per expert, weight Wr [E, d] in
    the [out, in] convention, no bias.
    """
    return np.asarray(X, dtype=np.float64) @ np.asarray(Wr, dtype=np.float64).T


def router_backward(X, Wr, dlogits):
    """Gradients of <dlogits, X Wr^T>: dX = dlogits Wr, dWr = dlogits^T X (fp64)."""
    X = np.asarray(X, dtype=np.float64)
    Wr = np.asarray(Wr, dtype=np.float64)
    G = np.asarray(dlogits, dtype=np.float64)
    return {"dX": G @ Wr, "dWr": G.T @ X}


# ----------------------------------------------------------------------------
# 1. Router: top-k experts per token and their gate weights.
# ----------------------------------------------------------------------------
def route(logits, k):
    """Top-k expert ids (logit descending, lower id on ties) and softmax-over-top-k weights.

    logits: [T, E] (fp32 values widened exactly).  Returns idx [T, k] int64,
    w [T, k] float64.
    """
    logits = np.asarray(logits, dtype=np.float64)
    if not np.all(np.isfinite(logits)):
        raise ValueError("router logits must be finite")
    T, E = logits.shape
    ids = np.broadcast_to(np.arange(E), (T, E))
    order = np.lexsort((ids, -logits), axis=-1)      # primary key -logit, then id
    idx = order[:, :k].astype(np.int64)
    sel = np.take_along_axis(logits, idx, axis=1)
    z = np.exp(sel - sel[:, :1])                      # sel[:, 0] is the row maximum
    w = z / z.sum(axis=1, keepdims=True)
    return idx, w


# ----------------------------------------------------------------------------
# 2. Layout: per-expert counts, contiguous placement, stable permutation.
# ----------------------------------------------------------------------------
def layout(idx, E):
    """Counts per expert, exclusive offsets, and the stable pair permutation.

    perm_src[r] = flat pair index (t*k + j) placed at sorted row r;
    dest[t, j]  = sorted row of pair (t, j).  Within one expert the pairs keep
    ascending flat index order.
    """
    idx = np.asarray(idx, dtype=np.int64)
    T, k = idx.shape
    flat = idx.reshape(-1)
    counts = np.bincount(flat, minlength=E).astype(np.int64)
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    perm_src = np.argsort(flat, kind="stable").astype(np.int64)
    dest = np.empty(T * k, dtype=np.int64)
    dest[perm_src] = np.arange(T * k)
    return {"counts": counts, "offsets": offsets, "perm_src": perm_src,
            "dest": dest.reshape(T, k)}


# ----------------------------------------------------------------------------
# 3. Experts and 4. combine (forward).
# ----------------------------------------------------------------------------
def _fmt(mx):
    """Quantisation recipe named by a call's ``mx`` argument: None (BF16
    arithmetic), "mxfp8" (True or "mxfp8") or "nvfp4"."""
    if mx is None or mx is False:
        return None
    if mx is True or mx == "mxfp8":
        return "mxfp8"
    if mx == "nvfp4":
        return "nvfp4"
    raise ValueError("mx must be False, True, 'mxfp8' or 'nvfp4'")


def _q(v, axis, fmt, g=1.0):
    """Dequantised image of v along axis in the recipe ``fmt`` (v itself for None).
    g is the NVFP4 tensor scale (weights); activations take 1."""
    if fmt == "mxfp8":
        return mxfp8.mx_fake_quant(v, axis)
    if fmt == "nvfp4":
        return nvfp4.nv_fake_quant(v, axis, g)
    return v


def _wscales(fmt, Wg, Wu, Wd, wscales):
    """NVFP4 tensor scales (g_gu, g_d) of the weights; (1, 1) for other recipes."""
    if fmt != "nvfp4":
        return 1.0, 1.0
    return wscales if wscales is not None else nvfp4.weight_scales(Wg, Wu, Wd)


def _segment_rows(lay, e):
    o = lay["offsets"]
    return lay["perm_src"][o[e]:o[e + 1]]


def forward(X, logits, Wg, Wu, Wd, k, mx=False, identity=False, wscales=None):
    """Layer forward.  Returns (Y [T, d] float64, ctx dict for :func:`backward`).

    mx=True (or "mxfp8") emulates the MXFP8 quantisation points: X, Wg, Wu
    along d; h along F; Wd along F (each GEMM operand along that GEMM's K).
    mx="nvfp4" emulates NVFP4 at the same points, the weights with their
    tensor scales (g_gu for Wg and Wu, g_d for Wd: ``wscales``, computed from
    the weights when None), the activations with tensor scale 1.
    identity=True replaces every expert by y = x (plumbing check).
    """
    X = np.asarray(X, dtype=np.float64)
    T, d = X.shape
    E = np.asarray(logits).shape[1]
    idx, w = route(logits, k)
    lay = layout(idx, E)
    R = T * k
    fmt = _fmt(mx)
    g_gu, g_d = (1.0, 1.0) if identity else _wscales(fmt, Wg, Wu, Wd, wscales)
    Xq = _q(X, 1, fmt)
    a_all = b_all = h_all = None
    if not identity:
        F = _expert(Wg, 0).shape[0]
        a_all = np.zeros((R, F))
        b_all = np.zeros((R, F))
        h_all = np.zeros((R, F))
    y_all = np.zeros((R, d))
    for e in range(E):
        rows = _segment_rows(lay, e)
        if rows.size == 0:
            continue
        x = Xq[rows // k]
        if identity:
            y_all[rows] = X[rows // k]
            continue
        wg, wu, wd = _expert(Wg, e), _expert(Wu, e), _expert(Wd, e)
        a = x @ _q(wg, 1, fmt, g_gu).T
        b = x @ _q(wu, 1, fmt, g_gu).T
        h = silu(a) * b
        y = _q(h, 1, fmt) @ _q(wd, 1, fmt, g_d).T
        a_all[rows], b_all[rows], h_all[rows], y_all[rows] = a, b, h, y
    Y = np.zeros((T, d))
    for j in range(k):
        Y += w[:, j:j + 1] * y_all[np.arange(T) * k + j]
    ctx = {"idx": idx, "w": w, "layout": lay, "a": a_all, "b": b_all, "h": h_all,
           "y": y_all, "k": k, "mx": fmt,
           "wscales": (g_gu, g_d)}
    return Y, ctx


def bf16_round(v):
    """Round to bfloat16 (8 significand bits), nearest even, through fp32:
    fp64 -> fp32 -> bf16, as the device rounds its fp32 values.  Finite input."""
    x = np.asarray(v, dtype=np.float32)
    b = x.view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000
    return b.astype(np.uint32).view(np.float32).astype(np.float64)


def stored_context(ctx):
    """The saved context as the layer stores it for the backward: the gate and
    up pre-activations a|b in bf16, h recomputed from them.  The backward's
    inputs are what the forward saved; the block-scaled backward decides the
    codes of dA|dB from these stored values."""
    out = dict(ctx)
    out["a"], out["b"] = bf16_round(ctx["a"]), bf16_round(ctx["b"])
    out["h"] = silu(out["a"]) * out["b"]
    return out


# ----------------------------------------------------------------------------
# 5. Backward (reverse combine, expert backward, reverse dispatch, dW, router).
# ----------------------------------------------------------------------------
def backward(dY, X, logits, Wg, Wu, Wd, ctx, sparse_dw=False):
    """Gradients of L = <dY, Y>.  Returns dict dX, dWg, dWu, dWd, dg, dlogits.

    sparse_dw=True stores the weight gradients as {expert: array} for the
    experts that received tokens (others are zero) instead of dense [E, ...]
    arrays -- storage only, for full-size layers on a sub-batch of tokens.

    MXFP8 / NVFP4 emulation (ctx["mx"]): dY along d and Wd along d for
    u = Wd^T dY; dA, dB along F and Wg, Wu along F for dX (NVFP4: the weights
    with the forward's tensor scales, activations with scale 1).  The weight
    gradients' operands (dY, w*h, dA/dB, x) are quantised along the tokens,
    i.e. along the expert's rows in sorted order, in blocks from the segment's
    first row (the last one zero-padded); dA/dB and w*h from the bf16 values
    the layer keeps of them (their codes are decided from those).
    """
    dY = np.asarray(dY, dtype=np.float64)
    X = np.asarray(X, dtype=np.float64)
    k, mx = ctx["k"], ctx["mx"]
    g_gu, g_d = ctx.get("wscales", (1.0, 1.0))
    idx, w, lay = ctx["idx"], ctx["w"], ctx["layout"]
    T, d = X.shape
    E = np.asarray(logits).shape[1]
    F = _expert(Wg, 0).shape[0]
    R = T * k
    wflat = w.reshape(-1)
    dYq = _q(dY, 1, mx)
    dX = np.zeros((T, d))
    if sparse_dw:
        dWg, dWu, dWd = {}, {}, {}
    else:
        dWg = np.zeros((E, F, d))
        dWu = np.zeros((E, F, d))
        dWd = np.zeros((E, d, F))
    dg = np.zeros(R)
    for e in range(E):
        rows = _segment_rows(lay, e)
        if rows.size == 0:
            continue
        tok = rows // k
        wg, wu, wd = _expert(Wg, e), _expert(Wu, e), _expert(Wd, e)
        a, b, h = ctx["a"][rows], ctx["b"][rows], ctx["h"][rows]
        wr = wflat[rows][:, None]
        u = dYq[tok] @ _q(wd, 0, mx, g_d)            # [m, F] = (Wd^T dY)^T, K = d
        dg[rows] = np.sum(u * h, axis=1)            # <dY, y> = <Wd^T dY, h>
        dh = wr * u
        sa = sigmoid(a)
        da = dh * b * sa * (1.0 + a * (1.0 - sa))
        db = dh * silu(a)
        dx = _q(da, 1, mx) @ _q(wg, 0, mx, g_gu) + _q(db, 1, mx) @ _q(wu, 0, mx, g_gu)
        np.add.at(dX, tok, dx)
        # weight gradients: K = the expert's tokens in sorted order
        dWd[e], dWg[e], dWu[e] = _weight_grads(dY[tok], X[tok], wr * h, da, db, mx)
    dg = dg.reshape(T, k)
    s = np.sum(w * dg, axis=1, keepdims=True)
    dsel = w * (dg - s)
    dlogits = np.zeros((T, E))
    np.put_along_axis(dlogits, idx, dsel, axis=1)
    return {"dX": dX, "dWg": dWg, "dWu": dWu, "dWd": dWd, "dg": dg, "dlogits": dlogits}


# ----------------------------------------------------------------------------
# Sampled forms for full-size layers: the same arithmetic restricted to a
# subset of tokens (per-token outputs) or of experts (per-expert dW).
# ----------------------------------------------------------------------------
def _weight_grads(dy, xs, wh, da, db, fmt):
    """(dWd, dWg, dWu) of one expert from its rows in sorted order (K = the
    rows).  Block-scaled recipes quantise every operand along the rows: dy and
    xs as given (bf16 inputs), w h, dA and dB from their bf16 values."""
    if not fmt:
        return dy.T @ wh, da.T @ xs, db.T @ xs
    qt = lambda v: _q(v, 0, fmt)
    xq = qt(xs)
    return (qt(dy).T @ qt(bf16_round(wh)), qt(bf16_round(da)).T @ xq, qt(bf16_round(db)).T @ xq)


def forward_backward_tokens(X, logits, Wg, Wu, Wd, dY, k, tokens, mx=False, wscales=None, stored=False):
    """Y, dX, dg, dlogits for the listed tokens only (BF16 arithmetic unless mx).

    Routing and every per-token quantity depend on that token alone, so this
    equals the corresponding rows of :func:`forward` / :func:`backward`
    (stored=True: of :func:`backward` on :func:`stored_context`, i.e. the
    backward reads a|b rounded to bf16).  NVFP4 takes the whole weights'
    tensor scales ``wscales`` (computed from the weights when None).
    """
    fmt = _fmt(mx)
    g_gu, g_d = _wscales(fmt, Wg, Wu, Wd, wscales)
    tokens = np.asarray(tokens, dtype=np.int64)
    logits = np.asarray(logits, dtype=np.float64)
    idx, w = route(logits[tokens], k)
    X = np.asarray(X, dtype=np.float64)[tokens]
    dY = np.asarray(dY, dtype=np.float64)[tokens]
    Xq, dYq = _q(X, 1, fmt), _q(dY, 1, fmt)
    n, d = X.shape
    E = logits.shape[1]
    Y = np.zeros((n, d))
    dX = np.zeros((n, d))
    dg = np.zeros((n, k))
    for e in np.unique(idx):
        wg, wu, wd = _expert(Wg, e), _expert(Wu, e), _expert(Wd, e)
        for i, j in zip(*np.nonzero(idx == e)):
            x = Xq[i]
            a = _q(wg, 1, fmt, g_gu) @ x
            b = _q(wu, 1, fmt, g_gu) @ x
            h = silu(a) * b
            hq = _q(h[None, :], 1, fmt)[0]       # h is quantised along F as one row
            y = _q(wd, 1, fmt, g_d) @ hq
            Y[i] += w[i, j] * y
            if stored:
                a, b = bf16_round(a), bf16_round(b)
                h = silu(a) * b
            u = _q(wd, 0, fmt, g_d).T @ dYq[i]
            dg[i, j] = u @ h
            dh = w[i, j] * u
            sa = sigmoid(a)
            da = dh * b * sa * (1.0 + a * (1.0 - sa))
            db = dh * silu(a)
            da, db = _q(da[None], 1, fmt)[0], _q(db[None], 1, fmt)[0]
            dX[i] += _q(wg, 0, fmt, g_gu).T @ da + _q(wu, 0, fmt, g_gu).T @ db
    s = np.sum(w * dg, axis=1, keepdims=True)
    dlogits = np.zeros((n, E))
    np.put_along_axis(dlogits, idx, w * (dg - s), axis=1)
    return {"Y": Y, "dX": dX, "dg": dg, "dlogits": dlogits, "idx": idx, "w": w}


def expert_weight_grads(X, logits, Wg, Wu, Wd, dY, k, e, mx=False, wscales=None, stored=False):
    """dWg[e], dWu[e], dWd[e] over every token routed to expert e (sorted order);
    stored=True: from a|b as the saved context stores them (bf16)."""
    fmt = _fmt(mx)
    g_gu, g_d = _wscales(fmt, Wg, Wu, Wd, wscales)
    idx, w = route(logits, k)
    E = np.asarray(logits).shape[1]
    lay = layout(idx, E)
    rows = _segment_rows(lay, e)
    wg, wu, wd = _expert(Wg, e), _expert(Wu, e), _expert(Wd, e)
    F, d = wg.shape
    if rows.size == 0:
        return np.zeros((F, d)), np.zeros((F, d)), np.zeros((d, F))
    tok = rows // k
    X = np.asarray(X, dtype=np.float64)[tok]
    dY = np.asarray(dY, dtype=np.float64)[tok]
    wr = w.reshape(-1)[rows][:, None]
    Xq, dYq = _q(X, 1, fmt), _q(dY, 1, fmt)
    a = Xq @ _q(wg, 1, fmt, g_gu).T
    b = Xq @ _q(wu, 1, fmt, g_gu).T
    if stored:
        a, b = bf16_round(a), bf16_round(b)
    h = silu(a) * b
    u = dYq @ _q(wd, 0, fmt, g_d)
    dh = wr * u
    sa = sigmoid(a)
    da = dh * b * sa * (1.0 + a * (1.0 - sa))
    db = dh * silu(a)
    dWd, dWg, dWu = _weight_grads(dY, X, wr * h, da, db, fmt)
    return dWg, dWu, dWd


# ----------------------------------------------------------------------------
# Minibatch floor (host heuristic), restated for the oracle's own pins.
# ----------------------------------------------------------------------------
def minibatch_floor(num_sms, tile_m, tile_n, n_out, waves=2):
    """Smallest minibatch (rows) whose grouped GEMM covers `waves` full waves.

    One wave gives every SM one tile; a minibatch of m rows yields
    (m / tile_m) * (n_out / tile_n) tiles, so m >= waves * S * tile_m * tile_n / n_out.
    (fluidifia page "Cursor ouvre MoK, un mégakernel qui accélère
    l'entraînement MoE", section "Comment MoK tente de gratter des
    millisecondes partout"; kucoin page, section 02.)
    """
    return waves * num_sms * tile_m * tile_n // n_out
