"""Oracle: exact softmax attention, masks, blockwise online-softmax fold and
streaming decode over a sink + sliding-window cache (float64).

TEST INFRASTRUCTURE ONLY -- see the package docstring.

Attention is the plain definition softmax(Q K^T / sqrt(d_k)) V ("Context
Window Scaling ...", Section 1).  The blockwise method the pages describe is
exact ("Long-context guide", Ring attention: an exact softmax accumulated as
key blocks arrive; "Context Length Extension", Ring Attention: partial results
combined by online softmax), so the oracle for every attention output is the
full softmax over the visible keys.  The blockwise fold below exists only to
check that claim on tiny inputs.
"""

from __future__ import annotations

import math

import numpy as np

from . import rope as _rope

MASKS = ("causal", "sink_window", "none")


def visible(m, n, mask: str, sink: int = 0, window: int = 0):
    """Visibility of key position n to query position m (broadcasting).

    * ``causal``      -- n <= m.
    * ``sink_window`` -- the cache of "Context Length Extension", Sliding
      Window + Attention Sinks: the first ``sink`` tokens plus the last
      ``window`` tokens up to and including m, i.e. n <= m and (n < sink or
      m - n < window).  Positions are 0-based; the page's x_1..x_s and
      x_{t-w+1}..x_t are the same sets 1-based.
    * ``none``        -- every key.
    """
    m = np.asarray(m)
    n = np.asarray(n)
    if mask == "none":
        return np.ones(np.broadcast(m, n).shape, dtype=bool)
    causal = n <= m
    if mask == "causal":
        return causal
    if mask == "sink_window":
        return causal & ((n < sink) | (m - n < window))
    raise ValueError(f"unknown mask {mask!r}")


def softmax_scale(kind: str, s: float, d: int, override: float = 0.0) -> float:
    """Logit multiplier.  Logits are q.k / sqrt(d) ("Context Window Scaling
    ...", Section 1) divided by the YaRN temperature t, where
    sqrt(1/t) = mscale = 0.1 ln(s) + 1 (Section 3 and its listing); dividing
    by t multiplies by mscale^2.  A positive ``override`` replaces the product.
    """
    if override > 0:
        return float(override)
    return _rope.mscale(kind, s) ** 2 / math.sqrt(d)


def attention_rows(q_rows, q_pos, k, v, mask: str, sink: int, window: int, scale: float,
                   k_pos=None):
    """Exact attention for selected query rows.

    ``q_rows`` [R, d] (already rotated), ``q_pos`` [R] their positions,
    ``k``/``v`` [S, d] (k already rotated), ``k_pos`` [S] (default 0..S-1).
    Returns ``(o [R, d], lse [R])`` with lse = ln sum_n exp(logit_n) over the
    visible keys; a row with no visible key gives o = 0 and lse = -inf.
    """
    q_rows = np.asarray(q_rows, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    S = k.shape[0]
    k_pos = np.arange(S) if k_pos is None else np.asarray(k_pos)
    logits = scale * (q_rows @ k.T)                                  # [R, S]
    vis = visible(np.asarray(q_pos)[:, None], k_pos[None, :], mask, sink, window)
    logits = np.where(vis, logits, -np.inf)
    mx = logits.max(axis=1, keepdims=True)
    empty = ~np.isfinite(mx[:, 0])
    mx = np.where(np.isfinite(mx), mx, 0.0)
    p = np.exp(logits - mx)
    l = p.sum(axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        o = (p @ v) / l[:, None]
        lse = mx[:, 0] + np.log(l)
    o[empty] = 0.0
    lse[empty] = -np.inf
    return o, lse


def ring_block_order(I: int, N: int, mask: str):
    """Order in which the holder of query block I sees the N key/value blocks
    as they rotate around the ring: at step t it holds block (I - t) mod N
    ("Context Window Scaling ...", Section 5: GPU i passes KV_j to GPU i+1, so
    it next receives the block of GPU i-1).  Under a causal or sink-window
    mask, blocks with a global index above I are future tokens and are skipped
    (Section 7, FAQ 2)."""
    order = [(I - t) % N for t in range(N)]
    if mask in ("causal", "sink_window"):
        order = [j for j in order if j <= I]
    return order


def fold_blockwise(q_row, q_pos, k, v, blocks, mask, sink, window, scale, k_pos=None):
    """Online-softmax accumulation of one query row over key blocks taken in
    the given order ("Context Length Extension", Ring Attention: partial
    results combined with online softmax).  ``blocks`` is a list of index
    arrays into the key axis.  State per row: running max mx, running sum l,
    unnormalised output acc; a block with logits x updates

        mx' = max(mx, max x);  l' = l e^(mx - mx') + sum e^(x - mx');
        acc' = acc e^(mx - mx') + sum e^(x - mx') v.

    Used only to check exactness against :func:`attention_rows`."""
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    S = k.shape[0]
    k_pos = np.arange(S) if k_pos is None else np.asarray(k_pos)
    mx, l, acc = -np.inf, 0.0, np.zeros(v.shape[1])
    for idx in blocks:
        idx = np.asarray(idx)
        x = scale * (k[idx] @ np.asarray(q_row, dtype=np.float64))
        x = np.where(visible(q_pos, k_pos[idx], mask, sink, window), x, -np.inf)
        bm = x.max() if x.size else -np.inf
        new = max(mx, bm)
        if new == -np.inf:
            continue
        corr = math.exp(mx - new) if mx != -np.inf else 0.0
        p = np.exp(x - new)
        l = l * corr + p.sum()
        acc = acc * corr + p @ v[idx]
        mx = new
    if mx == -np.inf:
        return np.zeros(v.shape[1]), -np.inf
    return acc / l, mx + math.log(l)


def merge_partials(parts):
    """Combine attention partials over disjoint key sets, each ``(o [R, d],
    lse [R])`` normalised over its own keys, into the attention over their
    union: lse = ln sum_j e^(lse_j), o = sum_j e^(lse_j - lse) o_j ("Context
    Length Extension", Ring Attention: partial results are combined using
    online softmax).  Rows where every lse is -inf are empty (o = 0)."""
    lses = np.stack([np.asarray(l, dtype=np.float64) for _, l in parts])      # [J, R]
    os_ = np.stack([np.asarray(o, dtype=np.float64) for o, _ in parts])       # [J, R, d]
    mx = lses.max(axis=0)
    empty = ~np.isfinite(mx)
    mx = np.where(empty, 0.0, mx)
    w = np.exp(lses - mx[None, :])                                          # e^-inf = 0
    tot = w.sum(axis=0)
    # an empty partial (lse = -inf) has weight 0 and no defined output: it is
    # not read at all
    contrib = np.where((w > 0)[:, :, None], w[:, :, None] * os_, 0.0)
    with np.errstate(divide="ignore", invalid="ignore"):
        lse = mx + np.log(tot)
        o = contrib.sum(axis=0) / tot[:, None]
    o[empty] = 0.0
    lse[empty] = -np.inf
    return o, lse


def prefill_head(q, k, v, rows, theta, scale, mask, sink=0, window=0):
    """Reference for one (batch, head): rotate the selected query rows at
    their positions and every key at its position, then exact attention.
    ``q``/``k``/``v`` are [S, d] raw (unrotated) inputs."""
    S = k.shape[0]
    rows = np.asarray(rows)
    k_rot = _rope.rotate(k, np.arange(S), theta)
    q_rot = _rope.rotate(np.asarray(q, dtype=np.float64)[rows], rows, theta)
    return attention_rows(q_rot, rows, k_rot, v, mask, sink, window, scale)


def decode_logical_to_physical(j, sink: int, window: int, ring_start: int):
    """Cache slot holding logical entry j of a sink + window cache: the first
    ``sink`` slots are pinned sinks; the next ``window`` slots are a ring whose
    oldest entry sits at slot sink + ring_start ("Context Length Extension",
    Sliding Window + Attention Sinks: s + w entries regardless of length;
    "Long-Context Scaling", Production defaults: 4 sinks pinned)."""
    j = np.asarray(j)
    return np.where(j < sink, j, sink + (ring_start + j - sink) % max(window, 1))


def decode_head(q, k_cache, v_cache, n_valid, ring_start, sink, window, theta, scale):
    """One new query token against one head of a sink + window cache.

    ``q`` [d] raw; ``k_cache``/``v_cache`` [sink + window, d] raw (keys are
    stored unrotated).  The positions are the logical cache indices: entry j
    sits at position j and the query, the newest entry, at n_valid - 1 (the
    StreamingLLM cache is used without changing RoPE, "Context Length
    Extension", Sliding Window + Attention Sinks).  Every logical entry
    j < n_valid is visible.  Returns ``(o [d], lse)``."""
    if n_valid <= 0:
        return np.zeros(np.asarray(q).shape[-1]), -np.inf
    j = np.arange(n_valid)
    phys = decode_logical_to_physical(j, sink, window, ring_start)
    k = _rope.rotate(np.asarray(k_cache, dtype=np.float64)[phys], j, theta)
    vv = np.asarray(v_cache, dtype=np.float64)[phys]
    qr = _rope.rotate(np.asarray(q, dtype=np.float64)[None, :], np.array([n_valid - 1]), theta)
    o, lse = attention_rows(qr, np.array([n_valid - 1]), k, vv, "none", 0, 0, scale)
    return o[0], lse[0]


def backward_head(q, k, v, do, q_pos, k_pos, theta, scale, mask, sink=0, window=0):
    """Gradients of L = sum(O * dO) for one (batch, head) of
    O = softmax(scale * <R_m q_m, R_n k_n>) V over visible keys, by the chain
    rule written out (the derivative of the softmax attention the pages
    define in "Context Window Scaling ...", Section 1, with the rotation of
    Section 2 applied to q and k):

        P = softmax rows of scale * Qr Kr^T (Qr, Kr the rotated q, k)
        dV = P^T dO;  dP = dO V^T;  D_m = sum_n P_mn dP_mn (= rowsum dO * O)
        dS = P * (dP - D);  dQr = scale dS Kr;  dKr = scale dS^T Qr
        dq = R_m^T dQr,  dk = R_n^T dKr  (the rotation is orthogonal)

    ``q``, ``do`` [Sq, d]; ``k``, ``v`` [Skv, d]; positions as in
    :func:`attention_rows`.  Returns (dq, dk, dv) in float64."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    q_pos = np.asarray(q_pos)
    k_pos = np.asarray(k_pos)
    qr = _rope.rotate(q, q_pos, theta)
    kr = _rope.rotate(k, k_pos, theta)
    logits = scale * (qr @ kr.T)
    vis = visible(q_pos[:, None], k_pos[None, :], mask, sink, window)
    logits = np.where(vis, logits, -np.inf)
    mx = logits.max(axis=1, keepdims=True)
    mx = np.where(np.isfinite(mx), mx, 0.0)
    p = np.exp(logits - mx)
    tot = p.sum(axis=1, keepdims=True)
    p = np.where(tot > 0, p / np.where(tot > 0, tot, 1.0), 0.0)
    dv = p.T @ do
    dp = do @ v.T
    D = (p * dp).sum(axis=1, keepdims=True)
    ds = p * (dp - D)
    dqr = scale * (ds @ kr)
    dkr = scale * (ds.T @ qr)
    # R^T is the rotation by the negated angle
    dq = _rope.rotate(dqr, q_pos, -np.asarray(theta))
    dk = _rope.rotate(dkr, k_pos, -np.asarray(theta))
    return dq, dk, dv


def backward_sampled(q, k, v, do, pos, theta, scale, mask, q_rows, k_rows, sink=0, window=0, chunk=512):
    """The gradients of :func:`backward_head` at selected rows only, for
    sequences too long for the full S x S matrices: dq at the query rows
    ``q_rows``, and dk, dv at the key rows ``k_rows``.  It is the same chain
    rule written per row.  The forward's lse and D = rowsum(dO * O) enter
    every key row's gradient, so they are computed for all query rows (in
    chunks of ``chunk`` rows).  Then, with P_mn = exp(scale <Qr_m, Kr_n> -
    lse_m) on visible pairs and dS_mn = P_mn (<dO_m, V_n> - D_m):

        dq_m = R_m^T scale sum_n dS_mn Kr_n          (row m of dS)
        dv_n = sum_m P_mn dO_m,  dk_n = R_n^T scale sum_m dS_mn Qr_m   (column n)

    Queries and keys share the positions ``pos`` (self-attention).  Returns
    (dq [len(q_rows), d], dk [len(k_rows), d], dv [len(k_rows), d]) in
    float64."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    pos = np.asarray(pos)
    neg_theta = -np.asarray(theta)
    qr = _rope.rotate(q, pos, theta)
    kr = _rope.rotate(k, pos, theta)
    S = q.shape[0]
    lse = np.empty(S)
    D = np.empty(S)
    for c0 in range(0, S, chunk):
        rows = slice(c0, min(S, c0 + chunk))
        o, l = attention_rows(qr[rows], pos[rows], kr, v, mask, sink, window, scale)
        lse[rows] = l
        D[rows] = (o * do[rows]).sum(axis=1)

    def probs(logits, lse_rows, vis):
        ok = vis & np.isfinite(lse_rows)
        return np.where(ok, np.exp(np.where(ok, logits - np.where(ok, lse_rows, 0.0), -np.inf)), 0.0)

    qi = np.asarray(q_rows)
    vis = visible(pos[qi][:, None], pos[None, :], mask, sink, window)
    p = probs(scale * (qr[qi] @ kr.T), lse[qi][:, None], vis)            # [Rq, S]
    ds = p * (do[qi] @ v.T - D[qi][:, None])
    dq = _rope.rotate(scale * (ds @ kr), pos[qi], neg_theta)

    ki = np.asarray(k_rows)
    vis = visible(pos[:, None], pos[ki][None, :], mask, sink, window)
    p = probs(scale * (qr @ kr[ki].T), lse[:, None], vis)                # [S, Rk]
    ds = p * (do @ v[ki].T - D[:, None])
    dv = p.T @ do
    dk = _rope.rotate(scale * (ds.T @ qr), pos[ki], neg_theta)
    return dq, dk, dv
