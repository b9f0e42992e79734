"""Pins for oracle.attention: brute force on tiny inputs, library softmax,
exact count probes, the sink + window set written out as Python sets, a
token-by-token streaming-cache simulation, and block-order invariance."""

import itertools
import json
import math
import os

import numpy as np
import pytest
from scipy.special import logsumexp, softmax

from oracle import attention as A
from oracle import rope


def _visible_set(m, S, mask, sink, window):
    """The cache of the page's sliding-window-plus-sinks section, written as a
    set: {x_1..x_s} U {x_{t-w+1}..x_t} with 1-based t = m + 1."""
    if mask == "none":
        return set(range(S))
    if mask == "causal":
        return set(range(m + 1))
    t = m + 1
    sinks = set(range(1, min(sink, t) + 1))
    recent = set(range(max(1, t - window + 1), t + 1))
    return {x - 1 for x in sinks | recent}


def _brute(q, k, v, m, mask, sink, window, scale):
    vis = sorted(_visible_set(m, k.shape[0], mask, sink, window))
    logits = [scale * sum(q[c] * k[n][c] for c in range(len(q))) for n in vis]
    mx = max(logits)
    w = [math.exp(x - mx) for x in logits]
    tot = sum(w)
    o = [sum(w[a] * v[n][c] for a, n in enumerate(vis)) / tot for c in range(v.shape[1])]
    return np.array(o), mx + math.log(tot)


@pytest.mark.parametrize("mask,sink,window", [("causal", 0, 0), ("none", 0, 0),
                                              ("sink_window", 2, 3), ("sink_window", 0, 1),
                                              ("sink_window", 4, 5)])
def test_attention_rows_brute_force(mask, sink, window):
    rng = np.random.default_rng(10)
    S, d = 11, 6
    q, k, v = rng.standard_normal((3, S, d))
    scale = 0.7
    rows = np.arange(S)
    o, lse = A.attention_rows(q, rows, k, v, mask, sink, window, scale)
    for m in range(S):
        ob, lb = _brute(q[m], k, v, m, mask, sink, window, scale)
        np.testing.assert_allclose(o[m], ob, atol=1e-12)
        assert lse[m] == pytest.approx(lb, abs=1e-12)


def test_attention_rows_library_softmax():
    rng = np.random.default_rng(11)
    S, d = 40, 16
    q, k, v = rng.standard_normal((3, S, d))
    o, lse = A.attention_rows(q, np.arange(S), k, v, "none", 0, 0, 0.25)
    logits = 0.25 * q @ k.T
    np.testing.assert_allclose(o, softmax(logits, axis=1) @ v, atol=1e-12)
    np.testing.assert_allclose(lse, logsumexp(logits, axis=1), atol=1e-12)


@pytest.mark.parametrize("mask,sink,window", [("causal", 0, 0), ("sink_window", 4, 7),
                                              ("sink_window", 0, 3), ("sink_window", 3, 100)])
def test_count_probe(mask, sink, window):
    # q = 0 makes every visible logit 0: lse = ln(count), o = mean of visible v
    S, d = 30, 4
    rng = np.random.default_rng(12)
    k = rng.standard_normal((S, d))
    v = np.arange(S, dtype=np.float64)[:, None] * np.ones((1, d))
    o, lse = A.attention_rows(np.zeros((S, d)), np.arange(S), k, v, mask, sink, window, 1.0)
    for m in range(S):
        vis = _visible_set(m, S, mask, sink, window)
        assert lse[m] == pytest.approx(math.log(len(vis)), abs=1e-13)
        assert o[m, 0] == pytest.approx(sum(vis) / len(vis), abs=1e-12)


def test_causal_row0_returns_v0():
    rng = np.random.default_rng(13)
    q, k, v = rng.standard_normal((3, 8, 5))
    o, _ = A.attention_rows(q, np.arange(8), k, v, "causal", 0, 0, 3.0)
    np.testing.assert_array_equal(o[0], v[0])


def test_window_covering_sequence_equals_causal():
    rng = np.random.default_rng(14)
    S = 25
    q, k, v = rng.standard_normal((3, S, 8))
    oc, lc = A.attention_rows(q, np.arange(S), k, v, "causal", 0, 0, 0.5)
    for sink in (0, 4):
        ow, lw = A.attention_rows(q, np.arange(S), k, v, "sink_window", sink, S, 0.5)
        np.testing.assert_array_equal(ow, oc)
        np.testing.assert_array_equal(lw, lc)


def test_window_one_no_sink_returns_own_value():
    rng = np.random.default_rng(15)
    q, k, v = rng.standard_normal((3, 9, 4))
    o, lse = A.attention_rows(q, np.arange(9), k, v, "sink_window", 0, 1, 1.0)
    np.testing.assert_allclose(o, v, atol=0)
    np.testing.assert_allclose(lse, np.einsum("sd,sd->s", q, k), atol=1e-13)


def test_empty_row():
    o, lse = A.attention_rows(np.ones((1, 4)), np.array([0]), np.ones((3, 4)), np.ones((3, 4)),
                              "causal", 0, 0, 1.0, k_pos=np.array([5, 6, 7]))
    assert np.all(o == 0) and lse[0] == -np.inf


@pytest.mark.parametrize("mask,sink,window", [("causal", 0, 0), ("none", 0, 0), ("sink_window", 2, 5)])
def test_blockwise_any_order_equals_full(mask, sink, window):
    # attention is an exact sum over key blocks ("Long-context guide", Ring attention)
    rng = np.random.default_rng(16)
    S, d = 16, 8
    q, k, v = rng.standard_normal((3, S, d))
    blocks = [np.arange(j, j + 4) for j in range(0, S, 4)]
    for m in (0, 3, 7, 12, 15):
        o_full, l_full = A.attention_rows(q[m:m + 1], np.array([m]), k, v, mask, sink, window, 0.8)
        for perm in itertools.permutations(range(4)):
            o, l = A.fold_blockwise(q[m], m, k, v, [blocks[p] for p in perm], mask, sink, window, 0.8)
            np.testing.assert_allclose(o, o_full[0], atol=1e-12)
            assert l == pytest.approx(l_full[0], abs=1e-12)


def test_ring_order_and_causal_block_skip():
    N = 6
    for I in range(N):
        order = A.ring_block_order(I, N, "causal")
        assert order[0] == I and sorted(order) == list(range(I + 1))  # no future block
        full = A.ring_block_order(I, N, "none")
        assert sorted(full) == list(range(N))
        assert all(full[t] == (I - t) % N for t in range(N))
    # folding in ring order reproduces full attention
    rng = np.random.default_rng(17)
    S, d, N = 24, 8, 4
    q, k, v = rng.standard_normal((3, S, d))
    bs = S // N
    for m in range(S):
        I = m // bs
        blocks = [np.arange(j * bs, (j + 1) * bs) for j in A.ring_block_order(I, N, "causal")]
        o, l = A.fold_blockwise(q[m], m, k, v, blocks, "causal", 0, 0, 0.5)
        of, lf = A.attention_rows(q[m:m + 1], np.array([m]), k, v, "causal", 0, 0, 0.5)
        np.testing.assert_allclose(o, of[0], atol=1e-12)


def _stream(tokens_k, tokens_v, sink, window):
    """Token-by-token streaming cache: pin the first `sink` tokens, keep the
    newest `window` in a ring buffer, overwrite the oldest on eviction.
    Returns (k_cache, v_cache, n_valid, ring_start, kept_token_ids)."""
    d = tokens_k.shape[1]
    kc = np.full((sink + window, d), np.nan)
    vc = np.full((sink + window, d), np.nan)
    ring_ids = []          # token ids in the ring, oldest first
    slot_of = {}
    write = 0              # next ring slot to write
    for t in range(tokens_k.shape[0]):
        if t < sink:
            kc[t], vc[t] = tokens_k[t], tokens_v[t]
            continue
        if len(ring_ids) == window:
            ring_ids.pop(0)
        slot = sink + write
        kc[slot], vc[slot] = tokens_k[t], tokens_v[t]
        slot_of[t] = write
        ring_ids.append(t)
        write = (write + 1) % window
    n_valid = min(tokens_k.shape[0], sink) + len(ring_ids)
    ring_start = slot_of[ring_ids[0]] if ring_ids else 0
    kept = list(range(min(tokens_k.shape[0], sink))) + ring_ids
    return kc, vc, n_valid, ring_start, kept


@pytest.mark.parametrize("T,sink,window", [(3, 4, 6), (4, 4, 6), (9, 4, 6), (10, 4, 6),
                                           (23, 4, 6), (40, 2, 7), (17, 0, 5)])
def test_decode_against_streaming_simulation(T, sink, window):
    rng = np.random.default_rng(20 + T)
    d = 16
    toks_k, toks_v = rng.standard_normal((2, T, d))
    q = rng.standard_normal(d)
    kc, vc, n_valid, ring_start, kept = _stream(toks_k, toks_v, sink, window)
    assert n_valid == len(kept) <= sink + window
    theta, _, _ = rope.inv_freq("plain", d, 1e4)
    scale = 1 / math.sqrt(d)
    o, lse = A.decode_head(q, kc, vc, n_valid, ring_start, sink, window, theta, scale)
    # positions are the logical cache indices 0..n_valid-1 (kept order)
    kk = rope.rotate(toks_k[kept], np.arange(n_valid), theta)
    qq = rope.rotate(q[None], [n_valid - 1], theta)[0]
    logits = scale * kk @ qq
    np.testing.assert_allclose(o, softmax(logits) @ toks_v[kept], atol=1e-12)
    assert lse == pytest.approx(logsumexp(logits), abs=1e-12)


def test_decode_ring_start_rotation_invariance():
    rng = np.random.default_rng(30)
    sink, window, d = 4, 10, 8
    kc, vc = rng.standard_normal((2, sink + window, d))
    q = rng.standard_normal(d)
    theta, _, _ = rope.inv_freq("yarn", d, 1e4, 16, 0, 4.0)
    o0, l0 = A.decode_head(q, kc, vc, sink + window, 0, sink, window, theta, 0.3)
    for shift in (1, 5, 9):
        # move ring contents so the oldest entry sits at slot sink + shift
        kc2, vc2 = kc.copy(), vc.copy()
        kc2[sink:] = np.roll(kc[sink:], shift, axis=0)
        vc2[sink:] = np.roll(vc[sink:], shift, axis=0)
        o, l = A.decode_head(q, kc2, vc2, sink + window, shift, sink, window, theta, 0.3)
        np.testing.assert_array_equal(o, o0)
        assert l == l0


def test_decode_sink_only_and_empty(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "streaming_defaults.json")))
    sink = g["sink"]
    rng = np.random.default_rng(31)
    kc, vc = rng.standard_normal((2, sink + 8, 8))
    theta, _, _ = rope.inv_freq("plain", 8, 1e4)
    for n in range(1, sink + 1):
        o, l = A.decode_head(np.zeros(8), kc, vc, n, 3, sink, 8, theta, 1.0)
        np.testing.assert_allclose(o, vc[:n].mean(axis=0), atol=1e-13)
        assert l == pytest.approx(math.log(n), abs=1e-13)
    o, l = A.decode_head(np.zeros(8), kc, vc, 0, 0, sink, 8, theta, 1.0)
    assert np.all(o == 0) and l == -np.inf


def test_softmax_scale_reading():
    assert A.softmax_scale("plain", 4.0, 128) == pytest.approx(1 / math.sqrt(128), rel=1e-15)
    assert A.softmax_scale("pi", 4.0, 128) == pytest.approx(1 / math.sqrt(128), rel=1e-15)
    ms = 0.1 * math.log(4.0) + 1
    assert A.softmax_scale("yarn", 4.0, 128) == pytest.approx(ms * ms / math.sqrt(128), rel=1e-15)
    assert A.softmax_scale("yarn", 4.0, 128, override=0.5) == 0.5
    # mscale applied to both rotated q and k reproduces the multiplier
    rng = np.random.default_rng(32)
    q, k = rng.standard_normal((2, 3, 128))
    th, _, m = rope.inv_freq("yarn", 128, 1e4, 4096, 0, 4.0)
    qa = rope.rope_apply(q, [0, 5, 9], "yarn", 128, 1e4, 4096, 0, 4.0, apply_mscale=True)
    ka = rope.rope_apply(k, [0, 5, 9], "yarn", 128, 1e4, 4096, 0, 4.0, apply_mscale=True)
    qr, kr = rope.rotate(q, [0, 5, 9], th), rope.rotate(k, [0, 5, 9], th)
    np.testing.assert_allclose((qa @ ka.T) / math.sqrt(128),
                               A.softmax_scale("yarn", 4.0, 128) * (qr @ kr.T), rtol=1e-13)


def test_prefill_head_small():
    rng = np.random.default_rng(33)
    S, d = 20, 8
    q, k, v = rng.standard_normal((3, S, d))
    theta, _, _ = rope.inv_freq("yarn", d, 1e4, 8, 0, 2.0)
    rows = np.array([0, 7, 19])
    o, lse = A.prefill_head(q, k, v, rows, theta, 0.4, "causal")
    qr = rope.rotate(q, np.arange(S), theta)
    kr = rope.rotate(k, np.arange(S), theta)
    for a, m in enumerate(rows):
        ob, lb = _brute(qr[m], kr, v, m, "causal", 0, 0, 0.4)
        np.testing.assert_allclose(o[a], ob, atol=1e-12)


@pytest.mark.parametrize("mask,sink,window", [("causal", 0, 0), ("sink_window", 2, 4), ("none", 0, 0)])
def test_merge_partials_equals_full_attention_by_brute_force(mask, sink, window):
    """Splitting the keys into blocks (any sizes, some blocks empty for some
    rows), attending per block and merging equals brute-force attention."""
    rng = np.random.default_rng(21)
    S, d = 13, 5
    q, k, v = rng.standard_normal((3, S, d))
    scale = 0.9
    rows = np.arange(S)
    edges = [0, 3, 4, 9, 13]
    parts = []
    for a, b in zip(edges[:-1], edges[1:]):
        kp = np.arange(a, b)
        parts.append(A.attention_rows(q, rows, k[a:b], v[a:b], mask, sink, window, scale, k_pos=kp))
    o, lse = A.merge_partials(parts[::-1])  # any order
    for m in range(S):
        ob, lb = _brute(q[m], k, v, m, mask, sink, window, scale)
        np.testing.assert_allclose(o[m], ob, atol=1e-12)
        assert lse[m] == pytest.approx(lb, abs=1e-12)


def test_merge_partials_lse_is_logsumexp_and_empty_rows():
    lse_a, lse_b = np.array([0.3, -np.inf, -np.inf]), np.array([-1.2, 2.0, -np.inf])
    o_a, o_b = np.ones((3, 2)), 2 * np.ones((3, 2))
    o, lse = A.merge_partials([(o_a, lse_a), (o_b, lse_b)])
    assert lse[0] == pytest.approx(logsumexp([0.3, -1.2]), abs=1e-15)
    assert lse[1] == 2.0 and np.all(o[1] == 2.0)
    assert np.isneginf(lse[2]) and np.all(o[2] == 0.0)


def test_merge_partials_ignores_the_output_of_an_empty_partial():
    o_a = np.full((2, 3), np.nan)
    o, lse = A.merge_partials([(o_a, np.array([-np.inf, -np.inf])), (np.ones((2, 3)), np.array([0.5, -np.inf]))])
    assert np.all(o[0] == 1.0) and lse[0] == 0.5
    assert np.all(o[1] == 0.0) and np.isneginf(lse[1])


@pytest.mark.parametrize("mask,sink,window", [("causal", 0, 0), ("sink_window", 1, 3), ("none", 0, 0)])
def test_backward_matches_finite_differences(mask, sink, window):
    """The hand-derived backward against central differences of the forward
    oracle's loss L = sum(O * G): independent of the chain-rule algebra."""
    rng = np.random.default_rng(31)
    S, d = 7, 6
    q, k, v, g = rng.standard_normal((4, S, d))
    theta = rope.base_frequencies(d, 100.0) / 3.0
    pos = np.arange(S)
    scale = 0.6

    def loss(q_, k_, v_):
        qr = rope.rotate(q_, pos, theta)
        kr = rope.rotate(k_, pos, theta)
        o, _ = A.attention_rows(qr, pos, kr, v_, mask, sink, window, scale)
        return float((o * g).sum())

    dq, dk, dv = A.backward_head(q, k, v, g, pos, pos, theta, scale, mask, sink, window)
    h = 1e-6
    for arr, grad, which in ((q, dq, 0), (k, dk, 1), (v, dv, 2)):
        num = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            args = [q.copy(), k.copy(), v.copy()]
            args[which][idx] += h
            up = loss(*args)
            args[which][idx] -= 2 * h
            dn = loss(*args)
            num[idx] = (up - dn) / (2 * h)
        np.testing.assert_allclose(grad, num, atol=1e-7, rtol=1e-6)


def test_backward_rows_and_blocks_are_consistent():
    """dV summed over query blocks equals dV of the whole (gradients are sums
    over query rows), and D = rowsum(dO * O)."""
    rng = np.random.default_rng(32)
    S, d = 12, 4
    q, k, v, g = rng.standard_normal((4, S, d))
    theta = rope.base_frequencies(d, 1e4)
    pos = np.arange(S)
    _, _, dv = A.backward_head(q, k, v, g, pos, pos, theta, 0.5, "causal")
    _, _, dv_a = A.backward_head(q[:5], k, v, g[:5], pos[:5], pos, theta, 0.5, "causal")
    _, _, dv_b = A.backward_head(q[5:], k, v, g[5:], pos[5:], pos, theta, 0.5, "causal")
    np.testing.assert_allclose(dv, dv_a + dv_b, atol=1e-12)


@pytest.mark.parametrize("mask,sink,window", [("causal", 0, 0), ("sink_window", 2, 9), ("none", 0, 0)])
def test_backward_sampled_rows_match_the_full_backward(mask, sink, window):
    """The row-sampled backward (used where S x S matrices do not fit) gives
    the rows of the full backward, which finite differences pin above; the
    sampled rows include the first, the last and rows split across its
    lse / D chunks."""
    rng = np.random.default_rng(33)
    S, d = 40, 8
    q, k, v, g = rng.standard_normal((4, S, d))
    theta = rope.base_frequencies(d, 1e4) / 2.0
    pos = np.arange(S)
    dq, dk, dv = A.backward_head(q, k, v, g, pos, pos, theta, 0.7, mask, sink, window)
    rows_q = np.array([0, 5, 16, 17, 39])
    rows_k = np.array([0, 1, 15, 30, 39])
    sq, sk, sv = A.backward_sampled(q, k, v, g, pos, theta, 0.7, mask, rows_q, rows_k, sink, window, chunk=16)
    np.testing.assert_allclose(sq, dq[rows_q], atol=1e-12, rtol=1e-10)
    np.testing.assert_allclose(sk, dk[rows_k], atol=1e-12, rtol=1e-10)
    np.testing.assert_allclose(sv, dv[rows_k], atol=1e-12, rtol=1e-10)
