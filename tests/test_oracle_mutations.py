"""The pins catch plausible mistakes: each case plants one mistake in the
oracle (on the CPU, through monkeypatch) and checks that a pin test fails."""

import math
import os

import numpy as np
import pytest

import oracle.attention as A
import oracle.rope as R
from tests import test_oracle_attention as TA
from tests import test_oracle_rope as TR


def _rotate_wrong_sign(x, positions, theta):
    return R.__dict__["_orig_rotate"](x, positions, -np.asarray(theta))


def _rotate_interleaved(x, positions, theta):
    x = np.asarray(x, dtype=np.float64)
    phi = np.asarray(positions, dtype=np.float64)[:, None] * np.asarray(theta)[None, :]
    c, s = np.cos(phi), np.sin(phi)
    a, b = x[..., 0::2], x[..., 1::2]
    y = np.empty_like(x)
    y[..., 0::2] = a * c - b * s
    y[..., 1::2] = a * s + b * c
    return y


def _visible_window_off_by_one(m, n, mask, sink=0, window=0):
    m, n = np.asarray(m), np.asarray(n)
    if mask == "sink_window":
        return (n <= m) & ((n < sink) | (m - n <= window))
    return R.__dict__["_orig_visible"](m, n, mask, sink, window)


def _ntk_wrong_exponent(b, s, d):
    return float(b) * float(s) ** (d / (d - 1.0))


def _mscale_missing_square(kind, s, d, override=0.0):
    if override > 0:
        return override
    return R.mscale(kind, s) / math.sqrt(d)


def _yarn_blend_reversed(kind, d, b, L_train=0.0, L_target=0.0, s=0.0, alpha=1.0, beta=32.0):
    th, cls, ms = R.__dict__["_orig_inv_freq"](kind, d, b, L_train, L_target, s, alpha, beta)
    if kind == "yarn":
        s_ = R.resolve_scale(L_train, L_target, s)
        g = R.ramp_gamma(float(L_train) / R.wavelength(d, b), alpha, beta)
        base = R.base_frequencies(d, b)
        th = g * base / s_ + (1 - g) * base
    return th, cls, ms


def _decode_ring_misindexed(j, sink, window, ring_start):
    j = np.asarray(j)
    return np.where(j < sink, j, sink + (ring_start + j) % max(window, 1))


@pytest.fixture(autouse=True)
def _keep_originals():
    R._orig_rotate = R.rotate
    R._orig_visible = A.visible
    R._orig_inv_freq = R.inv_freq
    yield


def _fails(fn, *args, **kw):
    try:
        fn(*args, **kw)
    except (AssertionError, ValueError):
        return True
    return False


def test_wrong_rotation_sign_is_caught(monkeypatch):
    monkeypatch.setattr(R, "rotate", _rotate_wrong_sign)
    assert _fails(TR.test_rotation_matches_complex_multiplication)


def test_interleaved_pairing_is_caught(monkeypatch):
    monkeypatch.setattr(R, "rotate", _rotate_interleaved)
    assert _fails(TR.test_rotation_direction_on_unit_vector)


def test_window_off_by_one_is_caught(monkeypatch):
    monkeypatch.setattr(A, "visible", _visible_window_off_by_one)
    assert _fails(TA.test_count_probe, "sink_window", 4, 7)


def test_ntk_exponent_is_caught(monkeypatch):
    monkeypatch.setattr(R, "ntk_base", _ntk_wrong_exponent)
    assert _fails(TR.test_ntk_base_by_root_finding, 128, 1e4, 4096, 8.0)


def test_missing_temperature_square_is_caught(monkeypatch):
    monkeypatch.setattr(A, "softmax_scale", _mscale_missing_square)
    assert _fails(TA.test_softmax_scale_reading)


def test_reversed_yarn_blend_is_caught(monkeypatch):
    monkeypatch.setattr(R, "inv_freq", _yarn_blend_reversed)
    assert _fails(TR.test_yarn_regimes, 128, 1e4, 4096, 4.0)


def test_ring_slot_misindex_is_caught(monkeypatch):
    monkeypatch.setattr(A, "decode_logical_to_physical", _decode_ring_misindexed)
    assert _fails(TA.test_decode_against_streaming_simulation, 23, 4, 6)


# --- the backward, the merge of partials and FP8 decoding -------------------

import oracle.quant as Q  # noqa: E402
from tests import test_oracle_quant as TQ  # noqa: E402


def _backward_without_inverse_rotation(q, k, v, do, q_pos, k_pos, theta, scale, mask, sink=0, window=0):
    # forgets R^T: the gradients of the rotated q and k are returned as they are
    dq, dk, dv = A.__dict__["_orig_backward"](q, k, v, do, q_pos, k_pos, theta, scale, mask, sink, window)
    return R.rotate(dq, q_pos, theta), R.rotate(dk, k_pos, theta), dv


def _backward_without_scale(q, k, v, do, q_pos, k_pos, theta, scale, mask, sink=0, window=0):
    # forgets the softmax scale in dq and dk
    dq, dk, dv = A.__dict__["_orig_backward"](q, k, v, do, q_pos, k_pos, theta, scale, mask, sink, window)
    return dq / scale, dk / scale, dv


def _backward_without_rowsum_term(q, k, v, do, q_pos, k_pos, theta, scale, mask, sink=0, window=0):
    # dS = P * dP, the D = rowsum(dO * O) term dropped
    qr, kr = R.rotate(np.asarray(q, float), q_pos, theta), R.rotate(np.asarray(k, float), k_pos, theta)
    logits = np.where(A.visible(np.asarray(q_pos)[:, None], np.asarray(k_pos)[None, :], mask, sink, window),
                      scale * (qr @ kr.T), -np.inf)
    p = np.exp(logits - logits.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    ds = p * (np.asarray(do, float) @ np.asarray(v, float).T)
    dq = R.rotate(scale * (ds @ kr), q_pos, -np.asarray(theta))
    dk = R.rotate(scale * (ds.T @ qr), k_pos, -np.asarray(theta))
    return dq, dk, p.T @ np.asarray(do, float)


def _merge_weights_swapped(parts):
    # two partials, each weighted by the other's share of the total
    (oa, la), (ob, _) = parts
    _, lse = A.__dict__["_orig_merge"](parts)
    with np.errstate(invalid="ignore"):
        wa = np.nan_to_num(np.exp(np.asarray(la) - lse))[:, None]
    return (1 - wa) * np.asarray(oa) + wa * np.asarray(ob), lse


def _e4m3_bias_8(codes):
    # exponent bias 8 instead of 7: every value halved
    return Q.__dict__["_orig_e4m3"](codes) / 2.0


@pytest.fixture(autouse=True)
def _keep_more_originals():
    A._orig_backward = A.backward_head
    A._orig_merge = A.merge_partials
    Q._orig_e4m3 = Q.e4m3_to_float
    yield


def test_backward_missing_inverse_rotation_is_caught(monkeypatch):
    monkeypatch.setattr(A, "backward_head", _backward_without_inverse_rotation)
    assert _fails(TA.test_backward_matches_finite_differences, "causal", 0, 0)


def test_backward_missing_scale_is_caught(monkeypatch):
    monkeypatch.setattr(A, "backward_head", _backward_without_scale)
    assert _fails(TA.test_backward_matches_finite_differences, "causal", 0, 0)


def test_backward_dropped_rowsum_term_is_caught(monkeypatch):
    monkeypatch.setattr(A, "backward_head", _backward_without_rowsum_term)
    assert _fails(TA.test_backward_matches_finite_differences, "none", 0, 0)


def test_merge_with_swapped_weights_is_caught(monkeypatch):
    monkeypatch.setattr(A, "merge_partials", _merge_weights_swapped)
    assert _fails(TA.test_merge_partials_lse_is_logsumexp_and_empty_rows)


def test_e4m3_wrong_exponent_bias_is_caught(monkeypatch):
    monkeypatch.setattr(Q, "e4m3_to_float", _e4m3_bias_8)
    assert _fails(TQ.test_e4m3_all_codes_match_torch)


# --- the YaRN ramp interior and the base frequencies, against hand values ---

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _ramp_denominator_beta(r, alpha, beta):
    # (r - alpha) / beta instead of (r - alpha) / (beta - alpha)
    return np.clip((np.asarray(r, dtype=np.float64) - alpha) / beta, 0.0, 1.0)


def _yarn_blend_divides(kind, d, b, L_train=0.0, L_target=0.0, s=0.0, alpha=1.0, beta=32.0, dim_scale=None):
    # the blend read as theta / ((1 - gamma) s + gamma): the factor blended, not the frequency
    th, cls, ms = R.__dict__["_orig_inv_freq"](kind, d, b, L_train, L_target, s, alpha, beta, dim_scale)
    if kind == "yarn":
        s_ = R.resolve_scale(L_train, L_target, s)
        g = R.ramp_gamma(float(L_train) / R.wavelength(d, b), alpha, beta)
        th = R.base_frequencies(d, b) / ((1 - g) * s_ + g)
    return th, cls, ms


def _base_exponent_i_over_d(d, b):
    # b^(-i/d) instead of b^(-2i/d)
    i = np.arange(d // 2, dtype=np.float64)
    return np.power(float(b), -i / d)


def test_ramp_denominator_is_caught_by_hand_values(monkeypatch):
    monkeypatch.setattr(R, "ramp_gamma", _ramp_denominator_beta)
    assert _fails(TR.test_yarn_ramp_hand_values, GOLDEN)


def test_blend_of_the_factor_is_caught_by_hand_values(monkeypatch):
    monkeypatch.setattr(R, "inv_freq", _yarn_blend_divides)
    assert _fails(TR.test_yarn_ramp_hand_values, GOLDEN)


def test_base_exponent_is_caught_by_hand_values(monkeypatch):
    monkeypatch.setattr(R, "base_frequencies", _base_exponent_i_over_d)
    assert _fails(TR.test_ntk_exercise2_and_base_frequencies_hand_values, GOLDEN)
