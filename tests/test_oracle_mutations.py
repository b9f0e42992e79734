"""The pins catch plausible mistakes: each case plants one mistake in the
oracle (on the CPU, through monkeypatch) and checks that a pin test fails."""

import math

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
