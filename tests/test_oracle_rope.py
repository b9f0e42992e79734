"""Pins for oracle.rope: each check ties the oracle to something other than
its own formula -- a value the pages print, the complex-number form of the
rotation, an invariant the pages state, or a closed form solved independently.
"""

import json
import math
import os

import numpy as np
import pytest
from scipy.optimize import brentq

from oracle import rope

CONFIG_SHAPES = [  # (d, theta_base, L_train, s) of the five workloads
    (64, 1e4, 64, 4.0),
    (128, 1e4, 4096, 4.0),
    (128, 1e4, 4096, 32.0),
    (128, 5e5, 8192, 4.0),
]


def _complex_rotate(x, positions, theta):
    """The rotation as complex multiplication: pair (x_i, x_{i+d/2}) is the
    complex number x_i + j x_{i+d/2}, rotated by e^{j m theta_i}
    ("Context Window Scaling ...", Section 2: the position lives in the phase of
    the complex representation)."""
    h = x.shape[-1] // 2
    z = x[..., :h] + 1j * x[..., h:]
    z = z * np.exp(1j * np.outer(positions, theta))
    return np.concatenate([z.real, z.imag], axis=-1)


def test_rotation_matches_complex_multiplication():
    rng = np.random.default_rng(1)
    for d in (2, 8, 64, 128):
        x = rng.standard_normal((37, d))
        pos = rng.integers(0, 200000, 37)
        theta = rope.base_frequencies(d, 1e4)
        np.testing.assert_allclose(rope.rotate(x, pos, theta), _complex_rotate(x, pos, theta),
                                   rtol=0, atol=1e-12)


def test_rotation_direction_on_unit_vector():
    # R [1, 0]^T = [cos, sin]^T: the first column of the page's 2x2 matrix.
    d = 16
    theta = rope.base_frequencies(d, 1e4)
    for i in range(d // 2):
        e = np.zeros((1, d))
        e[0, i] = 1.0
        y = rope.rotate(e, np.array([3]), theta)[0]
        assert y[i] == pytest.approx(math.cos(3 * theta[i]), abs=1e-15)
        assert y[i + d // 2] == pytest.approx(math.sin(3 * theta[i]), abs=1e-15)
        others = np.delete(y, [i, i + d // 2])
        assert np.all(others == 0.0)  # pair (i, i + d/2) mixes with nothing else


def test_exercise1_angle(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "exercise1_angle.json")))
    d, b = g["d"], g["theta_base"]
    theta = rope.base_frequencies(d, b)
    e = np.zeros((1, d))
    e[0, g["i"]] = 1.0
    y = rope.rotate(e, np.array([g["position"]]), theta)[0]
    phase = math.atan2(y[g["i"] + d // 2], y[g["i"]])
    want = math.remainder(g["angle_rad"], 2 * math.pi)
    assert phase == pytest.approx(want, abs=1e-9)
    assert g["position"] * theta[g["i"]] == g["angle_rad"]
    assert g["L_train"] * theta[g["i"]] == g["training_max_rad"]
    assert (g["angle_rad"] <= g["training_max_rad"]) == g["within_training_range"]


def test_frequency_wavelength_consistency():
    for d, b, _, _ in CONFIG_SHAPES:
        np.testing.assert_allclose(rope.base_frequencies(d, b) * rope.wavelength(d, b),
                                   2 * math.pi, rtol=1e-14)
        th = rope.base_frequencies(d, b)
        assert th[0] == 1.0 and np.all(np.diff(th) < 0)   # fastest dimension first


@pytest.mark.parametrize("kind", ["plain", "pi", "ntk", "yarn"])
def test_norm_preserved(kind):
    rng = np.random.default_rng(2)
    x = rng.standard_normal((50, 128))
    pos = rng.integers(0, 131072, 50)
    theta, _, _ = rope.inv_freq(kind, 128, 1e4, 4096, 0, 32.0)
    y = rope.rotate(x, pos, theta)
    np.testing.assert_allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-12)


@pytest.mark.parametrize("kind", ["plain", "pi", "ntk", "yarn"])
def test_relative_position_invariance(kind):
    # <R_m q, R_n k> depends only on m - n ("Context Window Scaling ...", Section 2).
    rng = np.random.default_rng(3)
    theta, _, _ = rope.inv_freq(kind, 128, 1e4, 4096, 0, 4.0)
    q, k = rng.standard_normal((2, 128))
    for _ in range(20):
        m, n, shift = rng.integers(0, 60000, 3)
        a = rope.rotate(q[None], [m], theta)[0] @ rope.rotate(k[None], [n], theta)[0]
        b = rope.rotate(q[None], [m + shift], theta)[0] @ rope.rotate(k[None], [n + shift], theta)[0]
        assert a == pytest.approx(b, abs=1e-9)


@pytest.mark.parametrize("d,b,L,s", CONFIG_SHAPES)
def test_scale_one_reduces_to_plain(d, b, L, s):
    plain, cls, ms = rope.inv_freq("plain", d, b, L)
    for kind in ("pi", "ntk", "yarn"):
        th, cls_k, ms_k = rope.inv_freq(kind, d, b, L, 0, 1.0)
        np.testing.assert_allclose(th, plain, rtol=1e-15, atol=0)
        np.testing.assert_array_equal(cls_k, cls)
        assert ms_k == 1.0


def test_none_is_identity():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((9, 64))
    th, _, ms = rope.inv_freq("none", 64, 1e4, 64, 0, 4.0)
    np.testing.assert_array_equal(rope.rotate(x, np.arange(9) * 1000, th), x)
    assert ms == 1.0


def test_pi_worked_example(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "pi_position_example.json")))
    d = 128
    th_pi, _, _ = rope.inv_freq("pi", d, 1e4, g["L_train"], g["L_target"])
    th = rope.base_frequencies(d, 1e4)
    rng = np.random.default_rng(5)
    x = rng.standard_normal((1, d))
    np.testing.assert_allclose(rope.rotate(x, [g["position"]], th_pi),
                               rope.rotate(x, [g["interpolated_position"]], th), atol=1e-12)
    # angles stay within the trained range: max angle at L_target equals that at L_train
    assert np.all(g["L_target"] * th_pi <= g["L_train"] * th + 1e-9)


@pytest.mark.parametrize("d,b,L,s", CONFIG_SHAPES + [(128, 1e4, 4096, 8.0)])
def test_ntk_base_by_root_finding(d, b, L, s):
    """Independent solve of the NTK reading: the base b' for which the lowest
    frequency is interpolated exactly by s, found numerically."""
    h = d // 2
    target = rope.base_frequencies(d, b)[h - 1] / s
    f = lambda bb: math.log(bb) * (-2.0 * (h - 1) / d) - math.log(target)
    b_root = brentq(f, b, b * s ** 4, xtol=1e-12, rtol=1e-15)
    assert rope.ntk_base(b, s, d) == pytest.approx(b_root, rel=1e-12)
    th, _, ms = rope.inv_freq("ntk", d, b, L, 0, s)
    base = rope.base_frequencies(d, b)
    assert th[0] == base[0]                                     # highest frequency kept
    assert th[h - 1] == pytest.approx(base[h - 1] / s, rel=1e-13)  # lowest interpolated by s
    ratio = th / base
    assert np.all(np.diff(ratio) < 0)                           # low dims scaled more
    assert ms == 1.0


def _class_boundaries(d, b, L, alpha, beta):
    """Closed-form regime boundaries: r_i = L b^(-2i/d) / (2 pi) is above beta
    for i < i_kept and below alpha for i > i_interp, solving the inequality
    with logarithms."""
    i_kept = (d / 2.0) * math.log(L / (2 * math.pi * beta)) / math.log(b)
    i_interp = (d / 2.0) * math.log(L / (2 * math.pi * alpha)) / math.log(b)
    return i_kept, i_interp


@pytest.mark.parametrize("d,b,L,s", CONFIG_SHAPES)
def test_yarn_regimes(d, b, L, s):
    th, cls, ms = rope.inv_freq("yarn", d, b, L, 0, s)
    base = rope.base_frequencies(d, b)
    i_kept, i_interp = _class_boundaries(d, b, L, 1.0, 32.0)
    for i in range(d // 2):
        if i < i_kept:
            assert cls[i] == rope.CLASS_KEPT and th[i] == base[i]           # no interpolation
        elif i > i_interp:
            assert cls[i] == rope.CLASS_INTERPOLATED and th[i] == pytest.approx(base[i] / s, rel=1e-15)
        else:
            assert cls[i] == rope.CLASS_RAMP
            assert base[i] / s <= th[i] <= base[i]
    # the blend moves monotonically from kept to interpolated
    frac = (th - base / s) / (base - base / s)
    assert np.all(np.diff(frac) <= 1e-15)
    assert ms == pytest.approx(0.1 * math.log(s) + 1.0, rel=1e-15)


def test_yarn_class_counts_for_workloads():
    # counts derived by hand from the closed-form boundaries above
    want = {(64, 1e4, 64): (23, 9, 0), (128, 1e4, 4096): (18, 25, 21),
            (128, 5e5, 8192): (29, 16, 19)}
    for (d, b, L), (n_interp, n_ramp, n_kept) in want.items():
        _, cls, _ = rope.inv_freq("yarn", d, b, L, 0, 4.0)
        assert (np.sum(cls == 0), np.sum(cls == 1), np.sum(cls == 2)) == (n_interp, n_ramp, n_kept)


def test_mscale_listing(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "mscale_listing.json")))
    for s, want in g["cases"]:
        assert rope.mscale("yarn", s) == want
    for s in (2.0, 4.0, 32.0):
        assert rope.mscale("pi", s) == 1.0 and rope.mscale("ntk", s) == 1.0
    assert rope.mscale("yarn", math.e ** 5) == pytest.approx(1.5, rel=1e-15)
    vals = [rope.mscale("yarn", s) for s in (1.5, 2, 4, 8, 32)]
    assert all(a < b for a, b in zip(vals, vals[1:]))


def test_resolve_scale():
    assert rope.resolve_scale(4096, 16384, 0) == 4.0
    assert rope.resolve_scale(4096, 16384, 2.0) == 2.0
    with pytest.raises(ValueError):
        rope.resolve_scale(0, 0, 0)


# ---- per-dimension scale vector (the form LongRoPE's search produces) -------

@pytest.mark.parametrize("d,b,L,s", CONFIG_SHAPES)
def test_perdim_uniform_vector_is_pi_and_ones_is_plain(d, b, L, s):
    h = d // 2
    th_pi, _, _ = rope.inv_freq("pi", d, b, L, 0, s)
    th_v, cls, ms = rope.inv_freq("perdim", d, b, L, dim_scale=np.full(h, s))
    np.testing.assert_allclose(th_v, th_pi, rtol=1e-15, atol=0)
    th_1, _, _ = rope.inv_freq("perdim", d, b, L, dim_scale=np.ones(h))
    np.testing.assert_array_equal(th_1, rope.base_frequencies(d, b))
    assert ms == 1.0


@pytest.mark.parametrize("d,b,L,s", CONFIG_SHAPES)
def test_perdim_reproduces_yarn_with_its_equivalent_vector(d, b, L, s):
    """YaRN is one particular non-uniform vector: the factor of dimension i is
    theta_i / theta'_i = 1 / ((1 - g_i) / s + g_i), with g_i from the ramp on
    r_i = L_train / lambda_i (written out here from the definitions)."""
    h = d // 2
    i = np.arange(h)
    r = L / (2 * math.pi * b ** (2.0 * i / d))
    g = np.clip((r - 1.0) / 31.0, 0.0, 1.0)
    lam = 1.0 / ((1 - g) / s + g)
    th_v, _, _ = rope.inv_freq("perdim", d, b, L, dim_scale=lam)
    th_y, _, _ = rope.inv_freq("yarn", d, b, L, 0, s)
    np.testing.assert_allclose(th_v, th_y, rtol=1e-14)


def test_perdim_rejects_bad_vectors():
    for bad in (None, np.ones(3), np.array([1.0] * 31 + [0.0]), np.array([1.0] * 31 + [np.nan])):
        with pytest.raises((ValueError, TypeError)):
            rope.inv_freq("perdim", 64, 1e4, 64, dim_scale=bad)


def test_yarn_ramp_hand_values(golden_dir):
    """The ramp's interior against values worked by hand from the page's
    definitions (wavelength, ratio to the training window, linear ramp,
    frequency blend): every field of every row, so a wrong denominator, a
    wrong blend or a wrong exponent changes at least one of them."""
    g = json.load(open(os.path.join(golden_dir, "yarn_ramp_hand.json")))
    for case in g["cases"]:
        d, b, L, s = case["d"], case["theta_base"], case["L_train"], case["s"]
        th_p, cls, _ = rope.inv_freq("yarn", d, b, L, 0, s)
        base = rope.base_frequencies(d, b)
        lam = rope.wavelength(d, b)
        for row in case["rows"]:
            i = row["i"]
            assert base[i] == pytest.approx(row["theta"], rel=1e-13)
            assert lam[i] == pytest.approx(row["lambda"], rel=1e-13)
            assert L / lam[i] == pytest.approx(row["r"], rel=1e-13)
            gam = float(rope.ramp_gamma(L / lam[i], 1.0, 32.0))
            assert gam == pytest.approx(row["gamma"], rel=1e-12, abs=1e-15)
            assert th_p[i] == pytest.approx(row["theta_prime"], rel=1e-13)
            assert int(cls[i]) == row["class"]


def test_ntk_exercise2_and_base_frequencies_hand_values(golden_dir):
    """Exercise 2 of the NTK section (4K -> 32K, d = 128) under the adopted
    reading, and the plain frequencies b^(-2i/d) at interior i, against values
    worked by hand."""
    g = json.load(open(os.path.join(golden_dir, "ntk_exercise2_hand.json")))
    d, b = g["d"], g["theta_base"]
    s = rope.resolve_scale(g["L_train"], g["L_target"], 0.0)
    assert s == g["s"]
    assert rope.ntk_base(b, s, d) == pytest.approx(g["ntk_base"], rel=1e-14)
    th, _, _ = rope.inv_freq("ntk", d, b, g["L_train"], g["L_target"])
    for i, want in g["ntk_theta"].items():
        assert th[int(i)] == pytest.approx(want, rel=1e-13)
    base = rope.base_frequencies(d, b)
    for i, want in g["plain_theta"].items():
        assert base[int(i)] == pytest.approx(want, rel=1e-14)
