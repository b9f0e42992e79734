"""Oracle: RoPE frequencies, context-extension rescaling and rotation (float64).

TEST INFRASTRUCTURE ONLY -- see the package docstring.  Plain definitions in
numpy float64; no code is shared with the CUDA library.

Notation follows the pages: ``d`` head dimension, ``b`` (``theta_base``) the
RoPE base, ``i`` in ``[0, d/2)`` the pair index, ``m`` a token position,
``L_train`` / ``L_target`` the trained and desired context lengths and
``s = L_target / L_train`` the scale factor ("Context Length Extension",
Notation, calls it alpha).
"""

from __future__ import annotations

import math

import numpy as np

KINDS = ("none", "plain", "pi", "ntk", "yarn", "perdim")

# Regime classes of a frequency dimension, per "Context Window Scaling ...",
# Section 3 (Decoupled Frequency Partitioning).
CLASS_INTERPOLATED = 0  # low frequency: full linear interpolation
CLASS_RAMP = 1          # mid frequency: blended by the ramp gamma(r)
CLASS_KEPT = 2          # high frequency: no interpolation


def resolve_scale(L_train: float, L_target: float, s: float) -> float:
    """Scale factor s.  A positive ``s`` is used as given; otherwise
    s = L_target / L_train ("Context Length Extension", Notation)."""
    if s > 0:
        return float(s)
    if L_train <= 0 or L_target <= 0:
        raise ValueError("need s > 0 or both L_train and L_target > 0")
    return float(L_target) / float(L_train)


def base_frequencies(d: int, b: float) -> np.ndarray:
    """theta_i = b^(-2i/d) for i in [0, d/2)  ("Context Window Scaling ...",
    Section 2, Formal RoPE Mechanics; "Context Length Extension", Why Models
    Fail: angle at position p is p / b^(2i/d))."""
    if d < 2 or d % 2:
        raise ValueError("head dimension must be even")
    i = np.arange(d // 2, dtype=np.float64)
    return np.power(float(b), -2.0 * i / d)


def wavelength(d: int, b: float) -> np.ndarray:
    """lambda_i = 2 pi b^(2i/d)  ("Context Window Scaling ...", Section 3)."""
    i = np.arange(d // 2, dtype=np.float64)
    return 2.0 * math.pi * np.power(float(b), 2.0 * i / d)


def ntk_base(b: float, s: float, d: int) -> float:
    """NTK-aware base b' ("Context Length Extension", NTK-Aware Scaling).

    The page states only the effect -- the base is scaled so that the lowest
    frequency is interpolated while the highest one is preserved -- and drops
    the formula.  Reading adopted: b' is the base for which theta'_0 = theta_0
    (automatic, b'^0 = 1) and theta'_{d/2-1} = theta_{d/2-1} / s, i.e.
    b'^(-(d-2)/d) = b^(-(d-2)/d) / s, giving b' = b * s^(d/(d-2)).
    """
    if d <= 2:
        raise ValueError("NTK scaling needs d > 2")
    return float(b) * float(s) ** (d / (d - 2.0))


def ramp_gamma(r: np.ndarray, alpha: float, beta: float) -> np.ndarray:
    """YaRN ramp gamma(r): 0 for r <= alpha, 1 for r >= beta, linear between
    ("Context Window Scaling ...", Section 3, item 3; bounds alpha=1 and
    beta=32 follow the section's code listing, beta_slow and beta_fast)."""
    return np.clip((np.asarray(r, dtype=np.float64) - alpha) / (beta - alpha), 0.0, 1.0)


def regime_classes(d: int, b: float, L_train: float, alpha: float, beta: float) -> np.ndarray:
    """Per-dimension regime, from r_i = L_train / lambda_i (the number of full
    rotations dimension i completes inside the training window):
    r < alpha -> interpolated, r > beta -> kept, otherwise ramp.
    ("Context Window Scaling ...", Section 3, the three regimes; "Long-context
    extension ...", "Not every RoPE dimension needs the same treatment".)
    With ``L_train <= 0`` no window is known and every dimension is kept."""
    h = d // 2
    if L_train <= 0:
        return np.full(h, CLASS_KEPT, dtype=np.int8)
    r = float(L_train) / wavelength(d, b)
    cls = np.full(h, CLASS_RAMP, dtype=np.int8)
    cls[r < alpha] = CLASS_INTERPOLATED
    cls[r > beta] = CLASS_KEPT
    return cls


def mscale(kind: str, s: float) -> float:
    """YaRN attention-temperature factor sqrt(1/t) = 0.1 ln(s) + 1 for s > 1,
    and 1 otherwise ("Context Window Scaling ...", Section 3, Attention
    Entropy, and its listing's get_mscale).  Only YaRN carries a temperature
    ("Context Window Scaling ...", FAQ 1; "Context Length Extension", YaRN)."""
    if kind != "yarn" or s <= 1.0:
        return 1.0
    return 0.1 * math.log(s) + 1.0


def inv_freq(kind: str, d: int, b: float, L_train: float = 0.0, L_target: float = 0.0,
             s: float = 0.0, alpha: float = 1.0, beta: float = 32.0, dim_scale=None):
    """Rescaled rotation frequencies theta'_i, regime classes and mscale.

    * ``none``  -- theta' = 0: the rotation is the identity (inputs arrive
      already rotated).
    * ``plain`` -- theta'_i = theta_i.
    * ``pi``    -- Position Interpolation, m' = m / s, equivalently
      theta'_i = theta_i / s ("Context Window Scaling ...", Section 2, The
      Failure of Naive PI; "Context Length Extension", Position Interpolation).
    * ``ntk``   -- theta'_i = b'^(-2i/d) with b' from :func:`ntk_base`.
    * ``yarn``  -- NTK-by-parts: theta'_i = (1 - gamma_i) theta_i / s
      + gamma_i theta_i with gamma_i = gamma(L_train / lambda_i).  High
      frequencies (gamma = 1) are kept, low ones (gamma = 0) fully
      interpolated, the band between blended ("Long-context extension ...",
      NTK-by-parts paragraph; "Context Length Extension", YaRN bullets).
      The blend acts on the frequencies, the reading of "blend the two
      treatments".
    * ``perdim`` -- a caller-given rescale factor per dimension,
      theta'_i = theta_i / lambda_i: the non-uniform scale vector that
      LongRoPE's search produces ("Context Window Scaling ...", Section 4,
      a unique scale vector for each dimension; FAQ 4, factors of the
      high-frequency dimensions kept near 1).  The search itself is not part
      of this path.  The page gives no temperature for it: mscale = 1.

    Returns ``(theta_prime[d/2] float64, classes[d/2] int8, mscale float)``.
    """
    if kind not in KINDS:
        raise ValueError(f"unknown kind {kind!r}")
    h = d // 2
    theta = base_frequencies(d, b)
    cls = regime_classes(d, b, L_train, alpha, beta)
    if kind == "none":
        return np.zeros(h), cls, 1.0
    if kind == "plain":
        return theta, cls, 1.0
    if kind == "perdim":
        lam = np.asarray(dim_scale, dtype=np.float64)
        if lam.shape != (h,) or not np.all(np.isfinite(lam)) or not np.all(lam > 0):
            raise ValueError("perdim needs d/2 finite factors > 0")
        return theta / lam, cls, 1.0
    s = resolve_scale(L_train, L_target, s)
    if kind == "pi":
        return theta / s, cls, 1.0
    if kind == "ntk":
        return base_frequencies(d, ntk_base(b, s, d)), cls, 1.0
    # yarn
    if L_train <= 0:
        raise ValueError("YaRN needs L_train > 0")
    lam = wavelength(d, b)
    gamma = ramp_gamma(float(L_train) / lam, alpha, beta)
    theta_p = (1.0 - gamma) * theta / s + gamma * theta
    return theta_p, cls, mscale(kind, s)


def rotate(x: np.ndarray, positions: np.ndarray, theta: np.ndarray) -> np.ndarray:
    """Rotate each pair (x_i, x_{i+d/2}) of the last axis by the angle
    phi = m * theta_i, m the row's position:

        y_i       = x_i cos(phi) - x_{i+d/2} sin(phi)
        y_{i+d/2} = x_i sin(phi) + x_{i+d/2} cos(phi)

    ("Context Window Scaling ...", Section 2: the 2x2 rotation applied to each
    of the d/2 pairs.)  The pairing (i, i + d/2) is the layout the section's
    listing builds with cat(freqs, freqs): dimension j and j + d/2 share
    frequency j.  ``x`` is [..., S, d]; ``positions`` is [S] (integers).
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    h = d // 2
    pos = np.asarray(positions, dtype=np.float64)
    phi = pos[:, None] * np.asarray(theta, dtype=np.float64)[None, :]  # [S, h]
    c, s_ = np.cos(phi), np.sin(phi)
    x1, x2 = x[..., :h], x[..., h:]
    return np.concatenate([x1 * c - x2 * s_, x1 * s_ + x2 * c], axis=-1)


def rope_apply(x, positions, kind, d, b, L_train=0.0, L_target=0.0, s=0.0,
               alpha=1.0, beta=32.0, apply_mscale=False, dim_scale=None):
    """Rotate ``x`` [..., S, d] with the rescaled frequencies; optionally
    multiply by mscale (the temperature split evenly over q and k: q.k then
    carries mscale^2 = 1/t)."""
    theta, _, ms = inv_freq(kind, d, b, L_train, L_target, s, alpha, beta, dim_scale)
    y = rotate(x, positions, theta)
    return y * ms if apply_mscale else y
