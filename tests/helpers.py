"""Shared test utilities: tolerances and comparisons (no method arithmetic)."""

import numpy as np
import pytest
import torch

# Tolerances stated for the path: rope_apply float32 max-abs 1e-5; bfloat16
# attention outputs max-abs 2e-2 and relative L2 1e-2; LSE abs 1e-2.
ROPE_F32_ATOL = 1e-5
ATTN_MAX_ABS = 2e-2
ATTN_REL_L2 = 1e-2
LSE_ATOL = 1e-2

gpu = pytest.mark.gpu


def need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def assert_attn_close(got: np.ndarray, want: np.ndarray, what: str = ""):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - want).max() if got.size else 0.0
    rel = np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-30)
    assert err <= ATTN_MAX_ABS, f"{what}: max-abs {err:.3e} > {ATTN_MAX_ABS}"
    assert rel <= ATTN_REL_L2, f"{what}: rel-L2 {rel:.3e} > {ATTN_REL_L2}"
    return err, rel


def assert_lse_close(got, want, what=""):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    both_inf = np.isneginf(got) & np.isneginf(want)
    with np.errstate(invalid="ignore"):
        err = np.abs(np.where(both_inf, 0.0, got - want)).max() if got.size else 0.0
    assert err <= LSE_ATOL, f"{what}: lse max-abs {err:.3e}"


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bfloat16 numbers at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(ax)) - 7)


def rope_bf16_bound(want: np.ndarray, x: np.ndarray) -> np.ndarray:
    """Bar for a bfloat16 rotation output: one bf16 ulp of the float64 value,
    plus the float32 error of the rotation itself.  Each output is a two-term
    sum x_i cos - x_(i+d/2) sin (or x_i sin + x_(i+d/2) cos) formed in float32
    from an angle carried to a few float32 ulps, so its absolute error scales
    with |x_i| + |x_(i+d/2)|, not with the output: 2^-20 of that sum (16
    float32 ulps) covers it.  Where the two terms nearly cancel, the output's
    own ulp is far smaller than that error; elsewhere the ulp dominates."""
    h = x.shape[-1] // 2
    pair = np.abs(x[..., :h]) + np.abs(x[..., h:])
    return bf16_ulp(want) + 2.0 ** -20 * np.concatenate([pair, pair], axis=-1)
