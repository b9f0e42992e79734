"""Oracle: FP8 E4M3 decoding and decode attention over an FP8 cache (float64).

TEST INFRASTRUCTURE ONLY -- see the package docstring.

KV-cache quantisation to FP8 ("Context Window Scaling ...", FAQ 3) stores
each cache entry as one OCP E4M3 byte; the dequantised value is the decoded
byte times a float32 scale of its (sequence, KV head).  The attention over
the dequantised cache is the plain decode definition in ``oracle.attention``.
"""

from __future__ import annotations

import numpy as np

from . import attention as _attn


def e4m3_to_float(codes) -> np.ndarray:
    """Decode OCP FP8 E4M3 bytes: 1 sign bit, 4 exponent bits (bias 7), 3
    mantissa bits.  Exponent field 0 is subnormal, value 2^-6 * m / 8; the
    all-ones pattern S.1111.111 is NaN; there are no infinities (the largest
    finite magnitude is 2^8 * 1.75 = 448)."""
    c = np.asarray(codes).astype(np.int64) & 0xFF
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    val = sign * mag
    return np.where((c & 0x7F) == 0x7F, np.nan, val)


def decode_head_fp8(q, k_codes, v_codes, k_scale, v_scale, n_valid, ring_start, sink, window, theta, scale):
    """One new query token against one head of an FP8 sink + window cache:
    dequantise (decoded byte x scale) and apply the plain decode definition."""
    k = e4m3_to_float(k_codes) * float(k_scale)
    v = e4m3_to_float(v_codes) * float(v_scale)
    return _attn.decode_head(q, k, v, n_valid, ring_start, sink, window, theta, scale)
