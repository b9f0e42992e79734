"""Pins for oracle.quant: E4M3 code points fixed by the format's definition,
and every code against torch's own float8_e4m3fn conversion."""

import math

import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import quant as Q
from oracle import rope


@pytest.mark.parametrize("code,value", [(0x00, 0.0), (0x38, 1.0), (0xB8, -1.0), (0x40, 2.0), (0xC0, -2.0),
                                        (0x7E, 448.0), (0xFE, -448.0), (0x08, 2.0 ** -6), (0x01, 2.0 ** -9),
                                        (0x07, 7 * 2.0 ** -9), (0x39, 1.125), (0x30, 0.5)])
def test_e4m3_code_points(code, value):
    assert Q.e4m3_to_float(code) == value


def test_e4m3_nan_codes_and_signed_zero():
    assert np.isnan(Q.e4m3_to_float(0x7F)) and np.isnan(Q.e4m3_to_float(0xFF))
    z = Q.e4m3_to_float(0x80)
    assert z == 0.0 and math.copysign(1.0, z) == -1.0


def test_e4m3_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = Q.e4m3_to_float(codes)
    nan = np.isnan(want)
    assert np.array_equal(nan, np.isnan(got))
    np.testing.assert_array_equal(got[~nan], want[~nan])


def test_decode_fp8_equals_decode_on_dequantised_cache():
    rng = np.random.default_rng(8)
    C, d = 20, 8
    kc = rng.integers(0, 256, (C, d)).astype(np.uint8)
    vc = rng.integers(0, 256, (C, d)).astype(np.uint8)
    kc[(kc & 0x7F) == 0x7F] = 0x38   # no NaN codes in a cache
    vc[(vc & 0x7F) == 0x7F] = 0x38
    q = rng.standard_normal(d)
    th = rope.base_frequencies(d, 1e4)
    o, l = Q.decode_head_fp8(q, kc, vc, 0.01, 0.02, 17, 5, 2, 18, th, 0.3)
    o2, l2 = A.decode_head(q, Q.e4m3_to_float(kc) * 0.01, Q.e4m3_to_float(vc) * 0.02, 17, 5, 2, 18, th, 0.3)
    np.testing.assert_array_equal(o, o2)
    assert l == l2
