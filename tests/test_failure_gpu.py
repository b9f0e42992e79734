"""The failure path on the GPU, by host-controlled fault injection.

Every wait in the decode and prefill kernels is bounded.  Here the host makes
one wait run out on purpose, in the allowed way: the producer never issues
one load unit, so the barrier that the consumers wait on is never completed,
and a short wait bound (about a millisecond) makes them give up.  The kernel
must then record the timeout, let the copies and products it did issue
finish, free its tensor memory and return; ``yr_sync_status`` reports
YR_ERR_TIMEOUT, and the next normal call on the same device must succeed and
match the oracle.
"""

import math

import numpy as np
import pytest
import torch

import oracle.attention as A
import oracle.rope as R
from tests.helpers import assert_attn_close, f64, gpu, need_cuda
from yarn_rope_scaling_ntk_b300 import api, workloads as W

pytestmark = gpu

SHORT_LIMIT = 2_000_000  # SM cycles: about 1 ms at 2 GHz


def _expect_timeout():
    with pytest.raises(api.YarnAttnError) as e:
        api.sync_status()
    assert e.value.status == 4, str(e.value)


def _decode_case():
    w = W.Decode("fault_decode", 81, 2, 4, 4, 128, 4, 60, W.RopeSpec("plain"), full=True)
    return w, W.decode_inputs(w, "cuda")


def _decode_oracle(w, inp):
    q, kc, vc, nv, rs = inp
    th = R.base_frequencies(w.d, 1e4)
    want = []
    for b in range(w.B):
        for h in range(w.Hq):
            o, _ = A.decode_head(f64(q[b, h]), f64(kc[b, h]), f64(vc[b, h]), int(nv[b]), int(rs[b]), w.sink,
                                 w.window, th, 1.0 / math.sqrt(w.d))
            want.append(o)
    return np.stack(want).reshape(w.B, w.Hq, w.d)


def test_decode_wait_runs_out_then_the_next_call_is_correct():
    need_cuda()
    w, inp = _decode_case()
    q, kc, vc, nv, rs = inp
    cfg = api.RopeConfig(kind="plain", head_dim=w.d)
    api.sync_status()
    try:
        api.debug_inject_wait_fault(SHORT_LIMIT, 0)  # the first cache chunk is never loaded
        api.attn_fwd_decode_sinkwindow(cfg, q, kc, vc, nv, rs, w.sink, w.window, num_splits=1)
        _expect_timeout()
    finally:
        api.debug_inject_wait_fault(0, -1)
    o = api.attn_fwd_decode_sinkwindow(cfg, q, kc, vc, nv, rs, w.sink, w.window, num_splits=1)
    api.sync_status()
    assert_attn_close(f64(o), _decode_oracle(w, inp), "decode after a timeout")


def _prefill_case():
    w = W.Prefill("fault_prefill", 82, 1, 2, 2, 256, 128, torch.bfloat16, W.RopeSpec("yarn", 1e4, 128, 0, 4.0))
    return w, W.prefill_inputs(w, "cuda")


def _prefill_check(w, q, k, v, o):
    th, _, _ = R.inv_freq("yarn", w.d, 1e4, 128, 0, 4.0)
    scale = A.softmax_scale("yarn", 4.0, w.d)
    for h in range(w.Hq):
        rows = np.arange(w.S)
        want, _ = A.prefill_head(f64(q[0, h]), f64(k[0, h]), f64(v[0, h]), rows, th, scale, "causal")
        assert_attn_close(f64(o[0, h]), want, f"prefill head {h} after a timeout")


@pytest.mark.parametrize("skip_unit", [0, 1, 2])
def test_prefill_wait_runs_out_then_the_next_call_is_correct(skip_unit):
    """Unit 0 is the first K tile, unit 1 the first V tile with the second K
    tile, unit 2 the last V tile: the MMA warp gives up before any product,
    between products, and before the last PV products."""
    need_cuda()
    w, (q, k, v) = _prefill_case()
    cfg = api.RopeConfig(kind="yarn", head_dim=w.d, L_train=128, s=4.0)
    api.sync_status()
    try:
        api.debug_inject_wait_fault(SHORT_LIMIT, skip_unit)
        api.attn_fwd_prefill(cfg, q, k, v)
        _expect_timeout()
    finally:
        api.debug_inject_wait_fault(0, -1)
    o = api.attn_fwd_prefill(cfg, q, k, v)
    api.sync_status()
    _prefill_check(w, q, k, v, o)


def test_a_short_bound_alone_changes_nothing():
    """With the short bound and no skipped unit every wait completes in time:
    the results are those of the default bound."""
    need_cuda()
    w, (q, k, v) = _prefill_case()
    cfg = api.RopeConfig(kind="yarn", head_dim=w.d, L_train=128, s=4.0)
    want = api.attn_fwd_prefill(cfg, q, k, v)
    api.sync_status()
    try:
        api.debug_inject_wait_fault(50 * SHORT_LIMIT, -1)
        got = api.attn_fwd_prefill(cfg, q, k, v)
        api.sync_status()
    finally:
        api.debug_inject_wait_fault(0, -1)
    assert torch.equal(got, want)
