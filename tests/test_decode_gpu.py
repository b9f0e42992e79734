"""attn_fwd_decode_sinkwindow on the GPU against the float64 oracle."""

import math
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle.attention as A
import oracle.rope as R
from tests.helpers import assert_attn_close, assert_lse_close, f64, gpu, need_cuda
from yarn_rope_scaling_ntk_b300 import api, workloads as W

pytestmark = gpu


def oracle_decode(w, q, kc, vc, n_valid, ring_start, rope):
    """Oracle outputs for every (sequence, query head)."""
    th, _, ms = R.inv_freq(rope.kind, w.d, rope.theta_base, rope.L_train, rope.L_target, rope.s)
    scale = A.softmax_scale(rope.kind, R.resolve_scale(rope.L_train, rope.L_target, rope.s)
                            if rope.kind in ("pi", "ntk", "yarn") else 1.0, w.d)
    qn, kn, vn = f64(q), f64(kc), f64(vc)
    nv, rs = n_valid.cpu().numpy(), ring_start.cpu().numpy()
    G = w.Hq // w.Hkv
    o = np.zeros((w.B, w.Hq, w.d))
    lse = np.zeros((w.B, w.Hq))
    for b in range(w.B):
        n = int(nv[b])
        if n == 0:
            lse[b] = -np.inf
            continue
        j = np.arange(n)
        phys = A.decode_logical_to_physical(j, w.sink, w.window, int(rs[b]))
        k_rot = R.rotate(kn[b][:, phys], j, th)                      # [Hkv, n, d]
        q_rot = R.rotate(qn[b][:, None, :], [n - 1], th)[:, 0]        # [Hq, d]
        for h in range(w.Hq):
            oo, ll = A.attention_rows(q_rot[h:h + 1], np.array([n - 1]), k_rot[h // G],
                                      vn[b][h // G][phys], "none", 0, 0, scale)
            o[b, h], lse[b, h] = oo[0], ll[0]
    return o, lse


def run(w, rope, num_splits=0, inputs=None):
    q, kc, vc, nv, rs = inputs if inputs is not None else W.decode_inputs(w, "cuda")
    cfg = api.RopeConfig(kind=rope.kind, head_dim=w.d, theta_base=rope.theta_base,
                         L_train=rope.L_train, L_target=rope.L_target, s=rope.s)
    o, lse = api.attn_fwd_decode_sinkwindow(cfg, q, kc, vc, nv, rs, w.sink, w.window,
                                            num_splits=num_splits, return_lse=True)
    torch.cuda.synchronize()
    return (q, kc, vc, nv, rs), o, lse


def test_decode_full_workload_all_heads():
    """64 sequences x 32 heads, 4 sinks + 4092-slot ring, every head compared."""
    need_cuda()
    w = W.DECODE
    inp, o, lse = run(w, w.rope)
    want_o, want_l = oracle_decode(w, *inp, w.rope)
    assert_attn_close(f64(o), want_o, "decode full")
    assert_lse_close(f64(lse), want_l, "decode full")


@pytest.mark.parametrize("splits", [1, 3, 8])
def test_decode_partial_caches_gqa_yarn(splits):
    need_cuda()
    w = W.Decode("partial_gqa", 31, 6, 32, 8, 128, 4, 1020, W.RopeSpec("yarn", 5e5, 256, 0, 4.0),
                 full=False)
    inp, o, lse = run(w, w.rope, num_splits=splits)
    want_o, want_l = oracle_decode(w, *inp, w.rope)
    assert_attn_close(f64(o), want_o, f"gqa splits={splits}")
    assert_lse_close(f64(lse), want_l)


@pytest.mark.parametrize("G", [1, 2, 8])
def test_decode_d64_and_group_sizes(G):
    need_cuda()
    w = W.Decode("d64", 32, 3, 4 * G, 4, 64, 4, 200, W.RopeSpec("ntk", 1e4, 64, 0, 8.0), full=False)
    inp, o, lse = run(w, w.rope, num_splits=2)
    want_o, want_l = oracle_decode(w, *inp, w.rope)
    assert_attn_close(f64(o), want_o, f"d64 G={G}")
    assert_lse_close(f64(lse), want_l)


def test_decode_count_probe_and_edges():
    """q = 0 makes every logit 0: lse = ln(n_valid) exactly and o = mean of
    the valid values; n_valid = 0 gives o = 0 and lse = -inf; sink = 0 works."""
    need_cuda()
    for sink in (4, 0):
        w = W.Decode("probe", 33, 5, 4, 4, 128, sink, 300, W.RopeSpec("plain"), full=False)
        q, kc, vc, nv, rs = W.decode_inputs(w, "cuda")
        q.zero_()
        nv = torch.tensor([0, 1, sink + 1, 77, sink + 300], dtype=torch.int32, device="cuda")
        _, o, lse = run(w, w.rope, num_splits=0, inputs=(q, kc, vc, nv, rs))
        l = f64(lse)
        for b, n in enumerate(nv.tolist()):
            if n == 0:
                assert np.all(np.isneginf(l[b])) and torch.all(o[b] == 0)
            else:
                assert np.abs(l[b] - math.log(n)).max() < 2e-6
        want_o, _ = oracle_decode(w, q, kc, vc, nv, rs, w.rope)
        assert_attn_close(f64(o), want_o, "probe")


def test_decode_ring_start_shift_invariance():
    """Rolling the ring contents and moving ring_start with them leaves the
    result unchanged (same values, same logical order)."""
    need_cuda()
    w = W.Decode("shift", 34, 2, 8, 8, 128, 4, 500, W.RopeSpec("yarn", 1e4, 128, 0, 4.0))
    q, kc, vc, nv, rs = W.decode_inputs(w, "cuda")
    rs.zero_()
    _, o0, l0 = run(w, w.rope, inputs=(q, kc, vc, nv, rs))
    kc2, vc2 = kc.clone(), vc.clone()
    kc2[:, :, 4:] = torch.roll(kc[:, :, 4:], 123, dims=2)
    vc2[:, :, 4:] = torch.roll(vc[:, :, 4:], 123, dims=2)
    _, o1, l1 = run(w, w.rope, inputs=(q, kc2, vc2, nv, torch.full_like(rs, 123)))
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
