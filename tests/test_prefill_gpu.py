"""attn_fwd_prefill on the GPU against the float64 oracle."""

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


def cfg_of(w, dim_scale=None):
    r = w.rope
    return api.RopeConfig(kind=r.kind, head_dim=w.d, theta_base=r.theta_base, L_train=r.L_train,
                          L_target=r.L_target, s=r.s, dim_scale=dim_scale)


def oracle_prefill(w, q, k, v, rows_per_head, extra_rows=()):
    """Oracle rows for every (batch, query head): returns {(b, h): (rows, o, lse)}."""
    r = w.rope
    th, _, _ = R.inv_freq(r.kind, w.d, r.theta_base, r.L_train, r.L_target, r.s)
    s = R.resolve_scale(r.L_train, r.L_target, r.s) if r.kind in ("pi", "ntk", "yarn") else 1.0
    scale = A.softmax_scale(r.kind, s, w.d)
    G = w.Hq // w.Hkv
    out = {}
    for b in range(w.B):
        for hk in range(w.Hkv):
            kr = R.rotate(f64(k[b, hk]), np.arange(w.S), th)
            vv = f64(v[b, hk])
            for h in range(hk * G, (hk + 1) * G):
                rows = W.sample_rows(w.S, rows_per_head, 100 * b + h, extra_rows).numpy()
                qr = R.rotate(f64(q[b, h, rows]), rows, th)
                o, lse = A.attention_rows(qr, rows, kr, vv, w.mask, w.sink, w.window, scale)
                out[(b, h)] = (rows, o, lse)
    return out


def check(w, q, k, v, rows_per_head, extra_rows=(), ring_blocks=None):
    o, lse = api.attn_fwd_prefill(cfg_of(w), q, k, v, mask=w.mask, sink=w.sink, window=w.window,
                                  ring_blocks=w.ring_blocks if ring_blocks is None else ring_blocks,
                                  return_lse=True)
    torch.cuda.synchronize()
    ref = oracle_prefill(w, q, k, v, rows_per_head, extra_rows)
    got_o, want_o, got_l, want_l = [], [], [], []
    for (b, h), (rows, oo, ll) in ref.items():
        got_o.append(f64(o[b, h, rows]))
        want_o.append(oo)
        got_l.append(f64(lse[b, h, rows]))
        want_l.append(ll)
    assert_attn_close(np.concatenate(got_o), np.concatenate(want_o), w.name)
    assert_lse_close(np.concatenate(got_l), np.concatenate(want_l), w.name)
    return o, lse


@pytest.mark.parametrize("kind", ["yarn", "pi", "ntk"])
def test_tiny_fp32_all_rows(kind):
    need_cuda()
    w = replace(W.TINY, rope=replace(W.TINY.rope, kind=kind))
    q, k, v = W.prefill_inputs(w, "cuda")
    o4, _ = check(w, q, k, v, 0)
    # natural order gives the same result up to rounding: P is rounded to
    # bfloat16 against a different running maximum (relative 2^-8), so the two
    # orders differ by about 1e-3 and each is within tolerance of the oracle
    o1, _ = check(w, q, k, v, 0, ring_blocks=1)
    assert (o4 - o1).abs().max().item() < 1e-2


@pytest.mark.parametrize("S,d,Hq,Hkv,mask,sink,window,ring", [
    (200, 128, 4, 4, "causal", 0, 0, 1),          # ragged tail
    (333, 64, 4, 2, "causal", 0, 0, 1),           # ragged, GQA, d = 64
    (512, 128, 8, 2, "sink_window", 4, 100, 1),   # sink + window
    (768, 128, 4, 1, "sink_window", 0, 64, 1),    # pure sliding window
    (640, 128, 2, 2, "sink_window", 4, 1000, 1),  # window covers the sequence
    (256, 128, 2, 2, "none", 0, 0, 2),            # no mask, full ring
    (1024, 128, 2, 1, "causal", 0, 0, 4),         # ring order, GQA
    (1, 128, 2, 2, "causal", 0, 0, 1),            # single token
    (130, 64, 2, 2, "none", 0, 0, 1),
])
def test_small_shapes_all_rows(S, d, Hq, Hkv, mask, sink, window, ring):
    need_cuda()
    w = W.Prefill(f"small_S{S}_d{d}", 50 + S % 97, 2, Hq, Hkv, S, d, torch.bfloat16,
                  W.RopeSpec("yarn", 1e4, 128, 0, 4.0), mask, sink, window, ring)
    q, k, v = W.prefill_inputs(w, "cuda")
    check(w, q, k, v, 0)


def test_count_probe_exact_mask():
    """Q = 0 (no rotation) makes every visible logit 0: lse = ln(count) with
    count from the mask definition, exact up to float32 rounding."""
    need_cuda()
    for mask, sink, window in (("causal", 0, 0), ("sink_window", 4, 37), ("sink_window", 0, 200)):
        w = W.Prefill("probe", 60, 1, 2, 2, 700, 128, torch.bfloat16, W.RopeSpec("none"), mask, sink, window)
        q, k, v = W.prefill_inputs(w, "cuda")
        q.zero_()
        _, lse = api.attn_fwd_prefill(cfg_of(w), q, k, v, mask=mask, sink=sink, window=window,
                                      return_lse=True)
        torch.cuda.synchronize()
        m = np.arange(w.S)
        if mask == "causal":
            count = m + 1
        else:
            in_window = np.minimum(m + 1, window)
            count = in_window + np.clip(np.minimum(sink, m + 1 - in_window), 0, None)
        assert np.abs(f64(lse[0, 0]) - np.log(count)).max() < 1e-5


def test_row0_returns_v0():
    need_cuda()
    w = W.Prefill("row0", 61, 1, 2, 2, 300, 128, torch.bfloat16, W.RopeSpec("yarn", 1e4, 128, 0, 4.0))
    q, k, v = W.prefill_inputs(w, "cuda")
    o = api.attn_fwd_prefill(cfg_of(w), q, k, v)
    torch.cuda.synchronize()
    assert torch.equal(o[0, :, 0], v[0, :, 0])


def test_llama2_7b_shape_sampled_rows():
    need_cuda()
    w = W.LLAMA2_7B
    q, k, v = W.prefill_inputs(w, "cuda")
    # 256 seeded query rows per head on all 32 heads, plus tile and block edges
    check(w, q, k, v, w.rows_per_head, extra_rows=(4095, 4096, 8191, 8192))


def test_ring_128k_sampled_rows():
    need_cuda()
    w = W.RING_128K
    q, k, v = W.prefill_inputs(w, "cuda")
    bs = w.S // w.ring_blocks
    edges = tuple(x for j in range(1, w.ring_blocks) for x in (j * bs - 1, j * bs, j * bs + 1))
    # 128 seeded query rows per head on all 32 heads, plus every ring-block edge
    check(w, q, k, v, w.rows_per_head, extra_rows=edges)


@pytest.mark.parametrize("wl", [W.LLAMA3_8B_GQA, W.LLAMA3_8B_GQA_SW])
def test_llama3_8b_gqa_sampled_rows(wl):
    need_cuda()
    q, k, v = W.prefill_inputs(wl, "cuda")
    # 32 seeded query rows per (sequence, head): 4096 rows per mask, plus the window edges
    check(wl, q, k, v, wl.rows_per_head, extra_rows=(8191, 8192, 8193, 8194, 8195, 8196, 8197, 16384))


def test_perdim_scale_vector_prefill_all_rows():
    """Attention with a per-dimension scale vector (LongRoPE's form) on the
    rotation, every row of a small ragged workload."""
    need_cuda()
    w = W.Prefill("perdim", 62, 1, 4, 2, 390, 128, torch.bfloat16, W.RopeSpec("perdim", 1e4, 128, 0, 0.0),
                  "causal")
    lam = np.concatenate([np.ones(20), np.linspace(1.0, 8.0, 30), np.full(14, 8.0)])
    q, k, v = W.prefill_inputs(w, "cuda")
    o, lse = api.attn_fwd_prefill(cfg_of(w, tuple(lam)), q, k, v, return_lse=True)
    torch.cuda.synchronize()
    th, _, _ = R.inv_freq("perdim", w.d, 1e4, 128, dim_scale=lam)
    scale = 1.0 / math.sqrt(w.d)
    got, want, gl, wl = [], [], [], []
    for h in range(w.Hq):
        rows = np.arange(w.S)
        kr = R.rotate(f64(k[0, h // 2]), rows, th)
        qr = R.rotate(f64(q[0, h]), rows, th)
        oo, ll = A.attention_rows(qr, rows, kr, f64(v[0, h // 2]), "causal", 0, 0, scale)
        got.append(f64(o[0, h])); want.append(oo); gl.append(f64(lse[0, h])); wl.append(ll)
    assert_attn_close(np.concatenate(got), np.concatenate(want), "perdim")
    assert_lse_close(np.concatenate(gl), np.concatenate(wl), "perdim")


def test_strided_inputs_all_rows():
    """Q, K, V given as [B, S, H, d] tensors viewed as [B, H, S, d] (row
    stride H * d): the rotation pass copies them row by row, V is read in place
    through its strides; every row against the oracle, and the same result as
    contiguous copies."""
    need_cuda()
    w = W.Prefill("strided", 63, 2, 4, 2, 300, 128, torch.bfloat16, W.RopeSpec("yarn", 1e4, 128, 0, 4.0), "causal")
    q, k, v = W.prefill_inputs(w, "cuda")
    qs, ks, vs = (t.transpose(1, 2).contiguous().transpose(1, 2) for t in (q, k, v))
    assert qs.stride(2) == w.Hq * w.d and ks.stride(2) == w.Hkv * w.d
    o, lse = api.attn_fwd_prefill(cfg_of(w), qs, ks, vs, return_lse=True)
    o_c = api.attn_fwd_prefill(cfg_of(w), q, k, v)
    torch.cuda.synchronize()
    assert torch.equal(o, o_c)
    ref = oracle_prefill(w, q, k, v, 0)
    got_o = np.concatenate([f64(o[b, h]) for (b, h) in ref])
    want_o = np.concatenate([oo for (_, oo, _) in ref.values()])
    assert_attn_close(got_o, want_o, "strided")
