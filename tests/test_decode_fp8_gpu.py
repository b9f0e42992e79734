"""attn_fwd_decode_sinkwindow_fp8 (FP8 E4M3 cache with per-(sequence, KV head)
scales) on the GPU against the float64 oracle on the dequantised cache."""

import math

import numpy as np
import pytest
import torch

import oracle.quant as Q
import oracle.rope as R
from tests.helpers import assert_attn_close, assert_lse_close, f64, gpu, need_cuda
from yarn_rope_scaling_ntk_b300 import api, workloads as W

pytestmark = gpu


def _oracle(w, q, kc, vc, ks, vs, nv, rs):
    r = w.rope
    th, _, ms = R.inv_freq(r.kind, w.d, r.theta_base, r.L_train, r.L_target, r.s)
    scale = ms * ms / math.sqrt(w.d)
    qn, kn, vn = f64(q), kc.cpu().numpy(), vc.cpu().numpy()
    ksn, vsn, nvn, rsn = f64(ks), f64(vs), nv.cpu().numpy(), rs.cpu().numpy()
    G = w.Hq // w.Hkv
    o = np.zeros((w.B, w.Hq, w.d))
    lse = np.zeros((w.B, w.Hq))
    for b in range(w.B):
        for h in range(w.Hq):
            hk = h // G
            o[b, h], lse[b, h] = Q.decode_head_fp8(qn[b, h], kn[b, hk], vn[b, hk], ksn[b, hk], vsn[b, hk],
                                                   int(nvn[b]), int(rsn[b]), w.sink, w.window, th, scale)
    return o, lse


def _run(w, splits=0):
    inp = W.decode_inputs_fp8(w, "cuda")
    q, kc, vc, ks, vs, nv, rs = inp
    r = w.rope
    cfg = api.RopeConfig(kind=r.kind, head_dim=w.d, theta_base=r.theta_base, L_train=r.L_train,
                         L_target=r.L_target, s=r.s)
    o, lse = api.attn_fwd_decode_sinkwindow_fp8(cfg, q, kc, vc, ks, vs, nv, rs, w.sink, w.window,
                                                num_splits=splits, return_lse=True)
    torch.cuda.synchronize()
    return inp, o, lse


def test_fp8_decode_full_workload_shape():
    """64 sequences x 32 heads, 4 sinks + 4092-slot ring, every head."""
    need_cuda()
    w = W.DECODE
    inp, o, lse = _run(w)
    want_o, want_l = _oracle(w, *inp)
    assert_attn_close(f64(o), want_o, "fp8 decode full")
    assert_lse_close(f64(lse), want_l, "fp8 decode full")


@pytest.mark.parametrize("splits,G,d", [(1, 4, 128), (3, 4, 128), (2, 1, 64), (0, 8, 64)])
def test_fp8_decode_partial_caches(splits, G, d):
    need_cuda()
    w = W.Decode("fp8_partial", 36, 5, 4 * G, 4, d, 4, 700, W.RopeSpec("yarn", 1e4, 256, 0, 4.0), full=False)
    inp, o, lse = _run(w, splits)
    want_o, want_l = _oracle(w, *inp)
    assert_attn_close(f64(o), want_o, f"fp8 G={G} d={d} splits={splits}")
    assert_lse_close(f64(lse), want_l)


def test_fp8_decode_matches_bf16_decode_on_the_dequantised_cache():
    """The same cache dequantised to bf16 through the bf16 entry point: the
    two differ only by the bf16 rounding of the dequantised values."""
    need_cuda()
    w = W.Decode("fp8_vs_bf16", 37, 3, 8, 8, 128, 4, 300, W.RopeSpec("plain"), full=False)
    q, kc, vc, ks, vs, nv, rs = W.decode_inputs_fp8(w, "cuda")
    cfg = api.RopeConfig(kind="plain", head_dim=128)
    o8 = api.attn_fwd_decode_sinkwindow_fp8(cfg, q, kc, vc, ks, vs, nv, rs, w.sink, w.window)
    kd = (kc.view(torch.float8_e4m3fn).float() * ks[:, :, None, None]).to(torch.bfloat16)
    vd = (vc.view(torch.float8_e4m3fn).float() * vs[:, :, None, None]).to(torch.bfloat16)
    o16 = api.attn_fwd_decode_sinkwindow(cfg, q, kd, vd, nv, rs, w.sink, w.window)
    torch.cuda.synchronize()
    assert (o8.float() - o16.float()).abs().max().item() < 2e-2
