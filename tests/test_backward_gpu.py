"""attn_bwd on the GPU against the float64 oracle.

O and LSE come from the oracle's forward (inputs to the CUDA path, never the
other way round), so every difference is the backward's own arithmetic:
bfloat16 operands (the rotated q and k, v, dO, and the bf16 P and dS fed to
the tensor cores) with float32 accumulation.  Tolerance, from that
arithmetic: each gradient element is a float32 sum of products whose bf16
factors carry a relative rounding of at most 2^-9; the errors are random in
sign, so the relative L2 error of a whole gradient stays near 2^-9 times a
small constant.  Bar: relative L2 <= 1e-2 per gradient (as for the forward
outputs) and max-abs <= 3e-2 of the gradient's largest magnitude.
"""

import math

import numpy as np
import pytest
import torch

import oracle.attention as A
import oracle.rope as R
from tests.helpers import f64, gpu, need_cuda
from yarn_rope_scaling_ntk_b300 import api, workloads as W

pytestmark = gpu

BWD_REL_L2 = 1e-2
BWD_MAX_REL = 3e-2


def _check(got, want, what):
    got, want = np.asarray(got, np.float64), np.asarray(want, np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite"
    rel = np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-30)
    mx = np.abs(got - want).max() / max(np.abs(want).max(), 1e-30)
    assert rel <= BWD_REL_L2, f"{what}: rel-L2 {rel:.3e}"
    assert mx <= BWD_MAX_REL, f"{what}: max-abs / max|ref| {mx:.3e}"
    return rel, mx


def _run(w, dtype_out=torch.float32, seed=0):
    r = w.rope
    cfg = api.RopeConfig(kind=r.kind, head_dim=w.d, theta_base=r.theta_base, L_train=r.L_train,
                         L_target=r.L_target, s=r.s)
    q, k, v = W.prefill_inputs(w, "cuda")
    g = torch.Generator(device="cuda").manual_seed(900 + seed)
    dout = torch.randn(q.shape, generator=g, device="cuda").to(q.dtype)
    th, _, ms = R.inv_freq(r.kind, w.d, r.theta_base, r.L_train, r.L_target, r.s)
    scale = ms * ms / math.sqrt(w.d)
    G = w.Hq // w.Hkv
    pos = np.arange(w.S)
    qn, kn, vn, gn = f64(q), f64(k), f64(v), f64(dout)
    o_ref = np.zeros(qn.shape)
    lse_ref = np.zeros(qn.shape[:3])
    dq_ref, dk_ref, dv_ref = np.zeros(qn.shape), np.zeros(kn.shape), np.zeros(vn.shape)
    for b in range(w.B):
        for h in range(w.Hq):
            hk = h // G
            qr = R.rotate(qn[b, h], pos, th)
            kr = R.rotate(kn[b, hk], pos, th)
            o_ref[b, h], lse_ref[b, h] = A.attention_rows(qr, pos, kr, vn[b, hk], w.mask, w.sink, w.window, scale)
            dq, dk, dv = A.backward_head(qn[b, h], kn[b, hk], vn[b, hk], gn[b, h], pos, pos, th, scale, w.mask,
                                         w.sink, w.window)
            dq_ref[b, h] = dq
            dk_ref[b, hk] += dk
            dv_ref[b, hk] += dv
    o_in = torch.from_numpy(o_ref).to("cuda", q.dtype)
    lse_in = torch.from_numpy(lse_ref).to("cuda", torch.float32).contiguous()
    dq, dk, dv = api.attn_bwd(cfg, q, k, v, o_in, dout, lse_in, mask=w.mask, sink=w.sink, window=w.window,
                              out_dtype=dtype_out)
    torch.cuda.synchronize()
    return (dq, dk, dv), (dq_ref, dk_ref, dv_ref)


@pytest.mark.parametrize("kind", ["yarn", "pi"])
def test_backward_tiny_fp32(kind):
    need_cuda()
    w = W.Prefill("bwd_tiny", 80, 1, 4, 4, 256, 64, torch.float32, W.RopeSpec(kind, 1e4, 64, 256, 0.0), "causal")
    got, want = _run(w)
    for g_, w_, n in zip(got, want, ("dq", "dk", "dv")):
        _check(f64(g_), w_, f"tiny {kind} {n}")


@pytest.mark.parametrize("mask,sink,window,Hq,Hkv,S", [
    ("causal", 0, 0, 4, 2, 384),
    ("sink_window", 4, 150, 4, 4, 512),
    ("none", 0, 0, 2, 1, 256),
    ("causal", 0, 0, 8, 2, 1024),
])
def test_backward_bf16_d128(mask, sink, window, Hq, Hkv, S):
    need_cuda()
    w = W.Prefill("bwd", 81 + S % 13, 2, Hq, Hkv, S, 128, torch.bfloat16, W.RopeSpec("yarn", 1e4, 128, 0, 4.0),
                  mask, sink, window)
    got, want = _run(w, seed=S)
    for g_, w_, n in zip(got, want, ("dq", "dk", "dv")):
        _check(f64(g_), w_, f"{mask} S={S} {n}")


def test_backward_bf16_outputs_and_errors():
    need_cuda()
    w = W.Prefill("bwd_bf16out", 85, 1, 2, 2, 256, 128, torch.bfloat16, W.RopeSpec("ntk", 1e4, 128, 0, 8.0))
    got, want = _run(w, dtype_out=torch.bfloat16)
    for g_, w_, n in zip(got, want, ("dq", "dk", "dv")):
        assert g_.dtype == torch.bfloat16
        _check(f64(g_), w_, f"bf16 out {n}")
    q = torch.zeros(1, 2, 200, 128, device="cuda", dtype=torch.bfloat16)
    lse = torch.zeros(1, 2, 200, device="cuda")
    with pytest.raises(api.YarnAttnError) as e:
        api.attn_bwd(api.RopeConfig(kind="plain", head_dim=128), q, q, q, q, q, lse)
    assert e.value.status == 2  # S not a multiple of 128


def _heads_per_group(units: int, n_tiles: int) -> int:
    """Heads per scheduling group of the backward kernels on this GPU (about
    four waves of CTAs per group), to place checks on both sides of a group
    boundary."""
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    return max(1, min(units, (4 * sm + n_tiles - 1) // n_tiles))


def test_backward_across_scheduling_groups():
    """2 x 40 (batch, head) units of 8 tiles each: more units than one
    scheduling group holds, so later groups' CTAs follow the first group's.
    O and LSE come from the oracle; the last unit of the first group, the
    first of the next and both ends are checked."""
    need_cuda()
    w = W.Prefill("bwd_groups", 86, 2, 40, 40, 1024, 128, torch.bfloat16, W.RopeSpec("yarn", 1e4, 256, 0, 4.0),
                  "causal")
    r = w.rope
    cfg = api.RopeConfig(kind=r.kind, head_dim=w.d, theta_base=r.theta_base, L_train=r.L_train,
                         L_target=r.L_target, s=r.s)
    q, k, v = W.prefill_inputs(w, "cuda")
    g = torch.Generator(device="cuda").manual_seed(902)
    dout = torch.randn(q.shape, generator=g, device="cuda").to(q.dtype)
    th, _, ms = R.inv_freq(r.kind, w.d, r.theta_base, r.L_train, r.L_target, r.s)
    scale = ms * ms / math.sqrt(w.d)
    pos = np.arange(w.S)
    qn, kn, vn, gn = f64(q), f64(k), f64(v), f64(dout)
    o_ref = np.zeros(qn.shape)
    lse_ref = np.zeros(qn.shape[:3])
    for b in range(w.B):
        for h in range(w.Hq):
            o_ref[b, h], lse_ref[b, h] = A.attention_rows(R.rotate(qn[b, h], pos, th), pos,
                                                          R.rotate(kn[b, h], pos, th), vn[b, h], w.mask, 0, 0,
                                                          scale)
    o_in = torch.from_numpy(o_ref).to("cuda", q.dtype)
    lse_in = torch.from_numpy(lse_ref).to("cuda", torch.float32).contiguous()
    dq, dk, dv = api.attn_bwd(cfg, q, k, v, o_in, dout, lse_in, mask=w.mask, out_dtype=torch.float32)
    torch.cuda.synchronize()
    units = w.B * w.Hq
    hg = _heads_per_group(units, w.S // 128)
    assert hg < units, "the case must span more than one scheduling group"
    for u in sorted({0, hg - 1, hg, units - 1}):
        b, h = divmod(u, w.Hq)
        want = A.backward_head(qn[b, h], kn[b, h], vn[b, h], gn[b, h], pos, pos, th, scale, w.mask)
        for got, ref, n in zip((dq[b, h], dk[b, h], dv[b, h]), want, ("dq", "dk", "dv")):
            _check(f64(got), ref, f"unit {u} (group {u // hg}) {n}")


def test_backward_full_size_sampled_rows():
    """The backward in the launch configuration the bench times: the
    Llama-2-7B shape (32 heads, S = 16384, causal, YaRN s = 4), O and LSE
    from the fused forward as the bench feeds them, several scheduling
    groups.  Sampled query rows (dq) and key rows (dk, dv) of a head in the
    first group, the first head of the second and the last head, against
    the row-sampled float64 oracle, which computes its own forward.  The bar
    is the one above; it also covers the forward's bf16 O entering
    D = rowsum(dO * O)."""
    need_cuda()
    w = W.LLAMA2_7B
    r = w.rope
    cfg = api.RopeConfig(kind=r.kind, head_dim=w.d, theta_base=r.theta_base, L_train=r.L_train,
                         L_target=r.L_target, s=r.s)
    q, k, v = W.prefill_inputs(w, "cuda")
    g = torch.Generator(device="cuda").manual_seed(901)
    dout = torch.randn(q.shape, generator=g, device="cuda").to(q.dtype)
    o, lse = api.attn_fwd_prefill(cfg, q, k, v, mask=w.mask, return_lse=True)
    dq, dk, dv = api.attn_bwd(cfg, q, k, v, o, dout, lse, mask=w.mask, out_dtype=torch.float32)
    torch.cuda.synchronize()
    th, _, ms = R.inv_freq(r.kind, w.d, r.theta_base, r.L_train, r.L_target, r.s)
    scale = ms * ms / math.sqrt(w.d)
    pos = np.arange(w.S)
    hg = _heads_per_group(w.B * w.Hq, w.S // 128)
    for h in sorted({0, min(hg, w.Hq - 1), w.Hq - 1}):
        rows_q = W.sample_rows(w.S, 48, h, extra=(4095, 4096, 8191)).numpy()
        rows_k = W.sample_rows(w.S, 48, 100 + h, extra=(4095, 4096, 16256)).numpy()
        sq, sk, sv = A.backward_sampled(f64(q[0, h]), f64(k[0, h]), f64(v[0, h]), f64(dout[0, h]), pos, th, scale,
                                        w.mask, rows_q, rows_k)
        _check(f64(dq[0, h, rows_q]), sq, f"head {h} dq rows")
        _check(f64(dk[0, h, rows_k]), sk, f"head {h} dk rows")
        _check(f64(dv[0, h, rows_k]), sv, f"head {h} dv rows")
