"""The per-device computation of ring attention on one GPU: attention of a
query block against one KV block at their own positions, exact merging of the
partials, and the whole ring schedule (query block I folds KV blocks I, I-1,
... and skips future blocks) against the fused kernel and the oracle."""

import math

import numpy as np
import pytest
import torch

import oracle.attention as A
import oracle.rope as R
from tests.helpers import assert_attn_close, assert_lse_close, f64, gpu, need_cuda
from yarn_rope_scaling_ntk_b300 import api, workloads as W

pytestmark = gpu

YARN = dict(kind="yarn", theta_base=1e4, L_train=256, s=4.0)


def _cfg(d):
    return api.RopeConfig(head_dim=d, **YARN)


def _oracle_block(q, k, v, q_pos0, k_pos0, mask, sink, window, d, G):
    th, _, ms = R.inv_freq("yarn", d, 1e4, 256, 0, 4.0)
    scale = ms * ms / math.sqrt(d)
    qn, kn, vn = f64(q), f64(k), f64(v)
    Sq, Skv = qn.shape[2], kn.shape[2]
    qp, kp = np.arange(Sq) + q_pos0, np.arange(Skv) + k_pos0
    out_o = np.zeros(qn.shape)
    out_l = np.zeros(qn.shape[:3])
    for b in range(qn.shape[0]):
        for h in range(qn.shape[1]):
            kr = R.rotate(kn[b, h // G], kp, th)
            qr = R.rotate(qn[b, h], qp, th)
            o, l = A.attention_rows(qr, qp, kr, vn[b, h // G], mask, sink, window, scale, k_pos=kp)
            out_o[b, h], out_l[b, h] = o, l
    return out_o, out_l


@pytest.mark.parametrize("mask,sink,window,q_pos0,k_pos0,Sq,Skv", [
    ("causal", 0, 0, 512, 256, 300, 256),        # block in the past, diagonal partly
    ("causal", 0, 0, 512, 512, 256, 384),        # diagonal block, keys beyond the rows
    ("causal", 0, 0, 100, 640, 128, 128),        # future block: empty
    ("sink_window", 4, 200, 700, 0, 256, 512),   # sinks + window edge inside the block
    ("none", 0, 0, 0, 333, 64, 200),
])
def test_kv_block_against_oracle(mask, sink, window, q_pos0, k_pos0, Sq, Skv):
    need_cuda()
    B, Hq, Hkv, d = 2, 4, 2, 128
    g = torch.Generator(device="cuda").manual_seed(q_pos0 + k_pos0 + Sq)
    q = torch.randn(B, Hq, Sq, d, generator=g, device="cuda").to(torch.bfloat16)
    k = torch.randn(B, Hkv, Skv, d, generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn(B, Hkv, Skv, d, generator=g, device="cuda").to(torch.bfloat16)
    o, lse = api.attn_fwd_prefill_kv_block(_cfg(d), q, k, v, q_pos0, k_pos0, mask=mask, sink=sink,
                                           window=window)
    torch.cuda.synchronize()
    want_o, want_l = _oracle_block(q, k, v, q_pos0, k_pos0, mask, sink, window, d, Hq // Hkv)
    assert_attn_close(f64(o), want_o, f"kv block {mask}")
    assert_lse_close(f64(lse), want_l, f"kv block {mask}")


@pytest.mark.parametrize("B,H,S,d,final_dtype", [(2, 3, 70, 128, torch.bfloat16),
                                                  (1, 5, 1001, 64, torch.float32),    # ragged row groups
                                                  (1, 2, 9, 256, torch.bfloat16)])    # two chunks per row
def test_merge_kernel_against_oracle(B, H, S, d, final_dtype):
    """Merge of two partials against the oracle's combination, with empty
    accumulator rows (NaN contents never read), empty partials and rows
    empty on both sides; rows taken several per warp in a grid-stride loop."""
    need_cuda()
    g = torch.Generator(device="cuda").manual_seed(5 + d)
    oa = torch.randn(B, H, S, d, generator=g, device="cuda")
    ob = torch.randn(B, H, S, d, generator=g, device="cuda")
    la = torch.randn(B, H, S, generator=g, device="cuda") * 3
    lb = torch.randn(B, H, S, generator=g, device="cuda") * 3
    n = B * H * S
    la.view(-1)[:5] = -math.inf               # accumulator empty: its O is never read
    oa.view(n, d)[:5] = float("nan")
    lb.view(-1)[n // 2:n // 2 + 4] = -math.inf  # partial empty
    la.view(-1)[n - 1] = lb.view(-1)[n - 1] = -math.inf   # both empty
    want_o, want_l = [], []
    for b in range(B):
        for h in range(H):
            o, l = A.merge_partials([(f64(oa[b, h]), f64(la[b, h])), (f64(ob[b, h]), f64(lb[b, h]))])
            want_o.append(o)
            want_l.append(l)
    final = torch.empty(B, H, S, d, dtype=final_dtype, device="cuda")
    api.attn_merge_partial(oa, la, ob, lb, out=final)
    torch.cuda.synchronize()
    got_o = f64(oa).reshape(-1, S, d)
    assert np.all(np.isfinite(got_o))
    np.testing.assert_allclose(got_o, np.stack(want_o), atol=1e-5, rtol=1e-5)
    gl, wl = f64(la).reshape(-1, S), np.stack(want_l)
    assert np.array_equal(np.isneginf(gl), np.isneginf(wl))
    np.testing.assert_allclose(np.where(np.isneginf(gl), 0, gl), np.where(np.isneginf(wl), 0, wl), atol=1e-5)
    assert torch.equal(final, oa.to(final_dtype))


@pytest.mark.parametrize("mask,sink,window", [("causal", 0, 0), ("sink_window", 4, 300)])
def test_ring_schedule_one_block_per_call_matches_fused_and_oracle(mask, sink, window):
    """Query block I takes KV blocks I, I-1, ... in ring order, skipping
    blocks j > I; each step computes a float32 partial and merges it."""
    need_cuda()
    w = W.Prefill("ring_steps", 70, 1, 4, 2, 1024, 128, torch.bfloat16, W.RopeSpec("yarn", 1e4, 256, 0, 4.0),
                  mask, sink, window)
    q, k, v = W.prefill_inputs(w, "cuda")
    N, bs = 4, w.S // 4
    cfg = _cfg(w.d)
    final = torch.empty_like(q)
    lse_all = torch.empty(w.B, w.Hq, w.S, dtype=torch.float32, device="cuda")
    for I in range(N):
        qi = q[:, :, I * bs:(I + 1) * bs]
        acc = torch.zeros(w.B, w.Hq, bs, w.d, dtype=torch.float32, device="cuda")
        lacc = torch.full((w.B, w.Hq, bs), -math.inf, dtype=torch.float32, device="cuda")
        order = [j for j in ((I - t) % N for t in range(N)) if j <= I]
        for step, j in enumerate(order):
            part, lpart = api.attn_fwd_prefill_kv_block(cfg, qi, k[:, :, j * bs:(j + 1) * bs],
                                                        v[:, :, j * bs:(j + 1) * bs], I * bs, j * bs,
                                                        mask=mask, sink=sink, window=window)
            api.attn_merge_partial(acc, lacc, part, lpart,
                                   out=final[:, :, I * bs:(I + 1) * bs] if step == len(order) - 1 else None)
        lse_all[:, :, I * bs:(I + 1) * bs] = lacc
    fused, fused_lse = api.attn_fwd_prefill(cfg, q, k, v, mask=mask, sink=sink, window=window, return_lse=True)
    torch.cuda.synchronize()
    assert (final.float() - fused.float()).abs().max().item() < 2e-2
    assert (lse_all - fused_lse).abs().max().item() < 1e-2
    th, _, ms = R.inv_freq("yarn", w.d, 1e4, 256, 0, 4.0)
    scale = ms * ms / math.sqrt(w.d)
    got, want = [], []
    for h in range(w.Hq):
        rows = W.sample_rows(w.S, 64, h, extra=(bs - 1, bs, 2 * bs, 3 * bs + 1)).numpy()
        kr = R.rotate(f64(k[0, h // 2]), np.arange(w.S), th)
        qr = R.rotate(f64(q[0, h, rows]), rows, th)
        o, _ = A.attention_rows(qr, rows, kr, f64(v[0, h // 2]), mask, sink, window, scale)
        got.append(f64(final[0, h, rows]))
        want.append(o)
    assert_attn_close(np.concatenate(got), np.concatenate(want), "ring steps")


def test_empty_kv_block_gives_empty_rows():
    need_cuda()
    q = torch.randn(1, 2, 40, 64, device="cuda").to(torch.bfloat16)
    k = torch.empty(1, 2, 0, 64, device="cuda", dtype=torch.bfloat16)
    o, lse = api.attn_fwd_prefill_kv_block(_cfg(64), q, k, k, 10, 0)
    torch.cuda.synchronize()
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))


def test_ring_blocks_full_size_sampled_rows():
    """The ring 128K workload in the launch configuration the bench times
    for the building blocks: Q and K rotated once by rope_apply, then query
    block I takes KV blocks I, I-1, ..., 0 of the rotated operands (kind
    "none", the YaRN softmax scale passed explicitly), one
    attn_fwd_prefill_kv_block call each into float32 partials merged by
    attn_merge_partial, the last merge writing bf16.  Sampled rows of three
    heads, with the block edges, against the float64 oracle."""
    need_cuda()
    w = W.RING_128K
    r = w.rope
    cfg_rot = api.RopeConfig(kind=r.kind, head_dim=w.d, theta_base=r.theta_base, L_train=r.L_train,
                             L_target=r.L_target, s=r.s)
    _, _, mscale = api.yarn_inv_freq(cfg_rot)
    cfg = api.RopeConfig(kind="none", head_dim=w.d)
    scale = mscale * mscale / math.sqrt(w.d)
    q0, k0, v = W.prefill_inputs(w, "cuda")
    q, k = api.rope_apply(cfg_rot, q0), api.rope_apply(cfg_rot, k0)
    N, bs = w.ring_blocks, w.S // w.ring_blocks
    final = torch.empty_like(q0)
    acc = torch.empty(w.B, w.Hq, bs, w.d, dtype=torch.float32, device="cuda")
    part, lacc, lpart = torch.empty_like(acc), acc.new_empty(w.B, w.Hq, bs), acc.new_empty(w.B, w.Hq, bs)
    for I in range(N):
        rows = slice(I * bs, (I + 1) * bs)
        for step, j in enumerate(range(I, -1, -1)):
            keys = slice(j * bs, (j + 1) * bs)
            last = j == 0
            if step == 0:
                api.attn_fwd_prefill_kv_block(cfg, q[:, :, rows], k[:, :, keys], v[:, :, keys], I * bs, j * bs,
                                              softmax_scale=scale, out=final[:, :, rows] if last else acc,
                                              lse=lacc)
                continue
            api.attn_fwd_prefill_kv_block(cfg, q[:, :, rows], k[:, :, keys], v[:, :, keys], I * bs, j * bs,
                                          softmax_scale=scale, out=part, lse=lpart)
            api.attn_merge_partial(acc, lacc, part, lpart, out=final[:, :, rows] if last else None)
    torch.cuda.synchronize()
    api.sync_status()
    th, _, ms = R.inv_freq(r.kind, w.d, r.theta_base, r.L_train, r.L_target, r.s)
    oscale = ms * ms / math.sqrt(w.d)
    pos = np.arange(w.S)
    edges = tuple(x for I in range(1, N) for x in (I * bs - 1, I * bs))
    got, want = [], []
    for h in (0, 13, 31):
        rws = W.sample_rows(w.S, 24, 200 + h, extra=edges).numpy()
        kr = R.rotate(f64(k0[0, h]), pos, th)
        qr = R.rotate(f64(q0[0, h, rws]), rws, th)
        o, _ = A.attention_rows(qr, rws, kr, f64(v[0, h]), w.mask, 0, 0, oscale)
        got.append(f64(final[0, h, rws]))
        want.append(o)
    assert_attn_close(np.concatenate(got), np.concatenate(want), "ring blocks 128K")


@pytest.mark.parametrize("world,mask,sink,window,Hq,Hkv", [(4, "causal", 0, 0, 4, 2), (3, "none", 0, 0, 2, 2),
                                                           (4, "sink_window", 4, 300, 4, 1)])
def test_ring_driver_all_ranks_in_one_process(world, mask, sink, window, Hq, Hkv):
    """The ring driver's per-rank computation with the library's kernels, all
    ranks of a ring run in lock step on one GPU (the exchange is a hand-over
    of the rotated blocks): every row of every rank against the oracle, and
    against the fused call in ring order."""
    need_cuda()
    from yarn_rope_scaling_ntk_b300 import ring
    B, bs, d = 1, 256, 128
    S = bs * world
    g = torch.Generator(device="cuda").manual_seed(4100 + world)
    q = torch.randn(B, Hq, S, d, generator=g, device="cuda").to(torch.bfloat16)
    k = torch.randn(B, Hkv, S, d, generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn(B, Hkv, S, d, generator=g, device="cuda").to(torch.bfloat16)
    blocks = lambda t: [t[:, :, i * bs:(i + 1) * bs].contiguous() for i in range(world)]
    res = ring.ring_attention_one_process(_cfg(d), blocks(q), blocks(k), blocks(v), mask=mask, sink=sink,
                                          window=window)
    api.sync_status()
    o = torch.cat([r[0] for r in res], dim=2)
    lse = torch.cat([r[1] for r in res], dim=2)
    want_o, want_l = _oracle_block(q, k, v, 0, 0, mask, sink, window, d, Hq // Hkv)
    assert_attn_close(f64(o), want_o, f"ring driver, {world} ranks")
    assert_lse_close(f64(lse), want_l, f"ring driver, {world} ranks")
    fused = api.attn_fwd_prefill(_cfg(d), q, k, v, mask=mask, sink=sink, window=window, ring_blocks=world)
    assert (fused.float() - o.float()).abs().max().item() < 2e-2
