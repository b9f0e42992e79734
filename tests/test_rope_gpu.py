"""rope_apply on the GPU against the float64 oracle."""

import numpy as np
import pytest
import torch

import oracle.rope as R
from tests.helpers import ROPE_F32_ATOL, f64, gpu, need_cuda, rope_bf16_bound
from yarn_rope_scaling_ntk_b300 import api, workloads as W

pytestmark = gpu


def _cfg(kind, d, b, L, Lt=0, s=0.0):
    return api.RopeConfig(kind=kind, head_dim=d, theta_base=b, L_train=L, L_target=Lt, s=s)


@pytest.mark.parametrize("kind", ["plain", "pi", "ntk", "yarn", "none"])
@pytest.mark.parametrize("apply_mscale", [False, True])
def test_rope_f32_tiny_all_rows(kind, apply_mscale):
    need_cuda()
    w = W.TINY
    q, _, _ = W.prefill_inputs(w, "cuda")
    cfg = _cfg(kind, w.d, w.rope.theta_base, w.rope.L_train, w.rope.L_target)
    y = api.rope_apply(cfg, q, apply_mscale=apply_mscale)
    torch.cuda.synchronize()
    want = R.rope_apply(f64(q), np.arange(w.S), kind, w.d, w.rope.theta_base, w.rope.L_train,
                        w.rope.L_target, 0.0, apply_mscale=apply_mscale)
    assert np.abs(f64(y) - want).max() <= ROPE_F32_ATOL


def test_rope_f32_long_positions_sampled():
    # positions up to 131071 at s = 32: the angle reduction must stay exact enough
    need_cuda()
    g = torch.Generator(device="cuda").manual_seed(41)
    S, d = 131072, 128
    x = torch.randn(1, 2, S, d, generator=g, device="cuda")
    cfg = _cfg("yarn", d, 1e4, 4096, s=32.0)
    y = api.rope_apply(cfg, x)
    rows = W.sample_rows(S, 2048, 41, extra=(S - 2, 65535, 65536, 100000))
    th, _, _ = R.inv_freq("yarn", d, 1e4, 4096, 0, 32.0)
    want = R.rotate(f64(x[:, :, rows]), rows.numpy(), th)
    assert np.abs(f64(y[:, :, rows]) - want).max() <= ROPE_F32_ATOL
    # plain RoPE (fastest dimension turns once per 2 pi positions) as well
    y2 = api.rope_apply(_cfg("plain", d, 1e4, 4096), x)
    want2 = R.rotate(f64(x[:, :, rows]), rows.numpy(), R.base_frequencies(d, 1e4))
    assert np.abs(f64(y2[:, :, rows]) - want2).max() <= ROPE_F32_ATOL


@pytest.mark.parametrize("wl", [W.LLAMA2_7B, W.RING_128K])
def test_rope_bf16_within_one_ulp(wl):
    need_cuda()
    g = torch.Generator(device="cuda").manual_seed(wl.index)
    x = torch.randn(1, 4, wl.S, wl.d, generator=g, device="cuda").to(torch.bfloat16)
    cfg = _cfg(wl.rope.kind, wl.d, wl.rope.theta_base, wl.rope.L_train, wl.rope.L_target)
    y = api.rope_apply(cfg, x)
    rows = W.sample_rows(wl.S, 1024, wl.index, extra=(wl.S // 2,))
    th, _, _ = R.inv_freq(wl.rope.kind, wl.d, wl.rope.theta_base, wl.rope.L_train, wl.rope.L_target)
    want = R.rotate(f64(x[:, :, rows]), rows.numpy(), th)
    got = f64(y[:, :, rows])
    assert np.all(np.abs(got - want) <= rope_bf16_bound(want, f64(x[:, :, rows])))


def test_rope_bench_launch_q_and_k_stacked():
    """The launch the bench times: Q and K of the Llama-2-7B-shaped workload
    stacked along the heads, [1, 64, 16384, 128] bf16, in one call; sampled
    rows of every head within the bf16 rotation bar of the oracle."""
    need_cuda()
    wl = W.LLAMA2_7B
    q, k, _ = W.prefill_inputs(wl, "cuda")
    qk = torch.cat([q, k], dim=1)
    cfg = _cfg(wl.rope.kind, wl.d, wl.rope.theta_base, wl.rope.L_train, wl.rope.L_target)
    y = api.rope_apply(cfg, qk)
    rows = W.sample_rows(wl.S, 512, wl.index + 7, extra=(wl.S // 2,))
    th, _, _ = R.inv_freq(wl.rope.kind, wl.d, wl.rope.theta_base, wl.rope.L_train, wl.rope.L_target)
    want = R.rotate(f64(qk[:, :, rows]), rows.numpy(), th)
    got = f64(y[:, :, rows])
    assert got.shape == (1, 2 * wl.Hq, len(rows), wl.d)
    assert np.all(np.abs(got - want) <= rope_bf16_bound(want, f64(qk[:, :, rows])))


def test_rope_positions_pos0_inplace_and_strides():
    need_cuda()
    g = torch.Generator(device="cuda").manual_seed(5)
    B, S, H, d = 2, 300, 3, 128
    base = torch.randn(B, S, H, d, generator=g, device="cuda")   # [B, S, H, d] storage
    x = base.transpose(1, 2)                                       # [B, H, S, d] view, strided
    cfg = _cfg("ntk", d, 1e4, 4096, s=8.0)
    th, _, _ = R.inv_freq("ntk", d, 1e4, 4096, 0, 8.0)
    # pos0 offset
    y = api.rope_apply(cfg, x, pos0=12345)
    want = R.rotate(f64(x), np.arange(S) + 12345, th)
    assert np.abs(f64(y) - want).max() <= ROPE_F32_ATOL
    # explicit positions
    pos = torch.randint(0, 1 << 20, (S,), generator=g, device="cuda", dtype=torch.int32)
    y = api.rope_apply(cfg, x, positions=pos)
    want = R.rotate(f64(x), pos.cpu().numpy(), th)
    assert np.abs(f64(y) - want).max() <= ROPE_F32_ATOL
    # in place on the strided view
    ref = f64(x)
    api.rope_apply(cfg, x, out=x)
    torch.cuda.synchronize()
    assert np.abs(f64(x) - R.rotate(ref, np.arange(S), th)).max() <= ROPE_F32_ATOL


def test_rope_small_and_empty():
    need_cuda()
    cfg = _cfg("yarn", 64, 1e4, 64, s=4.0)
    x = torch.randn(1, 1, 1, 64, device="cuda")
    y = api.rope_apply(cfg, x)
    th, _, _ = R.inv_freq("yarn", 64, 1e4, 64, 0, 4.0)
    assert np.abs(f64(y) - R.rotate(f64(x), [0], th)).max() <= ROPE_F32_ATOL
    e = torch.empty(0, 2, 5, 64, device="cuda")
    assert api.rope_apply(cfg, e).shape == e.shape
    for d in (16, 32, 256):
        x = torch.randn(2, 2, 33, d, device="cuda")
        y = api.rope_apply(_cfg("plain", d, 1e4, 0), x, pos0=7)
        want = R.rotate(f64(x), np.arange(33) + 7, R.base_frequencies(d, 1e4))
        assert np.abs(f64(y) - want).max() <= ROPE_F32_ATOL


def test_rope_perdim_scale_vector_f32():
    """A per-dimension scale vector (LongRoPE's form) through the rotation."""
    need_cuda()
    w = W.TINY
    q, _, _ = W.prefill_inputs(w, "cuda")
    lam = np.concatenate([np.ones(8), np.linspace(1.0, 4.0, 16), np.full(8, 4.0)])
    cfg = api.RopeConfig(kind="perdim", head_dim=w.d, theta_base=w.rope.theta_base, L_train=w.rope.L_train,
                         dim_scale=tuple(lam))
    y = api.rope_apply(cfg, q, pos0=1000)
    torch.cuda.synchronize()
    want = R.rope_apply(f64(q), np.arange(w.S) + 1000, "perdim", w.d, w.rope.theta_base, w.rope.L_train,
                        dim_scale=lam)
    assert np.abs(f64(y) - want).max() <= ROPE_F32_ATOL
