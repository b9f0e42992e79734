"""Host-side checks of the C-ABI library that need no GPU: it loads, exports
every symbol the header declares, computes the float64 frequency table like
the oracle (classes bit-exact), and rejects bad arguments before any launch."""

import ctypes
import os
import re

import numpy as np
import pytest
import torch

import oracle.rope as R
from yarn_rope_scaling_ntk_b300 import api
from yarn_rope_scaling_ntk_b300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build()
    return api.load_library()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "yarn_attn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(", text, flags=re.M)))


def test_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert {"yarn_inv_freq", "rope_apply", "attn_fwd_prefill", "attn_fwd_decode_sinkwindow"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
    assert lib.yr_version().decode().startswith("yarn_attn")


CASES = [("plain", 64, 1e4, 64, 0, 0.0), ("pi", 64, 1e4, 64, 256, 0.0), ("ntk", 64, 1e4, 64, 256, 0.0),
         ("yarn", 64, 1e4, 64, 256, 0.0), ("yarn", 128, 1e4, 4096, 16384, 0.0),
         ("yarn", 128, 1e4, 4096, 0, 32.0), ("yarn", 128, 5e5, 8192, 32768, 0.0),
         ("ntk", 128, 1e4, 4096, 0, 8.0), ("none", 128, 1e4, 4096, 0, 4.0), ("yarn", 128, 1e4, 4096, 0, 1.0),
         ("yarn", 256, 1e6, 32768, 0, 16.0), ("pi", 16, 500.0, 100, 0, 3.0)]


@pytest.mark.parametrize("kind,d,b,L,Lt,s", CASES)
def test_inv_freq_matches_oracle(lib, kind, d, b, L, Lt, s):
    cfg = api.RopeConfig(kind=kind, head_dim=d, theta_base=b, L_train=L, L_target=Lt, s=s)
    th, cls, ms = api.yarn_inv_freq(cfg)
    th_o, cls_o, ms_o = R.inv_freq(kind, d, b, L, Lt, s)
    np.testing.assert_array_equal(cls, cls_o)            # integer classes: bit-exact
    np.testing.assert_allclose(th, th_o, rtol=1e-12, atol=0)
    assert ms == pytest.approx(ms_o, rel=1e-15)


def test_inv_freq_errors(lib):
    bad = [api.RopeConfig(kind="yarn", head_dim=128, L_train=0, s=4.0),      # YaRN without L_train
           api.RopeConfig(kind="pi", head_dim=128, L_train=0, L_target=0),   # no scale
           api.RopeConfig(kind="plain", head_dim=7),                         # odd d
           api.RopeConfig(kind="plain", head_dim=128, theta_base=1.0),       # base <= 1
           api.RopeConfig(kind="yarn", head_dim=128, L_train=4096, s=4.0, ramp_alpha=5, ramp_beta=2)]
    for cfg in bad:
        with pytest.raises(api.YarnAttnError) as e:
            api.yarn_inv_freq(cfg)
        assert e.value.status == 1


def _i64(*v):
    return (ctypes.c_int64 * 3)(*v)


def test_argument_errors_before_launch(lib):
    cfg = api.RopeConfig(kind="yarn", head_dim=96, L_train=4096, s=4.0).c()
    st = lib.attn_fwd_prefill(ctypes.byref(cfg), None, None, None, None, None, 1, 1, 4, 4, 128, 96,
                              _i64(0, 0, 0), _i64(0, 0, 0), _i64(0, 0, 0), _i64(0, 0, 0), 0, 0, 0,
                              1, 0.0, None, 0, None)
    assert st == 2 and b"head dimension" in lib.yr_last_error_message()
    cfg = api.RopeConfig(kind="yarn", head_dim=128, L_train=4096, s=4.0).c()
    # Hq % Hkv != 0
    st = lib.attn_fwd_prefill(ctypes.byref(cfg), None, None, None, None, None, 1, 1, 6, 4, 128, 128,
                              _i64(0, 0, 0), _i64(0, 0, 0), _i64(0, 0, 0), _i64(0, 0, 0), 0, 0, 0,
                              1, 0.0, None, 0, None)
    assert st == 1
    # null pointers with work to do
    st = lib.attn_fwd_prefill(ctypes.byref(cfg), None, None, None, None, None, 1, 1, 4, 4, 128, 128,
                              _i64(0, 0, 0), _i64(0, 0, 0), _i64(0, 0, 0), _i64(0, 0, 0), 0, 0, 0,
                              1, 0.0, None, 0, None)
    assert st == 1
    # misaligned pointer
    st = lib.attn_fwd_prefill(ctypes.byref(cfg), ctypes.c_void_p(8), ctypes.c_void_p(16),
                              ctypes.c_void_p(16), ctypes.c_void_p(16), None, 1, 1, 4, 4, 128, 128,
                              _i64(0, 0, 128), _i64(0, 0, 128), _i64(0, 0, 128), _i64(0, 0, 128),
                              0, 0, 0, 1, 0.0, None, 0, None)
    assert st == 1
    # sink + window mask with window < 1
    st = lib.attn_fwd_prefill(ctypes.byref(cfg), None, None, None, None, None, 1, 1, 4, 4, 128, 128,
                              _i64(0, 0, 0), _i64(0, 0, 0), _i64(0, 0, 0), _i64(0, 0, 0), 1, 4, 0,
                              1, 0.0, None, 0, None)
    assert st == 1
    # ring blocks that do not divide S
    st = lib.attn_fwd_prefill(ctypes.byref(cfg), None, None, None, None, None, 1, 1, 4, 4, 100, 128,
                              _i64(0, 0, 0), _i64(0, 0, 0), _i64(0, 0, 0), _i64(0, 0, 0), 0, 0, 0,
                              3, 0.0, None, 0, None)
    assert st == 1
    # decode: GQA ratio outside {1, 2, 4, 8}; missing workspace for forced splits
    st = lib.attn_fwd_decode_sinkwindow(ctypes.byref(cfg), None, None, None, None, None, 2, 12, 4,
                                        128, 4, 60, None, None, 0, None, 0, None)
    assert st == 2
    st = lib.attn_fwd_decode_sinkwindow(ctypes.byref(cfg), ctypes.c_void_p(16), ctypes.c_void_p(16),
                                        ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16),
                                        2, 4, 4, 128, 4, 60, ctypes.c_void_p(16), None, 3, None, 0, None)
    assert st == 1 and b"workspace" in lib.yr_last_error_message()
    # rope_apply: unsupported d
    st = lib.rope_apply(ctypes.byref(api.RopeConfig(kind="plain", head_dim=48).c()), None, None, 1,
                        1, 1, 1, 48, _i64(0, 0, 0), _i64(0, 0, 0), 0, None, 0, None)
    assert st == 2


def test_empty_inputs_return_ok_without_launch(lib):
    cfg = api.RopeConfig(kind="yarn", head_dim=128, L_train=4096, s=4.0).c()
    st = lib.attn_fwd_prefill(ctypes.byref(cfg), None, None, None, None, None, 1, 0, 4, 4, 128, 128,
                              _i64(0, 0, 0), _i64(0, 0, 0), _i64(0, 0, 0), _i64(0, 0, 0), 0, 0, 0,
                              1, 0.0, None, 0, None)
    assert st == 0
    st = lib.rope_apply(ctypes.byref(cfg), None, None, 1, 0, 4, 16, 128, _i64(0, 0, 0), _i64(0, 0, 0),
                        0, None, 0, None)
    assert st == 0


def test_every_entry_point_accepts_empty_inputs(lib):
    """A zero batch or a zero length is a valid call with nothing to do: each
    entry point returns YR_OK before it touches a pointer or launches."""
    cfg = api.RopeConfig(kind="yarn", head_dim=128, L_train=4096, s=4.0).c()
    z = lambda: _i64(0, 0, 0)
    n0 = lib.yr_kernel_launch_count()
    # prefill: B = 0
    assert lib.attn_fwd_prefill(ctypes.byref(cfg), None, None, None, None, None, 1, 0, 4, 4, 256, 128,
                                z(), z(), z(), z(), 0, 0, 0, 1, 0.0, None, 0, None) == 0
    # one KV block with no queries (a block with queries but no keys is not
    # empty: it writes o = 0 and lse = -inf, and needs its pointers)
    none = api.RopeConfig(kind="none", head_dim=128).c()
    assert lib.attn_fwd_prefill_kv_block(ctypes.byref(none), None, None, None, None, None, 1, 0, 1, 4, 4, 0, 128,
                                         128, 0, 0, z(), z(), z(), z(), 0, 0, 0, 0.0, None, 0, None) == 0
    assert lib.attn_fwd_prefill_kv_block(ctypes.byref(none), None, None, None, None, None, 1, 0, 1, 4, 4, 128, 0,
                                         128, 0, 0, z(), z(), z(), z(), 0, 0, 0, 0.0, None, 0, None) == 1
    # decode, bf16 and FP8 caches: B = 0
    assert lib.attn_fwd_decode_sinkwindow(ctypes.byref(cfg), None, None, None, None, None, 0, 32, 8, 128, 4,
                                          4092, None, None, 0, None, 0, None) == 0
    assert lib.attn_fwd_decode_sinkwindow_fp8(ctypes.byref(cfg), None, None, None, None, None, None, None, 0, 32,
                                              8, 128, 4, 4092, None, None, 0, None, 0, None) == 0
    # merge: S = 0
    assert lib.attn_merge_partial(None, None, None, None, None, 0, 1, 4, 0, 128, z(), z(), z(), None) == 0
    # backward: S = 0
    assert lib.attn_bwd(ctypes.byref(cfg), None, None, None, None, None, None, None, None, None, 1, 1, 1, 4, 4, 0,
                        128, z(), z(), z(), z(), z(), z(), z(), z(), 0, 0, 0, 0.0, None, 0, None) == 0
    assert lib.yr_kernel_launch_count() == n0


def test_workspace_sizes(lib):
    cfg = api.RopeConfig(kind="yarn", head_dim=128, L_train=4096, s=4.0)
    assert api.prefill_workspace_bytes(cfg, torch.bfloat16, 1, 32, 8, 1024, 128) >= 8 * 1024 * 128 * 2
    assert api.prefill_workspace_bytes(api.RopeConfig(kind="none"), torch.bfloat16, 1, 32, 8, 1024, 128) == 0
    assert lib.yr_decode_auto_splits(64, 32, 4, 4092) == 1
    assert lib.yr_decode_auto_splits(1, 8, 4, 4092) > 1
    assert api.decode_workspace_bytes(64, 32, 32, 128, 4, 4092) == 0
    assert api.decode_workspace_bytes(2, 8, 8, 128, 4, 4092, 4) == 4 * 2 * 8 * 130 * 4


def test_library_is_the_product_path():
    """The binding refuses to run when the library is missing (no fallback)."""
    import importlib
    src = open(os.path.join(ROOT, "yarn_rope_scaling_ntk_b300", "api.py")).read()
    assert "oracle" not in src
    for f in os.listdir(os.path.join(ROOT, "yarn_rope_scaling_ntk_b300")):
        if f.endswith(".py"):
            assert "import oracle" not in open(os.path.join(ROOT, "yarn_rope_scaling_ntk_b300", f)).read()
    assert importlib.util.find_spec("yarn_rope_scaling_ntk_b300.api") is not None


def test_perdim_inv_freq_matches_oracle_and_rejects_bad_vectors(lib):
    lam = np.concatenate([np.ones(16), np.linspace(1.0, 6.0, 32), np.full(16, 6.0)])
    cfg = api.RopeConfig(kind="perdim", head_dim=128, L_train=4096, dim_scale=tuple(lam))
    th, cls, ms = api.yarn_inv_freq(cfg)
    th_o, cls_o, ms_o = R.inv_freq("perdim", 128, 1e4, 4096, dim_scale=lam)
    np.testing.assert_array_equal(cls, cls_o)
    np.testing.assert_allclose(th, th_o, rtol=1e-15, atol=0)
    assert ms == ms_o == 1.0
    for bad in (None, tuple([1.0] * 63 + [0.0]), tuple([1.0] * 63 + [float("inf")]), tuple([-1.0] * 64)):
        with pytest.raises(api.YarnAttnError) as e:
            api.yarn_inv_freq(api.RopeConfig(kind="perdim", head_dim=128, L_train=4096, dim_scale=bad))
        assert e.value.status == 1


def test_noalloc_reports_argument_errors_before_its_size_limit(lib):
    """The allocation-free decode entry reports the same argument errors as
    the workspace entry, even when the split count it is given would also
    exceed its fixed scratch array; no pointer is touched."""
    cfg = api.RopeConfig(kind="plain", head_dim=128).c()
    args = lambda B, Hq, Hkv, d, splits: (ctypes.byref(cfg), None, None, None, None, None, B, Hq, Hkv, d, 4,
                                          4092, None, None, splits, None)
    # Hq % Hkv != 0 with 4000 splits (far above the array): the shape error wins
    assert lib.attn_fwd_decode_sinkwindow_noalloc(*args(64, 30, 8, 128, 4000)) == 1
    assert b"Hq % Hkv" in lib.yr_last_error_message()
    # unsupported head dimension
    assert lib.attn_fwd_decode_sinkwindow_noalloc(*args(64, 32, 32, 96, 4000)) == 2
    assert b"head dimension" in lib.yr_last_error_message()
    # num_splits above the entry points' limit
    assert lib.attn_fwd_decode_sinkwindow_noalloc(*args(64, 32, 32, 128, 5000)) == 1
    assert b"num_splits" in lib.yr_last_error_message()
    # a valid shape whose split scratch exceeds the array
    assert lib.attn_fwd_decode_sinkwindow_noalloc(*args(64, 32, 32, 128, 64)) == 1
    assert b"scratch" in lib.yr_last_error_message()


def test_noalloc_python_wrapper_validates_like_its_sibling(lib):
    """The Python wrapper of the allocation-free entry checks shapes, dtypes
    and layouts before it calls the library (CPU tensors: the shape errors
    come before the device check)."""
    cfg = api.RopeConfig(kind="plain", head_dim=128)
    B, H, d, sink, win = 2, 4, 128, 4, 60
    q = torch.zeros(B, H, d, dtype=torch.bfloat16)
    kc = torch.zeros(B, H, sink + win, d, dtype=torch.bfloat16)
    nv = torch.full((B,), sink + win, dtype=torch.int32)
    rs = torch.zeros(B, dtype=torch.int32)
    bad = [
        dict(k_cache=kc[:, :, :-1].contiguous()),              # cache shorter than sink + window
        dict(q=q.float()),                                       # float32 query
        dict(v_cache=kc.transpose(2, 3).contiguous().transpose(2, 3)),  # not contiguous
        dict(n_valid=nv.long()),                                 # int64 counts
        dict(out=torch.zeros(B, H, d, dtype=torch.float32)),     # wrong output dtype
        dict(lse=torch.zeros(B, H + 1, dtype=torch.float32)),    # wrong lse shape
        dict(),                                                  # CPU tensors
    ]
    for change in bad:
        a = dict(q=q, k_cache=kc, v_cache=kc, n_valid=nv, ring_start=rs, out=None, lse=None)
        a.update(change)
        with pytest.raises(ValueError):
            api.attn_fwd_decode_sinkwindow_noalloc(cfg, a["q"], a["k_cache"], a["v_cache"], a["n_valid"],
                                                   a["ring_start"], sink, win, out=a["out"], lse=a["lse"])


def test_fault_injection_hook_checks_its_arguments(lib):
    assert lib.yr_debug_inject_wait_fault(-1, -1) == 1
    assert lib.yr_debug_inject_wait_fault(0, -2) == 1
    assert lib.yr_debug_inject_wait_fault(1000, 3) == 0
    assert lib.yr_debug_inject_wait_fault(0, -1) == 0  # off again


def test_launch_counter_does_not_count_refused_calls(lib):
    n = lib.yr_kernel_launch_count()
    cfg = api.RopeConfig(kind="yarn", head_dim=96, L_train=4096, s=4.0).c()
    assert lib.attn_fwd_prefill(ctypes.byref(cfg), None, None, None, None, None, 1, 1, 4, 4, 128, 96,
                                _i64(0, 0, 0), _i64(0, 0, 0), _i64(0, 0, 0), _i64(0, 0, 0), 0, 0, 0,
                                1, 0.0, None, 0, None) == 2
    assert lib.yr_kernel_launch_count() == n
