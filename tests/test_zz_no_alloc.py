"""The allocation-free decode entry point against the workspace one.

attn_fwd_decode_sinkwindow_noalloc serves callers that cannot allocate device
memory when they call (an engine hook that must not allocate, a process whose
memory another allocator holds): its split scratch is the library's own fixed
device array.  This file is collected last so that a failure here stops a
first-failure run only after every other test has run; it also passes alone
in a fresh process.
"""

import ctypes

import numpy as np
import pytest
import torch

from tests.helpers import assert_attn_close, f64, gpu, need_cuda
from yarn_rope_scaling_ntk_b300 import api, workloads as W

pytestmark = gpu


def _inputs(index, B, Hq, Hkv, sink, window):
    w = W.Decode(f"noalloc{index}", index, B, Hq, Hkv, 128, sink, window,
                 W.RopeSpec("yarn", 1e4, 256, 0, 4.0), full=False)
    return w, W.decode_inputs(w, "cuda")


def _call_noalloc(lib, cfg, w, inp, num_splits):
    """Through the C ABI, with caller-owned outputs and no workspace."""
    q, kc, vc, nv, rs = inp
    o = torch.empty_like(q)
    lse = torch.empty(w.B, w.Hq, dtype=torch.float32, device="cuda")
    c = cfg.c()
    st = lib.attn_fwd_decode_sinkwindow_noalloc(
        ctypes.byref(c), q.data_ptr(), kc.data_ptr(), vc.data_ptr(), nv.data_ptr(), rs.data_ptr(),
        w.B, w.Hq, w.Hkv, w.d, w.sink, w.window, o.data_ptr(), lse.data_ptr(), num_splits,
        torch.cuda.current_stream().cuda_stream)
    return st, o, lse


def test_noalloc_matches_workspace_entry_on_two_calls_in_a_row():
    need_cuda()
    lib = api.load_library()
    cfg = api.RopeConfig(kind="yarn", head_dim=128, L_train=256, s=4.0)
    cases = [(_inputs(71, 4, 32, 8, 4, 4092), 0),   # auto split count (8 slices)
             (_inputs(72, 3, 16, 16, 4, 1500), 5)]  # another shape, 5 slices
    for (w, inp), splits in cases:
        assert api.decode_workspace_bytes(w.B, w.Hq, w.Hkv, w.d, w.sink, w.window, splits) > 0
        q, kc, vc, nv, rs = inp
        want_o, want_l = api.attn_fwd_decode_sinkwindow(cfg, q, kc, vc, nv, rs, w.sink, w.window,
                                                        num_splits=splits, return_lse=True)
        st, o, lse = _call_noalloc(lib, cfg, w, inp, splits)
        assert st == 0, lib.yr_last_error_message()
        api.sync_status()
        assert_attn_close(f64(o), f64(want_o), "noalloc vs workspace entry")
        np.testing.assert_allclose(f64(lse), f64(want_l), atol=1e-2)


def test_noalloc_rejects_scratch_above_its_limit():
    need_cuda()
    lib = api.load_library()
    cfg = api.RopeConfig(kind="plain", head_dim=128)
    w, inp = _inputs(73, 64, 32, 32, 4, 4092)
    # 64 splits x 64 x 32 x 130 x 4 bytes is far above the fixed array
    st, _, _ = _call_noalloc(lib, cfg, w, inp, 64)
    assert st == 1 and b"scratch" in lib.yr_last_error_message()


def test_noalloc_python_wrapper_on_the_gpu():
    """The Python wrapper of the allocation-free entry, with caller-owned
    outputs, against the workspace entry (a split count that needs scratch)."""
    need_cuda()
    cfg = api.RopeConfig(kind="plain", head_dim=128)
    w, inp = _inputs(74, 2, 8, 4, 4, 700)
    q, kc, vc, nv, rs = inp
    want_o, want_l = api.attn_fwd_decode_sinkwindow(cfg, q, kc, vc, nv, rs, w.sink, w.window, num_splits=3,
                                                    return_lse=True)
    o = torch.empty_like(q)
    lse = torch.empty(w.B, w.Hq, dtype=torch.float32, device="cuda")
    api.attn_fwd_decode_sinkwindow_noalloc(cfg, q, kc, vc, nv, rs, w.sink, w.window, num_splits=3, out=o, lse=lse)
    api.sync_status()
    assert_attn_close(f64(o), f64(want_o), "noalloc wrapper vs workspace entry")
    np.testing.assert_allclose(f64(lse), f64(want_l), atol=1e-2)
