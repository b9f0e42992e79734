"""Python binding of ``libyarn_attn.so`` (ctypes).

Argument marshalling only: tensors become raw pointers and strides, the
caller's current CUDA stream is passed through, and every step of the path
runs in the library's kernels.  PyTorch provides device memory (outputs and
workspaces) and streams.  There is no CPU fallback: if the library is missing
or a call fails, an exception is raised.
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_NAME = "libyarn_attn.so"

KIND = {"none": 0, "plain": 1, "pi": 2, "ntk": 3, "yarn": 4, "perdim": 5}
MASK = {"causal": 0, "sink_window": 1, "none": 2}
F32, BF16 = 0, 1
STATUS = {0: "YR_OK", 1: "YR_ERR_INVALID_ARG", 2: "YR_ERR_UNSUPPORTED", 3: "YR_ERR_CUDA",
          4: "YR_ERR_TIMEOUT"}


class YarnAttnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


class _Cfg(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("theta_base", ctypes.c_double), ("L_train", ctypes.c_int32),
                ("L_target", ctypes.c_int32), ("s", ctypes.c_double),
                ("ramp_alpha", ctypes.c_double), ("ramp_beta", ctypes.c_double),
                ("mscale_override", ctypes.c_double), ("dim_scale", ctypes.POINTER(ctypes.c_double))]


@dataclass(frozen=True)
class RopeConfig:
    """The pages' problem statement: rescaling kind, head dim d, base b,
    L_train, L_target, scale s (<= 0: L_target / L_train), YaRN ramp bounds,
    an optional temperature override, and (kind "perdim") the d/2 factors of
    a per-dimension scale vector."""
    kind: str = "yarn"
    head_dim: int = 128
    theta_base: float = 10000.0
    L_train: int = 0
    L_target: int = 0
    s: float = 0.0
    ramp_alpha: float = 1.0
    ramp_beta: float = 32.0
    mscale_override: float = 0.0
    dim_scale: tuple | None = None

    def c(self) -> _Cfg:
        if self.kind not in KIND:
            raise ValueError(f"unknown rope kind {self.kind!r}")
        cfg = _Cfg(KIND[self.kind], int(self.head_dim), float(self.theta_base), int(self.L_train),
                   int(self.L_target), float(self.s), float(self.ramp_alpha),
                   float(self.ramp_beta), float(self.mscale_override), None)
        if self.dim_scale is not None:
            arr = (ctypes.c_double * len(self.dim_scale))(*[float(v) for v in self.dim_scale])
            cfg._dim_scale_buf = arr  # keeps the array alive with the struct
            cfg.dim_scale = ctypes.cast(arr, ctypes.POINTER(ctypes.c_double))
        return cfg


_lib = None
_i64x3 = ctypes.c_int64 * 3
_P = ctypes.c_void_p


def library_path() -> str:
    return os.path.join(_PKG, _LIB_NAME)


def load_library():
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing; build it with `python -m yarn_rope_scaling_ntk_b300.build`")
    lib = ctypes.CDLL(path)
    I32, SZ, D = ctypes.c_int32, ctypes.c_size_t, ctypes.c_double
    cfgp = ctypes.POINTER(_Cfg)
    sig = {
        "yarn_inv_freq": (I32, [cfgp, ctypes.POINTER(D), ctypes.POINTER(ctypes.c_int8), ctypes.POINTER(D)]),
        "rope_apply": (I32, [cfgp, _P, _P, I32, I32, I32, I32, I32, _i64x3, _i64x3, I32, _P, I32, _P]),
        "yr_prefill_workspace_bytes": (SZ, [cfgp, I32, I32, I32, I32, I32, I32]),
        "attn_fwd_prefill": (I32, [cfgp, _P, _P, _P, _P, _P, I32, I32, I32, I32, I32, I32,
                                   _i64x3, _i64x3, _i64x3, _i64x3, I32, I32, I32, I32,
                                   ctypes.c_float, _P, SZ, _P]),
        "yr_prefill_kv_block_workspace_bytes": (SZ, [cfgp, I32, I32, I32, I32, I32, I32, I32]),
        "attn_fwd_prefill_kv_block": (I32, [cfgp, _P, _P, _P, _P, _P, I32, I32, I32, I32, I32, I32, I32, I32,
                                            I32, I32, _i64x3, _i64x3, _i64x3, _i64x3, I32, I32, I32,
                                            ctypes.c_float, _P, SZ, _P]),
        "attn_merge_partial": (I32, [_P, _P, _P, _P, _P, I32, I32, I32, I32, I32, _i64x3, _i64x3, _i64x3, _P]),
        "yr_bwd_workspace_bytes": (SZ, [cfgp, I32, I32, I32, I32, I32, I32]),
        "attn_bwd": (I32, [cfgp, _P, _P, _P, _P, _P, _P, _P, _P, _P, I32, I32, I32, I32, I32, I32, I32,
                           _i64x3, _i64x3, _i64x3, _i64x3, _i64x3, _i64x3, _i64x3, _i64x3, I32, I32, I32,
                           ctypes.c_float, _P, SZ, _P]),
        "yr_decode_auto_splits": (I32, [I32, I32, I32, I32]),
        "yr_decode_workspace_bytes": (SZ, [I32, I32, I32, I32, I32, I32, I32]),
        "attn_fwd_decode_sinkwindow": (I32, [cfgp, _P, _P, _P, _P, _P, I32, I32, I32, I32, I32,
                                             I32, _P, _P, I32, _P, SZ, _P]),
        "attn_fwd_decode_sinkwindow_fp8": (I32, [cfgp, _P, _P, _P, _P, _P, _P, _P, I32, I32, I32, I32, I32,
                                                 I32, _P, _P, I32, _P, SZ, _P]),
        "attn_fwd_decode_sinkwindow_noalloc": (I32, [cfgp, _P, _P, _P, _P, _P, I32, I32, I32, I32,
                                                     I32, I32, _P, _P, I32, _P]),
        "yr_sync_status": (I32, [_P]),
        "yr_kernel_launch_count": (ctypes.c_uint64, []),
        "yr_debug_inject_wait_fault": (I32, [ctypes.c_int64, I32]),
        "yr_last_error_message": (ctypes.c_char_p, []),
        "yr_version": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    _lib = lib
    return lib


def _check(st: int):
    if st != 0:
        raise YarnAttnError(st, load_library().yr_last_error_message().decode())


def _stream(stream=None) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _strides(t: torch.Tensor):
    if t.stride(-1) != 1:
        raise ValueError("the last (head-dim) axis must be contiguous")
    return _i64x3(*t.stride()[:3])


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise ValueError(f"unsupported dtype {t.dtype}")


def yarn_inv_freq(cfg: RopeConfig):
    """Host-only: (theta'[d/2] float64, classes[d/2] int8, mscale)."""
    lib = load_library()
    h = cfg.head_dim // 2
    th = (ctypes.c_double * h)()
    cl = (ctypes.c_int8 * h)()
    ms = ctypes.c_double()
    c = cfg.c()
    _check(lib.yarn_inv_freq(ctypes.byref(c), th, cl, ctypes.byref(ms)))
    return np.array(th[:], dtype=np.float64), np.array(cl[:], dtype=np.int8), ms.value


def rope_apply(cfg: RopeConfig, x: torch.Tensor, out: torch.Tensor | None = None,
               positions: torch.Tensor | None = None, pos0: int = 0, apply_mscale: bool = False,
               stream=None) -> torch.Tensor:
    """Rotate x [B, H, S, d] (float32 or bfloat16); ``out`` may be ``x``."""
    lib = load_library()
    if x.dim() != 4:
        raise ValueError("x must be [B, H, S, d]")
    y = torch.empty_like(x) if out is None else out
    if positions is not None and (positions.dtype != torch.int32 or positions.device != x.device):
        raise ValueError("positions must be an int32 tensor on x's device")
    B, H, S, d = x.shape
    c = cfg.c()
    _check(lib.rope_apply(ctypes.byref(c), _ptr(x), _ptr(y), _dtype_code(x), B, H, S, d,
                          _strides(x), _strides(y), int(pos0), _ptr(positions),
                          int(bool(apply_mscale)), _stream(stream)))
    return y


def prefill_workspace_bytes(cfg: RopeConfig, dtype: torch.dtype, B, Hq, Hkv, S, d) -> int:
    c = cfg.c()
    code = F32 if dtype == torch.float32 else BF16
    return int(load_library().yr_prefill_workspace_bytes(ctypes.byref(c), code, B, Hq, Hkv, S, d))


def prefill_kv_block_workspace_bytes(cfg: RopeConfig, dtype: torch.dtype, B, Hq, Hkv, Sq, Skv, d) -> int:
    c = cfg.c()
    code = F32 if dtype == torch.float32 else BF16
    return int(load_library().yr_prefill_kv_block_workspace_bytes(ctypes.byref(c), code, B, Hq, Hkv, Sq, Skv, d))


def attn_fwd_prefill(cfg: RopeConfig, q, k, v, mask: str = "causal", sink: int = 0,
                     window: int = 0, ring_blocks: int = 1, softmax_scale: float = 0.0,
                     out=None, lse=None, return_lse: bool = False, workspace=None, stream=None):
    """Exact attention with RoPE rescaling fused: q [B, Hq, S, d], k/v
    [B, Hkv, S, d] (float32 or bfloat16).  Returns o (and lse [B, Hq, S])."""
    lib = load_library()
    B, Hq, S, d = q.shape
    Hkv = k.shape[1]
    if k.shape != (B, Hkv, S, d) or v.shape != k.shape:
        raise ValueError("k and v must be [B, Hkv, S, d] matching q")
    if not (q.dtype == k.dtype == v.dtype):
        raise ValueError("q, k and v must share a dtype")
    o = torch.empty_like(q) if out is None else out
    if return_lse and lse is None:
        lse = torch.empty(B, Hq, S, dtype=torch.float32, device=q.device)
    need = prefill_workspace_bytes(cfg, q.dtype, B, Hq, Hkv, S, d)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    c = cfg.c()
    _check(lib.attn_fwd_prefill(ctypes.byref(c), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                _dtype_code(q), B, Hq, Hkv, S, d, _strides(q), _strides(k),
                                _strides(v), _strides(o), MASK[mask], int(sink), int(window),
                                int(ring_blocks), float(softmax_scale), _ptr(workspace),
                                0 if workspace is None else workspace.numel() * workspace.element_size(),
                                _stream(stream)))
    return (o, lse) if return_lse else o


def attn_fwd_prefill_kv_block(cfg: RopeConfig, q, k, v, q_pos0: int, k_pos0: int, mask: str = "causal",
                              sink: int = 0, window: int = 0, softmax_scale: float = 0.0,
                              out_dtype: torch.dtype = torch.float32, out=None, lse=None, workspace=None,
                              stream=None):
    """One query block q [B, Hq, Sq, d] (rows at q_pos0 + r) against one KV
    block k/v [B, Hkv, Skv, d] (keys at k_pos0 + n).  Returns (o, lse); o in
    ``out_dtype`` (float32 keeps the partial exact for attn_merge_partial)."""
    lib = load_library()
    B, Hq, Sq, d = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    if k.shape != (B, Hkv, Skv, d) or v.shape != k.shape:
        raise ValueError("k and v must be [B, Hkv, Skv, d]")
    if not (q.dtype == k.dtype == v.dtype):
        raise ValueError("q, k and v must share a dtype")
    o = torch.empty(B, Hq, Sq, d, dtype=out_dtype, device=q.device) if out is None else out
    if lse is None:
        lse = torch.empty(B, Hq, Sq, dtype=torch.float32, device=q.device)
    c = cfg.c()
    code = F32 if q.dtype == torch.float32 else BF16
    need = int(lib.yr_prefill_kv_block_workspace_bytes(ctypes.byref(c), code, B, Hq, Hkv, Sq, Skv, d))
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check(lib.attn_fwd_prefill_kv_block(
        ctypes.byref(c), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _dtype_code(q), _dtype_code(o),
        B, Hq, Hkv, Sq, Skv, d, int(q_pos0), int(k_pos0), _strides(q), _strides(k), _strides(v), _strides(o),
        MASK[mask], int(sink), int(window), float(softmax_scale), _ptr(workspace),
        0 if workspace is None else workspace.numel() * workspace.element_size(), _stream(stream)))
    return o, lse


def attn_merge_partial(o_acc, lse_acc, o_part, lse_part, out=None, stream=None):
    """Merge the partial (o_part, lse_part) into (o_acc, lse_acc) in place
    (float32 [B, H, S, d] and [B, H, S]); if ``out`` is given (float32 or
    bfloat16) it receives the merged O too."""
    lib = load_library()
    B, H, S, d = o_acc.shape
    for t in (o_acc, o_part):
        if t.dtype != torch.float32 or t.shape != (B, H, S, d):
            raise ValueError("o_acc and o_part must be float32 [B, H, S, d]")
    for t in (lse_acc, lse_part):
        if t.dtype != torch.float32 or t.shape != (B, H, S) or not t.is_contiguous():
            raise ValueError("lse tensors must be contiguous float32 [B, H, S]")
    _check(lib.attn_merge_partial(_ptr(o_acc), _ptr(lse_acc), _ptr(o_part), _ptr(lse_part), _ptr(out),
                                  F32 if out is None else _dtype_code(out), B, H, S, d, _strides(o_acc),
                                  _strides(o_part), _strides(out) if out is not None else _i64x3(0, 0, 0),
                                  _stream(stream)))
    return o_acc, lse_acc


def lib_bwd_workspace_bytes(cfg: RopeConfig, dtype: torch.dtype, B, Hq, Hkv, S, d) -> int:
    c = cfg.c()
    code = F32 if dtype == torch.float32 else BF16
    return int(load_library().yr_bwd_workspace_bytes(ctypes.byref(c), code, B, Hq, Hkv, S, d))


def attn_bwd(cfg: RopeConfig, q, k, v, o, dout, lse, mask: str = "causal", sink: int = 0, window: int = 0,
             softmax_scale: float = 0.0, out_dtype: torch.dtype | None = None, workspace=None, stream=None):
    """Gradients (dq, dk, dv) of attn_fwd_prefill with respect to the
    unrotated q [B, Hq, S, d], k, v [B, Hkv, S, d], given o, dout and the
    forward's lse [B, Hq, S]."""
    lib = load_library()
    B, Hq, S, d = q.shape
    Hkv = k.shape[1]
    if k.shape != (B, Hkv, S, d) or v.shape != k.shape or o.shape != q.shape or dout.shape != q.shape:
        raise ValueError("shapes: q, o, dout [B, Hq, S, d]; k, v [B, Hkv, S, d]")
    if not (q.dtype == k.dtype == v.dtype == o.dtype == dout.dtype):
        raise ValueError("q, k, v, o and dout must share a dtype")
    if lse.dtype != torch.float32 or lse.shape != (B, Hq, S) or not lse.is_contiguous():
        raise ValueError("lse must be contiguous float32 [B, Hq, S]")
    od = q.dtype if out_dtype is None else out_dtype
    dq = torch.empty(B, Hq, S, d, dtype=od, device=q.device)
    dk = torch.empty(B, Hkv, S, d, dtype=od, device=q.device)
    dv = torch.empty(B, Hkv, S, d, dtype=od, device=q.device)
    c = cfg.c()
    code = _dtype_code(q)
    need = int(lib.yr_bwd_workspace_bytes(ctypes.byref(c), code, B, Hq, Hkv, S, d))
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check(lib.attn_bwd(ctypes.byref(c), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq),
                        _ptr(dk), _ptr(dv), code, _dtype_code(dq), B, Hq, Hkv, S, d, _strides(q), _strides(k),
                        _strides(v), _strides(o), _strides(dout), _strides(dq), _strides(dk), _strides(dv),
                        MASK[mask], int(sink), int(window), float(softmax_scale), _ptr(workspace),
                        0 if workspace is None else workspace.numel() * workspace.element_size(),
                        _stream(stream)))
    return dq, dk, dv


def _check_decode_args(q, k_cache, v_cache, n_valid, ring_start, sink, window, out=None, lse=None):
    """Shapes, dtypes and layouts of a bfloat16-cache decode call (the kernel
    indexes the caches as contiguous [B, Hkv, sink + window, d]); returns
    (B, Hq, d, Hkv)."""
    if q.dim() != 3 or k_cache.dim() != 4:
        raise ValueError("q must be [B, Hq, d] and the caches [B, Hkv, sink + window, d]")
    B, Hq, d = q.shape
    Hkv = k_cache.shape[1]
    for t in (q, k_cache, v_cache):
        if t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError("q and the caches must be contiguous bfloat16")
    if k_cache.shape != (B, Hkv, sink + window, d) or v_cache.shape != k_cache.shape:
        raise ValueError("caches must be [B, Hkv, sink + window, d]")
    for t in (n_valid, ring_start):
        if t.dtype != torch.int32 or t.shape != (B,):
            raise ValueError("n_valid and ring_start must be int32 [B]")
    if out is not None and (out.dtype != torch.bfloat16 or out.shape != (B, Hq, d) or not out.is_contiguous()):
        raise ValueError("out must be contiguous bfloat16 [B, Hq, d]")
    if lse is not None and (lse.dtype != torch.float32 or lse.shape != (B, Hq) or not lse.is_contiguous()):
        raise ValueError("lse must be contiguous float32 [B, Hq]")
    devs = {t.device for t in (q, k_cache, v_cache, n_valid, ring_start, out, lse) if t is not None}
    if len(devs) != 1 or next(iter(devs)).type != "cuda":
        raise ValueError("every tensor must be on the same CUDA device")
    return B, Hq, d, Hkv


def decode_workspace_bytes(B, Hq, Hkv, d, sink, window, num_splits=0) -> int:
    return int(load_library().yr_decode_workspace_bytes(B, Hq, Hkv, d, sink, window, num_splits))


def attn_fwd_decode_sinkwindow(cfg: RopeConfig, q, k_cache, v_cache, n_valid, ring_start,
                               sink: int, window: int, num_splits: int = 0, out=None, lse=None,
                               return_lse: bool = False, workspace=None, stream=None):
    """q [B, Hq, d] bf16; caches [B, Hkv, sink + window, d] bf16 (contiguous);
    n_valid / ring_start int32 [B].  Returns o [B, Hq, d] (and lse [B, Hq])."""
    lib = load_library()
    B, Hq, d, Hkv = _check_decode_args(q, k_cache, v_cache, n_valid, ring_start, sink, window, out, lse)
    o = torch.empty_like(q) if out is None else out
    if return_lse and lse is None:
        lse = torch.empty(B, Hq, dtype=torch.float32, device=q.device)
    need = decode_workspace_bytes(B, Hq, Hkv, d, sink, window, num_splits)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    c = cfg.c()
    _check(lib.attn_fwd_decode_sinkwindow(
        ctypes.byref(c), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(n_valid), _ptr(ring_start),
        B, Hq, Hkv, d, int(sink), int(window), _ptr(o), _ptr(lse), int(num_splits),
        _ptr(workspace), 0 if workspace is None else workspace.numel() * workspace.element_size(),
        _stream(stream)))
    return (o, lse) if return_lse else o


def attn_fwd_decode_sinkwindow_fp8(cfg: RopeConfig, q, k_cache, v_cache, k_scale, v_scale, n_valid,
                                   ring_start, sink: int, window: int, num_splits: int = 0, out=None,
                                   lse=None, return_lse: bool = False, workspace=None, stream=None):
    """Decode over an FP8 E4M3 cache: k_cache / v_cache [B, Hkv, sink + window,
    d] (torch.float8_e4m3fn or uint8 bytes), k_scale / v_scale float32
    [B, Hkv]; q [B, Hq, d] bfloat16.  Returns o (and lse)."""
    lib = load_library()
    B, Hq, d = q.shape
    Hkv = k_cache.shape[1]
    if q.dtype != torch.bfloat16 or not q.is_contiguous():
        raise ValueError("q must be contiguous bfloat16")
    for t in (k_cache, v_cache):
        if t.element_size() != 1 or not t.is_contiguous() or t.shape != (B, Hkv, sink + window, d):
            raise ValueError("caches must be contiguous 1-byte [B, Hkv, sink + window, d]")
    for t in (k_scale, v_scale):
        if t.dtype != torch.float32 or not t.is_contiguous() or t.numel() != B * Hkv:
            raise ValueError("scales must be contiguous float32 [B, Hkv]")
    for t in (n_valid, ring_start):
        if t.dtype != torch.int32 or t.shape != (B,):
            raise ValueError("n_valid and ring_start must be int32 [B]")
    o = torch.empty_like(q) if out is None else out
    if return_lse and lse is None:
        lse = torch.empty(B, Hq, dtype=torch.float32, device=q.device)
    need = decode_workspace_bytes(B, Hq, Hkv, d, sink, window, num_splits)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    c = cfg.c()
    _check(lib.attn_fwd_decode_sinkwindow_fp8(
        ctypes.byref(c), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(n_valid),
        _ptr(ring_start), B, Hq, Hkv, d, int(sink), int(window), _ptr(o), _ptr(lse), int(num_splits),
        _ptr(workspace), 0 if workspace is None else workspace.numel() * workspace.element_size(),
        _stream(stream)))
    return (o, lse) if return_lse else o


def attn_fwd_decode_sinkwindow_noalloc(cfg: RopeConfig, q, k_cache, v_cache, n_valid, ring_start,
                                       sink: int, window: int, num_splits: int = 0, out=None,
                                       lse=None, stream=None):
    """Decode without a workspace: the split scratch is the library's own
    fixed 4 MiB device array (for callers that cannot allocate when they
    call).  ``out`` and ``lse`` are the caller's; nothing is allocated when
    both are given."""
    lib = load_library()
    B, Hq, d, Hkv = _check_decode_args(q, k_cache, v_cache, n_valid, ring_start, sink, window, out, lse)
    o = torch.empty_like(q) if out is None else out
    c = cfg.c()
    _check(lib.attn_fwd_decode_sinkwindow_noalloc(
        ctypes.byref(c), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(n_valid), _ptr(ring_start),
        B, Hq, Hkv, d, int(sink), int(window), _ptr(o), _ptr(lse), int(num_splits), _stream(stream)))
    return o


def debug_inject_wait_fault(wait_limit_cycles: int = 0, skip_unit: int = -1):
    """Test hook for the failure path: bound the decode and prefill kernels'
    waits by ``wait_limit_cycles`` and make their producers skip load unit
    ``skip_unit``; ``(0, -1)`` turns it off.  Process-wide."""
    _check(load_library().yr_debug_inject_wait_fault(int(wait_limit_cycles), int(skip_unit)))


def kernel_launch_count() -> int:
    """Kernels the library has launched in this process so far."""
    return int(load_library().yr_kernel_launch_count())


def sync_status(stream=None):
    """Synchronise the stream and raise if a device-side bounded wait gave up."""
    _check(load_library().yr_sync_status(_stream(stream)))
