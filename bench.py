#!/usr/bin/env python3
"""Benchmark of the fused YaRN-RoPE + attention hot path on B300.

One step = one pass of the prefill hot path over the Llama-2-7B-shaped
workload (B=1, 32 heads, d=128, S=16384, bf16, YaRN s=4 from L_train=4096,
causal): frequency table, rotation of Q and K, QK^T, mask, online softmax and
PV folded over 128-key blocks, through the public ``attn_fwd_prefill`` call.
The same run also times the streaming decode over the sink + window cache
(B=64, 32 heads, 4 + 4092 slots) and standalone ``rope_apply`` on the
workload's Q and K, reported as sub-objects.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

``--impl reference`` times the float64 CPU oracle on a bounded sample of the
same workload (the oracle is the reference arm: the pages ship no code).
``--ring`` times ring attention over the N ranks on the 131072-token
workload instead (one KV block per rank, NCCL point-to-point exchange).
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from yarn_rope_scaling_ntk_b300 import api, workloads as W  # noqa: E402

METRIC = "fused YaRN-RoPE+attention TFLOP/s & % bf16 peak; decode HBM GB/s"
# Nominal figures beside the measured peaks: about 8 TB/s of HBM3e and
# 2.25 PFLOP/s of dense bf16 tensor throughput per B300.
NOMINAL_HBM_GBS = 8000.0
NOMINAL_BF16_TFLOPS = 2250.0

CSRC = os.path.join(ROOT, "yarn_rope_scaling_ntk_b300", "csrc")
# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) from
# one ncu capture of each kernel on the bench's workload, keyed by a hash of
# the kernel's source files at capture time.  A kernel whose sources changed
# since reports null.  The commands are in profiles/.
KERNEL_SOURCES = {
    "prefill_tc": ("prefill_tc.cu", "tc_ptx.cuh", "common.cuh"),
    "decode": ("decode.cu", "tc_ptx.cuh", "common.cuh"),
    "rope": ("rope.cu", "tc_ptx.cuh", "common.cuh"),
    "rotation_qk": ("rope.cu", "tc_ptx.cuh", "common.cuh"),
    "decode_fp8": ("decode.cu", "tc_ptx.cuh", "common.cuh"),
    "bwd_kv": ("backward_tc.cu", "tc_ptx.cuh", "common.cuh"),
    "bwd_q": ("backward_tc.cu", "tc_ptx.cuh", "common.cuh"),
}
TRAFFIC = {
    # kernel: (source hash, bytes per launch, what was captured)
    "prefill_tc": ("5f5deb7786a2f853", 515.94e6 + 120.82e6,
                   "bench.py --part prefill: Llama-2-7B shape S=16384, one launch"),
    "rotation_qk": ("f702d243b8631d22", 268.62e6 + 216.82e6,
                    "bench.py --part prefill: the step's rotation pass over Q and K, one launch"),
    "decode": ("3f0f6b32031b2712", 4295.89e6 + 3.59e6,
               "bench.py --part decode: 64 sequences x 32 heads x 4096 slots, one launch"),
    "decode_fp8": ("3f0f6b32031b2712", 2148.34e6 + 16.40e6,
                   "bench.py --part decode_fp8: the same cache shape in FP8 E4M3, one launch"),
    "rope": ("f702d243b8631d22", 268.63e6 + 214.95e6,
             "bench.py --part rope: Q and K stacked, [1, 64, 16384, 128] bf16, one launch"),
    "bwd_kv": ("9631e3af16d2f5fe", 550.11e6 + 237.83e6,
               "bench.py --part backward: Llama-2-7B shape S=16384, one launch"),
    "bwd_q": ("9631e3af16d2f5fe", 557.85e6 + 116.88e6,
              "bench.py --part backward: Llama-2-7B shape S=16384, one launch"),
}


def source_hash(kernel: str) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic(kernel: str):
    rec = TRAFFIC.get(kernel)
    if rec is None or rec[0] != source_hash(kernel):
        return None
    return rec[1]


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", 0)), "measured"
    except Exception:
        return 6400.0, 1800.0, 1400.0, "fallback"


def visible_pairs(S: int, mask: str, sink: int, window: int) -> int:
    """Number of visible (query, key) pairs of one head (integer formula of
    the mask definition)."""
    m = np.arange(S, dtype=np.int64)
    if mask == "none":
        return S * S
    if mask == "causal":
        return int((m + 1).sum())
    in_w = np.minimum(m + 1, window)
    return int((in_w + np.clip(np.minimum(sink, m + 1 - in_w), 0, None)).sum())


def prefill_flops(w) -> float:
    return 4.0 * w.d * visible_pairs(w.S, w.mask, w.sink, w.window) * w.B * w.Hq


def reduce_max(value: float, dist=None, device="cpu") -> float:
    """Max of a per-rank value over all ranks (the slowest rank's time); the
    value itself when there is no process group."""
    if dist is None:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(work_per_step: float, steps: int, world: int, max_total_ms: float) -> float:
    """Weak scaling: every rank runs the same per-rank work; the job's rate is
    all ranks' work divided by the slowest rank's time (units per second)."""
    return work_per_step * steps * world / (max_total_ms * 1e-3)


def step_config(w, n: int) -> dict:
    """The `config` object of the step's line, the same for both arms."""
    return {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "S": w.S, "d": w.d,
            "mask": w.mask, "rope": "yarn s=4 L_train=4096 theta_base=1e4",
            "l2": "inputs larger than L2 (537 MB Q/K/V/O vs 126 MB)", "parallelism": f"replicas x{n}"}


def cfg_of(w):
    r = w.rope
    return api.RopeConfig(kind=r.kind, head_dim=w.d, theta_base=r.theta_base, L_train=r.L_train,
                          L_target=r.L_target, s=r.s)


class _Nvml:
    """Read-only NVML queries through ctypes on the driver's libnvidia-ml."""

    def __init__(self, cuda_index: int):
        import ctypes
        self.c = ctypes
        self.lib = None
        for name in ("libnvidia-ml.so.1", "libnvidia-ml.so"):
            try:
                self.lib = ctypes.CDLL(name)
                break
            except OSError:
                continue
        if self.lib is None:
            raise RuntimeError("libnvidia-ml not found")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        p = torch.cuda.get_device_properties(cuda_index)
        bus = f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0".encode()
        self.h = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByPciBusId_v2(bus, ctypes.byref(self.h)) != 0:
            raise RuntimeError(f"no NVML handle for {bus!r}")

    def sm_clock(self, fn="nvmlDeviceGetClockInfo") -> int:
        v = self.c.c_uint()
        if getattr(self.lib, fn)(self.h, 1, self.c.byref(v)) != 0:  # 1 = NVML_CLOCK_SM
            raise RuntimeError(fn)
        return v.value

    def reasons(self) -> int:
        v = self.c.c_ulonglong()
        for fn in ("nvmlDeviceGetCurrentClocksEventReasons", "nvmlDeviceGetCurrentClocksThrottleReasons"):
            if hasattr(self.lib, fn) and getattr(self.lib, fn)(self.h, self.c.byref(v)) == 0:
                return v.value
        raise RuntimeError("clock event reasons unavailable")


class ClockSampler:
    """SM clock and clock-event reasons sampled through NVML every 5 ms on a
    background thread (read-only queries) while the timed region runs."""

    REASONS = {"hw_slowdown": 0x8, "hw_thermal_slowdown": 0x40, "sw_thermal_slowdown": 0x20,
               "sw_power_cap": 0x4}

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.stop = threading.Event()
        self.thread = None
        self.error = None
        self.max_mhz = None

    def __enter__(self):
        try:
            self.nv = _Nvml(self.index)
            self.max_mhz = self.nv.sm_clock("nvmlDeviceGetMaxClockInfo")
            self.thread = threading.Thread(target=self._run, daemon=True)
            self.thread.start()
        except Exception as e:  # noqa: BLE001 - reported in the JSON line
            self.error = str(e)
        return self

    def _run(self):
        while not self.stop.is_set():
            try:
                self.rows.append((self.nv.sm_clock(), self.nv.reasons()))
            except Exception as e:  # noqa: BLE001
                self.error = str(e)
            time.sleep(0.005)

    def __exit__(self, *exc):
        self.stop.set()
        if self.thread:
            self.thread.join(timeout=2)

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unsampled"],
                    "error": self.error}
        reasons = sorted({n for _, r in self.rows for n, bit in self.REASONS.items() if r & bit})
        return {"sm_mhz": statistics.median(sm for sm, _ in self.rows), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(self.rows), "source": "NVML, 5 ms"}


def timed(fn, steps: int, stream) -> list:
    """Per-call device time (ms) of ``fn`` with CUDA events on ``stream``."""
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in ev:
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def cpu_oracle_prefill(w, seconds: float = 12.0, seed: int = 0):
    """Float64 oracle on a bounded sample of the workload: all heads' K
    rotated, query rows sampled until ``seconds`` of CPU work.  Returns
    (TFLOP/s, sample description, threads)."""
    import oracle.attention as OA
    import oracle.rope as OR
    r = w.rope
    th, _, _ = OR.inv_freq(r.kind, w.d, r.theta_base, r.L_train, r.L_target, r.s)
    s = OR.resolve_scale(r.L_train, r.L_target, r.s)
    scale = OA.softmax_scale(r.kind, s, w.d)
    g = torch.Generator().manual_seed(4242 + seed)
    flops, rows_done, heads, t0 = 0.0, 0, 0, time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        q = torch.randn(w.S, w.d, generator=g).to(w.dtype).double().numpy()
        k = torch.randn(w.S, w.d, generator=g).to(w.dtype).double().numpy()
        v = torch.randn(w.S, w.d, generator=g).to(w.dtype).double().numpy()
        rows = np.sort(torch.randint(0, w.S, (64,), generator=g).numpy())
        OA.prefill_head(q, k, v, rows, th, scale, w.mask, w.sink, w.window)
        m = rows.astype(np.int64)
        if w.mask == "causal":
            vis = (m + 1).sum()
        elif w.mask == "none":
            vis = w.S * len(rows)
        else:
            in_w = np.minimum(m + 1, w.window)
            vis = (in_w + np.clip(np.minimum(w.sink, m + 1 - in_w), 0, None)).sum()
        flops += 4.0 * w.d * float(vis)
        rows_done += len(rows)
        heads += 1
    dt = time.perf_counter() - t0
    threads = torch.get_num_threads()
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        threads = max([i.get("num_threads", 1) for i in info] + [1])
    except Exception:
        pass
    desc = (f"{heads} heads x 64 sampled query rows of {w.name} (each head's full K rotated in "
            f"float64), {dt:.1f} s; TFLOP/s = 4*d*visible pairs of the sampled rows / time")
    return flops / dt / 1e12, desc, threads


def time_prefill_workload(w, dev, stream, reps: int = 3):
    """Device time of the whole fused call (rotation pass + attention) on one
    of the other prefill workloads; returns a JSON-ready dict."""
    cfg = cfg_of(w)
    q, k, v = W.prefill_inputs(w, dev)
    o = torch.empty_like(q)
    ws = torch.empty(api.prefill_workspace_bytes(cfg, q.dtype, w.B, w.Hq, w.Hkv, w.S, w.d),
                     dtype=torch.uint8, device=dev)
    call = lambda: api.attn_fwd_prefill(cfg, q, k, v, mask=w.mask, sink=w.sink, window=w.window,
                                        ring_blocks=w.ring_blocks, out=o, workspace=ws)
    call()
    torch.cuda.synchronize()
    ms = statistics.median(timed(call, reps, stream))
    api.sync_status()
    flops = prefill_flops(w)
    del q, k, v, o, ws
    torch.cuda.empty_cache()
    return {"workload": w.name, "ms": ms, "TFLOP/s": flops / (ms * 1e-3) / 1e12, "TFLOP": flops / 1e12,
            "ring_blocks": w.ring_blocks, "mask": w.mask}


def time_ring_blocks(w, dev, stream, reps: int = 2):
    """The ring workload computed as each device of a multi-GPU ring would:
    Q and K rotated once (each device rotates its own blocks), then query
    block I takes KV blocks I, I-1, ..., 0, one attn_fwd_prefill_kv_block
    call each on the rotated operands into a float32 partial, merged by
    attn_merge_partial (the last merge writes the bf16 output).  Device
    time of the rotation and all blocks' calls, with the merge kernel's
    share and bandwidth; no communication is included."""
    cfg_rot = cfg_of(w)
    _, _, mscale = api.yarn_inv_freq(cfg_rot)
    cfg = api.RopeConfig(kind="none", head_dim=w.d)
    scale = mscale * mscale / math.sqrt(w.d)
    q0, k0, v = W.prefill_inputs(w, dev)
    q, k = torch.empty_like(q0), torch.empty_like(k0)
    N = w.ring_blocks
    bs = w.S // N
    final = torch.empty_like(q)
    acc = torch.empty(w.B, w.Hq, bs, w.d, dtype=torch.float32, device=dev)
    part = torch.empty_like(acc)
    lacc = torch.empty(w.B, w.Hq, bs, dtype=torch.float32, device=dev)
    lpart = torch.empty_like(lacc)
    ws = torch.empty(max(1, api.prefill_kv_block_workspace_bytes(cfg, q.dtype, w.B, w.Hq, w.Hkv, bs, bs, w.d)),
                     dtype=torch.uint8, device=dev)
    merges = []

    def ring(record=False):
        api.rope_apply(cfg_rot, q0, out=q, stream=stream)
        api.rope_apply(cfg_rot, k0, out=k, stream=stream)
        for I in range(N):
            rows = slice(I * bs, (I + 1) * bs)
            qi = q[:, :, rows]
            order = list(range(I, -1, -1))  # I, I-1, ..., 0: the causal ring skips blocks after I
            for step, j in enumerate(order):
                keys = slice(j * bs, (j + 1) * bs)
                last = step == len(order) - 1
                if step == 0:
                    api.attn_fwd_prefill_kv_block(cfg, qi, k[:, :, keys], v[:, :, keys], I * bs, j * bs,
                                                  mask=w.mask, softmax_scale=scale,
                                                  out=final[:, :, rows] if last else acc, lse=lacc,
                                                  workspace=ws, stream=stream)
                    continue
                api.attn_fwd_prefill_kv_block(cfg, qi, k[:, :, keys], v[:, :, keys], I * bs, j * bs, mask=w.mask,
                                              softmax_scale=scale, out=part, lse=lpart, workspace=ws,
                                              stream=stream)
                if record:
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(stream)
                api.attn_merge_partial(acc, lacc, part, lpart, out=final[:, :, rows] if last else None,
                                       stream=stream)
                if record:
                    b.record(stream)
                    merges.append((a, b, last))

    ring()
    torch.cuda.synchronize()
    ms = statistics.median(timed(ring, reps, stream))
    ring(record=True)
    torch.cuda.synchronize()
    api.sync_status()
    fused = api.attn_fwd_prefill(cfg_rot, q0, k0, v, mask=w.mask, ring_blocks=N)
    diff = (fused.float() - final.float()).abs().max().item()
    del fused
    merge_ms = sum(a.elapsed_time(b) for a, b, _ in merges)
    # per merge: O_acc read + written, O_part read (float32), four lse vectors; the last one per query block
    # also writes the bf16 output
    per = w.B * w.Hq * bs
    merge_bytes = sum(per * w.d * 4 * 3 + per * 4 * 4 + (per * w.d * 2 if last else 0) for _, _, last in merges)
    flops = prefill_flops(w)
    del q0, k0, q, k, v, final, acc, part, lacc, lpart, ws
    torch.cuda.empty_cache()
    return {"workload": w.name + "_one_kv_block_per_call", "ms": ms, "TFLOP/s": flops / (ms * 1e-3) / 1e12,
            "kv_block_calls": N * (N + 1) // 2, "merges": len(merges), "merge_ms_total": merge_ms,
            "merge_GB/s": merge_bytes / (merge_ms * 1e-3) / 1e9, "max_abs_diff_vs_fused_call": diff}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = W.LLAMA2_7B
    vals, walls = [], []
    desc = ""
    threads = 1
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        v, desc, threads = cpu_oracle_prefill(w, seconds=6.0, seed=i)
        wall = time.perf_counter() - t0
        if i >= args.warmup:
            vals.append(v)
            walls.append(wall)
    value = statistics.median(vals)
    # a step is one bounded sample: its measured wall time, not the full workload's
    ms = statistics.mean(walls) * 1e3
    full_ms = prefill_flops(w) / (value * 1e12) * 1e3
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "full_workload_ms_extrapolated": full_ms,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": step_config(w, args.gpus),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def run_ours(args):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    hbm, tf_burst, tf_sust, peak_src = peaks()

    # ---- prefill (the step) ----------------------------------------------
    w = W.LLAMA2_7B
    cfg = cfg_of(w)
    q, k, v = W.prefill_inputs(w, dev, seed_index=w.index + 17 * rank)
    o = torch.empty_like(q)
    ws = torch.empty(api.prefill_workspace_bytes(cfg, q.dtype, w.B, w.Hq, w.Hkv, w.S, w.d),
                     dtype=torch.uint8, device=dev)
    step = lambda: api.attn_fwd_prefill(cfg, q, k, v, mask=w.mask, out=o, workspace=ws)
    for _ in range(max(3, args.warmup)):
        step()
    api.sync_status()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = api.kernel_launch_count()
    with ClockSampler(local) as clocks:
        times = timed(step, args.steps, stream)
    launches = api.kernel_launch_count() - launches0
    api.sync_status()
    total_ms = reduce_max(sum(times), dist, dev)
    flops = prefill_flops(w)
    value = whole_job_rate(flops, args.steps, world, total_ms) / 1e12
    ms_per_step = total_ms / args.steps

    # attention kernel alone (pre-rotated operands, same kernel): roofline
    nb = w.B * w.Hq * w.S * w.d * 2
    qr = ws[:nb].view(torch.bfloat16).view(w.B, w.Hq, w.S, w.d)
    kr = ws[nb:2 * nb].view(torch.bfloat16).view(w.B, w.Hkv, w.S, w.d)
    cfg_none = api.RopeConfig(kind="none", head_dim=w.d)
    _, _, mscale = api.yarn_inv_freq(cfg)  # the temperature the fused call folds into its scale
    scale = mscale * mscale / math.sqrt(w.d)
    attn = lambda: api.attn_fwd_prefill(cfg_none, qr, kr, v, mask=w.mask, out=o, softmax_scale=scale)
    for _ in range(3):
        attn()
    torch.cuda.synchronize()
    # A burst, like the peak it is divided by: after the step loop the GPU
    # idles briefly so that the power state of the long loop does not carry
    # over, then 10 launches; median launch time, clocks sampled meanwhile.
    time.sleep(0.3)
    with ClockSampler(local) as attn_clocks:
        attn_times = timed(attn, 10, stream)
    attn_ms = statistics.median(attn_times)
    attn_tflops = flops / (attn_ms * 1e-3) / 1e12

    # ---- end to end through the public call, host buffers -----------------
    # Q, K, V start in pinned host memory and O ends there, every step.  The
    # step is split into head chunks on three streams, so that the copy in of
    # chunk c + 1, the attention of chunk c and the copy out of chunk c - 1
    # overlap; steps do not overlap one another.
    hq_, hk_, hv_ = (t.cpu().pin_memory() for t in (q, k, v))
    ho = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
    dq_, dk_, dv_, do_ = (torch.empty_like(t) for t in (q, k, v, o))
    n_chunks = next(c for c in (8, 4, 2, 1) if w.Hq % c == 0 and w.Hkv % c == 0)
    hq_c, hk_c = w.Hq // n_chunks, w.Hkv // n_chunks
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(n_chunks)]
    ev_out = [torch.cuda.Event() for _ in range(n_chunks)]

    def e2e_step():
        s_in.wait_stream(stream)
        for c in range(n_chunks):
            qs, ks = slice(c * hq_c, (c + 1) * hq_c), slice(c * hk_c, (c + 1) * hk_c)
            with torch.cuda.stream(s_in):
                dq_[:, qs].copy_(hq_[:, qs], non_blocking=True)
                dk_[:, ks].copy_(hk_[:, ks], non_blocking=True)
                dv_[:, ks].copy_(hv_[:, ks], non_blocking=True)
                ev_in[c].record(s_in)
            stream.wait_event(ev_in[c])
            api.attn_fwd_prefill(cfg, dq_[:, qs], dk_[:, ks], dv_[:, ks], mask=w.mask, out=do_[:, qs],
                                 workspace=ws, stream=stream)
            ev_out[c].record(stream)
            s_out.wait_event(ev_out[c])
            with torch.cuda.stream(s_out):
                ho[:, qs].copy_(do_[:, qs], non_blocking=True)
        stream.wait_stream(s_out)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    e2e_times = timed(e2e_step, max(3, min(args.steps, 10)), stream)
    e2e_val = flops / (statistics.mean(e2e_times) * 1e-3) / 1e12
    h2d = sum(t.numel() * t.element_size() for t in (hq_, hk_, hv_))
    d2h = ho.numel() * ho.element_size()
    # the chunked end-to-end result against one device-resident call
    o_dev = api.attn_fwd_prefill(cfg, q, k, v, mask=w.mask, workspace=ws)
    e2e_diff = (ho.to(dev).float() - o_dev.float()).abs().max().item()
    del hq_, hk_, hv_, ho, dq_, dk_, dv_, do_, o_dev

    # ---- decode over the sink + window cache ------------------------------
    wd = W.DECODE
    dq, kc, vc, nv, rs = W.decode_inputs(wd, dev)
    dcfg = api.RopeConfig(kind="plain", head_dim=wd.d, theta_base=wd.rope.theta_base)
    do = torch.empty_like(dq)
    dws = torch.empty(max(1, api.decode_workspace_bytes(wd.B, wd.Hq, wd.Hkv, wd.d, wd.sink, wd.window)),
                      dtype=torch.uint8, device=dev)
    dec = lambda: api.attn_fwd_decode_sinkwindow(dcfg, dq, kc, vc, nv, rs, wd.sink, wd.window,
                                                  out=do, workspace=dws)
    for _ in range(3):
        dec()
    dec_ms = statistics.mean(timed(dec, max(10, args.steps), stream))
    dec_bytes = 2 * kc.numel() * 2 + dq.numel() * 2 + do.numel() * 2 + 2 * 4 * wd.B
    dec_gbs = dec_bytes / (dec_ms * 1e-3) / 1e9
    del kc, vc

    # ---- the same decode over an FP8 E4M3 cache (half the bytes) ----------
    fq, fkc, fvc, fks, fvs, fnv, frs = W.decode_inputs_fp8(wd, dev)
    dec8 = lambda: api.attn_fwd_decode_sinkwindow_fp8(dcfg, fq, fkc, fvc, fks, fvs, fnv, frs, wd.sink,
                                                       wd.window, out=do, workspace=dws)
    for _ in range(3):
        dec8()
    dec8_ms = statistics.mean(timed(dec8, max(10, args.steps), stream))
    dec8_bytes = 2 * fkc.numel() + 2 * 4 * fks.numel() + fq.numel() * 2 + do.numel() * 2 + 2 * 4 * wd.B
    dec8_gbs = dec8_bytes / (dec8_ms * 1e-3) / 1e9
    del fkc, fvc

    # ---- standalone rope_apply on Q and K of the prefill workload ---------
    # One call on Q and K stacked along the heads ([1, 64, 16384, 128], one
    # launch, the kernel's own rate), and two calls (Q, then K) as a caller
    # with separate tensors makes them.
    qk = torch.cat([q, k], dim=1)
    qk_out = torch.empty_like(qk)
    rope_one = lambda: api.rope_apply(cfg, qk, out=qk_out)
    def rope_qk():
        api.rope_apply(cfg, q, out=o)
        api.rope_apply(cfg, k, out=o)
    for _ in range(3):
        rope_one()
        rope_qk()
    rope_bytes = 2 * 2 * q.numel() * 2
    rope_ms = statistics.mean(timed(rope_one, max(10, args.steps), stream))
    rope_gbs = rope_bytes / (rope_ms * 1e-3) / 1e9
    rope2_ms = statistics.mean(timed(rope_qk, max(10, args.steps), stream))
    rope2_gbs = rope_bytes / (rope2_ms * 1e-3) / 1e9
    api.sync_status()
    del o, qk, qk_out
    torch.cuda.empty_cache()

    # ---- backward of the same prefill (whole call: rotation, rowsum, dK/dV, dQ)
    bwd = None
    if not args.no_backward:
        qb, kb, vb = W.prefill_inputs(w, dev)
        ob, lseb = api.attn_fwd_prefill(cfg, qb, kb, vb, mask=w.mask, return_lse=True)
        g = torch.Generator(device=dev).manual_seed(77)
        dob = torch.randn(qb.shape, generator=g, device=dev).to(qb.dtype)
        bws = torch.empty(api.lib_bwd_workspace_bytes(cfg, qb.dtype, w.B, w.Hq, w.Hkv, w.S, w.d),
                          dtype=torch.uint8, device=dev)
        bcall = lambda: api.attn_bwd(cfg, qb, kb, vb, ob, dob, lseb, mask=w.mask, workspace=bws)
        for _ in range(2):
            bcall()
        bwd_ms = statistics.median(timed(bcall, 5, stream))
        api.sync_status()
        # algorithmic: dV, dP, dQ, dK and one recompute of S, 2 d flops each per visible pair
        bflops = 2.5 * prefill_flops(w)
        bwd = {"workload": w.name, "ms": bwd_ms, "TFLOP/s": bflops / (bwd_ms * 1e-3) / 1e12,
               "frac_of_burst": bflops / (bwd_ms * 1e-3) / 1e12 / tf_burst,
               "flops": "10 d per visible pair (the kernels do 14 d: S and dP are recomputed in both)",
               "traffic_per_launch": {"bwd_kv_kernel": traffic("bwd_kv"), "bwd_q_kernel": traffic("bwd_q")}}
        del qb, kb, vb, ob, lseb, dob, bws
        torch.cuda.empty_cache()

    # ---- the other prefill workloads (whole fused call, device time) -------
    others = []
    if not args.no_other_workloads:
        for wo in (W.RING_128K, W.LLAMA3_8B_GQA, W.LLAMA3_8B_GQA_SW):
            r = time_prefill_workload(wo, dev, stream)
            r["frac_of_burst"] = r["TFLOP/s"] / tf_burst
            # tens of milliseconds per call under load: the sustained peak is the fair denominator
            r["frac_of_sustained"] = r["TFLOP/s"] / tf_sust
            others.append(r)
    ring_blocks = None
    if not args.no_other_workloads:
        ring_blocks = time_ring_blocks(W.RING_128K, dev, stream)
        ring_blocks["frac_of_burst"] = ring_blocks["TFLOP/s"] / tf_burst
        ring_blocks["frac_of_sustained"] = ring_blocks["TFLOP/s"] / tf_sust
        ring_blocks["merge_frac_of_hbm"] = ring_blocks["merge_GB/s"] / hbm

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return
    cs = clocks.summary()
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": step_config(w, world),
        "pct_bf16_peak": {"burst": value / world / tf_burst, "sustained": value / world / tf_sust,
                          "peaks": peak_src},
        "rotation_pass_traffic": traffic("rotation_qk"),
        "roofline": {"bound": "tensor", "achieved": attn_tflops, "peak": tf_burst, "unit": "TFLOP/s",
                     "frac": attn_tflops / tf_burst, "traffic": traffic("prefill_tc"),
                     "kernel": "prefill_tc_kernel alone on pre-rotated Q/K (the launch the step makes)",
                     "kernel_ms": attn_ms, "peak_kind": f"bf16 burst ({peak_src}; kernel timed alone)",
                     "timing": "median of 10 back-to-back launches after 0.3 s idle",
                     "kernel_ms_mean": statistics.mean(attn_times), "clocks": attn_clocks.summary(),
                     "frac_of_sustained": attn_tflops / tf_sust,
                     "frac_of_nominal": attn_tflops / NOMINAL_BF16_TFLOPS,
                     "nominal_peak": NOMINAL_BF16_TFLOPS},
        "e2e": {"value": e2e_val, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "pipeline": f"{n_chunks} head chunks, copy in / attention / copy out on 3 streams",
                "max_abs_diff_vs_device_call": e2e_diff},
        "gpu_launches": launches,  # the library's own launch counter over the timed steps
        "clocks": cs,
        "decode": {"workload": wd.name, "value": dec_gbs, "unit": "GB/s", "ms": dec_ms,
                   "roofline": {"bound": "hbm", "achieved": dec_gbs, "peak": hbm, "unit": "GB/s",
                                "frac": dec_gbs / hbm, "traffic": traffic("decode"),
                                "frac_of_nominal": dec_gbs / NOMINAL_HBM_GBS, "nominal_peak": NOMINAL_HBM_GBS,
                                "peak_note": "the measured peak is a copy (reads and writes); decode only reads"}},
        "decode_fp8": {"workload": wd.name + "_fp8_e4m3", "value": dec8_gbs, "unit": "GB/s", "ms": dec8_ms,
                       "speedup_vs_bf16_cache": dec_ms / dec8_ms,
                       "roofline": {"bound": "hbm", "achieved": dec8_gbs, "peak": hbm, "unit": "GB/s",
                                    "frac": dec8_gbs / hbm, "traffic": traffic("decode_fp8"),
                                    "frac_of_nominal": dec8_gbs / NOMINAL_HBM_GBS, "nominal_peak": NOMINAL_HBM_GBS}},
        "backward": bwd,
        "other_prefill_workloads": others,
        "ring_building_blocks": ring_blocks,
        "rope_apply": {"workload": "Q and K of " + w.name + ", stacked as one [1, 64, 16384, 128] tensor",
                       "value": rope_gbs, "unit": "GB/s", "ms": rope_ms,
                       "two_calls": {"what": "Q, then K, one call each", "ms": rope2_ms, "GB/s": rope2_gbs,
                                     "frac": rope2_gbs / hbm},
                       "roofline": {"bound": "hbm", "achieved": rope_gbs, "peak": hbm, "unit": "GB/s",
                                    "frac": rope_gbs / hbm, "traffic": traffic("rope"),
                                    "traffic_note": "per launch of the stacked call",
                                    "frac_of_nominal": rope_gbs / NOMINAL_HBM_GBS, "nominal_peak": NOMINAL_HBM_GBS}},
    }
    if not args.no_cpu_baseline:
        v_cpu, desc, threads = cpu_oracle_prefill(w, seconds=12.0)
        line["cpu_baseline"] = {"value": v_cpu, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                                "sample": desc}
    print(json.dumps(line))
    if dist:
        dist.destroy_process_group()


def run_part(args):
    """One kernel family alone, for profiling: ``--part prefill|decode|decode_fp8|rope|backward``
    runs W + K calls of that entry point; ``--small`` shrinks the workload
    (prefill S=4096, decode B=8) while keeping inputs larger than L2."""
    from dataclasses import replace
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    n = max(1, args.warmup) + max(1, args.steps)
    if args.part == "backward":
        w = W.LLAMA2_7B if not args.small else replace(W.LLAMA2_7B, S=4096, name="llama2_7b_shape_S4096")
        cfg = cfg_of(w)
        q, k, v = W.prefill_inputs(w, dev)
        o, lse = api.attn_fwd_prefill(cfg, q, k, v, mask=w.mask, return_lse=True)
        dout = torch.randn(q.shape, device=dev).to(q.dtype)
        ws = torch.empty(api.lib_bwd_workspace_bytes(cfg, q.dtype, w.B, w.Hq, w.Hkv, w.S, w.d),
                         dtype=torch.uint8, device=dev)
        for _ in range(n):
            api.attn_bwd(cfg, q, k, v, o, dout, lse, mask=w.mask, workspace=ws)
    elif args.part in ("prefill", "rope"):
        w = W.LLAMA2_7B if not args.small else replace(W.LLAMA2_7B, S=4096, name="llama2_7b_shape_S4096")
        cfg = cfg_of(w)
        q, k, v = W.prefill_inputs(w, dev)
        o = torch.empty_like(q)
        ws = torch.empty(api.prefill_workspace_bytes(cfg, q.dtype, w.B, w.Hq, w.Hkv, w.S, w.d),
                         dtype=torch.uint8, device=dev)
        if args.part == "rope":
            qk = torch.cat([q, k], dim=1)
            qk_out = torch.empty_like(qk)
        for _ in range(n):
            if args.part == "prefill":
                api.attn_fwd_prefill(cfg, q, k, v, mask=w.mask, out=o, workspace=ws)
            else:  # rope_apply on Q and K stacked along the heads, as the bench times it
                api.rope_apply(cfg, qk, out=qk_out)
    elif args.part == "decode_fp8":
        wd = W.DECODE if not args.small else replace(W.DECODE, B=8, name="decode_B8")
        dq, kc, vc, ks, vs, nv, rs = W.decode_inputs_fp8(wd, dev)
        dcfg = api.RopeConfig(kind="plain", head_dim=wd.d, theta_base=wd.rope.theta_base)
        for _ in range(n):
            api.attn_fwd_decode_sinkwindow_fp8(dcfg, dq, kc, vc, ks, vs, nv, rs, wd.sink, wd.window)
    else:
        wd = W.DECODE if not args.small else replace(W.DECODE, B=8, name="decode_B8")
        dq, kc, vc, nv, rs = W.decode_inputs(wd, dev)
        dcfg = api.RopeConfig(kind="plain", head_dim=wd.d, theta_base=wd.rope.theta_base)
        for _ in range(n):
            api.attn_fwd_decode_sinkwindow(dcfg, dq, kc, vc, nv, rs, wd.sink, wd.window)
    api.sync_status()
    print(json.dumps({"part": args.part, "small": args.small, "calls": n}))


def _ring_check_ops(seen: list):
    """Ring operations that do no attention, for the CPU check of the ring
    launch: every K block carries its block index as its value; ``block``
    records the index it was given and returns an empty partial, and the
    rotation and the merge leave their inputs as they are."""
    from yarn_rope_scaling_ntk_b300 import ring

    def rotate(cfg, x, pos0):
        return x

    def block(q, k, v, q_pos0, k_pos0, mask, sink, window, scale, out_dtype):
        seen.append((int(k.flatten()[0].item()), k_pos0))
        o = torch.zeros(q.shape, dtype=out_dtype)
        return o, torch.full(q.shape[:3], -math.inf, dtype=torch.float32)

    def merge(o_acc, lse_acc, o_part, lse_part, out):
        pass

    return ring.RingOps(rotate, block, merge)


def run_ring(args):
    """``--ring``: the long-sequence workload (B=1, H=32, S=131072, d=128,
    YaRN s=32, causal) as ring attention over the job's N ranks.  Rank I
    holds query and KV block I of S / N tokens; every step rotates its Q and
    K, passes KV blocks around the ring with ``torch.distributed``
    point-to-point transfers (NCCL) overlapped with the block attention, and
    merges the partials.  The total work is fixed as N grows (strong
    scaling); the value is the whole sequence's attention FLOPs over the
    slowest rank's time.  With ``--launcher-check`` the ranks join a gloo
    group on the CPU and run the exchange with operations that do no
    attention, checking that each rank is handed the blocks of the ring
    order (no GPU work)."""
    from yarn_rope_scaling_ntk_b300 import ring
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    w = W.RING_128K
    cfg = cfg_of(w)
    if w.S % (world * 128):
        raise SystemExit(f"--ring needs S = {w.S} to split into {world} blocks of a multiple of 128 tokens")
    bs = w.S // world
    import torch.distributed as dist
    if args.launcher_check:
        if world > 1:
            dist.init_process_group("gloo", rank=rank, world_size=world)
        kb = torch.full((1, 1, 128, 64), float(rank), dtype=torch.float64)
        ok = True
        for _ in range(max(1, args.steps)):
            seen = []
            ops = _ring_check_ops(seen)
            small = api.RopeConfig(kind="none", head_dim=64)
            if world > 1:
                ring.ring_attention(small, kb.clone(), kb.clone(), kb.clone(), mask="causal", ops=ops)
            else:
                ring.ring_attention_one_process(small, [kb], [kb], [kb], mask="causal", ops=ops)
            want = [(j, j * 128) for j in (ring.held_block(rank, t, world) for t in range(world)) if j <= rank]
            ok = ok and seen == want
        flag = torch.tensor([1.0 if ok else 0.0], dtype=torch.float64)
        if world > 1:
            dist.all_reduce(flag, op=dist.ReduceOp.MIN)
        if rank == 0:
            print(json.dumps({"launcher_check": True, "mode": "ring", "n_gpus": world,
                              "ring_order_ok": bool(flag.item() == 1.0), "steps": args.steps}))
        if world > 1:
            dist.destroy_process_group()
        return
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    q, k, v = W.prefill_inputs(w, dev)
    sl = slice(rank * bs, (rank + 1) * bs)
    qb, kb, vb = (t[:, :, sl].contiguous() for t in (q, k, v))
    del q, k, v
    torch.cuda.empty_cache()

    def step():
        if world > 1:
            return ring.ring_attention(cfg, qb, kb, vb, mask=w.mask)
        return ring.ring_attention_one_process(cfg, [qb], [kb], [vb], mask=w.mask)[0]

    for _ in range(max(3, args.warmup)):
        step()
    api.sync_status()

    def fence():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    fence()
    n0 = api.kernel_launch_count()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        a.record(stream)
        for _ in range(args.steps):
            step()
        b.record(stream)
        fence()
    launches = api.kernel_launch_count() - n0
    api.sync_status()
    ms = a.elapsed_time(b)
    mx = reduce_max(ms, dist if world > 1 else None, dev)
    mn = -reduce_max(-ms, dist if world > 1 else None, dev)
    flops = prefill_flops(w)
    if rank == 0:
        print(json.dumps({
            "metric": "ring attention TFLOP/s (causal, whole sequence over all ranks)", "mode": "ring",
            "value": flops * args.steps / (mx * 1e-3) / 1e12, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": mx / args.steps,
            "ms_per_step_fastest_rank": mn / args.steps, "higher_is_better": True, "scaling": "strong",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.Hq, "S": w.S, "d": w.d, "mask": w.mask,
                       "block_tokens": bs, "parallelism": f"ring{world}",
                       "exchange": "torch.distributed batch_isend_irecv (NCCL)" if world > 1 else "none (one rank)",
                       "l2": "inputs larger than L2"},
            "clocks": clk.summary(), "gpu_launches": launches,
        }))
    if world > 1:
        dist.destroy_process_group()


def _free_port() -> int:
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _rank_entry(rank: int, world: int, port: int, argv: list):
    """One rank of a self-launched multi-GPU run: the environment torchrun
    would give it, then the same code path as a torchrun rank."""
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world), LOCAL_WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    _dispatch(_parse(argv))


def launch_ranks(args, argv: list) -> None:
    """``--gpus N`` without a launcher's environment: start N rank processes
    (spawned, one per GPU, ranks 0..N-1 on 127.0.0.1) that form one process
    group, as ``torch.distributed.run --nproc-per-node N`` would."""
    import torch.multiprocessing as mp
    port = _free_port()
    mp.start_processes(_rank_entry, args=(args.gpus, port, argv), nprocs=args.gpus, join=True,
                       start_method="spawn")


def run_launcher_check(args):
    """The multi-rank path without a GPU: every rank joins a gloo group,
    times a fixed CPU step, the times are reduced to the slowest rank and
    rank 0 prints one line (a check of the launcher, not a bench line)."""
    import torch.distributed as dist
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1:
        dist.init_process_group("gloo", rank=rank, world_size=world)
        dist.barrier()
    a = torch.ones(256, 256, dtype=torch.float64)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        a = (a @ a) / 256.0
    ms = (time.perf_counter() - t0) * 1e3
    mx = reduce_max(ms, dist if world > 1 else None)
    ranks = torch.zeros(1, dtype=torch.float64) + 1.0
    if world > 1:
        dist.all_reduce(ranks)
    if rank == 0:
        print(json.dumps({"launcher_check": True, "n_gpus": world, "ranks_joined": int(ranks.item()),
                          "steps": args.steps, "max_ms_over_ranks": mx}))
    if world > 1:
        dist.destroy_process_group()


def _parse(argv):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-backward", action="store_true", help="skip timing the attention backward")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="skip timing the ring 128K and GQA prefill workloads")
    ap.add_argument("--part", choices=["prefill", "decode", "decode_fp8", "rope", "backward"], default=None,
                    help="profile one kernel family alone (prints no bench line)")
    ap.add_argument("--small", action="store_true", help="with --part: smaller workload")
    ap.add_argument("--launcher-check", action="store_true",
                    help="start the ranks on CPU (gloo) and print one line per job, no GPU work")
    ap.add_argument("--ring", action="store_true",
                    help="ring attention over the N ranks on the 131072-token workload (strong scaling)")
    return ap.parse_args(argv)


def _dispatch(args):
    if args.ring and args.impl == "ours" and not args.part:
        run_ring(args)
    elif args.launcher_check:
        run_launcher_check(args)
    elif args.part:
        run_part(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


def main():
    argv = sys.argv[1:]
    args = _parse(argv)
    # N ranks are needed and no launcher started them: start them here.  The
    # reference arm runs on rank 0 alone, so it never needs them.
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ and args.impl == "ours" and not args.part:
        launch_ranks(args, argv)
        return
    _dispatch(args)


if __name__ == "__main__":
    main()
