"""Synthetic workloads: shapes and seeded input generators.

This module holds no arithmetic of the method -- only the workload shapes and
random draws.  Tests hand the same generated tensors to the CUDA library and to
the float64 oracle; ``bench.py`` uses the same generators.

Every workload draws i.i.d. N(0, 1) values (the pages use no dataset; all
inputs are synthetic).  Q, K, V are drawn in that order from one
``torch.Generator`` seeded with ``1000 + index`` and then cast to the
workload's dtype.
"""

from __future__ import annotations

from dataclasses import dataclass, field, replace

import torch


@dataclass(frozen=True)
class RopeSpec:
    kind: str = "yarn"          # none | plain | pi | ntk | yarn
    theta_base: float = 10000.0
    L_train: int = 0
    L_target: int = 0
    s: float = 0.0              # <= 0: L_target / L_train
    ramp_alpha: float = 1.0
    ramp_beta: float = 32.0


@dataclass(frozen=True)
class Prefill:
    name: str
    index: int
    B: int
    Hq: int
    Hkv: int
    S: int
    d: int
    dtype: torch.dtype
    rope: RopeSpec
    mask: str = "causal"        # causal | sink_window | none
    sink: int = 0
    window: int = 0
    ring_blocks: int = 1
    rows_per_head: int = 0      # oracle rows sampled per head (0: all rows)


@dataclass(frozen=True)
class Decode:
    name: str
    index: int
    B: int
    Hq: int
    Hkv: int
    d: int
    sink: int
    window: int
    rope: RopeSpec = field(default_factory=lambda: RopeSpec(kind="plain"))
    full: bool = True           # every sequence has a full cache


TINY = Prefill("tiny_prefill_B1_H4_S256_d64_fp32_yarn4", 1, 1, 4, 4, 256, 64, torch.float32,
               RopeSpec("yarn", 1e4, 64, 256, 4.0), "causal", ring_blocks=4)
LLAMA2_7B = Prefill("llama2_7b_prefill_B1_H32_S16384_d128_bf16_yarn4", 2, 1, 32, 32, 16384, 128,
                    torch.bfloat16, RopeSpec("yarn", 1e4, 4096, 16384, 4.0), "causal",
                    rows_per_head=256)
DECODE = Decode("sink_window_decode_B64_H32_d128_sink4_win4092", 3, 64, 32, 32, 128, 4, 4092)
RING_128K = Prefill("ring_prefill_B1_H32_S131072_d128_bf16_yarn32_8blocks", 4, 1, 32, 32, 131072,
                    128, torch.bfloat16, RopeSpec("yarn", 1e4, 4096, 131072, 32.0), "causal",
                    ring_blocks=8, rows_per_head=128)
LLAMA3_8B_GQA = Prefill("llama3_8b_gqa_prefill_B4_Hq32_Hkv8_S32768_d128_bf16_yarn4", 5, 4, 32, 8,
                        32768, 128, torch.bfloat16, RopeSpec("yarn", 5e5, 8192, 32768, 4.0),
                        "causal", rows_per_head=32)
LLAMA3_8B_GQA_SW = replace(LLAMA3_8B_GQA, name=LLAMA3_8B_GQA.name + "_sink4_win8192",
                           mask="sink_window", sink=4, window=8192)

PREFILL_WORKLOADS = {w.name: w for w in (TINY, LLAMA2_7B, RING_128K, LLAMA3_8B_GQA, LLAMA3_8B_GQA_SW)}


def generator(index: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(1000 + index)
    return g


def prefill_inputs(w: Prefill, device="cpu", seed_index: int | None = None):
    """Q [B,Hq,S,d], K [B,Hkv,S,d], V [B,Hkv,S,d] in ``w.dtype``."""
    g = generator(w.index if seed_index is None else seed_index, device)
    q = torch.randn(w.B, w.Hq, w.S, w.d, generator=g, device=device, dtype=torch.float32)
    k = torch.randn(w.B, w.Hkv, w.S, w.d, generator=g, device=device, dtype=torch.float32)
    v = torch.randn(w.B, w.Hkv, w.S, w.d, generator=g, device=device, dtype=torch.float32)
    return q.to(w.dtype), k.to(w.dtype), v.to(w.dtype)


def decode_inputs(w: Decode, device="cpu", seed_index: int | None = None):
    """q [B,Hq,d], k_cache/v_cache [B,Hkv,sink+window,d] (bf16), n_valid [B]
    and ring_start [B] (int32).  A full cache has n_valid = sink + window and a
    seeded ring_start in [0, window); otherwise n_valid is drawn in
    [1, sink + window] and ring_start in [0, window)."""
    g = generator(w.index if seed_index is None else seed_index, device)
    C = w.sink + w.window
    q = torch.randn(w.B, w.Hq, w.d, generator=g, device=device).to(torch.bfloat16)
    kc = torch.randn(w.B, w.Hkv, C, w.d, generator=g, device=device).to(torch.bfloat16)
    vc = torch.randn(w.B, w.Hkv, C, w.d, generator=g, device=device).to(torch.bfloat16)
    ring_start = torch.randint(0, max(w.window, 1), (w.B,), generator=g, device=device,
                               dtype=torch.int32)
    if w.full:
        n_valid = torch.full((w.B,), C, dtype=torch.int32, device=device)
    else:
        n_valid = torch.randint(1, C + 1, (w.B,), generator=g, device=device, dtype=torch.int32)
    return q, kc, vc, n_valid, ring_start


def sample_rows(S: int, count: int, index: int, extra=()):
    """Seeded query rows of one head plus forced boundary rows: 0, 1, the
    128-row tile edges 127/128/129, S-1 and any ``extra`` rows (ring-block
    edges, window edges).  ``count <= 0`` returns every row."""
    if count <= 0 or count >= S:
        return torch.arange(S)
    g = torch.Generator().manual_seed(7000 + index)
    r = torch.randint(0, S, (count,), generator=g)
    forced = torch.tensor([x for x in (0, 1, 127, 128, 129, S - 1, *extra) if 0 <= x < S])
    return torch.unique(torch.cat([r, forced]))


def decode_inputs_fp8(w: Decode, device="cpu", seed_index: int | None = None):
    """The decode inputs with the caches stored as FP8 E4M3: K and V drawn
    N(0, 1) as in ``decode_inputs``, then each (sequence, KV head) stored as
    E4M3 bytes of x / scale with scale = max|x| / 448 (the largest E4M3
    magnitude).  Returns q (bf16), k_codes, v_codes (uint8), k_scale,
    v_scale (float32 [B, Hkv]), n_valid, ring_start."""
    g = generator(w.index if seed_index is None else seed_index, device)
    C = w.sink + w.window
    q = torch.randn(w.B, w.Hq, w.d, generator=g, device=device).to(torch.bfloat16)
    k = torch.randn(w.B, w.Hkv, C, w.d, generator=g, device=device)
    v = torch.randn(w.B, w.Hkv, C, w.d, generator=g, device=device)
    ring_start = torch.randint(0, max(w.window, 1), (w.B,), generator=g, device=device, dtype=torch.int32)
    if w.full:
        n_valid = torch.full((w.B,), C, dtype=torch.int32, device=device)
    else:
        n_valid = torch.randint(1, C + 1, (w.B,), generator=g, device=device, dtype=torch.int32)
    out = []
    for x in (k, v):
        scale = (x.abs().amax(dim=(2, 3)) / 448.0).clamp_min(1e-12)
        codes = (x / scale[:, :, None, None]).to(torch.float8_e4m3fn).view(torch.uint8)
        out += [codes.contiguous(), scale.float().contiguous()]
        del x
    kc, ks, vc, vs = out
    return q, kc, vc, ks, vs, n_valid, ring_start
