"""Seeded synthetic inputs for the Llama-3.1-8B grouped-query attention block.

This module is the one piece shared by the CUDA library's callers (tests,
bench) and the CPU oracle. It only *draws* tensors: it holds none of the
block's arithmetic (no projection, RoPE, table, softmax or rounding rule of the
method). Shapes and distributions follow the workloads described on the pages
"Llama 3.1 8B · Grouped-query attention" (the in/out/state header and the
parameter table) and "Llama 3.1 8B · Query projection".

Recipe (every tensor is a torch CPU tensor unless stated):
  * one ``torch.Generator('cpu')`` seeded with ``seed`` draws, in this order,
    Wq [4096,4096], Wk [1024,4096], Wv [1024,4096], Wo [4096,4096] as fp32
    normals scaled by 1/64 (variance 1/4096) and rounded to bf16, then
    x [B,T,4096] as N(0,1) rounded to bf16;
  * the cache draw uses its own generator seeded ``seed + 1``: rows
    0..P_b-1 of cache_k then cache_v get N(0,1) bf16 values, all other rows
    are zero. Caches above ``DEVICE_DRAW_THRESHOLD`` elements are drawn by
    torch's CUDA Philox generator on the device (the CPU Mersenne Twister
    needs minutes for the multi-GB caches); callers copy rows back to host
    memory when the oracle needs them;
  * per-sequence P for the batched-decode workload comes from a separate CPU
    generator seeded ``seed``: ``randint(512, 32769)`` (both ends inclusive).
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass
from typing import Optional, Sequence

import torch

__all__ = [
    "Dims", "RopeConfig", "Workload", "WORKLOADS", "LLAMA31_8B", "LLAMA31_8B_MHA", "LLAMA31_ROPE",
    "LLAMA3_ROPE", "draw_weights", "draw_x", "draw_cache", "draw_start_positions", "draw_norm_weight",
    "NORM_EPS",
    "workload", "DEVICE_DRAW_THRESHOLD",
]

# Caches with more elements than this (per K or V tensor) are drawn on the
# device; see the module docstring.
DEVICE_DRAW_THRESHOLD = 1 << 27


@dataclass(frozen=True)
class Dims:
    """Model dimensions of one attention block (catalogue entry arch_args)."""
    d_model: int = 4096
    n_heads: int = 32
    n_kv_heads: int = 8
    head_dim: int = 128

    @property
    def n_rep(self) -> int:
        return self.n_heads // self.n_kv_heads


@dataclass(frozen=True)
class RopeConfig:
    """Rotary-embedding settings: rope_theta and use_scaled_rope from the
    catalogue entries; the scaling constants are the Llama 3.1 values
    (factor 8, low/high frequency factor 1/4, original context 8192)."""
    theta: float = 500000.0
    scaled: bool = True
    factor: float = 8.0
    low_freq_factor: float = 1.0
    high_freq_factor: float = 4.0
    original_context: int = 8192


LLAMA31_8B = Dims()
# The multi-head variant the "Grouped-query attention" page sets against the
# model: 32 K/V heads, one per query head (repeat_kv is the identity).
LLAMA31_8B_MHA = Dims(n_kv_heads=32)
LLAMA31_ROPE = RopeConfig()
# "Llama 3 8B · Attention update" page: same dims, use_scaled_rope False.
LLAMA3_ROPE = RopeConfig(scaled=False)


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: batch B, new tokens T per sequence, cached
    positions (uniform ``start_pos`` or drawn per sequence) and cache rows."""
    name: str
    B: int
    T: int
    start_pos: Optional[int]          # uniform P; None = drawn per sequence
    p_range: Optional[tuple] = None   # (lo, hi) inclusive, when drawn
    s_max: Optional[int] = None       # cache rows per sequence
    seed: int = 0
    description: str = ""
    layers: int = 1                   # consecutive blocks per step (each with its own weights and cache)
    n_kv_heads: int = 8               # 32: the multi-head variant

    @property
    def dims(self) -> "Dims":
        return LLAMA31_8B if self.n_kv_heads == LLAMA31_8B.n_kv_heads else Dims(n_kv_heads=self.n_kv_heads)

    def start_positions(self) -> torch.Tensor:
        if self.start_pos is not None:
            return torch.full((self.B,), self.start_pos, dtype=torch.int32)
        return draw_start_positions(self.B, self.p_range, self.seed)

    def cache_rows(self) -> int:
        if self.s_max is not None:
            return self.s_max
        return int(self.start_positions().max()) + self.T


WORKLOADS = {
    w.name: w for w in [
        Workload("decode_b1_p15", B=1, T=1, start_pos=15, s_max=16,
                 description="decode, B=1, P=15 (16 keys)"),
        Workload("decode_b16_p1000", B=16, T=1, start_pos=1000, s_max=1001,
                 description="decode at P=1000, B=16 (1,001 keys read, row 1000 written)"),
        Workload("batched_decode_b64_p512_32768", B=64, T=1, start_pos=None,
                 p_range=(512, 32768),
                 description="batched decode, B=64, P_b ~ U[512, 32768]"),
        Workload("prefill_b1_t2048", B=1, T=2048, start_pos=0, s_max=2048,
                 description="causal prefill, B=1, T=2048"),
        Workload("prefill_b4_t2048", B=4, T=2048, start_pos=0, s_max=2048,
                 description="causal prefill, B=4, T=2048"),
        Workload("long_decode_b8_p131071", B=8, T=1, start_pos=131071, s_max=131072,
                 description="long-context decode, B=8, P=131071 (131,072 keys)"),
        Workload("mha_decode_b16_p1000", B=16, T=1, start_pos=1000, s_max=1001, n_kv_heads=32,
                 description="the multi-head variant (32 K/V heads) at the decode point P=1000, B=16: "
                             "4x the KV rows of the grouped model (16 KB per position)"),
        Workload("mha_prefill_b1_t2048", B=1, T=2048, start_pos=0, s_max=2048, n_kv_heads=32,
                 description="the multi-head variant's causal prefill, B=1, T=2048"),
        Workload("decode32_b16_p1000", B=16, T=1, start_pos=1000, s_max=1001, layers=32,
                 description="32 consecutive layers of one decode step at P=1000, B=16: the attention half "
                             "of each block with its norm and residual (h = x + attention(RMSNorm(x))), each "
                             "layer with its own weights and KV cache in device memory (copies of one seeded "
                             "draw), the output of one the input of the next"),
        Workload("prefill_chunk_b1_t1024_p7168", B=1, T=1024, start_pos=7168, s_max=8192,
                 description="chunked prefill: the last 1,024 tokens of an 8,192-token prompt "
                             "after 7,168 cached positions"),
    ]
}


def workload(name: str, **overrides) -> Workload:
    w = WORKLOADS[name]
    return dataclasses.replace(w, **overrides) if overrides else w


def _normal_bf16(gen: torch.Generator, shape, std: float) -> torch.Tensor:
    t = torch.randn(*shape, generator=gen, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(torch.bfloat16)


def draw_weights(dims: Dims = LLAMA31_8B, seed: int = 0):
    """Return (gen, dict) with bf16 Wq, Wk, Wv, Wo stored [out, in].

    The generator is returned so that ``draw_x`` continues the same stream."""
    gen = torch.Generator("cpu").manual_seed(seed)
    std = dims.d_model ** -0.5
    kv = dims.n_kv_heads * dims.head_dim
    w = {
        "wq": _normal_bf16(gen, (dims.n_heads * dims.head_dim, dims.d_model), std),
        "wk": _normal_bf16(gen, (kv, dims.d_model), std),
        "wv": _normal_bf16(gen, (kv, dims.d_model), std),
        "wo": _normal_bf16(gen, (dims.d_model, dims.n_heads * dims.head_dim), std),
    }
    return gen, w


def draw_x(gen: torch.Generator, B: int, T: int, dims: Dims = LLAMA31_8B) -> torch.Tensor:
    return _normal_bf16(gen, (B, T, dims.d_model), 1.0)


def draw_start_positions(B: int, p_range: Sequence[int], seed: int = 0) -> torch.Tensor:
    lo, hi = p_range
    gen = torch.Generator("cpu").manual_seed(seed)
    return torch.randint(lo, hi + 1, (B,), generator=gen, dtype=torch.int64).to(torch.int32)


def draw_cache(B: int, s_max: int, filled_rows: Sequence[int], dims: Dims = LLAMA31_8B,
               seed: int = 0, device: Optional[str] = None):
    """Return (cache_k, cache_v), bf16 [B, s_max, n_kv_heads, head_dim].

    Rows 0..filled_rows[b]-1 of sequence b hold N(0,1) draws; other rows are
    zero. ``device=None`` picks the CPU generator for small caches and the
    CUDA generator above DEVICE_DRAW_THRESHOLD elements."""
    row = dims.n_kv_heads * dims.head_dim
    n = B * s_max * row
    if device is None:
        device = "cuda" if n > DEVICE_DRAW_THRESHOLD else "cpu"
    gen = torch.Generator(device).manual_seed(seed + 1)
    out = []
    for _ in ("k", "v"):
        c = torch.zeros(B, s_max, dims.n_kv_heads, dims.head_dim, dtype=torch.bfloat16,
                        device=device)
        for b in range(B):
            p = int(filled_rows[b])
            if p > 0:
                vals = torch.randn(p, dims.n_kv_heads, dims.head_dim, generator=gen,
                                   dtype=torch.float32, device=device)
                c[b, :p] = vals.to(torch.bfloat16)
        out.append(c)
    return out[0], out[1]


# norm_eps of the catalogue entries
NORM_EPS = 1e-5


def draw_norm_weight(seed: int = 0, dims: Dims = LLAMA31_8B) -> torch.Tensor:
    """attention_norm weight g [d_model] bf16: 1 + 0.1 N(0,1) from a CPU
    generator seeded ``seed + 2`` (trained weights are not available; a
    weight near 1 with spread keeps the normalised rows at the block's scale
    and makes a dropped or misplaced g visible)."""
    gen = torch.Generator("cpu").manual_seed(seed + 2)
    return (1.0 + 0.1 * torch.randn(dims.d_model, generator=gen, dtype=torch.float32)).to(torch.bfloat16)

