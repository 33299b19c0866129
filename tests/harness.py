"""Test harness: run the CUDA library and the CPU oracle on the same seeded
inputs and compare. Used by the GPU parity tests, ``__graft_entry__.smoke``
and the bench's oracle leg; it is test infrastructure (it imports the oracle).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional, Sequence

import numpy as np
import torch

import gqa_inputs as I
from oracle import gqa as O

# Parity bar for delta_attn (bf16 I/O, fp32 accumulation).
REL_L2_TOL = 1e-2
MAX_ABS_TOL = 3e-2


@dataclass
class Case:
    B: int
    T: int
    start: list               # per-sequence start positions
    s_max: int
    seed: int = 0
    rope: I.RopeConfig = I.LLAMA31_ROPE
    dims: I.Dims = I.LLAMA31_8B
    dev: dict = field(default_factory=dict)     # device tensors
    host: dict = field(default_factory=dict)    # CPU copies of the inputs


def make_case(B: int, T: int, start: Sequence[int], s_max: int, seed: int = 0,
              rope: I.RopeConfig = I.LLAMA31_ROPE, weights=None, cache_device=None,
              dims: I.Dims = I.LLAMA31_8B) -> Case:
    """Seeded inputs on cuda:0 (weights may be shared between cases)."""
    start = [int(s) for s in start]
    c = Case(B, T, start, s_max, seed, rope, dims)
    if weights is None:
        gen, w = I.draw_weights(dims, seed=seed)
    else:
        gen, w = weights
    x = I.draw_x(gen, B, T)
    ck, cv = I.draw_cache(B, s_max, start, dims, seed=seed, device=cache_device)
    c.host = {"x": x, **w}
    c.dev = {k: v.to("cuda") for k, v in c.host.items()}
    c.dev["cache_k"] = ck.to("cuda")
    c.dev["cache_v"] = cv.to("cuda")
    c.dev["cache_k0"] = c.dev["cache_k"].clone()   # untouched copies for the canary check
    c.dev["cache_v0"] = c.dev["cache_v"].clone()
    return c


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


_W64 = {}


def weights64(c: Case):
    key = id(c.host["wq"])
    if key not in _W64:
        _W64.clear()
        _W64[key] = {k: f64(c.host[k]) for k in ("wq", "wk", "wv", "wo")}
    return _W64[key]


def oracle_sequence(c: Case, b: int, query_rows=None):
    """Oracle delta / new cache rows of sequence b, from the untouched cache."""
    r = c.rope
    freqs = O.rope_frequencies(128, r.theta, r.scaled, r.factor, r.low_freq_factor,
                               r.high_freq_factor, r.original_context)
    w = weights64(c)
    sp = c.start[b]
    ck = f64(c.dev["cache_k0"][b, :sp])
    cv = f64(c.dev["cache_v0"][b, :sp])
    return O.sequence_forward(f64(c.host["x"][b]), w["wq"], w["wk"], w["wv"], w["wo"], sp, ck, cv,
                              freqs, c.dims.n_heads, c.dims.n_kv_heads, query_rows)


def oracle_layer_sequence(c: Case, b: int, g: torch.Tensor, eps: float, query_rows=None):
    """Oracle h = x + attention(norm(x)) / new cache rows of sequence b."""
    r = c.rope
    freqs = O.rope_frequencies(128, r.theta, r.scaled, r.factor, r.low_freq_factor,
                               r.high_freq_factor, r.original_context)
    w = weights64(c)
    sp = c.start[b]
    ck = f64(c.dev["cache_k0"][b, :sp])
    cv = f64(c.dev["cache_v0"][b, :sp])
    return O.layer_sequence_forward(f64(c.host["x"][b]), f64(g), eps, w["wq"], w["wk"], w["wv"], w["wo"], sp,
                                    ck, cv, freqs, 32, 8, query_rows)


# Relative accuracy of the GPU's attention_norm before its bf16 rounding:
# fp32 sum of 4096 squares (at most ~2^-17 relative), one reciprocal square
# root and two products. A normalised value of the oracle (fp64) closer than
# this to a bf16 rounding midpoint may round to the neighbouring bf16 value
# on the GPU.
NORM_REL_ERR = 2.0 ** -17


def norm_flip_allowance(xn64: np.ndarray, w: np.ndarray) -> np.ndarray:
    """Per-output bound [T, rows of w] on how far x_n W^T (a K or V row before
    its bf16 rounding, RoPE partners included) can move when every normalised
    value within NORM_REL_ERR of a bf16 midpoint lands on the other side:
    sum over those inputs j of one bf16 spacing times (|W[f, j]| + |W[f^1, j]|)
    (a rotation moves one element of a pair by at most the pair's change).
    Computed from oracle values only."""
    u = bf16_ulp(xn64)
    frac = xn64 / u - np.floor(xn64 / u)
    amb = np.abs(frac - 0.5) * u <= NORM_REL_ERR * np.abs(xn64)
    aw = np.abs(w)
    aw = aw + aw.reshape(-1, 2, aw.shape[1])[:, ::-1, :].reshape(aw.shape)   # |W[f]| + |W[f ^ 1]|
    return (amb * u) @ aw.T


def compare_layer_sequence(c: Case, h: torch.Tensor, b: int, g: torch.Tensor, eps: float, query_rows=None):
    """Oracle vs GPU for the layer h = x + attention(norm(x)) of sequence b,
    everything on the oracle side from the case's own inputs: h at the delta
    bar; the written K/V rows within one bf16 ulp of the oracle layer's rows,
    widened by ``norm_flip_allowance`` for normalised values that sit on a
    bf16 rounding midpoint (where fp32 and fp64 may round apart)."""
    hl, nk, nv = oracle_layer_sequence(c, b, g, eps, query_rows)
    rows = slice(None) if query_rows is None else list(query_rows)
    got = f64(h[b])[rows]
    r2 = rel_l2(got, hl)
    ma = float(np.abs(got - hl).max())
    assert np.isfinite(got).all(), f"non-finite output in sequence {b}"
    assert r2 <= REL_L2_TOL, f"sequence {b}: rel L2 {r2:.3e} > {REL_L2_TOL}"
    assert ma <= MAX_ABS_TOL, f"sequence {b}: max abs {ma:.3e} > {MAX_ABS_TOL}"
    xn64 = O.rms_norm(f64(c.host["x"][b]), f64(g), eps)
    w = weights64(c)
    sp, T = c.start[b], c.T
    shape = nk.shape
    check_rows_within_one_ulp(c.dev["cache_k"][b, sp:sp + T], nk, f"cache_k rows of sequence {b}",
                              norm_flip_allowance(xn64, w["wk"]).reshape(shape))
    check_rows_within_one_ulp(c.dev["cache_v"][b, sp:sp + T], nv, f"cache_v rows of sequence {b}",
                              norm_flip_allowance(xn64, w["wv"]).reshape(shape))
    return r2, ma


def rel_l2(got: np.ndarray, ref: np.ndarray) -> float:
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30))


def ordered_bf16(t: torch.Tensor) -> np.ndarray:
    """bf16 bit patterns mapped to integers that order like the values."""
    bits = t.contiguous().view(torch.int16).to(torch.int32).numpy()
    mag = bits & 0x7FFF
    return np.where(bits < 0, -mag, mag)


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at |v| (8 significant bits, fp32 exponent range)."""
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, 2.0 ** (np.maximum(e, -126) - 7), 2.0 ** -133)


# Absolute floor of the cache-row check, relative to the RMS of the 128-value
# head row: an fp32 dot product of 4096 terms carries an error of order
# 2^-24 * sqrt(4096) = 2^-18 of the row scale, so values that cancel to
# nearly zero cannot be pinned to their own (tiny) bf16 ulp.
CACHE_FLOOR = 2.0 ** -16


def check_rows_within_one_ulp(got_bf16: torch.Tensor, ref64: np.ndarray, what: str, extra=None):
    """|got - ref| <= ulp_bf16(ref) + CACHE_FLOOR * rms(head row of ref)
    (+ ``extra``, an input-rounding allowance of the same shape, if given)."""
    got = got_bf16.detach().to("cpu", torch.float64).numpy()
    rms = np.sqrt(np.mean(ref64 ** 2, axis=-1, keepdims=True))
    tol = bf16_ulp(ref64) + CACHE_FLOOR * rms
    if extra is not None:
        tol = tol + extra
    err = np.abs(got - ref64)
    bad = err > tol
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} values beyond 1 bf16 ulp "
                           f"(worst excess {float((err - tol).max()):.3e}, at ref "
                           f"{float(ref64.reshape(-1)[np.argmax((err - tol).reshape(-1))]):.3e})")


def compare_sequence(c: Case, out: torch.Tensor, b: int, query_rows=None, check_cache=True):
    """Oracle vs GPU for sequence b; returns (rel_l2, max_abs)."""
    dl, nk, nv = oracle_sequence(c, b, query_rows)
    rows = slice(None) if query_rows is None else list(query_rows)
    got = f64(out[b])[rows]
    r2 = rel_l2(got, dl)
    ma = float(np.abs(got - dl).max())
    assert np.isfinite(got).all(), f"non-finite output in sequence {b}"
    assert r2 <= REL_L2_TOL, f"sequence {b}: rel L2 {r2:.3e} > {REL_L2_TOL}"
    assert ma <= MAX_ABS_TOL, f"sequence {b}: max abs {ma:.3e} > {MAX_ABS_TOL}"
    if check_cache:
        sp, T = c.start[b], c.T
        check_rows_within_one_ulp(c.dev["cache_k"][b, sp:sp + T], nk, f"cache_k rows of sequence {b}")
        check_rows_within_one_ulp(c.dev["cache_v"][b, sp:sp + T], nv, f"cache_v rows of sequence {b}")
    return r2, ma


def check_canaries(c: Case, seqs=None):
    """Cache rows outside [start_b, start_b + T) must be bit-identical."""
    for b in (range(c.B) if seqs is None else seqs):
        sp = c.start[b]
        for name in ("cache_k", "cache_v"):
            now, before = c.dev[name][b], c.dev[name + "0"][b]
            assert torch.equal(now[:sp], before[:sp]), f"{name}[{b}] rows before start_pos changed"
            assert torch.equal(now[sp + c.T:], before[sp + c.T:]), f"{name}[{b}] rows after the new ones changed"


def rope_for(c: Case, rows: Optional[int] = None):
    import grouped_query_attention_gemv_gb300 as G
    r = c.rope
    return G.rope_table(rows or c.s_max, r.theta, r.scaled, r.factor, r.low_freq_factor,
                        r.high_freq_factor, r.original_context)
