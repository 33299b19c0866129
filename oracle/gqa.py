"""CPU oracle for the Llama-3.1-8B grouped-query attention block (NumPy, fp64).

TEST INFRASTRUCTURE. Only the tests, the package smoke check and the bench's
CPU-baseline / reference leg may import this module. The CUDA library never
calls it and shares no code with it.

What it computes is the plain definition of the block as the pages state it
("Llama 3.1 8B · Grouped-query attention", mode decode, and its excerpts
``Attention.forward``, ``apply_rotary_emb``, ``repeat_kv``, the causal mask
built in ``Transformer.forward``; "Llama 3.1 8B · Query projection" for the
[out, in] weight storage read by ``F.linear``). Every step is exact
arithmetic in float64 except where the method itself stores a value:

  1. q = x Wq^T, k = x Wk^T, v = x Wv^T            (bias-free linears)
  2. q, k rotated pairwise by RoPE at absolute position start_pos + t
  3. k and v rounded to bf16 and appended to the cache at rows start_pos + t
  4. per query head h (KV head h // n_rep): softmax(q k^T / sqrt(d_h) + causal
     mask) over cache rows 0..start_pos+t, weights applied to the cached V
  5. heads merged (feature h*d_h + d) and projected: delta = o Wo^T

Readings of points the pages leave open are stated where they are used:
  * RoPE frequencies f_i = theta^(-2i/d_h) and the Llama 3.1 frequency
    rescaling (the pages name the rule but do not print it);
  * pair i of a head is the adjacent pair (x[2i], x[2i+1]) read as the complex
    number x[2i] + j x[2i+1] (``view_as_complex`` of a trailing reshape to 2);
  * the cache holds K after RoPE and V as projected, both in bf16, laid out
    [B, S_max, n_kv_heads, d_h]; only the stored cache rows are rounded.

The block's attention half with its residual (``rms_norm``,
``layer_sequence_forward``, ``layer_forward``) follows the handoff excerpt
h = x + attention(attention_norm(x)); RMSNorm's body is read as the usual
root-mean-square normalisation (the pages do not print it), and its output,
the attention's input tensor, is stored in bf16 like the block input.

Parity status: every function here is pinned by the CPU tests (page
figures, invariants, closed forms, brute force) except the exact values of
the scaled-RoPE frequencies inside the interpolation band, which the pages
never print: that part is "parity unpinned" beyond its band-edge and
limit-case pins.
"""
from __future__ import annotations

import math
from typing import Iterable, Optional, Sequence

import numpy as np

__all__ = [
    "param_counts", "kv_cache_bytes_per_token", "bf16_round", "rope_frequencies",
    "rope_cos_sin", "rope_rotate", "softmax", "sequence_forward", "block_forward",
]


# ---------------------------------------------------------------------------
# Sizes ("Parameters" tables and the "In numbers" KV-cache figures)
# ---------------------------------------------------------------------------

def param_counts(d_model: int, n_heads: int, n_kv_heads: int, head_dim: int) -> dict:
    """Per-block parameter counts of the four bias-free projections.

    Weights are stored [out, in]: Wq [H*d_h, d], Wk and Wv [H_kv*d_h, d],
    Wo [d, H*d_h] ("Exact per-instance accounting" table)."""
    q = n_heads * head_dim * d_model
    kv = n_kv_heads * head_dim * d_model
    o = d_model * n_heads * head_dim
    return {"wq": q, "wk": kv, "wv": kv, "wo": o, "total": q + 2 * kv + o}


def kv_cache_bytes_per_token(n_layers: int, n_kv_heads: int, head_dim: int,
                             bytes_per_value: int = 2) -> int:
    """K and V for every layer and KV head at one position ("In numbers")."""
    return 2 * n_layers * n_kv_heads * head_dim * bytes_per_value


# ---------------------------------------------------------------------------
# bf16 storage rounding
# ---------------------------------------------------------------------------

def bf16_round(a) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 value, ties to even.

    bfloat16 keeps 8 significant bits and fp32's exponent range: a normal
    value m * 2**e (0.5 <= |m| < 1) is rounded at a spacing of 2**(e-8);
    below 2**-126 the spacing stays 2**-133 (subnormals). Results at or
    above 2**128 overflow to infinity."""
    a = np.asarray(a, dtype=np.float64)
    out = a.copy()
    fin = np.isfinite(a) & (a != 0.0)
    v = a[fin]
    _, e = np.frexp(v)
    e = np.maximum(e, -125)
    r = np.ldexp(np.rint(np.ldexp(v, 8 - e)), e - 8)
    r = np.where(np.abs(r) >= 2.0 ** 128, np.copysign(np.inf, r), r)
    out[fin] = r
    return out


# ---------------------------------------------------------------------------
# Rotary embedding
# ---------------------------------------------------------------------------

def rope_frequencies(head_dim: int, theta: float, scaled: bool, factor: float = 8.0,
                     low_freq_factor: float = 1.0, high_freq_factor: float = 4.0,
                     original_context: int = 8192) -> np.ndarray:
    """Angular frequency of each of the head_dim/2 pairs.

    Base: f_i = theta^(-2i/d_h). With use_scaled_rope (Llama 3.1), pairs whose
    wavelength 2*pi/f_i is shorter than original_context/high_freq_factor
    keep f_i, those longer than original_context/low_freq_factor get
    f_i/factor, and the band between interpolates linearly in
    mu = (original_context/wavelength - low) / (high - low) between the two."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    f = theta ** (-2.0 * i / head_dim)
    if not scaled:
        return f
    wavelength = 2.0 * math.pi / f
    short_edge = original_context / high_freq_factor
    long_edge = original_context / low_freq_factor
    mu = (original_context / wavelength - low_freq_factor) / (high_freq_factor - low_freq_factor)
    mid = (1.0 - mu) * f / factor + mu * f
    return np.where(wavelength < short_edge, f, np.where(wavelength > long_edge, f / factor, mid))


def rope_cos_sin(positions: Iterable[int], freqs: np.ndarray):
    """cos and sin of position * f_i, shape [len(positions), d_h/2]."""
    p = np.asarray(list(positions) if not isinstance(positions, np.ndarray) else positions,
                   dtype=np.float64)
    ang = np.outer(p, freqs)
    return np.cos(ang), np.sin(ang)


def rope_rotate(v: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """Rotate adjacent pairs of the last axis: (a, b) -> (a c - b s, a s + b c).

    ``cos``/``sin`` broadcast against v[..., 0::2]; this is the complex
    product (a + j b) * (c + j s) of ``apply_rotary_emb``."""
    a = v[..., 0::2]
    b = v[..., 1::2]
    out = np.empty_like(v, dtype=np.float64)
    out[..., 0::2] = a * cos - b * sin
    out[..., 1::2] = a * sin + b * cos
    return out


def softmax(s: np.ndarray, axis: int = -1) -> np.ndarray:
    """exp(s - max) / sum(exp(s - max)); -inf entries get weight 0."""
    m = np.max(s, axis=axis, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=axis, keepdims=True)


# ---------------------------------------------------------------------------
# The block
# ---------------------------------------------------------------------------

def sequence_forward(x: np.ndarray, wq: np.ndarray, wk: np.ndarray, wv: np.ndarray,
                     wo: np.ndarray, start_pos: int, cached_k: np.ndarray,
                     cached_v: np.ndarray, freqs: np.ndarray, n_heads: int,
                     n_kv_heads: int, query_rows: Optional[Sequence[int]] = None):
    """One sequence of the block.

    x          [T, d] float64 (bf16-exact values)
    w*         [out, in] float64
    start_pos  cached positions before this call
    cached_k/v [start_pos, n_kv_heads, d_h] cache rows 0..start_pos-1
    freqs      per-pair angular frequencies (``rope_frequencies``)
    query_rows subset of t in [0, T) whose delta is wanted (default all)

    Returns (delta [len(query_rows), d], new_k [T, n_kv, d_h], new_v [T, n_kv, d_h]);
    new_k/new_v are the rows written to the cache at start_pos..start_pos+T-1.
    """
    T, d = x.shape
    head_dim = wq.shape[0] // n_heads
    n_rep = n_heads // n_kv_heads
    rows = np.arange(T) if query_rows is None else np.asarray(query_rows, dtype=np.int64)
    pos = start_pos + np.arange(T)
    cos, sin = rope_cos_sin(pos, freqs)

    # 1-2: projections, head split, RoPE on keys (all new rows) and queries
    k = (x @ wk.T).reshape(T, n_kv_heads, head_dim)
    v = (x @ wv.T).reshape(T, n_kv_heads, head_dim)
    k = rope_rotate(k, cos[:, None, :], sin[:, None, :])
    q = (x[rows] @ wq.T).reshape(len(rows), n_heads, head_dim)
    q = rope_rotate(q, cos[rows][:, None, :], sin[rows][:, None, :])

    # 3: the stored rows are bf16
    new_k = bf16_round(k)
    new_v = bf16_round(v)
    keys = np.concatenate([cached_k, new_k], axis=0)     # [start_pos+T, n_kv, d_h]
    values = np.concatenate([cached_v, new_v], axis=0)
    L = keys.shape[0]

    # 4: causal softmax attention; query row t sees keys j <= start_pos + t
    visible = np.arange(L)[None, :] <= (start_pos + rows)[:, None]      # [R, L]
    o = np.empty((len(rows), n_heads, head_dim))
    scale = 1.0 / math.sqrt(head_dim)
    R = len(rows)
    for g in range(n_kv_heads):
        heads = slice(g * n_rep, (g + 1) * n_rep)                 # KV head g serves h // n_rep == g
        qg = q[:, heads, :].reshape(R * n_rep, head_dim)          # (row, head) pairs
        s = (qg @ keys[:, g, :].T).reshape(R, n_rep, L) * scale
        s = np.where(visible[:, None, :], s, -np.inf)
        p = softmax(s, axis=-1)
        o[:, heads, :] = (p.reshape(R * n_rep, L) @ values[:, g, :]).reshape(R, n_rep, head_dim)

    # 5: merge heads (feature h*d_h + d) and project
    delta = o.reshape(len(rows), n_heads * head_dim) @ wo.T
    return delta, new_k, new_v


def block_forward(x: np.ndarray, weights: dict, start_pos, cache_k: np.ndarray,
                  cache_v: np.ndarray, freqs: np.ndarray, n_heads: int, n_kv_heads: int):
    """Whole batch: x [B, T, d]; start_pos an int or a length-B sequence;
    cache_k/v [B, S_max, n_kv, d_h] (float64, not modified).

    Returns (delta [B, T, d], cache_k', cache_v') with the new rows written."""
    B, T, _ = x.shape
    sp = [int(start_pos)] * B if np.isscalar(start_pos) else [int(s) for s in start_pos]
    delta = np.empty((B, T, weights["wo"].shape[0]))
    ck, cv = cache_k.copy(), cache_v.copy()
    for b in range(B):
        dl, nk, nv = sequence_forward(x[b], weights["wq"], weights["wk"], weights["wv"],
                                      weights["wo"], sp[b], cache_k[b, :sp[b]],
                                      cache_v[b, :sp[b]], freqs, n_heads, n_kv_heads)
        delta[b] = dl
        ck[b, sp[b]:sp[b] + T] = nk
        cv[b, sp[b]:sp[b] + T] = nv
    return delta, ck, cv


def rms_norm(x: np.ndarray, weight: np.ndarray, eps: float) -> np.ndarray:
    """attention_norm of the block: "Llama 3.1 8B · Grouped-query attention",
    handoff excerpt (``RMSNorm(args.dim, eps=args.norm_eps)``, norm_eps 1e-05 in
    the catalogue entry). The pages name the module without printing its body;
    read as y_i = g_i x_i / sqrt(mean_j x_j^2 + eps) over the model dimension
    (the last axis), float64, no intermediate rounding."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * weight


def layer_sequence_forward(x: np.ndarray, norm_weight: np.ndarray, eps: float, wq: np.ndarray,
                           wk: np.ndarray, wv: np.ndarray, wo: np.ndarray, start_pos: int,
                           cached_k: np.ndarray, cached_v: np.ndarray, freqs: np.ndarray,
                           n_heads: int, n_kv_heads: int, query_rows: Optional[Sequence[int]] = None):
    """The block's attention half with its residual for one sequence:
    h = x + attention(attention_norm(x)) (the handoff excerpt of "Llama 3.1 8B ·
    Grouped-query attention"; "Llama 3 8B · Attention update", block-residuals).

    The normalised rows are the attention's input tensor and are stored in
    bf16, as the block input x is: every module excerpt on the pages hands
    its result back in its input's dtype (apply_rotary_emb, the softmax), so
    they are rounded once here.

    Returns (h [len(query_rows), d], new_k, new_v) as ``sequence_forward``."""
    rows = np.arange(x.shape[0]) if query_rows is None else np.asarray(query_rows, dtype=np.int64)
    xn = bf16_round(rms_norm(x, norm_weight, eps))
    delta, new_k, new_v = sequence_forward(xn, wq, wk, wv, wo, start_pos, cached_k, cached_v, freqs, n_heads,
                                           n_kv_heads, query_rows)
    return x[rows] + delta, new_k, new_v


def layer_forward(x: np.ndarray, norm_weight: np.ndarray, eps: float, weights: dict, start_pos,
                  cache_k: np.ndarray, cache_v: np.ndarray, freqs: np.ndarray, n_heads: int,
                  n_kv_heads: int):
    """Whole batch of ``layer_sequence_forward``: returns (h [B, T, d], cache_k', cache_v')."""
    delta, ck, cv = block_forward(bf16_round(rms_norm(x, norm_weight, eps)), weights, start_pos, cache_k, cache_v,
                                  freqs, n_heads, n_kv_heads)
    return x + delta, ck, cv
