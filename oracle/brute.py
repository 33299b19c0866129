"""Pure-Python brute-force restatement of the attention block, for tiny shapes.

TEST INFRASTRUCTURE (same import rule as ``oracle.gqa``). It exists to pin the
NumPy oracle from a second, independent route: nested Python loops over
scalars, RoPE applied with Python ``complex`` arithmetic (the pages'
``view_as_complex`` + multiply by the unit phasor ``freqs_cis``), the GQA map
written as an explicit expansion of KV heads (``repeat_kv``: copy g of the
expanded axis is index g // n_rep), the causal mask added as -inf, and bf16
rounding done with ``math.frexp`` and Python's round-half-even ``round``.
It shares no helper with ``oracle.gqa``.
"""
from __future__ import annotations

import cmath
import math


def bf16(v: float) -> float:
    """Nearest bfloat16 value (8 significant bits, ties to even)."""
    if v == 0.0 or math.isinf(v) or math.isnan(v):
        return v
    m, e = math.frexp(v)
    e = max(e, -125)
    r = round(math.ldexp(v, 8 - e)) * 2.0 ** (e - 8)
    if abs(r) >= 2.0 ** 128:
        return math.copysign(math.inf, r)
    return r


def frequency(i: int, head_dim: int, theta: float, scaled: bool, factor: float = 8.0,
              low: float = 1.0, high: float = 4.0, ctx: int = 8192) -> float:
    base = 1.0 / (theta ** (2 * i / head_dim))
    if not scaled:
        return base
    wavelength = 2 * math.pi / base
    if wavelength < ctx / high:
        return base
    if wavelength > ctx / low:
        return base / factor
    mu = (ctx / wavelength - low) / (high - low)
    return (1 - mu) * base / factor + mu * base


def linear(x, w):
    """F.linear without bias: out[o] = sum_i x[i] * w[o][i], w stored [out, in]."""
    return [sum(x[i] * row[i] for i in range(len(x))) for row in w]


def rotate(vec, pos, freqs):
    out = []
    for i in range(len(vec) // 2):
        z = complex(vec[2 * i], vec[2 * i + 1]) * cmath.exp(1j * pos * freqs[i])
        out += [z.real, z.imag]
    return out


def block(x, wq, wk, wv, wo, start_pos, cache_k, cache_v, n_heads, n_kv_heads,
          theta=500000.0, scaled=True):
    """x: list[B][T][d]; cache_k/v: list[B][S][n_kv][d_h] (new rows overwritten
    in copies); start_pos: list of ints per sequence. Returns (delta, ck, cv)."""
    B, T = len(x), len(x[0])
    head_dim = len(wq) // n_heads
    n_rep = n_heads // n_kv_heads
    freqs = [frequency(i, head_dim, theta, scaled) for i in range(head_dim // 2)]
    ck = [[[list(h) for h in row] for row in seq] for seq in cache_k]
    cv = [[[list(h) for h in row] for row in seq] for seq in cache_v]
    delta = []
    for b in range(B):
        sp = start_pos[b]
        qs = []
        for t in range(T):
            pos = sp + t
            q = linear(x[b][t], wq)
            k = linear(x[b][t], wk)
            v = linear(x[b][t], wv)
            qh = [rotate(q[h * head_dim:(h + 1) * head_dim], pos, freqs) for h in range(n_heads)]
            for g in range(n_kv_heads):
                kg = rotate(k[g * head_dim:(g + 1) * head_dim], pos, freqs)
                ck[b][pos][g] = [bf16(e) for e in kg]
                cv[b][pos][g] = [bf16(e) for e in v[g * head_dim:(g + 1) * head_dim]]
            qs.append(qh)
        rows = []
        L = sp + T
        for t in range(T):
            # expanded key/value heads: copy c of KV head g sits at index g*n_rep + c
            merged = []
            for h in range(n_heads):
                g = [gg for gg in range(n_kv_heads) for _ in range(n_rep)][h]
                scores = []
                for j in range(L):
                    s = sum(qs[t][h][d] * ck[b][j][g][d] for d in range(head_dim))
                    s = s / math.sqrt(head_dim)
                    if j > sp + t:
                        s = s + (-math.inf)
                    scores.append(s)
                mx = max(scores)
                ex = [math.exp(s - mx) for s in scores]
                tot = sum(ex)
                probs = [e / tot for e in ex]
                merged += [sum(probs[j] * cv[b][j][g][d] for j in range(L))
                           for d in range(head_dim)]
            rows.append(linear(merged, wo))
        delta.append(rows)
    return delta, ck, cv
