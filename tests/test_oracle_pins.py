"""Pins for the CPU oracle: what the pages and the mathematics fix, checked
against ``oracle.gqa`` without trusting it. CPU only.

Each check is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign, a wrong GQA index, an off-by-one mask, a transposed weight)
fails at least one of them; ``test_oracle_mutations.py`` plants such slips and
confirms it.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import brute
from oracle import gqa as O

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_figures.json")))


def rand(rng, *shape, scale=1.0):
    """bf16-exact float64 test values."""
    return O.bf16_round(rng.standard_normal(shape) * scale)


def tiny_case(rng, d=16, H=4, Hkv=2, hd=4, B=2, T=3, S=12, start=(2, 5)):
    w = {"wq": rand(rng, H * hd, d, scale=d ** -0.5), "wk": rand(rng, Hkv * hd, d, scale=d ** -0.5),
         "wv": rand(rng, Hkv * hd, d, scale=d ** -0.5), "wo": rand(rng, d, H * hd, scale=d ** -0.5)}
    x = rand(rng, B, T, d)
    ck = np.zeros((B, S, Hkv, hd))
    cv = np.zeros((B, S, Hkv, hd))
    for b in range(B):
        ck[b, :start[b]] = rand(rng, start[b], Hkv, hd)
        cv[b, :start[b]] = rand(rng, start[b], Hkv, hd)
    return w, x, ck, cv


# --------------------------------------------------------------- page figures

def test_block_parameter_counts_match_page_table():
    g = GOLDEN["block_params"]
    c = O.param_counts(4096, 32, 8, 128)
    assert (c["wq"], c["wk"], c["wv"], c["wo"], c["total"]) == (g["wq"], g["wk"], g["wv"], g["wo"], g["total"])
    assert 32 * c["total"] == g["total_32_blocks"]
    q = GOLDEN["query_projection_params"]
    assert c["wq"] == q["per_instance"] and 32 * c["wq"] == q["total_32_blocks"]


def test_kv_cache_figures_match_in_numbers_section():
    g = GOLDEN["kv_cache"]
    per_tok = O.kv_cache_bytes_per_token(32, 8, 128)
    assert per_tok == g["per_token_all_layers_kib"] * 1024
    assert O.kv_cache_bytes_per_token(32, 32, 128) == g["per_token_all_layers_mha_kib"] * 1024
    assert round(per_tok * g["positions_after_decode_call"] / 2 ** 20, 1) == g["in_use_after_call_mib_1dp"]
    assert per_tok * g["full_context_tokens"] == g["full_context_gib"] * 2 ** 30
    assert O.kv_cache_bytes_per_token(32, 32, 128) * g["full_context_tokens"] == g["full_context_mha_gib"] * 2 ** 30


def test_decode_header_counts():
    # decode at P cached positions reads L = P + 1 keys and writes row P
    g = GOLDEN["decode_header"]
    rng = np.random.default_rng(0)
    P = 7
    w, x, ck, cv = tiny_case(rng, B=1, T=1, S=P + 1, start=(P,))
    _, nk, _ = O.sequence_forward(x[0], w["wq"], w["wk"], w["wv"], w["wo"], P, ck[0, :P], cv[0, :P],
                                  O.rope_frequencies(4, 500000.0, True), 4, 2)
    assert nk.shape[0] == 1
    assert g["keys_read"] == g["cached_positions"] + 1 and g["row_written"] == g["cached_positions"]
    assert g["rope_pairs"] == 128 // 2


# --------------------------------------------------------------- bf16 rounding

def test_bf16_round_matches_torch_on_fp32_values():
    # for fp32-representable inputs, fp64->bf16 equals torch's fp32->bf16 (RNE)
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000),
                        rng.standard_normal(1000) * 1e-39]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).float().numpy().astype(np.float64)
    np.testing.assert_array_equal(O.bf16_round(v.astype(np.float64)), ref)


def test_bf16_round_ties_and_limits():
    one = 1.0
    ulp = 2.0 ** -7
    assert O.bf16_round(one + ulp / 2) == one                 # tie -> even (1.0)
    assert O.bf16_round(one + 3 * ulp / 2) == one + 2 * ulp   # tie -> even (1+2ulp)
    assert O.bf16_round(one + ulp / 2 + 1e-12) == one + ulp
    assert O.bf16_round(-(one + ulp / 2)) == -one
    assert O.bf16_round(2.0 ** -133 * 0.75) == 2.0 ** -133    # subnormal spacing
    assert np.isinf(O.bf16_round(3.4e38 * 1.01))
    assert O.bf16_round(0.0) == 0.0


def test_bf16_round_matches_brute_on_fp64_values():
    rng = np.random.default_rng(2)
    v = rng.standard_normal(3000) * 10.0 ** rng.integers(-5, 5, 3000)
    np.testing.assert_array_equal(O.bf16_round(v), np.array([brute.bf16(float(e)) for e in v]))


# --------------------------------------------------------------- RoPE

FREQS = O.rope_frequencies(128, 500000.0, True)


def test_rope_preserves_norm_per_pair():
    rng = np.random.default_rng(3)
    v = rng.standard_normal((50, 128))
    c, s = O.rope_cos_sin(rng.integers(0, 131072, 50), FREQS)
    r = O.rope_rotate(v, c, s)
    n0 = v[:, 0::2] ** 2 + v[:, 1::2] ** 2
    n1 = r[:, 0::2] ** 2 + r[:, 1::2] ** 2
    np.testing.assert_allclose(n1, n0, rtol=1e-12, atol=1e-12)


def test_rope_dot_product_depends_only_on_relative_position():
    rng = np.random.default_rng(4)
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    def dot(m, n):
        cm, sm = O.rope_cos_sin([m], FREQS)
        cn, sn = O.rope_cos_sin([n], FREQS)
        return O.rope_rotate(q[None], cm, sm)[0] @ O.rope_rotate(k[None], cn, sn)[0]
    for m, n, shift in [(5, 2, 100), (1000, 999, 12345), (17, 40, 7)]:
        assert abs(dot(m, n) - dot(m + shift, n + shift)) < 1e-9
    assert abs(dot(5, 2) - dot(6, 2)) > 1e-6        # but it does depend on m - n


def test_rope_position_zero_is_identity():
    v = np.random.default_rng(5).standard_normal((3, 128))
    c, s = O.rope_cos_sin([0], FREQS)
    np.testing.assert_array_equal(O.rope_rotate(v, c, s), v)


def test_rope_pairs_are_adjacent_complex_numbers():
    # against Python complex multiplication (the view_as_complex reading)
    rng = np.random.default_rng(6)
    v = rng.standard_normal(128)
    for pos in (1, 77, 131071):
        c, s = O.rope_cos_sin([pos], FREQS)
        np.testing.assert_allclose(O.rope_rotate(v[None], c, s)[0],
                                   brute.rotate(list(v), pos, list(FREQS)), rtol=0, atol=1e-12)


def test_unscaled_frequencies_are_the_base_geometric_series():
    f = O.rope_frequencies(128, 500000.0, False)
    assert f[0] == 1.0
    np.testing.assert_allclose(f[1:] / f[:-1], 500000.0 ** (-2 / 128), rtol=1e-13)
    assert math.isclose(f[-1], 500000.0 ** (-126 / 128), rel_tol=1e-13)


def test_scaled_frequency_bands():
    base = O.rope_frequencies(128, 500000.0, False)
    f = O.rope_frequencies(128, 500000.0, True)
    wl = 2 * math.pi / base
    hi = wl < 8192 / 4
    lo = wl > 8192 / 1
    np.testing.assert_array_equal(f[hi], base[hi])            # short wavelengths untouched
    np.testing.assert_allclose(f[lo], base[lo] / 8, rtol=1e-15)  # long ones divided by the factor
    mid = ~hi & ~lo
    assert (hi.sum(), mid.sum(), lo.sum()) == (29, 6, 29)
    assert np.all(f[mid] < base[mid]) and np.all(f[mid] > base[mid] / 8)
    assert np.all(np.diff(f) < 0)                             # still strictly decreasing
    # factor 1 removes the rescaling everywhere (the band formula collapses to f)
    np.testing.assert_allclose(O.rope_frequencies(128, 500000.0, True, factor=1.0), base, rtol=1e-15)
    # matches the independent scalar restatement
    np.testing.assert_allclose(f, [brute.frequency(i, 128, 500000.0, True) for i in range(64)], rtol=1e-14)


def band_ratio_affine_residual(fr_scaled, fr_base, low=1.0, high=4.0, ctx=8192):
    """Largest distance of the band's points (f, f'/f) from their least-squares
    line, relative to the spread of f'/f. The reading interpolates linearly in
    mu, and mu is affine in 1/wavelength, i.e. in f: the points are collinear.
    A geometric blend (f/8 * 8^mu) or a blend linear in the wavelength puts
    them on a curve."""
    wl = 2 * math.pi / fr_base
    band = (wl >= ctx / high) & (wl <= ctx / low)
    f, r = fr_base[band], fr_scaled[band] / fr_base[band]
    assert band.sum() >= 3
    A = np.stack([f, np.ones_like(f)], axis=1)
    coef, *_ = np.linalg.lstsq(A, r, rcond=None)
    return float(np.abs(A @ coef - r).max() / (r.max() - r.min()))


def test_scaled_band_ratio_is_affine_in_frequency():
    base = O.rope_frequencies(128, 500000.0, False)
    assert band_ratio_affine_residual(O.rope_frequencies(128, 500000.0, True), base) < 1e-12
    # the pin separates the reading from the two other smooth blends that meet
    # both edges: geometric in mu, and linear in the wavelength
    wl = 2 * math.pi / base
    mu = (8192 / wl - 1) / 3
    geo = np.where(wl < 2048, base, np.where(wl > 8192, base / 8, base / 8 * 8.0 ** mu))
    lam = (8192 - wl) / (8192 - 2048)
    in_wl = np.where(wl < 2048, base, np.where(wl > 8192, base / 8, (1 - lam) * base / 8 + lam * base))
    assert band_ratio_affine_residual(geo, base) > 1e-3
    assert band_ratio_affine_residual(in_wl, base) > 1e-3


def test_scaled_band_formula_is_continuous_at_both_edges():
    # choose theta so that pair 1's wavelength sits exactly on each edge
    for edge, expect_div in ((8192 / 4, 1.0), (8192 / 1, 8.0)):
        # wavelength of pair 1 = 2*pi*theta^(2/hd); hd = 4 -> theta^(1/2)
        theta = (edge / (2 * math.pi)) ** 2
        f = O.rope_frequencies(4, theta, True)
        base = O.rope_frequencies(4, theta, False)
        assert math.isclose(f[1], base[1] / expect_div, rel_tol=1e-12)
        for eps in (1e-9, -1e-9):
            f2 = O.rope_frequencies(4, theta * (1 + eps), True)
            b2 = O.rope_frequencies(4, theta * (1 + eps), False)
            assert math.isclose(f2[1] / b2[1], 1 / expect_div, rel_tol=1e-6)


# --------------------------------------------------------------- softmax

def test_softmax_rows_sum_to_one_and_shift_invariant():
    rng = np.random.default_rng(7)
    s = rng.standard_normal((10, 1001)) * 30
    p = O.softmax(s)
    np.testing.assert_allclose(p.sum(-1), 1.0, atol=1e-12)
    np.testing.assert_allclose(O.softmax(s + 123.0), p, rtol=1e-12, atol=1e-300)
    s[:, 500:] = -np.inf
    p = O.softmax(s)
    assert np.all(p[:, 500:] == 0) and np.allclose(p.sum(-1), 1.0, atol=1e-12)


# --------------------------------------------------------------- block-level pins

def run(w, x, start, ck, cv, H, Hkv, scaled=True):
    hd = w["wq"].shape[0] // H
    return O.block_forward(x, w, start, ck, cv, O.rope_frequencies(hd, 500000.0, scaled), H, Hkv)


@pytest.mark.parametrize("shape", [
    dict(d=16, H=4, Hkv=2, hd=4, B=2, T=3, S=12, start=(2, 5)),
    dict(d=16, H=4, Hkv=2, hd=4, B=2, T=1, S=8, start=(0, 6)),
    dict(d=24, H=6, Hkv=3, hd=4, B=1, T=4, S=6, start=(0,)),
    dict(d=16, H=4, Hkv=4, hd=4, B=1, T=2, S=5, start=(3,)),   # MHA (n_rep = 1)
    dict(d=16, H=4, Hkv=1, hd=4, B=1, T=2, S=5, start=(2,)),   # MQA (n_rep = 4)
    dict(d=256, H=2, Hkv=1, hd=128, B=1, T=2, S=8, start=(5,)),  # real head width
])
def test_numpy_oracle_matches_brute_force(shape):
    rng = np.random.default_rng(hash(tuple(sorted(shape.items()))) % 2 ** 32)
    w, x, ck, cv = tiny_case(rng, **shape)
    H, Hkv = shape["H"], shape["Hkv"]
    d, k2, v2 = run(w, x, list(shape["start"]), ck, cv, H, Hkv)
    bd, bk, bv = brute.block(x.tolist(), w["wq"].tolist(), w["wk"].tolist(), w["wv"].tolist(),
                             w["wo"].tolist(), list(shape["start"]), ck.tolist(), cv.tolist(), H, Hkv)
    np.testing.assert_allclose(d, np.array(bd), rtol=1e-11, atol=1e-12)
    np.testing.assert_array_equal(k2, np.array(bk))
    np.testing.assert_array_equal(v2, np.array(bv))


def test_gqa_equals_mha_on_duplicated_kv_heads():
    # KV head g serves query heads g*n_rep .. g*n_rep+n_rep-1 (repeat_kv expands
    # each KV head into n_rep consecutive copies)
    rng = np.random.default_rng(8)
    H, Hkv, hd = 4, 2, 4
    w, x, ck, cv = tiny_case(rng, H=H, Hkv=Hkv, hd=hd, B=2, T=3, S=12, start=(2, 5))
    rep = H // Hkv
    w_mha = dict(w)
    w_mha["wk"] = np.repeat(w["wk"].reshape(Hkv, hd, -1), rep, axis=0).reshape(H * hd, -1)
    w_mha["wv"] = np.repeat(w["wv"].reshape(Hkv, hd, -1), rep, axis=0).reshape(H * hd, -1)
    ck_m, cv_m = np.repeat(ck, rep, axis=2), np.repeat(cv, rep, axis=2)
    d1, k1, _ = run(w, x, [2, 5], ck, cv, H, Hkv)
    d2, k2, _ = run(w_mha, x, [2, 5], ck_m, cv_m, H, H)
    np.testing.assert_allclose(d1, d2, rtol=1e-12, atol=1e-14)
    np.testing.assert_array_equal(np.repeat(k1, rep, axis=2), k2)


def test_cached_decode_equals_one_longer_prefill():
    rng = np.random.default_rng(9)
    w, x, ck, cv = tiny_case(rng, B=1, T=5, S=8, start=(0,))
    full, fk, fv = run(w, x, [0], ck, cv, 4, 2)
    pre, pk, pv = run(w, x[:, :4], [0], ck, cv, 4, 2)
    dec, dk, dv = run(w, x[:, 4:5], [4], pk, pv, 4, 2)
    np.testing.assert_allclose(dec[0, 0], full[0, 4], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(pre[0], full[0, :4], rtol=1e-12, atol=1e-14)
    np.testing.assert_array_equal(dk, fk)
    np.testing.assert_array_equal(dv, fv)


def test_chunked_prefill_equals_one_shot_prefill():
    rng = np.random.default_rng(10)
    w, x, ck, cv = tiny_case(rng, B=1, T=7, S=9, start=(0,))
    full, fk, fv = run(w, x, [0], ck, cv, 4, 2)
    a, ak, av = run(w, x[:, :3], [0], ck, cv, 4, 2)
    b, bk, bv = run(w, x[:, 3:], [3], ak, av, 4, 2)
    np.testing.assert_allclose(np.concatenate([a, b], axis=1), full, rtol=1e-12, atol=1e-14)
    np.testing.assert_array_equal(bk, fk)


def test_single_key_closed_form():
    # start_pos 0, T 1: every head attends only to its own new value row
    rng = np.random.default_rng(11)
    w, x, ck, cv = tiny_case(rng, B=1, T=1, S=1, start=(0,))
    d, k, v = run(w, x, [0], ck, cv, 4, 2)
    o = np.repeat(v[0, 0], 2, axis=0).reshape(-1)   # KV head h // 2 for h = 0..3
    np.testing.assert_allclose(d[0, 0], w["wo"] @ o, rtol=1e-13, atol=1e-15)
    np.testing.assert_array_equal(v[0, 0].reshape(-1), O.bf16_round(w["wv"] @ x[0, 0]))


def test_zero_query_weights_give_uniform_attention():
    rng = np.random.default_rng(12)
    w, x, ck, cv = tiny_case(rng, B=1, T=1, S=9, start=(8,))
    w["wq"] = np.zeros_like(w["wq"])
    d, k, v = run(w, x, [8], ck, cv, 4, 2)
    mean_v = v[0, :9].mean(axis=0)                       # [Hkv, hd]
    o = np.repeat(mean_v, 2, axis=0).reshape(-1)
    np.testing.assert_allclose(d[0, 0], w["wo"] @ o, rtol=1e-12, atol=1e-14)


def test_causal_mask_future_tokens_do_not_leak():
    rng = np.random.default_rng(13)
    w, x, ck, cv = tiny_case(rng, B=1, T=6, S=9, start=(3,))
    d1, _, _ = run(w, x, [3], ck, cv, 4, 2)
    x2 = x.copy()
    x2[0, 4:] += 1.0
    d2, _, _ = run(w, x2, [3], ck, cv, 4, 2)
    np.testing.assert_array_equal(d1[0, :4], d2[0, :4])
    assert np.abs(d1[0, 4:] - d2[0, 4:]).max() > 1e-6


def test_only_new_rows_of_the_cache_change():
    rng = np.random.default_rng(14)
    w, x, ck, cv = tiny_case(rng, B=2, T=3, S=12, start=(2, 5))
    ck[:, 9:] = 7.0     # canary rows beyond start_pos + T
    _, k2, v2 = run(w, x, [2, 5], ck, cv, 4, 2)
    for b, s in enumerate((2, 5)):
        keep = np.ones(12, bool)
        keep[s:s + 3] = False
        np.testing.assert_array_equal(k2[b, keep], ck[b, keep])
        np.testing.assert_array_equal(v2[b, keep], cv[b, keep])
        assert not np.array_equal(k2[b, s:s + 3], ck[b, s:s + 3])


def test_weight_orientation_is_out_by_in():
    # F.linear reads weights [out, in]: a non-square Wk must be (Hkv*hd, d)
    rng = np.random.default_rng(15)
    w, x, ck, cv = tiny_case(rng, d=16, H=4, Hkv=2, hd=4, B=1, T=1, S=1, start=(0,))
    assert w["wk"].shape == (8, 16)
    _, k, _ = run(w, x, [0], ck, cv, 4, 2)
    np.testing.assert_array_equal(k[0, 0].reshape(-1), O.bf16_round(w["wk"] @ x[0, 0]))


# ------------------------------------------------------------------ attention_norm and the residual

def test_rms_norm_closed_forms():
    """A constant row normalises to +-1; a [3, 4] row with eps = 3.5 has
    mean square 12.5 + 3.5 = 16, so it maps to [0.75, 1.0]; the weight
    multiplies the normalised row feature by feature."""
    x = np.array([[2.5] * 8, [-0.125] * 8])
    np.testing.assert_allclose(O.rms_norm(x, np.ones(8), 0.0), [[1.0] * 8, [-1.0] * 8], rtol=1e-15)
    np.testing.assert_allclose(O.rms_norm(np.array([3.0, 4.0]), np.ones(2), 3.5), [0.75, 1.0], rtol=1e-15)
    g = np.array([2.0, -0.5])
    np.testing.assert_allclose(O.rms_norm(np.array([3.0, 4.0]), g, 3.5), [1.5, -0.5], rtol=1e-15)


def test_rms_norm_rows_have_unit_rms_and_ignore_scale():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((3, 64)) * np.array([[0.01], [1.0], [300.0]])
    y = O.rms_norm(x, np.ones(64), 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, rtol=1e-13)
    np.testing.assert_allclose(O.rms_norm(7.0 * x, np.ones(64), 0.0), y, rtol=1e-13)


def test_layer_residual_is_the_input_when_the_output_projection_is_zero():
    rng = np.random.default_rng(6)
    d, H, Hkv, hd, T = 16, 4, 2, 4, 3
    w = {k: O.bf16_round(rng.standard_normal(s) * d ** -0.5) for k, s in
         (("wq", (H * hd, d)), ("wk", (Hkv * hd, d)), ("wv", (Hkv * hd, d)), ("wo", (d, H * hd)))}
    x = O.bf16_round(rng.standard_normal((1, T, d)))
    ck, cv = np.zeros((1, 8, Hkv, hd)), np.zeros((1, 8, Hkv, hd))
    g = O.bf16_round(1.0 + 0.1 * rng.standard_normal(d))
    fr = O.rope_frequencies(hd, 500000.0, True)
    w0 = dict(w, wo=np.zeros_like(w["wo"]))
    h, _, _ = O.layer_forward(x, g, 1e-5, w0, 0, ck, cv, fr, H, Hkv)
    np.testing.assert_array_equal(h, x)
    # with the projection back, h - x is the block on the normalised input (stored in bf16)
    h, k2, _ = O.layer_forward(x, g, 1e-5, w, 0, ck, cv, fr, H, Hkv)
    d2, k3, _ = O.block_forward(O.bf16_round(O.rms_norm(x, g, 1e-5)), w, 0, ck, cv, fr, H, Hkv)
    np.testing.assert_allclose(h - x, d2, rtol=1e-12, atol=1e-15)
    np.testing.assert_array_equal(k2, k3)

