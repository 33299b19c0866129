"""Plant plausible mistakes in a copy of the oracle (CPU only) and check that
the pins catch every one of them. The oracle's source text is edited in
memory and loaded as a throw-away module; the real module is untouched."""
import importlib.util
import os
import types

import numpy as np
import pytest

from oracle import brute

SRC_PATH = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "gqa.py")
SRC = open(SRC_PATH).read()

MUTANTS = {
    "gqa_map_modulo": ("heads = slice(g * n_rep, (g + 1) * n_rep)", "heads = slice(g, n_heads, n_kv_heads)"),
    "rope_sign": ("out[..., 1::2] = a * sin + b * cos", "out[..., 1::2] = a * sin - b * cos"),
    "rope_half_split_pairs": ("a = v[..., 0::2]\n    b = v[..., 1::2]",
                              "a = np.concatenate([v[..., :v.shape[-1] // 2]] * 1, -1)[..., :v.shape[-1] // 2]\n"
                              "    b = v[..., v.shape[-1] // 2:]"),
    "mask_sees_one_future_key": ("<= (start_pos + rows)[:, None]", "<= (start_pos + rows + 1)[:, None]"),
    "score_scale_dropped": ("scale = 1.0 / math.sqrt(head_dim)", "scale = 1.0"),
    "weight_not_transposed": ("q = (x[rows] @ wq.T)", "q = (x[rows] @ wq)"),
    "value_not_rounded": ("new_v = bf16_round(v)", "new_v = v"),
    "frequency_exponent": ("f = theta ** (-2.0 * i / head_dim)", "f = theta ** (-1.0 * i / head_dim)"),
    "band_swapped": ("np.where(wavelength < short_edge, f, np.where(wavelength > long_edge, f / factor, mid))",
                     "np.where(wavelength < short_edge, f / factor, np.where(wavelength > long_edge, f, mid))"),
    "rope_on_values": ("v = (x @ wv.T).reshape(T, n_kv_heads, head_dim)",
                       "v = rope_rotate((x @ wv.T).reshape(T, n_kv_heads, head_dim), cos[:, None, :], sin[:, None, :])"),
    "softmax_wrong_axis": ("return e / np.sum(e, axis=axis, keepdims=True)",
                                            "return e / np.sum(e, axis=0, keepdims=True)"),
    "rms_mean_over_rows": ("ms = np.mean(x * x, axis=-1, keepdims=True)", "ms = np.mean(x * x, axis=0, keepdims=True)"),
    "rms_no_sqrt": ("return x / np.sqrt(ms + eps) * weight", "return x / (ms + eps) * weight"),
    "rms_eps_outside_sqrt": ("return x / np.sqrt(ms + eps) * weight", "return x / (np.sqrt(ms) + eps) * weight"),
    "rms_weight_dropped": ("return x / np.sqrt(ms + eps) * weight", "return x / np.sqrt(ms + eps)"),
    "residual_on_normalised_input": ("    return x + delta, ck, cv", "    return rms_norm(x, norm_weight, eps) + delta, ck, cv"),
    # positions counted from the chunk, not the sequence (a chunked-prefill slip)
    "rope_position_from_chunk": ("    pos = start_pos + np.arange(T)", "    pos = np.arange(T)"),
    "keys_not_rotated": ("    k = rope_rotate(k, cos[:, None, :], sin[:, None, :])\n", ""),
    # heads merged as d * n_heads + h instead of h * d_h + d
    "head_merge_transposed": ("delta = o.reshape(len(rows), n_heads * head_dim) @ wo.T",
                              "delta = o.transpose(0, 2, 1).reshape(len(rows), n_heads * head_dim) @ wo.T"),
    "new_rows_written_at_zero": ("        ck[b, sp[b]:sp[b] + T] = nk", "        ck[b, :T] = nk"),
    # scaled-RoPE band blends that still meet both edges
    "band_geometric_blend": ("mid = (1.0 - mu) * f / factor + mu * f", "mid = f / factor * factor ** mu"),
    "band_linear_in_wavelength": (
        "mu = (original_context / wavelength - low_freq_factor) / (high_freq_factor - low_freq_factor)",
        "mu = (long_edge - wavelength) / (long_edge - short_edge)"),
}

BAND_MUTANTS = ("band_geometric_blend", "band_linear_in_wavelength")


def load(src):
    mod = types.ModuleType("oracle_mutant")
    exec(compile(src, "oracle_mutant", "exec"), mod.__dict__)
    return mod


def rnd(M, rng, *shape, scale=1.0):
    return M.bf16_round(rng.standard_normal(shape) * scale)


def case(M, rng, d, H, Hkv, hd, B, T, S, start):
    w = {k: rnd(M, rng, *s, scale=d ** -0.5) for k, s in
         (("wq", (H * hd, d)), ("wk", (Hkv * hd, d)), ("wv", (Hkv * hd, d)), ("wo", (d, H * hd)))}
    x = rnd(M, rng, B, T, d)
    ck, cv = np.zeros((B, S, Hkv, hd)), np.zeros((B, S, Hkv, hd))
    for b in range(B):
        ck[b, :start[b]] = rnd(M, rng, start[b], Hkv, hd)
        cv[b, :start[b]] = rnd(M, rng, start[b], Hkv, hd)
    return w, x, ck, cv


def pin_brute(M):
    for shape in (dict(d=16, H=4, Hkv=2, hd=4, B=2, T=3, S=12, start=(2, 5)),
                  dict(d=256, H=2, Hkv=1, hd=128, B=1, T=2, S=8, start=(5,))):
        rng = np.random.default_rng(0)
        w, x, ck, cv = case(M, rng, **shape)
        H, Hkv, hd = shape["H"], shape["Hkv"], shape["hd"]
        d, k2, v2 = M.block_forward(x, w, list(shape["start"]), ck, cv,
                                    M.rope_frequencies(hd, 500000.0, True), H, Hkv)
        bd, bk, bv = brute.block(x.tolist(), w["wq"].tolist(), w["wk"].tolist(), w["wv"].tolist(),
                                 w["wo"].tolist(), list(shape["start"]), ck.tolist(), cv.tolist(), H, Hkv)
        np.testing.assert_allclose(d, np.array(bd), rtol=1e-11, atol=1e-12)
        np.testing.assert_array_equal(k2, np.array(bk))
        np.testing.assert_array_equal(v2, np.array(bv))


def pin_scaled_frequencies(M):
    f = M.rope_frequencies(128, 500000.0, True)
    np.testing.assert_allclose(f, [brute.frequency(i, 128, 500000.0, True) for i in range(64)], rtol=1e-14)


def pin_band_affine(M):
    """Structural pin of the band (no restated formula): f'/f affine in f."""
    from tests.test_oracle_pins import band_ratio_affine_residual
    assert band_ratio_affine_residual(M.rope_frequencies(128, 500000.0, True),
                                      M.rope_frequencies(128, 500000.0, False)) < 1e-12


def pin_gqa_vs_mha(M):
    rng = np.random.default_rng(8)
    H, Hkv, hd = 4, 2, 4
    w, x, ck, cv = case(M, rng, 16, H, Hkv, hd, 2, 3, 12, (2, 5))
    wm = dict(w)
    wm["wk"] = np.repeat(w["wk"].reshape(Hkv, hd, -1), 2, axis=0).reshape(H * hd, -1)
    wm["wv"] = np.repeat(w["wv"].reshape(Hkv, hd, -1), 2, axis=0).reshape(H * hd, -1)
    fr = M.rope_frequencies(hd, 500000.0, True)
    d1, _, _ = M.block_forward(x, w, [2, 5], ck, cv, fr, H, Hkv)
    d2, _, _ = M.block_forward(x, wm, [2, 5], np.repeat(ck, 2, axis=2), np.repeat(cv, 2, axis=2), fr, H, H)
    np.testing.assert_allclose(d1, d2, rtol=1e-12, atol=1e-14)


def pin_rms_norm(M):
    x = np.array([[2.5] * 8, [-0.125] * 8])
    np.testing.assert_allclose(M.rms_norm(x, np.ones(8), 0.0), [[1.0] * 8, [-1.0] * 8], rtol=1e-15)
    np.testing.assert_allclose(M.rms_norm(np.array([3.0, 4.0]), np.array([2.0, -0.5]), 3.5), [1.5, -0.5], rtol=1e-15)
    rng = np.random.default_rng(5)
    y = M.rms_norm(rng.standard_normal((3, 64)) * np.array([[0.01], [1.0], [300.0]]), np.ones(64), 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, rtol=1e-13)


def pin_layer_residual(M):
    rng = np.random.default_rng(6)
    d, H, Hkv, hd = 16, 4, 2, 4
    w, x, ck, cv = case(M, rng, d, H, Hkv, hd, 1, 3, 8, (0,))
    w["wo"] = np.zeros_like(w["wo"])
    g = M.bf16_round(1.0 + 0.1 * rng.standard_normal(d))
    h, _, _ = M.layer_forward(x, g, 1e-5, w, 0, ck, cv, M.rope_frequencies(hd, 500000.0, True), H, Hkv)
    np.testing.assert_array_equal(h, x)


PINS = (pin_brute, pin_scaled_frequencies, pin_band_affine, pin_gqa_vs_mha, pin_rms_norm, pin_layer_residual)


def test_unmutated_oracle_passes_every_pin():
    M = load(SRC)
    for pin in PINS:
        pin(M)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name):
    old, new = MUTANTS[name]
    assert SRC.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    M = load(SRC.replace(old, new))
    failures = 0
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin(M)
        except (AssertionError, ValueError, IndexError):
            failures += 1
    assert failures > 0, f"no pin caught the planted mistake {name}"


@pytest.mark.parametrize("name", BAND_MUTANTS)
def test_band_blend_mistake_is_caught_by_the_structural_pin(name):
    """The affine-ratio pin alone catches a wrong band blend: it does not lean
    on the scalar restatement of the same formula."""
    old, new = MUTANTS[name]
    M = load(SRC.replace(old, new))
    with pytest.raises(AssertionError):
        pin_band_affine(M)
