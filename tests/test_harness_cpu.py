"""CPU checks of the parity harness's own bounds."""
import numpy as np
import torch

from oracle import gqa as O
from tests import harness as H


def _rotate_pairs(v, ang):
    c, s = np.cos(ang), np.sin(ang)
    out = v.copy()
    out[..., 0::2] = v[..., 0::2] * c - v[..., 1::2] * s
    out[..., 1::2] = v[..., 0::2] * s + v[..., 1::2] * c
    return out


def test_norm_flip_allowance_bounds_every_rounding_flip():
    """Round the ambiguous normalised values the other way (the worst a GPU
    norm within NORM_REL_ERR could do), project and rotate: the row moves by
    no more than the allowance, element by element; values on bf16 points
    give no allowance."""
    rng = np.random.default_rng(3)
    d, rows = 256, 16
    xn = rng.standard_normal((4, d))
    u = H.bf16_ulp(xn)
    # push a few values onto rounding midpoints
    xn[:, ::37] = (np.floor(xn[:, ::37] / u[:, ::37]) + 0.5) * u[:, ::37]
    w = O.bf16_round(rng.standard_normal((rows, d)) / 16)
    allow = H.norm_flip_allowance(xn, w)
    a = O.bf16_round(xn)
    frac = xn / u - np.floor(xn / u)
    amb = np.abs(frac - 0.5) * u <= H.NORM_REL_ERR * np.abs(xn)
    assert amb[:, ::37].all() and amb.sum() >= 4 * len(range(0, d, 37))
    flipped = np.where(amb, np.where(a > xn, a - u, a + u), a)
    ang = rng.uniform(0, 2 * np.pi, (4, rows // 2))
    diff = np.abs(_rotate_pairs(flipped @ w.T, ang) - _rotate_pairs(a @ w.T, ang))
    assert np.all(diff <= allow * (1 + 1e-12) + 1e-15)
    assert np.all(H.norm_flip_allowance(O.bf16_round(xn), w) == 0)


def test_cache_row_bar_is_one_ulp_without_allowance():
    ref = np.array([[1.0, -0.5, 3.0, 0.25]])
    got = torch.tensor(O.bf16_round(ref + H.bf16_ulp(ref) * 0.99), dtype=torch.float64).to(torch.bfloat16)
    H.check_rows_within_one_ulp(got, ref, "within")
    bad = torch.tensor(ref + 2.5 * H.bf16_ulp(ref), dtype=torch.float64).to(torch.bfloat16)
    try:
        H.check_rows_within_one_ulp(bad, ref, "beyond")
    except AssertionError:
        pass
    else:
        raise AssertionError("a 2-ulp difference passed the 1-ulp bar")
