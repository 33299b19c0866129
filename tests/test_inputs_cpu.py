"""The seeded input generators draw what the design states: weights
N(0, 1/4096) in bf16 stored [out, in], x and cached K/V rows N(0, 1) in bf16,
rows past each sequence's position zero, the norm weight near 1, the same
tensors for the same seed."""
import torch

import gqa_inputs as I


def test_weights_and_x():
    gen, w = I.draw_weights(seed=0)
    assert w["wq"].shape == (4096, 4096) and w["wk"].shape == (1024, 4096) and w["wo"].shape == (4096, 4096)
    assert all(t.dtype == torch.bfloat16 for t in w.values())
    sd = w["wq"].float().std().item()
    assert abs(sd - 1 / 64) < 1e-3
    x = I.draw_x(gen, 2, 3)
    assert x.shape == (2, 3, 4096) and abs(x.float().std().item() - 1.0) < 0.05
    gen2, w2 = I.draw_weights(seed=0)
    assert torch.equal(w["wv"], w2["wv"]) and torch.equal(x, I.draw_x(gen2, 2, 3))
    _, wm = I.draw_weights(I.LLAMA31_8B_MHA, seed=0)
    assert wm["wk"].shape == (4096, 4096)


def test_cache_rows():
    ck, cv = I.draw_cache(3, 40, [0, 7, 40], seed=0, device="cpu")
    assert ck.shape == (3, 40, 8, 128) and ck.dtype == torch.bfloat16
    assert not ck[0].any() and not cv[0].any()            # nothing cached
    assert ck[1, :7].abs().sum() > 0 and not ck[1, 7:].any()
    assert abs(ck[2].float().std().item() - 1.0) < 0.05


def test_norm_weight():
    g = I.draw_norm_weight(seed=0)
    assert g.shape == (4096,) and g.dtype == torch.bfloat16
    assert abs(g.float().mean().item() - 1.0) < 0.01 and abs(g.float().std().item() - 0.1) < 0.01
