"""gqa_decode_static: the decode step for callers that cannot allocate device
memory while they run a step (an engine plugin whose enqueue must not call
cudaMalloc, a real-time serving loop where a synchronous allocation would
stall the device). Its scratch is a static array inside the library instead
of a caller workspace.

Calls in a row on different inputs, each checked against gqa_decode on the
same inputs with the parity tolerance of the other tests and against the CPU
oracle; a later call must not see anything an earlier one left in the shared
array. The last case is a batch of 64 ragged sequences, the largest batch the
header promises fits the array. Collected last on purpose, and valid both
alone and after the other tests."""
import numpy as np
import pytest
import torch

import gqa_inputs as I
from tests import harness as H

pytestmark = pytest.mark.gpu

G = pytest.importorskip("grouped_query_attention_gemv_gb300")


def _decode_both_ways(c):
    d = c.dev
    sp = torch.tensor(c.start, dtype=torch.int32, device="cuda")
    mx = max(c.start)
    rope = H.rope_for(c)
    ref = G.decode(d["x"], sp, mx, d["wq"], d["wk"], d["wv"], d["wo"], rope, d["cache_k"], d["cache_v"],
                   workspace=G.make_workspace(c.B, 1, mx + 1))
    torch.cuda.synchronize()
    ref_k, ref_v = d["cache_k"].clone(), d["cache_v"].clone()
    # the same call again through the static-scratch entry point, on the untouched cache
    d["cache_k"].copy_(d["cache_k0"])
    d["cache_v"].copy_(d["cache_v0"])
    got = G.decode_static(d["x"], sp, mx, d["wq"], d["wk"], d["wv"], d["wo"], rope, d["cache_k"], d["cache_v"])
    torch.cuda.synchronize()
    assert G.static_device_status() == 0
    return ref, got, ref_k, ref_v


def test_decode_static_matches_decode_and_the_oracle_on_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from grouped_query_attention_gemv_gb300 import build
    build.build()
    weights = I.draw_weights(seed=0)
    ragged64 = [int(p) for p in np.random.default_rng(64).integers(0, 2048, 64)]
    cases = [H.make_case(6, 1, [1000, 3, 517, 64, 0, 2047], 2048, weights=weights),
             H.make_case(3, 1, [40, 129, 7], 160, seed=0, weights=weights),
             H.make_case(64, 1, ragged64, 2048, seed=1, weights=weights)]
    for c in cases:
        ref, got, ref_k, ref_v = _decode_both_ways(c)
        a, b = H.f64(got), H.f64(ref)
        assert np.isfinite(a).all()
        assert H.rel_l2(a, b) <= H.REL_L2_TOL
        assert np.abs(a - b).max() <= H.MAX_ABS_TOL
        for bi, sp in enumerate(c.start):
            for name, ref_c in (("cache_k", ref_k), ("cache_v", ref_v)):
                H.check_rows_within_one_ulp(c.dev[name][bi, sp:sp + 1], H.f64(ref_c[bi, sp:sp + 1]),
                                            f"{name} row of sequence {bi}")
        # and against the oracle on the same seeded inputs (delta and the written rows)
        for bi in range(0, c.B, max(1, c.B // 8)):
            H.compare_sequence(c, got, bi)
        H.check_canaries(c)
