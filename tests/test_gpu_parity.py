"""GPU parity: the CUDA library (through the C ABI) against the CPU oracle on
the same seeded inputs. Bar: delta_attn within rel-L2 1e-2 and max-abs 3e-2
(bf16 I/O, fp32 accumulation), written cache rows within 1 bf16 ulp, every
other cache row bit-identical, workspace status word clear."""
import math

import numpy as np
import pytest
import torch

import gqa_inputs as I
from oracle import gqa as O
from tests import harness as H

pytestmark = pytest.mark.gpu

G = pytest.importorskip("grouped_query_attention_gemv_gb300")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from grouped_query_attention_gemv_gb300 import build
    build.build()


@pytest.fixture(scope="module")
def weights():
    return I.draw_weights(seed=0)


class attention_split:
    """Run the block's fused decode grid with the given attention split
    ("position", "head" or "auto") inside the with-block."""

    def __init__(self, mode):
        self.mode = mode

    def __enter__(self):
        self.prev = G.set_decode_attention_split(self.mode)

    def __exit__(self, *exc):
        G.set_decode_attention_split(self.prev)


SPLITS = ["position", "head"]


def run_decode(c, max_start=None, ws=None, rope=None):
    d = c.dev
    sp = torch.tensor(c.start, dtype=torch.int32, device="cuda")
    max_start = max(c.start) if max_start is None else max_start
    ws = G.make_workspace(c.B, 1, max_start + 1) if ws is None else ws
    rope = H.rope_for(c) if rope is None else rope
    out = G.decode(d["x"], sp, max_start, d["wq"], d["wk"], d["wv"], d["wo"], rope, d["cache_k"], d["cache_v"],
                   workspace=ws)
    torch.cuda.synchronize()
    assert G.device_status(ws) == 0
    return out, ws


def run_prefill(c, ws=None, entry="prefill"):
    d = c.dev
    assert len(set(c.start)) == 1
    sp = c.start[0]
    ws = G.make_workspace(c.B, c.T, sp + c.T) if ws is None else ws
    fn = G.prefill if entry == "prefill" else G.block_forward
    out = fn(d["x"], sp, d["wq"], d["wk"], d["wv"], d["wo"], H.rope_for(c), d["cache_k"], d["cache_v"], workspace=ws)
    torch.cuda.synchronize()
    assert G.device_status(ws) == 0
    return out, ws


# ------------------------------------------------------------------ RoPE table

@pytest.mark.parametrize("scaled", [True, False])
def test_rope_table_matches_oracle(scaled):
    rows = 131072
    t = G.rope_table(rows, scaled=scaled).cpu().double().numpy()
    f = O.rope_frequencies(128, 500000.0, scaled)
    for lo in (0, 4097, rows - 2048):
        c, s = O.rope_cos_sin(np.arange(lo, lo + 2048), f)
        np.testing.assert_allclose(t[lo:lo + 2048, :, 0], c, rtol=0, atol=2e-7)
        np.testing.assert_allclose(t[lo:lo + 2048, :, 1], s, rtol=0, atol=2e-7)


# ------------------------------------------------------------------ decode

@pytest.mark.parametrize("B,starts,s_max", [
    (1, [0], 4),                          # one key: o_h = v_{h//4}
    (3, [0, 5, 130], 160),                # ragged tails, several splits
    (2, [63, 64], 80),                    # tile edges
    (16, list(range(0, 1600, 100)), 1600),
    (40, None, 700),                      # M = 40 token projection (n-tile padding)
    (64, None, 520),                      # largest few-token projection
    (80, None, 300),                      # tensor-core projection (M > 64)
])
@pytest.mark.parametrize("split", SPLITS)
def test_decode_small_matches_oracle(weights, B, starts, s_max, split):
    if starts is None:
        g = torch.Generator().manual_seed(B)
        starts = torch.randint(0, s_max, (B,), generator=g).tolist()
    c = H.make_case(B, 1, starts, s_max, weights=weights)
    with attention_split(split):
        out, _ = run_decode(c)
    assert G.last_launch_count() == (1 if B <= 64 else 3)   # one fused grid up to 64 sequences
    for b in range(B):
        H.compare_sequence(c, out, b)
    H.check_canaries(c)


@pytest.mark.parametrize("B,starts,s_max", [
    (3, [0, 5, 130], 160),
    (16, list(range(0, 1600, 100)), 1600),
    (64, None, 520),
])
def test_decode_three_kernel_path_matches_oracle(weights, B, starts, s_max):
    """The same step launched as three kernels (projection, attention, output
    projection) instead of the fused grid."""
    if starts is None:
        g = torch.Generator().manual_seed(B)
        starts = torch.randint(0, s_max, (B,), generator=g).tolist()
    c = H.make_case(B, 1, starts, s_max, weights=weights)
    prev = G.set_decode_fusion(False)
    try:
        out, _ = run_decode(c)
        assert G.last_launch_count() == 3
    finally:
        G.set_decode_fusion(prev)
    for b in range(B):
        H.compare_sequence(c, out, b)
    H.check_canaries(c)


@pytest.mark.parametrize("split", SPLITS)
@pytest.mark.parametrize("B", [1, 2])   # B=1: the one-token W_O path, W_O rows on the CTAs past the attention's
def test_decode_every_start_position_invalid_is_reported(weights, split, B):
    """No valid sequence: the fused grid must still finish (its last phase
    waits on no sequence) and leave every cache row untouched."""
    c = H.make_case(B, 1, [3, 4][:B], 16, weights=weights)
    d = c.dev
    sp = torch.tensor([11, 12][:B], dtype=torch.int32, device="cuda")   # > max_start_pos 9
    ws = G.make_workspace(B, 1, 10)
    with attention_split(split):
        G.decode(d["x"], sp, 9, d["wq"], d["wk"], d["wv"], d["wo"], H.rope_for(c), d["cache_k"], d["cache_v"],
                 workspace=ws)
    torch.cuda.synchronize()
    assert G.device_status(ws, clear=True) == 1
    assert torch.equal(d["cache_k"], d["cache_k0"]) and torch.equal(d["cache_v"], d["cache_v0"])
    # the workspace (its grid counters included) is ready for the next call
    sp.copy_(torch.tensor([3, 4][:B], dtype=torch.int32))
    with attention_split(split):
        out = G.decode(d["x"], sp, 9, d["wq"], d["wk"], d["wv"], d["wo"], H.rope_for(c), d["cache_k"],
                       d["cache_v"], workspace=ws)
    torch.cuda.synchronize()
    assert G.device_status(ws) == 0
    for b in range(B):
        H.compare_sequence(c, out, b)


def test_decode_is_repeatable_with_a_reused_workspace(weights):
    c = H.make_case(5, 1, [700, 10, 333, 1024, 1], 1100, weights=weights)
    out1, ws = run_decode(c)
    out1 = out1.clone()
    out2, _ = run_decode(c, ws=ws)
    assert H.rel_l2(H.f64(out2), H.f64(out1)) < 1e-3
    for b in range(5):
        H.compare_sequence(c, out2, b)


@pytest.mark.parametrize("split", SPLITS)
def test_decode_bad_start_position_is_reported_and_skipped(weights, split):
    c = H.make_case(3, 1, [5, 9, 7], 16, weights=weights)
    d = c.dev
    sp = torch.tensor([5, 12, 7], dtype=torch.int32, device="cuda")   # 12 > max_start_pos 9
    ws = G.make_workspace(3, 1, 10)
    out = torch.full_like(d["x"], float("nan"))
    with attention_split(split):
        G.decode(d["x"], sp, 9, d["wq"], d["wk"], d["wv"], d["wo"], H.rope_for(c), d["cache_k"], d["cache_v"],
                 out=out, workspace=ws)
    assert G.device_status(ws, clear=True) == 1
    assert torch.equal(d["cache_k"][1], d["cache_k0"][1])   # skipped sequence untouched
    c.start = [5, 9, 7]
    for b in (0, 2):
        H.compare_sequence(c, out, b)


@pytest.mark.parametrize("name", ["decode_b1_p15", "decode_b16_p1000"])
@pytest.mark.parametrize("split", SPLITS)
def test_decode_workloads_full(weights, name, split):
    w = I.workload(name)
    c = H.make_case(w.B, 1, w.start_positions().tolist(), w.cache_rows(), weights=weights)
    with attention_split(split):
        out, _ = run_decode(c)
    worst = 0.0
    for b in range(w.B):
        worst = max(worst, H.compare_sequence(c, out, b)[0])
    H.check_canaries(c)


@pytest.mark.parametrize("B,starts,s_max", [
    (1, [0], 2),                                  # one key per head: o_h = v_{h//4}
    (1, [1000], 1001),                            # one sequence over 8 stages (the one-token W_O path)
    (2, [127, 128], 130),                         # a stage of 128 keys whole, and one key past it
    (5, [126, 255, 256, 383, 1], 400),            # stage edges from both sides, ragged
    (19, [int(v) for v in np.random.default_rng(19).integers(0, 900, 19)], 900),  # every SM holds a pair
])
def test_decode_head_major_edges(weights, B, starts, s_max):
    """The head-major split at the edges of its 128-position stages: warps
    whose 16 keys lie past the sequence skip the stage, and the warps'
    states are combined in shared memory."""
    c = H.make_case(B, 1, starts, s_max, weights=weights)
    with attention_split("head"):
        out, _ = run_decode(c)
    for b in range(B):
        H.compare_sequence(c, out, b)
    H.check_canaries(c)


@pytest.mark.parametrize("split", SPLITS)
def test_decode_stale_new_row_never_reaches_the_scores(weights, split):
    """Row P of the cache holds NaN before the call. The head-major split
    requests the stage holding P before the projection has written that row
    (the warp holding key P then writes the new row over the stale copy); the
    position-major split reads it only after the gate. Either way the NaN
    must not reach the output, at one stage (P < 128) and at several."""
    starts = [0, 15, 127, 200, 383]
    c = H.make_case(len(starts), 1, starts, 400, weights=weights)
    for b, p in enumerate(starts):
        c.dev["cache_k"][b, p] = float("nan")
        c.dev["cache_v"][b, p] = float("nan")
    with attention_split(split):
        out, _ = run_decode(c)
    assert torch.isfinite(out.float()).all()
    for b in range(c.B):
        H.compare_sequence(c, out, b)
    H.check_canaries(c)


def test_decode_splits_alternate_on_one_workspace(weights):
    """Calls switching between the two attention splits share one workspace:
    each leaves the grid counters ready for the other."""
    c = H.make_case(6, 1, [1000, 3, 517, 64, 0, 130], 1100, weights=weights)
    ws = G.make_workspace(6, 1, 1001)
    for split in ("head", "position", "head", "auto", "position"):
        with attention_split(split):
            out, _ = run_decode(c, ws=ws)
        for b in range(6):
            H.compare_sequence(c, out, b)


def test_decode_split_setting_is_validated():
    assert G.lib().gqa_set_decode_attention_split(3) == -1
    assert G.lib().gqa_set_decode_attention_split(-1) == -1
    with pytest.raises(ValueError):
        G.set_decode_attention_split("rows")


class wait_limit:
    """Limit of the decode kernels' grid-wide waits inside the with-block."""

    def __init__(self, ns):
        self.ns = ns

    def __enter__(self):
        self.prev = G.set_wait_limit_ns(self.ns)

    def __exit__(self, *exc):
        G.set_wait_limit_ns(self.prev)


COUNTERS = 16   # byte offset of the grid counters in the workspace's status region


@pytest.mark.parametrize("path,split,counter", [
    ("fused", "head", 0),        # the Q|K|V gate of the one-kernel step
    ("fused", "head", 1),        # the W_O gate
    ("fused", "position", 0),
    ("fused", "position", 3),    # the attention's meeting before its merges
    ("three", "auto", 0),        # the standalone attention kernel's meeting
])
def test_grid_wait_timeout_is_reported_and_recovered(weights, path, split, counter):
    """Failure injected on the host: a grid counter in the workspace is set so
    far below its target that the wait on it cannot finish. With a 1 ms limit
    the call must end, record GQA_DEV_WAIT_TIMEOUT, leave every grid counter
    reset and every cache row outside the new ones untouched; the next call
    on the same workspace must pass parity."""
    c = H.make_case(3, 1, [1000, 517, 64], 1100, weights=weights)   # sequences split between CTAs
    d = c.dev
    sp = torch.tensor(c.start, dtype=torch.int32, device="cuda")
    ws = G.make_workspace(3, 1, 1001)
    counters = ws[COUNTERS:COUNTERS + 16].view(torch.int32)
    counters[counter] = -(1 << 30)
    prev = G.set_decode_fusion(path == "fused")
    try:
        with attention_split(split), wait_limit(1_000_000):
            G.decode(d["x"], sp, 1000, d["wq"], d["wk"], d["wv"], d["wo"], H.rope_for(c), d["cache_k"], d["cache_v"],
                     workspace=ws)
            torch.cuda.synchronize()
        assert G.device_status(ws, clear=True) == 2      # GQA_DEV_WAIT_TIMEOUT
        assert int(counters.abs().sum()) == 0, f"grid counters left {counters.tolist()}"
        H.check_canaries(c)
        # the same step again on the untouched cache, default limit: parity
        d["cache_k"].copy_(d["cache_k0"])
        d["cache_v"].copy_(d["cache_v0"])
        with attention_split(split):
            out, _ = run_decode(c, ws=ws)
    finally:
        G.set_decode_fusion(prev)
    for b in range(3):
        H.compare_sequence(c, out, b)
    H.check_canaries(c)


@pytest.mark.parametrize("counter", [0, 3])   # the Q|K|V gate after the three passes; the merges' meeting
def test_mha_fused_wait_timeout_is_reported_and_recovered(mha_weights, counter):
    """The multi-head one-grid step: a grid counter that cannot reach its
    target ends the call under a 1 ms limit with GQA_DEV_WAIT_TIMEOUT, every
    counter reset and no cache row outside the new ones changed; the next
    call on the same workspace passes parity."""
    starts = [1000, 517, 64]
    c = H.make_case(3, 1, starts, 1100, seed=3, weights=mha_weights, dims=I.LLAMA31_8B_MHA)
    d = c.dev
    sp = torch.tensor(starts, dtype=torch.int32, device="cuda")
    ws = G.make_workspace(3, 1, 1001)
    counters = ws[COUNTERS:COUNTERS + 16].view(torch.int32)
    counters[counter] = -(1 << 30)
    prev = G.set_decode_fusion(True)
    try:
        with wait_limit(1_000_000):
            G.decode(d["x"], sp, 1000, d["wq"], d["wk"], d["wv"], d["wo"], H.rope_for(c), d["cache_k"],
                     d["cache_v"], workspace=ws, n_kv_heads=32)
            torch.cuda.synchronize()
        assert G.last_launch_count() == 1
        assert G.device_status(ws, clear=True) == 2      # GQA_DEV_WAIT_TIMEOUT
        assert int(counters.abs().sum()) == 0, f"grid counters left {counters.tolist()}"
        H.check_canaries(c)
        d["cache_k"].copy_(d["cache_k0"])
        d["cache_v"].copy_(d["cache_v0"])
        out = G.decode(d["x"], sp, 1000, d["wq"], d["wk"], d["wv"], d["wo"], H.rope_for(c), d["cache_k"],
                       d["cache_v"], workspace=ws, n_kv_heads=32)
        torch.cuda.synchronize()
        assert G.device_status(ws) == 0
    finally:
        G.set_decode_fusion(prev)
    for b in range(3):
        H.compare_sequence(c, out, b)
    H.check_canaries(c)


def test_wait_limit_setting_round_trips():
    prev = G.set_wait_limit_ns(5_000_000)
    try:
        assert G.set_wait_limit_ns(0) == 5_000_000
        assert G.set_wait_limit_ns(prev) == 2_000_000_000   # 0 restored the default
    finally:
        G.set_wait_limit_ns(prev)


def test_block_forward_decode_matches_oracle(weights):
    c = H.make_case(4, 1, [37, 37, 37, 37], 40, weights=weights)
    d = c.dev
    ws = G.make_workspace(4, 1, 38)
    out = G.block_forward(d["x"], 37, d["wq"], d["wk"], d["wv"], d["wo"], H.rope_for(c), d["cache_k"],
                          d["cache_v"], workspace=ws)
    torch.cuda.synchronize()
    assert G.device_status(ws) == 0
    assert G.last_launch_count() == 1
    for b in range(4):
        H.compare_sequence(c, out, b)


# ------------------------------------------------------------------ prefill

@pytest.mark.parametrize("B,T,start,s_max", [
    (1, 5, 0, 8),          # few tokens: few-token projection path with T > 1
    (2, 37, 0, 40),        # M = 74: tensor-core projection, ragged M tile and query tile
    (1, 50, 70, 130),      # chunked prefill over a cached prefix
    (1, 300, 0, 300),      # three M tiles, ragged
    (3, 129, 200, 400),    # chunked, several sequences
])
def test_prefill_small_matches_oracle(weights, B, T, start, s_max):
    c = H.make_case(B, T, [start] * B, s_max, weights=weights)
    out, _ = run_prefill(c)
    for b in range(B):
        H.compare_sequence(c, out, b)
    H.check_canaries(c)


def test_prefill_then_decode_equals_longer_prefill(weights):
    c = H.make_case(1, 9, [0], 16, weights=weights)
    out9, _ = run_prefill(c)
    # decode the 10th token on top of the cache the prefill wrote
    x10 = I.draw_x(torch.Generator().manual_seed(99), 1, 1).cuda()
    d = c.dev
    sp = torch.tensor([9], dtype=torch.int32, device="cuda")
    o10 = G.decode(x10, sp, 9, d["wq"], d["wk"], d["wv"], d["wo"], H.rope_for(c), d["cache_k"], d["cache_v"])
    c2 = H.make_case(1, 10, [0], 16, weights=weights)
    c2.dev["x"][:, :9] = c.dev["x"]
    c2.dev["x"][:, 9:] = x10
    c2.host["x"] = c2.dev["x"].cpu()
    out10, _ = run_prefill(c2)
    torch.cuda.synchronize()
    ref = H.f64(out10[0, 9])
    got = H.f64(o10[0, 0])
    assert H.rel_l2(got, ref) < 1e-2
    for name in ("cache_k", "cache_v"):
        d1 = H.ordered_bf16(c.dev[name][0, :10].cpu()) - H.ordered_bf16(c2.dev[name][0, :10].cpu())
        assert np.abs(d1).max() <= 1


def test_chunked_prefill_large_matches_oracle(weights):
    """A 640-token chunk after 1800 cached positions: ragged against both the
    32-position query tiles and the 64-key tiles (the diagonal tile straddles
    the cached prefix); sampled query rows plus the first and the last."""
    c = H.make_case(2, 640, [1800, 1800], 2440, weights=weights)
    out, _ = run_prefill(c)
    g = np.random.default_rng(1)
    for b in range(c.B):
        q = sorted(set(g.choice(c.T, 48, replace=False).tolist()) | {0, 31, 32, c.T - 1})
        H.compare_sequence(c, out, b, query_rows=q)
    H.check_canaries(c)


@pytest.mark.parametrize("kind", ["decode", "prefill"])
def test_llama3_unscaled_rope_block_matches_oracle(weights, kind):
    """Llama 3 8B ("use_scaled_rope": false): same block, only the RoPE table
    differs. Positions past the 8192-token original context, where the scaled
    and unscaled tables disagree most; the scaled table's answer must then be
    far from the GPU's (the table really is the unscaled one)."""
    if kind == "decode":
        c = H.make_case(3, 1, [9000, 12345, 8191], 12346, rope=I.LLAMA3_ROPE, weights=weights)
        out, _ = run_decode(c)
    else:
        c = H.make_case(1, 96, [9000], 9096, rope=I.LLAMA3_ROPE, weights=weights)
        out, _ = run_prefill(c)
    for b in range(c.B):
        H.compare_sequence(c, out, b)
    H.check_canaries(c)
    import dataclasses
    scaled = dataclasses.replace(c, rope=I.LLAMA31_ROPE)
    other, _, _ = H.oracle_sequence(scaled, 0)
    assert H.rel_l2(H.f64(out[0]), other) > 0.1


@pytest.mark.parametrize("name,rows", [("prefill_b1_t2048", None), ("prefill_b4_t2048", 192)])
def test_prefill_workloads_full(weights, name, rows):
    w = I.workload(name)
    c = H.make_case(w.B, w.T, w.start_positions().tolist(), w.cache_rows(), weights=weights)
    out, _ = run_prefill(c, entry="block_forward")
    g = np.random.default_rng(0)
    for b in range(w.B):
        q = None if rows is None else sorted(set(g.choice(w.T, rows, replace=False).tolist()) | {0, w.T - 1})
        H.compare_sequence(c, out, b, query_rows=q)
    H.check_canaries(c)


@pytest.mark.parametrize("name,sample", [("batched_decode_b64_p512_32768", 4), ("long_decode_b8_p131071", 2)])
def test_large_decode_workloads_sampled(weights, name, sample):
    w = I.workload(name)
    starts = w.start_positions().tolist()
    c = H.make_case(w.B, 1, starts, w.cache_rows(), weights=weights, cache_device="cuda")
    out, _ = run_decode(c)
    order = np.argsort(starts)
    seqs = sorted({int(order[0]), int(order[-1])} | set(list(range(0, w.B, max(1, w.B // sample)))[:sample]))
    for b in seqs:
        H.compare_sequence(c, out, b)
    # every written row and the rows around it, for all sequences
    for b in range(w.B):
        sp = starts[b]
        for name_ in ("cache_k", "cache_v"):
            now, before = c.dev[name_][b], c.dev[name_ + "0"][b]
            lo = max(0, sp - 64)
            assert torch.equal(now[lo:sp], before[lo:sp])
            assert torch.equal(now[sp + 1:sp + 65], before[sp + 1:sp + 65])


# ------------------------------------------------------------------ the layer: h = x + attention(norm(x))

@pytest.mark.parametrize("B,starts,s_max,fused", [
    (16, [3, 40, 17, 100] * 4, 128, "position"),   # the fused decode grid, both attention splits
    (16, [3, 40, 17, 100] * 4, 128, "head"),
    (16, [3, 40, 17, 100] * 4, 128, False),        # three kernels
    (80, list(range(5, 85)), 100, "auto"),         # above the fused grid's batch: tensor-core projections
])
def test_layer_decode_matches_oracle(weights, B, starts, s_max, fused):
    c = H.make_case(B, 1, starts, s_max, weights=weights)
    g = I.draw_norm_weight(seed=0).cuda()
    d = c.dev
    sp = torch.tensor(starts, dtype=torch.int32, device="cuda")
    ws = G.make_workspace(B, 1, max(starts) + 1)
    prev = G.set_decode_fusion(bool(fused))
    try:
        with attention_split(fused if fused else "auto"):
            h = G.layer_decode(d["x"], sp, max(starts), g, I.NORM_EPS, d["wq"], d["wk"], d["wv"], d["wo"],
                               H.rope_for(c), d["cache_k"], d["cache_v"], workspace=ws)
        torch.cuda.synchronize()
    finally:
        G.set_decode_fusion(prev)
    assert G.device_status(ws) == 0
    for b in range(0, B, max(1, B // 8)):
        H.compare_layer_sequence(c, h, b, g, I.NORM_EPS)
    H.check_canaries(c)


@pytest.mark.parametrize("B,T,start,s_max", [
    (1, 5, 0, 8),         # few tokens: stream-K projections
    (2, 37, 0, 40),       # tensor-core projections with a ragged tile
    (1, 96, 300, 400),    # chunked
])
def test_layer_prefill_matches_oracle(weights, B, T, start, s_max):
    c = H.make_case(B, T, [start] * B, s_max, weights=weights)
    g = I.draw_norm_weight(seed=0).cuda()
    d = c.dev
    ws = G.make_workspace(B, T, start + T)
    h = G.layer_forward(d["x"], start, g, I.NORM_EPS, d["wq"], d["wk"], d["wv"], d["wo"], H.rope_for(c),
                        d["cache_k"], d["cache_v"], workspace=ws)
    torch.cuda.synchronize()
    assert G.device_status(ws) == 0
    for b in range(B):
        H.compare_layer_sequence(c, h, b, g, I.NORM_EPS)
    H.check_canaries(c)
    # the residual is really there: h - x is the normalised block's delta, not h
    assert float((h.float() - d["x"].float()).abs().max()) < float(h.float().abs().max())


def test_rms_norm_matches_oracle():
    """The norm alone: every value within one bf16 ulp of the oracle's (fp32
    arithmetic on the GPU, one rounding), nearly all identical; the x rows
    span four orders of magnitude."""
    gen = torch.Generator().manual_seed(11)
    x = (torch.randn(64, 4096, generator=gen) * torch.logspace(-2, 2, 64).unsqueeze(1)).to(torch.bfloat16)
    g = I.draw_norm_weight(seed=3)
    y = G.rms_norm(x.cuda(), g.cuda(), I.NORM_EPS).cpu()
    ref = O.bf16_round(O.rms_norm(H.f64(x), H.f64(g), I.NORM_EPS))
    got = H.f64(y)
    assert np.all(np.abs(got - ref) <= H.bf16_ulp(ref))
    assert (got != ref).mean() < 1e-3



@pytest.mark.parametrize("fused", [True, False])
def test_layer_decode_chained_layers_match_oracle(fused):
    """Three consecutive layers of one decode step, each with its own weights
    and KV cache, one shared workspace, the output of one the input of the
    next, against the oracle chained in fp64 from the same seeded input (h
    rounded to bf16 between layers, as the block stores it). Layer 0 (whose
    input is the seeded x) is held to the layer bars of
    ``compare_layer_sequence``; the cache rows of later layers, whose inputs
    are earlier layers' outputs, to the delta bar; the final h to the delta
    bar, its max-abs bar widened by one bf16 ulp of h per layer for the
    roundings between layers."""
    B, starts, s_max, L = 4, [0, 17, 128, 300], 320, 3
    cases = [H.make_case(B, 1, starts, s_max, seed=10 + l) for l in range(L)]
    gs = [I.draw_norm_weight(seed=10 + l).cuda() for l in range(L)]
    sp = torch.tensor(starts, dtype=torch.int32, device="cuda")
    ws = G.make_workspace(B, 1, max(starts) + 1)
    prev = G.set_decode_fusion(fused)
    try:
        xs = [cases[0].dev["x"]]
        for l, c in enumerate(cases):
            d = c.dev
            xs.append(G.layer_decode(xs[-1], sp, max(starts), gs[l], I.NORM_EPS, d["wq"], d["wk"], d["wv"], d["wo"],
                                     H.rope_for(c), d["cache_k"], d["cache_v"], workspace=ws))
        torch.cuda.synchronize()
    finally:
        G.set_decode_fusion(prev)
    assert G.device_status(ws) == 0
    for b in range(B):
        H.compare_layer_sequence(cases[0], xs[1], b, gs[0], I.NORM_EPS)
    for c in cases:
        H.check_canaries(c)
    r = I.LLAMA31_ROPE
    freqs = O.rope_frequencies(128, r.theta, r.scaled, r.factor, r.low_freq_factor, r.high_freq_factor,
                               r.original_context)
    for b in range(B):
        h = H.f64(cases[0].host["x"][b])
        for l, c in enumerate(cases):
            w = H.weights64(c)
            sp_b = starts[b]
            h, nk, nv = O.layer_sequence_forward(h, H.f64(gs[l]), I.NORM_EPS, w["wq"], w["wk"], w["wv"], w["wo"],
                                                 sp_b, H.f64(c.dev["cache_k0"][b, :sp_b]),
                                                 H.f64(c.dev["cache_v0"][b, :sp_b]), freqs, 32, 8)
            h = O.bf16_round(h)
            if l > 0:
                for name, ref in (("cache_k", nk), ("cache_v", nv)):
                    got = H.f64(c.dev[name][b, sp_b:sp_b + 1])
                    assert H.rel_l2(got, ref) <= H.REL_L2_TOL, f"layer {l} {name} row of sequence {b}"
                    assert float(np.abs(got - ref).max()) <= H.MAX_ABS_TOL, f"layer {l} {name} row of sequence {b}"
        got = H.f64(xs[-1][b])
        assert H.rel_l2(got, h) <= H.REL_L2_TOL
        # both sides round h to bf16 after every layer: where they land on
        # neighbouring values an element differs by one ulp of h (0.0625 for
        # |h| in [8, 16)), and the residual carries that difference into the
        # next layer's h unchanged, so L layers allow L ulps on top of the
        # delta bar
        err = np.abs(got - h) - L * H.bf16_ulp(np.abs(h))
        assert float(err.max()) <= H.MAX_ABS_TOL


# ------------------------------------------------------------ multi-head variant

@pytest.fixture(scope="module")
def mha_weights():
    return I.draw_weights(I.LLAMA31_8B_MHA, seed=3)


@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("B,starts,s_max", [
    (1, [15], 16),                                    # one sequence, one unit
    (4, [0, 17, 128, 300], 320),                      # ragged positions, split sequences
    (9, [int(v) for v in np.random.default_rng(9).integers(0, 700, 9)], 704),  # 16 padded tokens, 36 head groups
    (80, [int(v) for v in np.random.default_rng(5).integers(0, 90, 80)], 96),  # tcgen05 GEMM projections
])
def test_mha_decode_matches_oracle(mha_weights, B, starts, s_max, fused):
    """32 KV heads (query head h with KV head h): the decode path over head
    groups, against the oracle with n_kv_heads = 32. Up to 16 sequences the
    step runs as one grid (Q|K|V in three passes over Wq, Wk, Wv) or as
    three kernels; above, as three kernels either way."""
    c = H.make_case(B, 1, starts, s_max, seed=3, weights=mha_weights, dims=I.LLAMA31_8B_MHA)
    d = c.dev
    sp = torch.tensor(starts, dtype=torch.int32, device="cuda")
    ws = G.make_workspace(B, 1, max(starts) + 1)
    prev = G.set_decode_fusion(fused)
    try:
        out = G.decode(d["x"], sp, max(starts), d["wq"], d["wk"], d["wv"], d["wo"], H.rope_for(c), d["cache_k"],
                       d["cache_v"], workspace=ws, n_kv_heads=32)
        torch.cuda.synchronize()
        launches = G.last_launch_count()
    finally:
        G.set_decode_fusion(prev)
    assert launches == (1 if fused and B <= 16 else 3), launches
    assert G.device_status(ws) == 0
    for b in range(0, B, max(1, B // 6)):
        H.compare_sequence(c, out, b)
    H.check_canaries(c)


@pytest.mark.parametrize("B,T,start,s_max", [
    (1, 5, 0, 8),          # few tokens
    (2, 37, 0, 40),        # one ragged 128-position tile
    (1, 300, 0, 304),      # two CTAs' worth of 256 positions, ragged
    (1, 96, 300, 400),     # chunked: 96 tokens after 300 cached
])
def test_mha_prefill_matches_oracle(mha_weights, B, T, start, s_max):
    c = H.make_case(B, T, [start] * B, s_max, seed=3, weights=mha_weights, dims=I.LLAMA31_8B_MHA)
    d = c.dev
    ws = G.make_workspace(B, T, start + T)
    out = G.block_forward(d["x"], start, d["wq"], d["wk"], d["wv"], d["wo"], H.rope_for(c), d["cache_k"],
                          d["cache_v"], workspace=ws, n_kv_heads=32)
    torch.cuda.synchronize()
    assert G.device_status(ws) == 0
    rows = None if T <= 96 else sorted({0, 1, 127, 128, 129, 255, 256, T - 1})
    for b in range(B):
        H.compare_sequence(c, out, b, query_rows=rows, check_cache=rows is None)
    if rows is not None:
        # every new cache row, checked against the oracle's rows from one full pass
        _, nk, nv = H.oracle_sequence(c, 0, [0])
        H.check_rows_within_one_ulp(d["cache_k"][0, start:start + T], nk, "cache_k rows")
        H.check_rows_within_one_ulp(d["cache_v"][0, start:start + T], nv, "cache_v rows")
    H.check_canaries(c)


def test_mha_with_duplicated_kv_heads_equals_gqa(weights):
    """The multi-head path run on K/V heads duplicated 4 times (and the
    matching weights) gives the grouped path's result: the repeat_kv map
    h // 4 pinned on the GPU."""
    B, starts, s_max = 3, [5, 40, 77], 80
    c = H.make_case(B, 1, starts, s_max, weights=weights)
    d = c.dev
    rep4 = lambda w: w.view(8, 128, 4096).repeat_interleave(4, dim=0).reshape(4096, 4096).contiguous()
    ck4 = d["cache_k0"].repeat_interleave(4, dim=2).contiguous()
    cv4 = d["cache_v0"].repeat_interleave(4, dim=2).contiguous()
    sp = torch.tensor(starts, dtype=torch.int32, device="cuda")
    rope = H.rope_for(c)
    g = G.decode(d["x"], sp, max(starts), d["wq"], d["wk"], d["wv"], d["wo"], rope, d["cache_k"], d["cache_v"])
    m = G.decode(d["x"], sp, max(starts), d["wq"], rep4(d["wk"]), rep4(d["wv"]), d["wo"], rope, ck4, cv4,
                 n_kv_heads=32)
    torch.cuda.synchronize()
    # the two runs accumulate in different kernels (the grouped decode step is
    # one fused grid): equal up to rounding, where a wrong head map is O(1) off
    r2 = H.rel_l2(H.f64(m), H.f64(g))
    assert r2 <= 5e-3, r2
    for b in range(B):
        for cm, cg in ((ck4, d["cache_k"]), (cv4, d["cache_v"])):
            # each of the four copies of a KV head (rows of different CTAs of
            # the Wk / Wv pass, whose sums over k start at different stages)
            # within an ulp of the grouped row
            new = cm[b, starts[b]].view(8, 4, 128)
            for r in range(4):
                H.check_rows_within_one_ulp(new[:, r], H.f64(cg[b, starts[b]]), f"new row {r} of sequence {b}")


@pytest.mark.parametrize("name,rows", [("prefill_chunk_b1_t1024_p7168", 64), ("mha_prefill_b1_t2048", 96)])
def test_next_prefill_workloads_full(weights, mha_weights, name, rows):
    """The bench's chunked and multi-head prefill workloads at full size, on
    sampled query rows (plus the first and last, and the rows either side of a
    128-position tile edge)."""
    w = I.workload(name)
    wts = mha_weights if w.n_kv_heads == 32 else weights
    seed = 3 if w.n_kv_heads == 32 else 0
    c = H.make_case(w.B, w.T, w.start_positions().tolist(), w.cache_rows(), seed=seed, weights=wts, dims=w.dims)
    d = c.dev
    ws = G.make_workspace(w.B, w.T, c.start[0] + w.T)
    out = G.block_forward(d["x"], c.start[0], d["wq"], d["wk"], d["wv"], d["wo"], H.rope_for(c), d["cache_k"],
                          d["cache_v"], workspace=ws, n_kv_heads=w.n_kv_heads)
    torch.cuda.synchronize()
    assert G.device_status(ws) == 0
    g = np.random.default_rng(2)
    q = sorted(set(g.choice(w.T, rows, replace=False).tolist()) | {0, 127, 128, w.T - 1})
    H.compare_sequence(c, out, 0, query_rows=q)
    H.check_canaries(c)


def test_mha_decode_workload_full(mha_weights):
    w = I.workload("mha_decode_b16_p1000")
    c = H.make_case(w.B, 1, w.start_positions().tolist(), w.cache_rows(), seed=3, weights=mha_weights, dims=w.dims)
    d = c.dev
    sp = torch.tensor(c.start, dtype=torch.int32, device="cuda")
    ws = G.make_workspace(w.B, 1, max(c.start) + 1)
    out = G.decode(d["x"], sp, max(c.start), d["wq"], d["wk"], d["wv"], d["wo"], H.rope_for(c), d["cache_k"],
                   d["cache_v"], workspace=ws, n_kv_heads=32)
    torch.cuda.synchronize()
    assert G.device_status(ws) == 0
    for b in range(w.B):
        H.compare_sequence(c, out, b)
    H.check_canaries(c)


# ------------------------------------------------------------ host-buffer entries

def test_host_buffer_entries_match_device_entries(weights):
    """decode_host / block_forward_host (x and the result in host memory,
    uploads on the library's copy stream, two stage buffers in turn) give the
    device entries' results bit for bit over consecutive calls."""
    B, starts, s_max = 4, [3, 40, 77, 120], 128
    c = H.make_case(B, 1, starts, s_max, weights=weights)
    d = c.dev
    ck2, cv2 = d["cache_k0"].clone(), d["cache_v0"].clone()
    sp = torch.tensor(starts, dtype=torch.int32, device="cuda")
    rope = H.rope_for(c)
    stage = G.make_host_stage(B, 1)
    ws = G.make_workspace(B, 1, max(starts) + 1)
    g = torch.Generator().manual_seed(7)
    xs = [I.draw_x(g, B, 1).pin_memory() for _ in range(3)]
    outs = []
    for xh in xs:   # three calls: both stage pairs, then the first again
        outs.append(G.decode_host(xh, sp, max(starts), d["wq"], d["wk"], d["wv"], d["wo"], rope, ck2, cv2,
                                  stage=stage))
    G.host_stage_wait(stage)
    torch.cuda.current_stream().synchronize()
    for xh, oh in zip(xs, outs):
        ref = G.decode(xh.cuda(), sp, max(starts), d["wq"], d["wk"], d["wv"], d["wo"], rope, d["cache_k"],
                       d["cache_v"], workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(oh, ref.cpu())
    assert torch.equal(ck2, d["cache_k"]) and torch.equal(cv2, d["cache_v"])
    G.release_host_stage(stage)

    cp = H.make_case(1, 40, [0], 48, weights=weights)
    dp = cp.dev
    ck3, cv3 = dp["cache_k0"].clone(), dp["cache_v0"].clone()
    stage = G.make_host_stage(1, 40)
    oh = G.block_forward_host(cp.host["x"].pin_memory(), 0, dp["wq"], dp["wk"], dp["wv"], dp["wo"], H.rope_for(cp),
                              ck3, cv3, stage=stage)
    G.host_stage_wait(stage)
    ref = G.block_forward(dp["x"], 0, dp["wq"], dp["wk"], dp["wv"], dp["wo"], H.rope_for(cp), dp["cache_k"],
                          dp["cache_v"])
    torch.cuda.synchronize()
    assert torch.equal(oh, ref.cpu())
    assert torch.equal(ck3, dp["cache_k"])
    G.release_host_stage(stage)


def test_decode_reused_workspace_across_batch_shapes(weights):
    """One workspace for a large step (every CTA leaves partials) and then a
    small one whose few units leave most CTAs empty: the small step's merges
    read the partials of the CTAs that hold its units only, never the slots
    the large step left behind."""
    big = H.make_case(16, 1, list(range(200, 1800, 100)), 1800, weights=weights)
    ws = G.make_workspace(16, 1, 1800)
    with attention_split("position"):
        run_decode(big, ws=ws)
    for fused, split in ((True, "position"), (True, "head"), (False, "auto")):
        small = H.make_case(3, 1, [0, 5, 130], 160, seed=1)
        prev = G.set_decode_fusion(fused)
        try:
            with attention_split(split):
                out, _ = run_decode(small, ws=ws)
        finally:
            G.set_decode_fusion(prev)
        for b in range(3):
            H.compare_sequence(small, out, b)


@pytest.mark.parametrize("kind", ["decode_fused", "decode_fused_head", "decode_three", "prefill"])
def test_workspace_and_output_guards_untouched(weights, kind):
    """Bytes past the workspace size the library asks for, and past the
    output rows, keep their pattern: no kernel writes outside its buffers."""
    guard = 1 << 16
    B, T, starts, s_max = (4, 1, [3, 40, 77, 120], 128) if kind != "prefill" else (2, 37, [0, 0], 40)
    c = H.make_case(B, T, starts, s_max, weights=weights)
    d = c.dev
    need = G.workspace_bytes(B, T, max(starts) + T)
    ws_full = torch.zeros(need + guard, dtype=torch.uint8, device="cuda")
    ws_full[need:] = 0xA5
    out_full = torch.full((B * T * 4096 + guard // 2,), 7.0, dtype=torch.bfloat16, device="cuda")
    out = out_full[:B * T * 4096].view(B, T, 4096)
    ws = ws_full[:need]
    rope = H.rope_for(c)
    if kind == "prefill":
        G.block_forward(d["x"], 0, d["wq"], d["wk"], d["wv"], d["wo"], rope, d["cache_k"], d["cache_v"], out=out,
                        workspace=ws)
    else:
        sp = torch.tensor(starts, dtype=torch.int32, device="cuda")
        prev = G.set_decode_fusion(kind != "decode_three")
        try:
            with attention_split("head" if kind == "decode_fused_head" else "position"):
                G.decode(d["x"], sp, max(starts), d["wq"], d["wk"], d["wv"], d["wo"], rope, d["cache_k"],
                         d["cache_v"], out=out, workspace=ws)
        finally:
            G.set_decode_fusion(prev)
    torch.cuda.synchronize()
    assert G.device_status(ws) == 0
    assert bool((ws_full[need:] == 0xA5).all()), "a write past the workspace"
    assert bool((out_full[B * T * 4096:] == 7.0).all()), "a write past the output"
    for b in range(B):
        H.compare_sequence(c, out, b)
    H.check_canaries(c)


def test_host_buffer_entry_with_the_default_stage(weights):
    """decode_host without a stage uses the binding's default stage for the
    device and shape; host_stage_wait on it joins the read-back."""
    B, starts, s_max = 2, [10, 90], 96
    c = H.make_case(B, 1, starts, s_max, weights=weights)
    d = c.dev
    ck2, cv2 = d["cache_k0"].clone(), d["cache_v0"].clone()
    sp = torch.tensor(starts, dtype=torch.int32, device="cuda")
    rope = H.rope_for(c)
    xh = c.host["x"].pin_memory()
    oh = G.decode_host(xh, sp, max(starts), d["wq"], d["wk"], d["wv"], d["wo"], rope, ck2, cv2)
    G.host_stage_wait(G.default_host_stage(B, 1))
    torch.cuda.current_stream().synchronize()
    ref = G.decode(d["x"], sp, max(starts), d["wq"], d["wk"], d["wv"], d["wo"], rope, d["cache_k"], d["cache_v"])
    torch.cuda.synchronize()
    assert torch.equal(oh, ref.cpu())
