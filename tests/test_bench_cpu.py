"""The bench's algorithmic work counts (the roofline's numerators), checked
against the figures the design derives from the pages' sizes: bytes of a
decode step (weights, K/V rows read and written, x, q, o, delta) and FLOPs of
a causal prefill (projections plus the visible (query, key) pairs)."""
import bench
import gqa_inputs as I


def test_decode_step_bytes():
    # B=16 at P=1000: 83,886,080 weight bytes + 16 x 1,001 positions x 4,096
    # + 16 new rows x 4,096 + x and delta (2 x 16 x 8,192)
    b = bench.step_bytes(16, [1000] * 16)
    assert b["step"] == 83886080 + 16 * 1001 * 4096 + 16 * 4096 + 2 * 16 * 8192 == 149815296
    assert b["decode_step"] == b["step"]
    # B=1 at P=15 (16 keys)
    assert bench.step_bytes(1, [15])["step"] == 83972096
    # B=8 at P=131,071: 512 MiB of K and V per sequence
    assert bench.step_bytes(8, [131071] * 8)["step"] == 4379017216
    # the three-kernel split covers the weights exactly once
    assert (bench.step_bytes(16, [1000] * 16)["qkv_projection"] - 16 * (8192 + 8192 + 4096)
            + bench.step_bytes(16, [1000] * 16)["o_projection"] - 2 * 16 * 8192) == bench.weight_bytes()


def test_decode_step_bytes_multi_head():
    # 32 KV heads: 134,217,728 weight bytes, 16,384 bytes per position
    assert bench.weight_bytes(4096) == 4 * 4096 * 4096 * 2
    b = bench.step_bytes(16, [1000] * 16, kv_row=4096)
    assert b["step"] == 134217728 + 16 * 1001 * 16384 + 16 * 16384 + 2 * 16 * 8192


def test_prefill_flops():
    # T=2048 from position 0: 2 x 41,943,040 per token + 16,384 per visible pair
    f = bench.step_flops(1, 2048, 0)
    pairs = 2048 * 2049 // 2
    assert f["step"] == 2.0 * 41943040 * 2048 + 16384.0 * pairs
    assert abs(f["step"] - 2.0618e11) / 2.0618e11 < 1e-4
    assert abs(bench.step_flops(4, 2048, 0)["step"] - 8.2470e11) / 8.2470e11 < 1e-4
    # a chunk after 7,168 cached positions sees them all
    chunk = bench.step_flops(1, 1024, 7168)["prefill_attention"]
    assert chunk == 16384.0 * sum(7168 + t + 1 for t in range(1024))
    # 32 KV heads: the Q|K|V projection is 12,288 outputs wide
    assert bench.step_flops(1, 2048, 0, kv_row=4096)["qkv_projection"] == 2.0 * 2048 * 4096 * 12288


def test_workloads_match_their_descriptions():
    w = I.workload("decode_b16_p1000")
    assert (w.B, w.T, w.start_pos, w.cache_rows()) == (16, 1, 1000, 1001)
    w = I.workload("batched_decode_b64_p512_32768")
    p = w.start_positions()
    assert w.B == 64 and int(p.min()) >= 512 and int(p.max()) <= 32768
    assert I.workload("mha_decode_b16_p1000").dims.n_kv_heads == 32
    assert I.workload("decode32_b16_p1000").layers == 32


def test_headline_line_carries_every_other_configuration():
    """The headline (B=16 at 1,001 keys) and the five secondary workloads are
    the benchmark's six configurations: B=1 at 16 keys, the batched decode,
    the two prefills and the long-context decode."""
    names = [n for n, _, _ in bench.SECONDARY]
    assert bench.args_default_workload() == "decode_b16_p1000"
    assert sorted(names) == sorted(["decode_b1_p15", "batched_decode_b64_p512_32768", "long_decode_b8_p131071",
                                    "prefill_b1_t2048", "prefill_b4_t2048"])
    assert all(cap > 0 and reps >= 1 for _, cap, reps in bench.SECONDARY)


def test_clock_summary_falls_back_to_the_soak():
    c = bench.ClockSampler(0)
    row = "0, {mhz}, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, {cap}"
    c.rows = [(1.0, row.format(mhz=1500, cap="Not Active")), (5.0, row.format(mhz=2070, cap="Active")),
              (5.5, row.format(mhz=2060, cap="Not Active"))]
    c.t0, c.t1, c.s0, c.s1 = 2.0, 2.001, 4.9, 6.0     # no sample inside a 1 ms timed region
    s = c.summary(soak_replays=64)
    assert s["samples_in_timed_region"] == 0 and s["source"] == "soak"
    assert s["sm_mhz"] == 2065 and s["soak"]["samples"] == 2 and s["reasons"] == ["sw_power_cap"]
    c.t0, c.t1 = 0.5, 1.5
    assert c.summary()["source"] == "timed region" and c.summary()["sm_mhz"] == 1500
