"""C-ABI checks that need no GPU: the library builds for sm_103a, loads,
exports every function include/gqa.h declares, sizes workspaces, and rejects
bad arguments on the host before anything is launched.

Every call below fails validation by construction (the pointers are fake
but are never dereferenced, because validation runs before any launch)."""
import ctypes

import pytest

import grouped_query_attention_gemv_gb300 as G
from grouped_query_attention_gemv_gb300 import build as gbuild


@pytest.fixture(scope="module")
def lib():
    gbuild.build()
    return G.lib()


def test_every_declared_symbol_is_exported(lib):
    names = G.exported_symbols()
    assert set(names) >= {"gqa_block_forward", "gqa_decode", "gqa_prefill", "gqa_workspace_bytes",
                          "gqa_strerror", "gqa_rope_table"}
    for n in names:
        assert hasattr(lib, n), f"{n} declared in gqa.h but not exported"


def test_strerror_covers_codes(lib):
    for code in (0, -1, -2, -3, -4, -5):
        assert lib.gqa_strerror(code)
    assert b"unknown" in lib.gqa_strerror(-99)


def test_workspace_sizes(lib):
    ws = G.workspace_bytes
    assert ws(0, 1, 1) == 0 and ws(1, 0, 1) == 0 and ws(1, 4, 3) == 0   # max_keys < T
    a, b = ws(16, 1, 1001), ws(16, 1, 131072)
    assert 0 < a == b          # decode scratch is per warp of the grid, not per cached position
    assert ws(32, 1, 1001) > a  # ... but grows with the batch
    assert ws(1, 2048, 2048) >= 2 * 2048 * 4096 * 2    # rotated q + attention output, bf16
    assert ws(64, 1, 32769) % 256 == 0


FAKE = 1 << 20   # aligned, never dereferenced


def call_block(lib, **kw):
    a = dict(x=FAKE, B=2, T=1, start_pos=5, wq=FAKE, wk=FAKE, wv=FAKE, wo=FAKE, rope=FAKE, rope_rows=64,
             ck=FAKE, cv=FAKE, s_max=64, out=FAKE, ws=FAKE, ws_bytes=1 << 40, stream=None)
    a.update(kw)
    return lib.gqa_block_forward(a["x"], a["B"], a["T"], a["start_pos"], a["wq"], a["wk"], a["wv"], a["wo"],
                                 a["rope"], a["rope_rows"], a["ck"], a["cv"], a["s_max"], a["out"], a["ws"],
                                 a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(x=None), -1), (dict(wo=None), -1), (dict(ws=None), -1), (dict(rope=None), -1),
    (dict(B=0), -1), (dict(T=0), -1), (dict(start_pos=-1), -1),
    (dict(start_pos=60, T=5), -1),          # start_pos + T > s_max
    (dict(start_pos=60, T=4, rope_rows=63), -1),   # beyond the rope table
    (dict(x=FAKE + 2), -2), (dict(ck=FAKE + 8), -2), (dict(out=FAKE + 4), -2),
    (dict(ws_bytes=16), -3),
])
def test_block_forward_rejects_bad_arguments(lib, kw, code):
    assert call_block(lib, **kw) == code


def test_decode_rejects_bad_arguments(lib):
    d = lib.gqa_decode
    args = [FAKE, 4, FAKE, 10, FAKE, FAKE, FAKE, FAKE, FAKE, 64, FAKE, FAKE, 64, FAKE, FAKE, 1 << 40, None]
    bad = list(args)
    bad[2] = None          # start_pos array
    assert d(*bad) == -1
    bad = list(args)
    bad[3] = 64            # max_start_pos + 1 > s_max
    assert d(*bad) == -1
    bad = list(args)
    bad[2] = FAKE + 2      # start_pos array misaligned
    assert d(*bad) == -2
    bad = list(args)
    bad[15] = 100          # workspace too small
    assert d(*bad) == -3


def test_rope_table_rejects_bad_arguments(lib):
    f = lib.gqa_rope_table
    assert f(None, 16, 5e5, 1, 8.0, 1.0, 4.0, 8192.0, None) == -1
    assert f(FAKE, 0, 5e5, 1, 8.0, 1.0, 4.0, 8192.0, None) == -1
    assert f(FAKE, 16, 5e5, 1, 8.0, 4.0, 1.0, 8192.0, None) == -1   # high <= low
    assert f(FAKE + 4, 16, 5e5, 1, 8.0, 1.0, 4.0, 8192.0, None) == -2


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(G, "_LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(G, "_lib", None)
    with pytest.raises(ImportError):
        G.lib()


def test_decode_static_scratch_holds_every_batch_up_to_64_at_any_length(lib):
    # the header promises that any batch of up to 64 sequences fits the static
    # scratch at any cached length: a decode workspace does not grow with the
    # length, and B = 64 is the largest (the few-token projection's partials)
    need = [G.workspace_bytes(B, 1, 1 << 30) for B in range(1, 65)]
    assert all(n > 0 for n in need)
    assert max(need) <= G.STATIC_SCRATCH_BYTES
    assert need[-1] == max(need)
    assert all(G.workspace_bytes(64, 1, k) == need[-1] for k in (1, 1001, 131072))


def test_decode_static_rejects_requests_beyond_its_scratch(lib):
    # B = 2048 needs far more than the static scratch: rejected on the host
    # before any device work
    assert G.workspace_bytes(2048, 1, 1024) > G.STATIC_SCRATCH_BYTES
    r = lib.gqa_decode_static(FAKE, 2048, FAKE, 1023, FAKE, FAKE, FAKE, FAKE, FAKE, 1024, FAKE, FAKE, 1024,
                              FAKE, None)
    assert r == -6
    assert b"static" in lib.gqa_strerror(-6)
    assert lib.gqa_decode_static(FAKE, 0, FAKE, 10, FAKE, FAKE, FAKE, FAKE, FAKE, 64, FAKE, FAKE, 64, FAKE, None) == -1


def test_layer_entries_reject_bad_arguments(lib):
    """Validation of the norm weight, eps and the output buffer happens on the
    host before anything else (no device needed)."""
    f = lib.gqa_layer_forward
    ok = [FAKE, 1, 4, 0, FAKE, 1e-5, FAKE, FAKE, FAKE, FAKE, FAKE, 64, FAKE, FAKE, 64, FAKE + 4096, FAKE, 0, None]
    for i, v, code in ((4, None, -1),          # no norm weight
                       (5, 0.0, -1),           # eps must be > 0
                       (5, -1e-5, -1),
                       (5, float("nan"), -1),
                       (4, FAKE + 8, -2),      # norm weight misaligned
                       (15, FAKE, -1)):        # h is x itself
        bad = list(ok)
        bad[i] = v
        assert f(*bad) == code, (i, v)
    d = lib.gqa_layer_decode
    okd = [FAKE, 4, FAKE, 10, FAKE, 1e-5, FAKE, FAKE, FAKE, FAKE, FAKE, 64, FAKE, FAKE, 64, FAKE + 4096, FAKE, 0,
           None]
    bad = list(okd)
    bad[4] = None
    assert d(*bad) == -1
    bad = list(okd)
    bad[15] = FAKE
    assert d(*bad) == -1


def test_kv_head_entries_reject_bad_arguments(lib):
    """gqa_block_forward_nkv / gqa_decode_nkv take 8 or 32 KV heads only; the
    multi-head decode caps the batch at 512 (its 4 head groups per sequence
    are attention units of their own), and every decode call refuses a unit
    count that the 32-bit split of the work could not hold."""
    f = lib.gqa_block_forward_nkv
    ok = [FAKE, 2, 1, 5, 8, FAKE, FAKE, FAKE, FAKE, FAKE, 64, FAKE, FAKE, 64, FAKE, FAKE, 1 << 40, None]
    for n_kv in (0, 1, 4, 16, 64, -8):
        bad = list(ok)
        bad[4] = n_kv
        assert f(*bad) == -1, n_kv
    bad = list(ok)
    bad[0] = None
    assert f(*bad) == -1
    d = lib.gqa_decode_nkv
    okd = [FAKE, 4, FAKE, 10, 32, FAKE, FAKE, FAKE, FAKE, FAKE, 64, FAKE, FAKE, 64, FAKE, FAKE, 1 << 40, None]
    bad = list(okd)
    bad[4] = 16
    assert d(*bad) == -1
    bad = list(okd)
    bad[1] = 513          # 32 KV heads: at most 512 sequences
    assert d(*bad) == -1
    big = (1 << 30) + 1   # 2^26 units per sequence: 32-bit unit arithmetic would overflow
    for fn, a in ((lib.gqa_decode, [FAKE, 64, FAKE, 1 << 30, FAKE, FAKE, FAKE, FAKE, FAKE, big, FAKE, FAKE, big,
                                    FAKE, FAKE, 1 << 40, None]),
                  (d, [FAKE, 64, FAKE, 1 << 30, 32, FAKE, FAKE, FAKE, FAKE, FAKE, big, FAKE, FAKE, big, FAKE, FAKE,
                       1 << 40, None])):
        assert fn(*a) == -1


def test_host_entries_reject_bad_arguments(lib):
    """The host-buffer entries check their own arguments (host pointers, the
    stage's size and alignment) and the block's before anything is created
    or enqueued."""
    sb = lib.gqa_host_stage_bytes
    assert sb(0, 1) == 0 and sb(1, 0) == 0
    assert sb(16, 1) == 4 * 16 * 4096 * 2 and sb(3, 5) % 256 == 0
    d = lib.gqa_decode_host
    ok = [FAKE, 4, FAKE, 10, 8, FAKE, FAKE, FAKE, FAKE, FAKE, 64, FAKE, FAKE, 64, FAKE + 4096, FAKE, sb(4, 1),
          FAKE, 1 << 40, None]
    for i, v, code in ((0, None, -1),            # no host input
                       (14, None, -1),           # no host output
                       (15, None, -1),           # no stage
                       (15, FAKE + 8, -2),       # stage misaligned
                       (16, 64, -3),             # stage too small
                       (4, 16, -1),              # n_kv_heads
                       (2, None, -1),            # no start positions
                       (3, 64, -1),              # max_start_pos + 1 > s_max
                       (18, 16, -3)):            # workspace too small
        bad = list(ok)
        bad[i] = v
        assert d(*bad) == code, (i, v)
    f = lib.gqa_block_forward_host
    okf = [FAKE, 1, 8, 0, 32, FAKE, FAKE, FAKE, FAKE, FAKE, 64, FAKE, FAKE, 64, FAKE + 4096, FAKE, sb(1, 8),
           FAKE, 1 << 40, None]
    for i, v, code in ((0, None, -1), (16, 100, -3), (3, 60, -1), (4, 9, -1)):
        bad = list(okf)
        bad[i] = v
        assert f(*bad) == code, (i, v)
    assert lib.gqa_host_stage_release(None) == -1
    assert lib.gqa_host_stage_wait(None, None) == -1
