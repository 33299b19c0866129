"""The Python binding checks its arguments before it calls into the library
(no device is touched for a bad call), and fails loudly rather than falling
back when something is wrong."""
import pytest
import torch

import grouped_query_attention_gemv_gb300 as G


def _cpu_block(B=2, T=1, n_kv=8):
    bf = torch.bfloat16
    return dict(x=torch.zeros(B, T, 4096, dtype=bf), wq=torch.zeros(4096, 4096, dtype=bf),
                wk=torch.zeros(n_kv * 128, 4096, dtype=bf), wv=torch.zeros(n_kv * 128, 4096, dtype=bf),
                wo=torch.zeros(4096, 4096, dtype=bf), rope=torch.zeros(16, 64, 2),
                ck=torch.zeros(B, 16, n_kv, 128, dtype=bf), cv=torch.zeros(B, 16, n_kv, 128, dtype=bf))


def test_host_tensors_are_refused_by_the_device_entries():
    a = _cpu_block()
    with pytest.raises(ValueError, match="CUDA tensor"):
        G.block_forward(a["x"], 0, a["wq"], a["wk"], a["wv"], a["wo"], a["rope"], a["ck"], a["cv"])


def test_kv_head_count_is_checked():
    a = _cpu_block()
    with pytest.raises(ValueError, match="n_kv_heads"):
        G._weight_args(2, a["wq"], a["wk"], a["wv"], a["wo"], a["rope"], a["ck"], a["cv"], 16)


def test_host_buffer_entry_checks_its_host_tensors():
    a = _cpu_block()
    sp = torch.zeros(2, dtype=torch.int32)
    with pytest.raises(ValueError, match="x_host"):
        G.decode_host(a["x"].float(), sp, 4, a["wq"], a["wk"], a["wv"], a["wo"], a["rope"], a["ck"], a["cv"])
    with pytest.raises(ValueError, match="out_host"):
        G.decode_host(a["x"], sp, 4, a["wq"], a["wk"], a["wv"], a["wo"], a["rope"], a["ck"], a["cv"],
                      out_host=torch.zeros(1, 1, 4096, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="CUDA tensor"):   # the weights must be on the device
        G.decode_host(a["x"], sp, 4, a["wq"], a["wk"], a["wv"], a["wo"], a["rope"], a["ck"], a["cv"],
                      out_host=torch.zeros(2, 1, 4096, dtype=torch.bfloat16))


def test_shapes_are_checked():
    a = _cpu_block()
    with pytest.raises(ValueError):
        G._weight_args(2, a["wq"], a["wk"][:512], a["wv"], a["wo"], a["rope"], a["ck"], a["cv"], 8)
