"""GB300 grouped-query attention block (Llama 3.1 8B) — Python binding.

A thin ctypes layer over the C ABI in ``include/gqa.h`` (``lib/libgqa.so``,
built in-tree by ``python -m grouped_query_attention_gemv_gb300.build``).
It only checks and marshals arguments: every step of the block runs in the
library's CUDA kernels. PyTorch supplies device memory and streams.

Functions mirror the C entry points: ``block_forward`` / ``decode`` /
``prefill`` (``n_kv_heads`` 8, or 32 for the multi-head variant), the layer
entries ``layer_forward`` / ``layer_decode`` / ``rms_norm``, the host-buffer
entries ``block_forward_host`` / ``decode_host`` (with ``make_host_stage``,
``host_stage_wait``, ``release_host_stage``), ``decode_static``,
``rope_table``, ``workspace_bytes``, ``device_status``, ``last_launch_count``.
If the library has not been built every call raises ``ImportError``; there is
no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

import torch

__all__ = [
    "GQAError", "D_MODEL", "N_HEADS", "N_KV_HEADS", "HEAD_DIM", "library_path", "lib",
    "exported_symbols", "workspace_bytes", "make_workspace", "rope_table", "block_forward",
    "decode", "prefill", "device_status", "last_launch_count", "set_profile_events",
    "set_decode_fusion", "set_decode_attention_split", "set_wait_limit_ns", "decode_static", "rms_norm", "layer_forward", "layer_decode", "static_device_status",
    "STATIC_SCRATCH_BYTES", "make_host_stage", "default_host_stage", "host_stage_wait", "release_host_stage",
    "decode_host",
    "block_forward_host",
]

D_MODEL, N_HEADS, N_KV_HEADS, HEAD_DIM = 4096, 32, 8, 128
STATIC_SCRATCH_BYTES = 16 << 20
_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "lib", "libgqa.so")
_HEADER = os.path.join(os.path.dirname(_PKG), "include", "gqa.h")

_vp, _i, _sz, _d = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_double
_SIGNATURES = {
    "gqa_workspace_bytes": (_sz, [_i, _i, _i]),
    "gqa_workspace_init": (_i, [_vp, _sz, _vp]),
    "gqa_device_status": (_i, [_vp, ctypes.POINTER(_i), _i]),
    "gqa_rope_table": (_i, [_vp, _i, _d, _i, _d, _d, _d, _d, _vp]),
    "gqa_block_forward": (_i, [_vp, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _i, _vp, _vp, _i, _vp, _vp, _sz, _vp]),
    "gqa_prefill": (_i, [_vp, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _i, _vp, _vp, _i, _vp, _vp, _sz, _vp]),
    "gqa_decode": (_i, [_vp, _i, _vp, _i, _vp, _vp, _vp, _vp, _vp, _i, _vp, _vp, _i, _vp, _vp, _sz, _vp]),
    "gqa_block_forward_nkv": (_i, [_vp, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _i, _vp, _vp, _i, _vp, _vp, _sz,
                                   _vp]),
    "gqa_decode_nkv": (_i, [_vp, _i, _vp, _i, _i, _vp, _vp, _vp, _vp, _vp, _i, _vp, _vp, _i, _vp, _vp, _sz, _vp]),
    "gqa_rms_norm": (_i, [_vp, _i, _vp, ctypes.c_float, _vp, _vp]),
    "gqa_layer_forward": (_i, [_vp, _i, _i, _i, _vp, ctypes.c_float, _vp, _vp, _vp, _vp, _vp, _i, _vp, _vp, _i, _vp,
                               _vp, _sz, _vp]),
    "gqa_layer_decode": (_i, [_vp, _i, _vp, _i, _vp, ctypes.c_float, _vp, _vp, _vp, _vp, _vp, _i, _vp, _vp, _i, _vp,
                              _vp, _sz, _vp]),
    "gqa_host_stage_bytes": (_sz, [_i, _i]),
    "gqa_block_forward_host": (_i, [_vp, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _i, _vp, _vp, _i, _vp, _vp, _sz,
                                    _vp, _sz, _vp]),
    "gqa_decode_host": (_i, [_vp, _i, _vp, _i, _i, _vp, _vp, _vp, _vp, _vp, _i, _vp, _vp, _i, _vp, _vp, _sz, _vp,
                             _sz, _vp]),
    "gqa_host_stage_wait": (_i, [_vp, _vp]),
    "gqa_host_stage_release": (_i, [_vp]),
    "gqa_strerror": (ctypes.c_char_p, [_i]),
    "gqa_last_launch_count": (_i, []),
    "gqa_set_decode_fusion": (_i, [_i]),
    "gqa_set_decode_attention_split": (_i, [_i]),
    "gqa_set_wait_limit_ns": (ctypes.c_ulonglong, [ctypes.c_ulonglong]),
    "gqa_set_profile_events": (_i, [ctypes.POINTER(_vp), _i]),
    "gqa_decode_static": (_i, [_vp, _i, _vp, _i, _vp, _vp, _vp, _vp, _vp, _i, _vp, _vp, _i, _vp, _vp]),
    "gqa_static_device_status": (_i, [ctypes.POINTER(_i), _i]),
}


class GQAError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = lib().gqa_strerror(status).decode()
        super().__init__(f"{where}: {msg} (status {status})")
        self.status = status


_lib = None


def library_path() -> str:
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    """The loaded libgqa; raises ImportError when it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise ImportError(f"libgqa.so is not built ({_LIB_PATH}); run "
                              "`python -m grouped_query_attention_gemv_gb300.build`")
        handle = ctypes.CDLL(_LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def exported_symbols():
    """Names of the functions declared in include/gqa.h."""
    text = open(_HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w]+\s*\*?\s*(gqa_\w+)\s*\(", text, re.M)))


def _p(t: Optional[torch.Tensor]):
    # a plain int: ctypes passes it as the void* the signature declares
    return None if t is None else t.data_ptr()


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _s(stream, device=None):
    """The CUDA stream handle: ``stream`` or, when None, torch's current
    stream on ``device`` (the raw handle lookup is a few times cheaper than
    building a Stream object on every call)."""
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None and device is not None and device.index is not None:
        return _raw_stream(device.index)
    return torch.cuda.current_stream().cuda_stream


def _check(t: torch.Tensor, name: str, dtype, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not (t.is_cuda and t.dtype == dtype and t.is_contiguous()):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if t.dtype != dtype:
            raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and t.shape != shape:
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def workspace_bytes(B: int, T: int, max_keys: int) -> int:
    return int(lib().gqa_workspace_bytes(B, T, max_keys))


def make_workspace(B: int, T: int, max_keys: int, device=None) -> torch.Tensor:
    """A zero-filled uint8 workspace sized for (B, T, max_keys)."""
    n = workspace_bytes(B, T, max_keys)
    if n == 0:
        raise ValueError(f"invalid workspace request B={B} T={T} max_keys={max_keys}")
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def rope_table(rows: int, theta: float = 500000.0, scaled: bool = True, factor: float = 8.0,
               low_freq_factor: float = 1.0, high_freq_factor: float = 4.0,
               original_context: float = 8192.0, device=None, stream=None) -> torch.Tensor:
    """fp32 [rows, 64, 2] table of (cos, sin), built on the device."""
    out = torch.empty(rows, 64, 2, dtype=torch.float32, device=device or "cuda")
    r = lib().gqa_rope_table(_p(out), rows, theta, int(scaled), factor, low_freq_factor,
                             high_freq_factor, original_context, _s(stream, out.device))
    if r:
        raise GQAError(r, "gqa_rope_table")
    return out


def _block_args(x, wq, wk, wv, wo, rope, cache_k, cache_v, out, T, n_kv=N_KV_HEADS):
    B = x.shape[0]
    _check(x, "x", torch.bfloat16, (B, T, D_MODEL))
    _weight_args(B, wq, wk, wv, wo, rope, cache_k, cache_v, n_kv)
    if out is None:
        out = torch.empty_like(x)
    _check(out, "out", torch.bfloat16, (B, T, D_MODEL))
    return B, out


def _weight_args(B, wq, wk, wv, wo, rope, cache_k, cache_v, n_kv):
    if n_kv not in (N_KV_HEADS, N_HEADS):
        raise ValueError(f"n_kv_heads must be {N_KV_HEADS} or {N_HEADS}, got {n_kv}")
    _check(wq, "wq", torch.bfloat16, (N_HEADS * HEAD_DIM, D_MODEL))
    _check(wk, "wk", torch.bfloat16, (n_kv * HEAD_DIM, D_MODEL))
    _check(wv, "wv", torch.bfloat16, (n_kv * HEAD_DIM, D_MODEL))
    _check(wo, "wo", torch.bfloat16, (D_MODEL, N_HEADS * HEAD_DIM))
    _check(rope, "rope", torch.float32)
    if rope.dim() != 3 or rope.shape[1:] != (64, 2):
        raise ValueError("rope must be [rows, 64, 2]")
    _check(cache_k, "cache_k", torch.bfloat16)
    _check(cache_v, "cache_v", torch.bfloat16, cache_k.shape)
    if cache_k.dim() != 4 or cache_k.shape[0] != B or cache_k.shape[2:] != (n_kv, HEAD_DIM):
        raise ValueError(f"cache must be [B, S_max, {n_kv}, 128], got {tuple(cache_k.shape)}")


def _ws(workspace, B, T, max_keys, device):
    if workspace is None:
        workspace = make_workspace(B, T, max_keys, device)
    _check(workspace, "workspace", torch.uint8)
    return workspace


def block_forward(x, start_pos: int, wq, wk, wv, wo, rope, cache_k, cache_v, out=None,
                  workspace=None, stream=None, n_kv_heads: int = N_KV_HEADS) -> torch.Tensor:
    """delta_attn for x [B, T, 4096] after ``start_pos`` cached rows; updates the cache.
    ``n_kv_heads`` 32 is the multi-head variant (wk, wv [4096, 4096], cache [B, S, 32, 128])."""
    T = x.shape[1]
    B, out = _block_args(x, wq, wk, wv, wo, rope, cache_k, cache_v, out, T, n_kv_heads)
    workspace = _ws(workspace, B, T, start_pos + T, x.device)
    if n_kv_heads == N_KV_HEADS:
        r = lib().gqa_block_forward(_p(x), B, T, int(start_pos), _p(wq), _p(wk), _p(wv), _p(wo), _p(rope),
                                    rope.shape[0], _p(cache_k), _p(cache_v), cache_k.shape[1], _p(out),
                                    _p(workspace), workspace.numel(), _s(stream, x.device))
        where = "gqa_block_forward"
    else:
        r = lib().gqa_block_forward_nkv(_p(x), B, T, int(start_pos), int(n_kv_heads), _p(wq), _p(wk), _p(wv),
                                        _p(wo), _p(rope), rope.shape[0], _p(cache_k), _p(cache_v), cache_k.shape[1],
                                        _p(out), _p(workspace), workspace.numel(), _s(stream, x.device))
        where = "gqa_block_forward_nkv"
    if r:
        raise GQAError(r, where)
    return out


def prefill(x, start_pos: int, wq, wk, wv, wo, rope, cache_k, cache_v, out=None, workspace=None,
            stream=None) -> torch.Tensor:
    T = x.shape[1]
    B, out = _block_args(x, wq, wk, wv, wo, rope, cache_k, cache_v, out, T)
    workspace = _ws(workspace, B, T, start_pos + T, x.device)
    r = lib().gqa_prefill(_p(x), B, T, int(start_pos), _p(wq), _p(wk), _p(wv), _p(wo), _p(rope),
                          rope.shape[0], _p(cache_k), _p(cache_v), cache_k.shape[1], _p(out),
                          _p(workspace), workspace.numel(), _s(stream, x.device))
    if r:
        raise GQAError(r, "gqa_prefill")
    return out


def decode(x, start_pos: torch.Tensor, max_start_pos: int, wq, wk, wv, wo, rope, cache_k, cache_v,
           out=None, workspace=None, stream=None, n_kv_heads: int = N_KV_HEADS) -> torch.Tensor:
    """One decode step; ``start_pos`` is a device int32 [B] of cached rows per sequence.
    ``n_kv_heads`` as in ``block_forward``."""
    B, out = _block_args(x, wq, wk, wv, wo, rope, cache_k, cache_v, out, 1, n_kv_heads)
    _check(start_pos, "start_pos", torch.int32, (B,))
    workspace = _ws(workspace, B, 1, max_start_pos + 1, x.device)
    if n_kv_heads == N_KV_HEADS:
        r = lib().gqa_decode(_p(x), B, _p(start_pos), int(max_start_pos), _p(wq), _p(wk), _p(wv), _p(wo),
                             _p(rope), rope.shape[0], _p(cache_k), _p(cache_v), cache_k.shape[1], _p(out),
                             _p(workspace), workspace.numel(), _s(stream, x.device))
        where = "gqa_decode"
    else:
        r = lib().gqa_decode_nkv(_p(x), B, _p(start_pos), int(max_start_pos), int(n_kv_heads), _p(wq), _p(wk),
                                 _p(wv), _p(wo), _p(rope), rope.shape[0], _p(cache_k), _p(cache_v), cache_k.shape[1],
                                 _p(out), _p(workspace), workspace.numel(), _s(stream, x.device))
        where = "gqa_decode_nkv"
    if r:
        raise GQAError(r, where)
    return out


def rms_norm(x, norm_w, eps: float, out=None, stream=None) -> torch.Tensor:
    """attention_norm of rows of 4096 features (bf16 in and out)."""
    _check(x, "x", torch.bfloat16)
    _check(norm_w, "norm_w", torch.bfloat16, (4096,))
    if x.shape[-1] != 4096:
        raise ValueError("x: last dimension must be 4096")
    out = torch.empty_like(x) if out is None else out
    _check(out, "out", torch.bfloat16, tuple(x.shape))
    r = lib().gqa_rms_norm(_p(x), x.numel() // 4096, _p(norm_w), float(eps), _p(out), _s(stream, x.device))
    if r:
        raise GQAError(r, "gqa_rms_norm")
    return out


def layer_forward(x, start_pos: int, norm_w, eps: float, wq, wk, wv, wo, rope, cache_k, cache_v, out=None,
                  workspace=None, stream=None) -> torch.Tensor:
    """h = x + attention(RMSNorm(x)) for B sequences of T tokens after ``start_pos`` cached rows."""
    B, out = _block_args(x, wq, wk, wv, wo, rope, cache_k, cache_v, out, x.shape[1])
    _check(norm_w, "norm_w", torch.bfloat16, (4096,))
    workspace = _ws(workspace, B, x.shape[1], int(start_pos) + x.shape[1], x.device)
    r = lib().gqa_layer_forward(_p(x), B, x.shape[1], int(start_pos), _p(norm_w), float(eps), _p(wq), _p(wk),
                                _p(wv), _p(wo), _p(rope), rope.shape[0], _p(cache_k), _p(cache_v), cache_k.shape[1],
                                _p(out), _p(workspace), workspace.numel(), _s(stream, x.device))
    if r:
        raise GQAError(r, "gqa_layer_forward")
    return out


def layer_decode(x, start_pos: torch.Tensor, max_start_pos: int, norm_w, eps: float, wq, wk, wv, wo, rope,
                 cache_k, cache_v, out=None, workspace=None, stream=None) -> torch.Tensor:
    """One decode step of h = x + attention(RMSNorm(x)); ``start_pos`` as in ``decode``."""
    B, out = _block_args(x, wq, wk, wv, wo, rope, cache_k, cache_v, out, 1)
    _check(start_pos, "start_pos", torch.int32, (B,))
    _check(norm_w, "norm_w", torch.bfloat16, (4096,))
    workspace = _ws(workspace, B, 1, max_start_pos + 1, x.device)
    r = lib().gqa_layer_decode(_p(x), B, _p(start_pos), int(max_start_pos), _p(norm_w), float(eps), _p(wq),
                               _p(wk), _p(wv), _p(wo), _p(rope), rope.shape[0], _p(cache_k), _p(cache_v),
                               cache_k.shape[1], _p(out), _p(workspace), workspace.numel(), _s(stream, x.device))
    if r:
        raise GQAError(r, "gqa_layer_decode")
    return out


def device_status(workspace: torch.Tensor, clear: bool = False) -> int:
    """Synchronise and return the workspace status word (0 = no device error)."""
    st = ctypes.c_int(0)
    r = lib().gqa_device_status(_p(workspace), ctypes.byref(st), int(clear))
    if r not in (0, -5):
        raise GQAError(r, "gqa_device_status")
    return st.value


def last_launch_count() -> int:
    return int(lib().gqa_last_launch_count())


def set_decode_fusion(enable: bool) -> bool:
    """Run decode steps of at most 64 sequences on this thread as one fused
    persistent kernel (True, the default) or as three kernels (False).
    Returns the previous setting."""
    return bool(lib().gqa_set_decode_fusion(1 if enable else 0))


def set_wait_limit_ns(ns: int) -> int:
    """Limit (ns) of the decode kernels' grid-wide waits on this thread; 0
    restores the default (2 s). Returns the previous limit."""
    if ns < 0:
        raise ValueError("the wait limit is a non-negative number of nanoseconds")
    return int(lib().gqa_set_wait_limit_ns(int(ns)))


_SPLITS = {"auto": 0, "position": 1, "head": 2}


def set_decode_attention_split(mode: str) -> str:
    """How the one-kernel decode step splits its attention on this thread:
    "auto" (chosen per call, the default), "position" (16-position units over
    the grid, split sequences merged) or "head" (one (sequence, KV head) pair
    per CTA where the batch fits, nothing merged). Returns the previous mode."""
    if mode not in _SPLITS:
        raise ValueError(f"split must be one of {sorted(_SPLITS)}, not {mode!r}")
    prev = lib().gqa_set_decode_attention_split(_SPLITS[mode])
    return {v: k for k, v in _SPLITS.items()}[prev]


_prof_keep = None


def set_profile_events(events) -> None:
    """Record ``events[0]`` before and ``events[i]`` after kernel i of every
    following call on this thread (torch.cuda.Event objects with timing);
    ``None`` stops it."""
    global _prof_keep
    if not events:
        _prof_keep = None
        lib().gqa_set_profile_events(None, 0)
        return
    arr = (_vp * len(events))(*[e.cuda_event for e in events])
    _prof_keep = (arr, events)
    r = lib().gqa_set_profile_events(arr, len(events))
    if r:
        raise GQAError(r, "gqa_set_profile_events")


def decode_static(x, start_pos: torch.Tensor, max_start_pos: int, wq, wk, wv, wo, rope, cache_k, cache_v,
                  out=None, stream=None) -> torch.Tensor:
    """``decode`` without a workspace: the library's own static device scratch
    (``STATIC_SCRATCH_BYTES``) is used, so nothing is allocated for scratch.
    For callers that must not allocate device memory per step. Calls share
    that scratch: do not overlap them on the GPU."""
    B, out = _block_args(x, wq, wk, wv, wo, rope, cache_k, cache_v, out, 1)
    _check(start_pos, "start_pos", torch.int32, (B,))
    r = lib().gqa_decode_static(_p(x), B, _p(start_pos), int(max_start_pos), _p(wq), _p(wk), _p(wv), _p(wo),
                                _p(rope), rope.shape[0], _p(cache_k), _p(cache_v), cache_k.shape[1], _p(out),
                                _s(stream, x.device))
    if r:
        raise GQAError(r, "gqa_decode_static")
    return out


def static_device_status(clear: bool = False) -> int:
    """Status word of the static scratch on the current device (synchronises)."""
    st = ctypes.c_int(0)
    r = lib().gqa_static_device_status(ctypes.byref(st), int(clear))
    if r not in (0, -5):
        raise GQAError(r, "gqa_static_device_status")
    return st.value


# ------------------------------------------------------------ host-buffer entries

def make_host_stage(B: int, T: int, device=None) -> torch.Tensor:
    """Device stage of the host-buffer entries (two input and two output buffers)."""
    n = int(lib().gqa_host_stage_bytes(B, T))
    if n == 0:
        raise ValueError(f"invalid stage request B={B} T={T}")
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


_default_stages = {}
_MAX_DEFAULT_STAGES = 8


def _default_stage(B: int, T: int, device) -> torch.Tensor:
    """One stage per (device, B, T), kept for the calls that pass none (the
    library keeps copy streams per stage: a fresh stage per call would make
    new ones every time)."""
    d = torch.device(device)
    index = d.index if d.index is not None else torch.cuda.current_device()
    key = (index, B, T)
    st = _default_stages.get(key)
    if st is None:
        if len(_default_stages) >= _MAX_DEFAULT_STAGES:   # drop the oldest shape's stage
            old_key = next(iter(_default_stages))
            with torch.cuda.device(old_key[0]):
                stage = _default_stages.pop(old_key)
                r = lib().gqa_host_stage_release(_p(stage))
                if r not in (0, -1):          # -1: no call ever ran on it
                    raise GQAError(r, "gqa_host_stage_release")
        st = _default_stages[key] = make_host_stage(B, T, torch.device("cuda", index))
    return st


def default_host_stage(B: int, T: int, device=None) -> torch.Tensor:
    """The stage the host-buffer calls of this device and shape use when they
    are given none."""
    return _default_stage(B, T, device or "cuda")


def host_stage_wait(stage: torch.Tensor, stream=None) -> None:
    """Order ``stream`` after the read-backs of every call made on ``stage``:
    their results are in host memory once ``stream`` reaches this point."""
    r = lib().gqa_host_stage_wait(_p(stage), _s(stream, stage.device))
    if r:
        raise GQAError(r, "gqa_host_stage_wait")


def release_host_stage(stage: torch.Tensor) -> None:
    """Free the copy stream and events the library keeps for ``stage``."""
    r = lib().gqa_host_stage_release(_p(stage))
    if r:
        raise GQAError(r, "gqa_host_stage_release")


def _host_args(x_host, out_host, T):
    if not isinstance(x_host, torch.Tensor) or x_host.is_cuda:
        raise ValueError("x_host must be a CPU tensor")
    B = x_host.shape[0]
    if x_host.dtype != torch.bfloat16 or not x_host.is_contiguous() or x_host.shape != (B, T, D_MODEL):
        raise ValueError(f"x_host must be a contiguous bf16 [B, {T}, {D_MODEL}] tensor")
    if out_host is None:
        out_host = torch.empty(x_host.shape, dtype=torch.bfloat16).pin_memory()
    if out_host.is_cuda or out_host.dtype != torch.bfloat16 or not out_host.is_contiguous() \
            or out_host.shape != x_host.shape:
        raise ValueError("out_host must be a contiguous bf16 CPU tensor shaped like x_host")
    return B, out_host


def decode_host(x_host, start_pos: torch.Tensor, max_start_pos: int, wq, wk, wv, wo, rope, cache_k, cache_v,
                out_host=None, stage=None, workspace=None, stream=None, n_kv_heads: int = N_KV_HEADS) -> torch.Tensor:
    """``decode`` with x and the result in host memory (pinned for asynchronous
    copies); out_host holds the result once ``stream`` has reached a later
    ``host_stage_wait(stage)`` (with ``stage=None``: the default stage of this
    device and shape, ``host_stage_wait(default_host_stage(B, 1, device))``)."""
    B, out_host = _host_args(x_host, out_host, 1)
    _weight_args(B, wq, wk, wv, wo, rope, cache_k, cache_v, n_kv_heads)
    dev = start_pos.device
    _check(start_pos, "start_pos", torch.int32, (B,))
    workspace = _ws(workspace, B, 1, max_start_pos + 1, dev)
    stage = _default_stage(B, 1, dev) if stage is None else stage
    r = lib().gqa_decode_host(x_host.data_ptr(), B, _p(start_pos), int(max_start_pos), int(n_kv_heads), _p(wq),
                              _p(wk), _p(wv), _p(wo), _p(rope), rope.shape[0], _p(cache_k), _p(cache_v),
                              cache_k.shape[1], out_host.data_ptr(), _p(stage), stage.numel(), _p(workspace),
                              workspace.numel(), _s(stream, dev))
    if r:
        raise GQAError(r, "gqa_decode_host")
    return out_host


def block_forward_host(x_host, start_pos: int, wq, wk, wv, wo, rope, cache_k, cache_v, out_host=None, stage=None,
                       workspace=None, stream=None, n_kv_heads: int = N_KV_HEADS) -> torch.Tensor:
    """``block_forward`` with x and delta_attn in host memory."""
    T = x_host.shape[1]
    B, out_host = _host_args(x_host, out_host, T)
    _weight_args(B, wq, wk, wv, wo, rope, cache_k, cache_v, n_kv_heads)
    dev = wq.device
    workspace = _ws(workspace, B, T, start_pos + T, dev)
    stage = _default_stage(B, T, dev) if stage is None else stage
    r = lib().gqa_block_forward_host(x_host.data_ptr(), B, T, int(start_pos), int(n_kv_heads), _p(wq), _p(wk),
                                     _p(wv), _p(wo), _p(rope), rope.shape[0], _p(cache_k), _p(cache_v),
                                     cache_k.shape[1], out_host.data_ptr(), _p(stage), stage.numel(), _p(workspace),
                                     workspace.numel(), _s(stream, dev))
    if r:
        raise GQAError(r, "gqa_block_forward_host")
    return out_host
