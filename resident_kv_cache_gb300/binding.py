"""Thin ctypes binding of librkv_attn.so: the C ABI's entry points under the same names.

Only argument marshalling happens here (tensor -> device pointer, current CUDA
stream, status -> exception).  All computation runs in the library's kernels;
there is no CPU path, and every function raises if the library is missing.

Tensor arguments may be torch tensors (their ``data_ptr()`` is passed) or raw
integer device addresses.  ``stream`` defaults to torch's current CUDA stream.
"""
from __future__ import annotations

import ctypes
import os
import re

from . import build as _build

LIB_PATH = _build.LIB
HEADER = os.path.join(_build.INCLUDE, "rkv_attn.h")

RKV_OK, RKV_ERR_INVALID_ARG, RKV_ERR_UNSUPPORTED, RKV_ERR_LAUNCH, RKV_ERR_DEVICE = range(5)
RKV_FLAG_WAIT_TIMEOUT, RKV_FLAG_LEN_CLAMPED, RKV_FLAG_NEGATIVE_INPUT, RKV_FLAG_BAD_POINTER = 0x1, 0x2, 0x4, 0x8
RKV_FLAG_BOUNDS = 0x10   # raised only by the checked build
RKV_DECODE_TICKET_BYTES = 32768   # head of a decode workspace: completion tickets

_lib = None


class RkvError(RuntimeError):
    """A non-OK status from the library."""

    def __init__(self, op: str, status: int, message: str):
        super().__init__(f"{op}: status {status} ({_status_name(status)}): {message}")
        self.op, self.status, self.message = op, status, message


def _status_name(s: int) -> str:
    return {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "launch", 4: "device"}.get(s, "?")


def declared_functions() -> list[str]:
    """Names of the functions include/rkv_attn.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(",
                                 text, flags=re.M)))


def load():
    """Load the built library (raises FileNotFoundError if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise FileNotFoundError(
            f"{LIB_PATH} is missing: build it with resident_kv_cache_gb300.build.build() "
            "(the attention path has no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.rkv_version.restype = I
    lib.rkv_version.argtypes = []
    lib.rkv_status_string.restype = ctypes.c_char_p
    lib.rkv_status_string.argtypes = [I]
    lib.rkv_last_error.restype = ctypes.c_char_p
    lib.rkv_last_error.argtypes = []
    lib.rkv_read_device_flags.restype = I
    lib.rkv_read_device_flags.argtypes = [ctypes.POINTER(ctypes.c_uint), I, P]
    lib.rkv_check_wait_timeout.restype = I
    lib.rkv_check_wait_timeout.argtypes = [ctypes.c_uint, P]
    lib.rkv_check_tf32_round.restype = I
    lib.rkv_check_tf32_round.argtypes = [P, P, P, I, P]
    lib.attn_prefill.restype = I
    lib.attn_prefill.argtypes = [P, P, P, P, I, I, I, I, I, I, P, F, P]
    lib.attn_prefill_fill_cache.restype = I
    lib.attn_prefill_fill_cache.argtypes = [P, P, P, P, I, I, I, I, I, I, F, P, P, I, P]
    lib.attn_prefill_chunked.restype = I
    lib.attn_prefill_chunked.argtypes = [P, P, P, P, I, I, I, I, I, I, I, P, P, F, P]
    lib.attn_decode_workspace_bytes.restype = SZ
    lib.attn_decode_workspace_bytes.argtypes = [I, I, I, I, I]
    lib.attn_decode_batched.restype = I
    lib.attn_decode_batched.argtypes = [P, P, P, P, I, I, I, I, I, P, F, P, SZ, P]
    lib.attn_decode_batched_noalloc.restype = I
    lib.attn_decode_batched_noalloc.argtypes = [P, P, P, P, I, I, I, I, I, P, F, P]
    lib.attn_decode_append.restype = I
    lib.attn_decode_append.argtypes = [P, P, P, P, P, P, I, I, I, I, I, P, F, P, SZ, P]
    lib.attn_decode_batched_ptrs.restype = I
    lib.attn_decode_batched_ptrs.argtypes = [P, P, P, P, I, I, I, I, I, P, F, P, SZ, P]
    lib.kv_cache_scatter_ptrs.restype = I
    lib.kv_cache_scatter_ptrs.argtypes = [P, P, P, P, I, I, I, I, I, P, P, P]
    lib.kv_append_rope.restype = I
    lib.kv_append_rope.argtypes = [P, P, P, P, P, I, I, I, I, I, I, P, I, F, P, P]
    lib.kv_cache_scatter.restype = I
    lib.kv_cache_scatter.argtypes = [P, P, P, P, I, I, I, I, I, P, P, P]
    _lib = lib
    return lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(op: str, status: int):
    if status != RKV_OK:
        raise RkvError(op, status, rkv_last_error())


def rkv_version() -> int:
    return load().rkv_version()


def rkv_status_string(status: int) -> str:
    return load().rkv_status_string(status).decode()


def rkv_last_error() -> str:
    return load().rkv_last_error().decode()


def rkv_read_device_flags(clear: bool = False, stream=None) -> int:
    """Device flag word (RKV_FLAG_*); synchronises the stream."""
    out = ctypes.c_uint(0)
    _check("rkv_read_device_flags", load().rkv_read_device_flags(ctypes.byref(out), int(clear),
                                                                  _stream(stream)))
    return out.value


def rkv_check_wait_timeout(limit_us: int, stream=None) -> None:
    """Run the bounded on-chip wait on a barrier nothing completes (gives up after limit_us)."""
    _check("rkv_check_wait_timeout", load().rkv_check_wait_timeout(int(limit_us), _stream(stream)))


def rkv_check_tf32_round(x, ours, ref, n, stream=None) -> None:
    """The prefill's operand rounding (ours) and the hardware cvt.rna.tf32.f32 (ref) of n f32 bit patterns."""
    _check("rkv_check_tf32_round", load().rkv_check_tf32_round(_ptr(x), _ptr(ours), _ptr(ref), int(n),
                                                               _stream(stream)))


def attn_prefill(q, k, v, o, batch, seq_len, n_heads, n_kv_heads, head_dim, causal,
                 seq_lens=None, scale=0.0, stream=None):
    _check("attn_prefill", load().attn_prefill(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), batch, seq_len, n_heads, n_kv_heads, head_dim,
        int(bool(causal)), _ptr(seq_lens), float(scale), _stream(stream)))


def attn_prefill_fill_cache(q, k, v, o, batch, seq_len, n_heads, n_kv_heads, head_dim, causal, k_cache, v_cache,
                            max_len, scale=0.0, stream=None):
    _check("attn_prefill_fill_cache", load().attn_prefill_fill_cache(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), batch, seq_len, n_heads, n_kv_heads, head_dim, int(bool(causal)),
        float(scale), _ptr(k_cache), _ptr(v_cache), max_len, _stream(stream)))


def attn_prefill_chunked(q, k_cache, v_cache, o, M, T, n_heads, n_kv_heads, head_dim, max_len, causal,
                         start_pos, q_lens=None, scale=0.0, stream=None):
    _check("attn_prefill_chunked", load().attn_prefill_chunked(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o), M, T, n_heads, n_kv_heads, head_dim, max_len,
        int(bool(causal)), _ptr(start_pos), _ptr(q_lens), float(scale), _stream(stream)))


def attn_decode_workspace_bytes(M, n_heads, n_kv_heads, head_dim, max_len) -> int:
    return int(load().attn_decode_workspace_bytes(M, n_heads, n_kv_heads, head_dim, max_len))


def attn_decode_batched(q, k_cache, v_cache, o, M, n_heads, n_kv_heads, head_dim, max_len, seq_lens,
                        scale, workspace, workspace_bytes, stream=None):
    _check("attn_decode_batched", load().attn_decode_batched(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o), M, n_heads, n_kv_heads, head_dim, max_len,
        _ptr(seq_lens), float(scale), _ptr(workspace), int(workspace_bytes), _stream(stream)))


def attn_decode_batched_noalloc(q, k_cache, v_cache, o, M, n_heads, n_kv_heads, head_dim, max_len,
                                seq_lens, scale, stream=None):
    """attn_decode_batched with the library's built-in scratch instead of a caller workspace."""
    _check("attn_decode_batched_noalloc", load().attn_decode_batched_noalloc(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o), M, n_heads, n_kv_heads, head_dim, max_len,
        _ptr(seq_lens), float(scale), _stream(stream)))


def kv_cache_scatter(k_new, v_new, k_cache, v_cache, M, T, n_kv_heads, head_dim, max_len, start_pos,
                     overflow=None, stream=None):
    _check("kv_cache_scatter", load().kv_cache_scatter(
        _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), M, T, n_kv_heads, head_dim, max_len,
        _ptr(start_pos), _ptr(overflow), _stream(stream)))


def kv_append_rope(q, k_new, v_new, k_cache, v_cache, M, T, n_heads, n_kv_heads, head_dim, max_len, start_pos,
                   rotary_ndims=None, theta=10000.0, overflow=None, stream=None):
    """RoPE (GPT-NeoX half-split) of q and k_new in place at start_pos + t, then K/V into the cache."""
    _check("kv_append_rope", load().kv_append_rope(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), M, T, n_heads, n_kv_heads, head_dim,
        max_len, _ptr(start_pos), head_dim if rotary_ndims is None else int(rotary_ndims), float(theta),
        _ptr(overflow), _stream(stream)))


def attn_decode_batched_ptrs(q, k_ptrs, v_ptrs, o, M, n_heads, n_kv_heads, head_dim, max_len, seq_lens, scale,
                             workspace, workspace_bytes, stream=None):
    """attn_decode_batched with per-sequence caches: k_ptrs / v_ptrs are device int64 arrays of M addresses."""
    _check("attn_decode_batched_ptrs", load().attn_decode_batched_ptrs(
        _ptr(q), _ptr(k_ptrs), _ptr(v_ptrs), _ptr(o), M, n_heads, n_kv_heads, head_dim, max_len, _ptr(seq_lens),
        float(scale), _ptr(workspace), int(workspace_bytes), _stream(stream)))


def kv_cache_scatter_ptrs(k_new, v_new, k_ptrs, v_ptrs, M, T, n_kv_heads, head_dim, max_len, start_pos,
                          overflow=None, stream=None):
    """kv_cache_scatter into per-sequence caches (device int64 arrays of M addresses)."""
    _check("kv_cache_scatter_ptrs", load().kv_cache_scatter_ptrs(
        _ptr(k_new), _ptr(v_new), _ptr(k_ptrs), _ptr(v_ptrs), M, T, n_kv_heads, head_dim, max_len,
        _ptr(start_pos), _ptr(overflow), _stream(stream)))


def attn_decode_append(q, k_new, v_new, k_cache, v_cache, o, M, n_heads, n_kv_heads, head_dim, max_len, seq_lens,
                       scale, workspace, workspace_bytes, stream=None):
    """One decode step: append the new rows at seq_lens-1, then decode (one launch)."""
    _check("attn_decode_append", load().attn_decode_append(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(o), M, n_heads, n_kv_heads, head_dim,
        max_len, _ptr(seq_lens), float(scale), _ptr(workspace), int(workspace_bytes), _stream(stream)))
