"""CPU oracle for resident attention (prefill, batched decode, KV scatter).

TEST INFRASTRUCTURE ONLY.  The library never imports this package; only the
tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` use
it.  The arithmetic lives in ``rkv_oracle.c`` (plain C, f64 accumulation,
two-pass softmax); this module only builds it with gcc and marshals numpy
arrays through ctypes.  It shares no code with the CUDA library.

Page citations are in the C file's header; the functions here follow it:
  prefill  -- trustformers-core attention.rs, fn attention_prefill_gpu_to_gpu
              (causal from-empty-cache mask) and trueno-gpu attention.rs,
              fn batched_multihead_attention (non-causal, scale 1/sqrt(d)).
  decode   -- trustformers-core attention.rs, fn attention_decode_gpu_to_gpu;
              cache layout from realizar cache_from_cache_from_kv_cache.rs,
              fn init_batched_kv_cache_gpu.
  scatter  -- trueno-gpu attention.rs, fn kv_cache_scatter_gpu.
  rope     -- GPT-NeoX half-split rotary embedding at explicit positions:
              trustformers-core attention.rs, fn rope_neox_gpu_to_gpu and
              realizar cache_from_cache_from_kv_cache.rs, fn apply_rope_to_buffer.
  prefill_cached -- a prefill appended behind an existing cache, which
              trustformers-core attention.rs, fn attention_prefill_gpu_to_gpu
              says must run the decode path once per token: query i of the
              chunk sees cache rows 0..start_pos+i.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rkv_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "librkv_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-fopenmp) into oracle/_build/."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        _lib = _configure(ctypes.CDLL(build()))
    return _lib


@contextlib.contextmanager
def using_library(lib_path: str):
    """Test hook: run this module's wrappers against another build of the oracle
    (the mutation tests compile copies with planted mistakes)."""
    global _lib
    saved = _lib
    _lib = _configure(ctypes.CDLL(lib_path))
    try:
        yield
    finally:
        _lib = saved


def _configure(lib):
    P = ctypes.c_void_p
    I = ctypes.c_int
    D = ctypes.c_double
    L = ctypes.c_int64
    lib.rkv_oracle_prefill.argtypes = [P, P, P, P, I, I, I, I, I, I, P, D]
    lib.rkv_oracle_prefill_rows.argtypes = [P, P, P, I, I, I, I, I, I, P, D, P, L, P]
    lib.rkv_oracle_prefill_probs.argtypes = [P, P, P, I, I, I, I, I, I, P, D, I, I, I, P]
    lib.rkv_oracle_decode.argtypes = [P, P, P, P, I, I, I, I, I, P, D]
    lib.rkv_oracle_scatter.argtypes = [P, P, P, P, I, I, I, I, I, P, P]
    lib.rkv_oracle_prefill_cached.argtypes = [P, P, P, P, I, I, I, I, I, I, I, P, P, D]
    lib.rkv_oracle_rope.argtypes = [P, P, L, I, I, I, P, D]
    for f in ("rkv_oracle_prefill", "rkv_oracle_prefill_rows", "rkv_oracle_prefill_probs",
              "rkv_oracle_decode", "rkv_oracle_scatter", "rkv_oracle_num_threads",
              "rkv_oracle_prefill_cached", "rkv_oracle_rope"):
        getattr(lib, f).restype = ctypes.c_int
    return lib


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _i32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.int32)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def default_scale(head_dim: int) -> float:
    """1/sqrt(head_dim): trueno-gpu attention.rs, fn batched_multihead_attention."""
    return 1.0 / float(np.sqrt(head_dim))


def num_threads() -> int:
    return int(_load().rkv_oracle_num_threads())


def prefill(q, k, v, B, S, H, Hk, D, causal, seq_lens=None, scale=None):
    """O[B, S, H*D] (float64) for interleaved Q [B,S,H*D], K/V [B,S,Hk*D]."""
    q, k, v = _f32(q), _f32(k), _f32(v)
    assert q.size == B * S * H * D and k.size == B * S * Hk * D and v.size == k.size
    sl = _i32(seq_lens)
    o = np.zeros((B, S, H * D), dtype=np.float64)
    rc = _load().rkv_oracle_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(o), B, S, H, Hk, D,
                                    int(bool(causal)), _ptr(sl),
                                    default_scale(D) if scale is None else float(scale))
    if rc != 0:
        raise ValueError("oracle prefill rejected its arguments")
    return o


def prefill_rows(q, k, v, B, S, H, Hk, D, causal, rows, seq_lens=None, scale=None):
    """Output rows for flat ids rows[n] = (b*H + h)*S + i; returns [n, D] float64."""
    q, k, v = _f32(q), _f32(k), _f32(v)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    sl = _i32(seq_lens)
    out = np.zeros((rows.size, D), dtype=np.float64)
    rc = _load().rkv_oracle_prefill_rows(_ptr(q), _ptr(k), _ptr(v), B, S, H, Hk, D,
                                         int(bool(causal)), _ptr(sl),
                                         default_scale(D) if scale is None else float(scale),
                                         _ptr(rows), rows.size, _ptr(out))
    if rc != 0:
        raise ValueError("oracle prefill_rows rejected its arguments")
    return out


def prefill_probs(q, k, v, B, S, H, Hk, D, causal, b, h, i, seq_lens=None, scale=None):
    """Softmax probability row [S] (float64) of query (b, h, i)."""
    q, k, v = _f32(q), _f32(k), _f32(v)
    sl = _i32(seq_lens)
    p = np.zeros(S, dtype=np.float64)
    rc = _load().rkv_oracle_prefill_probs(_ptr(q), _ptr(k), _ptr(v), B, S, H, Hk, D,
                                          int(bool(causal)), _ptr(sl),
                                          default_scale(D) if scale is None else float(scale),
                                          b, h, i, _ptr(p))
    if rc != 0:
        raise ValueError("oracle prefill_probs rejected its arguments")
    return p


def decode(q, k_cache, v_cache, M, H, Hk, D, Lmax, seq_lens, scale=None):
    """O[M, H*D] (float64): one query per sequence against cache [M,Hk,Lmax,D]."""
    q, kc, vc = _f32(q), _f32(k_cache), _f32(v_cache)
    assert q.size == M * H * D and kc.size == M * Hk * Lmax * D and vc.size == kc.size
    sl = _i32(seq_lens)
    o = np.zeros((M, H * D), dtype=np.float64)
    rc = _load().rkv_oracle_decode(_ptr(q), _ptr(kc), _ptr(vc), _ptr(o), M, H, Hk, D, Lmax,
                                   _ptr(sl), default_scale(D) if scale is None else float(scale))
    if rc != 0:
        raise ValueError("oracle decode rejected its arguments (a length above max_len?)")
    return o


def scatter(k_new, v_new, k_cache, v_cache, M, T, Hk, D, Lmax, start_pos, inplace=False):
    """Scatter into copies of the caches (or into the given arrays themselves when inplace,
    which must then be C-contiguous float32); returns (k_cache, v_cache, overflow)."""
    kn, vn = _f32(k_new), _f32(v_new)
    if inplace:
        kc, vc = k_cache, v_cache
        for a in (kc, vc):
            if a.dtype != np.float32 or not a.flags.c_contiguous:
                raise ValueError("in-place scatter needs C-contiguous float32 caches")
    else:
        kc = np.array(k_cache, dtype=np.float32, copy=True, order="C")
        vc = np.array(v_cache, dtype=np.float32, copy=True, order="C")
    sp = _i32(start_pos)
    ov = np.zeros(1, dtype=np.int32)
    rc = _load().rkv_oracle_scatter(_ptr(kn), _ptr(vn), _ptr(kc), _ptr(vc), M, T, Hk, D, Lmax,
                                    _ptr(sp), _ptr(ov))
    if rc != 0:
        raise ValueError("oracle scatter rejected its arguments")
    return kc, vc, int(ov[0])


def prefill_cached(q, k_cache, v_cache, B, T, H, Hk, D, Lmax, causal, start_pos, q_lens=None,
                   scale=None):
    """O[B, T, H*D] (float64): a chunk of T queries per sequence at positions start_pos[b]+i
    against cache [B,Hk,Lmax,D] that already holds the chunk's own K/V rows."""
    q, kc, vc = _f32(q), _f32(k_cache), _f32(v_cache)
    assert q.size == B * T * H * D and kc.size == B * Hk * Lmax * D and vc.size == kc.size
    sp, ql = _i32(start_pos), _i32(q_lens)
    o = np.zeros((B, T, H * D), dtype=np.float64)
    rc = _load().rkv_oracle_prefill_cached(_ptr(q), _ptr(kc), _ptr(vc), _ptr(o), B, T, H, Hk, D, Lmax,
                                           int(bool(causal)), _ptr(sp), _ptr(ql),
                                           default_scale(D) if scale is None else float(scale))
    if rc != 0:
        raise ValueError("oracle prefill_cached rejected its arguments (start + length above max_len?)")
    return o


def rope(x, n_heads, head_dim, positions, theta=10000.0, rotary_ndims=None):
    """x [..., n_heads*head_dim] rows at absolute `positions` (one per row), rotated (float64)."""
    x = _f32(x)
    rows = x.size // (n_heads * head_dim)
    assert x.size == rows * n_heads * head_dim
    pos = _i32(np.broadcast_to(np.asarray(positions, np.int32), (rows,)).copy())
    out = np.zeros(x.shape, dtype=np.float64)
    r = head_dim if rotary_ndims is None else int(rotary_ndims)
    rc = _load().rkv_oracle_rope(_ptr(x), _ptr(out), rows, n_heads, head_dim, r, _ptr(pos), float(theta))
    if rc != 0:
        raise ValueError("oracle rope rejected its arguments")
    return out
