"""Seeded synthetic inputs for the resident-attention workloads.

This module only draws random numbers and names shapes; it holds none of the
attention arithmetic.  Tests, the benchmark and the oracle-side checks all take
their inputs from here so that both sides see identical data.

Distributions follow the workloads the three reference pages imply: Q, K, V and
cache contents are i.i.d. N(0, 1) f32; decode lengths are uniform integers.
numpy's PCG64 generator is used, so a seed gives the same bits on any host.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

# Fixed default seeds: Q, K, V, lengths.
SEED_Q, SEED_K, SEED_V, SEED_LEN = 0, 1, 2, 3


def normal(shape, seed) -> np.ndarray:
    """i.i.d. N(0,1) float32 array of the given shape (seed: int or tuple of ints)."""
    return np.random.default_rng(seed).standard_normal(size=shape, dtype=np.float32)


def uniform_lengths(m: int, lo: int, hi: int, seed: int) -> np.ndarray:
    """m integers uniform in [lo, hi] (inclusive), int32."""
    return np.random.default_rng(seed).integers(lo, hi + 1, size=m, dtype=np.int64).astype(np.int32)


def sample_indices(n_total: int, n: int, seed: int) -> np.ndarray:
    """n distinct sorted indices in [0, n_total) (n clipped to n_total)."""
    n = min(n, n_total)
    return np.sort(np.random.default_rng(seed).choice(n_total, size=n, replace=False)).astype(np.int64)


@dataclass(frozen=True)
class PrefillShape:
    name: str
    B: int
    S: int
    H: int
    Hk: int
    D: int
    causal: bool

    @property
    def flops(self) -> float:
        """Algorithmic FLOP: 2 GEMMs x 2 flop per MAC, causal counts i+1 keys per row."""
        keys = self.S * (self.S + 1) / 2 if self.causal else float(self.S * self.S)
        return 4.0 * self.B * self.H * self.D * keys


@dataclass(frozen=True)
class DecodeShape:
    name: str
    M: int
    H: int
    Hk: int
    D: int
    Lmax: int
    extra: dict = field(default_factory=dict)


# The five workloads: a tiny MHA prefill, an encoder prefill, a causal GQA prefill with its cache
# fill, a batched decode step and a long-context decode.
TINY = PrefillShape("tiny non-causal MHA prefill S=32 H=2 D=16", 1, 32, 2, 2, 16, False)
ENCODER = PrefillShape("encoder non-causal MHA prefill S=1500 H=8 D=64", 1, 1500, 8, 8, 64, False)
CAUSAL_GQA = PrefillShape("causal GQA prefill B=4 S=2048 H=32 Hk=8 D=128", 4, 2048, 32, 8, 128, True)
CAUSAL_GQA_CACHE_LEN = 4096          # cache capacity the causal GQA prefill fills
BATCHED_DECODE = DecodeShape("batched decode M=32 H=32 Hk=8 D=128 Lmax=4096", 32, 32, 8, 128, 4096)
LONG_DECODE = DecodeShape("long-context decode M=1 H=32 Hk=8 D=128 Lmax=32768 x256 steps",
                          1, 32, 8, 128, 32768, {"steps": 256})
LONG_DECODE_PREFILLED = 32768 - 256  # rows present before the first of the 256 steps


def prefill_inputs(shape: PrefillShape, seed_q=SEED_Q, seed_k=SEED_K, seed_v=SEED_V):
    """Interleaved Q [B,S,H*D], K/V [B,S,Hk*D] float32."""
    q = normal((shape.B, shape.S, shape.H * shape.D), seed_q)
    k = normal((shape.B, shape.S, shape.Hk * shape.D), seed_k)
    v = normal((shape.B, shape.S, shape.Hk * shape.D), seed_v)
    return q, k, v


def batched_decode_inputs(shape: DecodeShape = BATCHED_DECODE, seed_q=SEED_Q, seed_k=SEED_K,
                          seed_v=SEED_V, seed_len=SEED_LEN):
    """One batched decode step.

    Returns dict with caches [M,Hk,Lmax,D], q [M,H*D], new rows k_new/v_new
    [M,1,Hk*D], and lens [M]: the attended length INCLUDING the new token,
    uniform in [1, Lmax]; the new row goes to position lens-1.
    """
    M, H, Hk, D, L = shape.M, shape.H, shape.Hk, shape.D, shape.Lmax
    k_cache = normal((M, Hk, L, D), seed_k)
    v_cache = normal((M, Hk, L, D), seed_v)
    q = normal((M, H * D), seed_q)
    k_new = normal((M, 1, Hk * D), (seed_k, 1))
    v_new = normal((M, 1, Hk * D), (seed_v, 1))
    lens = uniform_lengths(M, 1, L, seed_len)
    return {"k_cache": k_cache, "v_cache": v_cache, "q": q, "k_new": k_new, "v_new": v_new,
            "lens": lens, "start_pos": (lens - 1).astype(np.int32)}


def long_decode_step_inputs(step: int, shape: DecodeShape = LONG_DECODE, seed_q=SEED_Q,
                            seed_k=SEED_K, seed_v=SEED_V):
    """Per-step inputs of the long-context decode: q [1,H*D], k_new/v_new [1,1,Hk*D].

    Step t writes row LONG_DECODE_PREFILLED + t and attends to that many + 1 rows.
    """
    H, Hk, D = shape.H, shape.Hk, shape.D
    return {"q": normal((1, H * D), (seed_q, 2, step)),
            "k_new": normal((1, 1, Hk * D), (seed_k, 2, step)),
            "v_new": normal((1, 1, Hk * D), (seed_v, 2, step)),
            "pos": LONG_DECODE_PREFILLED + step,
            "len": LONG_DECODE_PREFILLED + step + 1}
