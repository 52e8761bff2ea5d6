"""Seeded random shapes for every entry point of the path, against the oracle.

The hand-picked cases in the other GPU tests cover the edges one by one; this sweep draws the
shape parameters at random (fixed seeds, so every run sees the same cases) across everything
the entry points accept: head dims 16/32/64/128, GQA group sizes, sequence lengths that end
anywhere in a tile (including 0, 1 and the full length), causal and non-causal, padded batches,
chunk offsets and clamped lengths.  Tolerances are the same as the per-entry tests: 3e-3 max /
1e-3 mean abs for the TF32 prefill, 1e-4 for the f32 decode, bit-exact for cache writes.
"""
import numpy as np
import pytest

from resident_kv_cache_gb300 import inputs
from tests.gpu_util import assert_close, torch_cuda
from tests.test_gpu_decode import _decode
from tests.test_gpu_decode_append import _run_pair
from tests.test_gpu_prefill import _prefill
from tests.test_gpu_prefill_chunked import _chunked

pytestmark = pytest.mark.gpu
PF_MAX, PF_MEAN, DEC_TOL = 3e-3, 1e-3, 1e-4
N_CASES = 12
HEAD_DIMS = (16, 32, 64, 128)          # cycled, so every head dim meets both mask modes


def _lens(rng, n, hi):
    """n lengths in [0, hi], with the ends of the range drawn often."""
    out = rng.integers(0, hi + 1, size=n)
    ends = rng.random(n)
    out[ends < 0.15] = 0
    out[(ends >= 0.15) & (ends < 0.3)] = 1
    out[(ends >= 0.3) & (ends < 0.45)] = hi
    return [int(x) for x in out]


def _prefill_case(i):
    rng = np.random.default_rng(1000 + i)
    D = HEAD_DIMS[i % 4]
    Hk = int(rng.choice([1, 2, 4]))
    H = Hk * int(rng.choice([1, 2, 3, 4, 8]))
    B = int(rng.integers(1, 4))
    S = int(rng.integers(1, 321))
    causal = (i // 4) % 2 == 0
    lens = _lens(rng, B, S) if rng.random() < 0.5 else None
    return B, S, H, Hk, D, causal, lens


def _decode_case(i):
    rng = np.random.default_rng(2000 + i)
    D = HEAD_DIMS[i % 4]
    Hk = int(rng.choice([1, 2, 4]))
    H = Hk * int(rng.choice([1, 2, 4, 8]))
    M = int(rng.integers(1, 33))
    L = int(rng.integers(1, 701))
    return M, H, Hk, D, L, _lens(rng, M, L)


def _chunked_case(i):
    rng = np.random.default_rng(3000 + i)
    D = HEAD_DIMS[i % 4]
    Hk = int(rng.choice([1, 2, 4]))
    H = Hk * int(rng.choice([1, 2, 4]))
    M = int(rng.integers(1, 4))
    T = int(rng.integers(1, 200))
    L = int(rng.integers(T, T + 400))
    start = [int(rng.integers(0, L - T + 1)) for _ in range(M)]
    causal = (i // 4) % 2 == 0
    q_lens = _lens(rng, M, T) if rng.random() < 0.5 else None
    return M, T, H, Hk, D, L, causal, start, q_lens


@pytest.mark.parametrize("ci", range(N_CASES))
def test_random_prefill(rkv, oracle_mod, ci):
    torch = torch_cuda()
    B, S, H, Hk, D, causal, lens = _prefill_case(ci)
    q = inputs.normal((B, S, H * D), (ci, 710))
    k = inputs.normal((B, S, Hk * D), (ci, 711))
    v = inputs.normal((B, S, Hk * D), (ci, 712))
    got = _prefill(rkv, torch, q, k, v, B, S, H, Hk, D, causal, lens)
    want = oracle_mod.prefill(q, k, v, B, S, H, Hk, D, causal, seq_lens=lens)
    assert_close(got, want, PF_MAX, PF_MEAN, what=f"prefill case {_prefill_case(ci)}")
    if lens is not None:
        for b, n in enumerate(lens):
            assert np.all(got[b, n:] == 0.0)


@pytest.mark.parametrize("ci", range(N_CASES))
def test_random_decode(rkv, oracle_mod, ci):
    torch = torch_cuda()
    M, H, Hk, D, L, lens = _decode_case(ci)
    q = inputs.normal((M, H * D), (ci, 720))
    kc = inputs.normal((M, Hk, L, D), (ci, 721))
    vc = inputs.normal((M, Hk, L, D), (ci, 722))
    got, _ = _decode(rkv, torch, q, kc, vc, M, H, Hk, D, L, lens)
    want = oracle_mod.decode(q, kc, vc, M, H, Hk, D, L, np.array(lens))
    assert_close(got, want, DEC_TOL, what=f"decode case {_decode_case(ci)}")


@pytest.mark.parametrize("ci", range(N_CASES))
def test_random_decode_append(rkv, oracle_mod, ci):
    torch = torch_cuda()
    M, H, Hk, D, L, lens = _decode_case(N_CASES + ci)
    (q, kc, vc, kn, vn), (o1, k1, v1), (o2, k2, v2) = _run_pair(rkv, torch, M, H, Hk, D, L, lens, 730 + ci)
    assert torch.equal(o1, o2) and torch.equal(k1, k2) and torch.equal(v1, v2)
    hk, hv, _ = oracle_mod.scatter(kn.reshape(M, 1, Hk * D), vn.reshape(M, 1, Hk * D), kc, vc, M, 1, Hk, D, L,
                                   np.array(lens, np.int32) - 1)
    assert np.array_equal(k2.cpu().numpy(), hk) and np.array_equal(v2.cpu().numpy(), hv)
    want = oracle_mod.decode(q, hk, hv, M, H, Hk, D, L, np.minimum(np.array(lens), L))
    assert_close(o2.cpu().numpy(), want, DEC_TOL, what=f"decode append case {(M, H, Hk, D, L, lens)}")


@pytest.mark.parametrize("ci", range(N_CASES))
def test_random_chunked_prefill(rkv, oracle_mod, ci):
    torch = torch_cuda()
    M, T, H, Hk, D, L, causal, start, q_lens = _chunked_case(ci)
    q = inputs.normal((M, T, H * D), (ci, 740))
    kc = inputs.normal((M, Hk, L, D), (ci, 741))
    vc = inputs.normal((M, Hk, L, D), (ci, 742))
    got = _chunked(rkv, torch, q, kc, vc, M, T, H, Hk, D, L, causal, start, q_lens)
    want = oracle_mod.prefill_cached(q, kc, vc, M, T, H, Hk, D, L, causal, np.array(start), q_lens=q_lens)
    assert_close(got, want, PF_MAX, PF_MEAN, what=f"chunked case {_chunked_case(ci)}")
    if q_lens is not None:
        for b, n in enumerate(q_lens):
            assert np.all(got[b, n:] == 0.0)


def test_random_cases_span_the_parameter_space():
    """The drawn cases reach every head dim and both mask modes (a host check of the sweep)."""
    pf = [_prefill_case(i) for i in range(N_CASES)]
    dec = [_decode_case(i) for i in range(2 * N_CASES)]
    ch = [_chunked_case(i) for i in range(N_CASES)]
    assert {c[4] for c in pf} | {c[4] for c in ch} == {16, 32, 64, 128}
    assert {c[3] for c in dec} == {16, 32, 64, 128}
    assert {c[5] for c in pf} == {True, False} and {c[6] for c in ch} == {True, False}
    assert any(0 in c[5] for c in dec) and any(c[5].count(c[4]) for c in dec)
