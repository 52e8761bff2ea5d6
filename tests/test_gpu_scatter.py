"""KV-cache scatter on the GPU against the oracle: bit-exact, untouched rows intact.

trueno-gpu attention.rs, fn kv_cache_scatter_gpu (row -> cache[h, pos, :],
pos < max_seq_len); batched layout of realizar fn init_batched_kv_cache_gpu.
"""
import numpy as np
import pytest

from resident_kv_cache_gb300 import inputs
from tests.gpu_util import Guarded, torch_cuda

pytestmark = pytest.mark.gpu


def _run(rkv, oracle_mod, M, T, Hk, D, L, start, seed):
    torch = torch_cuda()
    kn = inputs.normal((M, T, Hk * D), (seed, 0))
    vn = inputs.normal((M, T, Hk * D), (seed, 1))
    kc0 = inputs.normal((M, Hk, L, D), (seed, 2))
    vc0 = inputs.normal((M, Hk, L, D), (seed, 3))
    start = np.asarray(start, np.int32)
    g_kn, g_vn = Guarded(torch, kn), Guarded(torch, vn)
    g_kc, g_vc = Guarded(torch, kc0), Guarded(torch, vc0)
    g_sp = Guarded(torch, start, np.int32)
    ov = torch.zeros(1, dtype=torch.int32, device="cuda")
    rkv.kv_cache_scatter(g_kn.t, g_vn.t, g_kc.t, g_vc.t, M, T, Hk, D, L, g_sp.t, ov)
    torch.cuda.synchronize()
    want_k, want_v, want_ov = oracle_mod.scatter(kn, vn, kc0, vc0, M, T, Hk, D, L, start)
    assert np.array_equal(g_kc.numpy(), want_k)
    assert np.array_equal(g_vc.numpy(), want_v)
    assert int(ov.item()) == want_ov
    for g in (g_kn, g_vn, g_kc, g_vc):
        assert g.guards_intact()
    return want_ov


@pytest.mark.parametrize("D", [16, 32, 64, 128])
def test_scatter_small_all_head_dims(rkv, oracle_mod, D):
    _run(rkv, oracle_mod, M=3, T=5, Hk=2, D=D, L=12, start=[0, 7, 3], seed=D)


def test_scatter_overflow_and_negative_positions(rkv, oracle_mod):
    ov = _run(rkv, oracle_mod, M=4, T=6, Hk=3, D=32, L=10, start=[8, -2, 4, 9], seed=5)
    assert ov == (4 + 2 + 0 + 5)
    flags = rkv.rkv_read_device_flags(clear=True)
    assert flags & rkv.RKV_FLAG_NEGATIVE_INPUT


def test_scatter_ragged_token_chunks(rkv, oracle_mod):
    # T not a multiple of the tokens-per-block chunk; several blocks per sequence
    _run(rkv, oracle_mod, M=2, T=37, Hk=8, D=128, L=64, start=[1, 27], seed=11)


def test_scatter_causal_gqa_cache_fill_full_size(rkv, oracle_mod):
    """B=4, T=2048, Hk=8, D=128 rows into a [4,8,4096,128] cache at positions 0..2047."""
    s = inputs.CAUSAL_GQA
    _run(rkv, oracle_mod, M=s.B, T=s.S, Hk=s.Hk, D=s.D, L=inputs.CAUSAL_GQA_CACHE_LEN,
         start=[0] * s.B, seed=21)


def test_scatter_batched_decode_step_full_size(rkv, oracle_mod):
    """M=32 single-token appends at position len-1 of a [32,8,4096,128] cache."""
    d = inputs.BATCHED_DECODE
    lens = inputs.uniform_lengths(d.M, 1, d.Lmax, inputs.SEED_LEN)
    _run(rkv, oracle_mod, M=d.M, T=1, Hk=d.Hk, D=d.D, L=d.Lmax, start=lens - 1, seed=22)
