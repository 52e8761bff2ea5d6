"""Prefill fused with the cache fill (attn_prefill_fill_cache) on the GPU.

The attention output must equal attn_prefill's to the bit (same kernel arithmetic) and
therefore the oracle within the prefill tolerance; the cache rows 0..S-1 must equal the
oracle's scatter (trueno-gpu attention.rs, fn kv_cache_scatter_gpu; realizar batched
layout) bit for bit, and every other cache row must keep its canary.
"""
import numpy as np
import pytest

from resident_kv_cache_gb300 import inputs
from tests.gpu_util import Guarded, assert_close, empty_guarded, torch_cuda

pytestmark = pytest.mark.gpu
MAX_ABS, MEAN_ABS = 3e-3, 1e-3
FILL = np.float32(-5.5e30)

CASES = [
    # B, S, H, Hk, D, causal, L
    (1, 1, 1, 1, 16, True, 4),
    (2, 37, 4, 2, 32, True, 64),
    (2, 130, 4, 2, 64, False, 200),
    (2, 300, 8, 2, 128, True, 300),
    (1, 300, 8, 8, 128, False, 512),
    (3, 257, 6, 3, 16, True, 400),
    (4, 129, 8, 1, 128, True, 160),
]


@pytest.mark.parametrize("ci", range(len(CASES)))
def test_prefill_fill_cache_matches_prefill_and_scatter(rkv, oracle_mod, ci):
    torch = torch_cuda()
    B, S, H, Hk, D, causal, L = CASES[ci]
    q = inputs.normal((B, S, H * D), (ci, 40))
    k = inputs.normal((B, S, Hk * D), (ci, 41))
    v = inputs.normal((B, S, Hk * D), (ci, 42))
    g_q, g_k, g_v = Guarded(torch, q), Guarded(torch, k), Guarded(torch, v)
    g_o = empty_guarded(torch, (B, S, H * D))
    g_kc = Guarded(torch, np.full((B, Hk, L, D), FILL, np.float32))
    g_vc = Guarded(torch, np.full((B, Hk, L, D), FILL, np.float32))
    rkv.attn_prefill_fill_cache(g_q.t, g_k.t, g_v.t, g_o.t, B, S, H, Hk, D, causal, g_kc.t, g_vc.t, L)
    o_ref = torch.empty((B, S, H * D), device="cuda")
    rkv.attn_prefill(g_q.t, g_k.t, g_v.t, o_ref, B, S, H, Hk, D, causal)
    torch.cuda.synchronize()
    for g in (g_q, g_k, g_v, g_o, g_kc, g_vc):
        assert g.guards_intact()
    got = g_o.numpy()
    assert np.array_equal(got, o_ref.cpu().numpy()), "fused output differs from attn_prefill"
    want = oracle_mod.prefill(q, k, v, B, S, H, Hk, D, causal)
    assert_close(got, want, MAX_ABS, MEAN_ABS, what=f"case {ci}")
    hk, hv, ov = oracle_mod.scatter(k, v, np.full((B, Hk, L, D), FILL, np.float32),
                                    np.full((B, Hk, L, D), FILL, np.float32), B, S, Hk, D, L,
                                    np.zeros(B, np.int32))
    assert ov == 0
    assert np.array_equal(g_kc.numpy(), hk) and np.array_equal(g_vc.numpy(), hv)


def test_fused_fill_causal_gqa_workload(rkv):
    """B=4, S=2048, H=32, Hk=8, D=128 into [4,8,4096,128]: output bitwise equal to attn_prefill and
    caches bitwise equal to kv_cache_scatter at positions 0..2047 (rows 2048.. untouched)."""
    torch = torch_cuda()
    s = inputs.CAUSAL_GQA
    L = inputs.CAUSAL_GQA_CACHE_LEN
    q, k, v = (torch.from_numpy(a).cuda() for a in inputs.prefill_inputs(s))
    o1 = torch.empty_like(q)
    o2 = torch.empty_like(q)
    kc1 = torch.full((s.B, s.Hk, L, s.D), 7.0, device="cuda")
    vc1 = torch.full_like(kc1, -7.0)
    kc2, vc2 = kc1.clone(), vc1.clone()
    rkv.attn_prefill(q, k, v, o1, s.B, s.S, s.H, s.Hk, s.D, True)
    rkv.kv_cache_scatter(k, v, kc1, vc1, s.B, s.S, s.Hk, s.D, L, torch.zeros(s.B, dtype=torch.int32, device="cuda"))
    rkv.attn_prefill_fill_cache(q, k, v, o2, s.B, s.S, s.H, s.Hk, s.D, True, kc2, vc2, L)
    torch.cuda.synchronize()
    assert rkv.rkv_read_device_flags() & rkv.RKV_FLAG_WAIT_TIMEOUT == 0
    assert torch.equal(o1, o2)
    assert torch.equal(kc1, kc2) and torch.equal(vc1, vc2)
