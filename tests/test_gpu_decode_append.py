"""One decode step in one launch (attn_decode_append) against the same step as two launches
(kv_cache_scatter at seq_lens-1, then attn_decode_batched) and the oracle.

trueno-gpu attention.rs, fn kv_cache_scatter_gpu then fn incremental_attention_gpu; realizar
batched cache layout.  Same kernel arithmetic, so the output must match the two-launch step bit
for bit, and the cache must match the scatter bit for bit.
"""
import numpy as np
import pytest

from resident_kv_cache_gb300 import inputs
from tests.gpu_util import assert_close, torch_cuda

pytestmark = pytest.mark.gpu

CASES = [
    # M, H, Hk, D, L, lens
    (1, 1, 1, 16, 5, [5]),
    (3, 8, 2, 64, 200, [200, 1, 77]),
    (4, 16, 4, 128, 300, [300, 0, 2000, 129]),      # an empty sequence and a clamped one (no row written)
    (6, 32, 8, 128, 1000, [1000, 999, 513, 2, 64, 1]),
    (2, 8, 8, 32, 90, [90, 33]),
]


def _run_pair(rkv, torch, M, H, Hk, D, L, lens, seed):
    q = inputs.normal((M, H * D), (seed, 0))
    kc = inputs.normal((M, Hk, L, D), (seed, 1))
    vc = inputs.normal((M, Hk, L, D), (seed, 2))
    kn = inputs.normal((M, Hk * D), (seed, 3))
    vn = inputs.normal((M, Hk * D), (seed, 4))
    dq, dkn, dvn = (torch.from_numpy(a).cuda() for a in (q, kn, vn))
    ln = torch.tensor(lens, dtype=torch.int32, device="cuda")
    n = rkv.attn_decode_workspace_bytes(M, H, Hk, D, L)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    k1, v1 = torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda()
    k2, v2 = k1.clone(), v1.clone()
    o1 = torch.full((M, H * D), float("nan"), device="cuda")
    o2 = torch.full((M, H * D), float("nan"), device="cuda")
    rkv.kv_cache_scatter(dkn, dvn, k1, v1, M, 1, Hk, D, L, ln - 1)
    rkv.attn_decode_batched(dq, k1, v1, o1, M, H, Hk, D, L, ln, 0.0, ws, n)
    rkv.attn_decode_append(dq, dkn, dvn, k2, v2, o2, M, H, Hk, D, L, ln, 0.0, ws, n)
    torch.cuda.synchronize()
    return (q, kc, vc, kn, vn), (o1, k1, v1), (o2, k2, v2)


@pytest.mark.parametrize("ci", range(len(CASES)))
def test_decode_append_equals_scatter_then_decode(rkv, oracle_mod, ci):
    torch = torch_cuda()
    M, H, Hk, D, L, lens = CASES[ci]
    (q, kc, vc, kn, vn), (o1, k1, v1), (o2, k2, v2) = _run_pair(rkv, torch, M, H, Hk, D, L, lens, 600 + ci)
    assert torch.equal(o1, o2)
    assert torch.equal(k1, k2) and torch.equal(v1, v2)
    hk, hv, _ = oracle_mod.scatter(kn.reshape(M, 1, Hk * D), vn.reshape(M, 1, Hk * D), kc, vc, M, 1, Hk, D, L,
                                   np.array(lens, np.int32) - 1)
    assert np.array_equal(k2.cpu().numpy(), hk) and np.array_equal(v2.cpu().numpy(), hv)
    want = oracle_mod.decode(q, hk, hv, M, H, Hk, D, L, np.minimum(np.array(lens), L))
    assert_close(o2.cpu().numpy(), want, 1e-4)


def test_decode_append_batched_decode_workload(rkv):
    """M=32, H=32, Hk=8, D=128, cache [32,8,4096,128], lengths U{1..4096}."""
    torch = torch_cuda()
    d = inputs.BATCHED_DECODE
    x = inputs.batched_decode_inputs(d)
    M, H, Hk, D, L = d.M, d.H, d.Hk, d.D, d.Lmax
    dq = torch.from_numpy(x["q"]).cuda()
    kn = torch.from_numpy(x["k_new"]).cuda()
    vn = torch.from_numpy(x["v_new"]).cuda()
    ln = torch.from_numpy(x["lens"]).cuda()
    sp = torch.from_numpy(x["start_pos"]).cuda()
    n = rkv.attn_decode_workspace_bytes(M, H, Hk, D, L)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    k1, v1 = torch.from_numpy(x["k_cache"]).cuda(), torch.from_numpy(x["v_cache"]).cuda()
    k2, v2 = k1.clone(), v1.clone()
    o1 = torch.empty((M, H * D), device="cuda")
    o2 = torch.empty((M, H * D), device="cuda")
    rkv.kv_cache_scatter(kn, vn, k1, v1, M, 1, Hk, D, L, sp)
    rkv.attn_decode_batched(dq, k1, v1, o1, M, H, Hk, D, L, ln, 0.0, ws, n)
    rkv.attn_decode_append(dq, kn, vn, k2, v2, o2, M, H, Hk, D, L, ln, 0.0, ws, n)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)
    assert torch.equal(k1, k2) and torch.equal(v1, v2)
