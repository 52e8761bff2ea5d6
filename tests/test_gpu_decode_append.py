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


def test_long_context_decode_as_timed(rkv, oracle_mod):
    """The long-context decode exactly as it is timed: M=1, H=32, Hk=8, D=128, cache
    [1,8,32768,128] prefilled to 32512 rows, 256 steps of attn_decode_append (row 32512+t
    appended and 32513+t rows attended; one (sequence, kv head) split over every CTA and
    merged in the launch), issued eagerly and replayed from one CUDA graph.  Steps 0, 1, 127
    and 255 are checked against the oracle (trueno-gpu fn kv_cache_scatter_gpu then
    fn incremental_attention_gpu), the graph replay against the eager run bit for bit, and
    the final caches against the oracle's scatter bit for bit."""
    torch = torch_cuda()
    rkv.rkv_read_device_flags(clear=True)   # flags left by earlier tests
    d = inputs.LONG_DECODE
    H, Hk, D, L, T = d.H, d.Hk, d.D, d.Lmax, d.extra["steps"]
    k0 = inputs.normal((1, Hk, L, D), inputs.SEED_K)
    v0 = inputs.normal((1, Hk, L, D), inputs.SEED_V)
    steps = [inputs.long_decode_step_inputs(t) for t in range(T)]
    qs = torch.from_numpy(np.stack([x["q"] for x in steps])).cuda()
    kn = torch.from_numpy(np.stack([x["k_new"] for x in steps])).cuda()
    vn = torch.from_numpy(np.stack([x["v_new"] for x in steps])).cuda()
    lens = torch.tensor([x["len"] for x in steps], dtype=torch.int32, device="cuda")
    n = rkv.attn_decode_workspace_bytes(1, H, Hk, D, L)

    def run(kc, vc, ws, outs):
        for t in range(T):
            rkv.attn_decode_append(qs[t], kn[t], vn[t], kc, vc, outs[t], 1, H, Hk, D, L, lens[t:t + 1], 0.0,
                                   ws, n)

    ka, va = torch.from_numpy(k0).cuda(), torch.from_numpy(v0).cuda()
    wa = torch.zeros(n, dtype=torch.uint8, device="cuda")
    oa = torch.full((T, 1, H * D), float("nan"), device="cuda")
    run(ka, va, wa, oa)
    torch.cuda.synchronize()
    kb, vb = torch.from_numpy(k0).cuda(), torch.from_numpy(v0).cuda()
    wb = torch.zeros(n, dtype=torch.uint8, device="cuda")
    ob = torch.full((T, 1, H * D), float("nan"), device="cuda")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run(kb, vb, wb, ob)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(ob, oa), "graph replay differs from the eager launches"
    assert torch.equal(kb, ka) and torch.equal(vb, va)
    assert rkv.rkv_read_device_flags(clear=True) == 0

    got = oa.cpu().numpy()
    kn_all = np.concatenate([x["k_new"] for x in steps], axis=1)   # [1, 256, Hk*D]
    vn_all = np.concatenate([x["v_new"] for x in steps], axis=1)
    start = np.array([inputs.LONG_DECODE_PREFILLED], np.int32)
    for t in (0, 1, 127, 255):
        hk, hv, _ = oracle_mod.scatter(kn_all[:, :t + 1], vn_all[:, :t + 1], k0, v0, 1, t + 1, Hk, D, L, start)
        want = oracle_mod.decode(steps[t]["q"], hk, hv, 1, H, Hk, D, L, np.array([steps[t]["len"]]))
        assert_close(got[t], want, 1e-4, what=f"step {t}")
    hk, hv, _ = oracle_mod.scatter(kn_all, vn_all, k0, v0, 1, T, Hk, D, L, start)
    assert np.array_equal(ka.cpu().numpy(), hk) and np.array_equal(va.cpu().numpy(), hv)
