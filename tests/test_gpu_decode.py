"""Split-KV batched decode on the GPU against the oracle (tolerance 1e-4 max abs).

trueno-gpu attention.rs, fn incremental_attention_gpu (single query per head,
first seq_len cache rows, zero row for seq_len == 0); trustformers-core
attention.rs, fn attention_decode_gpu_to_gpu (no mask); batched cache of
realizar fn init_batched_kv_cache_gpu (M <= 32, per-sequence lengths).
"""
import numpy as np
import pytest

from resident_kv_cache_gb300 import inputs
from tests.gpu_util import Guarded, assert_close, empty_guarded, torch_cuda

pytestmark = pytest.mark.gpu
TOL = 1e-4


def _workspace(torch, rkv, M, H, Hk, D, L):
    n = rkv.attn_decode_workspace_bytes(M, H, Hk, D, L)
    return torch.zeros(n, dtype=torch.uint8, device="cuda"), n


def _decode(rkv, torch, q, kc, vc, M, H, Hk, D, L, lens, ws=None, scale=0.0):
    g_q, g_k, g_v = Guarded(torch, q), Guarded(torch, kc), Guarded(torch, vc)
    g_o = empty_guarded(torch, (M, H * D))
    g_l = Guarded(torch, np.asarray(lens, np.int32), np.int32)
    if ws is None:
        ws = _workspace(torch, rkv, M, H, Hk, D, L)
    rkv.attn_decode_batched(g_q.t, g_k.t, g_v.t, g_o.t, M, H, Hk, D, L, g_l.t, scale, ws[0], ws[1])
    torch.cuda.synchronize()
    for g in (g_q, g_k, g_v, g_o):
        assert g.guards_intact()
    return g_o.numpy(), ws


CASES = [
    # M, H, Hk, D, L, lens
    (1, 1, 1, 16, 5, [5]),
    (2, 4, 4, 32, 70, [70, 1]),
    (3, 8, 4, 64, 200, [200, 64, 65]),
    (4, 16, 4, 128, 300, [300, 1, 0, 129]),
    (5, 32, 4, 128, 1000, [1000, 999, 513, 2, 64]),
    (2, 16, 2, 128, 257, [257, 100]),
    (3, 8, 8, 128, 90, [90, 33, 7]),
    (2, 8, 1, 64, 150, [150, 150]),
    (4, 64, 8, 16, 40, [40, 3, 0, 17]),
    (1, 8, 1, 32, 2048, [2048]),
    (32, 8, 2, 64, 96, list(range(1, 97, 3))),
]


@pytest.mark.parametrize("ci", range(len(CASES)))
def test_decode_matches_oracle(rkv, oracle_mod, ci):
    torch = torch_cuda()
    M, H, Hk, D, L, lens = CASES[ci]
    q = inputs.normal((M, H * D), (ci, 0))
    kc = inputs.normal((M, Hk, L, D), (ci, 1))
    vc = inputs.normal((M, Hk, L, D), (ci, 2))
    got, _ = _decode(rkv, torch, q, kc, vc, M, H, Hk, D, L, lens)
    want = oracle_mod.decode(q, kc, vc, M, H, Hk, D, L, np.array(lens))
    assert_close(got, want, TOL, what=f"case {ci}")


def test_decode_explicit_scale(rkv, oracle_mod):
    torch = torch_cuda()
    M, H, Hk, D, L, lens = 2, 8, 2, 64, 100, [100, 37]
    q = inputs.normal((M, H * D), 91)
    kc, vc = inputs.normal((M, Hk, L, D), 92), inputs.normal((M, Hk, L, D), 93)
    got, _ = _decode(rkv, torch, q, kc, vc, M, H, Hk, D, L, lens, scale=0.3)
    want = oracle_mod.decode(q, kc, vc, M, H, Hk, D, L, np.array(lens), scale=0.3)
    assert_close(got, want, TOL)


def test_decode_clamps_lengths_above_max_len(rkv, oracle_mod):
    torch = torch_cuda()
    rkv.rkv_read_device_flags(clear=True)
    M, H, Hk, D, L = 2, 8, 2, 128, 64
    q = inputs.normal((M, H * D), 81)
    kc, vc = inputs.normal((M, Hk, L, D), 82), inputs.normal((M, Hk, L, D), 83)
    got, _ = _decode(rkv, torch, q, kc, vc, M, H, Hk, D, L, [1000, -5])
    assert rkv.rkv_read_device_flags(clear=True) & rkv.RKV_FLAG_LEN_CLAMPED
    want = oracle_mod.decode(q, kc, vc, M, H, Hk, D, L, np.array([L, 0]))
    assert_close(got, want, TOL)


def test_workspace_reuse_and_tickets_reset(rkv, oracle_mod):
    """Two calls on one workspace give identical results and leave the tickets zero."""
    torch = torch_cuda()
    M, H, Hk, D, L = 4, 32, 8, 128, 3000
    lens = [3000, 2999, 1500, 1]
    q = inputs.normal((M, H * D), 71)
    kc, vc = inputs.normal((M, Hk, L, D), 72), inputs.normal((M, Hk, L, D), 73)
    o1, ws = _decode(rkv, torch, q, kc, vc, M, H, Hk, D, L, lens)
    o2, _ = _decode(rkv, torch, q, kc, vc, M, H, Hk, D, L, lens, ws=ws)
    assert np.array_equal(o1, o2)
    assert int(ws[0][: rkv.RKV_DECODE_TICKET_BYTES].view(torch.int32).abs().sum().item()) == 0
    want = oracle_mod.decode(q, kc, vc, M, H, Hk, D, L, np.array(lens))
    assert_close(o1, want, TOL)


def test_one_workspace_serves_calls_of_different_sizes(rkv, oracle_mod):
    """A workspace sized for the largest call, zero-filled once, reused by calls whose
    (M, n_kv_heads) differ: the tickets sit at fixed places at its head, so a larger call's
    tickets never land on a smaller call's records.  Lengths are long enough that every
    (sequence, kv head) is split over several CTAs and merged through its ticket."""
    torch = torch_cuda()
    rkv.rkv_read_device_flags(clear=True)   # flags left by earlier tests
    H, D, L = 32, 128, 4096
    shapes = [(8, 8), (16, 8), (8, 8), (4, 16), (16, 8), (2, 32)]   # (M, Hk)
    n = max(rkv.attn_decode_workspace_bytes(M, H, Hk, D, L) for M, Hk in shapes)
    ws = (torch.zeros(n, dtype=torch.uint8, device="cuda"), n)
    for i, (M, Hk) in enumerate(shapes):
        lens = [4096 - 37 * m for m in range(M)]
        q = inputs.normal((M, H * D), (900 + i, 0))
        kc, vc = inputs.normal((M, Hk, L, D), (900 + i, 1)), inputs.normal((M, Hk, L, D), (900 + i, 2))
        got, _ = _decode(rkv, torch, q, kc, vc, M, H, Hk, D, L, lens, ws=ws)
        want = oracle_mod.decode(q, kc, vc, M, H, Hk, D, L, np.array(lens))
        assert_close(got, want, TOL, what=f"call {i}: M={M}, Hk={Hk}")
        tickets = ws[0][: rkv.RKV_DECODE_TICKET_BYTES].view(torch.int32)
        assert int(tickets.abs().sum().item()) == 0, f"call {i} left a ticket set"
    assert rkv.rkv_read_device_flags(clear=True) == 0


def test_batched_decode_step_full_size(rkv, oracle_mod):
    """M=32, H=32, Hk=8, D=128, cache [32,8,4096,128], lengths U{1..4096}: scatter the new
    row at len-1, then decode over len rows (the batched decode workload)."""
    torch = torch_cuda()
    d = inputs.BATCHED_DECODE
    x = inputs.batched_decode_inputs(d)
    M, H, Hk, D, L = d.M, d.H, d.Hk, d.D, d.Lmax
    kc = torch.from_numpy(x["k_cache"]).cuda()
    vc = torch.from_numpy(x["v_cache"]).cuda()
    kn = torch.from_numpy(x["k_new"]).cuda()
    vn = torch.from_numpy(x["v_new"]).cuda()
    sp = torch.from_numpy(x["start_pos"]).cuda()
    ln = torch.from_numpy(x["lens"]).cuda()
    q = torch.from_numpy(x["q"]).cuda()
    o = torch.full((M, H * D), float("nan"), device="cuda")
    ws, nws = _workspace(torch, rkv, M, H, Hk, D, L)
    rkv.kv_cache_scatter(kn, vn, kc, vc, M, 1, Hk, D, L, sp)
    rkv.attn_decode_batched(q, kc, vc, o, M, H, Hk, D, L, ln, 0.0, ws, nws)
    torch.cuda.synchronize()
    hk, hv, ov = oracle_mod.scatter(x["k_new"], x["v_new"], x["k_cache"], x["v_cache"], M, 1, Hk, D, L,
                                    x["start_pos"])
    assert ov == 0
    assert np.array_equal(kc.cpu().numpy(), hk) and np.array_equal(vc.cpu().numpy(), hv)
    want = oracle_mod.decode(x["q"], hk, hv, M, H, Hk, D, L, x["lens"])
    assert_close(o.cpu().numpy(), want, TOL, what="batched decode step")


def test_long_context_decode_sampled_steps(rkv, oracle_mod):
    """M=1, cache [1,8,32768,128] prefilled to 32512 rows, 256 append+decode steps; steps
    0, 1, 127, 255 are checked against the oracle and the final cache bit-exactly."""
    torch = torch_cuda()
    d = inputs.LONG_DECODE
    H, Hk, D, L = d.H, d.Hk, d.D, d.Lmax
    k0 = inputs.normal((1, Hk, L, D), inputs.SEED_K)
    v0 = inputs.normal((1, Hk, L, D), inputs.SEED_V)
    kc, vc = torch.from_numpy(k0).cuda(), torch.from_numpy(v0).cuda()
    ws, nws = _workspace(torch, rkv, 1, H, Hk, D, L)
    o = torch.empty((1, H * D), device="cuda")
    pos_t = torch.zeros(1, dtype=torch.int32, device="cuda")
    len_t = torch.zeros(1, dtype=torch.int32, device="cuda")
    sampled = {0: None, 1: None, 127: None, 255: None}
    steps = [inputs.long_decode_step_inputs(t) for t in range(256)]
    for t, x in enumerate(steps):
        pos_t.fill_(x["pos"])
        len_t.fill_(x["len"])
        rkv.kv_cache_scatter(torch.from_numpy(x["k_new"]).cuda(), torch.from_numpy(x["v_new"]).cuda(),
                             kc, vc, 1, 1, Hk, D, L, pos_t)
        rkv.attn_decode_batched(torch.from_numpy(x["q"]).cuda(), kc, vc, o, 1, H, Hk, D, L, len_t, 0.0,
                                ws, nws)
        if t in sampled:
            sampled[t] = o.cpu().numpy().copy()
    torch.cuda.synchronize()
    kn_all = np.concatenate([x["k_new"] for x in steps], axis=1)   # [1, 256, Hk*D]
    vn_all = np.concatenate([x["v_new"] for x in steps], axis=1)
    start = np.array([inputs.LONG_DECODE_PREFILLED], np.int32)
    for t, got in sampled.items():
        hk, hv, _ = oracle_mod.scatter(kn_all[:, :t + 1], vn_all[:, :t + 1], k0, v0, 1, t + 1, Hk, D, L,
                                       start)
        want = oracle_mod.decode(steps[t]["q"], hk, hv, 1, H, Hk, D, L, np.array([steps[t]["len"]]))
        assert_close(got, want, TOL, what=f"step {t}")
    hk, hv, _ = oracle_mod.scatter(kn_all, vn_all, k0, v0, 1, 256, Hk, D, L, start)
    assert np.array_equal(kc.cpu().numpy(), hk) and np.array_equal(vc.cpu().numpy(), hv)


def test_append_and_decode_steps_replay_from_a_cuda_graph(rkv):
    """Scatter + decode launches captured in a CUDA graph replay to the same bits as the
    eager launches (the library never syncs, allocates or reads the host inside a call)."""
    torch = torch_cuda()
    M, H, Hk, D, L, steps = 2, 32, 8, 128, 1024, 8
    kc0 = torch.from_numpy(inputs.normal((M, Hk, L, D), 501)).cuda()
    vc0 = torch.from_numpy(inputs.normal((M, Hk, L, D), 502)).cuda()
    qs = torch.from_numpy(inputs.normal((steps, M, H * D), 503)).cuda()
    kn = torch.from_numpy(inputs.normal((steps, M, 1, Hk * D), 504)).cuda()
    vn = torch.from_numpy(inputs.normal((steps, M, 1, Hk * D), 505)).cuda()
    pos = torch.tensor([[500 + t, 900 + t] for t in range(steps)], dtype=torch.int32, device="cuda")
    n = rkv.attn_decode_workspace_bytes(M, H, Hk, D, L)

    def run(kc, vc, ws, outs):
        for t in range(steps):
            rkv.kv_cache_scatter(kn[t], vn[t], kc, vc, M, 1, Hk, D, L, pos[t])
            rkv.attn_decode_batched(qs[t], kc, vc, outs[t], M, H, Hk, D, L, pos[t] + 1, 0.0, ws, n)

    ka, va = kc0.clone(), vc0.clone()
    wa = torch.zeros(n, dtype=torch.uint8, device="cuda")
    oa = torch.empty((steps, M, H * D), device="cuda")
    run(ka, va, wa, oa)
    torch.cuda.synchronize()
    kb, vb = kc0.clone(), vc0.clone()
    wb = torch.zeros(n, dtype=torch.uint8, device="cuda")
    ob = torch.full((steps, M, H * D), float("nan"), device="cuda")
    lens_b = pos + 1                      # allocated before capture
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for t in range(steps):
            rkv.kv_cache_scatter(kn[t], vn[t], kb, vb, M, 1, Hk, D, L, pos[t])
            rkv.attn_decode_batched(qs[t], kb, vb, ob[t], M, H, Hk, D, L, lens_b[t], 0.0, wb, n)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(ob, oa)
    assert torch.equal(kb, ka) and torch.equal(vb, va)
