"""Prefill appended behind an existing cache (attn_prefill_chunked) on the GPU against
the oracle.

Semantics: trustformers-core attention.rs, fn attention_prefill_gpu_to_gpu (doc: a
prefill behind an existing cache runs the decode path once per token) and
fn attention_decode_gpu_to_gpu; cache layout of realizar cache_from_cache_from_kv_cache.rs,
fn init_batched_kv_cache_gpu.  Tolerance: 3e-3 max abs and 1e-3 mean abs on N(0,1) inputs,
as for attn_prefill (same kernel, TF32 products, f32 accumulation).
"""
import numpy as np
import pytest

from resident_kv_cache_gb300 import inputs
from tests.gpu_util import Guarded, assert_close, empty_guarded, torch_cuda

pytestmark = pytest.mark.gpu
MAX_ABS, MEAN_ABS = 3e-3, 1e-3


def _chunked(rkv, torch, q, kc, vc, M, T, H, Hk, D, L, causal, start, q_lens=None, scale=0.0):
    g_q, g_k, g_v = Guarded(torch, q), Guarded(torch, kc), Guarded(torch, vc)
    g_o = empty_guarded(torch, (M, T, H * D))
    g_s = Guarded(torch, np.asarray(start, np.int32), np.int32)
    g_n = None if q_lens is None else Guarded(torch, np.asarray(q_lens, np.int32), np.int32)
    rkv.attn_prefill_chunked(g_q.t, g_k.t, g_v.t, g_o.t, M, T, H, Hk, D, L, causal, g_s.t,
                             None if g_n is None else g_n.t, scale)
    torch.cuda.synchronize()
    for g in (g_q, g_k, g_v, g_o):
        assert g.guards_intact()
    return g_o.numpy()


CASES = [
    # M, T, H, Hk, D, L, causal, start_pos, q_lens
    (1, 1, 1, 1, 16, 8, True, [0], None),
    (2, 37, 4, 2, 32, 200, True, [0, 100], None),
    (2, 130, 8, 2, 64, 400, True, [5, 270], [130, 64]),
    (1, 300, 8, 8, 128, 1000, False, [123], None),
    (3, 129, 4, 1, 128, 700, True, [0, 1, 571], [129, 1, 129]),
    (2, 64, 16, 4, 128, 256, True, [192, 64], [64, 0]),
    (1, 200, 2, 2, 16, 300, False, [100], [150]),
    (4, 65, 8, 8, 64, 1100, False, [1035, 0, 500, 999], None),
]


@pytest.mark.parametrize("ci", range(len(CASES)))
def test_prefill_chunked_matches_oracle(rkv, oracle_mod, ci):
    torch = torch_cuda()
    M, T, H, Hk, D, L, causal, sp, ql = CASES[ci]
    q = inputs.normal((M, T, H * D), (ci, 20))
    kc = inputs.normal((M, Hk, L, D), (ci, 21))
    vc = inputs.normal((M, Hk, L, D), (ci, 22))
    got = _chunked(rkv, torch, q, kc, vc, M, T, H, Hk, D, L, causal, sp, ql)
    want = oracle_mod.prefill_cached(q, kc, vc, M, T, H, Hk, D, L, causal, np.array(sp), q_lens=ql)
    assert_close(got, want, MAX_ABS, MEAN_ABS, what=f"case {ci}")
    if ql is not None:
        for b, n in enumerate(ql):
            assert np.all(got[b, n:] == 0.0)


def test_prefill_chunked_ignores_non_finite_rows_outside_the_chunk(rkv, oracle_mod):
    """Cache rows past start+n and padded query rows hold NaN/Inf: the valid outputs still
    match the oracle and padded rows are exact zeros."""
    torch = torch_cuda()
    M, T, H, Hk, D, L = 2, 100, 8, 2, 128, 512
    sp, ql = np.array([60, 300], np.int32), np.array([100, 37], np.int32)
    q = inputs.normal((M, T, H * D), 301)
    q[1, 37:] = np.nan
    kc = inputs.normal((M, Hk, L, D), 302)
    vc = inputs.normal((M, Hk, L, D), 303)
    for b in range(M):
        kc[b, :, sp[b] + ql[b]:, :] = np.inf
        vc[b, :, sp[b] + ql[b]:, :] = np.nan
    for causal in (True, False):
        got = _chunked(rkv, torch, q, kc, vc, M, T, H, Hk, D, L, causal, sp, ql)
        kf, vf = np.nan_to_num(kc, posinf=0.0), np.nan_to_num(vc)
        want = oracle_mod.prefill_cached(np.nan_to_num(q), kf, vf, M, T, H, Hk, D, L, causal, sp, q_lens=ql)
        assert_close(got, want, MAX_ABS, MEAN_ABS, what=f"causal={causal}")
        assert np.all(got[1, 37:] == 0.0)


def test_prefill_chunked_from_empty_cache_is_bitwise_attn_prefill(rkv):
    """start_pos = 0 and the cache filled by kv_cache_scatter: same kernel, same tiles, so the
    result equals attn_prefill's bit for bit."""
    torch = torch_cuda()
    B, S, H, Hk, D, L = 2, 333, 16, 4, 128, 1024
    q, k, v = (inputs.normal((B, S, n * D), (311, t)) for t, n in enumerate((H, Hk, Hk)))
    dq, dk, dv = (torch.from_numpy(a).cuda() for a in (q, k, v))
    kc = torch.randn((B, Hk, L, D), device="cuda")
    vc = torch.randn((B, Hk, L, D), device="cuda")
    zero = torch.zeros(B, dtype=torch.int32, device="cuda")
    lens = torch.tensor([333, 200], dtype=torch.int32, device="cuda")
    rkv.kv_cache_scatter(dk, dv, kc, vc, B, S, Hk, D, L, zero)
    for causal in (True, False):
        o1 = torch.empty((B, S, H * D), device="cuda")
        o2 = torch.empty((B, S, H * D), device="cuda")
        rkv.attn_prefill(dq, dk, dv, o1, B, S, H, Hk, D, causal, lens)
        rkv.attn_prefill_chunked(dq, kc, vc, o2, B, S, H, Hk, D, L, causal, zero, lens)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2), f"causal={causal}"


def test_prefill_chunked_single_token_matches_decode(rkv):
    """T = 1 is one decode step of length start+1 (GPU decode vs GPU chunked prefill)."""
    torch = torch_cuda()
    M, H, Hk, D, L = 5, 32, 8, 128, 2000
    q = torch.from_numpy(inputs.normal((M, H * D), 321)).cuda()
    kc = torch.from_numpy(inputs.normal((M, Hk, L, D), 322)).cuda()
    vc = torch.from_numpy(inputs.normal((M, Hk, L, D), 323)).cuda()
    sp = torch.tensor([0, 1, 999, 1500, 1999], dtype=torch.int32, device="cuda")
    o1 = torch.empty((M, H * D), device="cuda")
    o2 = torch.empty((M, H * D), device="cuda")
    n = rkv.attn_decode_workspace_bytes(M, H, Hk, D, L)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    rkv.attn_decode_batched(q, kc, vc, o1, M, H, Hk, D, L, sp + 1, 0.0, ws, n)
    rkv.attn_prefill_chunked(q, kc, vc, o2, M, 1, H, Hk, D, L, True, sp)
    torch.cuda.synchronize()
    assert_close(o2.cpu().numpy(), o1.cpu().numpy(), MAX_ABS)


def test_prefill_chunked_clamps_chunk_past_capacity(rkv, oracle_mod):
    """start + n > max_len: keys past max_len are not read and the clamp flag is raised."""
    torch = torch_cuda()
    rkv.rkv_read_device_flags(clear=True)
    M, T, H, Hk, D, L = 1, 10, 4, 2, 64, 140
    q = inputs.normal((M, T, H * D), 331)
    kc, vc = inputs.normal((M, Hk, L, D), 332), inputs.normal((M, Hk, L, D), 333)
    got = _chunked(rkv, torch, q, kc, vc, M, T, H, Hk, D, L, True, [134])
    assert rkv.rkv_read_device_flags(clear=True) & rkv.RKV_FLAG_LEN_CLAMPED
    # tokens 0..5 fit (positions 134..139); tokens 6..9 see the whole cache of 140 rows
    want = oracle_mod.prefill_cached(q[:, :6], kc, vc, M, 6, H, Hk, D, L, True, np.array([134]))
    assert_close(got[:, :6], want, MAX_ABS, MEAN_ABS)
    full = oracle_mod.decode(q[0, 6:], np.repeat(kc, 4, 0), np.repeat(vc, 4, 0), 4, H, Hk, D, L,
                             np.full(4, L))
    assert_close(got[0, 6:], full, MAX_ABS, MEAN_ABS)


def test_chunked_causal_gqa_second_half_sampled(rkv, oracle_mod):
    """The causal GQA workload (B=4, H=32, Hk=8, D=128) prefilled in two chunks of 1024 tokens
    into a [4,8,4096,128] cache: the second chunk equals rows 1024..2047 of the one-shot causal
    prefill (the oracle's chunk-composition pin), checked on sampled rows."""
    torch = torch_cuda()
    s = inputs.CAUSAL_GQA
    L, c = inputs.CAUSAL_GQA_CACHE_LEN, 1024
    q, k, v = inputs.prefill_inputs(s)
    dq, dk, dv = (torch.from_numpy(a).cuda() for a in (q, k, v))
    kc = torch.zeros((s.B, s.Hk, L, s.D), device="cuda")
    vc = torch.zeros_like(kc)
    rkv.kv_cache_scatter(dk, dv, kc, vc, s.B, s.S, s.Hk, s.D, L, torch.zeros(s.B, dtype=torch.int32, device="cuda"))
    o = torch.full((s.B, s.S - c, s.H * s.D), float("nan"), device="cuda")
    start = torch.full((s.B,), c, dtype=torch.int32, device="cuda")
    rkv.attn_prefill_chunked(dq[:, c:].contiguous(), kc, vc, o, s.B, s.S - c, s.H, s.Hk, s.D, L, True, start)
    torch.cuda.synchronize()
    got_all = o.cpu().numpy()
    assert np.all(np.isfinite(got_all))
    rows = set()
    for b in range(s.B):
        for h in (0, 3, 4, s.H - 1):
            for i in (c, c + 1, c + 127, c + 128, s.S - 1):
                rows.add((b * s.H + h) * s.S + i)
    rng_rows = inputs.sample_indices(s.B * s.H * (s.S - c), 300, 23)
    for r in rng_rows:
        bh, i = divmod(int(r), s.S - c)
        rows.add(bh * s.S + c + i)
    rows = np.array(sorted(rows), np.int64)
    want = oracle_mod.prefill_rows(q, k, v, s.B, s.S, s.H, s.Hk, s.D, True, rows)
    b, h, i = rows // (s.H * s.S), (rows // s.S) % s.H, rows % s.S
    got = np.stack([got_all[bb, ii - c, hh * s.D:(hh + 1) * s.D] for bb, hh, ii in zip(b, h, i)])
    assert_close(got, want, MAX_ABS, MEAN_ABS, what="chunked causal GQA sample")
