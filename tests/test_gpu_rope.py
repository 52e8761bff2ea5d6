"""Rotary position embedding fused with the append (kv_append_rope) on the GPU against the oracle.

GPT-NeoX half-split RoPE: trustformers-core attention.rs, fn rope_neox_gpu_to_gpu (partial, at a
position offset) and realizar cache_from_cache_from_kv_cache.rs, fn apply_rope_to_buffer.
Rotated q and k match the f64 oracle within 1e-5 abs on N(0,1) inputs (f32 products and a
float sincos of an angle reduced in double); the cache receives exactly the rotated k the call
leaves in k_new and the v rows bit for bit.  A decode step and a prefill with the RoPE prologue
then match the oracle within their attention tolerances.
"""
import numpy as np
import pytest

from resident_kv_cache_gb300 import inputs
from tests.gpu_util import Guarded, assert_close, torch_cuda

pytestmark = pytest.mark.gpu
ROPE_TOL = 1e-5
FILL = np.float32(3.25e30)

CASES = [
    # M, T, H, Hk, D, L, rotary, theta, start_pos
    (1, 1, 1, 1, 16, 4, 16, 1e4, [2]),
    (2, 5, 4, 2, 32, 64, 32, 1e4, [0, 59]),
    (3, 7, 8, 2, 64, 40, 32, 1e6, [3, 33, 38]),      # partial rotary; two tokens past the cache
    (2, 3, 32, 8, 128, 32768, 128, 1e6, [32765, 20000]),
    (4, 1, 32, 8, 128, 4096, 128, 1e4, [0, 1, 2047, 4095]),
    (1, 130, 16, 4, 128, 300, 64, 1e4, [100]),
]


@pytest.mark.parametrize("ci", range(len(CASES)))
def test_kv_append_rope_matches_oracle(rkv, oracle_mod, ci):
    torch = torch_cuda()
    M, T, H, Hk, D, L, r, theta, sp = CASES[ci]
    q = inputs.normal((M, T, H * D), (ci, 60))
    kn = inputs.normal((M, T, Hk * D), (ci, 61))
    vn = inputs.normal((M, T, Hk * D), (ci, 62))
    g_q, g_k, g_v = Guarded(torch, q), Guarded(torch, kn), Guarded(torch, vn)
    g_kc = Guarded(torch, np.full((M, Hk, L, D), FILL, np.float32))
    g_vc = Guarded(torch, np.full((M, Hk, L, D), FILL, np.float32))
    g_sp = Guarded(torch, np.array(sp, np.int32), np.int32)
    g_ov = Guarded(torch, np.zeros(1, np.int32), np.int32)
    rkv.kv_append_rope(g_q.t, g_k.t, g_v.t, g_kc.t, g_vc.t, M, T, H, Hk, D, L, g_sp.t, rotary_ndims=r, theta=theta,
                       overflow=g_ov.t)
    torch.cuda.synchronize()
    for g in (g_q, g_k, g_v, g_kc, g_vc):
        assert g.guards_intact()
    pos = (np.array(sp)[:, None] + np.arange(T)[None, :]).reshape(-1)
    want_q = oracle_mod.rope(q.reshape(M * T, H * D), H, D, pos, theta=theta, rotary_ndims=r).reshape(q.shape)
    want_k = oracle_mod.rope(kn.reshape(M * T, Hk * D), Hk, D, pos, theta=theta, rotary_ndims=r).reshape(kn.shape)
    got_q, got_k = g_q.numpy(), g_k.numpy()
    assert_close(got_q, want_q, ROPE_TOL, what="q")
    assert_close(got_k, want_k, ROPE_TOL, what="k")
    assert np.array_equal(g_v.numpy(), vn)
    # the cache holds the rotated k the call left in k_new, and v, at rows start_pos + t < L
    hk, hv, ov = oracle_mod.scatter(got_k, vn, np.full((M, Hk, L, D), FILL, np.float32),
                                    np.full((M, Hk, L, D), FILL, np.float32), M, T, Hk, D, L, np.array(sp, np.int32))
    assert np.array_equal(g_kc.numpy(), hk) and np.array_equal(g_vc.numpy(), hv)
    assert int(g_ov.numpy()[0]) == ov


def test_decode_step_with_rope_prologue(rkv, oracle_mod):
    """Append with RoPE at len-1, then decode over len rows; the oracle rotates q and the new k at
    len-1, scatters, and decodes (the batched decode workload's shapes, smaller cache)."""
    torch = torch_cuda()
    M, H, Hk, D, L = 8, 32, 8, 128, 1024
    lens = inputs.uniform_lengths(M, 1, L, 77)
    q = inputs.normal((M, 1, H * D), 70)
    kn = inputs.normal((M, 1, Hk * D), 71)
    vn = inputs.normal((M, 1, Hk * D), 72)
    kc0 = inputs.normal((M, Hk, L, D), 73)
    vc0 = inputs.normal((M, Hk, L, D), 74)
    dq, dk, dv = (torch.from_numpy(a).cuda() for a in (q, kn, vn))
    kc, vc = torch.from_numpy(kc0).cuda(), torch.from_numpy(vc0).cuda()
    sp = torch.from_numpy((lens - 1).astype(np.int32)).cuda()
    ln = torch.from_numpy(lens).cuda()
    rkv.kv_append_rope(dq, dk, dv, kc, vc, M, 1, H, Hk, D, L, sp, theta=1e6)
    n = rkv.attn_decode_workspace_bytes(M, H, Hk, D, L)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    o = torch.empty((M, H * D), device="cuda")
    rkv.attn_decode_batched(dq.view(M, H * D), kc, vc, o, M, H, Hk, D, L, ln, 0.0, ws, n)
    torch.cuda.synchronize()
    qr = oracle_mod.rope(q.reshape(M, H * D), H, D, lens - 1, theta=1e6).astype(np.float32)
    kr = oracle_mod.rope(kn.reshape(M, Hk * D), Hk, D, lens - 1, theta=1e6).astype(np.float32)
    hk, hv, _ = oracle_mod.scatter(kr.reshape(M, 1, Hk * D), vn, kc0, vc0, M, 1, Hk, D, L, lens - 1)
    want = oracle_mod.decode(qr, hk, hv, M, H, Hk, D, L, lens)
    assert_close(o.cpu().numpy(), want, 1e-4, what="decode with RoPE")


def test_prefill_with_rope_prologue(rkv, oracle_mod):
    """kv_append_rope over the whole sequence (start 0) then attn_prefill on the rotated q, k equals
    the oracle prefill of rope(q), rope(k) within the prefill tolerance; the cache holds rope(k)."""
    torch = torch_cuda()
    B, S, H, Hk, D, L = 2, 300, 16, 4, 128, 512
    q, k, v = (inputs.normal((B, S, n * D), (80, t)) for t, n in enumerate((H, Hk, Hk)))
    dq, dk, dv = (torch.from_numpy(a).cuda() for a in (q, k, v))
    kc = torch.zeros((B, Hk, L, D), device="cuda")
    vc = torch.zeros_like(kc)
    zero = torch.zeros(B, dtype=torch.int32, device="cuda")
    rkv.kv_append_rope(dq, dk, dv, kc, vc, B, S, H, Hk, D, L, zero, theta=1e4)
    o = torch.empty((B, S, H * D), device="cuda")
    rkv.attn_prefill(dq, dk, dv, o, B, S, H, Hk, D, True)
    torch.cuda.synchronize()
    pos = np.tile(np.arange(S), B)
    qr = oracle_mod.rope(q.reshape(B * S, H * D), H, D, pos).astype(np.float32).reshape(q.shape)
    kr = oracle_mod.rope(k.reshape(B * S, Hk * D), Hk, D, pos).astype(np.float32).reshape(k.shape)
    want = oracle_mod.prefill(qr, kr, v, B, S, H, Hk, D, True)
    assert_close(o.cpu().numpy(), want, 3e-3, 1e-3, what="prefill with RoPE")
    assert np.array_equal(kc.cpu().numpy()[:, :, :S, :], dk.cpu().numpy().reshape(B, S, Hk, D).transpose(0, 2, 1, 3))


def test_decode_step_with_rope_prologue_full_size(rkv, oracle_mod):
    """The batched decode step with the RoPE prologue exactly as it is timed: the batched decode
    workload's inputs (M=32, H=32, Hk=8, D=128, cache [32,8,4096,128], lengths U{1..4096}),
    kv_append_rope at len-1 (theta 1e6, every dim rotated), then attn_decode_batched over len rows;
    the whole output against the oracle and the caches bit for bit."""
    torch = torch_cuda()
    d = inputs.BATCHED_DECODE
    x = inputs.batched_decode_inputs(d)
    M, H, Hk, D, L = d.M, d.H, d.Hk, d.D, d.Lmax
    dq = torch.from_numpy(x["q"]).cuda()
    dk = torch.from_numpy(x["k_new"]).cuda()
    dv = torch.from_numpy(x["v_new"]).cuda()
    kc, vc = torch.from_numpy(x["k_cache"]).cuda(), torch.from_numpy(x["v_cache"]).cuda()
    sp, ln = torch.from_numpy(x["start_pos"]).cuda(), torch.from_numpy(x["lens"]).cuda()
    rkv.kv_append_rope(dq, dk, dv, kc, vc, M, 1, H, Hk, D, L, sp, theta=1e6)
    n = rkv.attn_decode_workspace_bytes(M, H, Hk, D, L)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    o = torch.full((M, H * D), float("nan"), device="cuda")
    rkv.attn_decode_batched(dq, kc, vc, o, M, H, Hk, D, L, ln, 0.0, ws, n)
    torch.cuda.synchronize()
    pos = x["start_pos"]
    qr = oracle_mod.rope(x["q"], H, D, pos, theta=1e6).astype(np.float32)
    kr = oracle_mod.rope(x["k_new"].reshape(M, Hk * D), Hk, D, pos, theta=1e6).astype(np.float32)
    assert np.abs(dq.cpu().numpy() - qr).max() <= 1e-5
    # the cache receives exactly the rotated k the call left in k_new
    hk, hv, _ = oracle_mod.scatter(dk.cpu().numpy(), x["v_new"], x["k_cache"], x["v_cache"], M, 1, Hk, D, L, pos)
    assert np.array_equal(kc.cpu().numpy(), hk) and np.array_equal(vc.cpu().numpy(), hv)
    assert np.abs(dk.cpu().numpy().reshape(M, Hk * D) - kr).max() <= 1e-5
    want = oracle_mod.decode(qr, hk, hv, M, H, Hk, D, L, x["lens"])
    assert_close(o.cpu().numpy(), want, 1e-4, what="decode step with RoPE, full size")
