"""Per-sequence caches through pointer arrays (attn_decode_batched_ptrs, kv_cache_scatter_ptrs).

realizar cache_from_cache_from_kv_cache.rs keeps device arrays of per-sequence K and V
pointers (batched_k_ptrs / batched_v_ptrs) for batched attention; each sequence's cache
[n_kv_heads, max_len, head_dim] may then live anywhere.  The pointer-array entries run the
same kernels as the batched-cache entries, so results must be identical to them bit for bit
(and to the oracle within 1e-4 / exactly for the scatter).  Rollback (realizar
fn rollback_kv_cache_gpu) is a shorter seq_lens and needs no kernel.
"""
import numpy as np
import pytest

from resident_kv_cache_gb300 import inputs
from tests.gpu_util import assert_close, torch_cuda

pytestmark = pytest.mark.gpu


def _scattered_caches(torch, kc, vc):
    """One allocation per sequence (with allocations of other sizes in between), as separate tensors."""
    keep, ks, vs = [], [], []
    for m in range(kc.shape[0]):
        keep.append(torch.empty(4096 * (m + 1), device="cuda"))        # spacers
        ks.append(torch.from_numpy(np.ascontiguousarray(kc[m])).cuda())
        keep.append(torch.empty(1000 + 64 * m, device="cuda"))
        vs.append(torch.from_numpy(np.ascontiguousarray(vc[m])).cuda())
    kp = torch.tensor([t.data_ptr() for t in ks], dtype=torch.int64, device="cuda")
    vp = torch.tensor([t.data_ptr() for t in vs], dtype=torch.int64, device="cuda")
    return ks, vs, kp, vp, keep


def test_decode_ptrs_equals_batched_decode(rkv, oracle_mod):
    torch = torch_cuda()
    M, H, Hk, D, L = 6, 32, 8, 128, 700
    lens = np.array([700, 1, 350, 0, 699, 64], np.int32)
    q = inputs.normal((M, H * D), 401)
    kc, vc = inputs.normal((M, Hk, L, D), 402), inputs.normal((M, Hk, L, D), 403)
    ks, vs, kp, vp, keep = _scattered_caches(torch, kc, vc)
    dq = torch.from_numpy(q).cuda()
    ln = torch.from_numpy(lens).cuda()
    n = rkv.attn_decode_workspace_bytes(M, H, Hk, D, L)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    o1 = torch.empty((M, H * D), device="cuda")
    o2 = torch.empty((M, H * D), device="cuda")
    rkv.attn_decode_batched(dq, torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda(), o1, M, H, Hk, D, L, ln, 0.0,
                            ws, n)
    rkv.attn_decode_batched_ptrs(dq, kp, vp, o2, M, H, Hk, D, L, ln, 0.0, ws, n)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)
    assert_close(o2.cpu().numpy(), oracle_mod.decode(q, kc, vc, M, H, Hk, D, L, lens), 1e-4)


def test_scatter_ptrs_then_decode_and_rollback(rkv, oracle_mod):
    """Append 5 tokens per sequence into separate caches, decode over them, then roll two
    sequences back (shorter lengths) and decode again: rows past the lengths are ignored."""
    torch = torch_cuda()
    M, H, Hk, D, L, T = 4, 16, 4, 64, 256, 5
    base = np.array([10, 0, 200, 251], np.int32)              # 251 + 5 = 256: the last one ends at the capacity
    kc, vc = inputs.normal((M, Hk, L, D), 411), inputs.normal((M, Hk, L, D), 412)
    kn, vn = inputs.normal((M, T, Hk * D), 413), inputs.normal((M, T, Hk * D), 414)
    q = inputs.normal((M, H * D), 415)
    ks, vs, kp, vp, keep = _scattered_caches(torch, kc, vc)
    rkv.kv_cache_scatter_ptrs(torch.from_numpy(kn).cuda(), torch.from_numpy(vn).cuda(), kp, vp, M, T, Hk, D, L,
                              torch.from_numpy(base).cuda())
    hk, hv, ov = oracle_mod.scatter(kn, vn, kc, vc, M, T, Hk, D, L, base)
    torch.cuda.synchronize()
    for m in range(M):
        assert np.array_equal(ks[m].cpu().numpy(), hk[m]) and np.array_equal(vs[m].cpu().numpy(), hv[m])
    n = rkv.attn_decode_workspace_bytes(M, H, Hk, D, L)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    dq = torch.from_numpy(q).cuda()
    for lens in (base + T, np.array([12, 5, 201, 256], np.int32)):      # full, then rolled back
        o = torch.empty((M, H * D), device="cuda")
        rkv.attn_decode_batched_ptrs(dq, kp, vp, o, M, H, Hk, D, L, torch.from_numpy(lens).cuda(), 0.0, ws, n)
        torch.cuda.synchronize()
        assert_close(o.cpu().numpy(), oracle_mod.decode(q, hk, hv, M, H, Hk, D, L, lens), 1e-4)


def test_bad_pointer_entries_are_skipped_and_flagged(rkv, oracle_mod):
    """A NULL entry and an entry 4 bytes into a valid allocation (not 16-byte aligned) are never
    dereferenced: those sequences give zero rows (decode) or are left alone (scatter), the others
    are exact, and the device flag says so."""
    torch = torch_cuda()
    rkv.rkv_read_device_flags(clear=True)
    M, H, Hk, D, L = 3, 8, 2, 64, 128
    kc, vc = inputs.normal((M, Hk, L, D), 421), inputs.normal((M, Hk, L, D), 422)
    ks, vs, kp, vp, keep = _scattered_caches(torch, kc, vc)
    kp_bad = kp.clone()
    kp_bad[0] = 0                                              # NULL
    kp_bad[2] = ks[2].data_ptr() + 4                           # misaligned, inside a valid allocation
    lens = np.array([100, 128, 50], np.int32)
    q = inputs.normal((M, H * D), 423)
    n = rkv.attn_decode_workspace_bytes(M, H, Hk, D, L)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    o = torch.full((M, H * D), float("nan"), device="cuda")
    rkv.attn_decode_batched_ptrs(torch.from_numpy(q).cuda(), kp_bad, vp, o, M, H, Hk, D, L,
                                 torch.from_numpy(lens).cuda(), 0.0, ws, n)
    torch.cuda.synchronize()
    assert rkv.rkv_read_device_flags(clear=True) & rkv.RKV_FLAG_BAD_POINTER
    got = o.cpu().numpy()
    assert np.all(got[0] == 0.0) and np.all(got[2] == 0.0)
    assert_close(got[1:2], oracle_mod.decode(q, kc, vc, M, H, Hk, D, L, lens)[1:2], 1e-4)
    kn = inputs.normal((M, 1, Hk * D), 424)
    rkv.kv_cache_scatter_ptrs(torch.from_numpy(kn).cuda(), torch.from_numpy(kn).cuda(), kp_bad, vp, M, 1, Hk, D, L,
                              torch.from_numpy(lens).cuda())
    torch.cuda.synchronize()
    assert rkv.rkv_read_device_flags(clear=True) & rkv.RKV_FLAG_BAD_POINTER
    assert np.array_equal(ks[0].cpu().numpy(), kc[0]) and np.array_equal(ks[2].cpu().numpy(), kc[2])
    assert np.array_equal(vs[0].cpu().numpy(), vc[0]) and np.array_equal(vs[2].cpu().numpy(), vc[2])
    # sequence 1 got its row at position lens[1] = 128 -> outside the cache: nothing written there either
    assert np.array_equal(ks[1].cpu().numpy(), kc[1])
