"""Every entry point through the checked build (device index checks compiled in), in a fresh
process: results match the oracle and no kernel computes an index outside its buffer
(RKV_FLAG_BOUNDS stays clear).  The cases reach the guarded paths: clamped, zero and negative
lengths and positions, a NULL per-sequence cache pointer, padded prefill rows, a chunk behind a
cache, the fused cache fill and the RoPE prologue."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import sys
sys.path.insert(0, ROOT)
import numpy as np, torch
import oracle
from resident_kv_cache_gb300 import binding as rkv, build, inputs
from tests.gpu_util import assert_close
rkv.LIB_PATH = build.CHECKED_LIB
rkv.load()
oracle.build()
dev = "cuda"
to = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
rkv.rkv_read_device_flags(clear=True)

def bounds_clear(what):
    f = rkv.rkv_read_device_flags(clear=True)
    assert not (f & rkv.RKV_FLAG_BOUNDS), f"{what}: RKV_FLAG_BOUNDS raised (flags {f:#x})"

# scatter: in range, overflowing and negative start positions
M, T, Hk, D, L = 3, 5, 2, 32, 8
kn, vn = inputs.normal((M, T, Hk * D), (70, 0)), inputs.normal((M, T, Hk * D), (70, 1))
kc, vc = inputs.normal((M, Hk, L, D), (70, 2)), inputs.normal((M, Hk, L, D), (70, 3))
sp = np.array([0, 6, -2], np.int32)
dk, dv = to(kc), to(vc)
ov = torch.zeros(1, dtype=torch.int32, device=dev)
rkv.kv_cache_scatter(to(kn), to(vn), dk, dv, M, T, Hk, D, L, to(sp), ov)
hk, hv, n_ov = oracle.scatter(kn, vn, kc, vc, M, T, Hk, D, L, sp)
torch.cuda.synchronize()
assert np.array_equal(dk.cpu().numpy(), hk) and np.array_equal(dv.cpu().numpy(), hv)
assert int(ov.item()) == n_ov
bounds_clear("kv_cache_scatter")

# decode: full, single, empty and clamped lengths; then the one-launch step
M, H, Hk, D, L = 4, 8, 2, 64, 300
q = inputs.normal((M, H * D), (71, 0))
kc, vc = inputs.normal((M, Hk, L, D), (71, 1)), inputs.normal((M, Hk, L, D), (71, 2))
lens = np.array([L, 1, 0, L + 5], np.int32)
n = rkv.attn_decode_workspace_bytes(M, H, Hk, D, L)
ws = torch.zeros(n, dtype=torch.uint8, device=dev)
o = torch.full((M, H * D), float("nan"), device=dev)
dk, dv = to(kc), to(vc)
rkv.attn_decode_batched(to(q), dk, dv, o, M, H, Hk, D, L, to(lens), 0.0, ws, n)
torch.cuda.synchronize()
assert_close(o.cpu().numpy(), oracle.decode(q, kc, vc, M, H, Hk, D, L, np.minimum(np.maximum(lens, 0), L)), 1e-4)
bounds_clear("attn_decode_batched")
lens2 = np.array([L, 2, 0, 150], np.int32)
kn, vn = inputs.normal((M, Hk * D), (71, 3)), inputs.normal((M, Hk * D), (71, 4))
rkv.attn_decode_append(to(q), to(kn), to(vn), dk, dv, o, M, H, Hk, D, L, to(lens2), 0.0, ws, n)
hk, hv, _ = oracle.scatter(kn[:, None], vn[:, None], kc, vc, M, 1, Hk, D, L, lens2 - 1)
torch.cuda.synchronize()
assert np.array_equal(dk.cpu().numpy(), hk) and np.array_equal(dv.cpu().numpy(), hv)
assert_close(o.cpu().numpy(), oracle.decode(q, hk, hv, M, H, Hk, D, L, lens2), 1e-4)
bounds_clear("attn_decode_append")

# per-sequence caches with a NULL entry
per = [to(np.ascontiguousarray(kc[m])) for m in range(M)], [to(np.ascontiguousarray(vc[m])) for m in range(M)]
kp = torch.tensor([t.data_ptr() for t in per[0]], dtype=torch.int64, device=dev)
vp = torch.tensor([t.data_ptr() for t in per[1]], dtype=torch.int64, device=dev)
kp[1] = 0
lens3 = np.array([L, 7, 3, 200], np.int32)
rkv.attn_decode_batched_ptrs(to(q), kp, vp, o, M, H, Hk, D, L, to(lens3), 0.0, ws, n)
torch.cuda.synchronize()
want = oracle.decode(q, kc, vc, M, H, Hk, D, L, np.where(np.arange(M) == 1, 0, lens3))
assert_close(o.cpu().numpy(), want, 1e-4)
f = rkv.rkv_read_device_flags(clear=True)
assert f & rkv.RKV_FLAG_BAD_POINTER and not (f & rkv.RKV_FLAG_BOUNDS), f

# RoPE prologue at mixed positions
M, T, H, Hk, D, L = 2, 3, 4, 2, 64, 16
qr, kr, vr = (inputs.normal((M, T, n * D), (72, i)) for i, n in enumerate((H, Hk, Hk)))
sp = np.array([0, 14], np.int32)
dq, dk_new = to(qr), to(kr)
kc, vc = torch.zeros((M, Hk, L, D), device=dev), torch.zeros((M, Hk, L, D), device=dev)
rkv.kv_append_rope(dq, dk_new, to(vr), kc, vc, M, T, H, Hk, D, L, to(sp), rotary_ndims=32)
torch.cuda.synchronize()
pos = (sp[:, None] + np.arange(T)[None, :]).reshape(-1)
assert_close(dq.cpu().numpy().reshape(M * T, H * D), oracle.rope(qr.reshape(M * T, H * D), H, D, pos, rotary_ndims=32), 1e-5)
bounds_clear("kv_append_rope")

# prefill with per-sequence lengths (a zero length: padded rows), chunked, fused fill
B, S, H, Hk, D = 3, 130, 4, 2, 64
q, k, v = (inputs.normal((B, S, n * D), (73, i)) for i, n in enumerate((H, Hk, Hk)))
sl = np.array([130, 0, 77], np.int32)
o = torch.full((B, S, H * D), float("nan"), device=dev)
rkv.attn_prefill(to(q), to(k), to(v), o, B, S, H, Hk, D, True, to(sl))
torch.cuda.synchronize()
assert_close(o.cpu().numpy(), oracle.prefill(q, k, v, B, S, H, Hk, D, True, seq_lens=sl), 3e-3, 1e-3)
bounds_clear("attn_prefill")
L = 256
kcache, vcache = torch.zeros((B, Hk, L, D), device=dev), torch.zeros((B, Hk, L, D), device=dev)
o2 = torch.empty((B, S, H * D), device=dev)
rkv.attn_prefill_fill_cache(to(q), to(k), to(v), o2, B, S, H, Hk, D, True, kcache, vcache, L)
torch.cuda.synchronize()
assert np.array_equal(kcache[:, :, :S].cpu().numpy(), k.reshape(B, S, Hk, D).transpose(0, 2, 1, 3))
bounds_clear("attn_prefill_fill_cache")
p0 = np.array([100, 0, 30], np.int32)
qc = inputs.normal((B, 20, H * D), (73, 9))
oc = torch.empty((B, 20, H * D), device=dev)
rkv.attn_prefill_chunked(to(qc), kcache, vcache, oc, B, 20, H, Hk, D, L, True, to(p0))
torch.cuda.synchronize()
want = oracle.prefill_cached(qc, kcache.cpu().numpy(), vcache.cpu().numpy(), B, 20, H, Hk, D, L, True, p0)
assert_close(oc.cpu().numpy(), want, 3e-3, 1e-3)
bounds_clear("attn_prefill_chunked")

# the same three at head_dim 128 with pairs of query heads per kv head (the CTA-pair kernel)
B, S, H, Hk, D = 3, 130, 4, 2, 128
q, k, v = (inputs.normal((B, S, n * D), (74, i)) for i, n in enumerate((H, Hk, Hk)))
o = torch.full((B, S, H * D), float("nan"), device=dev)
rkv.attn_prefill(to(q), to(k), to(v), o, B, S, H, Hk, D, True, to(sl))
torch.cuda.synchronize()
assert_close(o.cpu().numpy(), oracle.prefill(q, k, v, B, S, H, Hk, D, True, seq_lens=sl), 3e-3, 1e-3)
bounds_clear("attn_prefill (pair)")
kcache, vcache = torch.zeros((B, Hk, L, D), device=dev), torch.zeros((B, Hk, L, D), device=dev)
o2 = torch.empty((B, S, H * D), device=dev)
rkv.attn_prefill_fill_cache(to(q), to(k), to(v), o2, B, S, H, Hk, D, True, kcache, vcache, L)
torch.cuda.synchronize()
assert np.array_equal(kcache[:, :, :S].cpu().numpy(), k.reshape(B, S, Hk, D).transpose(0, 2, 1, 3))
assert_close(o2.cpu().numpy(), oracle.prefill(q, k, v, B, S, H, Hk, D, True), 3e-3, 1e-3)
bounds_clear("attn_prefill_fill_cache (pair)")
qc = inputs.normal((B, 20, H * D), (74, 9))
oc = torch.empty((B, 20, H * D), device=dev)
rkv.attn_prefill_chunked(to(qc), kcache, vcache, oc, B, 20, H, Hk, D, L, True, to(p0))
torch.cuda.synchronize()
want = oracle.prefill_cached(qc, kcache.cpu().numpy(), vcache.cpu().numpy(), B, 20, H, Hk, D, L, True, p0)
assert_close(oc.cpu().numpy(), want, 3e-3, 1e-3)
bounds_clear("attn_prefill_chunked (pair)")
print("CHECKED BUILD OK")
'''


@pytest.mark.gpu
def test_every_entry_point_through_the_checked_build():
    from tests.gpu_util import torch_cuda
    torch_cuda()
    from resident_kv_cache_gb300 import build
    build.build(checked=True)
    r = subprocess.run([sys.executable, "-c", f"ROOT = {ROOT!r}\n" + CHILD], capture_output=True, text=True,
                       cwd=ROOT, timeout=600)
    assert r.returncode == 0 and "CHECKED BUILD OK" in r.stdout, r.stdout[-3000:] + r.stderr[-3000:]
