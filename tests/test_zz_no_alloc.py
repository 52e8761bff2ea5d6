"""The allocation-free decode entry point against the regular one.

attn_decode_batched_noalloc exists for callers that cannot allocate device
memory while decoding (an allocator they do not own, a host that forbids
allocation after start-up, a loop that must not block in cudaMalloc); it uses a
fixed scratch array inside the library instead of a caller workspace.  These
tests call it through the C ABI and compare it with attn_decode_batched on the
same inputs, twice in a row, since the shared array keeps the previous call's
contents.  The file is named to be collected last.
"""
import numpy as np
import pytest

from resident_kv_cache_gb300 import inputs
from tests.gpu_util import assert_close, torch_cuda

TOL = 1e-4   # the decode tolerance the other decode tests use


def _inputs(torch, M, H, Hk, D, L, lens, seed):
    q = torch.from_numpy(inputs.normal((M, H * D), (seed, 0))).cuda()
    kc = torch.from_numpy(inputs.normal((M, Hk, L, D), (seed, 1))).cuda()
    vc = torch.from_numpy(inputs.normal((M, Hk, L, D), (seed, 2))).cuda()
    ln = torch.from_numpy(np.asarray(lens, np.int32)).cuda()
    return q, kc, vc, ln


@pytest.mark.gpu
@pytest.mark.parametrize("M,H,Hk,D,L,lens", [
    (32, 32, 8, 128, 4096, None),                 # the batched decode workload's shape
    (3, 8, 2, 64, 700, [700, 1, 333]),
    (2, 4, 4, 16, 50, [0, 50]),
])
def test_noalloc_matches_workspace_entry_point_twice(rkv, oracle_mod, M, H, Hk, D, L, lens):
    """Same kernel, same arithmetic, same split of the rows: the output must equal
    attn_decode_batched's bit for bit, on both calls, and match the oracle."""
    torch = torch_cuda()
    rkv.rkv_read_device_flags(clear=True)   # flags left by earlier tests
    if lens is None:
        lens = inputs.uniform_lengths(M, 1, L, inputs.SEED_LEN)
    q, kc, vc, ln = _inputs(torch, M, H, Hk, D, L, lens, seed=M + D)
    n = rkv.attn_decode_workspace_bytes(M, H, Hk, D, L)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    ref = torch.empty((M, H * D), device="cuda")
    rkv.attn_decode_batched(q, kc, vc, ref, M, H, Hk, D, L, ln, 0.0, ws, n)
    torch.cuda.synchronize()
    want = oracle_mod.decode(q.cpu().numpy(), kc.cpu().numpy(), vc.cpu().numpy(), M, H, Hk, D, L,
                             np.asarray(lens, np.int32))
    for call in range(2):
        out = torch.full((M, H * D), float("nan"), device="cuda")
        rkv.attn_decode_batched_noalloc(q, kc, vc, out, M, H, Hk, D, L, ln, 0.0)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"call {call}: differs from attn_decode_batched"
        assert_close(out.cpu().numpy(), want, TOL, what=f"call {call} against the oracle")
    assert rkv.rkv_read_device_flags(clear=True) == 0


@pytest.mark.gpu
def test_noalloc_rejects_sizes_beyond_its_scratch(rkv):
    torch_cuda()
    # 32 sequences x 64 kv heads x group 8 at head_dim 128 need far more than 4 MiB of scratch
    need = rkv.attn_decode_workspace_bytes(32, 512, 64, 128, 1024)
    assert need > 4 << 20
    with pytest.raises(rkv.RkvError) as e:
        rkv.attn_decode_batched_noalloc(16, 16, 16, 32, 32, 512, 64, 128, 1024, 16, 0.0)
    assert e.value.status == rkv.RKV_ERR_UNSUPPORTED
    assert "scratch" in e.value.message
