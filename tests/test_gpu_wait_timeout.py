"""The failure path of the kernels' on-chip waits, exercised without a fault.

Every mbarrier wait in the kernels is bounded; on expiry the kernel sets RKV_FLAG_WAIT_TIMEOUT,
unwinds and returns.  rkv_check_wait_timeout runs that same bounded wait on a barrier that
nothing completes: the wait must give up after its limit, raise the flag, and leave the context
usable for the next call.
"""
import time

import numpy as np
import pytest

from resident_kv_cache_gb300 import inputs
from tests.gpu_util import assert_close, torch_cuda

pytestmark = pytest.mark.gpu


def test_wait_gives_up_raises_the_flag_and_the_context_survives(rkv, oracle_mod):
    torch = torch_cuda()
    rkv.rkv_read_device_flags(clear=True)
    limit_us = 20000
    t0 = time.perf_counter()
    rkv.rkv_check_wait_timeout(limit_us)
    flags = rkv.rkv_read_device_flags(clear=True)            # synchronises
    elapsed = time.perf_counter() - t0
    assert flags & rkv.RKV_FLAG_WAIT_TIMEOUT
    assert limit_us * 1e-6 <= elapsed < 2.0                   # gave up after the limit, not later
    assert rkv.rkv_read_device_flags() == 0                   # the flag was cleared

    # the context is still usable: a decode right after is correct and raises no flag
    M, H, Hk, D, L, lens = 3, 8, 2, 64, 200, [200, 1, 77]
    q = inputs.normal((M, H * D), (5, 800))
    kc = inputs.normal((M, Hk, L, D), (5, 801))
    vc = inputs.normal((M, Hk, L, D), (5, 802))
    dq, dk, dv = (torch.from_numpy(a).cuda() for a in (q, kc, vc))
    o = torch.empty((M, H * D), device="cuda")
    ln = torch.tensor(lens, dtype=torch.int32, device="cuda")
    n = rkv.attn_decode_workspace_bytes(M, H, Hk, D, L)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    rkv.attn_decode_batched(dq, dk, dv, o, M, H, Hk, D, L, ln, 0.0, ws, n)
    assert rkv.rkv_read_device_flags(clear=True) == 0
    assert_close(o.cpu().numpy(), oracle_mod.decode(q, kc, vc, M, H, Hk, D, L, np.array(lens)), 1e-4)
