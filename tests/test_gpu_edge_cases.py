"""Degenerate batches on the GPU: every sequence empty.

With no valid row anywhere the split-KV decode has nothing to partition (R = 0 rows), the
prefill has no visible key for any query, and the one-launch decode step has no row to append.
Every output row must be exact zeros, the caches untouched, and no device flag raised (an empty
sequence is valid input, not a clamped or negative one).
"""
import numpy as np
import pytest

from resident_kv_cache_gb300 import inputs
from tests.gpu_util import torch_cuda

pytestmark = pytest.mark.gpu


def _nan_like(torch, shape):
    return torch.full(shape, float("nan"), device="cuda")


def test_decode_all_sequences_empty(rkv):
    torch = torch_cuda()
    M, H, Hk, D, L = 4, 16, 4, 128, 64
    q = torch.from_numpy(inputs.normal((M, H * D), (1, 900))).cuda()
    kc = torch.from_numpy(inputs.normal((M, Hk, L, D), (1, 901))).cuda()
    vc = torch.from_numpy(inputs.normal((M, Hk, L, D), (1, 902))).cuda()
    o = _nan_like(torch, (M, H * D))
    lens = torch.zeros(M, dtype=torch.int32, device="cuda")
    n = rkv.attn_decode_workspace_bytes(M, H, Hk, D, L)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    rkv.rkv_read_device_flags(clear=True)
    rkv.attn_decode_batched(q, kc, vc, o, M, H, Hk, D, L, lens, 0.0, ws, n)
    assert rkv.rkv_read_device_flags(clear=True) == 0
    assert torch.count_nonzero(o).item() == 0 and not torch.isnan(o).any().item()


def test_decode_step_all_sequences_empty_appends_nothing(rkv):
    torch = torch_cuda()
    M, H, Hk, D, L = 3, 8, 2, 64, 50
    q = torch.from_numpy(inputs.normal((M, H * D), (2, 900))).cuda()
    kn = torch.from_numpy(inputs.normal((M, Hk * D), (2, 901))).cuda()
    vn = torch.from_numpy(inputs.normal((M, Hk * D), (2, 902))).cuda()
    kc = torch.from_numpy(inputs.normal((M, Hk, L, D), (2, 903))).cuda()
    vc = torch.from_numpy(inputs.normal((M, Hk, L, D), (2, 904))).cuda()
    k0, v0 = kc.clone(), vc.clone()
    o = _nan_like(torch, (M, H * D))
    lens = torch.zeros(M, dtype=torch.int32, device="cuda")
    n = rkv.attn_decode_workspace_bytes(M, H, Hk, D, L)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    rkv.rkv_read_device_flags(clear=True)
    rkv.attn_decode_append(q, kn, vn, kc, vc, o, M, H, Hk, D, L, lens, 0.0, ws, n)
    assert rkv.rkv_read_device_flags(clear=True) == 0
    assert torch.equal(kc, k0) and torch.equal(vc, v0)
    assert torch.count_nonzero(o).item() == 0 and not torch.isnan(o).any().item()


@pytest.mark.parametrize("D", [64, 128])
def test_prefill_all_sequences_empty(rkv, D):
    torch = torch_cuda()
    B, S, H, Hk = 2, 150, 4, 2
    q = torch.from_numpy(inputs.normal((B, S, H * D), (3, 900))).cuda()
    k = torch.from_numpy(inputs.normal((B, S, Hk * D), (3, 901))).cuda()
    v = torch.from_numpy(inputs.normal((B, S, Hk * D), (3, 902))).cuda()
    o = _nan_like(torch, (B, S, H * D))
    lens = torch.zeros(B, dtype=torch.int32, device="cuda")
    rkv.rkv_read_device_flags(clear=True)
    rkv.attn_prefill(q, k, v, o, B, S, H, Hk, D, True, lens)
    assert rkv.rkv_read_device_flags(clear=True) == 0
    assert torch.count_nonzero(o).item() == 0 and not torch.isnan(o).any().item()


def test_chunked_prefill_all_chunks_empty(rkv):
    torch = torch_cuda()
    M, T, H, Hk, D, L = 2, 70, 8, 2, 128, 300
    q = torch.from_numpy(inputs.normal((M, T, H * D), (4, 900))).cuda()
    kc = torch.from_numpy(inputs.normal((M, Hk, L, D), (4, 901))).cuda()
    vc = torch.from_numpy(inputs.normal((M, Hk, L, D), (4, 902))).cuda()
    o = _nan_like(torch, (M, T, H * D))
    start = torch.tensor([0, 200], dtype=torch.int32, device="cuda")
    q_lens = torch.zeros(M, dtype=torch.int32, device="cuda")
    rkv.rkv_read_device_flags(clear=True)
    rkv.attn_prefill_chunked(q, kc, vc, o, M, T, H, Hk, D, L, True, start, q_lens, 0.0)
    assert rkv.rkv_read_device_flags(clear=True) == 0
    assert torch.count_nonzero(o).item() == 0 and not torch.isnan(o).any().item()
