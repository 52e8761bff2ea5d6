"""The CTA-pair prefill (head_dim 128, an even number of query heads per kv head) against the
oracle.

Two CTAs of a cluster take two query heads of one kv group over the same 128-query tile and
share every tensor-core product, so the cases here vary what that pairing depends on: the group
size (2, 6, 8: one, three and four head pairs per kv head), sequence lengths that end anywhere in
a tile, per-sequence lengths with empty and one-token sequences (whole tiles without keys), the
fused cache fill, and a launch with more work items than resident pairs.  Odd group sizes and
other head sizes take the single-CTA kernel; one such case runs beside them as a control.
Tolerance as for every prefill test: 3e-3 max abs, 1e-3 mean abs (TF32 products, f32 sums).
Semantics: trueno-gpu attention.rs, fn batched_multihead_attention_optimized, and
trustformers-core attention.rs, fn attention_prefill_gpu_to_gpu.
"""
import numpy as np
import pytest

from resident_kv_cache_gb300 import inputs
from tests.gpu_util import assert_close, torch_cuda
from tests.test_gpu_prefill import _prefill

pytestmark = pytest.mark.gpu
MAX_ABS, MEAN_ABS = 3e-3, 1e-3

CASES = [
    # B, S, H, Hk, causal, seq_lens          (head_dim 128 throughout)
    (1, 1, 2, 1, True, None),                # one query, one key
    (1, 127, 2, 1, True, None),              # one tile, one row short
    (2, 128, 4, 2, False, None),             # exactly one tile
    (1, 129, 12, 2, True, None),             # group 6: three pairs per kv head; ragged second tile
    (2, 300, 8, 1, False, None),             # group 8, non-causal, ragged third tile
    (3, 257, 4, 2, True, [257, 0, 1]),       # an empty and a one-token sequence
    (2, 384, 16, 2, True, [200, 384]),       # padded rows inside the last tiles
    (1, 300, 6, 2, True, None),              # group 3 (odd): the single-CTA kernel, as a control
]


@pytest.mark.parametrize("ci", range(len(CASES)))
def test_pair_prefill_matches_oracle(rkv, oracle_mod, ci):
    torch = torch_cuda()
    B, S, H, Hk, causal, lens = CASES[ci]
    D = 128
    q = inputs.normal((B, S, H * D), (ci, 810))
    k = inputs.normal((B, S, Hk * D), (ci, 811))
    v = inputs.normal((B, S, Hk * D), (ci, 812))
    got = _prefill(rkv, torch, q, k, v, B, S, H, Hk, D, causal, lens)
    want = oracle_mod.prefill(q, k, v, B, S, H, Hk, D, causal, seq_lens=lens)
    assert_close(got, want, MAX_ABS, MEAN_ABS, what=f"case {ci}")
    if lens is not None:          # padded query rows are exactly zero
        for b, n in enumerate(lens):
            assert np.all(got[b, n:] == 0.0)


def test_pair_prefill_more_items_than_pairs(rkv, oracle_mod):
    """B=2, S=1024, H=16, Hk=2 (group 8): 8 tiles x 2 x 2 kv heads x 4 head pairs = 128 work items,
    more than the 76 pairs that fit on the GPU, so clusters walk several items each, heaviest
    first, and rings and barrier phases run on from item to item.  Whole output checked."""
    torch = torch_cuda()
    B, S, H, Hk, D = 2, 1024, 16, 2, 128
    q, k, v = (inputs.normal((B, S, n * D), (40, t)) for t, n in enumerate((H, Hk, Hk)))
    got = _prefill(rkv, torch, q, k, v, B, S, H, Hk, D, True)
    want = oracle_mod.prefill(q, k, v, B, S, H, Hk, D, True)
    mx = assert_close(got, want, MAX_ABS, MEAN_ABS, what="more items than pairs")
    print(f"max abs {mx:.3e}")


def test_pair_prefill_heads_of_a_pair_are_independent(rkv, oracle_mod):
    """The two heads of a pair share K and V but not Q: a query head whose input is all zeros
    sees uniform weights (the mean of the visible V rows) while its partner is unaffected."""
    torch = torch_cuda()
    B, S, H, Hk, D = 1, 200, 2, 1, 128
    q = inputs.normal((B, S, H * D), (41, 0))
    q[:, :, D:] = 0.0                       # head 1: zero queries
    k, v = (inputs.normal((B, S, Hk * D), (41, t)) for t in (1, 2))
    got = _prefill(rkv, torch, q, k, v, B, S, H, Hk, D, True)
    want = oracle_mod.prefill(q, k, v, B, S, H, Hk, D, True)
    assert_close(got, want, MAX_ABS, MEAN_ABS, what="zero-query head")
    # causal row i of the zero head is the mean of V rows 0..i
    mean_v = np.cumsum(v[0].astype(np.float64), axis=0) / np.arange(1, S + 1)[:, None]
    assert np.max(np.abs(got[0, :, D:] - mean_v)) < MAX_ABS


def test_pair_fused_fill_equals_plain_prefill(rkv, oracle_mod):
    """attn_prefill_fill_cache runs the same pair kernel as attn_prefill (the fill is a
    programmatic dependent): identical output bit for bit, and the cache rows exact."""
    torch = torch_cuda()
    B, S, H, Hk, D, L = 2, 300, 8, 2, 128, 512
    q, k, v = (inputs.normal((B, S, n * D), (42, t)) for t, n in enumerate((H, Hk, Hk)))
    dq, dk, dv = (torch.from_numpy(a).cuda() for a in (q, k, v))
    o1 = torch.empty((B, S, H * D), device="cuda")
    o2 = torch.empty((B, S, H * D), device="cuda")
    kc = torch.zeros((B, Hk, L, D), device="cuda")
    vc = torch.zeros((B, Hk, L, D), device="cuda")
    rkv.attn_prefill(dq, dk, dv, o1, B, S, H, Hk, D, True)
    rkv.attn_prefill_fill_cache(dq, dk, dv, o2, B, S, H, Hk, D, True, kc, vc, L)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)
    assert np.array_equal(kc[:, :, :S].cpu().numpy(), k.reshape(B, S, Hk, D).transpose(0, 2, 1, 3))
    assert np.array_equal(vc[:, :, :S].cpu().numpy(), v.reshape(B, S, Hk, D).transpose(0, 2, 1, 3))
    assert_close(o1.cpu().numpy(), oracle_mod.prefill(q, k, v, B, S, H, Hk, D, True), MAX_ABS, MEAN_ABS)
