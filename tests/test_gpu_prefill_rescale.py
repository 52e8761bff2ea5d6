"""The prefill's lazy rescale of O, on inputs built to take it at every key block.

The kernels keep a running row maximum m and rescale the output accumulator O (and the row sum)
only when a block's maximum exceeds m by more than 2^8 in the exponent (trustformers-core
attention.rs, mod gpu_tests, fn prefill_reference computes the plain max-subtracted softmax; the
online form with a rescale is the flash-attention restatement of it).  With N(0,1) inputs at
head_dim 32 to 128 the scores never jump that far, so the rescale path would go untested.  Here
every query row is the unit vector e0 and key j is e0 scaled by 100 * (j // 128) + (j % 4): each
128-key block's scores sit 100 above the previous block's (12.7 in log2 units after the 1/sqrt(D)
scale at D = 128, more at smaller D), so every row that sees a new block rescales O by about
2^-12.7 and the earlier blocks keep a small but non-negligible share of the weight.  The scores
are integers below 2^11, exact in TF32, so the only TF32 error is V's rounding and P's
truncation, as in every prefill test; the oracle computes the exact softmax in f64.
"""
import numpy as np
import pytest

from resident_kv_cache_gb300 import inputs
from tests.gpu_util import assert_close, torch_cuda
from tests.test_gpu_prefill import _prefill

pytestmark = pytest.mark.gpu
MAX_ABS, MEAN_ABS = 3e-3, 1e-3

CASES = [
    # B, S, H, Hk, D, causal     (head_dim 128 with an even group: the CTA-pair kernel; else one CTA)
    (1, 640, 2, 1, 128, True),
    (1, 640, 2, 1, 128, False),
    (2, 600, 4, 2, 128, True),
    (1, 640, 1, 1, 128, True),
    (1, 640, 2, 1, 64, False),
    (1, 600, 3, 1, 32, True),
    (1, 300, 2, 2, 16, False),
]


def _rescale_inputs(B, S, H, Hk, D, seed):
    q = np.zeros((B, S, H, D), np.float32)
    q[..., 0] = 1.0
    j = np.arange(S)
    kj = (100 * (j // 128) + (j % 4)).astype(np.float32)          # integers < 2^11: exact in TF32
    k = np.zeros((B, S, Hk, D), np.float32)
    k[..., 0] = kj[None, :, None]
    v = inputs.normal((B, S, Hk * D), (seed, 2))
    return q.reshape(B, S, H * D), k.reshape(B, S, Hk * D), v


@pytest.mark.parametrize("ci", range(len(CASES)))
def test_prefill_rescales_o_at_every_block(rkv, oracle_mod, ci):
    torch = torch_cuda()
    B, S, H, Hk, D, causal = CASES[ci]
    q, k, v = _rescale_inputs(B, S, H, Hk, D, 900 + ci)
    got = _prefill(rkv, torch, q, k, v, B, S, H, Hk, D, causal)
    want = oracle_mod.prefill(q, k, v, B, S, H, Hk, D, causal)
    assert_close(got, want, MAX_ABS, MEAN_ABS, what=f"case {ci}")
