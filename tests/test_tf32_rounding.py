"""The prefill's TF32 operand rounding: the bit method against the definition (host),
and the device code against the definition and the hardware conversion (GPU).

The tensor core reads an f32 operand of a kind::tf32 product by dropping its 13 low
mantissa bits (truncation).  The prefill rounds Q and V to nearest first by adding half
a TF32 unit in the last place to the bit pattern, so that the drop lands on the nearest
TF32 value, ties away from zero; infinities and positive NaNs keep their class.
"""
import numpy as np
import pytest

from tests.tf32_util import LOW, add_half_bits, rna_exact, sweep_bits


def _is_nan_bits(b):
    b = np.asarray(b, np.uint32)
    return ((b & np.uint32(0x7F800000)) == np.uint32(0x7F800000)) & ((b & np.uint32(0x007FE000)) != 0)


def test_add_half_then_drop_is_round_to_nearest_ties_away():
    bits = sweep_bits()
    got = add_half_bits(bits) & ~LOW
    want = np.array([rna_exact(b) for b in bits], np.uint32)
    x = bits.view(np.float32)
    finite = np.isfinite(x)
    assert np.array_equal(got[finite], want[finite])
    inf = np.isinf(x)
    assert np.array_equal(got[inf], bits[inf])              # infinities unchanged
    # a NaN stays NaN (or becomes the infinity that dropping its low bits gives anyway),
    # except a negative NaN at 0xFFFFF000 or above, which wraps to +0
    nan = np.isnan(x)
    wraps = bits >= np.uint32(0xFFFFF000)
    keep = nan & ~wraps
    assert np.all(_is_nan_bits(got[keep]) | ((got[keep] & ~np.uint32(0x80000000)) == np.uint32(0x7F800000)))
    assert np.all(got[nan & wraps] == 0)


def test_worked_values():
    # 1 + 2^-11 is exactly halfway between 1 and 1 + 2^-10: ties away -> 1 + 2^-10
    one_half = int(np.float32(1 + 2 ** -11).view(np.uint32))
    assert rna_exact(one_half) == int(np.float32(1 + 2 ** -10).view(np.uint32))
    # just below halfway rounds down, just above rounds up
    assert rna_exact(one_half - 1) == 0x3F800000
    assert rna_exact(one_half + 1) == int(np.float32(1 + 2 ** -10).view(np.uint32))
    # ties away from zero on the negative side too
    assert rna_exact(one_half | 0x80000000) == int(np.float32(-(1 + 2 ** -10)).view(np.uint32))
    # the largest finite float32 rounds past the largest TF32 value to infinity
    assert rna_exact(0x7F7FFFFF) == 0x7F800000
    # the error of rounding to nearest is at most half a unit: 2^-11 relative to the binade
    for v in (3.999, 4.0017, -5.3, 0.123456):
        r = float(np.uint32(rna_exact(int(np.float32(v).view(np.uint32)))).view(np.float32))
        assert abs(r - np.float32(v)) <= 2.0 ** (np.floor(np.log2(abs(v))) - 11)
    # the canonical NaN pattern would carry into the sign bit without the signed maximum
    assert add_half_bits(np.array([0x7FFFFFFF], np.uint32))[0] == 0x7FFFFFFF
    # negative numbers: the signed add grows the magnitude; -(1 + 2^-11) is a tie and goes
    # away from zero to -(1 + 2^-10)
    neg_tie = np.array([one_half | 0x80000000], np.uint32)
    assert (add_half_bits(neg_tie) & ~LOW)[0] == int(np.float32(-(1 + 2 ** -10)).view(np.uint32))


@pytest.mark.gpu
def test_device_rounding_matches_definition_and_cvt_rna(rkv):
    from tests.gpu_util import torch_cuda
    torch = torch_cuda()
    host = sweep_bits(n_random=1 << 20, seed=11)
    x = torch.from_numpy(host.view(np.int32)).cuda()
    ours = torch.empty_like(x)
    ref = torch.empty_like(x)
    rkv.rkv_check_tf32_round(x, ours, ref, x.numel())
    torch.cuda.synchronize()
    ours_h = ours.cpu().numpy().view(np.uint32)
    ref_h = ref.cpu().numpy().view(np.uint32)
    finite = np.isfinite(host.view(np.float32))
    assert np.array_equal(ours_h[finite], ref_h[finite]), "differs from cvt.rna.tf32.f32"
    assert np.array_equal(ours_h, add_half_bits(host) & ~LOW)   # the device runs the method exactly
    sub = np.arange(0, host.size, 97)
    want = np.array([rna_exact(b) for b in host[sub]], np.uint32)
    fin = finite[sub]
    assert np.array_equal(ours_h[sub][fin], want[fin])
