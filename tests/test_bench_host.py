"""Host-side helpers of bench.py (no GPU): the decode step's one-buffer input staging and the
datasheet fraction added beside every roofline entry."""
import numpy as np
import pytest

import bench
from resident_kv_cache_gb300 import inputs


def _small_decode_inputs():
    shape = inputs.DecodeShape("small decode", 5, 8, 2, 64, 40)
    return inputs.batched_decode_inputs(shape)


def test_packed_decode_inputs_round_trip_through_views():
    torch = pytest.importorskip("torch")
    x = _small_decode_inputs()
    buf = torch.from_numpy(bench.pack_decode_inputs(x))
    qd, kn, vn, ln = bench.decode_input_views(torch, buf, x)
    assert np.array_equal(qd.numpy(), x["q"]) and qd.shape == x["q"].shape
    assert np.array_equal(kn.numpy(), x["k_new"]) and np.array_equal(vn.numpy(), x["v_new"])
    assert ln.dtype == torch.int32 and np.array_equal(ln.numpy(), x["lens"])
    # every part starts on a 16-byte boundary (the kernels load 16-byte vectors)
    for t in (qd, kn, vn, ln):
        assert (t.data_ptr() - buf.data_ptr()) % 16 == 0
    # the views alias the one buffer: a single copy into it moves every input
    assert buf.numel() * 4 == sum(t.numel() * t.element_size() for t in (qd, kn, vn, ln))


def test_nominal_fraction_beside_each_roofline():
    r = bench.with_nominal({"unit": "GB/s", "achieved": 3950.0})
    assert r["nominal"]["peak"] == 7900.0 and abs(r["nominal"]["frac"] - 0.5) < 1e-12
    r = bench.with_nominal({"unit": "TFLOP/s", "value": 550.0})
    assert r["nominal"]["peak"] == 1100.0 and abs(r["nominal"]["frac"] - 0.5) < 1e-12
    assert "nominal" not in bench.with_nominal({"unit": "us", "value": 3.0})
