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


def test_traffic_figures_are_keyed_to_every_source_of_their_kernel():
    """bench.py reports an ncu DRAM figure only while the source hash it was taken on matches:
    the hashed file set of each kernel must exist and take in every source its launch compiles
    (both prefill kernels, which share one launch path), or a changed kernel would keep a stale
    figure."""
    import glob
    import json
    import os
    csrc = os.path.join(bench.ROOT, "resident_kv_cache_gb300", "csrc")
    for kernel, files in bench.KERNEL_FILES.items():
        for f in files:
            assert os.path.exists(os.path.join(csrc, f)), (kernel, f)
    prefill_sources = {os.path.basename(p) for p in glob.glob(os.path.join(csrc, "prefill_*"))
                       if not os.path.basename(p).endswith("_guarded.cu")}
    assert prefill_sources <= set(bench.KERNEL_FILES["prefill"])
    assert "rkv_internal.cuh" in bench.KERNEL_FILES["prefill"]
    assert "decode_splitkv.cu" in bench.KERNEL_FILES["decode"]
    with open(os.path.join(bench.ROOT, "profiles", "ncu_traffic.json")) as fh:
        table = json.load(fh)
    for kernel, entry in table.items():
        assert kernel in bench.KERNEL_FILES
        h = entry["source_hash"]
        assert len(h) == 16 and all(c in "0123456789abcdef" for c in h)
        assert entry["dram_bytes_per_launch"] > 0
