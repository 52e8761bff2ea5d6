"""Host-only checks of the C ABI (no GPU needed).

The library builds for sm_103a, loads, exports every function the header
declares, and rejects invalid arguments on the host before touching the GPU --
the pages' hardware-free validation tests (trustformers-core attention.rs,
mod plan_tests: exact fit, empty, overrun) carried over to this ABI.
"""
import ctypes

import pytest

from resident_kv_cache_gb300 import binding, build

pytestmark = pytest.mark.filterwarnings("ignore")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def test_library_exports_every_declared_function(lib):
    names = binding.declared_functions()
    assert set(names) >= {"attn_prefill", "attn_prefill_chunked", "attn_prefill_fill_cache", "kv_append_rope",
                          "attn_decode_batched", "attn_decode_batched_ptrs", "kv_cache_scatter_ptrs",
                          "attn_decode_append",
                          "attn_decode_workspace_bytes",
                          "kv_cache_scatter", "rkv_last_error", "rkv_status_string",
                          "rkv_read_device_flags", "rkv_version"}
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/rkv_attn.h but not exported"


def test_status_strings(lib):
    for s in range(5):
        assert binding.rkv_status_string(s)
    assert binding.rkv_version() >= 1


def _expect(status, fn, *args, **kw):
    with pytest.raises(binding.RkvError) as e:
        fn(*args, **kw)
    assert e.value.status == status, str(e.value)
    assert e.value.message
    return e.value


A = 1 << 20   # a fake 16-byte-aligned address: never dereferenced, validation fails first
INV, UNS = binding.RKV_ERR_INVALID_ARG, binding.RKV_ERR_UNSUPPORTED


@pytest.mark.parametrize("args,status", [
    ((A, A, A, A, 1, 8, 3, 2, 64, 1), INV),      # n_heads % n_kv_heads != 0
    ((A, A, A, A, 1, 8, 4, 2, 48, 1), UNS),      # head_dim not supported
    ((A, A, A, A, 1, 8, 4, 0, 64, 1), INV),      # n_kv_heads == 0
    ((A, A, A, A, -1, 8, 4, 2, 64, 1), INV),     # negative batch
    ((A, A, A, A, 1, -8, 4, 2, 64, 1), INV),     # negative seq_len
    ((None, A, A, A, 1, 8, 4, 2, 64, 1), INV),   # NULL q
    ((A + 4, A, A, A, 1, 8, 4, 2, 64, 1), INV),  # misaligned q
    ((A, A, A, A, 1, 8, 4, 2, 64, 1), INV),      # o aliases q
    ((A, A, A, 2 * A, 1 << 16, 8, 4, 2, 64, 1), UNS),  # batch*heads beyond grid limit
])
def test_prefill_host_validation(lib, args, status):
    _expect(status, binding.attn_prefill, *args, stream=0)


def test_prefill_rejects_bad_scale(lib):
    _expect(INV, binding.attn_prefill, A, A, A, 2 * A, 1, 8, 4, 2, 64, 1, scale=-1.0, stream=0)
    _expect(INV, binding.attn_prefill, A, A, A, 2 * A, 1, 8, 4, 2, 64, 1, scale=float("nan"), stream=0)


def test_zero_sized_work_is_a_noop(lib):
    binding.attn_prefill(None, None, None, None, 0, 8, 4, 2, 64, 1, stream=0)
    binding.attn_prefill(None, None, None, None, 2, 0, 4, 2, 64, 0, stream=0)
    binding.kv_cache_scatter(None, None, None, None, 0, 1, 8, 128, 16, None, stream=0)
    binding.kv_cache_scatter(None, None, None, None, 4, 0, 8, 128, 16, None, stream=0)
    binding.attn_decode_batched(None, None, None, None, 0, 32, 8, 128, 16, None, 0.0, None, 0,
                                stream=0)


@pytest.mark.parametrize("args,status", [
    ((A, A, A, A, 33, 32, 8, 128, 4096, A, 0.0, A, 1 << 30), INV),   # M > 32 (batched cache limit)
    ((A, A, A, A, 4, 32, 8, 96, 4096, A, 0.0, A, 1 << 30), UNS),     # head_dim
    ((A, A, A, A, 4, 48, 3, 128, 4096, A, 0.0, A, 1 << 30), UNS),    # group 16 unsupported
    ((A, A, A, A, 4, 32, 8, 128, 0, A, 0.0, A, 1 << 30), INV),       # max_len 0
    ((A, A, A, A, 4, 32, 8, 128, 4096, None, 0.0, A, 1 << 30), INV), # seq_lens NULL
    ((A, A, A, A, 4, 32, 8, 128, 4096, A, 0.0, A + 16, 1 << 30), INV),  # workspace alignment
    ((A, A, A, A, 4, 32, 8, 128, 4096, A, 0.0, A, 64), INV),         # workspace too small
])
def test_decode_host_validation(lib, args, status):
    _expect(status, binding.attn_decode_batched, *args, stream=0)


def test_decode_workspace_query(lib):
    n = binding.attn_decode_workspace_bytes(32, 32, 8, 128, 4096)
    assert n > 0 and n % 4 == 0
    assert binding.attn_decode_workspace_bytes(33, 32, 8, 128, 4096) == 0
    assert binding.attn_decode_workspace_bytes(4, 32, 7, 128, 4096) == 0
    # grows with the record size
    assert binding.attn_decode_workspace_bytes(4, 32, 8, 64, 4096) < \
        binding.attn_decode_workspace_bytes(4, 32, 8, 128, 4096)
    # the tickets take a fixed block at the head, whatever the sizes; the records grow with M * n_kv_heads
    tb = binding.RKV_DECODE_TICKET_BYTES
    assert binding.attn_decode_workspace_bytes(1, 8, 8, 16, 1) > tb
    a8 = binding.attn_decode_workspace_bytes(8, 32, 8, 128, 4096)
    a16 = binding.attn_decode_workspace_bytes(16, 32, 8, 128, 4096)
    assert (a16 - tb) - (a8 - tb) == 8 * 8 * (4 * 128 + 2 * 4) * 4
    # at most RKV_DECODE_TICKET_BYTES / 4 (sequence, kv head) pairs
    assert binding.attn_decode_workspace_bytes(32, 256, 256, 16, 64) > 0
    assert binding.attn_decode_workspace_bytes(32, 257, 257, 16, 64) == 0
    assert binding.attn_decode_workspace_bytes(1, 8192, 8192, 16, 64) > 0
    assert binding.attn_decode_workspace_bytes(1, 8193, 8193, 16, 64) == 0


def test_checked_build_exports_every_declared_function():
    """The debug build with the device index checks compiled in (librkv_attn_checked.so)."""
    path = build.build(checked=True)
    lib = ctypes.CDLL(path)
    for n in binding.declared_functions():
        assert hasattr(lib, n), f"{n} missing from the checked build"


def test_bounds_flag_matches_the_header():
    import os
    import re
    hdr = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "rkv_attn.h")
    m = re.search(r"#define\s+RKV_FLAG_BOUNDS\s+(0x[0-9a-fA-F]+)u", open(hdr).read())
    assert m and int(m.group(1), 16) == binding.RKV_FLAG_BOUNDS


def test_ticket_block_size_matches_the_header():
    import os
    import re
    hdr = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "rkv_attn.h")
    m = re.search(r"#define\s+RKV_DECODE_TICKET_BYTES\s+(\d+)", open(hdr).read())
    assert m and int(m.group(1)) == binding.RKV_DECODE_TICKET_BYTES


def test_decode_rejects_more_pairs_than_tickets(lib):
    # 32 sequences x 257 kv heads: more (sequence, kv head) pairs than the ticket block holds
    _expect(UNS, binding.attn_decode_batched, A, A, A, A, 32, 257, 257, 16, 64, A, 0.0, A, 1 << 40, stream=0)


@pytest.mark.parametrize("args,status", [
    ((A, A, A, A, 33, 1, 8, 128, 4096, A), INV),    # M > 32
    ((A, A, A, A, 4, 5000, 8, 128, 4096, A), INV),  # T > max_len
    ((A, A, A, A, 4, 1, 8, 80, 4096, A), UNS),      # head_dim
    ((A, A, A, A, 4, 1, 8, 128, 4096, None), INV),  # start_pos NULL
    ((A, A + 8, A, A, 4, 1, 8, 128, 4096, A), INV),  # misaligned v_new
    ((A, A, A, A, 4, -1, 8, 128, 4096, A), INV),    # negative T
])
def test_scatter_host_validation(lib, args, status):
    _expect(status, binding.kv_cache_scatter, *args, stream=0)


@pytest.mark.parametrize("args,status", [
    ((A, A, A, 2 * A, 33, 8, 4, 2, 64, 128, 1, A), INV),       # M > 32 (batched cache limit)
    ((A, A, A, 2 * A, 2, 200, 4, 2, 64, 128, 1, A), INV),      # T > max_len
    ((A, A, A, 2 * A, 2, 8, 4, 2, 64, 0, 1, A), INV),          # max_len 0
    ((A, A, A, 2 * A, 2, 8, 6, 4, 64, 128, 1, A), INV),        # n_heads % n_kv_heads
    ((A, A, A, 2 * A, 2, 8, 4, 2, 96, 128, 1, A), UNS),        # head_dim
    ((A, A, A, 2 * A, 2, 8, 4, 2, 64, 128, 1, None), INV),     # start_pos NULL
    ((A, A + 4, A, 2 * A, 2, 8, 4, 2, 64, 128, 1, A), INV),    # misaligned cache
    ((A, A, A, A, 2, 8, 4, 2, 64, 128, 1, A), INV),            # o aliases q
    ((A, A, A, 2 * A, 2, -1, 4, 2, 64, 128, 1, A), INV),       # negative T
])
def test_prefill_chunked_host_validation(lib, args, status):
    _expect(status, binding.attn_prefill_chunked, *args, stream=0)


def test_prefill_chunked_zero_sized_is_a_noop(lib):
    binding.attn_prefill_chunked(None, None, None, None, 0, 8, 4, 2, 64, 128, 1, None, stream=0)
    binding.attn_prefill_chunked(None, None, None, None, 3, 0, 4, 2, 64, 128, 1, None, stream=0)


B_ = 3 * A   # a second fake address for the caches
@pytest.mark.parametrize("args,status", [
    ((A, A, A, 2 * A, 33, 8, 4, 2, 64, 1, 0.0, B_, 4 * A, 16), INV),     # batch > 32 (batched cache limit)
    ((A, A, A, 2 * A, 2, 32, 4, 2, 64, 1, 0.0, B_, 4 * A, 16), INV),     # seq_len > max_len
    ((A, A, A, 2 * A, 2, 8, 4, 2, 64, 1, 0.0, None, 4 * A, 16), INV),   # NULL cache
    ((A, A, A, 2 * A, 2, 8, 4, 2, 64, 1, 0.0, A, 4 * A, 16), INV),      # cache aliases q
    ((A, A, A, 2 * A, 2, 8, 4, 2, 64, 1, 0.0, B_, B_, 16), INV),        # k_cache == v_cache
    ((A, A, A, 2 * A, 2, 8, 4, 2, 64, 1, 0.0, B_ + 8, 4 * A, 16), INV),  # misaligned cache
    ((A, A, A, 2 * A, 2, 8, 4, 2, 96, 1, 0.0, B_, 4 * A, 16), UNS),     # head_dim
    ((A, A, A, 2 * A, 2, 8, 4, 2, 64, 1, -1.0, B_, 4 * A, 16), INV),    # negative scale
])
def test_prefill_fill_cache_host_validation(lib, args, status):
    q, k, v, o, B, S, H, Hk, D, causal, scale, kc, vc, L = args
    _expect(status, binding.attn_prefill_fill_cache, q, k, v, o, B, S, H, Hk, D, causal, kc, vc, L,
            scale=scale, stream=0)


@pytest.mark.parametrize("kw,status", [
    ({"M": 33}, INV), ({"T": 70}, INV), ({"rotary_ndims": 0}, INV), ({"rotary_ndims": 130}, INV),
    ({"rotary_ndims": 7}, INV), ({"rotary_ndims": 12}, UNS), ({"theta": 0.0}, INV),
    ({"theta": float("inf")}, INV), ({"head_dim": 96}, UNS), ({"v_cache": B_}, INV), ({"q": A + 4}, INV),
    ({"start_pos": None}, INV),
])
def test_kv_append_rope_host_validation(lib, kw, status):
    a = dict(q=A, k_new=2 * A, v_new=4 * A, k_cache=B_, v_cache=5 * A, M=2, T=8, n_heads=8, n_kv_heads=2,
             head_dim=128, max_len=64, start_pos=6 * A, rotary_ndims=128, theta=1e4)
    a.update(kw)
    _expect(status, binding.kv_append_rope, a["q"], a["k_new"], a["v_new"], a["k_cache"], a["v_cache"], a["M"],
            a["T"], a["n_heads"], a["n_kv_heads"], a["head_dim"], a["max_len"], a["start_pos"],
            rotary_ndims=a["rotary_ndims"], theta=a["theta"], stream=0)


def test_pointer_array_entries_host_validation(lib):
    n = binding.attn_decode_workspace_bytes(4, 32, 8, 128, 64)
    _expect(INV, binding.attn_decode_batched_ptrs, A, None, 2 * A, 3 * A, 4, 32, 8, 128, 64, A, 0.0, A, n, stream=0)
    _expect(INV, binding.attn_decode_batched_ptrs, A, 2 * A + 4, 3 * A, 4 * A, 4, 32, 8, 128, 64, A, 0.0, A, n,
            stream=0)                                            # pointer array not 8-byte aligned
    _expect(INV, binding.attn_decode_batched_ptrs, A, 2 * A, 3 * A, 4 * A, 33, 32, 8, 128, 64, A, 0.0, A, n,
            stream=0)
    _expect(INV, binding.kv_cache_scatter_ptrs, A, A, None, 2 * A, 4, 1, 8, 128, 64, A, stream=0)
    _expect(UNS, binding.kv_cache_scatter_ptrs, A, A, 2 * A, 3 * A, 4, 1, 8, 96, 64, A, stream=0)
    binding.attn_decode_batched_ptrs(None, None, None, None, 0, 32, 8, 128, 64, None, 0.0, None, 0, stream=0)
    binding.kv_cache_scatter_ptrs(None, None, None, None, 0, 1, 8, 128, 64, None, stream=0)


def test_decode_append_host_validation(lib):
    n = binding.attn_decode_workspace_bytes(4, 32, 8, 128, 64)
    _expect(INV, binding.attn_decode_append, A, None, 2 * A, 3 * A, 4 * A, 5 * A, 4, 32, 8, 128, 64, A, 0.0, A, n,
            stream=0)                                              # k_new NULL
    _expect(INV, binding.attn_decode_append, A, 2 * A, 2 * A + 8, 3 * A, 4 * A, 5 * A, 4, 32, 8, 128, 64, A, 0.0, A,
            n, stream=0)                                           # v_new misaligned
    _expect(INV, binding.attn_decode_append, A, 2 * A, 6 * A, 2 * A, 4 * A, 5 * A, 4, 32, 8, 128, 64, A, 0.0, A, n,
            stream=0)                                              # k_cache aliases k_new
    _expect(INV, binding.attn_decode_append, A, 2 * A, 6 * A, 3 * A, 3 * A, 5 * A, 4, 32, 8, 128, 64, A, 0.0, A, n,
            stream=0)                                              # k_cache == v_cache
    binding.attn_decode_append(None, None, None, None, None, None, 0, 32, 8, 128, 64, None, 0.0, None, 0, stream=0)


def test_wait_check_host_validation(lib):
    _expect(INV, binding.rkv_check_wait_timeout, 0, stream=0)           # no limit
    _expect(INV, binding.rkv_check_wait_timeout, 1000001, stream=0)     # above 1 s
    assert "limit_us" in binding.rkv_last_error()


def test_last_error_is_per_call(lib):
    _expect(INV, binding.attn_prefill, A, A, A, A, 1, 8, 3, 2, 64, 1, stream=0)
    assert "multiple" in binding.rkv_last_error()
    binding.attn_prefill(None, None, None, None, 0, 8, 4, 2, 64, 1, stream=0)
    assert binding.rkv_last_error() == ""


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "LIB_PATH", str(tmp_path / "absent.so"))
    with pytest.raises(FileNotFoundError):
        binding.load()
