"""Pins for the CPU oracle: checks against things other than the oracle itself.

- hand-derived worked examples in tests/golden/ (each file cites its page);
- an independent brute-force implementation (dense score tensor, scipy's
  softmax) on tiny shapes, to 1e-12;
- invariants the pages and the mathematics fix: probability rows sum to 1,
  constant V passes through, identical keys average V, causal row 0 copies
  V[0], decode equals the last row of a causal prefill (the parity test of
  trustformers-core attention.rs, mod gpu_tests, decode test), GQA equals MHA
  with repeated kv heads, softmax shift invariance, scatter read-back.
"""
import glob
import json
import os

import numpy as np
import pytest
from scipy.special import softmax as scipy_softmax

from resident_kv_cache_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- brute force
def brute_prefill(q, k, v, B, S, H, Hk, D, causal, seq_lens=None, scale=None):
    """Dense [B,H,S,S] scores, -inf mask, scipy softmax, einsum with V (float64)."""
    scale = 1.0 / np.sqrt(D) if scale is None else scale
    q4 = np.asarray(q, np.float64).reshape(B, S, H, D)
    k4 = np.asarray(k, np.float64).reshape(B, S, Hk, D)
    v4 = np.asarray(v, np.float64).reshape(B, S, Hk, D)
    grp = np.arange(H) // (H // Hk)
    kx, vx = k4[:, :, grp, :], v4[:, :, grp, :]            # [B,S,H,D]
    sc = np.einsum("bihd,bjhd->bhij", q4, kx) * scale        # [B,H,S,S]
    lens = np.full(B, S) if seq_lens is None else np.asarray(seq_lens)
    i_idx = np.arange(S)[:, None]
    j_idx = np.arange(S)[None, :]
    out = np.zeros((B, S, H, D))
    for b in range(B):
        vis = (j_idx < lens[b]) & (i_idx < lens[b])
        if causal:
            vis &= j_idx <= i_idx
        s = np.where(vis[None], sc[b], -np.inf)
        with np.errstate(invalid="ignore"):
            p = scipy_softmax(s, axis=-1)
        p = np.where(vis[None], p, 0.0)
        p = np.nan_to_num(p)
        out[b] = np.einsum("hij,jhd->ihd", p, vx[b])
    return out.reshape(B, S, H * D)


def brute_decode(q, kc, vc, M, H, Hk, D, L, lens, scale=None):
    scale = 1.0 / np.sqrt(D) if scale is None else scale
    q3 = np.asarray(q, np.float64).reshape(M, H, D)
    grp = np.arange(H) // (H // Hk)
    out = np.zeros((M, H, D))
    for m in range(M):
        n = int(lens[m])
        if n <= 0:
            continue
        kk = np.asarray(kc, np.float64)[m][grp, :n, :]        # [H,n,D]
        vv = np.asarray(vc, np.float64)[m][grp, :n, :]
        s = np.einsum("hd,hnd->hn", q3[m], kk) * scale
        out[m] = np.einsum("hn,hnd->hd", scipy_softmax(s, axis=-1), vv)
    return out.reshape(M, H * D)


# ------------------------------------------------------------------- golden
@pytest.mark.parametrize("name", ["two_keys_closed_form.json", "equal_scores_mean.json",
                                  "gqa_single_key.json"])
@pytest.mark.parametrize("causal", [False, True])
def test_golden_prefill(oracle_mod, name, causal):
    g = _golden(name)
    q = np.array(g["q"], np.float32)
    k = np.array(g["k"], np.float32)
    v = np.array(g["v"], np.float32)
    o = oracle_mod.prefill(q, k, v, g["B"], g["S"], g["H"], g["Hk"], g["D"], causal,
                           scale=g.get("scale"))
    want = np.array(g["expected_causal" if causal else "expected_noncausal"], np.float64)
    assert np.max(np.abs(o.reshape(want.shape) - want)) <= g["tolerance"]


def test_golden_decode(oracle_mod):
    g = _golden("decode_ignores_rows_past_length.json")
    o = oracle_mod.decode(np.array(g["q"], np.float32), np.array(g["k_cache"], np.float32),
                          np.array(g["v_cache"], np.float32), g["M"], g["H"], g["Hk"], g["D"],
                          g["Lmax"], np.array(g["lens"]), scale=g["scale"])
    assert np.max(np.abs(o - np.array(g["expected"]))) <= g["tolerance"]


def test_golden_scatter(oracle_mod):
    g = _golden("scatter_overflow.json")
    M, T, Hk, D, L = g["M"], g["T"], g["Hk"], g["D"], g["Lmax"]
    kn = np.array(g["k_new"], np.float32)
    vn = kn + 100.0
    kc = np.full((M, Hk, L, D), g["fill"], np.float32)
    vc = np.full((M, Hk, L, D), g["fill"], np.float32)
    k2, v2, ov = oracle_mod.scatter(kn, vn, kc, vc, M, T, Hk, D, L, np.array(g["start_pos"]))
    want_k = np.array(g["expected_k_cache"], np.float32)
    want_v = np.where(want_k == g["fill"], g["fill"], want_k + 100.0).astype(np.float32)
    assert np.array_equal(k2, want_k)
    assert np.array_equal(v2, want_v)
    assert ov == g["expected_overflow"]


def test_every_golden_file_has_a_citation():
    files = glob.glob(os.path.join(GOLDEN, "*.json"))
    assert files
    for f in files:
        with open(f) as fh:
            g = json.load(fh)
        assert g.get("citation") and g.get("derivation"), f


# --------------------------------------------------------------- brute force
_TINY_CASES = [
    # B, S, H, Hk, D, causal, seq_lens
    (1, 1, 1, 1, 1, False, None),
    (1, 5, 2, 2, 3, False, None),
    (1, 5, 2, 2, 3, True, None),
    (2, 7, 4, 2, 4, True, [7, 3]),
    (2, 8, 4, 1, 2, False, [5, 8]),
    (3, 6, 3, 3, 4, True, [6, 1, 0]),
    (1, 8, 4, 4, 4, False, [4]),
    (2, 4, 2, 1, 1, True, None),
]


@pytest.mark.parametrize("ci", range(len(_TINY_CASES)))
def test_prefill_matches_brute_force(oracle_mod, ci):
    B, S, H, Hk, D, causal, lens = _TINY_CASES[ci]
    seed = 1000 + ci
    q = inputs.normal((B, S, H * D), (seed, 0))
    k = inputs.normal((B, S, Hk * D), (seed, 1))
    v = inputs.normal((B, S, Hk * D), (seed, 2))
    got = oracle_mod.prefill(q, k, v, B, S, H, Hk, D, causal, seq_lens=lens)
    want = brute_prefill(q, k, v, B, S, H, Hk, D, causal, seq_lens=lens)
    assert np.max(np.abs(got - want)) < 1e-12


def test_page_worked_example_shape(oracle_mod):
    """trustformers-core attention.rs, mod gpu_tests, prefill parity test: H=2, seq=3, d=2,
    q_i = sin(0.37 i), k_i = cos(0.53 i), v_i = 0.25 i - 1 over the heads-major [H,seq,d]
    buffer.  The page prints no expected values, so the check is against brute force."""
    H, S, D = 2, 3, 2
    n = H * S * D
    idx = np.arange(n, dtype=np.float32)
    hm = lambda a: np.transpose(a.reshape(H, S, D), (1, 0, 2)).reshape(1, S, H * D)
    q = hm(np.sin(idx * np.float32(0.37)).astype(np.float32))
    k = hm(np.cos(idx * np.float32(0.53)).astype(np.float32))
    v = hm((idx * np.float32(0.25) - 1).astype(np.float32))
    got = oracle_mod.prefill(q, k, v, 1, S, H, H, D, True)
    want = brute_prefill(q, k, v, 1, S, H, H, D, True)
    assert np.max(np.abs(got - want)) < 1e-12


@pytest.mark.parametrize("M,H,Hk,D,L,lens", [
    (1, 1, 1, 1, 1, [1]),
    (3, 4, 2, 4, 9, [9, 1, 5]),
    (4, 8, 2, 8, 16, [0, 16, 7, 2]),
    (2, 2, 2, 3, 5, [3, 5]),
])
def test_decode_matches_brute_force(oracle_mod, M, H, Hk, D, L, lens):
    seed = M * 1000 + L
    q = inputs.normal((M, H * D), (seed, 0))
    kc = inputs.normal((M, Hk, L, D), (seed, 1))
    vc = inputs.normal((M, Hk, L, D), (seed, 2))
    got = oracle_mod.decode(q, kc, vc, M, H, Hk, D, L, np.array(lens))
    want = brute_decode(q, kc, vc, M, H, Hk, D, L, lens)
    assert np.max(np.abs(got - want)) < 1e-12


# ---------------------------------------------------------------- invariants
@pytest.mark.parametrize("causal", [False, True])
def test_probability_rows_sum_to_one(oracle_mod, causal):
    """trueno-gpu attention.rs, fn batched_multihead_attention debug check: softmax rows sum to 1."""
    B, S, H, Hk, D = 2, 9, 4, 2, 4
    q, k, v = (inputs.normal((B, S, n * D), (5, t)) for t, n in enumerate((H, Hk, Hk)))
    lens = np.array([9, 6])
    for b in range(B):
        for h in range(H):
            for i in range(S):
                p = oracle_mod.prefill_probs(q, k, v, B, S, H, Hk, D, causal, b, h, i,
                                             seq_lens=lens)
                if i < lens[b]:
                    assert abs(p.sum() - 1.0) < 1e-12
                    assert np.all(p >= 0)
                    visible = (i + 1) if causal else lens[b]
                    assert np.all(p[visible:] == 0.0)
                else:
                    assert np.all(p == 0.0)


@pytest.mark.parametrize("causal", [False, True])
def test_constant_v_passes_through(oracle_mod, causal):
    B, S, H, Hk, D = 1, 11, 4, 2, 8
    q = inputs.normal((B, S, H * D), 11)
    k = inputs.normal((B, S, Hk * D), 12)
    col = np.linspace(-2, 3, Hk * D).astype(np.float32)
    v = np.broadcast_to(col, (B, S, Hk * D)).copy()
    o = oracle_mod.prefill(q, k, v, B, S, H, Hk, D, causal)
    grp = np.arange(H) // (H // Hk)
    want = col.reshape(Hk, D)[grp].reshape(-1)
    assert np.max(np.abs(o - want[None, None, :])) < 1e-12


def test_identical_keys_average_v(oracle_mod):
    B, S, H, Hk, D = 1, 6, 2, 2, 4
    q = inputs.normal((B, S, H * D), 21)
    k = np.broadcast_to(inputs.normal((1, 1, Hk * D), 22), (B, S, Hk * D)).copy()
    v = inputs.normal((B, S, Hk * D), 23)
    o_nc = oracle_mod.prefill(q, k, v, B, S, H, Hk, D, False)
    o_c = oracle_mod.prefill(q, k, v, B, S, H, Hk, D, True)
    v64 = v.astype(np.float64)
    assert np.max(np.abs(o_nc - v64.mean(axis=1, keepdims=True))) < 1e-12
    running = np.cumsum(v64, axis=1) / np.arange(1, S + 1)[None, :, None]
    assert np.max(np.abs(o_c - running)) < 1e-12


def test_causal_row0_is_v0(oracle_mod):
    B, S, H, Hk, D = 2, 5, 4, 2, 4
    q, k, v = (inputs.normal((B, S, n * D), (31, t)) for t, n in enumerate((H, Hk, Hk)))
    o = oracle_mod.prefill(q, k, v, B, S, H, Hk, D, True)
    grp = np.arange(H) // (H // Hk)
    want = v[:, 0, :].reshape(B, Hk, D)[:, grp, :].reshape(B, H * D)
    assert np.array_equal(o[:, 0, :], want.astype(np.float64))


def test_decode_equals_last_row_of_causal_prefill(oracle_mod):
    """trustformers-core attention.rs, mod gpu_tests: decode must equal the last row of
    a causal prefill on the same data."""
    S, H, Hk, D = 7, 4, 2, 4
    q, k, v = (inputs.normal((1, S, n * D), (41, t)) for t, n in enumerate((H, Hk, Hk)))
    full = oracle_mod.prefill(q, k, v, 1, S, H, Hk, D, True)
    L = S + 3
    kc = np.zeros((1, Hk, L, D), np.float32)
    vc = np.zeros((1, Hk, L, D), np.float32)
    kc[0, :, :S, :] = k.reshape(S, Hk, D).transpose(1, 0, 2)
    vc[0, :, :S, :] = v.reshape(S, Hk, D).transpose(1, 0, 2)
    kc[0, :, S:, :] = 1e30                        # must not be read
    dec = oracle_mod.decode(q[:, S - 1, :], kc, vc, 1, H, Hk, D, L, np.array([S]))
    assert np.max(np.abs(dec - full[:, S - 1, :])) < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_gqa_equals_mha_with_repeated_kv(oracle_mod, causal):
    B, S, H, Hk, D = 2, 6, 6, 2, 3
    q, k, v = (inputs.normal((B, S, n * D), (51, t)) for t, n in enumerate((H, Hk, Hk)))
    grp = np.arange(H) // (H // Hk)
    rep = lambda a: a.reshape(B, S, Hk, D)[:, :, grp, :].reshape(B, S, H * D)
    gqa = oracle_mod.prefill(q, k, v, B, S, H, Hk, D, causal)
    mha = oracle_mod.prefill(q, rep(k), rep(v), B, S, H, H, D, causal)
    assert np.array_equal(gqa, mha)


def test_softmax_shift_invariance(oracle_mod):
    """Adding one vector u to every key shifts all scores of a row equally; the output must
    not move, even when the shift is large enough to overflow an unshifted exp."""
    B, S, H, Hk, D = 1, 5, 2, 1, 4
    q = np.abs(inputs.normal((B, S, H * D), 61)) + 1.0
    # keys on a 2^-10 grid so that k + 400 is exact in f32
    k = (np.round(inputs.normal((B, S, Hk * D), 62) * 1024) / 1024).astype(np.float32)
    v = inputs.normal((B, S, Hk * D), 63)
    u = np.full(Hk * D, 400.0, np.float32)        # shift ~ 400*|q|*4/2 >> 709
    o1 = oracle_mod.prefill(q, k, v, B, S, H, Hk, D, True)
    o2 = oracle_mod.prefill(q, k + u, v, B, S, H, Hk, D, True)
    assert np.all(np.isfinite(o2))
    assert np.max(np.abs(o1 - o2)) < 1e-9


def test_explicit_scale_equals_scaled_query(oracle_mod):
    B, S, H, Hk, D = 1, 6, 2, 2, 4
    q, k, v = (inputs.normal((B, S, n * D), (71, t)) for t, n in enumerate((H, Hk, Hk)))
    o1 = oracle_mod.prefill(q, k, v, B, S, H, Hk, D, True, scale=0.5)
    o2 = oracle_mod.prefill(q * np.float32(0.25), k, v, B, S, H, Hk, D, True, scale=2.0)
    assert np.max(np.abs(o1 - o2)) < 1e-12


def test_padded_query_rows_are_zero(oracle_mod):
    B, S, H, Hk, D = 2, 6, 2, 1, 4
    q, k, v = (inputs.normal((B, S, n * D), (81, t)) for t, n in enumerate((H, Hk, Hk)))
    lens = np.array([4, 0])
    o = oracle_mod.prefill(q, k, v, B, S, H, Hk, D, False, seq_lens=lens)
    assert np.all(o[0, 4:] == 0) and np.all(o[1] == 0)
    # the valid part equals a prefill of the truncated sequence
    o4 = oracle_mod.prefill(q[:1, :4], k[:1, :4], v[:1, :4], 1, 4, H, Hk, D, False)
    assert np.max(np.abs(o[0, :4] - o4[0])) < 1e-12


def test_all_empty_batches_give_zero_rows(oracle_mod):
    """Reading O3/O7 for a batch with no valid row at all (the decode has nothing to attend,
    the prefill and the chunked prefill no valid query): every output row is exactly zero."""
    M, H, Hk, D, L = 3, 4, 2, 8, 5
    q = inputs.normal((M, H * D), (82, 0))
    kc, vc = inputs.normal((M, Hk, L, D), (82, 1)), inputs.normal((M, Hk, L, D), (82, 2))
    assert np.all(oracle_mod.decode(q, kc, vc, M, H, Hk, D, L, np.zeros(M, np.int32)) == 0)
    B, S = 2, 6
    qp, kp, vp = (inputs.normal((B, S, n * D), (83, t)) for t, n in enumerate((H, Hk, Hk)))
    for causal in (False, True):
        assert np.all(oracle_mod.prefill(qp, kp, vp, B, S, H, Hk, D, causal, seq_lens=np.zeros(B)) == 0)
    qc = inputs.normal((B, 3, H * D), (84, 0))
    kc2, vc2 = inputs.normal((B, Hk, 10, D), (84, 1)), inputs.normal((B, Hk, 10, D), (84, 2))
    got = oracle_mod.prefill_cached(qc, kc2, vc2, B, 3, H, Hk, D, 10, True, np.array([0, 5], np.int32),
                                    q_lens=np.zeros(B, np.int32))
    assert np.all(got == 0)


def test_prefill_rows_matches_full(oracle_mod):
    B, S, H, Hk, D = 2, 9, 4, 2, 8
    q, k, v = (inputs.normal((B, S, n * D), (91, t)) for t, n in enumerate((H, Hk, Hk)))
    full = oracle_mod.prefill(q, k, v, B, S, H, Hk, D, True)
    rows = inputs.sample_indices(B * H * S, 25, 7)
    got = oracle_mod.prefill_rows(q, k, v, B, S, H, Hk, D, True, rows)
    for t, r in enumerate(rows):
        b, h, i = r // (H * S), (r // S) % H, r % S
        assert np.array_equal(got[t], full[b, i, h * D:(h + 1) * D])


def test_scatter_readback_identity_and_canaries(oracle_mod):
    M, T, Hk, D, L = 3, 4, 2, 8, 10
    kn = inputs.normal((M, T, Hk * D), 101)
    vn = inputs.normal((M, T, Hk * D), 102)
    kc0 = inputs.normal((M, Hk, L, D), 103)
    vc0 = inputs.normal((M, Hk, L, D), 104)
    start = np.array([0, 5, 8], np.int32)          # third sequence overflows by 2 tokens
    kc, vc, ov = oracle_mod.scatter(kn, vn, kc0, vc0, M, T, Hk, D, L, start)
    assert ov == 2
    written = np.zeros((M, Hk, L), bool)
    for m in range(M):
        for t in range(T):
            p = start[m] + t
            if p >= L:
                continue
            written[m, :, p] = True
            np.testing.assert_array_equal(kc[m, :, p, :], kn[m, t].reshape(Hk, D))
            np.testing.assert_array_equal(vc[m, :, p, :], vn[m, t].reshape(Hk, D))
    assert np.array_equal(kc[~written], kc0[~written])
    assert np.array_equal(vc[~written], vc0[~written])


# ------------------------------------------------- prefill behind an existing cache
def brute_prefill_cached(q, kc, vc, B, T, H, Hk, D, L, causal, start_pos, q_lens=None, scale=None):
    """Dense scores over the whole cache, a mask on absolute positions, scipy softmax."""
    scale = 1.0 / np.sqrt(D) if scale is None else scale
    q4 = np.asarray(q, np.float64).reshape(B, T, H, D)
    grp = np.arange(H) // (H // Hk)
    n_q = np.full(B, T) if q_lens is None else np.asarray(q_lens)
    out = np.zeros((B, T, H, D))
    pos_key = np.arange(L)[None, :]
    for b in range(B):
        kk = np.asarray(kc, np.float64)[b][grp]                  # [H, L, D]
        vv = np.asarray(vc, np.float64)[b][grp]
        sc = np.einsum("ihd,hjd->hij", q4[b], kk) * scale        # [H, T, L]
        pos_q = start_pos[b] + np.arange(T)[:, None]              # absolute query positions
        vis = (np.arange(T)[:, None] < n_q[b]) & (pos_key < start_pos[b] + n_q[b])
        if causal:
            vis &= pos_key <= pos_q
        s = np.where(vis[None], sc, -np.inf)
        with np.errstate(invalid="ignore"):
            p = np.nan_to_num(np.where(vis[None], scipy_softmax(s, axis=-1), 0.0))
        out[b] = np.einsum("hij,hjd->ihd", p, vv)
    return out.reshape(B, T, H * D)


@pytest.mark.parametrize("causal", [False, True])
def test_golden_prefill_cached(oracle_mod, causal):
    g = _golden("chunk_behind_cache_closed_form.json")
    B, T, H, Hk, D, L = g["B"], g["T"], g["H"], g["Hk"], g["D"], g["Lmax"]
    q = np.array(g["q"], np.float32).reshape(B, T, H * D)
    kc = np.array(g["k_cache"], np.float32).reshape(B, Hk, L, D)
    vc = np.array(g["v_cache"], np.float32).reshape(B, Hk, L, D)
    o = oracle_mod.prefill_cached(q, kc, vc, B, T, H, Hk, D, L, causal, np.array(g["start_pos"]),
                                  q_lens=np.array(g["q_lens"]), scale=g["scale"])
    want = np.array(g["expected_causal" if causal else "expected_noncausal"], np.float64)
    assert np.max(np.abs(o.reshape(want.shape) - want)) <= g["tolerance"]


_CACHED_CASES = [
    # B, T, H, Hk, D, L, causal, start_pos, q_lens
    (1, 1, 1, 1, 1, 1, True, [0], None),
    (1, 3, 2, 2, 3, 8, True, [5], None),
    (1, 3, 2, 2, 3, 8, False, [5], None),
    (2, 4, 4, 2, 4, 9, True, [0, 3], [4, 2]),
    (3, 5, 6, 3, 2, 12, False, [7, 0, 2], [5, 0, 3]),
    (2, 2, 4, 1, 4, 6, True, [4, 1], None),
]


@pytest.mark.parametrize("ci", range(len(_CACHED_CASES)))
def test_prefill_cached_matches_brute_force(oracle_mod, ci):
    B, T, H, Hk, D, L, causal, sp, ql = _CACHED_CASES[ci]
    seed = 2000 + ci
    q = inputs.normal((B, T, H * D), (seed, 0))
    kc = inputs.normal((B, Hk, L, D), (seed, 1))
    vc = inputs.normal((B, Hk, L, D), (seed, 2))
    got = oracle_mod.prefill_cached(q, kc, vc, B, T, H, Hk, D, L, causal, np.array(sp), q_lens=ql)
    want = brute_prefill_cached(q, kc, vc, B, T, H, Hk, D, L, causal, np.array(sp), q_lens=ql)
    assert np.max(np.abs(got - want)) < 1e-12


def _cache_of(k, v, B, S, Hk, D, L, fill=1e30):
    """Caches [B,Hk,L,D] holding the interleaved rows k/v [B,S,Hk*D] at positions 0..S-1; the
    rows after them hold `fill`, which would dominate any result that read them."""
    kc = np.full((B, Hk, L, D), fill, np.float32)
    vc = np.full((B, Hk, L, D), fill, np.float32)
    kc[:, :, :S, :] = k.reshape(B, S, Hk, D).transpose(0, 2, 1, 3)
    vc[:, :, :S, :] = v.reshape(B, S, Hk, D).transpose(0, 2, 1, 3)
    return kc, vc


@pytest.mark.parametrize("causal", [False, True])
def test_prefill_cached_from_empty_cache_equals_prefill(oracle_mod, causal):
    """start_pos = 0: the chunk is the whole sequence, so the result is the ordinary prefill
    (padding included: q_lens plays the role of seq_lens)."""
    B, S, H, Hk, D = 2, 7, 4, 2, 4
    q, k, v = (inputs.normal((B, S, n * D), (2101, t)) for t, n in enumerate((H, Hk, Hk)))
    lens = np.array([7, 4])
    kc, vc = _cache_of(k, v, B, S, Hk, D, S + 3)
    for b in range(B):               # keys past a sequence's length are not part of it
        kc[b, :, lens[b]:, :] = 1e30
        vc[b, :, lens[b]:, :] = 1e30
    got = oracle_mod.prefill_cached(q, kc, vc, B, S, H, Hk, D, S + 3, causal, np.zeros(B, np.int32),
                                    q_lens=lens)
    want = oracle_mod.prefill(q, k, v, B, S, H, Hk, D, causal, seq_lens=lens)
    assert np.max(np.abs(got - want)) < 1e-12


def test_prefill_cached_single_token_equals_decode(oracle_mod):
    """T = 1: the chunk is one decode step of length start_pos + 1 (the page's per-token rule)."""
    M, H, Hk, D, L = 3, 4, 2, 4, 10
    q = inputs.normal((M, 1, H * D), (2201, 0))
    kc = inputs.normal((M, Hk, L, D), (2201, 1))
    vc = inputs.normal((M, Hk, L, D), (2201, 2))
    sp = np.array([0, 6, 9], np.int32)
    got = oracle_mod.prefill_cached(q, kc, vc, M, 1, H, Hk, D, L, True, sp)
    want = oracle_mod.decode(q.reshape(M, H * D), kc, vc, M, H, Hk, D, L, sp + 1)
    assert np.max(np.abs(got.reshape(M, H * D) - want)) < 1e-12


def test_prefill_cached_chunks_compose_to_full_prefill(oracle_mod):
    """A causal prefill of S tokens equals a first chunk of c tokens followed by a second chunk
    of S - c tokens behind it (both reading the cache that holds all S rows)."""
    B, S, H, Hk, D, c = 2, 9, 4, 1, 4, 4
    q, k, v = (inputs.normal((B, S, n * D), (2301, t)) for t, n in enumerate((H, Hk, Hk)))
    full = oracle_mod.prefill(q, k, v, B, S, H, Hk, D, True)
    kc, vc = _cache_of(k, v, B, S, Hk, D, S + 2)
    first = oracle_mod.prefill_cached(q[:, :c], kc, vc, B, c, H, Hk, D, S + 2, True, np.zeros(B, np.int32))
    second = oracle_mod.prefill_cached(q[:, c:], kc, vc, B, S - c, H, Hk, D, S + 2, True,
                                       np.full(B, c, np.int32))
    assert np.max(np.abs(first - full[:, :c])) < 1e-12
    assert np.max(np.abs(second - full[:, c:])) < 1e-12


def test_prefill_cached_rejects_chunk_past_capacity(oracle_mod):
    q = inputs.normal((1, 3, 4), 1)
    kc = inputs.normal((1, 1, 5, 4), 2)
    with pytest.raises(ValueError):
        oracle_mod.prefill_cached(q, kc, kc, 1, 3, 1, 1, 4, 5, True, np.array([3]))


# ------------------------------------------------------------ rotary embedding
def test_golden_rope(oracle_mod):
    g = _golden("rope_neox_closed_form.json")
    full = oracle_mod.rope(np.array([g["x_full"]], np.float32), 1, 4, [g["position"]], theta=g["theta"])
    assert np.max(np.abs(full[0] - np.array(g["expected_full"]))) <= g["tolerance"]
    part = oracle_mod.rope(np.array([g["x_partial"]], np.float32), 1, 6, [g["position"]], theta=g["theta"],
                           rotary_ndims=g["rotary_ndims_partial"])
    assert np.max(np.abs(part[0] - np.array(g["expected_partial"]))) <= g["tolerance"]
    same = oracle_mod.rope(np.array([g["x_full"]], np.float32), 1, 4, [0], theta=g["theta"])
    assert np.array_equal(same[0], np.array(g["x_full"], np.float64))


def test_rope_preserves_pair_norms(oracle_mod):
    H, D, r = 3, 16, 12
    x = inputs.normal((5, H * D), 3001)
    pos = np.array([0, 1, 17, 4095, 32767])
    out = oracle_mod.rope(x, H, D, pos, theta=1e6, rotary_ndims=r).reshape(5, H, D)
    x3 = x.astype(np.float64).reshape(5, H, D)
    h = r // 2
    n_in = x3[..., :h] ** 2 + x3[..., h:r] ** 2
    n_out = out[..., :h] ** 2 + out[..., h:r] ** 2
    assert np.max(np.abs(n_in - n_out)) < 1e-9
    assert np.array_equal(out[..., r:], x3[..., r:])       # dims past rotary_ndims untouched


@pytest.mark.parametrize("r", [8, 16])
def test_rope_scores_depend_only_on_relative_position(oracle_mod, r):
    """q at m and k at n score the same as q at m - n and k at 0: the property RoPE exists for."""
    D = 16
    q = inputs.normal((1, D), 3011)
    k = inputs.normal((1, D), 3012)
    for m, n in ((5, 3), (100, 100), (4097, 15), (30000, 29000)):
        a = oracle_mod.rope(q, 1, D, [m], rotary_ndims=r)[0] @ oracle_mod.rope(k, 1, D, [n], rotary_ndims=r)[0]
        b = oracle_mod.rope(q, 1, D, [m - n], rotary_ndims=r)[0] @ oracle_mod.rope(k, 1, D, [0], rotary_ndims=r)[0]
        assert abs(a - b) < 1e-9


def test_rope_rejects_bad_shapes(oracle_mod):
    x = inputs.normal((1, 8), 1)
    for kw in ({"rotary_ndims": 3}, {"rotary_ndims": 10}, {"theta": 0.0}):
        with pytest.raises(ValueError):
            oracle_mod.rope(x, 1, 8, [1], **kw)
