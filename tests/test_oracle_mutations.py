"""The oracle's pins must catch plausible mistakes.

Each case copies rkv_oracle.c, plants one mistake (a dropped term, a wrong sign
or index, a swapped operand, an off-by-one mask), compiles the copy with gcc and
runs the pin checks of test_oracle_pins against it: at least one must fail.
Everything happens on the CPU.
"""
import os
import subprocess

import numpy as np
import pytest

import oracle
import tests.test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "rkv_oracle.c")

MUTATIONS = {
    "causal_off_by_one": ("return causal ? i + 1 : len;", "return causal ? i : len;"),
    "gqa_modulo_grouping": ("return h / (H / Hk);", "return h % Hk;"),
    "scale_dropped": ("scores[j] = acc * scale;", "scores[j] = acc;"),
    "not_normalised": ("double p = scores[j] / sum;", "double p = scores[j];"),
    "values_from_keys": ("const float* vj = v_base", "const float* vj = k_base"),
    "exponent_sign": ("exp(scores[j] - smax)", "exp(smax - scores[j])"),
    "padded_rows_kept": ("if (i >= len) return 0;", "if (i >= len) return len;"),
    "decode_reads_full_cache": ("seq_lens[m] > 0 ? seq_lens[m] : 0", "Lmax"),
    "scatter_row_index": ("+ kh) * Lmax + pos) * D;", "+ kh) * Lmax + t) * D;"),
    "scatter_head_stride": ("* Hk * D + (int64_t)kh * D;", "* Hk * D;"),
    "query_head_offset": ("* q_row + (int64_t)h * D;\n            const float* kb",
                          "* q_row;\n            const float* kb"),
    "chunk_causal_off_by_one": ("n_keys = causal ? p0 + i + 1 : p0 + n;", "n_keys = causal ? p0 + i : p0 + n;"),
    "chunk_ignores_start": ("n_keys = causal ? p0 + i + 1 : p0 + n;", "n_keys = causal ? i + 1 : n;"),
    "chunk_noncausal_sees_capacity": ("n_keys = causal ? p0 + i + 1 : p0 + n;",
                                      "n_keys = causal ? p0 + i + 1 : Lmax;"),
    "chunk_padded_rows_kept": ("if (i < n) n_keys", "if (i < T) n_keys"),
    "rope_rotation_sign": ("oh[i] = x1 * c - x2 * s;", "oh[i] = x1 * c + x2 * s;"),
    "rope_adjacent_pairs": ("x2 = (double)xh[i + half];", "x2 = (double)xh[i ^ 1];"),
    "rope_frequency_over_head_dim": ("(double)i / (double)rotary_ndims", "(double)i / (double)head_dim"),
    "rope_position_ignored": ("const double pos = (double)positions[row];", "const double pos = 1.0;"),
}


def _pin_checks():
    """(name, callable) for every pin; each raises AssertionError on failure."""
    om = oracle
    checks = []
    for name in ("two_keys_closed_form.json", "equal_scores_mean.json", "gqa_single_key.json"):
        for causal in (False, True):
            checks.append(lambda n=name, c=causal: pins.test_golden_prefill(om, n, c))
    checks.append(lambda: pins.test_golden_decode(om))
    checks.append(lambda: pins.test_golden_scatter(om))
    for ci in range(len(pins._TINY_CASES)):
        checks.append(lambda ci=ci: pins.test_prefill_matches_brute_force(om, ci))
    checks.append(lambda: pins.test_decode_matches_brute_force(om, 3, 4, 2, 4, 9, [9, 1, 5]))
    checks.append(lambda: pins.test_decode_equals_last_row_of_causal_prefill(om))
    checks.append(lambda: pins.test_scatter_readback_identity_and_canaries(om))
    checks.append(lambda: pins.test_padded_query_rows_are_zero(om))
    for causal in (False, True):
        checks.append(lambda c=causal: pins.test_golden_prefill_cached(om, c))
        checks.append(lambda c=causal: pins.test_prefill_cached_from_empty_cache_equals_prefill(om, c))
    for ci in range(len(pins._CACHED_CASES)):
        checks.append(lambda ci=ci: pins.test_prefill_cached_matches_brute_force(om, ci))
    checks.append(lambda: pins.test_prefill_cached_single_token_equals_decode(om))
    checks.append(lambda: pins.test_prefill_cached_chunks_compose_to_full_prefill(om))
    checks.append(lambda: pins.test_golden_rope(om))
    checks.append(lambda: pins.test_rope_preserves_pair_norms(om))
    for r in (8, 16):
        checks.append(lambda r=r: pins.test_rope_scores_depend_only_on_relative_position(om, r))
    return checks


def test_unmutated_oracle_passes_every_check():
    for chk in _pin_checks():
        chk()


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(tmp_path, name):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fopenmp", str(mutated),
                    "-o", str(lib), "-lm"], check=True)
    caught = 0
    with oracle.using_library(str(lib)):
        for chk in _pin_checks():
            try:
                with np.errstate(all="ignore"):
                    chk()
            except (AssertionError, ValueError):
                caught += 1
    assert caught > 0, f"planted mistake {name!r} passed every pin"
