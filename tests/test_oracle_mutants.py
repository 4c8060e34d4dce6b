"""Plant plausible mistakes in copies of the oracle (on the CPU) and check that the
pins catch every one: a dropped term, a wrong sign, a transposed operand, a wrong
scale or rank, an unstable or miscounting segment builder, a wrong row index."""
import pytest

import oracle
import oracle_pins


def _nth_replace(text, old, new, nth):
    start = -1
    for _ in range(nth + 1):
        start = text.find(old, start + 1)
        assert start >= 0, "mutation site not found: %r (#%d)" % (old, nth)
    return text[:start] + new + text[start + len(old):]


MUTANTS = {
    "rows_missing_scale": ("yi[n] += scale * d;", "yi[n] += d;", 0),
    "grouped_missing_scale": ("yi[n] += scale * d;", "yi[n] += d;", 1),
    "rows_alpha_not_over_r": ("alpha[s] / (double)r", "alpha[s]", 0),
    "grouped_alpha_not_over_r": ("alpha[s] / (double)r", "alpha[s]", 1),
    "merged_alpha_not_over_r": ("alpha[s] / (double)r", "alpha[s]", 2),
    "rows_delta_sign": ("yi[n] += scale * d;", "yi[n] -= scale * d;", 0),
    "rows_A_transposed": ("acc += xi[k] * As[(size_t)k * R + j];",
                          "acc += xi[k] * As[(size_t)j * K + k];", 0),
    "grouped_A_transposed": ("+= xv * As[(size_t)k * R + j];", "+= xv * As[(size_t)j * K + k];", 0),
    "merged_B_transposed": ("* Bs[(size_t)j * N + n];\n                    Wm",
                            "* Bs[(size_t)n * R + j];\n                    Wm", 0),
    "rows_padded_rank": ("const int r = rank[s];", "const int r = R;", 0),
    "grouped_padded_rank": ("const int r = rank[s];", "const int r = R;", 1),
    "rows_base_dropped": ("yi[n] += xk * Wk[n];", "yi[n] += 0.0 * Wk[n];", 0),
    "grouped_base_dropped": ("yi[n] += xk * Wk[n];", "yi[n] += 0.0 * Wk[n];", 1),
    "merged_base_dropped": ("yi[n] += xk * Wk[n];", "yi[n] += 0.0 * Wk[n];", 2),
    "segments_unstable": ("for (int i = 0; i < T; i++) {\n            if (slot[i] == s)",
                          "for (int i = T - 1; i >= 0; i--) {\n            if (slot[i] == s)", 0),
    "segments_bad_ids_uncounted": ("if (slot[i] < -1 || slot[i] >= S) bad++;",
                                   "if (slot[i] < -1) bad++;", 0),
    "merged_wrong_rows": ("if (si != s) continue;", "if (si == s) continue;", 0),
    "rows_expand_columns_reversed": ("d += v[j] * Bs[(size_t)j * N + n];",
                                     "d += v[j] * Bs[(size_t)j * N + (N - 1 - n)];", 0),
    "rows_sample_index_for_row": ("const double* xi = x + (size_t)i * K;\n            double* yi",
                                  "const double* xi = x + (size_t)q * K;\n            double* yi", 0),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new, nth = MUTANTS[name]
    src = _nth_replace(oracle.source_text(), old, new, nth)
    lib = oracle.compile_variant(src, str(tmp_path / ("mut_%s.so" % name)))
    caught = []
    for pin in oracle_pins.PINS:
        try:
            pin(lib)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, "no pin caught mutant %s" % name
