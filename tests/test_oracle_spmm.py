"""The fp64 SpMM-family oracle against what the definition fixes (CPU only),
and planted mistakes that the pins must catch."""
import pytest

import oracle
import oracle_pins_spmm as pins

MUTANTS = {
    "mean_divides_by_source_degree": (
        "if (norm == 1) return di > 0 ? 1.0 / (double)di : 0.0;",
        "if (norm == 1) return dj > 0 ? 1.0 / (double)dj : 0.0;"),
    "sym_uses_destination_twice": ("return 1.0 / sqrt((double)di * (double)dj);",
                                   "return 1.0 / sqrt((double)di * (double)di);"),
    "sym_zero_degree_not_masked": ("if (di == 0 || dj == 0) return 0.0;", ""),
    "backward_scatters_to_destination": ("dx[j * F + f] += c * v;", "dx[i * F + f] += c * v;"),
    "forward_gathers_destination_row": (
        "const double v = spmm_widen(x, dtype, j * F + f);",
        "const double v = spmm_widen(x, dtype, i * F + f);"),
    "backward_uses_forward_coefficient_order": (
        "      const double c = spmm_coef(norm, row_ptr, i, j);\n      for (int64_t f = 0; f < F; ++f) {\n        const double v = spmm_widen(dout",
        "      const double c = spmm_coef(norm, row_ptr, j, i);\n      for (int64_t f = 0; f < F; ++f) {\n        const double v = spmm_widen(dout"),
    "multi_edge_counted_once": (
        "    for (int64_t p = row_ptr[i]; p < row_ptr[i + 1]; ++p) {\n      const int64_t j = col[p];\n      const double c = spmm_coef(norm, row_ptr, i, j);\n      for (int64_t f = 0; f < F; ++f) {\n        const double v = spmm_widen(x,",
        "    for (int64_t p = row_ptr[i]; p < row_ptr[i + 1]; ++p) {\n      const int64_t j = col[p];\n      if (p > row_ptr[i] && col[p - 1] == j) continue;\n      const double c = spmm_coef(norm, row_ptr, i, j);\n      for (int64_t f = 0; f < F; ++f) {\n        const double v = spmm_widen(x,"),
}


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_spmm_oracle_pin(pin):
    pin(oracle.Oracle())


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_spmm_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = oracle.source_text("spmm_oracle.c")
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    path = oracle.compile_variant(src.replace(old, new), str(tmp_path / f"mut_{name}.so"),
                                  "spmm_oracle.c")
    mutant = oracle.Oracle(path)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(mutant)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake {name}"
