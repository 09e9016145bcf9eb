"""The fp64 reduction-family oracle against what the definition fixes (CPU
only), and planted mistakes that the pins must catch."""
import pytest

import oracle
import oracle_pins_reduce as pins

MUTANTS = {
    "tie_goes_to_largest_source": ("(v == best && j < *who)", "(v == best && j > *who)"),
    "empty_row_minus_infinity": ("  double best = 0.0;\n  *who = -1;",
                                 "  double best = -INFINITY;\n  *who = -1;"),
    "min_uses_max": ("const int better = op == 0 ? v > best : v < best;",
                     "const int better = v > best;"),
    "gradient_to_destination": ("      dx[j * F + f] += g;", "      dx[i * F + f] += g;"),
    "reads_destination_row": ("const double v = red_widen(x, dtype, j * F + f);",
                              "const double v = red_widen(x, dtype, i * F + f);"),
    "first_edge_skipped": ("  for (int64_t p = row_ptr[i]; p < row_ptr[i + 1]; ++p) {\n    const int64_t j = col[p];",
                           "  for (int64_t p = row_ptr[i] + 1; p < row_ptr[i + 1]; ++p) {\n    const int64_t j = col[p];"),
}


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_reduce_oracle_pin(pin):
    pin(oracle.Oracle())


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_reduce_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = oracle.source_text("reduce_oracle.c")
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    path = oracle.compile_variant(src.replace(old, new), str(tmp_path / f"mut_{name}.so"),
                                  "reduce_oracle.c")
    mutant = oracle.Oracle(path)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(mutant)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake {name}"
