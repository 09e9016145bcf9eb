"""The fp64 GATv2 oracle against what the definition fixes (CPU only), and
planted mistakes that the pins must catch."""
import pytest

import oracle
import oracle_pins_gatv2 as pins

MUTANTS = {
    "value_from_destination_side": ("const double x = v2_feat(&g, xl, col[b + q], k, d);",
                                    "const double x = v2_feat(&g, xr, col[b + q], k, d);"),
    "score_without_nonlinearity": (
        "         v2_leaky(v2_feat(g, g->xr, i, k, d) + v2_feat(g, g->xl, j, k, d), g->slope);",
        "         (v2_feat(g, g->xr, i, k, d) + v2_feat(g, g->xl, j, k, d));"),
    "kink_derivative_one": ("static double v2_leaky_grad(double z, double s) { return z > 0.0 ? 1.0 : s; }",
                            "static double v2_leaky_grad(double z, double s) { return z >= 0.0 ? 1.0 : s; }"),
    "softmax_jacobian_sign": ("          const double de = alpha[q] * (da[q] - delta);\n          const double dm = alpha[q] * (fabs(da[q]) + fabs(delta));\n          for (int d = 0; d < D; ++d) {\n            const double z = v2_feat(&g, xr, i, k, d) + v2_feat(&g, xl, j, k, d);\n            const double a = att[k * D + d];",
                              "          const double de = alpha[q] * (delta - da[q]);\n          const double dm = alpha[q] * (fabs(da[q]) + fabs(delta));\n          for (int d = 0; d < D; ++d) {\n            const double z = v2_feat(&g, xr, i, k, d) + v2_feat(&g, xl, j, k, d);\n            const double a = att[k * D + d];"),
    "datt_without_nonlinearity": ("            pa[k * D + d] += de * v2_leaky(z, slope);",
                                  "            pa[k * D + d] += de * z;"),
    "value_term_unweighted": ("            dxl[x] += alpha[q] * gd + de * a * v2_leaky_grad(z, slope);",
                              "            dxl[x] += gd + de * a * v2_leaky_grad(z, slope);"),
    "lse_without_log": ("  return m + log(l);", "  return m + l;"),
}


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_gatv2_oracle_pin(pin):
    pin(oracle.Oracle())


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_gatv2_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = oracle.source_text("gatv2_oracle.c")
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    path = oracle.compile_variant(src.replace(old, new), str(tmp_path / f"mut_{name}.so"),
                                  "gatv2_oracle.c")
    mutant = oracle.Oracle(path)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(mutant)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake {name}"
