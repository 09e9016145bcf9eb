"""The fp64 graph-transformer attention oracle against what the definition
fixes (CPU only), and planted mistakes that the pins must catch."""
import pytest

import oracle
import oracle_pins_transformer as pins

MUTANTS = {
    "no_scale": ("alpha[q] = g->scale * gt_dot(g, g->q, i, g->key, g->col[b + q], k);",
                 "alpha[q] = gt_dot(g, g->q, i, g->key, g->col[b + q], k);"),
    "value_from_key": ("const double x = gt_feat(&g, val, col[b + e], k, d);",
                       "const double x = gt_feat(&g, key, col[b + e], k, d);"),
    "score_with_destination_key": ("alpha[q] = g->scale * gt_dot(g, g->q, i, g->key, g->col[b + q], k);",
                                   "alpha[q] = g->scale * gt_dot(g, g->q, i, g->key, i, k);"),
    "softmax_jacobian_sign": ("const double de = alpha[e] * (da[e] - delta);",
                              "const double de = alpha[e] * (delta - da[e]);"),
    "dkey_from_key": ("const double qv = gt_feat(&g, q, i, k, d), gv",
                      "const double qv = gt_feat(&g, key, i, k, d), gv"),
    "dval_unweighted": ("dval[x] += alpha[e] * gv;", "dval[x] += gv;"),
    "delta_from_key": ("da[q] = gt_dot(g, dout, i, g->val, g->col[b + q], k);",
                       "da[q] = gt_dot(g, dout, i, g->key, g->col[b + q], k);"),
}


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_gt_oracle_pin(pin):
    pin(oracle.Oracle())


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_gt_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = oracle.source_text("transformer_oracle.c")
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    path = oracle.compile_variant(src.replace(old, new), str(tmp_path / f"mut_{name}.so"),
                                  "transformer_oracle.c")
    mutant = oracle.Oracle(path)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(mutant)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake {name}"
