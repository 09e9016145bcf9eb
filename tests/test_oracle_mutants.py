"""Plant plausible mistakes in a copy of the oracle and check that the pins
catch every one of them (each mistake must make at least one pin fail)."""
import pytest

import oracle
import oracle_pins

MUTANTS = {
    "drop_dst_score_term": ("dh[x] += ds_src[j * H + k] * as + ds_dst[j * H + k] * ad;",
                            "dh[x] += ds_src[j * H + k] * as;"),
    "a_src_for_destination": ("const double sd = head_dot(g, g->a_dst, g->h, i, k);",
                              "const double sd = head_dot(g, g->a_src, g->h, i, k);"),
    "kink_derivative_one": ("return z > 0.0 ? 1.0 : slope;", "return z >= 0.0 ? 1.0 : slope;"),
    "softmax_jacobian_sign": ("ds += alpha[q] * (da[q] - delta) * leaky_grad(z[q], g->slope);",
                              "ds += alpha[q] * (delta - da[q]) * leaky_grad(z[q], g->slope);"),
    "value_from_destination": ("const double x = feat(&g, h, col[b + q], k, d);",
                               "const double x = feat(&g, h, i, k, d);"),
    "no_leaky_slope": ("return z > 0.0 ? z : slope * z;", "return z > 0.0 ? z : z;"),
    "lse_without_log": ("return m + log(l);", "return m + l;"),
    "da_dst_from_src_side": ("da_dst[k * D + d] += ds_dst[j * H + k] * hv;",
                             "da_dst[k * D + d] += ds_src[j * H + k] * hv;"),
    "value_term_unweighted": ("dh[(j * H + k) * (int64_t)D + d] += alpha[q] * x;",
                              "dh[(j * H + k) * (int64_t)D + d] += x;"),
    "row_source_offset": ("const int64_t j = g->col[b + q];\n    z[q]",
                          "const int64_t j = g->col[b + (q + 1) % deg];\n    z[q]"),
    # the per-node backward rows
    "rows_alpha_from_max": ("const double alpha = exp(leaky(zz, slope) - s[1]);",
                            "const double alpha = exp(leaky(zz, slope) - s[0]);"),
    "rows_drop_dst_term": ("row[d] += ds_src * as + sj[3] * ad;", "row[d] += ds_src * as;"),
    "rows_delta_sign": ("ds_src += alpha * (da - s[2]) * leaky_grad(zz, slope);",
                        "ds_src += alpha * (da + s[2]) * leaky_grad(zz, slope);"),
    # the kink ambiguity
    "kink_without_weight": ("fabs(1.0 - g->slope) * alpha[q] * fabs(da[q] - delta) : 0.0;",
                            "fabs(1.0 - g->slope) * fabs(da[q] - delta) : 0.0;"),
    "kink_src_to_dst_vector": ("dh_kink[x] = kink_src[j * H + k] * fabs(as) + kink_dst[j * H + k] * fabs(ad);",
                               "dh_kink[x] = kink_src[j * H + k] * fabs(ad) + kink_dst[j * H + k] * fabs(as);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = oracle.source_text()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    path = oracle.compile_variant(src.replace(old, new), str(tmp_path / f"mut_{name}.so"))
    mutant = oracle.Oracle(path)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(mutant)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake {name}"
