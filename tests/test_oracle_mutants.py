"""Planted mistakes: each mutant of the oracle's C source must fail a pin.

Every mutant is a plausible slip (a dropped scale, an off-by-one in the mask, a
wrong sign in the softmax backward, the wrong GQA head map, a transposed
operand).  The mutant is compiled into a temporary library on the CPU and the
pins of test_oracle.py are run against it; at least one of them must fail.
"""
import importlib.util
import os

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))

MUTANTS = {
    "gqa_map_modulo": ("int g = h / R;", "int g = h % G;"),
    "rows_gqa_map_modulo": ("long g = h / R;", "long g = h % G;"),
    "drop_scale": ("s[j] = scale * dot;", "s[j] = dot;"),
    "causal_off_by_one": ("if (causal && j > i)", "if (causal && j >= i)"),
    "window_off_by_one": ("(j > i - (long)window)", "(j >= i - (long)window)"),
    "sinks_ignored": ("(j < (long)n_sink)", "(j < 0L)"),
    "lse_without_max": ("return m + log(l);", "return log(l);"),
    "softmax_bwd_sign": ("double ds = p[j] * (dp[j] - D);", "double ds = p[j] * (dp[j] + D);"),
    "dq_no_scale": ("dqi[c] += scale * ds * kg[j * (long)d + c];", "dqi[c] += ds * kg[j * (long)d + c];"),
    "dk_wrong_operand": ("dk_t[j * (long)d + c] += scale * ds * qi[c];",
                         "dk_t[j * (long)d + c] += scale * ds * doi[c];"),
    "dv_wrong_operand": ("dv_t[j * (long)d + c] += p[j] * doi[c];",
                         "dv_t[j * (long)d + c] += p[j] * qi[c];"),
    "softmax_not_normalised": ("        p[j] /= l;\n", "        p[j] /= 1.0;\n"),
}


def _pins():
    spec = importlib.util.spec_from_file_location("pins", os.path.join(HERE, "test_oracle.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    calls = [
        mod.test_p5_forward_closed_form,
        mod.test_p5_gradients_closed_form_and_page_gradcheck,
        mod.test_p5_gqa_head_map,
        mod.test_causal_row0_is_v0,
        lambda: mod.test_window_sink_mask_literal_sets("window_sink_mask_w4_s2.json"),
        lambda: mod.test_window_sink_mask_literal_sets("window_sink_mask_w1_s5.json"),
        mod.test_causal_and_full_masks_literal,
        mod.test_equal_keys_closed_form_backward,
        lambda: mod.test_against_torch_sdpa_float64(2, 6, 2, 13, 5, True, 4, 2),
        mod.test_rows_and_group_entry_points_match_full,
    ]
    return calls


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(os.path.join(os.path.dirname(oracle.__file__), "gqa_oracle.c")).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutant = src.replace(old, new)
    c_path = tmp_path / f"{name}.c"
    c_path.write_text(mutant)
    so = oracle.build(force=True, src=str(c_path), out=str(tmp_path / f"lib{name}.so"))
    lib = oracle.load(so)
    saved = oracle._lib
    oracle._lib = lib
    failures = 0
    try:
        for pin in _pins():
            try:
                pin()
            except AssertionError:
                failures += 1
    finally:
        oracle._lib = saved
    assert failures > 0, f"no pin caught the planted mistake {name}"
