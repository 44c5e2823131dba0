"""The pins must catch plausible mistakes in the oracle.

Each case plants one mistake in a copy of oracle.c (on the CPU, in a
temporary directory), rebuilds that copy and reruns the pin tests against
it: at least one pin has to fail.  The shipped oracle is never modified."""
import importlib.util
import os

import pytest

import test_oracle_ffn as FFN
import test_oracle_routing as R
import test_residency as RES

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTANTS = {
    "tie_break_to_higher_id": ("(la == lb && a < b)", "(la == lb && a > b)"),
    "phase2_ignores_union": ("if (in_base[o[j]])", "if (1)"),
    "top_p_count_off_by_one": ("if (prefix >= p)\n            return t;",
                               "if (prefix >= p)\n            return t + 1;"),
    "baseline_ignores_top_p": ("nbase[i] = t < k0 ? t : k0;", "nbase[i] = k0;"),
    "partition_drops_one_expert": ("for (int e = 0; e < N; ++e)\n        Z += expf",
                                   "for (int e = 1; e < N; ++e)\n        Z += expf"),
    "weights_not_renormalised": ("ww[j] = exp((double)l[ii[j]] - m) / Z;",
                                 "ww[j] = exp((double)l[ii[j]] - m);"),
    "silu_sign": ("return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    "down_transposed": ("w_down[(size_t)j * F + f]", "w_down[(size_t)f * d + j]"),
    "gate_up_swapped": ("h[f] = silu(g) * u;", "h[f] = silu(u) * g;"),
    "combine_ignores_weight": ("o[c] += w[(size_t)i * kslots + j] * y[c];", "o[c] += y[c];"),
    "bias_subtracted": ("acc += (double)bias[e];", "acc -= (double)bias[e];"),
    "grouping_tokens_descending": ("for (int i = 0; i < B; ++i)\n            if (sel[",
                                   "for (int i = B - 1; i >= 0; --i)\n            if (sel["),
    "padding_tokens_join_union": ("if (i >= B_valid) {\n                nbase[i] = 0;\n                continue;",
                                  "if (0) {\n                nbase[i] = 0;\n                continue;"),
    "max_depth_ignored": ("const int depth = maxP < N ? maxP : N;", "const int depth = N;"),
    "int4_nibble_pairs_swapped": ("const int bit = 4 * (o / 2) + 16 * (o % 2);",
                                  "const int bit = 16 * (o / 2 % 2) + 4 * (o % 2) + 8 * (o / 4);"),
    "int4_scale_row_ignored": ("(size_t)rb * 64 + (size_t)rr * 2;", "(size_t)rb * 64;"),
    "int4_chunk_order_swapped": ("((size_t)rbi * nkb + kb) * chunk", "((size_t)kb * (rows / rb) + rbi) * chunk"),
    "given_baseline_sizes_ignored": ("nbase[i] = nbase_in[i];", "nbase[i] = k0;"),
    "policy_keeps_oea_for_one_token": ("if (B_valid <= 1) {", "if (B_valid < 1) {"),
    "hysteresis_margin_ignored": ("!(S[o] > S[i] + margin)", "!(S[o] > S[i])"),
    "ema_weights_swapped": ("S[e] = alpha * S[e] + (1.0 - alpha) * c[e];", "S[e] = (1.0 - alpha) * S[e] + alpha * c[e];"),
    "selection_ties_to_higher_outsider": ("(o < 0 || S[e] > S[o])", "(o < 0 || S[e] >= S[o])"),
    "policy_smaller_k0_at_small_batches": ("if (B_valid < 16)\n        return (5 * k + 7) / 8;",
                                           "if (B_valid < 16)\n        return (3 * k + 7) / 8;"),
}


def pins():
    """Every pin test, bound to fixed parameters."""
    out = [R.test_topk_invariants_and_grouping, R.test_weights_are_renormalised_scores,
           R.test_top_p_worked_example, R.test_special_cases_reduce_to_known_routers,
           R.test_padding_tokens_select_nothing, R.test_batch_size_policy,
           FFN.test_swiglu_worked_example, FFN.test_expert_algebra,
           FFN.test_combine_is_weighted_sum_in_slot_order, FFN.test_router_logits_match_library,
           FFN.test_dequant_int4_codes_and_layout, FFN.test_int4_round_trip_within_half_step]
    out += [lambda s=s: R.test_topk_matches_brute_force_with_ties(s) for s in range(6)]
    for args in [(2, 0.5, 16, 4), (2, 0.7, 6, 4), (2, 0.6, 5, 5)]:
        out += [lambda s=s, a=args: R.test_oea_matches_brute_force(s, *a) for s in range(4)]
    for d, F in [(8, 5), (96, 40)]:
        out.append(lambda d=d, F=F: FFN.test_expert_matches_library_fp64(d, F))
    out.append(lambda: R.test_union_size_monte_carlo(16, R.OEA, 3))
    out += [lambda s=s: R.test_given_baseline_sizes_follow_the_definitions(s, 2, 12, 4) for s in range(3)]
    out += [RES.test_ema_closed_form, RES.test_margin_zero_gives_the_top_n, RES.test_worked_example_and_hysteresis,
            RES.test_every_member_set_on_tiny_cases]
    out += [lambda s=s, m=m: RES.test_selection_matches_pairing(s, m) for s in range(6) for m in (0.0, 2.0)]
    return out


def load_mutant(tmp_path, name, old, new):
    src = open(os.path.join(ROOT, "oracle", "oracle.c")).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    spec = importlib.util.spec_from_file_location(f"oracle_mutant_{name}",
                                                  os.path.join(ROOT, "oracle", "__init__.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod._SRC = str(path)
    mod._LIB_PATH = str(tmp_path / f"lib{name}.so")
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path, monkeypatch):
    mod = load_mutant(tmp_path, name, *MUTANTS[name])
    monkeypatch.setattr(R, "oracle", mod)
    monkeypatch.setattr(FFN, "oracle", mod)
    monkeypatch.setattr(RES, "oracle", mod)
    caught = 0
    for pin in pins():
        try:
            pin()
        except (AssertionError, ValueError):
            caught += 1
        except pytest.skip.Exception:
            pass
    assert caught > 0, f"no pin fails with the planted mistake {name}"
