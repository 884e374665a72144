"""Planted mistakes in the oracle: each mutant is a copy of the oracle's C source with
one plausible error (a dropped term, a wrong sign, an off-by-one, a transposed index
or operand), compiled with the oracle's own flags and loaded in its place; at least
one pin of test_oracle.py must reject every mutant.  A control build of the
unchanged source must pass all of them, so that a rejection means the mistake, not
the harness.  CPU only; the builds go to a git-ignored folder beside the oracle."""
import os

import pytest

import oracle
import test_oracle as pins

_DIR = os.path.join(os.path.dirname(oracle.__file__), "_mutants")
_SRC = os.path.join(os.path.dirname(oracle.__file__), "focus_oracle.c")

# name: (text in the source, replacement, which occurrence)
MUTANTS = {
    "score_drops_last_term": (
        "for (int t = 0; t < DG; ++t) s += (double)ri[t] * (double)cg[t];",
        "for (int t = 0; t < DG - 1; ++t) s += (double)ri[t] * (double)cg[t];", 0),
    "topk_ties_go_high": ("(best < 0 || key[g] > key[best])", "(best < 0 || key[g] >= key[best])", 0),
    "sinkhorn_column_step_sign": (
        "beta[g] = log((double)N / (double)K) - logsumexp(col, N, 1);",
        "beta[g] = log((double)N / (double)K) + logsumexp(col, N, 1);", 0),
    "sinkhorn_marginal_inverted": ("log((double)N / (double)K)", "log((double)K / (double)N)", 0),
    "sinkhorn_row_step_drops_beta": (
        "for (int g = 0; g < K; ++g) row[g] = L[i * K + g] + beta[g];",
        "for (int g = 0; g < K; ++g) row[g] = L[i * K + g];", 0),
    "window_off_by_one": ("if (i - j < w) return 1;", "if (i - j <= w) return 1;", 0),
    "exact_group_set_instead_of_overlap": ("return (mi & mj) != 0;", "return mi == mj;", 0),
    "diagonal_excluded": ("if (j > i) return 0;", "if (j >= i) return 0;", 0),
    "logits_unscaled": ("s *= J->scale;", "s *= 1.0;", 0),
    "lse_drops_the_max": ("const double lse = mx + log(sum);", "const double lse = log(sum);", 0),
    "kv_head_map_transposed": ("const int kvh = h / (J->H / J->H_kv);", "const int kvh = h % J->H_kv;", 0),
    "routing_head_map_transposed": ("const int rho = kvh / (J->H_kv / J->R);", "const int rho = kvh % J->R;", 0),
    "value_row_of_the_query": (
        "const uint16_t* vj = J->v + (((int64_t)b * J->N + j_buf[a]) * J->H_kv + kvh) * d;",
        "const uint16_t* vj = J->v + (((int64_t)b * J->N + i) * J->H_kv + kvh) * d;", 0),
    "ds_sign": ("const double ds = p * (dp_buf[a] - D);", "const double ds = p * (dp_buf[a] + D);", 0),
    "dk_drops_scale": ("dk[t] += J->scale * ds * qv[t];", "dk[t] += ds * qv[t];", 0),
    "dv_uses_ds": ("dv[t] += p * gv[t];", "dv[t] += ds * gv[t];", 0),
    "dq_transposed_operand": (
        "for (int t = 0; t < d; ++t) dq[t] += J->scale * ds * bf16_to_double(kj[t]);",
        "for (int t = 0; t < d; ++t) dq[t] += J->scale * ds * qv[t];", 0),
    "D_drops_probability": (
        "for (int64_t a = 0; a < n; ++a) D += exp(s_buf[a] - lse) * dp_buf[a];",
        "for (int64_t a = 0; a < n; ++a) D += dp_buf[a];", 0),
    "backward_kv_head_map_transposed": (
        "const int kvh = h / (J->H / J->H_kv);", "const int kvh = h % J->H_kv;", 1),
    "backward_routing_head_map_transposed": (
        "const int rho = kvh / (J->H_kv / J->R);", "const int rho = kvh % J->R;", 1),
    "backward_logits_unscaled": ("s_buf[n] = s * J->scale;", "s_buf[n] = s;", 0),
}

PINS = [
    lambda: pins.test_scores_match_matmul_and_topk_is_best_subset(4, 2),
    lambda: pins.test_topk_matches_stable_argsort_and_ties_go_low(),
    lambda: pins.test_sinkhorn_marginals_converge_to_balanced_groups(),
    lambda: pins.test_sinkhorn_matches_probability_domain_matrix_scaling(),
    lambda: pins.test_sinkhorn_first_column_potentials_closed_form(),
    lambda: pins.test_allowed_pairs_brute_force_and_closed_forms(),
    lambda: pins.test_attention_matches_dense_masked_softmax(1, 70, 2, 2, 1, 16, 4, 2, 5),
    lambda: pins.test_attention_matches_dense_masked_softmax(2, 97, 4, 2, 2, 8, 5, 1, 9),
    lambda: pins.test_attention_matches_dense_masked_softmax(1, 60, 8, 4, 2, 8, 4, 2, 5),
    lambda: pins.test_special_cases_reduce_to_dense_causal("K1"),
    lambda: pins.test_identical_keys_reveal_the_attended_set(),
    lambda: pins.test_gradients_reduce_to_dense_causal_autograd("K1"),
    lambda: pins.test_gradients_match_dense_masked_softmax_autograd(1, 60, 8, 4, 2, 8, 4, 2, 5),
    lambda: pins.test_gradient_sum_rules(2, 80, 4, 2, 2, 8, 5, 2, 6),
]


def _mutate(text: str, old: str, new: str, occurrence: int) -> str:
    at = -1
    for _ in range(occurrence + 1):
        at = text.index(old, at + 1)
    return text[:at] + new + text[at + len(old):]


def _build(name: str, source: str) -> str:
    os.makedirs(_DIR, exist_ok=True)
    return oracle.compile_variant(source, os.path.join(_DIR, f"{name}_{os.getpid()}.so"))


def _failing_pins(path: str) -> list[int]:
    failed = []
    with oracle.use_library(path):
        for f in (path, path[:-3] + ".c"):  # loaded: the files are no longer needed
            os.remove(f)
        for n, pin in enumerate(PINS):
            try:
                pin()
            except Exception:  # an assertion, or values a pin cannot use (NaN, inf)
                failed.append(n)
    return failed


def test_control_build_passes_every_pin():
    src = open(_SRC).read()
    assert _failing_pins(_build("control", src)) == []


@pytest.mark.parametrize("name", list(MUTANTS))
def test_pins_reject_planted_mistake(name):
    old, new, occurrence = MUTANTS[name]
    src = open(_SRC).read()
    mutant = _mutate(src, old, new, occurrence)
    assert mutant != src
    failed = _failing_pins(_build(name, mutant))
    assert failed, f"no pin rejects the mutant {name}"
