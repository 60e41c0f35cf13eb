"""The pins have power: each plausible mistake planted in a copy of the oracle (a dropped term,
a wrong sign, a wrong index, a flipped comparison) makes at least one pin fail.

The mistakes are planted by text substitution into a temporary copy of oracle/spec_oracle.c,
compiled on the CPU; the real oracle is never modified.
"""

import os
import tempfile

import pytest

import oracle
import oracle_pins as pins

# (name, original text, planted mistake); every original must occur in the oracle source.
MUTANTS = [
    ("alpha_inverted", "px / qx;", "qx / px;"),
    ("alpha_without_min", "(qx == 0.0 || px >= qx) ? 1.0 : px / qx", "(qx == 0.0) ? 1.0 : px / qx"),
    ("accept_strict_less", "if ((double)r[n] <= alpha[n])", "if ((double)r[n] < alpha[n])"),
    ("accept_test_dropped", "if ((double)r[n] <= alpha[n])", "if (1)"),
    ("residual_sign_flipped", "double d = pk[i] - qk[i];", "double d = qk[i] - pk[i];"),
    ("residual_not_clamped", "w[i] = d > 0.0 ? d : 0.0;", "w[i] = d;"),
    ("bonus_from_first_row", "/* R6 bonus: draw from p */\n            w[i] = pk[i];",
     "/* R6 bonus: draw from p */\n            w[i] = p[i];"),
    ("softmax_temperature_dropped", "p[i] = exp((l[i] - m) / T);", "p[i] = exp(l[i] - m);"),
    ("softmax_temperature_multiplied", "p[i] = exp((l[i] - m) / T);", "p[i] = exp((l[i] - m) * T);"),
    ("softmax_not_normalised", "p[i] = p[i] / Z;", "p[i] = p[i];"),
    ("cdf_non_strict", "if (C > target) {", "if (C >= target) {"),
    ("cdf_off_by_one", "if (C > target) {\n            pick = i;",
     "if (C > target) {\n            pick = i + 1 < V ? i + 1 : i;"),
    ("cdf_tie_flag_dropped", "if (fabs(Cprev / S - u) <= tol || fabs(C / S - u) <= tol)", "if (0)"),
    ("accept_tie_flag_dropped", "if (fabs((double)r[n] - alpha[n]) <= tol)", "if (0)"),
    ("zero_residual_fallback_dropped", "c = oracle_inverse_cdf(pk, V, (double)u, tol, &S2, &fl);",
     "c = 0;"),
    ("argmax_last_on_ties", "if (l[i] > l[a])", "if (l[i] >= l[a])"),
    ("tree_compares_child_row", "parents[c] == cur && tokens[c] == a)",
     "parents[c] == cur && tokens[c] == amax[c])"),
    ("tree_final_token_from_root", "out_tokens[len] = amax[cur];", "out_tokens[len] = amax[0];"),
    ("tree_parent_check_dropped", "if (parents[i] < 0 || parents[i] >= i)", "if (0)"),
    ("bf16_widening_shift", "[i] << 16;", "[i] << 15;"),
    ("f16_subnormal_scale", "ldexp((double)man, -24)", "ldexp((double)man, -25)"),
    ("ngram_onehot_weight", "q[(size_t)k * V + xb[k]] = 1.0;", "q[(size_t)k * V + xb[k]] = 0.5;"),
    ("greedy_compares_next_row", "while (n < K && x[n] == cand[n])", "while (n < K && x[n] == cand[n + 1])"),
    ("residual_band_not_scaled", "oracle_inverse_cdf(w, V, (double)u, tol / S, &S3, &flw);",
     "oracle_inverse_cdf(w, V, (double)u, tol, &S3, &flw);"),
    ("residual_wide_tier_dropped", "        if (flw)\n            f |= ORF_CDF_TIE_WIDE;", ""),
    ("tree_sample_no_residual_update", "p[i] = w[i] / S;", "p[i] = p[i];"),
    ("tree_sample_residual_not_normalised", "p[i] = w[i] / S;", "p[i] = w[i];"),
    ("tree_sample_residual_sign_flipped", "double d = p[i] - q[i];", "double d = q[i] - p[i];"),
    ("tree_sample_alpha_inverted", "1.0 : p[x] / q[x]; /* step 1, R2 */", "1.0 : q[x] / p[x]; /* step 1, R2 */"),
    ("tree_sample_draw_from_node_p", "tok = oracle_inverse_cdf(p, V, (double)u, tol, &S2, &fl);",
     "tok = oracle_inverse_cdf(p0, V, (double)u, tol, &S2, &fl);"),
    ("tree_sample_draw_band_not_scaled", "oracle_inverse_cdf(p, V, (double)u, tol / R, &S2, &flw);",
     "oracle_inverse_cdf(p, V, (double)u, tol, &S2, &flw);"),
    ("tree_sample_band_not_scaled", "else if (fabs((double)r[c] - a) <= tol / R)",
     "else if (fabs((double)r[c] - a) <= tol)"),
    ("tree_sample_strict_band_scaled", "if (fabs((double)r[c] - a) <= tol)\n                *req_flag |= ORF_ACCEPT_TIE;",
     "if (fabs((double)r[c] - a) <= tol / R)\n                *req_flag |= ORF_ACCEPT_TIE;"),
    ("tree_sample_mass_not_accumulated", "R *= S;", "R = S;"),
    ("tree_sample_accept_strict_less", "int acc = (double)r[c] <= a; /* step 2: accepted */",
     "int acc = (double)r[c] < a; /* step 2: accepted */"),
    ("tree_greedy_walk_final_token", "out_tokens[len] = a;\n            break;",
     "out_tokens[len] = tokens[cur];\n            break;"),
    ("ngram_draft_earliest_occurrence", "for (int i = L - n - 1; i >= 0; i--) {",
     "for (int i = 0; i <= L - n - 1; i++) {"),
    ("ngram_draft_shortest_first", "for (int n = n_max; n >= n_min && n >= 1; n--) {",
     "for (int n = (n_min > 1 ? n_min : 1); n <= n_max; n++) {"),
    ("ngram_draft_no_overlap", "for (int i = L - n - 1; i >= 0; i--) {", "for (int i = L - 2 * n; i >= 0; i--) {"),
    ("ngram_draft_shifted", "draft[k] = ctx[e + k];", "draft[k] = ctx[e + k - 1];"),
    ("kv_compact_wrong_destination",
     "memcpy(cache + (size_t)slots[j] * row_bytes, tmp + (size_t)(j - 1) * row_bytes,",
     "memcpy(cache + (size_t)slots[path[j]] * row_bytes, tmp + (size_t)(j - 1) * row_bytes,"),
    ("kv_compact_last_row_dropped", "for (int j = 1; j <= L; j++) /* read every accepted row before any slot is written */",
     "for (int j = 1; j < L; j++) /* read every accepted row before any slot is written */"),
    ("kv_compact_path_check_dropped", "ok = pt[j] > 0 && pt[j] < N1 && pa[pt[j]] == pt[j - 1];", "ok = 1;"),
    ("tree_walk_per_request_temperature_ignored", "float Tb = temps ? temps[b] : T;", "float Tb = T;"),
    ("draw_rows_no_empty_residual_fallback", "if (!(S > 0.0)) /* R5 */", "if (0) /* R5 */"),
    ("draw_cdf_not_normalised", "cdf[i] = S > 0.0 ? C / S : 0.0;", "cdf[i] = C;"),
    ("walk_draw_row_from_node_p", "const double *wd = p;", "const double *wd = p0;"),
    ("walk_flip_not_applied", "acc = !acc;", "acc = acc;"),
    ("wmax_margin_subtracted", "double d = p[i] - q[i] + 0.5 * tol * (p[i] + q[i]);",
     "double d = p[i] - q[i] - 0.5 * tol * (p[i] + q[i]);"),
    ("walk_wmax_not_normalised", "draw_wmax[i] /= Slast;", "draw_wmax[i] /= 1.0;"),
    ("walk_flip_any_test", "if (flip && fabs((double)r[c] - a) <= tol / R) {", "if (flip) {"),
    ("chain_per_request_temperature_ignored", "*Tb = temps ? temps[b] : T;", "*Tb = T;"),
    ("chain_bad_temperature_accepted", "return (*Tb >= 0.0f) && !isinf(*Tb);", "return 1;"),
    ("bad_token_check_dropped", "if (xb[k] < 0 || xb[k] >= V)\n                e |= ORE_BAD_TOKEN;",
     "if (0)\n                e |= ORE_BAD_TOKEN;"),
]

SRC = open(oracle.SRC).read()


def _first_failing_pin(lib):
    for pin in pins.FAST_PINS + [lambda l: pins.pin_tree_walk_vs_bruteforce(l, n_trees=300),
                                 pins.pin_hand_tree_cases]:
        try:
            pin(lib)
        except (AssertionError, IndexError, ValueError):
            return getattr(pin, "__name__", "tree_bruteforce")
    return None


def test_real_oracle_passes_every_pin():
    assert _first_failing_pin(oracle.load()) is None


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(name, old, new, tmp_path):
    assert old in SRC, f"mutant {name}: original text not found in the oracle source"
    src = tmp_path / "mutant.c"
    src.write_text(SRC.replace(old, new))
    so = oracle.build(str(src), str(tmp_path / f"lib_{name}.so"))
    caught = _first_failing_pin(oracle.load(so))
    assert caught is not None, f"no pin catches the planted mistake '{name}'"
