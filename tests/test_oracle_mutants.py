"""Planted mistakes: each mutant is a copy of the oracle source with one
plausible error (a transposed operand, a wrong sign, a dropped term, a wrong
index or row, an inclusive comparison).  The oracle's pins must reject every
mutant; a mutant that passes all pins would show a gap in the pins."""
from __future__ import annotations

import os
import tempfile

import pytest

import oracle
from oracle import build as obuild
from oracle_pins import ALL_CHECKS

MUTANTS = {
    "ratio_transposed": ("double r = exp(lp - lq);", "double r = exp(lq - lp);"),
    "residual_sign": ("double d = p - q;", "double d = q - p;"),
    "lse_drops_max": ("*lse = M + log(s);", "*lse = log(s);"),
    "draft_rows_unscaled": ("if (row_lse(rd, V, T, &ld[i]) != 0) return;",
                            "if (row_lse(rd, V, 1.0, &ld[i]) != 0) return;"),
    "bonus_wrong_row": ("load_row(a->target, a->dtype, ot + k, V, rt);",
                        "load_row(a->target, a->dtype, ot + k - (k > 0), V, rt);"),
    "resample_uniform_index": ("const double ur = (double)a->u_resample[ot + j];",
                               "const double ur = (double)a->u_resample[od + j];"),
    "accept_inclusive": ("if (u < alpha[i]) continue;", "if (u <= alpha[i]) continue;"),
    "cdf_inclusive": ("if (C > t) {", "if (C >= t) {"),
    "greedy_emits_first_argmax": ("a->out_tokens[ot + n] = am[n];", "a->out_tokens[ot + n] = am[0];"),
    "argmax_last_tie": ("if (z[v] > bv) {", "if (z[v] >= bv) {"),
    "no_stop_at_first_reject": ("j = i;\n        break;", "j = i;"),
    "residual_wrong_draft_row": ("load_row(a->draft, a->dtype, od + j, V, rd);",
                                 "load_row(a->draft, a->dtype, od, V, rd);"),
    "residual_uses_q_for_p": ("double p = exp(rt[v] / T - lt[j]);",
                              "double p = exp(rt[v] / T - lt[0]);"),
    "accept_ratio_no_min": ("alpha[i] = r < 1.0 ? r : 1.0;", "alpha[i] = r;"),
}


@pytest.fixture(scope="module")
def mutant_dir():
    with tempfile.TemporaryDirectory() as d:
        yield d


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name, mutant_dir):
    old, new = MUTANTS[name]
    src = open(obuild.SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique/absent"
    path = os.path.join(mutant_dir, f"{name}.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    lib = oracle.load(obuild.compile_oracle(path, os.path.join(mutant_dir, f"lib_{name}.so")))
    failed = []
    for check_name, check in ALL_CHECKS.items():
        try:
            check(lib)
        except AssertionError:
            failed.append(check_name)
    assert failed, f"mutant {name} passed every pin"
