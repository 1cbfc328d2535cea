"""CPU pins of the oracle's tree verify and tree drafting, and planted
mistakes in copies of the oracle that the pins must reject."""
from __future__ import annotations

import os
import tempfile

import pytest

import oracle
from oracle import build as obuild
from tree_pins import TREE_CHECKS


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("name", sorted(TREE_CHECKS))
def test_tree_pin(lib, name):
    TREE_CHECKS[name](lib)


MUTANTS = {
    "no_residual_update": ("for (int v = 0; v < V; ++v) p[v] = w[v] / Z;", ";"),
    "residual_not_normalised": ("p[v] = w[v] / Z;", "p[v] = w[v];"),
    "later_candidates_against_p0": ("double r = p[x] / q[x];",
                                    "double r = exp((rt[x] / T - Lt) - (rd[x] / T - Ld));"),
    "draw_with_root_uniform": ("token = inverse_cdf(w, V, (double)a->u_resample[u], &m);",
                               "token = inverse_cdf(w, V, (double)a->u_resample[g0], &m);"),
    "greedy_last_matching_child": ("c < g0 + n && next < 0; ++c)", "c < g0 + n; ++c)"),
    "accept_inclusive": ("if (uc < alpha) {", "if (uc <= alpha) {"),
    "drafting_from_own_row": ("load_row(draft_logits, dtype, pa, V, z);", "load_row(draft_logits, dtype, g, V, z);"),
    "stay_at_parent": ("            path[nacc++] = a->tokens[next];\n            u = next;\n            continue;\n        }\n        /* every",
                       "            path[nacc++] = a->tokens[next];\n            break;\n        }\n        /* every"),
}


@pytest.fixture(scope="module")
def mutant_dir():
    with tempfile.TemporaryDirectory() as d:
        yield d


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_tree_pins_reject_mutant(name, mutant_dir):
    old, new = MUTANTS[name]
    src = open(obuild.SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique/absent"
    path = os.path.join(mutant_dir, f"{name}.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    mlib = oracle.load(obuild.compile_oracle(path, os.path.join(mutant_dir, f"lib_{name}.so")))
    failed = []
    for check_name, check in TREE_CHECKS.items():
        try:
            check(mlib)
        except (AssertionError, IndexError, ValueError):
            failed.append(check_name)
    assert failed, f"mutant {name} passed every tree pin"
