"""Mutation check of the oracle's pins.

Each case plants one plausible mistake (a flipped sign, a wrong neighbour
index, a dropped term, a swapped operand) in a private copy of the oracle
source, builds it, and runs the pin suite against it in a subprocess: at
least one pin must fail.  The oracle itself is never modified.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle_pcg.c")

MUTANTS = {
    "vertical_sign": ("return -g->a_v / (0.5 * (g->h[k] + g->h[k + 1]));",
                      "return g->a_v / (0.5 * (g->h[k] + g->h[k + 1]));"),
    "lower_face_index": ("return -g->a_v / (0.5 * (g->h[k - 1] + g->h[k]));",
                         "return -g->a_v / (0.5 * (g->h[k - 1] + g->h[k - 1]));"),
    "face_mean_wrong_cell": ("nb.ae = -0.5 * (g->ah[c] + g->ah[nb.e]);",
                             "nb.ae = -0.5 * (g->ah[c] + g->ah[nb.w]);"),
    "north_is_south": ("nb.n = (int64_t)jp * g->nx + i;", "nb.n = (int64_t)jm * g->nx + i;"),
    "dropped_south_term": ("y += nb.as * d * x[nb.s * nz + k];", ""),
    "mass_not_volume_scaled": ("return g->mass * g->h[k];", "return g->mass;"),
    "diag_sign_alpha": ("double diag = (a - b - c) - alpha_T * d;                  /* eq. (8) */",
                        "double diag = (a - b - c) + alpha_T * d;"),
    "thomas_sub_sup_swapped": ("double sub = c, sup = b;", "double sub = b, sup = c;"),
    "back_substitution_sign": ("z[k] = y[k] - phi[k] * z[k + 1];",
                               "z[k] = y[k] + phi[k] * z[k + 1];"),
    "precond_drops_horizontal_diag": (
        "  double alpha_T = nb.ae + nb.aw + nb.an + nb.as;\n  int nz = g->nz;",
        "  double alpha_T = 0.0;\n  int nz = g->nz;"),
    "beta_inverted": ("double beta = kappa_new / kappa;", "double beta = kappa / kappa_new;"),
    "direction_unpreconditioned": ("p[l] = z[l] + beta * p[l];", "p[l] = r[l] + beta * p[l];"),
    "residual_sign": ("r[l] -= alpha * q[l];", "r[l] += alpha * q[l];"),
    "solution_uses_q": ("x[l] += alpha * p[l];", "x[l] += alpha * q[l];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, "mutation anchor not found: " + name
    mutated = tmp_path / "oracle_mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = tmp_path / "liboracle_mutant.so"
    subprocess.run(["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
                    "-o", str(lib), str(mutated), "-lm"], check=True)
    env = dict(os.environ, ORACLE_LIB=str(lib))
    res = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                          "-k", "not manufactured", os.path.join(ROOT, "tests",
                                                                 "test_oracle_pins.py")],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert res.returncode != 0, "mutant %s survived the pins:\n%s" % (name, res.stdout[-2000:])
