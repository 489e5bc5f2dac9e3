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
    "vertical_sign": ("return -g->a_v / (0.5 * (g->h[k] + g->h[k + 1])) * g->area;",
                      "return g->a_v / (0.5 * (g->h[k] + g->h[k + 1])) * g->area;"),
    "lower_face_index": ("return -g->a_v / (0.5 * (g->h[k - 1] + g->h[k])) * g->area;",
                         "return -g->a_v / (0.5 * (g->h[k - 1] + g->h[k - 1])) * g->area;"),
    "face_mean_wrong_cell": ("nb.ae = -0.5 * (g->ah[c] + g->ah[nb.e]);",
                             "nb.ae = -0.5 * (g->ah[c] + g->ah[nb.w]);"),
    "north_is_south": ("nb.n = (int64_t)jp * g->nx + i;", "nb.n = (int64_t)jm * g->nx + i;"),
    "dropped_south_term": ("y += nb.as * d * x[nb.s * nz + k];", ""),
    "mass_not_volume_scaled": ("return g->mass * g->h[k] * g->area;", "return g->mass * g->area;"),
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
    "stopping_ratio_squared": ("double res = rnorm / rho0;",
                               "double res = (rnorm * rnorm) / (rho0 * rho0);"),
}

# Mistakes in the multigrid part, checked against its own pins.
MG_MUTANTS = {
    "mg_area_not_quadrupled": ("4.0 * f->area};", "2.0 * f->area};"),
    "mg_mass_not_area_scaled": ("return g->mass * g->h[k] * g->area;", "return g->mass * g->h[k];"),
    "mg_restriction_averages": (
        "rc[cc + k] = rf[c00 + k] + rf[c10 + k] + rf[c01 + k] + rf[c11 + k];",
        "rc[cc + k] = 0.25 * (rf[c00 + k] + rf[c10 + k] + rf[c01 + k] + rf[c11 + k]);"),
    "mg_prolongation_halved": ("for (int k = 0; k < nz; ++k) xf[cf + k] += ec[cc + k];",
                               "for (int k = 0; k < nz; ++k) xf[cf + k] += 0.5 * ec[cc + k];"),
    "mg_coarse_ah_cell_twice": ("ahf[(2 * J + 1) * nxf + 2 * I + 1];",
                                "ahf[(2 * J + 1) * nxf + 2 * I];"),
    "mg_smoother_undamped": ("for (int64_t i = 0; i < n; ++i) x[i] += mg->omega * z[i];",
                             "for (int64_t i = 0; i < n; ++i) x[i] += z[i];"),
    "mg_residual_sign": ("for (int64_t i = 0; i < n; ++i) mg->t[l][i] = mg->b[l][i] - mg->t[l][i];",
                         "for (int64_t i = 0; i < n; ++i) mg->t[l][i] = mg->t[l][i] - mg->b[l][i];"),
    "mg_no_post_smoothing": ("  mg_prolong_add(g, mg->x[l + 1], mg->x[l]);\n  for (int s = 0; s < mg->nu; ++s) {",
                             "  mg_prolong_add(g, mg->x[l + 1], mg->x[l]);\n  for (int s = 0; s < 0; ++s) {"),
}


def build_mutant(tmp_path, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, "mutation anchor not found: " + old
    mutated = tmp_path / "oracle_mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = tmp_path / "liboracle_mutant.so"
    subprocess.run(["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
                    "-o", str(lib), str(mutated), "-lm"], check=True)
    return lib


def run_pins(lib, pin_file, deselect="not manufactured"):
    env = dict(os.environ, ORACLE_LIB=str(lib))
    return subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                           "-k", deselect, os.path.join(ROOT, "tests", pin_file)],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    lib = build_mutant(tmp_path, *MUTANTS[name])
    res = run_pins(lib, "test_oracle_pins.py")
    assert res.returncode != 0, "mutant %s survived the pins:\n%s" % (name, res.stdout[-2000:])


@pytest.mark.parametrize("name", sorted(MG_MUTANTS))
def test_multigrid_pins_catch_planted_mistake(name, tmp_path):
    lib = build_mutant(tmp_path, *MG_MUTANTS[name])
    res = run_pins(lib, "test_oracle_mg_pins.py", deselect="not fewer_iterations")
    assert res.returncode != 0, "mutant %s survived the pins:\n%s" % (name, res.stdout[-2000:])
