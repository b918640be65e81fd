"""The oracle's pins must catch plausible mistakes.  Each case copies the oracle
source, plants one mistake on the CPU, builds the copy with gcc and runs the pin
suites against it in a subprocess; at least one pin has to fail."""
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "spec_oracle.c")

MUTANTS = {
    "residual_sign": ("fmax(0.0, P[i] - Q[i])", "fmax(0.0, Q[i] - P[i])"),
    "residual_unnormalised": ("P[i] = fmax(0.0, P[i] - Q[i]) / z;", "P[i] = fmax(0.0, P[i] - Q[i]);"),
    "alpha_inverted": ("fmin(1.0, P[x] / Q[x])", "fmin(1.0, Q[x] / P[x])"),
    "ties_to_higher_index": ("return (x->idx < y->idx) ? -1 : (x->idx > y->idx);",
                             "return (x->idx > y->idx) ? -1 : (x->idx < y->idx);"),
    "top_p_strict": ("if (cum / s_k >= top_p) {", "if (cum / s_k > top_p) {"),
    "top_k_off_by_one": ("int K = (top_k > 0 && top_k < V) ? top_k : V;",
                         "int K = (top_k > 0 && top_k < V) ? top_k + 1 : V;"),
    "temperature_dropped": ("w[j] = exp((r[j].z - m) / T);", "w[j] = exp(r[j].z - m);"),
    "inverse_cdf_off_by_one": ("if (P[i] > 0.0 && cum >= target) {",
                               "if (P[i] > 0.0 && prev >= target) {"),
    "philox_multiplier": ("mult0 = 0xD2511F53u", "mult0 = 0xD2511F55u"),
    "philox_no_key_bump": ("k0 += weyl0;", "k0 += 0;"),
    "uniform_closed_at_zero": ("((x >> 8) + 1u)", "((x >> 8) + 0u)"),
    "no_reset_after_accept": ("for (int c = u + 1; c < N && next < 0; ++c) {\n      if (par[c] != u) continue;\n      int x = tok[c];",
                              "for (int c = u + 1; c < N && next < 0; ++c) {\n      if (par[c] != u) continue;\n      if (u > 0 && c == u + 1) continue;\n      int x = tok[c];"),
    "greedy_first_rejects": ("int ok = (tok[c] == pi.argmax);", "int ok = (tok[c] == pi.argmax) && c != u + 1;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name):
    find, repl = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(find) >= 1, f"mutation anchor for {name} not found"
    with tempfile.TemporaryDirectory() as d:
        c_path = os.path.join(d, "mutant.c")
        so_path = os.path.join(d, "libmutant.so")
        with open(c_path, "w") as f:
            f.write(src.replace(find, repl))
        subprocess.run(["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-o", so_path, c_path,
                        "-lm", "-lpthread"], check=True)
        env = dict(os.environ, SPEC_ORACLE_LIB=so_path)
        r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                            "tests/test_oracle_pins.py", "tests/test_oracle_walk.py"],
                           cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
        assert r.returncode != 0, f"mutant {name} passed every pin:\n{r.stdout[-2000:]}"
