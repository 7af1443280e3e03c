"""Planted mistakes in the oracle must be caught by its pins.

Each case below is a plausible slip in oracle/dcp_oracle.c -- a dropped term,
a wrong sign, a swapped index or stride, a wrong bias or offset, an inverted
flag.  The test writes the mutated C file to a scratch directory, compiles it
exactly as the oracle is compiled, and runs tests/test_oracle.py against that
build (through DCP_ORACLE_LIB).  Every mutant must make at least one pin fail,
so the pins are shown to constrain each part of the oracle rather than merely
agree with it.  CPU only; the mistakes are planted in the oracle, never in the
CUDA path.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "dcp_oracle.c")

# (what the slip is, exact text in dcp_oracle.c, the slip)
MUTANTS = [
    ("logsumexp drops the max term", "return m + log(s);", "return log(s);"),
    ("weight exponent sign flipped", "w[r] = exp(x[r] - G);", "w[r] = exp(G - x[r]);"),
    ("non-finite weight mapped to 1", "if (!isfinite(w[r])) w[r] = 0.0;", "if (!isfinite(w[r])) w[r] = 1.0;"),
    ("NaN LSE class ignored", "if (any_nan) return NAN;", "(void)any_nan;"),
    ("+inf LSE taken as the running max", "else if (x[r] == INFINITY) any_pinf = 1;\n        else if (x[r] > m)",
     "else if (x[r] > m)"),
    ("base-2 input converted the wrong way", "return base == ORACLE_BASE_2 ? l * ln2() : l;",
     "return base == ORACLE_BASE_2 ? l / ln2() : l;"),
    ("returned LSE left in natural-log units", "return base == ORACLE_BASE_2 ? G / ln2() : G;",
     "return G;"),
    ("sanitise flag inverted", "if ((flags & ORACLE_SANITIZE_O) && !isfinite(o)) o = 0.0;",
     "if (!(flags & ORACLE_SANITIZE_O) && !isfinite(o)) o = 0.0;"),
    ("first rank left out of the sum", "for (int r = 0; r < N; ++r) {\n            double o = load_elem",
     "for (int r = 1; r < N; ++r) {\n            double o = load_elem"),
    ("pack peer taken round-robin", "const int p = h / H_pr;", "const int p = h % N;"),
    ("pack local head taken round-robin", "const int hl = h % H_pr;", "const int hl = h / N;"),
    ("pack LSE read from the local head", "&lse[g * l_sg + b * l_sb + h * l_sh], 4);",
     "&lse[g * l_sg + b * l_sb + hl * l_sh], 4);"),
    ("combine rank and token strides swapped", "(g * o_sg + r * o_sn + b * o_sb + h * o_sh)",
     "(g * o_sg + r * o_sb + b * o_sn + h * o_sh)"),
    ("single rank sent through the merge", "if (N == 1) {\n                    const void* src",
     "if (N == 0) {\n                    const void* src"),
    ("unpack LSE word one element early", "memcpy(&lw, rp + (int64_t)D * e, 4);",
     "memcpy(&lw, rp + (int64_t)(D - 1) * e, 4);"),
    ("unpack rank and token strides swapped", "(g * r_sg + r * r_sn + b * r_sb + h * r_sh)",
     "(g * r_sg + r * r_sb + b * r_sn + h * r_sh)"),
    ("fp16 exponent bias off by one", "ldexp((double)(man + 1024), ex - 25)",
     "ldexp((double)(man + 1024), ex - 24)"),
    ("bf16 bits shifted one place short", "uint32_t bits = (uint32_t)h << 16;",
     "uint32_t bits = (uint32_t)h << 15;"),
    ("fp8 exponent bias off by one", "ldexp((double)(man + 8), ex - 10)", "ldexp((double)(man + 8), ex - 11)"),
    ("fp8 top exponent all NaN", "if (ex == 15 && man == 7) {", "if (ex == 15) {"),
    ("bf16 given one element per LSE word", "if (dtype == ORACLE_F16 || dtype == ORACLE_BF16) return 2;",
     "if (dtype == ORACLE_F16) return 2;"),
    ("round-robin share off by one", "return L / n + (r < L % n ? 1 : 0);",
     "return L / n + (r <= L % n ? 1 : 0);"),
    ("empty rank not neutral", "            lse[r] = -INFINITY;\n            continue;",
     "            lse[r] = 0.0;\n            continue;"),
    ("attention probabilities without the scale", "const double p = exp(s * scale - l);",
     "const double p = exp(s - l);"),
    ("latent value read from the rope end", "Or[d] += prob * row[d];", "Or[d] += prob * row[Dk - Dv + d];"),
    ("latent probabilities scored over the value part only",
     "const double prob = exp(scale * latent_dot(q, row, Dk) - lse_nat);",
     "const double prob = exp(scale * latent_dot(q, row, Dv) - lse_nat);"),
    ("latent LSE left in natural-log units for base 2",
     "lse[r] = base == ORACLE_BASE_2 ? lse_nat / ln2() : lse_nat;", "lse[r] = lse_nat;"),
    ("latent attention skips each rank's first token", "for (int t = r; t < L; t += n) z +=",
     "for (int t = r + n; t < L; t += n) z +="),
]


def test_every_mutant_is_distinct_and_present():
    src = open(SRC).read()
    for name, old, new in MUTANTS:
        assert src.count(old) == 1, f"{name}: the original text must occur exactly once"
        assert old != new, name


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(name, old, new, tmp_path):
    src = open(SRC).read()
    assert src.count(old) == 1
    c = tmp_path / "dcp_oracle_mutant.c"
    c.write_text(src.replace(old, new))
    so = tmp_path / "liboracle_mutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", str(so), str(c), "-lm"], check=True)
    env = dict(os.environ, DCP_ORACLE_LIB=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle.py"),
                        "-x", "-q", "-p", "no:cacheprovider", "-m", "not gpu"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    # 1: a pin failed; a negative code: the mutant crashed the pins' process
    assert r.returncode == 1 or r.returncode < 0, (
        f"no pin caught the planted mistake '{name}' (pytest exit {r.returncode}):\n{r.stdout[-1500:]}")
