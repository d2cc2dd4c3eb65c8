"""Planted mistakes: each one is a plausible slip in the oracle's arithmetic
(a dropped term, a wrong sign, a swapped index, the wrong rounding); the pins
of tests/test_oracle.py must fail on every one.  The mistakes go into a copy
of oracle.c built in a temporary directory (CPU only; the package's oracle is
untouched), which a child pytest loads through MOE_ORACLE_LIB."""
import os
import subprocess
import sys

import pytest

REPO = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(REPO, "oracle", "oracle.c")

# (name, original text, planted text)
MUTANTS = [
    ("int4 sign", "return v >= 8 ? v - 16 : v;", "return v;"),
    ("int4 nibble order", "int v = high ? (byte >> 4) & 0xF : byte & 0xF;", "int v = high ? byte & 0xF : (byte >> 4) & 0xF;"),
    ("int2 sign", "return v >= 2 ? v - 4 : v;", "return v;"),
    ("int2 field order", "int v = (byte >> (2 * pos)) & 0x3;", "int v = (byte >> (6 - 2 * pos)) & 0x3;"),
    ("int2 byte index", "orc_unpack2(row[k >> 2], (int)(k & 3))", "orc_unpack2(row[k >> 1], (int)(k & 3))"),
    ("route tie to higher index", "if (best < 0 || l[e] > l[best] || (isnan(l[best]) && !isnan(l[e]))) best = e;",
     "if (best < 0 || l[e] >= l[best] || (isnan(l[best]) && !isnan(l[e]))) best = e;"),
    ("route NaN first", "if (best < 0 || l[e] > l[best] || (isnan(l[best]) && !isnan(l[e]))) best = e;",
     "if (best < 0 || l[e] > l[best]) best = e;"),
    ("group scale dropped", "out[n] = a_scale * acc;", "out[n] = acc;"),
    ("gate and up swapped", "h[i] = orc_silu(Gv[i]) * Gv[I + i];", "h[i] = orc_silu(Gv[I + i]) * Gv[i];"),
    ("SiLU sign", "return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    ("requant rounding", "float q = (s > 0.0f) ? rintf((float)h[i] / s) : 0.0f;",
     "float q = (s > 0.0f) ? roundf((float)h[i] / s) : 0.0f;"),
    ("requant scale", "*sh = s;", "*sh = s * 1.0001f;"),
    ("shared expert dropped", "for (int64_t s = 0; s < d->n_shared; ++s) {", "for (int64_t s = 0; s < 0; ++s) {"),
    ("routing weight dropped", "for (int64_t n = 0; n < H; ++n) o[n] += w[j] * y[n];",
     "for (int64_t n = 0; n < H; ++n) o[n] += y[n];"),
    ("permute not stable", "int32_t pos = offsets[e] + cursor[e];", "int32_t pos = offsets[e + 1] - 1 - cursor[e];"),
    ("partials index", "acc += (int32_t)a[kk] * code_at(row, kk, bits);", "acc += (int32_t)a[kk] * code_at(row, kk ^ 1, bits);"),
    ("group scale order", "acc += (double)s[n * ng + q] * (double)P[n * ng + q];",
     "acc += (double)s[n * ng + (ng - 1 - q)] * (double)P[n * ng + q];"),
    ("S0 scale", "        float s = amax / 127.0f;\n        x_scale[t] = s;", "        float s = amax / 128.0f;\n        x_scale[t] = s;"),
    ("S0 rounding", "float q = (s > 0.0f) ? rintf(v / s) : 0.0f;", "float q = (s > 0.0f) ? roundf(v / s) : 0.0f;"),
    ("S0 widening", "uint32_t bits = (uint32_t)x[t * H + h] << 16;\n            float v;\n            memcpy(&v, &bits, sizeof v);\n            float q",
     "uint32_t bits = (uint32_t)x[t * H + h] << 15;\n            float v;\n            memcpy(&v, &bits, sizeof v);\n            float q"),
]


@pytest.mark.parametrize("name,orig,planted", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(name, orig, planted, tmp_path):
    src = open(SRC).read()
    assert src.count(orig) == 1, f"{name}: the original text is not in oracle.c exactly once"
    mutated = tmp_path / "oracle.c"
    mutated.write_text(src.replace(orig, planted))
    lib = tmp_path / "liboracle_mutant.so"
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
                    "-I", os.path.join(REPO, "oracle"), "-o", str(lib), str(mutated), "-lm"], check=True)
    env = dict(os.environ, MOE_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(REPO, "tests", "test_oracle.py"), "-x", "-q",
                        "-p", "no:cacheprovider"], cwd=REPO, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"{name}: the oracle pins did not catch it\n{r.stdout[-2000:]}"


def test_unmodified_copy_passes_the_same_harness(tmp_path):
    """Control: the same build and child run on an unmodified copy passes (the mutants fail for their mistake)."""
    lib = tmp_path / "liboracle_copy.so"
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
                    "-I", os.path.join(REPO, "oracle"), "-o", str(lib), SRC, "-lm"], check=True)
    env = dict(os.environ, MOE_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(REPO, "tests", "test_oracle.py"), "-x", "-q",
                        "-p", "no:cacheprovider"], cwd=REPO, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:]
