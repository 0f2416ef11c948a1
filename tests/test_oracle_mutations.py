"""The oracle's pins must catch plausible mistakes.  Each case plants one bug in
a copy of oracle.c (on the CPU), builds it, runs the pin suite against it and
expects a failure.  The real oracle is untouched."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = {
    "forward drops the scale": ("        srow[j] = scale * acc;", "        srow[j] = acc;"),
    "forward exponent sign": ("exp(srow[j] - m)", "exp(m - srow[j])"),
    "causal mask off by one": ("        if (causal && j > i) {\n            srow[j] = -INFINITY;",
                               "        if (causal && j >= i && j > 0) {\n            srow[j] = -INFINITY;"),
    "lse drops the max": ("    return m + log(l);", "    return log(l);"),
    "tiled rescale direction": ("exp(m[r] - ref)", "exp(ref - m[r])"),
    "dV reads P transposed": ("av += P[(size_t)i * N + j] * doh[i * d + c];",
                              "av += P[(size_t)j * N + i] * doh[i * d + c];"),
    "dS drops delta": ("dSi[j] = Pi[j] * (dp - dl);", "dSi[j] = Pi[j] * dp;"),
    "dK misses the scale": ("dkh[j * d + c] = scale * ak;", "dkh[j * d + c] = ak;"),
    "dQ uses V instead of K": ("a += dSi[j] * kh[j * d + c];", "a += dSi[j] * vh[j * d + c];"),
    "E4M3 exponent bias": ("ldexp(1.0 + (double)mant / 8.0, e - 7)", "ldexp(1.0 + (double)mant / 8.0, e - 8)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_bug(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not unique: {old!r}"
    mutant = tmp_path / "oracle_mutant.c"
    mutant.write_text(src.replace(old, new))
    lib = tmp_path / "liboracle_mutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", str(lib),
                    str(mutant), "-lm"], check=True)
    env = dict(os.environ, ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                        "-x", "-q", "-p", "no:cacheprovider"], cwd=ROOT, env=env,
                       stdout=subprocess.PIPE, stderr=subprocess.STDOUT, timeout=600)
    assert r.returncode != 0, f"the pins did not catch: {name}\n" + r.stdout.decode()[-2000:]
