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
    "dV reads P transposed": ("dvh[j * d + c] += Pi[j] * doh[i * d + c];",
                              "dvh[j * d + c] += P[(size_t)j * N + i] * doh[i * d + c];"),
    "dS drops delta": ("dSi[j] = Pi[j] * (dp - dl);", "dSi[j] = Pi[j] * dp;"),
    "dK misses the scale": ("dkh[j * d + c] *= scale;", "dkh[j * d + c] *= 1.0;"),
    "dQ uses V instead of K": ("dqi[c] += dSi[j] * kh[j * d + c];", "dqi[c] += dSi[j] * vh[j * d + c];"),
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


# Mistakes planted in the Python part of the oracle (grouped-query, key shards, the
# merge, per-block E4M3 factors): a mutated copy of the package shadows the real one
# (same compiled library) while the pins run.
PY_MUTANTS = {
    "per-block factor reaches the wrong rows": (
        "    return x * f[..., np.arange(N) // block][..., None]",
        "    return x * f[..., np.arange(N) % f.shape[-1]][..., None]"),
    "GQA dK averages the group instead of summing": (
        "    return (dq, dk.reshape(B, H_kv, g, N, d).sum(axis=2),",
        "    return (dq, dk.reshape(B, H_kv, g, N, d).mean(axis=2),"),
    "key shard: causal offsets swapped": (
        "        masked = (kv_offset + np.arange(Nkv))[None, :] > (q_offset + np.arange(Nq))[:, None]",
        "        masked = (q_offset + np.arange(Nkv))[None, :] > (kv_offset + np.arange(Nq))[:, None]"),
    "key shard: lse drops the max": (
        "    lse = np.where(seen, m + np.log(np.where(seen, l, 1.0)), -np.inf)\n    return o, lse",
        "    lse = np.where(seen, np.log(np.where(seen, l, 1.0)), -np.inf)\n    return o, lse"),
    "merge weights inverted": ("    w = np.exp(L - mm[None])", "    w = np.exp(mm[None] - L)"),
}


@pytest.mark.parametrize("name", sorted(PY_MUTANTS) + ["(unchanged copy)"])
def test_pins_catch_planted_python_bug(name, tmp_path):
    import shutil
    import oracle
    real_lib = oracle.lib()._name  # built once; the copy loads it through ORACLE_LIB
    # the control: an unchanged copy must pass, so a caught mutant is caught by a pin
    old, new = PY_MUTANTS.get(name, ('"""fp64 CPU oracle', '"""fp64 CPU oracle'))
    pkg = tmp_path / "oracle"
    shutil.copytree(os.path.join(ROOT, "oracle"), pkg, ignore=shutil.ignore_patterns("_lib", "__pycache__"))
    src = (pkg / "__init__.py").read_text()
    assert src.count(old) == 1, f"mutation anchor not unique: {old!r}"
    (pkg / "__init__.py").write_text(src.replace(old, new))
    env = dict(os.environ, ORACLE_LIB=real_lib,
               PYTHONPATH=os.pathsep.join([str(tmp_path), ROOT] + [p for p in [os.environ.get("PYTHONPATH")] if p]))
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                        "-x", "-q", "-p", "no:cacheprovider"], cwd=str(tmp_path), env=env,
                       stdout=subprocess.PIPE, stderr=subprocess.STDOUT, timeout=600)
    out = r.stdout.decode()
    assert "passed" in out or "failed" in out, out[-2000:]
    if name not in PY_MUTANTS:
        assert r.returncode == 0, "the unchanged copy fails the pins\n" + out[-2000:]
        return
    assert r.returncode != 0, f"the pins did not catch: {name}\n" + out[-2000:]
