"""Plant mistakes in a copy of the oracle's C source and check that the pins
in test_oracle_pins.py catch every one.

Each mutant is compiled from oracle.c with one textual change (a dropped
term, a wrong sign, a transposed or mis-indexed operand, a flipped filter, a
wrong padding sign, swapped filter axes) and the pin suite runs against it in
a child process (ORACLE_LIB points the loader at the mutant). The child must
fail; if it passes, the pins are blind to that mistake.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = {
    "dropped_last_k": ("for (int64_t k = 0; k < K; ++k)", "for (int64_t k = 0; k < K - 1; ++k)"),
    "wrong_sign": ("sum += prod;\n                sabs", "sum -= prod;\n                sabs"),
    "abs_not_abs": ("sabs += fabs(prod);\n            }\n            ref[ii", "sabs += prod;\n            }\n            ref[ii"),
    "b_row_index": ("B[j * ldb + k]", "B[(j + (k & 1)) % N * ldb + k]"),
    "a_index_shift": ("A[i * lda + k]", "A[i * lda + (K - 1 - k)]"),
    "conv_flipped_filter": ("w + ((k * R + r) * S + s) * C", "w + ((k * R + (R - 1 - r)) * S + (S - 1 - s)) * C"),
    "conv_pad_sign": ("const int64_t h = p * st - pad + r;", "const int64_t h = p * st + pad + r;"),
    "conv_swapped_rs": ("const int64_t h = p * st - pad + r;", "const int64_t h = p * st - pad + (r * S + 0) % R;"),
    "conv_q_stride": ("const int64_t ww = q * st - pad + s;", "const int64_t ww = q - pad + s;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, "mutation anchor not found"
    mutant_c = tmp_path / "mutant.c"
    mutant_c.write_text(src.replace(old, new, 1))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", str(mutant_c), "-o", str(lib), "-lm"],
                   check=True, capture_output=True)
    env = dict(os.environ, ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"pins did not catch mutant {name}:\n{r.stdout[-2000:]}"


# Mistakes in the acceptance rule (oracle/__init__.py), planted in a copy of
# the package that the pin suite then imports in place of the real one.
TOLERANCE_MUTANTS = {
    "bf16_term_2_pow_7": ("np.abs(ref) * 2.0 ** -8", "np.abs(ref) * 2.0 ** -7"),
    "bf16_term_2_pow_9": ("np.abs(ref) * 2.0 ** -8", "np.abs(ref) * 2.0 ** -9"),
    "bf16_term_signed": ("np.abs(ref) * 2.0 ** -8", "ref * 2.0 ** -8"),
    "bf16_term_on_fp32": ("    if out_bf16:\n        tol = tol + np.abs(ref)", "    if True:\n        tol = tol + np.abs(ref)"),
    "abs_scale_1e_2": ("tol = 1e-3 * ab + 1e-6", "tol = 1e-2 * ab + 1e-6"),
}

_LOAD_MUTANT = """
import importlib.util, sys
pkg = sys.argv[1]
spec = importlib.util.spec_from_file_location("oracle", pkg + "/__init__.py", submodule_search_locations=[pkg])
mod = importlib.util.module_from_spec(spec)
sys.modules["oracle"] = mod
spec.loader.exec_module(mod)
import pytest
sys.exit(pytest.main(["-q", "-x", "-p", "no:cacheprovider", sys.argv[2]]))
"""


@pytest.mark.parametrize("name", sorted(TOLERANCE_MUTANTS))
def test_pins_catch_planted_tolerance_mistake(name, tmp_path):
    import shutil

    sys.path.insert(0, ROOT)
    from oracle import build as oracle_build

    lib = oracle_build.build()
    old, new = TOLERANCE_MUTANTS[name]
    pkg = tmp_path / "oracle"
    pkg.mkdir()
    for f in ("__init__.py", "build.py", "oracle.c"):
        shutil.copy(os.path.join(ROOT, "oracle", f), pkg / f)
    src = (pkg / "__init__.py").read_text()
    assert src.count(old) == 1, "mutation anchor not found"
    (pkg / "__init__.py").write_text(src.replace(old, new, 1))
    env = dict(os.environ, ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-c", _LOAD_MUTANT, str(pkg),
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"pins did not catch mutant {name}:\n{r.stdout[-2000:]}"


def test_unmutated_copy_passes_the_pins(tmp_path):
    # The loader above runs the real acceptance rule cleanly, so a failing
    # mutant run means its planted mistake, not the harness.
    import shutil

    sys.path.insert(0, ROOT)
    from oracle import build as oracle_build

    lib = oracle_build.build()
    pkg = tmp_path / "oracle"
    pkg.mkdir()
    for f in ("__init__.py", "build.py", "oracle.c"):
        shutil.copy(os.path.join(ROOT, "oracle", f), pkg / f)
    env = dict(os.environ, ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-c", _LOAD_MUTANT, str(pkg),
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:]
