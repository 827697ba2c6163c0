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
