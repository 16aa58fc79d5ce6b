"""Plants plausible mistakes in a COPY of the oracle's C source and checks that a pin catches each.

This is the evidence that the pins in oracle_pins.py are strong enough: a
dropped term, a wrong sign, a swapped index, a transposed operand, a float
accumulator or a read of C when beta == 0 each fail at least one pin.  Every
mutant is compiled with gcc into a temporary directory and exercised in a
child process, so a mutant that reads out of bounds cannot take the test
runner down (a crash counts as caught).  Nothing here touches a GPU.
"""
import json
import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTATIONS = [
    ("drop the last k term", "for (int64_t k = 0; k < K; ++k)", "for (int64_t k = 0; k < K - 1; ++k)"),
    ("skip the first k term", "for (int64_t k = 0; k < K; ++k)", "for (int64_t k = 1; k < K; ++k)"),
    ("transposed B index", "oracle_op_elem(B, ldb, tb, k, j)", "oracle_op_elem(B, ldb, tb, j, k)"),
    ("transposed A index", "oracle_op_elem(A, lda, ta, i, k)", "oracle_op_elem(A, lda, ta, k, i)"),
    ("op flag inverted", "return trans ? (double)X[c * ld + r] : (double)X[r * ld + c];",
     "return trans ? (double)X[r * ld + c] : (double)X[c * ld + r];"),
    ("wrong sign of beta", "const double bc = (double)beta * c_old;", "const double bc = -(double)beta * c_old;"),
    ("alpha applied to beta*C", "const double r = (double)alpha * sum + bc;", "const double r = (double)alpha * (sum + bc);"),
    ("alpha dropped", "const double r = (double)alpha * sum + bc;", "const double r = sum + bc;"),
    ("C read when beta == 0", "const int read_c = (beta != 0.0f);", "const int read_c = 1;"),
    ("A, B read when alpha == 0", "const int read_ab = (alpha != 0.0f) && (K > 0);", "const int read_ab = (K > 0);"),
    ("float accumulator", "double sum = 0.0;", "float sum = 0.0f;"),
    ("signed magnitude in S", "sum_abs += fabs(p);", "sum_abs += p;"),
    ("ldc ignored", "C[i * ldc + j] = (float)r;", "C[i * N + j] = (float)r;"),
    ("column index modulo M", "const int64_t j = e % N;", "const int64_t j = e % (M > 0 ? M : 1);"),
    ("'C' not accepted as transpose", "t == 'C' || t == 'c'", "t == 'C' && t == 'c'"),
    ("batch: last product dropped", "for (int64_t b = 0; b < batch; ++b)", "for (int64_t b = 0; b < batch - 1; ++b)"),
    ("batch: A advanced by B's stride", "A ? A + b * strideA : A", "A ? A + b * strideB : A"),
    ("batch: C taken as packed", "C ? C + b * strideC : C", "C ? C + b * M * ldc : C"),
    ("batch: S not advanced", "S ? S + b * strideS : S", "S"),
    ("batch: negative stride accepted", "strideA < 0 || strideB", "strideB"),
    ("tf32: truncation instead of rounding", "floor(a / q + 0.5) * q", "floor(a / q) * q"),
    ("tf32: ties to even magnitude down", "floor(a / q + 0.5) * q", "ceil(a / q - 0.5) * q"),
    ("tf32: 11 fraction bits", "int qexp = (e - 1) - 10;", "int qexp = (e - 1) - 11;"),
    ("tf32: no subnormal quantum", "if (qexp < -136) qexp = -136;", "if (qexp < -149) qexp = -149;"),
    ("tf32: sign dropped", "const double y = x < 0.0f ? -r : r;", "const double y = r;"),
    ("bf16: ties away from zero", "(frac > 0.5 || (frac == 0.5 && fmod(m, 2.0) != 0.0))", "(frac >= 0.5)"),
    ("bf16: truncation", "if (frac > 0.5 || (frac == 0.5 && fmod(m, 2.0) != 0.0)) m += 1.0;", ""),
    ("bf16: 8 fraction bits", "int qexp = (e - 1) - 7;", "int qexp = (e - 1) - 8;"),
    ("bf16: no subnormal quantum", "if (qexp < -133) qexp = -133;", "if (qexp < -149) qexp = -149;"),
    ("bf16: ties to odd", "fmod(m, 2.0) != 0.0", "fmod(m, 2.0) == 0.0"),
    ("bf16: sign dropped", "const double y = (x < 0.0f) ? -r : r;", "const double y = r;"),
]

_CHILD = r"""
import json, sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import oracle, oracle_pins as P
lib = oracle.load_library({lib!r})
failed = []
pins = [p for p in P.ALL_PINS if p is not P.pin_integer_pattern]
for pin in pins:
    try:
        pin(lib)
    except Exception as e:   # AssertionError or an oracle error both count as caught
        failed.append(pin.__name__)
try:
    P.pin_integer_pattern(lib, M=100, N=130, K=70)
except Exception:
    failed.append("pin_integer_pattern")
print(json.dumps(failed))
"""


@pytest.mark.parametrize("desc,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_mutant_is_caught(tmp_path, desc, old, new):
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, f"mutation anchor not found once: {old!r}"
    mutant = tmp_path / "mutant.c"
    mutant.write_text(src.replace(old, new))
    lib = oracle.compile_library(str(mutant), str(tmp_path / "libmutant.so"))
    code = _CHILD.format(root=ROOT, tests=os.path.join(ROOT, "tests"), lib=lib)
    proc = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300,
                          env={**os.environ, "OMP_NUM_THREADS": "2"})
    if proc.returncode != 0:
        return   # the mutant crashed the child (e.g. read out of bounds): caught
    failed = json.loads(proc.stdout.strip().splitlines()[-1])
    assert failed, f"no pin caught the mutation '{desc}'"
