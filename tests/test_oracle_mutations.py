"""The oracle's pins reject plausible mistakes.

Each case compiles a copy of the oracle with one planted error (on the CPU,
in a temporary directory) and runs the pin suite against it in a child
process; every mutant must make the pins fail.  This shows that the pins
constrain the oracle rather than restate it.
"""
import inspect
import os
import subprocess
import sys

import numpy as np
import pytest

import hermitian_pins
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "tp_oracle.c")

MUTANTS = {
    "rotation-transposed": ("p[j] = s * (R[0 * dim + j] * kx + R[1 * dim + j] * ky);",
                            "p[j] = s * (R[j * dim + 0] * kx + R[j * dim + 1] * ky);"),
    "phase-sign": ("double ang = -2.0 * M_PI", "double ang = 2.0 * M_PI"),
    "friedel-read-no-conj": ("if (cj)\n                    v = cconj(v);", ""),
    "friedel-reflect-x-only": ("m[1] = -m[1];\n        m[2] = -m[2];", ""),
    "cubic-tap-offset": ("tap[j] = x0 - 1 + j;", "tap[j] = x0 + j;"),
    "keys-a": ("const double a = -0.5;\n    double u = fabs(t);\n    if (u <= 1.0)\n        return (a + 2.0)",
               "const double a = -0.75;\n    double u = fabs(t);\n    if (u <= 1.0)\n        return (a + 2.0)"),
    "adjoint-friedel-no-conj": ("double im = wt * (cj ? -c.im : c.im);", "double im = wt * c.im;"),
    "adjoint-phase-not-conj": ("cplx c = cmul(cconj(phase_of(t, kx, ky, N)), yk);",
                               "cplx c = cmul(phase_of(t, kx, ky, N), yk);"),
    "grad-shift-sign": ("cplx dy = {0.0, -2.0 * M_PI * k[a] / (double)N};",
                        "cplx dy = {0.0, 2.0 * M_PI * k[a] / (double)N};"),
    "linear-derivative": ("dw[0] = -1.0;\n    dw[1] = 1.0;", "dw[0] = 1.0;\n    dw[1] = -1.0;"),
    "keys-derivative": ("return sg * (3.0 * (a + 2.0) * u * u - 2.0 * (a + 3.0) * u);",
                        "return sg * (3.0 * (a + 2.0) * u * u - 1.0 * (a + 3.0) * u);"),
    "radius-exclusive": ("if (kx * kx + ky * ky > r * r)\n                    continue;\n                double p[3];\n                sample_position(R, dim, s, kx, ky, p);\n                cplx S",
                         "if (kx * kx + ky * ky >= r * r)\n                    continue;\n                double p[3];\n                sample_position(R, dim, s, kx, ky, p);\n                cplx S"),
    "weight-ignores-omega": ("W[e] += wt * omega;", "W[e] += wt;"),
    "grad-rot-no-scale": ("gR[i * dim + j] += s * k[i] * d.re;", "gR[i * dim + j] += k[i] * d.re;"),
    # The outermost shell: -M/2 is a stored row, +M/2 and columns beyond M/2 are not, and
    # the Friedel reflection comes before the range test.
    "nyquist-row-accepted": ("if (f < -M / 2 || f > M / 2 - 1)", "if (f < -M / 2 || f > M / 2)"),
    "nyquist-row-rejected": ("if (f < -M / 2 || f > M / 2 - 1)", "if (f <= -M / 2 || f > M / 2 - 1)"),
    "periodic-rows": ("    if (f < -M / 2 || f > M / 2 - 1)\n        return -1;\n    return (f < 0) ? f + M : f;",
                      "    return ((f % M) + M) % M;"),
    "nyquist-column-rejected": ("if (m[0] > s.M / 2)\n        return -1;",
                                "if (m[0] >= s.M / 2)\n        return -1;"),
    "periodic-columns": ("if (m[0] > s.M / 2)\n        return -1;",
                         "if (m[0] > s.M / 2) {\n        m[0] = s.M - m[0];\n        m[1] = -m[1];\n"
                         "        m[2] = -m[2];\n        *conj = !*conj;\n    }"),
    "range-test-before-reflection": ("    *conj = 0;\n    if (m[0] < 0) {",
                                     "    *conj = 0;\n    if (row_of(m[1], s.M) < 0 || (s.dim == 3 && row_of(m[2], s.M) < 0))\n"
                                     "        return -1;\n    if (m[0] < 0) {"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    mutant = tmp_path / "mutant.c"
    mutant.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c99", "-fopenmp", "-fPIC", "-shared", "-o", str(lib),
                    str(mutant), "-lm"], check=True)
    env = dict(os.environ, TP_ORACLE_LIB=str(lib), OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"pins accepted mutant {name}:\n{r.stdout[-2000:]}"


# Planted mistakes in the symmetrised zero-frequency axis (a Python function
# of the oracle): each copy must fail at least one of its pins.
HERMITIAN_MUTANTS = {
    "mirror-without-modulo": ("neg = (-np.arange(M)) % M", "neg = np.arange(M)[::-1]"),
    "no-conj": ("0.5 * (plane + np.conj(mirror))", "0.5 * (plane + mirror)"),
    "no-half": ("0.5 * (plane + np.conj(mirror))", "(plane + np.conj(mirror))"),
    "2d-no-conj": ("0.5 * (col + np.conj(col[:, neg]))", "0.5 * (col + col[:, neg])"),
    "mirror-one-axis": ("mirror = plane[:, neg][:, :, neg]", "mirror = plane[:, neg]"),
    "weight-not-mirrored": ("0.5 * (wp + wp[:, neg][:, :, neg])", "0.5 * (wp + wp)"),
}


@pytest.mark.parametrize("name", sorted(HERMITIAN_MUTANTS))
def test_hermitian_pins_reject_mutant(name):
    old, new = HERMITIAN_MUTANTS[name]
    src = inspect.getsource(oracle.hermitian_x0)
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    ns = {"np": np}
    exec(src.replace(old, new), ns)
    mutant = ns["hermitian_x0"]
    failed = 0
    for check in hermitian_pins.ALL:
        try:
            check(mutant)
        except AssertionError:
            failed += 1
    assert failed > 0, f"pins accepted mutant {name}"
