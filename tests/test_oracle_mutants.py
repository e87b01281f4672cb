"""The pins are strong enough: every plausible slip planted in the oracle fails one.

Each case below copies the float64 oracle's C source, plants one mistake of
the kind that is easy to make when writing the Mamba-3 recurrence (a sign, a
dropped factor, the wrong frame for the delayed write, the wrong index), builds
it, swaps it in for the real oracle and runs the pins of test_oracle_pins.py.
The real oracle passes all of them; each mutant must fail at least one.
"""
import os
import shutil
import subprocess
import tempfile

import pytest

import oracle
import test_oracle_pins as pins
import test_oracle_prep_pins as prep_pins

SRC = os.path.join(os.path.dirname(os.path.abspath(oracle.__file__)), "m3_oracle.c")

# name -> list of (exact source text, replacement)
MUTANTS = {
    "rotation turns the other way": [
        ("h0[p] = cs * u0 - sn * u1 + gamma * v0[p];", "h0[p] = cs * u0 + sn * u1 + gamma * v0[p];"),
        ("h1[p] = sn * u0 + cs * u1 + gamma * v1[p];", "h1[p] = -sn * u0 + cs * u1 + gamma * v1[p];"),
    ],
    "beta without the decay alpha": [
        ("const double beta = (1.0 - l) * d * alpha;", "const double beta = (1.0 - l) * d;"),
    ],
    "gamma weighted by 1 - lambda": [
        ("const double gamma = l * d;", "const double gamma = (1.0 - l) * d;"),
    ],
    "delayed write not rotated": [
        ("const double u0 = alpha * h0[p] + beta * vp0[p];", "const double u0 = alpha * h0[p];"),
        ("const double u1 = alpha * h1[p] + beta * vp1[p];", "const double u1 = alpha * h1[p];"),
        ("h0[p] = cs * u0 - sn * u1 + gamma * v0[p];", "h0[p] = cs * u0 - sn * u1 + beta * vp0[p] + gamma * v0[p];"),
        ("h1[p] = sn * u0 + cs * u1 + gamma * v1[p];", "h1[p] = sn * u0 + cs * u1 + beta * vp1[p] + gamma * v1[p];"),
    ],
    "angle without the step size": [
        ("const double phi = d * wt[j];", "const double phi = wt[j];"),
    ],
    "readout mixes the ranks": [
        ("s += h[n * P + p] * ct[r * N + n];", "s += h[n * P + p] * ct[n];"),
    ],
    "delayed write taken from the current token": [
        ("sp += bprev[r * N + n] * xprev[r * P + p];", "sp += bt[r * N + n] * xt[r * P + p];"),
    ],
    "pairs split in halves instead of interleaved": [
        ("double* h0 = h + (2 * j) * P;", "double* h0 = h + j * P;"),
        ("double* h1 = h + (2 * j + 1) * P;", "double* h1 = h + (j + N / 2) * P;"),
        ("const double* vp0 = vp + (2 * j) * P;", "const double* vp0 = vp + j * P;"),
        ("const double* vp1 = vp + (2 * j + 1) * P;", "const double* vp1 = vp + (j + N / 2) * P;"),
        ("const double* v0 = v + (2 * j) * P;", "const double* v0 = v + j * P;"),
        ("const double* v1 = v + (2 * j + 1) * P;", "const double* v1 = v + (j + N / 2) * P;"),
    ],
    "decay exponent sign flipped": [
        ("const double alpha = exp(d * a);", "const double alpha = exp(-d * a);"),
    ],
    "per-token decay generator taken from the first token": [
        ("const double a = a_seq[t * a_stride];", "const double a = a_seq[0];"),
    ],
    "per-token decay generator taken from the previous token": [
        ("const double a = a_seq[t * a_stride];", "const double a = a_seq[(t > 0 ? t - 1 : 0) * a_stride];"),
    ],
}

# Pins that run in well under a second each (name, callable).
PIN_SUITE = [
    ("mamba2 reduction", pins.test_mamba2_reduction),
    ("matrix form T=17", lambda: pins.test_matrix_form_equals_scan(17, 1)),
    ("matrix form MIMO", lambda: pins.test_matrix_form_equals_scan(33, 3)),
    ("two-band closed form", pins.test_two_band_constant_coefficients_match_closed_form),
    ("complex/rotating frame R=1", lambda: pins.test_complex_and_rotating_frame_equal_scan(1)),
    ("complex/rotating frame R=2", lambda: pins.test_complex_and_rotating_frame_equal_scan(2)),
    ("closed form two steps", pins.test_closed_form_two_steps),
    ("closed form three steps", pins.test_closed_form_three_steps_delayed_term_rotation),
    ("parity construction", pins.test_parity_construction_golden),
    ("norm under pure rotation", pins.test_rotation_preserves_norm_without_decay),
    ("single-token MIMO R=3", lambda: pins.test_single_token_mimo_write_and_readout(3)),
    ("lambda = 1 drops the delayed write", pins.test_lambda_one_ignores_delayed_write),
    ("chunked = sequential", lambda: pins.test_chunked_equals_sequential_T256(64)),
    ("per-token A: Mamba-2 reduction", prep_pins.test_mamba2_reduction_per_token_A),
    ("per-token A: chunked = sequential", lambda: prep_pins.test_chunked_per_token_A(16)),
    ("per-token A: two steps closed form", prep_pins.test_closed_form_two_steps_per_token_A),
]


def _run_suite():
    failed = []
    for name, fn in PIN_SUITE:
        try:
            fn()
        except (AssertionError, ValueError):
            failed.append(name)
    return failed


def _build(text: str, d: str) -> str:
    src = os.path.join(d, "mutant.c")
    lib = os.path.join(d, "libmutant.so")
    with open(src, "w") as f:
        f.write(text)
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", lib, src, "-lm"])
    return lib


def test_real_oracle_passes_the_suite():
    assert _run_suite() == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_fails_a_pin(name, monkeypatch):
    text = open(SRC).read()
    for old, new in MUTANTS[name]:
        assert old in text, f"mutation site not found: {old}"
        text = text.replace(old, new, 1)
    d = tempfile.mkdtemp(prefix="m3o_mutant_")
    try:
        path = _build(text, d)
        real = oracle._load()
        import ctypes
        lib = ctypes.CDLL(path)
        lib.m3o_scan.argtypes = real.m3o_scan.argtypes
        lib.m3o_scan.restype = real.m3o_scan.restype
        lib.m3o_scan_tok.argtypes = real.m3o_scan_tok.argtypes
        lib.m3o_scan_tok.restype = real.m3o_scan_tok.restype
        lib.m3o_num_threads.argtypes = []
        lib.m3o_num_threads.restype = ctypes.c_int
        monkeypatch.setattr(oracle, "_lib", lib)
        failed = _run_suite()
    finally:
        shutil.rmtree(d, ignore_errors=True)
    assert failed, f"mutant '{name}' passed every pin"
