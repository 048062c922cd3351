"""Do the oracle's pins catch plausible mistakes?  Each case plants one mistake
in a copy of the C oracle (built on the CPU under the test's temp dir), swaps it
in, runs the pin tests of tests/test_oracle_pins.py, and requires at least one
of them to fail."""
import ctypes
import inspect
import os
import shutil
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "bitlinear_oracle.c")

# (name, text in the oracle, planted replacement)
MUTATIONS = [
    ("round half away from zero", "float r = nearbyintf(t);", "float r = roundf(t);"),
    ("weight eps 1e-6", "float sw = 1.0f / fmaxf(mean, 1e-5f);", "float sw = 1.0f / fmaxf(mean, 1e-6f);"),
    ("mean over N only", "float mean = (float)(S / (double)(N * K));", "float mean = (float)(S / (double)N);"),
    ("act scale 128", "float s = 127.0f / fmaxf(amax, 1e-5f);", "float s = 128.0f / fmaxf(amax, 1e-5f);"),
    ("act eps 1e-4", "float s = 127.0f / fmaxf(amax, 1e-5f);", "float s = 127.0f / fmaxf(amax, 1e-4f);"),
    ("code bit position", "*shift = (int)(2 * (i / 4));", "*shift = (int)(2 * (i % 4));"),
    ("chunk order transposed", "return (kb * N + n) * 16 + 4 * w + (i % 4);", "return (n * 1 + kb * N) * 16 + 4 * (3 - w) + (i % 4);"),
    ("code offset", "*q = code - 1;", "*q = code - 2;"),
    ("rmsnorm without /K", "float inv = (float)(1.0 / sqrt(S / (double)K + eps));", "float inv = (float)(1.0 / sqrt(S + eps));"),
    ("rmsnorm without sqrt", "float inv = (float)(1.0 / sqrt(S / (double)K + eps));", "float inv = (float)(1.0 / (S / (double)K + eps));"),
    ("gamma ignored", "h[k] = t * gamma[k];", "h[k] = t;"),
    ("no relu", "float r = fmaxf(xr[k], 0.0f);", "float r = xr[k];"),
    ("relu not squared", "float rr = r * r;", "float rr = r;"),
    ("rescale without sw", "if (y) y[m * N + n] = (double)a / ((double)sx[m] * (double)sw);\n    }\n  }\n  return ORACLE_OK;\n}\n\n/* Same",
     "if (y) y[m * N + n] = (double)a / ((double)sx[m]);\n    }\n  }\n  return ORACLE_OK;\n}\n\n/* Same"),
    ("sticky bit dropped", "if (round_bit && (sticky || (m & 1u))) {", "if (round_bit && (m & 1u)) {"),
    ("subnormal exponent", "if (e == 0) { *mant = frac; *e2 = -149; }", "if (e == 0) { *mant = frac; *e2 = -150; }"),
    ("lost carry", "a->d[j + 1] += c;", "a->d[j + 1] += 0 * c;"),
    ("argmax ties to the last", "if (y[m * N + n] > y[m * N + best]) best = n;",
     "if (y[m * N + n] >= y[m * N + best]) best = n;"),
    ("argmax misses the last column", "for (int64_t n = 1; n < N; ++n)", "for (int64_t n = 1; n < N - 1; ++n)"),
    ("fp64 weight decision", "float t = W[i] * sw;\n    Wq[i] = (int8_t)rne_clamp(t, -1, 1);",
     "double t = (double)W[i] * (double)sw;\n    double rr = nearbyint(t);\n    Wq[i] = (int8_t)(rr < -1 ? -1 : (rr > 1 ? 1 : rr));"),
    ("fp64 activation decision", "float t = h[k] * s;\n      xq[m * K + k] = (int8_t)rne_clamp(t, -128, 127);",
     "double t = (double)h[k] * (double)s;\n      double rr = nearbyint(t);\n"
     "      xq[m * K + k] = (int8_t)(rr < -128 ? -128 : (rr > 127 ? 127 : rr));"),
]


def _pin_cases():
    """Every pin test with its first parameter set (enough to exercise each)."""
    cases = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        marks = getattr(fn, "pytestmark", [])
        params = [m for m in marks if m.name == "parametrize"]
        if not params:
            cases.append((name, fn, {}))
            continue
        argnames, values = params[0].args[0], params[0].args[1]
        argnames = [a.strip() for a in argnames.split(",")] if isinstance(argnames, str) else list(argnames)
        for v in list(values)[:2]:
            v = v if isinstance(v, (tuple, list)) and len(argnames) > 1 else (v,)
            cases.append((name, fn, dict(zip(argnames, v))))
    return cases


@pytest.fixture(scope="module")
def mutant_dir(tmp_path_factory):
    return tmp_path_factory.mktemp("oracle_mutants")


def test_unmutated_oracle_passes_every_pin():
    for name, fn, kw in _pin_cases():
        fn(**kw)


@pytest.mark.parametrize("label,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(mutant_dir, label, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not found once: {label}"
    path = mutant_dir / (label.replace(" ", "_").replace("/", "_") + ".c")
    path.write_text(src.replace(old, new))
    so = str(path) + ".so"
    subprocess.check_call(["gcc", *oracle.CFLAGS, str(path), "-o", so, "-lm"])
    real = oracle._load()
    mutant = ctypes.CDLL(so)
    for attr in ("oracle_exact_abs_sum", "oracle_exact_sq_sum", "oracle_weight_quant", "oracle_packed_bytes",
                 "oracle_pack", "oracle_unpack", "oracle_act_quant", "oracle_forward", "oracle_forward_unpacked"):
        getattr(mutant, attr).argtypes = getattr(real, attr).argtypes
        getattr(mutant, attr).restype = getattr(real, attr).restype
    failures = []
    oracle._lib = mutant
    try:
        for name, fn, kw in _pin_cases():
            try:
                fn(**kw)
            except (Exception, pytest.fail.Exception):  # assertion, oracle error, pytest.raises miss
                failures.append(name)
    finally:
        oracle._lib = real
    assert failures, f"no pin caught the planted mistake '{label}'"
