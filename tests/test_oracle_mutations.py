"""Mutation checks of the oracle's pins (CPU): each test plants one plausible mistake in a
copy of the oracle -- the C source recompiled into a scratch library, or the numpy attention
module re-executed from edited source -- and requires at least one pin of
tests/test_oracle.py to fail against it.  The product library is not involved."""
import os
import subprocess
import sys
import types

import pytest

import oracle
import oracle.attention as attention

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
import test_oracle  # noqa: E402  (the pins)

ORACLE_C = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")


def _pins(prefixes):
    """The pins of tests/test_oracle.py that take no arguments (the parametrized ones are
    covered by their unparametrized siblings here)."""
    import inspect
    return [getattr(test_oracle, n) for n in sorted(dir(test_oracle))
            if n.startswith("test_") and any(n.startswith(p) for p in prefixes)
            and not inspect.signature(getattr(test_oracle, n)).parameters]


def _failures(pins):
    failed = []
    for fn in pins:
        try:
            fn()
        except Exception:          # a failed assertion, or the mutant refusing its input
            failed.append(fn.__name__)
    return failed


def _with_c_mutant(tmp_path, old, new):
    """Compile oracle.c with `old` replaced by `new` into a scratch library and swap it in."""
    with open(ORACLE_C) as fh:
        src = fh.read()
    assert src.count(old) == 1, old
    path = tmp_path / "oracle_mut.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / "liboracle_mut.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
                           "-fPIC", "-shared", str(path), "-o", str(lib), "-lm"])
    return str(path), str(lib)


C_MUTANTS = {
    "scale sign dropped": ("acc += oracle_half_to_double(scales[n * G + g]) * inner;",
                           "acc += fabs(oracle_half_to_double(scales[n * G + g])) * inner;"),
    "wrong group of scales": ("acc += oracle_half_to_double(scales[n * G + g]) * inner;",
                              "acc += oracle_half_to_double(scales[n * G + (G - 1 - g)]) * inner;"),
    "reciprocal instead of divide": ("float r = nearbyintf(a / sm);",
                                     "float r = nearbyintf(a * (1.0f / sm));"),
    "halves rounded away from zero": ("float r = nearbyintf(a / sm);", "float r = roundf(a / sm);"),
    "W4A8 scale sign dropped": ("acc += oracle_half_to_double(scales[n * G + g]) * (double)inner;",
                                "acc += fabs(oracle_half_to_double(scales[n * G + g])) * (double)inner;"),
    "gather scale sign dropped": ("out[t * D + k] = oracle_double_to_half((double)codes[v * D + k] * s);",
                                  "out[t * D + k] = oracle_double_to_half((double)codes[v * D + k] * fabs(s));"),
    "top-k ties to the larger index": ("return (i < j) ? -1 : (i > j) ? 1 : 0;",
                                      "return (i < j) ? 1 : (i > j) ? -1 : 0;"),
}


@pytest.mark.parametrize("name", sorted(C_MUTANTS))
def test_c_oracle_mutant_is_caught(tmp_path, name):
    old, new = C_MUTANTS[name]
    src, lib = _with_c_mutant(tmp_path, old, new)
    saved = (oracle._SRC, oracle._LIB, oracle._lib)
    try:
        oracle._SRC, oracle._LIB, oracle._lib = src, lib, None
        failed = _failures(_pins(["test_"]))
    finally:
        oracle._SRC, oracle._LIB, oracle._lib = saved
    assert failed, f"no pin catches: {name}"


ATTN_MUTANTS = {
    "no 1/sqrt(d)": ("inv_sqrt_d = 1.0 / np.sqrt(np.float64(d))", "inv_sqrt_d = 1.0"),
    "no causal mask": ("visible = np.arange(S)[None, :] <= pos", "visible = np.ones((T, S), bool)"),
    "heads mapped modulo": ("g = h // group", "g = h % Hkv"),
    "no smoothing": ("kq, ks = quant_rows_f32(smooth_k(k))", "kq, ks = quant_rows_f32(k.astype(np.float32))"),
    "reciprocal in the row quantizer": ("q = np.rint((x / safe[..., None]).astype(np.float32))",
                                        "q = np.rint((x * (np.float32(1.0) / safe)[..., None]).astype(np.float32))"),
    "mean not divided by S": ("mean = (total / np.float64(S)).astype(np.float32)",
                              "mean = total.astype(np.float32)"),
}


@pytest.mark.parametrize("name", sorted(ATTN_MUTANTS))
def test_attention_oracle_mutant_is_caught(name):
    old, new = ATTN_MUTANTS[name]
    with open(attention.__file__) as fh:
        src = fh.read()
    assert src.count(old) == 1, old
    mod = types.ModuleType("attention_mutant")
    exec(compile(src.replace(old, new), "attention_mutant", "exec"), mod.__dict__)
    saved = (oracle.attn_int8qk, oracle.quant_rows_f32, oracle.smooth_k)
    try:
        oracle.attn_int8qk, oracle.quant_rows_f32, oracle.smooth_k = \
            mod.attn_int8qk, mod.quant_rows_f32, mod.smooth_k
        failed = _failures(_pins(["test_attn_"]))
    finally:
        oracle.attn_int8qk, oracle.quant_rows_f32, oracle.smooth_k = saved
    assert failed, f"no pin catches: {name}"


def test_unmutated_oracle_passes_every_pin():
    assert _failures(_pins(["test_"])) == []
