"""Plant plausible mistakes in copies of the oracle and check that the pins catch each.

Every mutant is a text edit of ``oracle/sgemm_oracle.c`` compiled into a
temporary library on the CPU; the pin functions of ``test_oracle_pins`` are then
run against it.  A mutant that passes every pin would mean the pins cannot tell
that mistake from the definition.
"""
import importlib.util
import multiprocessing as mp
import os
import shutil
import sys

import pytest

import test_oracle_pins as pins

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTANTS = {
    "wrong_sign_in_row_sum": ("acc[j] += a * (double)brow[j];", "acc[j] -= a * (double)brow[j];"),
    "transposed_A_index": ("return transA ? A[k * lda + i] : A[i * lda + k];",
                           "return transA ? A[i * lda + k] : A[k * lda + i];"),
    "transposed_B_index": ("return transB ? B[j * ldb + k] : B[k * ldb + j];",
                           "return transB ? B[k * ldb + j] : B[j * ldb + k];"),
    "dropped_beta_term": ("ref[(int64_t)i * N + j] = (use_ab ? alpha * acc[j] : 0.0) + bc;",
                          "ref[(int64_t)i * N + j] = (use_ab ? alpha * acc[j] : 0.0);"),
    "alpha_not_applied": ("ref[(int64_t)i * N + j] = (use_ab ? alpha * acc[j] : 0.0) + bc;",
                          "ref[(int64_t)i * N + j] = (use_ab ? acc[j] : 0.0) + bc;"),
    "last_k_dropped": ("for (int k = 0; k < K; ++k) {\n                    const double a = (double)opA",
                       "for (int k = 0; k < K - 1; ++k) {\n                    const double a = (double)opA"),
    "magnitude_missing_b": ("mag[j] += aa * fabs((double)brow[j]);", "mag[j] += aa;"),
    "c_read_with_wrong_ld": ("const double c = (beta != 0.0) ? (double)C[(int64_t)i * ldc + j] : 0.0;",
                             "const double c = (beta != 0.0) ? (double)C[(int64_t)i * N + j] : 0.0;"),
    "entries_wrong_operand": ("s += a * b;", "s += a * a;"),
    "c_read_when_beta_zero": ("const double c = (beta != 0.0) ? (double)C[(int64_t)i * ldc + j] : 0.0;",
                              "const double c = (double)C[(int64_t)i * ldc + j];"),
}

# every pin, with one parameter set for the parametrised ones
PIN_CALLS = [
    ("hand", lambda m: pins.test_hand_worked_example(m)),
    ("fma", lambda m: pins.test_fma_count_is_mnk(m, 3, 5, 7)),
    ("idl", lambda m: pins.test_identity_left(m, 0.75, -1.25)),
    ("idr", lambda m: pins.test_identity_right(m, 0.75, -1.25)),
    ("ones", lambda m: pins.test_all_ones(m, 100)),
    ("a0", lambda m: pins.test_alpha_zero_gives_beta_c(m)),
    ("b0", lambda m: pins.test_beta_zero_does_not_read_c(m)),
    ("int", lambda m: pins.test_small_integer_exactness(m, 0)),
    ("frac", lambda m: pins.test_fraction_brute_force(m, True, True, 0)),
    ("frac_nn", lambda m: pins.test_fraction_brute_force(m, False, False, 1)),
    ("tr", lambda m: pins.test_transpose_identity(m)),
    ("lin", lambda m: pins.test_linearity_in_alpha(m)),
    ("pad", lambda m: pins.test_padded_leading_dims(m)),
    ("ent", lambda m: pins.test_entries_match_full(m, False, False)),
]


def _load_mutant(tmp_path, name, old, new):
    pkg = tmp_path / f"oracle_{name}"
    shutil.copytree(os.path.join(ROOT, "oracle"), pkg,
                    ignore=shutil.ignore_patterns("*.so", "__pycache__", "*.tmp*"))
    src = pkg / "sgemm_oracle.c"
    text = src.read_text()
    assert text.count(old) >= 1, f"mutation site for {name} not found"
    src.write_text(text.replace(old, new, 1))
    spec = importlib.util.spec_from_file_location(f"oracle_{name}", pkg / "__init__.py",
                                                  submodule_search_locations=[str(pkg)])
    mod = importlib.util.module_from_spec(spec)
    sys.modules[spec.name] = mod
    spec.loader.exec_module(mod)
    mod.build(force=True)
    return mod


def _run_pins(tmp, name, old, new, queue):
    import pathlib

    sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, ROOT)
    mod = _load_mutant(pathlib.Path(tmp), name, old, new)
    caught = []
    for pin, call in PIN_CALLS:
        try:
            call(mod)
        except Exception:
            caught.append(pin)
        queue.put(("progress", pin))
    queue.put(("caught", caught))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    """Each mutant runs in a child process: a mutant that crashes (for example by
    reading an operand that is not there) counts as caught."""
    old, new = MUTANTS[name]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    p = ctx.Process(target=_run_pins, args=(str(tmp_path), name, old, new, q))
    p.start()
    p.join(300)
    if p.is_alive():
        p.kill()
    result = None
    while not q.empty():
        kind, val = q.get()
        if kind == "caught":
            result = val
    crashed = p.exitcode != 0
    assert crashed or result, f"mutant {name} passed every pin"


def test_unmutated_copy_passes_every_pin(tmp_path):
    mod = _load_mutant(tmp_path, "none", "#include <math.h>", "#include <math.h>")
    for _, call in PIN_CALLS:
        call(mod)
