"""Plant plausible mistakes in a copy of the oracle (on the CPU) and check that the pins catch each one.

Every mutant is compiled from a textually edited copy of oracle/oracle.c into a temporary directory and
swapped in for the real oracle library while the pin checks run; at least one pin must fail per mutant.
"""
import ctypes
import importlib.util
import os
import subprocess
import sys

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(os.path.dirname(HERE), "oracle", "oracle.c")

MUTANTS = {
    "drop_one_minus_beta1": ("(1.0 - b1) * g", "g"),
    "update_sign": ("(double)*th - lr * mh", "(double)*th + lr * mh"),
    "bias_power_off_by_one": ("pow(b1, (double)w->t_new)", "pow(b1, (double)w->t_new + 1.0)"),
    "beta_transposed": ("b2 * (double)*vv", "b1 * (double)*vv"),
    "eps_inside_sqrt": ("lr * mh / (sqrt(vh) + eps)", "lr * mh / sqrt(vh + eps)"),
    "average_over_n_times_a": ("(double)p->n * (double)p->loss_scale", "(double)(p->n * p->a) * (double)p->loss_scale"),
    "no_skip": ("      w->found = 1;\n", "\n"),
    "replica_from_wrong_rank": ("p->replicas[r][i] = oracle_f32_to_bf16(p->master[r][i])",
                                "p->replicas[r][i] = oracle_f32_to_bf16(p->master[0][i] * 0.5f)"),
    "replica_from_moment": ("uint16_t b = oracle_f32_to_bf16(p->master[owner][j]);",
                            "uint16_t b = oracle_f32_to_bf16(p->m[owner][j]);"),
    "local_offset_dropped": ("int64_t j = l0 + (i - g0);", "int64_t j = i - g0;"),
    "bf16_truncates": ("nearbyint(ldexp(x, -q))", "trunc(ldexp(x, -q))"),
    "second_moment_linear": ("(1.0 - b2) * g * g", "(1.0 - b2) * g"),
    "last_micro_step_dropped": ("for (int q = 0; q < na; ++q)", "for (int q = 0; q < na - 1; ++q)"),
}


def _load_pins():
    spec = importlib.util.spec_from_file_location("_pins", os.path.join(HERE, "test_oracle_pins.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _checks(P):
    return [
        lambda: P.test_sum_matches_fsum_library(),
        lambda: P.test_global_batch_example_256_samples(),
        lambda: P.test_adam_matches_torch_optim_adam(7),
        lambda: P.test_adam_cold_start_closed_form(),
        lambda: P.test_adam_constant_gradient_closed_form(),
        lambda: P.test_skip_on_nonfinite_leaves_state("middle", 0x7F80),
        lambda: P.test_replicas_identical_and_equal_bf16_of_master(),
        lambda: P.test_sharded_equals_unsharded("random"),
        lambda: P.test_bf16_rounding_vs_torch_library(),
    ]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    pytest.importorskip("torch")
    src = open(SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) >= 1, "mutation site vanished: " + name
    mutated = src.replace(old, new, 1)
    c = tmp_path / "oracle_mut.c"
    c.write_text(mutated)
    so = tmp_path / "liboracle_mut.so"
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-D_GNU_SOURCE", "-ffp-contract=off", "-fPIC", "-shared",
                           "-o", str(so), str(c), "-lm", "-lpthread"])
    child = subprocess.run([sys.executable, "-c", _CHILD, str(so)], cwd=os.path.dirname(HERE),
                           capture_output=True, text=True, timeout=600)
    assert child.returncode == 0, child.stdout + child.stderr
    caught = [int(x) for x in child.stdout.split() if x.isdigit()]
    assert caught, "no pin caught the planted mistake " + name


_CHILD = r"""
import ctypes, sys, importlib.util, os
sys.path.insert(0, os.getcwd())
import oracle
L = ctypes.CDLL(sys.argv[1])
for fn in ("oracle_step", "oracle_reduce"):
    getattr(L, fn).argtypes = [ctypes.POINTER(oracle.Problem)]
    getattr(L, fn).restype = ctypes.c_int
L.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
L.oracle_f32_to_bf16.restype = ctypes.c_uint16
L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
L.oracle_bf16_to_double.restype = ctypes.c_double
oracle._LIB = L
spec = importlib.util.spec_from_file_location("_pins", os.path.join("tests", "test_oracle_pins.py"))
P = importlib.util.module_from_spec(spec)
spec.loader.exec_module(P)
sys.path.insert(0, "tests")
import test_oracle_mutations as T
for k, chk in enumerate(T._checks(P)):
    try:
        chk()
    except (AssertionError, RuntimeError, FloatingPointError):
        print(k)
"""
