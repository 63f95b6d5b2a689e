"""The pins catch plausible mistakes: each test builds a copy of the oracle with
one mistake planted (on the CPU, in a temporary directory), points the oracle
module at it, and requires at least one pin to fail."""
import ctypes
import inspect
import os
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

MUTANTS = {
    "euler_instead_of_zoh": ("(An != 0.0) ? expm1(dA) / An : dt", "dt"),
    "abar_sign": ("double abar = exp(dA);", "double abar = exp(-dA);"),
    "no_softplus": ("return x > 0.0 ? x + log1p(exp(-x)) : log1p(exp(x));", "return x;"),
    "bias_dropped": ("in_val(delta, bf16, row * L + t) + bias;", "in_val(delta, bf16, row * L + t);"),
    "readout_before_update": (
        "      h[n] = abar * h[n] + bbar * (double)B_b[n * bc_ld + t] * ut;\n"
        "      acc += (double)C_b[n * bc_ld + t] * h[n];",
        "      acc += (double)C_b[n * bc_ld + t] * h[n];\n"
        "      h[n] = abar * h[n] + bbar * (double)B_b[n * bc_ld + t] * ut;"),
    "D_dropped": ("double yv = acc + Dd * ut;", "double yv = acc;"),
    "gate_sign": ("yv *= zt / (1.0 + exp(-zt));", "yv *= zt / (1.0 + exp(zt));"),
    "B_time_shift": ("bbar * (double)B_b[n * bc_ld + t] * ut",
                     "bbar * (double)B_b[n * bc_ld + (t > 0 ? t - 1 : 0)] * ut"),
    "C_uses_B": ("acc += (double)C_b[n * bc_ld + t] * h[n];", "acc += (double)B_b[n * bc_ld + t] * h[n];"),
    "init_state_ignored": ("h[n] = h0 ? h0[n] : 0.0;", "h[n] = 0.0;"),
}


def _pin_calls():
    calls = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_") or name == "test_rel_err_metric":
            continue
        marks = getattr(fn, "pytestmark", [])
        params = [m for m in marks if m.name == "parametrize"]
        if params:
            argname, values = params[0].args
            for v in values:
                calls.append((name, lambda fn=fn, v=v, a=argname: fn(**{a: v})))
        else:
            calls.append((name, fn))
    return calls


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_pins_catch_planted_mistake(mutant, tmp_path, monkeypatch):
    old, new = MUTANTS[mutant]
    src = open(oracle._SRC).read()
    assert src.count(old) == 1, "mutation site not found: " + mutant
    path = os.path.join(tmp_path, "mutant.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    so = os.path.join(tmp_path, "libmutant.so")
    subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-o", so, path, "-lm"])
    real = oracle._load()
    lib = ctypes.CDLL(so)
    for fname in ("ssm_oracle_scan", "ssm_oracle_step", "ssm_oracle_max_threads"):
        getattr(lib, fname).argtypes = getattr(real, fname).argtypes
        getattr(lib, fname).restype = getattr(real, fname).restype
    monkeypatch.setattr(oracle, "_lib", lib)
    caught = []
    for name, call in _pin_calls():
        try:
            call()
        except AssertionError:
            caught.append(name)
    assert caught, "no pin caught mutant " + mutant
