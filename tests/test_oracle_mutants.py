"""The pins catch plausible mistakes: each test builds a copy of the oracle with
one mistake planted (on the CPU, in a temporary directory), points the oracle
module at it, and requires at least one pin to fail."""
import ctypes
import inspect
import os
import subprocess

import pytest

import oracle
import test_oracle_bwd_pins as bwd_pins
import test_oracle_conv_pins as conv_pins
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
    "euler_flag_ignored": ("double bbar = euler ? dt : ((An != 0.0)", "double bbar = 0 ? dt : ((An != 0.0)"),
}


# mistakes in the backward (derivative) part of the oracle
BWD_MUTANTS = {
    "bwd_no_state_carry": ("      lam[n] *= abar;\n", ""),
    "bwd_dbbar_dA_sign": ("(dt * abar - bbar) / An", "(bbar - dt * abar) / An"),
    "bwd_zero_A_limit": ("0.5 * dt * dt", "dt * dt"),
    "bwd_softplus_chain_dropped": ("double dx = softplus_on ? ddt * sigmoid(xs[t]) : ddt;",
                                   "double dx = ddt;"),
    "bwd_dC_uses_previous_state": ("dC_b[n * L + t] += ds * hs[t * N + n];",
                                   "dC_b[n * L + t] += ds * prev;"),
    "bwd_dB_without_bbar": ("dB_b[n * L + t] += lam[n] * bbar * ut;",
                            "dB_b[n * L + t] += lam[n] * ut;"),
    "bwd_ddelta_without_A": ("ddt += lam[n] * (prev * An * abar + Bn * ut * dbbar_ddt);",
                             "ddt += lam[n] * (prev * abar + Bn * ut * dbbar_ddt);"),
    "bwd_euler_slope": ("double dbbar_ddt = euler ? 1.0 : abar;", "double dbbar_ddt = abar;"),
    "bwd_euler_dA": ("double dbbar_dA = euler ? 0.0 :", "double dbbar_dA = euler ? 0.5 * dt * dt :"),
    "bwd_dz_without_silu_slope": ("sg * (1.0 + zt * (1.0 - sg))", "sg"),
    "bwd_dfinal_ignored": ("lam[n] = dfinal ? dfinal[n] : 0.0;", "lam[n] = 0.0;"),
    "bwd_du_without_D": ("double du = ds * Dd;", "double du = 0.0;"),
    "bwd_gate_missing_in_ds": ("double ds = dy_row[t] * g;", "double ds = dy_row[t];"),
}


# mistakes in the front end (causal conv1d + SiLU)
CONV_MUTANTS = {
    "conv_anticausal": ("const int64_t s = t - (K - 1) + k;  /* input time */",
                        "const int64_t s = t + k;  /* input time */"),
    "conv_kernel_flipped": ("v += (double)w[d * K + k] * xv;", "v += (double)w[d * K + (K - 1 - k)] * xv;"),
    "conv_bias_dropped": ("double v = bias ? (double)bias[d] : 0.0;", "double v = 0.0;"),
    "conv_silu_sign": ("v / (1.0 + exp(-v))", "v / (1.0 + exp(v))"),
    "conv_state_ignored": ("else xv = state_in ? state_in[i * (K - 1) + (K - 1 + s)] : 0.0;\n        v +=",
                           "else xv = 0.0;\n        v +="),
    "conv_state_out_shift": ("const int64_t s = L - (K - 1) + j;", "const int64_t s = L - K + j;"),
}


def _pin_calls(module=pins):
    calls = []
    for name, fn in inspect.getmembers(module, inspect.isfunction):
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


def _run_mutant(old, new, tmp_path, monkeypatch, module, part):
    """Plant `old` -> `new` in one part of the oracle source: "fwd" (the scan and
    the decode step), "bwd" (the derivatives, from the sigmoid helper on) or
    "conv" (the front end)."""
    src = open(oracle._SRC).read()
    c1 = src.index("static double sigmoid(")
    c2 = src.index("/*\n * Front end of the scan")
    bounds = {"fwd": (0, c1), "bwd": (c1, c2), "conv": (c2, len(src))}[part]
    region = src[bounds[0]:bounds[1]]
    assert region.count(old) == 1, "mutation site not found: " + old
    path = os.path.join(tmp_path, "mutant.c")
    with open(path, "w") as f:
        f.write(src[:bounds[0]] + region.replace(old, new) + src[bounds[1]:])
    so = os.path.join(tmp_path, "libmutant.so")
    subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-o", so, path, "-lm"])
    real = oracle._load()
    lib = ctypes.CDLL(so)
    for fname in ("ssm_oracle_scan", "ssm_oracle_step", "ssm_oracle_scan_bwd",
                  "ssm_oracle_conv1d", "ssm_oracle_max_threads"):
        getattr(lib, fname).argtypes = getattr(real, fname).argtypes
        getattr(lib, fname).restype = getattr(real, fname).restype
    monkeypatch.setattr(oracle, "_lib", lib)
    caught = []
    for name, call in _pin_calls(module):
        try:
            call()
        except AssertionError:
            caught.append(name)
    return caught


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_pins_catch_planted_mistake(mutant, tmp_path, monkeypatch):
    old, new = MUTANTS[mutant]
    assert _run_mutant(old, new, tmp_path, monkeypatch, pins, "fwd"), "no pin caught mutant " + mutant


@pytest.mark.parametrize("mutant", sorted(BWD_MUTANTS))
def test_backward_pins_catch_planted_mistake(mutant, tmp_path, monkeypatch):
    """The backward pins (finite differences of the forward, the transposed
    convolution, the transition product) catch each planted derivative mistake;
    the forward part of the oracle is left intact, so the finite differences
    still see the true forward."""
    old, new = BWD_MUTANTS[mutant]
    assert _run_mutant(old, new, tmp_path, monkeypatch, bwd_pins, "bwd"), "no pin caught " + mutant


@pytest.mark.parametrize("mutant", sorted(CONV_MUTANTS))
def test_conv_pins_catch_planted_mistake(mutant, tmp_path, monkeypatch):
    old, new = CONV_MUTANTS[mutant]
    assert _run_mutant(old, new, tmp_path, monkeypatch, conv_pins, "conv"), "no pin caught " + mutant


# mistakes in the front end's backward (oracle.conv1d_bwd, numpy): planted in a
# copy of the function's source, which then stands in for the real one
CONV_BWD_MUTANTS = {
    "convbwd_taps_flipped": ("dxp[:, :, k:k + L] += w[None, :, k, None] * g",
                             "dxp[:, :, k:k + L] += w[None, :, K - 1 - k, None] * g"),
    "convbwd_dw_unshifted": ("dw[:, k] = np.sum(g * xp[:, :, k:k + L], axis=(0, 2))",
                             "dw[:, k] = np.sum(g * xp[:, :, K - 1:K - 1 + L], axis=(0, 2))"),
    "convbwd_silu_slope": ("g = g * sg * (1.0 + p * (1.0 - sg))", "g = g * sg"),
    "convbwd_bias_not_in_p": ("p += np.asarray(bias, dtype=np.float64)[None, :, None]",
                              "p += 0.0 * np.asarray(bias, dtype=np.float64)[None, :, None]"),
    "convbwd_state_grad_dropped": ("dstate=dxp[:, :, :K - 1])", "dstate=0.0 * dxp[:, :, :K - 1])"),
    "convbwd_dbias_sign": ("dbias=np.sum(g, axis=(0, 2))", "dbias=-np.sum(g, axis=(0, 2))"),
}


@pytest.mark.parametrize("mutant", sorted(CONV_BWD_MUTANTS))
def test_conv_backward_pins_catch_planted_mistake(mutant, monkeypatch):
    old, new = CONV_BWD_MUTANTS[mutant]
    src = inspect.getsource(oracle.conv1d_bwd)
    assert src.count(old) == 1, "mutation site not found: " + old
    ns = dict(vars(oracle))
    exec(compile(src.replace(old, new), "conv1d_bwd_mutant", "exec"), ns)
    monkeypatch.setattr(oracle, "conv1d_bwd", ns["conv1d_bwd"])
    caught = []
    for name, call in _pin_calls(conv_pins):
        if not name.startswith("test_backward"):
            continue
        try:
            call()
        except AssertionError:
            caught.append(name)
    assert caught, "no pin caught " + mutant


# mistakes in the SSD backward's summing of the tied parameters (oracle.ssd_bwd)
SSD_BWD_MUTANTS = {
    "ssdbwd_ddt_one_channel": ("r[\"ddelta\"].reshape(batch, H, P, L).sum(axis=2)",
                               "r[\"ddelta\"].reshape(batch, H, P, L)[:, :, 0]"),
    "ssdbwd_head_sum_skips_batch": ("a.reshape(batch, H, P, -1).sum(axis=(0, 2, 3))",
                                    "a.reshape(batch, H, P, -1)[0].sum(axis=(1, 2))"),
    "ssdbwd_groups_swapped": ("unit_b = (bb * G + hh // hpg).ravel()",
                              "unit_b = (bb * G + (G - 1 - hh // hpg)).ravel()"),
    "ssdbwd_dx_time_reversed": ("back = lambda a: np.transpose(a.reshape(batch, H, P, L), (0, 3, 1, 2))",
                                "back = lambda a: np.transpose(a.reshape(batch, H, P, L)[..., ::-1], (0, 3, 1, 2))"),
}


@pytest.mark.parametrize("mutant", sorted(SSD_BWD_MUTANTS))
def test_ssd_backward_pins_catch_planted_mistake(mutant, monkeypatch):
    import test_oracle_ssd_pins as ssd_pins
    old, new = SSD_BWD_MUTANTS[mutant]
    src = inspect.getsource(oracle.ssd_bwd)
    assert src.count(old) == 1, "mutation site not found: " + old
    ns = dict(vars(oracle))
    exec(compile(src.replace(old, new), "ssd_bwd_mutant", "exec"), ns)
    monkeypatch.setattr(oracle, "ssd_bwd", ns["ssd_bwd"])
    caught = []
    for name, call in _pin_calls(ssd_pins):
        if not name.startswith("test_backward"):
            continue
        try:
            call()
        except AssertionError:
            caught.append(name)
    assert caught, "no pin caught " + mutant
