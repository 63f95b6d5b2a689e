"""Pins of the fp64 backward oracle (the derivatives of the scan).

The summary page ("Mamba: Linear-Time Sequence Modeling", section 4c) trains the
layer with the states recomputed in the backward pass but prints no gradient
formula, so the backward oracle is the chain rule applied to the forward
definition.  None of these checks re-derives that chain rule: each compares the
oracle with another route to the same number --

* central finite differences of the (separately pinned) forward oracle, for every
  input that has a derivative, on problems where every term of every gradient is
  of the same order (so a dropped or mis-signed term moves the result well past
  the finite-difference error);
* the transposed causal convolution: in the LTI special case (constant Δ, B, C;
  the summary page's convolution mode, section 4b) y = K * u + D u, so
  dLoss/du is the cross-correlation of dy with the kernel K;
* the state-transition product: with dy = 0 only the final state carries a
  derivative and dLoss/dh_{-1} = exp(A ΣΔ) dLoss/dh_{L-1} elementwise.
"""
import numpy as np
import pytest

import oracle


def _problem(seed, batch=2, dim=3, L=19, N=3, softplus=True, with_z=True, zero_a=False):
    rng = np.random.default_rng(seed)
    f32 = np.float32
    x = dict(
        u=rng.standard_normal((batch, dim, L)).astype(f32),
        delta=(0.8 * rng.standard_normal((batch, dim, L)) + (0.0 if softplus else 0.6)).astype(f32),
        z=rng.standard_normal((batch, dim, L)).astype(f32) if with_z else None,
        A=(-0.2 - 1.3 * rng.random((dim, N))).astype(f32),
        B=rng.standard_normal((batch, N, L)).astype(f32),
        C=rng.standard_normal((batch, N, L)).astype(f32),
        D=rng.standard_normal(dim).astype(f32),
        bias=(0.3 * rng.standard_normal(dim)).astype(f32),
        h0=rng.standard_normal((batch, dim, N)),
    )
    if not softplus:
        x["delta"] = np.abs(x["delta"]) + f32(0.05)
        x["bias"] = np.abs(x["bias"])
    if zero_a:
        x["A"][1, 0] = 0.0
    dy = rng.standard_normal((batch, dim, L))
    dfin = rng.standard_normal((batch, dim, N))
    return x, dy, dfin


def _loss(x, dy, dfin, softplus, euler=False):
    y, hN = oracle.scan(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"], x["bias"],
                        softplus, x["h0"], euler=euler)
    return float(np.sum(y * dy) + np.sum(hN * dfin))


def _fd(x, dy, dfin, softplus, name, step=2.0 ** -11, euler=False):
    """Central differences of the loss over every element of input `name`, dividing by
    the difference of the values actually fed (float32 inputs round)."""
    base = x[name]
    g = np.empty(base.shape, dtype=np.float64)
    for idx in np.ndindex(base.shape):
        v0 = base[idx]
        xp = dict(x)
        arr = base.copy()
        arr[idx] = v0 + step
        hi = float(arr[idx])
        xp[name] = arr
        lp = _loss(xp, dy, dfin, softplus, euler)
        arr = base.copy()
        arr[idx] = v0 - step
        lo = float(arr[idx])
        xp[name] = arr
        lm = _loss(xp, dy, dfin, softplus, euler)
        g[idx] = (lp - lm) / (hi - lo)
    return g


def _grads(x, dy, dfin, softplus, euler=False):
    return oracle.scan_bwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"], x["bias"],
                           softplus, x["h0"], dy, dfin, euler=euler)


NAMES = {"u": "du", "delta": "ddelta", "z": "dz", "A": "dA", "B": "dB", "C": "dC", "D": "dD",
         "bias": "dbias", "h0": "dinit"}


@pytest.mark.parametrize("case", ["softplus_gate", "no_softplus_no_gate", "zero_A", "euler"])
def test_gradients_match_finite_differences(case):
    softplus = case != "no_softplus_no_gate"
    euler = case == "euler"
    x, dy, dfin = _problem({"softplus_gate": 1, "no_softplus_no_gate": 2, "zero_A": 3,
                            "euler": 5}[case],
                           softplus=softplus, with_z=case != "no_softplus_no_gate",
                           zero_a=case in ("zero_A", "euler"))
    g = _grads(x, dy, dfin, softplus, euler)
    for name, key in NAMES.items():
        if x[name] is None:
            assert g[key] is None
            continue
        fd = _fd(x, dy, dfin, softplus, name, euler=euler)
        scale = np.max(np.abs(fd))
        assert scale > 1e-3, name
        err = np.max(np.abs(g[key] - fd)) / scale
        assert err < 2e-5, (name, err)


def test_lti_input_gradient_is_correlation_with_kernel():
    """Constant Δ, B, C, softplus off, no gate: y = K * u + D u with
    K_k = Σ_n C_n Ā_n^k B̄_n ([S] 4b convolution mode), so
    dLoss/du_t = Σ_{k>=0} K_k dy_{t+k} + D dy_t."""
    rng = np.random.default_rng(9)
    L, N = 64, 4
    A = -np.array([[0.4, 1.0, 2.2, 5.0]], dtype=np.float32)
    dt = np.float32(0.11)
    Bc = rng.standard_normal(N).astype(np.float32)
    Cc = rng.standard_normal(N).astype(np.float32)
    u = rng.standard_normal((1, 1, L)).astype(np.float32)
    dl = np.full((1, 1, L), dt, dtype=np.float32)
    Bt = np.repeat(Bc[None, :, None], L, axis=2)
    Ct = np.repeat(Cc[None, :, None], L, axis=2)
    D = np.array([0.7], dtype=np.float32)
    dy = rng.standard_normal((1, 1, L))
    g = oracle.scan_bwd(u, dl, A, Bt, Ct, D, None, None, False, None, dy)
    a = np.exp(np.float64(dt) * A[0].astype(np.float64))
    bb = np.expm1(np.float64(dt) * A[0].astype(np.float64)) / A[0].astype(np.float64)
    K = np.array([np.sum(Cc * a ** k * bb * Bc) for k in range(L)])
    ref = np.correlate(dy[0, 0], K, mode="full")[L - 1:] + np.float64(D[0]) * dy[0, 0]
    assert np.max(np.abs(g["du"][0, 0] - ref)) < 1e-12 * np.max(np.abs(ref)) * L


def test_final_state_derivative_decays_by_transition_product():
    """dy = 0: only dLoss/dh_{L-1} is non-zero, and h_{L-1} depends on h_{-1}
    through Π_t Ā_t = exp(A Σ_t Δ_t) per state ([S] 4b equation (4))."""
    x, _, dfin = _problem(4, L=37, N=4)
    dy = np.zeros_like(x["u"], dtype=np.float64)
    g = _grads(x, dy, dfin, True)
    xb = x["delta"].astype(np.float64) + x["bias"].astype(np.float64)[None, :, None]
    sdt = np.sum(np.logaddexp(0.0, xb), axis=2)                     # Σ_t softplus
    ref = np.exp(sdt[:, :, None] * x["A"].astype(np.float64)[None]) * dfin
    assert np.max(np.abs(g["dinit"] - ref)) < 1e-13
    # with dy = 0 nothing reaches C or the gate, and dD = 0
    assert np.max(np.abs(g["dC"])) == 0.0
    assert np.max(np.abs(g["dz"])) == 0.0 and np.max(np.abs(g["dD"])) == 0.0
