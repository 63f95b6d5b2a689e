"""Pins of the fp64 oracle to facts the pages and the mathematics fix.

None of these checks re-evaluates the oracle's own formula: each compares it
with a different route to the same number (a closed form, a library routine,
an ODE integration, a brute-force sum) chosen so that a plausible slip in the
oracle (a dropped term, a wrong sign, an off-by-one time index, Euler instead
of zero-order hold, reading the state before the update, a gate in the wrong
place) fails at least one of them.

Citations name the page and its section or equation:
  [S]  "Mamba: Linear-Time Sequence Modeling" summary page (Paper2Web), 4b/4c/4d.
  [C]  "14.1 SSM(State Space Models)과 Mamba 아키텍처의 부상" chapter page, 3.1-4.2.
"""
import math

import numpy as np
import pytest
import scipy.integrate
import scipy.linalg
import scipy.special

import oracle
import synth


def _rows(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _scan1(u, dl, A, B, C, D=None, z=None, bias=None, softplus=True, h0=None):
    """Single unit (batch 0, channel 0) helper: u, dl (L,), A (N,), B, C (N, L)."""
    L = len(u)
    N = len(A)
    y, h = oracle.scan_rows(_rows(u)[None], _rows(dl)[None], None if z is None else _rows(z)[None],
                            [0], [0], _rows(A)[None], _rows(B)[None], _rows(C)[None],
                            None if D is None else _rows([D]), None if bias is None else _rows([bias]),
                            softplus, None if h0 is None else np.asarray(h0, np.float64)[None])
    return y[0], h[0]


def _zoh_vanloan(a, b, dt):
    """ZOH pair (Ā, B̄) of the scalar system h' = a h + b x with x held for dt,
    from the matrix exponential of the augmented generator (Van Loan 1978)."""
    M = np.array([[a * dt, b * dt], [0.0, 0.0]])
    E = scipy.linalg.expm(M)
    return E[0, 0], E[0, 1]


# --- Theorem 1 ([S] 4b, equation (5)) -------------------------------------------------

def test_theorem1_gated_rnn():
    """N=1, A=-1, B=1, C=1, softplus on: the scan is h_t = (1-g_t) h_{t-1} + g_t x_t with
    g_t = sigmoid(Δraw_t + bias) ([S] 4b, Theorem 1 and its derivation)."""
    rng = np.random.default_rng(11)
    L = 300
    u = rng.standard_normal(L).astype(np.float32)
    draw = (2.0 * rng.standard_normal(L)).astype(np.float32)
    bias = np.float32(-0.75)
    y, hN = _scan1(u, draw, [-1.0], np.ones((1, L)), np.ones((1, L)), bias=bias)
    g = scipy.special.expit(draw.astype(np.float64) + np.float64(bias))
    h = 0.0
    ref = np.empty(L)
    for t in range(L):
        h = (1.0 - g[t]) * h + g[t] * float(u[t])
        ref[t] = h
    assert np.max(np.abs(y - ref)) < 1e-12
    assert abs(hN[0] - ref[-1]) < 1e-12


# --- LTI special case equals the causal convolution ([S] 4b, eq. (2) derivation) -------

@pytest.mark.parametrize("dt", [1e-3, 0.05, 0.7])
def test_lti_equals_convolution(dt):
    """Constant Δ, B, C (softplus off): y = u * K + D u with
    K_k = Σ_n C_n Ā_n^k B̄_n ([S] 4b convolution mode; [C] 3.3 y = x * K̄)."""
    rng = np.random.default_rng(5)
    L, N = 200, 5
    A = -np.array([0.3, 1.0, 2.5, 4.0, 9.0])
    Bc = rng.standard_normal(N)
    Cc = rng.standard_normal(N)
    D = 0.8
    u = rng.standard_normal(L).astype(np.float32)
    A32 = A.astype(np.float32)
    B32 = Bc.astype(np.float32)
    C32 = Cc.astype(np.float32)
    y, _ = _scan1(u, np.full(L, dt, np.float32), A32, np.repeat(B32[:, None], L, 1),
                  np.repeat(C32[:, None], L, 1), D=D, softplus=False)
    dt64 = float(np.float32(dt))
    K = np.zeros(L)
    for n in range(N):
        abar, bbar = _zoh_vanloan(float(A32[n]), float(B32[n]), dt64)
        K += float(C32[n]) * bbar * abar ** np.arange(L)
    u64 = u.astype(np.float64)
    ref = np.convolve(u64, K)[:L] + float(np.float32(D)) * u64
    assert np.max(np.abs(y - ref)) <= 1e-11 * max(1.0, np.max(np.abs(ref)))


# --- N = 1, constant inputs: closed form of the held-input ODE ([S] eq. (4) derivation) -

def test_n1_constant_closed_form():
    """h_t = (-B u / A)(1 - exp(ΔA (t+1))): the exact solution of h' = A h + B u with u
    held; the steady state -B u / A does not depend on Δ ([S] 4b, ZOH derivation)."""
    L = 500
    A, B, C, D, u, dt = -1.7, 0.6, 1.3, 0.25, 0.9, 0.01
    f = lambda v: float(np.float32(v))
    A, B, C, D, u, dt = map(f, (A, B, C, D, u, dt))
    y, hN = _scan1(np.full(L, u, np.float32), np.full(L, dt, np.float32), [A],
                   np.full((1, L), B), np.full((1, L), C), D=D, softplus=False)
    t = np.arange(L)
    h = (-B * u / A) * (-np.expm1(dt * A * (t + 1)))
    assert np.max(np.abs(y - (C * h + D * u))) < 1e-13
    assert abs(hN[0] - h[-1]) < 1e-13


# --- brute-force unrolling on tiny inputs ([S] eq. (2a)/(2b), Algorithm 2) --------------

def test_brute_force_unrolled_sum():
    """y_t = silu(z_t) (Σ_n C_{n,t} Σ_{s<=t} (Π_{r=s+1..t} Ā_{n,r}) B̄_{n,s} u_s + D u_t),
    with Ā, B̄ from the matrix exponential of each step's held-input system."""
    rng = np.random.default_rng(3)
    batch, dim, L, N = 2, 3, 9, 3
    u = rng.standard_normal((batch, dim, L)).astype(np.float32)
    draw = rng.standard_normal((batch, dim, L)).astype(np.float32)
    z = rng.standard_normal((batch, dim, L)).astype(np.float32)
    A = (-rng.uniform(0.2, 3.0, (dim, N))).astype(np.float32)
    B = rng.standard_normal((batch, N, L)).astype(np.float32)
    C = rng.standard_normal((batch, N, L)).astype(np.float32)
    D = rng.uniform(0.5, 1.5, dim).astype(np.float32)
    bias = rng.uniform(-3, 0, dim).astype(np.float32)
    y, hN = oracle.scan(u, draw, A, B, C, D, z, bias, True)
    for b in range(batch):
        for d in range(dim):
            dts = np.logaddexp(0.0, draw[b, d].astype(np.float64) + float(bias[d]))  # softplus
            for t in range(L):
                acc = 0.0
                for n in range(N):
                    for s in range(t + 1):
                        decay = 1.0
                        for r in range(s + 1, t + 1):
                            decay *= _zoh_vanloan(float(A[d, n]), 1.0, dts[r])[0]
                        bbar = _zoh_vanloan(float(A[d, n]), float(B[b, n, s]), dts[s])[1]
                        acc += float(C[b, n, t]) * decay * bbar * float(u[b, d, s])
                pre = acc + float(D[d]) * float(u[b, d, t])
                ref = pre * float(z[b, d, t]) * scipy.special.expit(float(z[b, d, t]))
                assert abs(y[b, d, t] - ref) < 1e-12 * max(1.0, abs(ref)), (b, d, t)


# --- time-varying ZOH against direct ODE integration ([S] eq. (1a), ZOH reading) --------

def test_matches_ode_integration_with_held_input():
    """Integrate h' = A h + B_t u_t with (B_t, u_t) held over each interval of length Δ_t
    ([S] 4b: ZOH assumes the input constant over the step) and compare the states."""
    rng = np.random.default_rng(8)
    L, N = 12, 3
    A = np.array([-0.5, -2.0, -6.0], np.float32)
    u = rng.standard_normal(L).astype(np.float32)
    dts = rng.uniform(0.05, 0.6, L).astype(np.float32)
    B = rng.standard_normal((N, L)).astype(np.float32)
    C = np.zeros((N, L), np.float32)
    h = np.zeros(N)
    for t in range(L):
        y_t, h_or = _scan1(u[:t + 1], dts[:t + 1], A, B[:, :t + 1], C[:, :t + 1], softplus=False)
        sol = scipy.integrate.solve_ivp(
            lambda _s, x: A.astype(np.float64) * x + B[:, t].astype(np.float64) * float(u[t]),
            (0.0, float(dts[t])), h, method="DOP853", rtol=1e-13, atol=1e-15)
        h = sol.y[:, -1]
        assert np.max(np.abs(h_or - h)) < 1e-10, t


# --- limits of equation (4) ([S] 4b table: Δ→0 gives ΔB; large Δ resets) ---------------

def test_zoh_small_step_tends_to_euler():
    """B̄ / (Δ B) -> 1 as Δ -> 0 ([S] 4b, the B̄ row of the equation (4) table)."""
    for dt in (1e-4, 1e-6, 1e-8):
        y, _ = _scan1([1.0], [dt], [-3.0], [[0.7]], [[1.0]], softplus=False)
        bb = float(np.float32(0.7))
        ratio = y[0] / (float(np.float32(dt)) * bb)
        assert abs(ratio - 1.0) < 3.0 * float(np.float32(dt)) + 1e-12


def test_zoh_large_step_resets_state():
    """Δ large, A < 0: Ā -> 0 and h_t -> -B u_t / A, forgetting h_{t-1} ([S] 4b)."""
    L = 6
    u = np.array([1.0, -2.0, 0.5, 3.0, -1.0, 2.0], np.float32)
    y, _ = _scan1(u, np.full(L, 60.0, np.float32), [-1.5], np.full((1, L), 0.8),
                  np.ones((1, L)), softplus=False)
    ref = -float(np.float32(0.8)) * u.astype(np.float64) / -1.5
    assert np.max(np.abs(y - ref)) < 1e-12


def test_zero_A_is_the_continuous_limit():
    """A = 0 takes the limit B̄ = Δ B (pure integrator) and agrees with tiny |A|."""
    rng = np.random.default_rng(2)
    L = 50
    u = rng.standard_normal(L).astype(np.float32)
    dts = rng.uniform(0.01, 0.2, L).astype(np.float32)
    B = rng.standard_normal((1, L)).astype(np.float32)
    C = np.ones((1, L), np.float32)
    y0, _ = _scan1(u, dts, [0.0], B, C, softplus=False)
    ref = np.cumsum(dts.astype(np.float64) * B[0].astype(np.float64) * u.astype(np.float64))
    assert np.max(np.abs(y0 - ref)) < 1e-12
    ys, _ = _scan1(u, dts, [-1e-12], B, C, softplus=False)
    assert np.max(np.abs(y0 - ys)) < 1e-9


# --- selection: softplus and bias ([S] 4b Algorithm 2, parameterisation; [C] 4.1) -------

def test_softplus_and_bias_placement():
    """One step from h = 0 with N = 1: y = C B̄(Δ) B u with Δ = softplus(Δraw + bias)
    (softplus on) or Δ = Δraw + bias (off); Δ here from numpy's logaddexp."""
    for raw, bias, sp in ((0.3, -2.0, True), (-25.0, 1.0, True), (30.0, 0.5, True),
                          (0.4, 0.1, False)):
        y, _ = _scan1([1.0], [raw], [-2.0], [[1.0]], [[1.0]], bias=bias, softplus=sp)
        x = float(np.float32(raw)) + float(np.float32(bias))
        dt = float(np.logaddexp(0.0, x)) if sp else x
        _, bbar = _zoh_vanloan(-2.0, 1.0, dt)
        assert abs(y[0] - bbar) <= 1e-14 + 1e-12 * abs(bbar), (raw, bias, sp)


# --- the gate and the direct term ([S] 4a shape table; [C] 3.1) --------------------------

def test_gate_multiplies_ssm_output_including_D():
    rng = np.random.default_rng(9)
    w = synth.scaled(synth.TINY, dim=4, seqlen=64, d_one=False)
    x = synth.make_scan_inputs(w)
    y_nz, _ = oracle.scan(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], None, x["delta_bias"])
    y_z, _ = oracle.scan(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"])
    z = x["z"].astype(np.float64)
    np.testing.assert_allclose(y_z, y_nz * z * scipy.special.expit(z), rtol=1e-13, atol=1e-15)
    y_d0, _ = oracle.scan(x["u"], x["delta"], x["A"], x["B"], x["C"], None, None, x["delta_bias"])
    np.testing.assert_allclose(y_nz - y_d0, x["D"][None, :, None].astype(np.float64) * x["u"],
                               rtol=1e-12, atol=1e-13)
    del rng


# --- invariants: causality, linearity, chunk carry, decode == scan ([S] 4b, 4d) --------

def _tiny_bf16():
    w = synth.scaled(synth.MAMBA_130M, batch=2, dim=8, seqlen=96, seed=21)
    return w, synth.make_scan_inputs(w)


def test_causal_and_linear_in_u():
    w, x = _tiny_bf16()
    u = synth.bf16_to_f32(x["u"])
    dl = synth.bf16_to_f32(x["delta"])
    args = (x["A"], x["B"], x["C"], x["D"], None, x["delta_bias"])
    y1, _ = oracle.scan(u, dl, *args)
    u2 = u.copy()
    u2[:, :, 50] += 1.0
    y2, _ = oracle.scan(u2, dl, *args)
    assert np.array_equal(y1[:, :, :50], y2[:, :, :50])
    assert np.max(np.abs(y1[:, :, 50:] - y2[:, :, 50:])) > 0
    y3, _ = oracle.scan((2.0 * u).astype(np.float32), dl, *args)
    np.testing.assert_allclose(y3, 2.0 * y1, rtol=1e-12, atol=1e-13)


def test_bf16_inputs_decode_exactly():
    w, x = _tiny_bf16()
    f = {k: synth.bf16_to_f32(x[k]) for k in ("u", "delta", "z")}
    ya, ha = oracle.scan(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"])
    yb, hb = oracle.scan(f["u"], f["delta"], x["A"], x["B"], x["C"], x["D"], f["z"], x["delta_bias"])
    assert np.array_equal(ya, yb) and np.array_equal(ha, hb)
    assert synth.bf16_to_f32(np.array([0x3F80, 0xC000, 0x0001], np.uint16)).tolist() == \
        [1.0, -2.0, 2.0 ** -133]


def test_chunked_scan_with_carried_state_equals_one_shot():
    w, x = _tiny_bf16()
    full_y, full_h = oracle.scan(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                                 x["delta_bias"])
    h = None
    ys = []
    for t0, t1 in ((0, 17), (17, 64), (64, 96)):
        yk, h = oracle.scan(np.ascontiguousarray(x["u"][:, :, t0:t1]),
                            np.ascontiguousarray(x["delta"][:, :, t0:t1]), x["A"],
                            np.ascontiguousarray(x["B"][:, :, t0:t1]),
                            np.ascontiguousarray(x["C"][:, :, t0:t1]), x["D"],
                            np.ascontiguousarray(x["z"][:, :, t0:t1]), x["delta_bias"],
                            init_state=h)
        ys.append(yk)
    np.testing.assert_allclose(np.concatenate(ys, axis=2), full_y, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(h, full_h, rtol=1e-12, atol=1e-12)


def test_decode_steps_equal_scan():
    """The recurrent mode ([S] 4b: O(N) state update per token) run for L steps equals the
    scan over the same L inputs."""
    w, x = _tiny_bf16()
    L = 20
    y_ref, h_ref = oracle.scan(np.ascontiguousarray(x["u"][:, :, :L]),
                               np.ascontiguousarray(x["delta"][:, :, :L]), x["A"],
                               np.ascontiguousarray(x["B"][:, :, :L]),
                               np.ascontiguousarray(x["C"][:, :, :L]), x["D"],
                               np.ascontiguousarray(x["z"][:, :, :L]), x["delta_bias"])
    st = np.zeros((w.batch, w.dim, w.dstate))
    for t in range(L):
        yt, st = oracle.step(st, x["u"][:, :, t], x["delta"][:, :, t], x["A"], x["B"][:, :, t],
                             x["C"][:, :, t], x["D"], x["z"][:, :, t], x["delta_bias"])
        np.testing.assert_allclose(yt, y_ref[:, :, t], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(st, h_ref, rtol=1e-12, atol=1e-12)


def test_rel_err_metric():
    assert oracle.rel_err([1.0, 2.0], [1.0, 2.0]) == 0.0
    assert math.isclose(oracle.rel_err([1.0, 2.5], [1.0, 2.0]), 0.25)


def test_golden_snapshot_of_tiny_workload():
    """Regression snapshot (tests/golden, written by make_golden.py from the oracle)."""
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "tiny_s6_fp32_oracle.txt")
    w = synth.TINY
    x = synth.make_scan_inputs(w)
    y, h = oracle.scan(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"])
    n = 0
    for line in open(path):
        if line.startswith("#"):
            continue
        kind, b, d, i, v = line.split()
        got = y[int(b), int(d), int(i)] if kind == "y" else h[int(b), int(d), int(i)]
        assert abs(got - float(v)) <= 1e-14 * max(1.0, abs(float(v)))
        n += 1
    assert n == w.dim * (7 + w.dstate)


# --- Euler variant of B̄ ([S] §4b, the first-order form beside equation (4)) -----------

def test_euler_variant_closed_form_and_first_step():
    """Euler B̄ = Δ B with the exact Ā: for constant inputs (N = 1, softplus off)
    h_t = Δ B u (1 - Ā^{t+1}) / (1 - Ā), a geometric series; the first step from a zero
    state differs from the ZOH one by exactly the factor expm1(ΔA) / (ΔA)."""
    L, dt, a_, b_, u_ = 40, 0.37, -1.7, 0.8, 1.3
    u = np.full(L, u_, np.float32)
    dl = np.full(L, dt, np.float32)
    dtf, af, bf, uf = (float(np.float32(v)) for v in (dt, a_, b_, u_))
    ye, he = oracle.scan_rows(_rows(u)[None], _rows(dl)[None], None, [0], [0], _rows([[a_]]),
                              _rows(np.full((1, 1, L), b_)), _rows(np.ones((1, 1, L))), None, None,
                              False, None, 1, 0, euler=True)
    abar = np.exp(dtf * af)
    t = np.arange(L)
    ref = dtf * bf * uf * (1.0 - abar ** (t + 1)) / (1.0 - abar)
    assert np.max(np.abs(ye[0] - ref)) < 1e-13
    yz, _ = _scan1(u, dl, [a_], np.full((1, L), b_), np.ones((1, L)), softplus=False)
    assert abs(yz[0] / ye[0, 0] - np.expm1(dtf * af) / (dtf * af)) < 1e-14
