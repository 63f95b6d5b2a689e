"""Pins of the complex-A oracle (oracle.scan_complex) against what the mathematics
fixes: the real case reduces to the real oracle; a time-invariant system is a
convolution with the kernel Re(Σ_n C_n B̄_n B_n Ā_n^k) (numpy powers and
numpy.convolve); a brute-force sum over the products of the step factors on tiny
inputs (no recurrence); a conjugate pair of states gives twice the real part of one."""
import cmath
import math

import numpy as np

import oracle
import synth


def _rng(seed):
    return np.random.default_rng(seed)


def _complex_A(rng, dim, N):
    return (-rng.uniform(0.2, 2.0, (dim, N)) + 1j * rng.uniform(-3.0, 3.0, (dim, N)))


def test_real_A_reduces_to_the_real_oracle():
    w = synth.scaled(synth.MAMBA_130M, batch=2, dim=5, seqlen=40, dstate=4, io="f32", seed=500)
    x = synth.make_scan_inputs(w)
    y_r, h_r = oracle.scan(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                           x["delta_bias"])
    y_c, h_c = oracle.scan_complex(x["u"], x["delta"], x["A"].astype(np.complex128),
                                   x["B"].astype(np.complex128), x["C"].astype(np.complex128),
                                   x["D"], x["z"], x["delta_bias"])
    assert oracle.rel_err(y_c, y_r) < 1e-12
    assert np.max(np.abs(h_c.imag)) == 0.0
    assert oracle.rel_err(h_c.real, h_r) < 1e-12


def test_time_invariant_system_is_a_convolution():
    rng = _rng(501)
    dim, N, L, dt = 3, 4, 60, 0.07
    A = _complex_A(rng, dim, N)
    Bn = rng.standard_normal((1, N)) + 1j * rng.standard_normal((1, N))
    Cn = rng.standard_normal((1, N)) + 1j * rng.standard_normal((1, N))
    B = np.repeat(Bn[:, :, None], L, axis=2)
    C = np.repeat(Cn[:, :, None], L, axis=2)
    u = rng.standard_normal((1, dim, L)).astype(np.float32)
    delta = np.zeros((1, dim, L), np.float32)
    bias = np.full(dim, dt, np.float32)
    D = rng.standard_normal(dim).astype(np.float32)
    y, _ = oracle.scan_complex(u, delta, A, B, C, D, None, bias, delta_softplus=False)
    dtf = float(np.float32(dt))
    for d in range(dim):
        Abar = np.exp(dtf * A[d])
        Bbar = (Abar - 1.0) / A[d]
        k = np.arange(L)
        K = np.real(np.sum((Cn[0] * Bbar * Bn[0])[None, :] * np.power(Abar[None, :], k[:, None]), axis=1))
        ud = u[0, d].astype(np.float64)
        ref = np.convolve(ud, K)[:L] + float(D[d]) * ud
        assert oracle.rel_err(y[0, d], ref) < 1e-12


def _brute(u, delta, A, B, C, D, z, bias, softplus, euler):
    """h_t = Σ_{k<=t} (Π_{j=k+1..t} Ā_j) B̄_k B_k u_k for every t from scratch."""
    batch, dim, L = u.shape
    N = A.shape[1]
    y = np.zeros((batch, dim, L))
    for b in range(batch):
        for d in range(dim):
            dts = []
            for t in range(L):
                x = float(delta[b, d, t]) + float(bias[d])
                dts.append(math.log1p(math.exp(x)) if softplus else x)
            for t in range(L):
                acc = 0.0
                for n in range(N):
                    a = complex(A[d, n])
                    hn = 0j
                    for k in range(t + 1):
                        prod = 1 + 0j
                        for j in range(k + 1, t + 1):
                            prod *= cmath.exp(dts[j] * a)
                        bb = dts[k] if euler else (cmath.exp(dts[k] * a) - 1) / a
                        hn += prod * bb * complex(B[b, n, k]) * float(u[b, d, k])
                    acc += (complex(C[b, n, t]) * hn).real
                yv = acc + float(D[d]) * float(u[b, d, t])
                if z is not None:
                    zt = float(z[b, d, t])
                    yv *= zt / (1.0 + math.exp(-zt))
                y[b, d, t] = yv
    return y


def test_brute_force_sum_on_tiny_inputs():
    rng = _rng(502)
    batch, dim, L, N = 1, 2, 6, 3
    A = _complex_A(rng, dim, N)
    B = rng.standard_normal((batch, N, L)) + 1j * rng.standard_normal((batch, N, L))
    C = rng.standard_normal((batch, N, L)) + 1j * rng.standard_normal((batch, N, L))
    u = rng.standard_normal((batch, dim, L)).astype(np.float32)
    delta = (0.5 * rng.standard_normal((batch, dim, L))).astype(np.float32)
    z = rng.standard_normal((batch, dim, L)).astype(np.float32)
    D = rng.standard_normal(dim).astype(np.float32)
    bias = np.array([-2.0, -1.0], np.float32)
    for euler in (False, True):
        y, _ = oracle.scan_complex(u, delta, A, B, C, D, z, bias, euler=euler)
        ref = _brute(u, delta, A, B, C, D, z, bias, True, euler)
        assert oracle.rel_err(y, ref) < 1e-12, euler


def test_a_conjugate_pair_gives_twice_the_real_part_of_one_state():
    rng = _rng(503)
    batch, dim, L = 2, 3, 30
    A1 = _complex_A(rng, dim, 1)
    B1 = rng.standard_normal((batch, 1, L)) + 1j * rng.standard_normal((batch, 1, L))
    C1 = rng.standard_normal((batch, 1, L)) + 1j * rng.standard_normal((batch, 1, L))
    u = rng.standard_normal((batch, dim, L)).astype(np.float32)
    delta = (0.5 * rng.standard_normal((batch, dim, L))).astype(np.float32)
    bias = np.full(dim, -1.5, np.float32)
    y1, _ = oracle.scan_complex(u, delta, A1, B1, 2.0 * C1, None, None, bias)
    y2, h2 = oracle.scan_complex(u, delta, np.concatenate([A1, A1.conj()], 1),
                                 np.concatenate([B1, B1.conj()], 1),
                                 np.concatenate([C1, C1.conj()], 1), None, None, bias)
    assert oracle.rel_err(y2, y1) < 1e-12
    assert np.max(np.abs(h2[:, :, 1] - h2[:, :, 0].conj())) < 1e-12


def test_zero_A_takes_the_limit():
    rng = _rng(504)
    A = np.zeros((2, 2), np.complex128)
    B = rng.standard_normal((1, 2, 5)) + 1j * rng.standard_normal((1, 2, 5))
    C = rng.standard_normal((1, 2, 5)) + 1j * rng.standard_normal((1, 2, 5))
    u = rng.standard_normal((1, 2, 5)).astype(np.float32)
    delta = (0.3 * rng.standard_normal((1, 2, 5))).astype(np.float32)
    bias = np.zeros(2, np.float32)
    y, h = oracle.scan_complex(u, delta, A, B, C, None, None, bias)
    # the A = 0 limit: Ā = 1, B̄ = Δ (the Euler weight, exactly)
    ref = _brute(u, delta, A + 1e-300, B, C, np.zeros(2), None, bias, True, True)
    assert oracle.rel_err(y, ref) < 1e-9
    assert np.isfinite(h).all()
