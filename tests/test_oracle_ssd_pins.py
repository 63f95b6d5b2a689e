"""Pins of the oracle of Mamba-2's scalar-A SSM (SSD).

The chapter page ("14.1 SSM(State Space Models)과 Mamba 아키텍처의 부상", §5.1-5.2)
restricts A to a scalar per step times the identity and states the duality
Y = (L ∘ C Bᵀ) X, L the lower-triangular matrix of cumulative products of the
scalar decays; §5.2 computes it chunk by chunk (quadratic form inside a chunk,
states passed between chunks).  The oracle is the plain recurrence; these pins
reach the same numbers by those two other routes, with numpy matrix products:

* the masked-attention (quadratic) form over the whole sequence, with the initial
  state's contribution exp(Σ Δ a) C h0 and the final state as a decayed sum;
* the chunked form (intra-chunk quadratic product + inter-chunk state passing).

Readings: head h uses B, C of group h // (H / G); the discrete input weight is the
selective scan's (zero-order hold: (exp(Δ a) - 1) / a; or Δ with the Euler flag),
a scalar per (step, head) that scales x."""
import numpy as np
import pytest

import oracle


def _problem(seed, batch=2, L=37, H=4, P=3, G=2, N=5):
    rng = np.random.default_rng(seed)
    f = np.float32
    return dict(
        x=rng.standard_normal((batch, L, H, P)).astype(f),
        dt=(0.6 * rng.standard_normal((batch, L, H))).astype(f),
        A=-(0.3 + 2.0 * rng.random(H)).astype(f),
        B=rng.standard_normal((batch, L, G, N)).astype(f),
        C=rng.standard_normal((batch, L, G, N)).astype(f),
        D=rng.standard_normal(H).astype(f),
        z=rng.standard_normal((batch, L, H, P)).astype(f),
        bias=(0.3 * rng.standard_normal(H)).astype(f),
        h0=rng.standard_normal((batch, H, P, N)),
    )


def _terms(p, b, h, euler):
    """Per head: Δ, a, cumulative log-decay s, input weight β, and the group's B, C."""
    H, G = p["x"].shape[2], p["B"].shape[2]
    g = h // (H // G)
    xdt = p["dt"][b, :, h].astype(np.float64) + np.float64(p["bias"][h])
    dlt = np.logaddexp(0.0, xdt)                      # softplus
    a = np.float64(p["A"][h])
    s = np.cumsum(dlt * a)
    beta = dlt if euler else np.expm1(dlt * a) / a
    return dlt, a, s, beta, p["B"][b, :, g].astype(np.float64), p["C"][b, :, g].astype(np.float64)


def _gate(y, z):
    return y * z / (1.0 + np.exp(-z))


@pytest.mark.parametrize("euler", [False, True])
def test_duality_masked_attention_form(euler):
    p = _problem(1)
    y, hN = oracle.ssd(p["x"], p["dt"], p["A"], p["B"], p["C"], p["D"], p["z"], p["bias"], True,
                       p["h0"], euler=euler)
    batch, L, H, P = p["x"].shape
    for b in range(batch):
        for h in range(H):
            dlt, a, s, beta, Bm, Cm = _terms(p, b, h, euler)
            Lm = np.tril(np.exp(s[:, None] - s[None, :]))           # L[t, τ] = Π_{τ<k<=t} ā_k
            X = p["x"][b, :, h, :].astype(np.float64)
            Yq = (Lm * (Cm @ Bm.T)) @ (beta[:, None] * X)            # (L ∘ C Bᵀ) X̃
            Yq += np.exp(s)[:, None] * (Cm @ p["h0"][b, h].T)        # the initial state
            Yq += np.float64(p["D"][h]) * X
            ref = _gate(Yq, p["z"][b, :, h, :].astype(np.float64))
            assert np.max(np.abs(y[b, :, h, :] - ref)) < 1e-11 * max(1.0, np.max(np.abs(ref)))
            # final state: Σ_τ exp(s_L - s_τ) β_τ x_τ ⊗ B_τ + exp(s_L) h0
            w = np.exp(s[-1] - s) * beta
            href = (w[:, None] * X).T @ Bm + np.exp(s[-1]) * p["h0"][b, h]
            assert np.max(np.abs(hN[b, h] - href)) < 1e-11 * max(1.0, np.max(np.abs(href)))


@pytest.mark.parametrize("Q", [1, 4, 8])
def test_chunked_decomposition(Q):
    """Inside each chunk of Q steps the quadratic form; between chunks the state
    H_c = exp(Σ_chunk Δ a) H_{c-1} + Σ_τ exp(s_end - s_τ) β_τ x_τ ⊗ B_τ, and the
    chunk's outputs read the entering state through exp(s_t - s_start) C_t H_{c-1}."""
    p = _problem(2, L=29)
    y, hN = oracle.ssd(p["x"], p["dt"], p["A"], p["B"], p["C"], None, None, p["bias"], True,
                       p["h0"])
    batch, L, H, P = p["x"].shape
    for b in range(batch):
        for h in range(H):
            dlt, a, s, beta, Bm, Cm = _terms(p, b, h, False)
            X = beta[:, None] * p["x"][b, :, h, :].astype(np.float64)
            Hs = p["h0"][b, h].copy()
            out = np.zeros((L, P))
            for c0 in range(0, L, Q):
                c1 = min(L, c0 + Q)
                sl = np.concatenate([[0.0], np.cumsum(dlt[c0:c1] * a)])[1:]  # decay within the chunk
                Lm = np.tril(np.exp(sl[:, None] - sl[None, :]))
                out[c0:c1] = (Lm * (Cm[c0:c1] @ Bm[c0:c1].T)) @ X[c0:c1]
                out[c0:c1] += np.exp(sl)[:, None] * (Cm[c0:c1] @ Hs.T)
                w = np.exp(sl[-1] - sl)
                Hs = np.exp(sl[-1]) * Hs + (w[:, None] * X[c0:c1]).T @ Bm[c0:c1]
            assert np.max(np.abs(y[b, :, h, :] - out)) < 1e-11 * max(1.0, np.max(np.abs(out)))
            assert np.max(np.abs(hN[b, h] - Hs)) < 1e-11 * max(1.0, np.max(np.abs(Hs)))


# ---------------------------------------------------------------------------
# the backward (oracle.ssd_bwd: the scan backward's per-channel terms summed over
# the tied parameters) against central finite differences of the forward oracle
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("euler", [False, True])
def test_backward_matches_finite_differences(euler):
    p = _problem(3, batch=2, L=11, H=4, P=2, G=2, N=3)
    rng = np.random.default_rng(4)
    dy = rng.standard_normal(p["x"].shape)
    dfin = rng.standard_normal(p["h0"].shape)
    g = oracle.ssd_bwd(p["x"], p["dt"], p["A"], p["B"], p["C"], p["D"], p["z"], p["bias"], True,
                       p["h0"], dy=dy, d_final_state=dfin, euler=euler)
    h = 2.0 ** -9

    def loss(q):
        y, hN = oracle.ssd(q["x"], q["dt"], q["A"], q["B"], q["C"], q["D"], q["z"], q["bias"], True,
                           q["h0"], euler=euler)
        return float(np.sum(y * dy) + np.sum(hN * dfin))

    def fd(name, idx):
        up, dn = dict(p), dict(p)
        up[name] = p[name].copy()
        dn[name] = p[name].copy()
        up[name][idx] += h
        dn[name][idx] -= h
        return (loss(up) - loss(dn)) / (2 * h)

    # two batch rows: the head parameters' derivatives sum over both
    checks = [("x", "dx", (0, 5, 1, 1)), ("x", "dx", (1, 0, 3, 0)), ("z", "dz", (1, 7, 2, 1)),
              ("dt", "ddt", (0, 3, 0)), ("dt", "ddt", (1, 10, 3)), ("A", "dA", (1,)),
              ("A", "dA", (2,)), ("B", "dB", (0, 4, 1, 2)), ("B", "dB", (1, 9, 0, 0)),
              ("C", "dC", (1, 6, 0, 1)), ("D", "dD", (3,)), ("bias", "ddt_bias", (0,)),
              ("h0", "dinit", (1, 2, 1, 2))]
    for name, gname, idx in checks:
        ref = fd(name, idx)
        got = g[gname][idx]
        assert abs(got - ref) < 1e-4 * max(1.0, abs(ref)), (name, idx, got, ref)
