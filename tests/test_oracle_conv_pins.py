"""Pins of the fp64 oracle of the scan's front end: causal depthwise conv1d + SiLU.

The summary page ("Mamba: Linear-Time Sequence Modeling", section 4a shape table:
"Conv1d -> SiLU" on (B, L, ED) ahead of the SSM) and the configuration page
("2. Mamba 상세", d_conv = 4) fix the operation.  Each pin reaches the same number
by another route: numpy's full convolution, scipy's logistic function, the
elementwise closed form of a width-1 kernel, and the equality of a chunked pass
(state carried) with a single pass."""
import numpy as np
import pytest
import scipy.special

import oracle


def _x(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape).astype(np.float32)


@pytest.mark.parametrize("K", [2, 3, 4])
def test_linear_part_is_numpy_causal_convolution(K):
    """Without SiLU, bias or state, out = (x * w reversed)[:L], numpy's full convolution
    truncated to the first L outputs (the causal part)."""
    x = _x((2, 5, 33), K)
    w = _x((5, K), 10 + K)
    out, _ = oracle.conv1d(x, w, None, None, silu=False)
    for b in range(2):
        for d in range(5):
            ref = np.convolve(x[b, d].astype(np.float64), w[d, ::-1].astype(np.float64))[:33]
            assert np.max(np.abs(out[b, d] - ref)) < 1e-12


def test_silu_and_bias_follow_the_logistic_function():
    x = _x((1, 4, 40), 1)
    w = _x((4, 4), 2)
    bias = _x((4,), 3)
    lin, _ = oracle.conv1d(x, w, None, None, silu=False)
    out, _ = oracle.conv1d(x, w, bias, None, silu=True)
    v = lin + bias.astype(np.float64)[None, :, None]
    assert np.max(np.abs(out - v * scipy.special.expit(v))) < 1e-13


def test_width_one_is_elementwise():
    x = _x((2, 3, 17), 4)
    w = _x((3, 1), 5)
    bias = _x((3,), 6)
    out, st = oracle.conv1d(x, w, bias, None, silu=True)
    v = w.astype(np.float64)[None, :, :1] * x + bias.astype(np.float64)[None, :, None]
    assert np.max(np.abs(out - v / (1.0 + np.exp(-v)))) < 1e-13
    assert st.shape == (2, 3, 0)


@pytest.mark.parametrize("cut", [1, 2, 7, 20])
def test_chunked_with_state_equals_one_shot(cut):
    """Split the sequence at `cut`: the first part's state (its last K-1 inputs, with
    the initial state in front when the part is shorter) starts the second part."""
    x = _x((2, 3, 21), 7)
    w = _x((3, 4), 8)
    bias = _x((3,), 9)
    s0 = _x((2, 3, 3), 10).astype(np.float64)
    whole, s_whole = oracle.conv1d(x, w, bias, s0)
    a, s_a = oracle.conv1d(np.ascontiguousarray(x[..., :cut]), w, bias, s0)
    b, s_b = oracle.conv1d(np.ascontiguousarray(x[..., cut:]), w, bias, s_a)
    assert np.max(np.abs(np.concatenate([a, b], axis=-1) - whole)) < 1e-14
    assert np.max(np.abs(s_b - s_whole)) == 0.0
    # the state is the last K-1 inputs of the extended sequence (state, x)
    ext = np.concatenate([s0, x.astype(np.float64)], axis=-1)
    assert np.array_equal(s_whole, ext[..., -3:])
    if cut < 3:
        assert np.array_equal(s_a, np.concatenate([s0, x[..., :cut].astype(np.float64)], -1)[..., -3:])


def test_state_enters_the_first_outputs_only():
    """A non-zero initial state changes outputs t < K-1 and nothing after."""
    x = _x((1, 2, 12), 11)
    w = _x((2, 4), 12)
    s0 = _x((1, 2, 3), 13).astype(np.float64)
    a, _ = oracle.conv1d(x, w, None, None, silu=False)
    b, _ = oracle.conv1d(x, w, None, s0, silu=False)
    assert np.all(np.abs(a[..., :3] - b[..., :3]) > 0)
    assert np.array_equal(a[..., 3:], b[..., 3:])
    # and by linearity the difference is the convolution of the state alone
    ref = np.zeros((2, 3))
    for d in range(2):
        for t in range(3):
            ref[d, t] = sum(float(w[0 + d, k]) * s0[0, d, 3 + t - 3 + k] for k in range(4) if t - 3 + k < 0)
    assert np.max(np.abs((b - a)[0, :, :3] - ref)) < 1e-12


# ---------------------------------------------------------------------------
# the backward of the front end (oracle.conv1d_bwd, numpy fp64) against the
# forward oracle (the C code): finite differences, and the exact adjoint identity
# of the linear part
# ---------------------------------------------------------------------------

def _loss(x, w, bias, s0, silu, dout):
    out, _ = oracle.conv1d(x, w, bias, s0, silu=silu)
    return float(np.sum(out * dout))


@pytest.mark.parametrize("K", [1, 2, 4])
def test_backward_linear_part_is_the_adjoint(K):
    """Without SiLU the conv is linear in (state, x) and in (w, bias), so
    <out, dout> = <x, dx> + <state, dstate> = Σ w·dw + Σ bias·dbias exactly (up to
    fp64 rounding): a wrong index, sign or dropped term breaks one of the two."""
    x = _x((2, 3, 19), 20 + K)
    w = _x((3, K), 21)
    bias = _x((3,), 22)
    s0 = _x((2, 3, K - 1), 23)
    dout = _x((2, 3, 19), 24).astype(np.float64)
    g = oracle.conv1d_bwd(x, w, None, s0, False, dout)
    lhs = _loss(x, w, None, s0.astype(np.float64), False, dout)
    rhs = np.sum(x.astype(np.float64) * g["dx"]) + np.sum(s0.astype(np.float64) * g["dstate"])
    assert abs(lhs - rhs) < 1e-11 * max(1.0, abs(lhs))
    gb = oracle.conv1d_bwd(x, w, bias, s0, False, dout)
    lhs_b = _loss(x, w, bias, s0.astype(np.float64), False, dout)
    rhs_b = np.sum(w.astype(np.float64) * gb["dweight"]) + np.sum(bias.astype(np.float64) * gb["dbias"])
    assert abs(lhs_b - rhs_b) < 1e-11 * max(1.0, abs(lhs_b))


@pytest.mark.parametrize("K", [3, 4])
def test_backward_matches_finite_differences(K):
    """With SiLU: central differences of <conv1d(...), dout> (the forward oracle, float32
    inputs perturbed by h = 2^-7, exactly representable) for sampled x, state, weight and
    bias entries."""
    rng = np.random.default_rng(30 + K)
    x = _x((1, 2, 12), 31)
    w = (0.5 * _x((2, K), 32)).astype(np.float32)
    bias = _x((2,), 33)
    s0 = _x((1, 2, K - 1), 34)
    dout = _x((1, 2, 12), 35).astype(np.float64)
    g = oracle.conv1d_bwd(x, w, bias, s0, True, dout)
    h = np.float32(2.0 ** -7)

    def fd(arr, idx, name):
        a, b = arr.copy(), arr.copy()
        a[idx] += h
        b[idx] -= h
        args = dict(x=x, w=w, bias=bias, s0=s0)
        args[name] = a
        up = _loss(args["x"], args["w"], args["bias"], args["s0"].astype(np.float64), True, dout)
        args[name] = b
        dn = _loss(args["x"], args["w"], args["bias"], args["s0"].astype(np.float64), True, dout)
        return (up - dn) / (2 * float(h))

    for _ in range(6):
        i = (0, int(rng.integers(2)), int(rng.integers(12)))
        assert abs(fd(x, i, "x") - g["dx"][i]) < 2e-4 * max(1.0, abs(g["dx"][i]))
    for j in range(K - 1):
        i = (0, 1, j)
        assert abs(fd(s0, i, "s0") - g["dstate"][i]) < 2e-4 * max(1.0, abs(g["dstate"][i]))
    for k in range(K):
        i = (1, k)
        assert abs(fd(w, i, "w") - g["dweight"][i]) < 2e-4 * max(1.0, abs(g["dweight"][i]))
    assert abs(fd(bias, (0,), "bias") - g["dbias"][0]) < 2e-4 * max(1.0, abs(g["dbias"][0]))
