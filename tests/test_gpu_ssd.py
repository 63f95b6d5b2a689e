"""GPU parity of the chunked scalar-A SSM (Mamba-2 SSD) against the fp64 oracle (the
plain recurrence, pinned by the masked-attention duality and the chunked
decomposition).

Inputs are bf16 (x, dt, z, B, C) as the products run in bf16; the oracle reads the
same bits.  Bar: max|gpu - ref| / max|ref| <= 1e-2 for y and the final state."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_128_b300 as ssm
import synth
from _gpu import dev_f32, dev_io, host64

pytestmark = pytest.mark.gpu

TOL = 1e-2


def _inputs(batch, L, H, G, N, seed, P=64):
    f = lambda s, n, std: synth.fill(seed, s, 0, n, synth.NORMAL, 0.0, std, dtype="bf16")
    x = f(synth.S_U, batch * L * H * P, 1.0).reshape(batch, L, H, P)
    z = f(synth.S_Z, batch * L * H * P, 1.0).reshape(batch, L, H, P)
    dt = f(synth.S_DELTA, batch * L * H, 0.5).reshape(batch, L, H)
    B = f(synth.S_B, batch * L * G * N, 1.0).reshape(batch, L, G, N)
    C = f(synth.S_C, batch * L * G * N, 1.0).reshape(batch, L, G, N)
    # per head: A from [-8, -1], D ~ U(0.5, 1.5), bias from dt ~ logU[1e-3, 0.1]
    A = -synth.fill(seed, synth.S_DT, 0, H, synth.UNIFORM, 1.0, 8.0)
    D = synth.fill(seed, synth.S_D, 0, H, synth.UNIFORM, 0.5, 1.5)
    bias = synth.gen_delta_bias(seed, H)
    h0 = synth.fill(seed, synth.S_H0, 0, batch * H * P * N, synth.NORMAL, 0.0, 1.0).reshape(batch, H, P, N)
    return dict(x=x, z=z, dt=dt, B=B, C=C, A=A, D=D, bias=bias, h0=h0)


def _f32(bits):
    return synth.bf16_to_f32(bits)


@pytest.mark.parametrize("case", ["n64_g2", "n128_g1", "ragged", "no_gate_no_D", "init_state",
                                  "euler", "no_softplus", "one_chunk", "single_step",
                                  "three_heads_per_group"])
def test_ssd_matches_oracle(case):
    cfg = dict(batch=2, L=200, H=4, G=2, N=64)
    cfg.update(dict(n128_g1=dict(N=128, G=1), ragged=dict(L=131), one_chunk=dict(L=64),
                    single_step=dict(L=1), init_state=dict(L=150),
                    three_heads_per_group=dict(H=6, G=2, L=100)).get(case, {}))
    x = _inputs(seed=300 + len(case), **cfg)
    use_z = case != "no_gate_no_D"
    use_D = case != "no_gate_no_D"
    h0 = x["h0"] if case == "init_state" else None
    euler = case == "euler"
    softplus = case != "no_softplus"
    if not softplus:  # Δ used as given: a positive step
        x["dt"] = synth.f32_to_bf16(np.abs(_f32(x["dt"])) * 0.1 + 0.01)
        x["bias"] = None
    y_ref, h_ref = oracle.ssd(x["x"], x["dt"], x["A"], _f32(x["B"]), _f32(x["C"]),
                              x["D"] if use_D else None, x["z"] if use_z else None, x["bias"],
                              softplus, None if h0 is None else h0.astype(np.float64), euler=euler)
    y, h = ssm.ssd(dev_io(x["x"]), dev_io(x["dt"]), dev_f32(x["A"]), dev_io(x["B"]), dev_io(x["C"]),
                   dev_f32(x["D"]) if use_D else None, dev_io(x["z"]) if use_z else None,
                   dev_f32(x["bias"]) if x["bias"] is not None else None, softplus,
                   dev_f32(h0) if h0 is not None else None, euler=euler)
    torch.cuda.synchronize()
    ey, eh = oracle.rel_err(host64(y), y_ref), oracle.rel_err(host64(h), h_ref)
    assert np.isfinite(host64(y)).all()
    assert ey <= TOL, ey
    assert eh <= TOL, eh


@pytest.mark.slow
def test_ssd_bench_shape_sampled():
    """The bench's Mamba-2-130M-shaped layer (batch 8, L 2048, 24 heads x 64, N 128) on
    the GPU; the oracle recomputes 3 sampled (batch, head) pairs over the whole
    sequence (y at every step, and the final state)."""
    cfg = dict(batch=8, L=2048, H=24, G=1, N=128)
    x = _inputs(seed=350, **cfg)
    y, h = ssm.ssd(dev_io(x["x"]), dev_io(x["dt"]), dev_f32(x["A"]), dev_io(x["B"]),
                   dev_io(x["C"]), dev_f32(x["D"]), dev_io(x["z"]), dev_f32(x["bias"]))
    torch.cuda.synchronize()
    yh, hh = host64(y), host64(h)
    for b, hd in ((0, 0), (3, 11), (7, 23)):
        sl = lambda a: np.ascontiguousarray(a[b:b + 1, :, hd:hd + 1])
        y_ref, h_ref = oracle.ssd(sl(x["x"]), sl(x["dt"]), x["A"][hd:hd + 1],
                                  _f32(x["B"][b:b + 1]), _f32(x["C"][b:b + 1]),
                                  x["D"][hd:hd + 1], sl(x["z"]), x["bias"][hd:hd + 1], True)
        assert oracle.rel_err(yh[b:b + 1, :, hd:hd + 1], y_ref) <= TOL
        assert oracle.rel_err(hh[b:b + 1, hd:hd + 1], h_ref) <= TOL


# ---------------------------------------------------------------------------
# the backward (ssm_ssd_bwd) against oracle.ssd_bwd
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("case", ["n64_g2", "n128_g1", "n128_g2_three_chunks", "euler",
                                  "no_gate_no_D", "single_step", "three_heads_per_group",
                                  "no_init_no_dfinal"])
def test_ssd_backward_matches_oracle(case):
    cfg = dict(batch=2, L=90, H=4, G=2, N=64)
    cfg.update(dict(n128_g1=dict(N=128, G=1, L=70), n128_g2_three_chunks=dict(N=128, G=2, L=150),
                    single_step=dict(L=1), three_heads_per_group=dict(H=6, G=2, L=50)).get(case, {}))
    x = _inputs(seed=400 + len(case), **cfg)
    use_z = use_D = case != "no_gate_no_D"
    euler = case == "euler"
    rng = np.random.default_rng(7)
    dy = synth.f32_to_bf16(rng.standard_normal(x["x"].shape).astype(np.float32))
    dfin = rng.standard_normal(x["h0"].shape).astype(np.float32)
    states = case != "no_init_no_dfinal"
    ref = oracle.ssd_bwd(x["x"], x["dt"], x["A"], _f32(x["B"]), _f32(x["C"]),
                         x["D"] if use_D else None, x["z"] if use_z else None, x["bias"], True,
                         x["h0"].astype(np.float64) if states else None,
                         dy=_f32(dy).astype(np.float64),
                         d_final_state=dfin.astype(np.float64) if states else None, euler=euler)
    out = ssm.ssd_bwd(dev_io(x["x"]), dev_io(x["dt"]), dev_f32(x["A"]), dev_io(x["B"]), dev_io(x["C"]),
                      dev_f32(x["D"]) if use_D else None, dev_io(x["z"]) if use_z else None,
                      dev_f32(x["bias"]), True, dev_f32(x["h0"]) if states else None, dy=dev_io(dy),
                      d_final_state=dev_f32(dfin) if states else None, euler=euler)
    torch.cuda.synchronize()
    pairs = [("dx", "dx", 1e-2), ("ddt", "ddt", 1e-2), ("dA", "dA", 1e-4), ("dB", "dB", 1e-4),
             ("dC", "dC", 1e-4), ("ddt_bias", "ddt_bias", 1e-4), ("dinit", "dinit", 1e-4)]
    if use_z:
        pairs.append(("dz", "dz", 1e-2))
    if use_D:
        pairs.append(("dD", "dD", 1e-4))
    for k, rk, tol in pairs:
        got = host64(out[k])
        assert np.isfinite(got).all(), k
        assert oracle.rel_err(got, ref[rk]) <= tol, (k, oracle.rel_err(got, ref[rk]))


def test_ssd_backward_empty_sequence():
    """L = 0: no step, so the head parameters' derivatives are zero and d init_state is
    d final_state."""
    x = _inputs(batch=2, L=1, H=4, G=2, N=64, seed=450)
    e = lambda a: a[:, :0]
    dfin = np.random.default_rng(8).standard_normal(x["h0"].shape).astype(np.float32)
    out = ssm.ssd_bwd(dev_io(e(x["x"])), dev_io(e(x["dt"])), dev_f32(x["A"]), dev_io(e(x["B"])),
                      dev_io(e(x["C"])), dev_f32(x["D"]), dev_io(e(x["z"])), dev_f32(x["bias"]), True,
                      dev_f32(x["h0"]), dy=dev_io(e(x["x"])), d_final_state=dev_f32(dfin))
    torch.cuda.synchronize()
    assert out["dx"].shape == (2, 0, 4, 64)
    for k in ("dA", "dD", "ddt_bias"):
        assert out[k].abs().max().item() == 0.0, k
    assert np.array_equal(host64(out["dinit"]), dfin.astype(np.float64))


@pytest.mark.slow
def test_ssd_backward_bench_shape_sampled():
    """The backward at the bench's layer size (batch 8, L 2048, 24 heads x 64, N 128): dx,
    ddt, dz of 3 sampled (batch, head) pairs over the whole sequence, and dB, dC of one
    batch row in full (they sum over its 24 heads), against the oracle; every output
    finite."""
    cfg = dict(batch=8, L=2048, H=24, G=1, N=128)
    x = _inputs(seed=360, **cfg)
    rng = np.random.default_rng(9)
    dy = synth.f32_to_bf16(rng.standard_normal(x["x"].shape).astype(np.float32))
    out = ssm.ssd_bwd(dev_io(x["x"]), dev_io(x["dt"]), dev_f32(x["A"]), dev_io(x["B"]),
                      dev_io(x["C"]), dev_f32(x["D"]), dev_io(x["z"]), dev_f32(x["bias"]), True,
                      dy=dev_io(dy))
    torch.cuda.synchronize()
    for k in ("dx", "ddt", "dz", "dB", "dC", "dA", "dD", "ddt_bias"):
        assert torch.isfinite(out[k].float()).all().item(), k
    dy64 = _f32(dy).astype(np.float64)
    for b, hd in ((0, 0), (3, 11), (7, 23)):
        sl = lambda a: np.ascontiguousarray(a[b:b + 1, :, hd:hd + 1])
        ref = oracle.ssd_bwd(sl(x["x"]), sl(x["dt"]), x["A"][hd:hd + 1], _f32(x["B"][b:b + 1]),
                             _f32(x["C"][b:b + 1]), x["D"][hd:hd + 1], sl(x["z"]),
                             x["bias"][hd:hd + 1], True, dy=sl(dy64))
        for k in ("dx", "dz"):
            assert oracle.rel_err(host64(out[k][b:b + 1, :, hd:hd + 1]), ref[k]) <= TOL, k
        assert oracle.rel_err(host64(out["ddt"][b:b + 1, :, hd:hd + 1]), ref["ddt"]) <= TOL
    b = 5
    sb = lambda a: np.ascontiguousarray(a[b:b + 1])
    ref = oracle.ssd_bwd(sb(x["x"]), sb(x["dt"]), x["A"], _f32(sb(x["B"])), _f32(sb(x["C"])),
                         x["D"], sb(x["z"]), x["bias"], True, dy=sb(dy64))
    for k in ("dB", "dC"):
        assert oracle.rel_err(host64(out[k][b:b + 1]), ref[k]) <= 1e-4, k
