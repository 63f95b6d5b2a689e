"""GPU parity of the Euler variant (B̄ = Δ B; flag SSM_EULER_B) against the fp64
oracle in the same mode: the scan (one pass and the split plan with carried
segments), the decode step and the backward pass.

Bar: the forward's, 1e-4 for float32 I/O and 1e-2 for bfloat16 I/O, relative
to the largest reference value of each output."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_128_b300 as ssm
import synth
from _gpu import dev_f32, dev_io, host64, upload_scan

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 1e-2}


@pytest.mark.parametrize("io", ["bf16", "f32"])
@pytest.mark.parametrize("N", [1, 4, 16, 64, 128])
def test_scan_euler_matches_oracle(io, N):
    w = synth.scaled(synth.MAMBA_130M, name="euler_scan", batch=2, dim=70, seqlen=150,
                     dstate=N, io=io, seed=90 + N)
    x = synth.make_scan_inputs(w)
    y_ref, h_ref = oracle.scan(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                               x["delta_bias"], True, euler=True)
    g = upload_scan(x)
    y, h = ssm.scan(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"], g["delta_bias"],
                    True, euler=True)
    torch.cuda.synchronize()
    assert oracle.rel_err(host64(y), y_ref) <= TOL[io]
    assert oracle.rel_err(host64(h), h_ref) <= TOL[io]
    # and it is not the zero-order hold
    y_zoh, _ = oracle.scan(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                           x["delta_bias"], True)
    assert oracle.rel_err(y_zoh, y_ref) > 2 * TOL[io] or N == 1


def test_scan_euler_split_plan():
    """Few channels, long sequence: the plan splits L into segments whose carries are
    folded with exp(A ΣΔ); the Euler B̄ changes only the segments' inputs."""
    w = synth.scaled(synth.MAMBA_130M, name="euler_split", batch=1, dim=64, seqlen=8192,
                     seed=95)
    x = synth.make_scan_inputs(w)
    assert ssm.ssm_scan_workspace_bytes(1, 64, 8192, 16, ssm.SSM_BF16) > 0
    y_ref, h_ref = oracle.scan(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                               x["delta_bias"], True, euler=True)
    g = upload_scan(x)
    y, h = ssm.scan(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"], g["delta_bias"],
                    True, euler=True)
    torch.cuda.synchronize()
    assert oracle.rel_err(host64(y), y_ref) <= 1e-2
    assert oracle.rel_err(host64(h), h_ref) <= 1e-2


@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_decode_euler_matches_oracle(io):
    dw = synth.DecodeWorkload("euler_dec", 3, 50, 16, 5, 32, 96, io=io)
    s = synth.make_decode_step_inputs(dw, 0, dw.steps)
    A = synth.gen_A(dw.dim, 16)
    D = synth.fill(97, synth.S_D, 0, dw.dim, synth.UNIFORM, 0.5, 1.5)
    bias = synth.gen_delta_bias(97, dw.dim)
    st0 = np.random.default_rng(3).standard_normal((dw.batch, dw.dim, 16)).astype(np.float32)
    st_ref = st0.astype(np.float64)
    st = dev_f32(st0)
    flags = ssm.SSM_SOFTPLUS | ssm.SSM_EULER_B
    for i in range(dw.steps):
        y_ref, st_ref = oracle.step(st_ref, s["u"][i], s["delta"][i], A, s["B"][i], s["C"][i], D,
                                    s["z"][i], bias, True, euler=True)
        u = dev_io(s["u"][i])
        y = torch.empty_like(u)
        ssm.ssm_state_update_ex(st, u, dev_io(s["delta"][i]), dev_f32(bias), flags, dev_f32(A),
                                dev_f32(s["B"][i]), dev_f32(s["C"][i]), dev_f32(D),
                                dev_io(s["z"][i]), y)
        torch.cuda.synchronize()
        assert oracle.rel_err(host64(y), y_ref) <= TOL[io]
        assert oracle.rel_err(host64(st), st_ref) <= TOL[io]


@pytest.mark.parametrize("io,N", [("bf16", 16), ("f32", 16), ("bf16", 128)])
def test_backward_euler_matches_oracle(io, N):
    w = synth.scaled(synth.MAMBA_130M, name="euler_bwd", batch=2, dim=40, seqlen=70, io=io,
                     dstate=N, seed=98)
    x = synth.make_scan_inputs(w)
    x["A"][1, ::2] = 0.0
    e = synth.make_bwd_inputs(w)
    dy64 = (synth.bf16_to_f32(e["dy"]) if io == "bf16" else e["dy"]).astype(np.float64)
    ref = oracle.scan_bwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                          x["delta_bias"], True, e["init_state"].astype(np.float64), dy64,
                          e["d_final_state"].astype(np.float64), euler=True)
    g = upload_scan(x)
    out = ssm.scan_bwd(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"],
                       g["delta_bias"], True, init_state=dev_f32(e["init_state"]),
                       dy=dev_io(e["dy"]), d_final_state=dev_f32(e["d_final_state"]),
                       want_init_grad=True, euler=True)
    torch.cuda.synchronize()
    for k in ("du", "ddelta", "dz", "dA", "dB", "dC", "dD", "dbias", "dinit"):
        assert oracle.rel_err(host64(out[k]), ref[k]) <= TOL[io], k
