"""GPU parity of the (batch, L, dim) layout (SSM_LAYOUT_BLD; Algorithm 2's (B, L, D))
for the scan, the training forward, the backward and the conv1d front end.

Each case runs the oracle on the (batch, dim, L) transposes of the same inputs (bar:
1e-4 for float32 I/O, 1e-2 for bfloat16) and also requires the result to equal, bit
for bit, the transpose of the (batch, dim, L) run: the layout changes only where
elements are read and written, not the arithmetic."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_128_b300 as ssm
import synth
from _gpu import dev_f32, dev_io, host64, upload_scan

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 1e-2}


def _bld(t):
    """(batch, dim, L) device tensor -> contiguous (batch, L, dim)."""
    return None if t is None else t.transpose(1, 2).contiguous()


@pytest.mark.parametrize("io,N,dim,L", [
    ("bf16", 16, 96, 200),   # TMA staging: rows of 96 bf16 are 16-byte multiples
    ("bf16", 16, 70, 77),    # element-wise staging: rows of 70 bf16 are not
    ("f32", 16, 40, 50),
    ("bf16", 1, 130, 64),
    ("bf16", 4, 64, 33),
    ("bf16", 64, 40, 48),
])
def test_scan_bld_matches_oracle_and_the_dim_major_run(io, N, dim, L):
    w = synth.scaled(synth.MAMBA_130M, name="bld_scan", batch=2, dim=dim, seqlen=L, dstate=N,
                     io=io, seed=140 + N + dim)
    x = synth.make_scan_inputs(w)
    y_ref, h_ref = oracle.scan(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                               x["delta_bias"], True)
    g = upload_scan(x)
    y0, h0 = ssm.scan(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"], g["delta_bias"])
    y1, h1 = ssm.scan(_bld(g["u"]), _bld(g["delta"]), g["A"], g["B"], g["C"], g["D"], _bld(g["z"]),
                      g["delta_bias"], bld=True)
    torch.cuda.synchronize()
    assert y1.shape == (2, L, dim)
    assert oracle.rel_err(host64(y1.transpose(1, 2)), y_ref) <= TOL[io]
    assert oracle.rel_err(host64(h1), h_ref) <= TOL[io]
    assert torch.equal(y1.transpose(1, 2), y0) and torch.equal(h1, h0)


def test_scan_bld_split_plan():
    w = synth.scaled(synth.MAMBA_130M, name="bld_split", batch=1, dim=64, seqlen=8192, seed=150)
    x = synth.make_scan_inputs(w)
    g = upload_scan(x)
    y0, h0 = ssm.scan(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"], g["delta_bias"])
    y1, h1 = ssm.scan(_bld(g["u"]), _bld(g["delta"]), g["A"], g["B"], g["C"], g["D"], _bld(g["z"]),
                      g["delta_bias"], bld=True)
    torch.cuda.synchronize()
    assert torch.equal(y1.transpose(1, 2), y0) and torch.equal(h1, h0)


@pytest.mark.parametrize("io,N,dim,L", [("bf16", 16, 96, 130), ("f32", 16, 40, 45),
                                        ("bf16", 4, 70, 300), ("bf16", 32, 33, 40),
                                        ("bf16", 128, 20, 70)])
def test_backward_bld_matches_oracle(io, N, dim, L):
    w = synth.scaled(synth.MAMBA_130M, name="bld_bwd", batch=2, dim=dim, seqlen=L, dstate=N,
                     io=io, seed=160 + N)
    x = synth.make_scan_inputs(w)
    e = synth.make_bwd_inputs(w)
    dy64 = (synth.bf16_to_f32(e["dy"]) if io == "bf16" else e["dy"]).astype(np.float64)
    ref = oracle.scan_bwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                          x["delta_bias"], True, e["init_state"].astype(np.float64), dy64,
                          e["d_final_state"].astype(np.float64))
    g = upload_scan(x)
    kw = dict(init_state=dev_f32(e["init_state"]), d_final_state=dev_f32(e["d_final_state"]),
              want_init_grad=True)
    args = (g["A"], g["B"], g["C"], g["D"])
    out0 = ssm.scan_bwd(g["u"], g["delta"], *args, g["z"], g["delta_bias"], True,
                        dy=dev_io(e["dy"]), **kw)
    bl = {k: _bld(g[k]) for k in ("u", "delta", "z")}
    out1 = ssm.scan_bwd(bl["u"], bl["delta"], *args, bl["z"], g["delta_bias"], True,
                        dy=_bld(dev_io(e["dy"])), bld=True, **kw)
    # the training forward in the same layout, and the backward from its saved states
    _, _, saved = ssm.scan_train(bl["u"], bl["delta"], *args, bl["z"], g["delta_bias"], True,
                                 init_state=kw["init_state"], bld=True)
    out2 = ssm.scan_bwd(bl["u"], bl["delta"], *args, bl["z"], g["delta_bias"], True,
                        dy=_bld(dev_io(e["dy"])), bld=True, saved=saved, **kw)
    torch.cuda.synchronize()
    for k in ("du", "ddelta", "dz"):
        got = out1[k].transpose(1, 2)
        assert oracle.rel_err(host64(got), ref[k]) <= TOL[io], k
        assert torch.equal(got, out0[k]), k
        assert torch.equal(out2[k], out1[k]), k
    for k in ("dA", "dB", "dC", "dD", "dbias", "dinit"):
        assert oracle.rel_err(host64(out1[k]), ref[k]) <= TOL[io], k
        assert torch.equal(out1[k], out0[k]), k


@pytest.mark.parametrize("io,dim,L", [("bf16", 48, 40), ("bf16", 37, 21), ("f32", 12, 33)])
def test_conv1d_bld(io, dim, L):
    batch, K = 3, 4
    n = batch * dim * L
    x = synth.fill(170 + dim, synth.S_U, 0, n, synth.NORMAL, 0.0, 1.0, dtype=io).reshape(batch, dim, L)
    wt = synth.fill(171, synth.S_B, 0, dim * K, synth.NORMAL, 0.0, 0.5).reshape(dim, K)
    bias = synth.fill(172, synth.S_D, 0, dim, synth.NORMAL, 0.0, 0.2)
    st = synth.fill(173, synth.S_Z, 0, batch * dim * (K - 1), synth.NORMAL, 0.0, 1.0,
                    dtype=io).reshape(batch, dim, K - 1)
    st64 = (synth.bf16_to_f32(st) if io == "bf16" else st).astype(np.float64)
    ref, sref = oracle.conv1d(x, wt, bias, st64, silu=True)
    gx = dev_io(x)
    out0, s0 = ssm.conv1d(gx, dev_f32(wt), dev_f32(bias), dev_io(st), True, want_state=True)
    out1, s1 = ssm.conv1d(_bld(gx), dev_f32(wt), dev_f32(bias), dev_io(st), True, want_state=True,
                          bld=True)
    torch.cuda.synchronize()
    assert oracle.rel_err(host64(out1.transpose(1, 2)), ref) <= TOL[io]
    assert torch.equal(out1.transpose(1, 2), out0)
    assert torch.equal(s1, s0) and np.array_equal(host64(s1), sref)
