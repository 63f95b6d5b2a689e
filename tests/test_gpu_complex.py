"""GPU parity of ssm_scan_fwd_complex (the scan with a complex diagonal A, complex B
and C) against oracle.scan_complex (complex128, pinned in test_oracle_complex_pins).

Bar: max|gpu - oracle| / max|oracle| <= 1e-4 for float32 I/O and 1e-2 for bfloat16
(the real scan's bars), for y and the final state.  Sizes span several chunks and
channel blocks with ragged tails."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_128_b300 as ssm
import synth
from _gpu import dev_f32, dev_io, host64

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 1e-2}


def _inputs(io, batch, dim, L, N, seed, zero_a=False):
    w = synth.scaled(synth.MAMBA_130M, batch=batch, dim=dim, seqlen=L, dstate=N, io=io, seed=seed)
    x = synth.make_scan_inputs(w)
    rng = np.random.default_rng(seed)
    # A: real part the recipe's -(n + 1) scaled down, imaginary part a spread of frequencies
    A = (x["A"] * 0.5 + 1j * np.pi * rng.uniform(-1.0, 1.0, x["A"].shape)).astype(np.complex64)
    if zero_a:
        A[1, ::2] = 0
    B = (x["B"] + 1j * rng.standard_normal(x["B"].shape)).astype(np.complex64)
    C = (x["C"] + 1j * rng.standard_normal(x["C"].shape)).astype(np.complex64)
    h0 = (rng.standard_normal((batch, dim, N)) + 1j * rng.standard_normal((batch, dim, N))
          ).astype(np.complex64)
    return x, A, B, C, h0


def _dev_c(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("io,N,dim,L", [("bf16", 16, 70, 300), ("f32", 16, 40, 77),
                                        ("f32", 4, 33, 129), ("bf16", 64, 20, 50),
                                        ("f32", 1, 130, 40), ("f32", 2, 65, 33),
                                        ("f32", 32, 40, 70), ("bf16", 8, 64, 64)])
def test_complex_scan_matches_oracle(io, N, dim, L):
    x, A, B, C, h0 = _inputs(io, 2, dim, L, N, seed=600 + N + dim)
    y_ref, h_ref = oracle.scan_complex(x["u"], x["delta"], A, B, C, x["D"], x["z"],
                                       x["delta_bias"], True, h0)
    y, h = ssm.scan_complex(dev_io(x["u"]), dev_io(x["delta"]), _dev_c(A), _dev_c(B), _dev_c(C),
                            dev_f32(x["D"]), dev_io(x["z"]), dev_f32(x["delta_bias"]), True,
                            _dev_c(h0))
    torch.cuda.synchronize()
    assert oracle.rel_err(host64(y), y_ref) <= TOL[io]
    hc = h.cpu().numpy()
    assert oracle.rel_err(np.concatenate([hc.real, hc.imag]), np.concatenate([h_ref.real, h_ref.imag])) <= TOL[io]


@pytest.mark.parametrize("case", ["euler", "zero_a", "no_optionals", "no_softplus", "in_place"])
def test_complex_scan_variants(case):
    x, A, B, C, h0 = _inputs("f32", 2, 40, 90, 16, seed=650, zero_a=case == "zero_a")
    kw = dict(D=x["D"], z=x["z"], bias=x["delta_bias"], softplus=True, h0=h0, euler=False)
    if case == "euler":
        kw["euler"] = True
    if case == "no_optionals":
        kw.update(D=None, z=None, bias=None, h0=None)
    if case == "no_softplus":
        d = (np.abs(x["delta"]) * 0.2).astype(np.float32)
        x["delta"] = d
        kw.update(softplus=False, bias=np.full_like(x["delta_bias"], 0.01))
    y_ref, h_ref = oracle.scan_complex(x["u"], x["delta"], A, B, C, kw["D"], kw["z"], kw["bias"],
                                       kw["softplus"], kw["h0"], euler=kw["euler"])
    args = (dev_io(x["u"]), dev_io(x["delta"]), _dev_c(A), _dev_c(B), _dev_c(C), dev_f32(kw["D"]),
            dev_io(kw["z"]), dev_f32(kw["bias"]), kw["softplus"])
    if case == "in_place":
        # final_state == init_state: the state carried in place
        st = _dev_c(h0)
        y = torch.empty_like(args[0])
        ssm.ssm_scan_fwd_complex(args[0], args[1], args[7], args[2], args[3], args[4], args[5],
                                 args[6], ssm._flags(True), y, st, st)
        h = st
    else:
        y, h = ssm.scan_complex(*args, init_state=_dev_c(kw["h0"]), euler=kw["euler"])
    torch.cuda.synchronize()
    assert oracle.rel_err(host64(y), y_ref) <= TOL["f32"]
    hc = h.cpu().numpy()
    assert oracle.rel_err(np.concatenate([hc.real, hc.imag]),
                          np.concatenate([h_ref.real, h_ref.imag])) <= TOL["f32"]


def test_real_A_agrees_with_the_real_scan():
    """With zero imaginary parts the complex scan computes the real scan (its own
    precise-flavour arithmetic; the real kernel's fp32 path is pinned separately)."""
    w = synth.scaled(synth.MAMBA_130M, batch=2, dim=48, seqlen=200, dstate=16, io="f32", seed=660)
    x = synth.make_scan_inputs(w)
    y_r, h_r = ssm.scan(dev_io(x["u"]), dev_io(x["delta"]), dev_f32(x["A"]), dev_f32(x["B"]),
                        dev_f32(x["C"]), dev_f32(x["D"]), dev_io(x["z"]), dev_f32(x["delta_bias"]))
    y_c, h_c = ssm.scan_complex(dev_io(x["u"]), dev_io(x["delta"]),
                                _dev_c(x["A"].astype(np.complex64)),
                                _dev_c(x["B"].astype(np.complex64)),
                                _dev_c(x["C"].astype(np.complex64)), dev_f32(x["D"]),
                                dev_io(x["z"]), dev_f32(x["delta_bias"]))
    torch.cuda.synchronize()
    assert oracle.rel_err(host64(y_c), host64(y_r)) <= 1e-5
    assert oracle.rel_err(h_c.real.cpu().numpy(), host64(h_r)) <= 1e-5
    assert h_c.imag.abs().max().item() == 0.0
