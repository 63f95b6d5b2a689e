"""GPU parity of the scan on strided views (ssm_scan_fwd_strided).

The summary page's section 4a shape table feeds the SSM from one input projection
Linear(2ED) whose output is split into the SSM input and the gate; with strided
views, u and z are the two halves of that output without a copy.  Each case
builds such views (time-major (batch, 2 dim, L) and channel-major (batch, L, 2 dim)
projections, y written into a strided view of a larger buffer) and requires:

* the oracle's result on the same values within the workload bar (1e-2 for
  bfloat16 I/O, 1e-4 for float32);
* bit-equality with ssm_scan_fwd_ex on contiguous copies of the views when both
  take the same kernel (the strides change only where elements are read and
  written);
* y's buffer untouched outside the view."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_128_b300 as ssm
import synth
from _gpu import host64, upload_scan

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 1e-2}


def _inputs(batch, dim, L, N=16, io="bf16", seed=300):
    w = synth.scaled(synth.MAMBA_130M, batch=batch, dim=dim, seqlen=L, dstate=N, io=io, seed=seed)
    x = synth.make_scan_inputs(w)
    return w, x, upload_scan(x)


def _contiguous_run(g, w):
    y = torch.empty_like(g["u"])
    h = torch.empty((w.batch, w.dim, w.dstate), dtype=torch.float32, device="cuda")
    ssm.ssm_scan_fwd_ex(g["u"], g["delta"], g["delta_bias"], g["A"], g["B"], g["C"], g["D"],
                        g["z"], True, y, h)
    return y, h


def _strided_run(g, w, u, z, delta, y):
    h = torch.empty((w.batch, w.dim, w.dstate), dtype=torch.float32, device="cuda")
    ssm.ssm_scan_fwd_strided(u, delta, g["delta_bias"], g["A"], g["B"], g["C"], g["D"], z, True,
                             y, h)
    return h


@pytest.mark.parametrize("io,N,dim,L", [("bf16", 16, 96, 256), ("bf16", 16, 40, 200),
                                        ("f32", 16, 48, 64), ("bf16", 64, 32, 96)])
def test_halves_of_a_time_major_projection(io, N, dim, L):
    """u and z are xz[:, :dim] and xz[:, dim:] of one (batch, 2 dim, L) projection."""
    w, x, g = _inputs(2, dim, L, N, io, seed=310 + dim)
    xz = torch.cat([g["u"], g["z"]], dim=1)          # (batch, 2 dim, L)
    u, z = xz[:, :dim], xz[:, dim:]
    assert not u.is_contiguous()
    ybuf = torch.full((w.batch, dim + 8, L), float("nan"), dtype=g["u"].dtype, device="cuda")
    y = ybuf[:, 4:4 + dim]                            # a view with a channel offset
    h = _strided_run(g, w, u, z, g["delta"], y)
    y0, h0 = _contiguous_run(g, w)
    torch.cuda.synchronize()
    assert torch.equal(y, y0) and torch.equal(h, h0)
    assert torch.isnan(ybuf[:, :4].float()).all() and torch.isnan(ybuf[:, 4 + dim:].float()).all()
    y_o, h_o = oracle.scan(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                           x["delta_bias"])
    assert oracle.rel_err(host64(y), y_o) <= TOL[io]
    assert oracle.rel_err(host64(h), h_o) <= TOL[io]


@pytest.mark.parametrize("dim,L", [(96, 256), (64, 8192)])
def test_halves_of_a_channel_major_projection(dim, L):
    """Algorithm 2's (B, L, D): u, z are xz[..., :dim], xz[..., dim:] of a (batch, L, 2 dim)
    projection (row stride 2 dim), delta is (batch, L, dim), y a (batch, L, dim) buffer; as
    (batch, dim, L) views their channel stride is 1.  The longer case splits the sequence."""
    w, x, g = _inputs(1 if L > 1000 else 2, dim, L, seed=320 + dim)
    xz = torch.cat([g["u"], g["z"]], dim=1).transpose(1, 2).contiguous()   # (batch, L, 2 dim)
    u = xz[..., :dim].transpose(1, 2)
    z = xz[..., dim:].transpose(1, 2)
    delta = g["delta"].transpose(1, 2).contiguous().transpose(1, 2)
    ybld = torch.empty((w.batch, L, dim), dtype=g["u"].dtype, device="cuda")
    y = ybld.transpose(1, 2)
    assert u.stride() == (L * 2 * dim, 1, 2 * dim)
    h = _strided_run(g, w, u, z, delta, y)
    y0, h0 = _contiguous_run(g, w)
    torch.cuda.synchronize()
    assert torch.equal(y, y0) and torch.equal(h, h0)
    y_o, h_o = oracle.scan(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                           x["delta_bias"])
    assert oracle.rel_err(host64(y), y_o) <= 1e-2


def test_strides_that_are_not_16_byte_multiples():
    """Row strides of an odd number of elements take the element-wise path; results still
    match the oracle."""
    dim, L = 24, 100
    w, x, g = _inputs(2, dim, L, seed=330)
    big = torch.empty((w.batch, dim, L + 3), dtype=g["u"].dtype, device="cuda")
    big[..., :L] = g["u"]
    u = big[..., :L]                                  # time stride 1, channel stride L + 3
    assert u.stride(1) == L + 3
    y = torch.empty_like(g["u"])
    h = _strided_run(g, w, u, g["z"], g["delta"], y)
    torch.cuda.synchronize()
    y_o, h_o = oracle.scan(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                           x["delta_bias"])
    assert oracle.rel_err(host64(y), y_o) <= 1e-2
    assert oracle.rel_err(host64(h), h_o) <= 1e-2
