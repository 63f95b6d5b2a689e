"""GPU parity of the scan's front end (causal depthwise conv1d + SiLU, and its
one-token form on a rolling state) against the fp64 oracle.

Bar: max|gpu - ref| / max|ref| <= 1e-4 for float32 I/O and <= 1e-2 for bfloat16
I/O (the outputs are rounded to the I/O type); states are copies of inputs and
must match exactly."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_128_b300 as ssm
import synth
from _gpu import dev_f32, dev_io, host64

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 1e-2}


def _inputs(io, batch, dim, L, K, seed, state=True):
    n = batch * dim * L
    x = synth.fill(seed, synth.S_U, 0, n, synth.NORMAL, 0.0, 1.0, dtype=io).reshape(batch, dim, L)
    wt = synth.fill(seed, synth.S_B, 0, dim * K, synth.NORMAL, 0.0, 0.5).reshape(dim, K)
    bias = synth.fill(seed, synth.S_D, 0, dim, synth.NORMAL, 0.0, 0.2)
    st = None
    if state and K > 1:
        st = synth.fill(seed, synth.S_Z, 0, batch * dim * (K - 1), synth.NORMAL, 0.0, 1.0,
                        dtype=io).reshape(batch, dim, K - 1)
    return x, wt, bias, st


def _as64(a):
    return None if a is None else (synth.bf16_to_f32(a).astype(np.float64) if a.dtype == np.uint16
                                   else a.astype(np.float64))


@pytest.mark.parametrize("io", ["bf16", "f32"])
@pytest.mark.parametrize("K", [1, 2, 3, 4])
@pytest.mark.parametrize("L", [64, 67, 5])
def test_conv1d_matches_oracle(io, K, L):
    x, wt, bias, st = _inputs(io, 3, 37, L, K, seed=70 + K + L)
    ref, sref = oracle.conv1d(x, wt, bias, _as64(st), silu=True)
    out, snew = ssm.conv1d(dev_io(x), dev_f32(wt), dev_f32(bias), dev_io(st), True,
                           want_state=True)
    torch.cuda.synchronize()
    assert oracle.rel_err(host64(out), ref) <= TOL[io]
    if K > 1:
        assert np.array_equal(host64(snew), sref)


def test_conv1d_without_silu_bias_or_state():
    x, wt, _, _ = _inputs("f32", 2, 16, 40, 4, seed=80, state=False)
    ref, _ = oracle.conv1d(x, wt, None, None, silu=False)
    out = ssm.conv1d(dev_io(x), dev_f32(wt), None, None, False)
    torch.cuda.synchronize()
    assert oracle.rel_err(host64(out), ref) <= 1e-6


def test_chunked_in_place_state_equals_one_shot():
    x, wt, bias, st = _inputs("bf16", 2, 24, 96, 4, seed=81)
    gx, gw, gb = dev_io(x), dev_f32(wt), dev_f32(bias)
    whole, s_whole = ssm.conv1d(gx, gw, gb, dev_io(st), True, want_state=True)
    state = dev_io(st).clone()
    parts = []
    for a, b in ((0, 40), (40, 42), (42, 96)):
        xc = gx[..., a:b].contiguous()
        out = torch.empty_like(xc)
        ssm.ssm_conv1d_fwd(xc, gw, gb, state, True, out, state)  # state updated in place
        parts.append(out)
    torch.cuda.synchronize()
    assert torch.equal(torch.cat(parts, -1), whole)
    assert torch.equal(state, s_whole)


@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_decode_update_steps_equal_sequence(io):
    """T one-token updates on the rolling state give the sequence pass's outputs."""
    K, L = 4, 12
    x, wt, bias, st = _inputs(io, 4, 40, L, K, seed=82)
    ref, sref = oracle.conv1d(x, wt, bias, _as64(st), silu=True)
    state = dev_io(st).clone()
    gx, gw, gb = dev_io(x), dev_f32(wt), dev_f32(bias)
    outs = []
    for t in range(L):
        xt = gx[..., t].contiguous()
        o = torch.empty_like(xt)
        ssm.ssm_conv1d_update(state, xt, gw, gb, True, o)
        outs.append(o)
    torch.cuda.synchronize()
    got = torch.stack(outs, -1)
    assert oracle.rel_err(host64(got), ref) <= TOL[io]
    assert np.array_equal(host64(state), sref)


def test_conv1d_feeds_the_scan():
    """u = silu(conv(x)) computed on the GPU and scanned equals the oracle's
    composition of the two steps (the pages' Conv1d -> SiLU -> SSM order)."""
    w = synth.scaled(synth.MAMBA_130M, name="conv_scan", batch=2, dim=64, seqlen=160, seed=83)
    xs = synth.make_scan_inputs(w)
    x, wt, bias, _ = _inputs("bf16", 2, 64, 160, 4, seed=84, state=False)
    u_ref, _ = oracle.conv1d(x, wt, bias, None, silu=True)
    u_gpu = ssm.conv1d(dev_io(x), dev_f32(wt), dev_f32(bias))
    torch.cuda.synchronize()
    # the scan's input is the GPU's bf16 u; the oracle scans the same bits
    u_bits = u_gpu.view(torch.int16).cpu().numpy().view(np.uint16)
    assert oracle.rel_err(synth.bf16_to_f32(u_bits), u_ref) <= 1e-2
    y_ref, _ = oracle.scan(u_bits, xs["delta"], xs["A"], xs["B"], xs["C"], xs["D"], xs["z"],
                           xs["delta_bias"])
    y, _ = ssm.scan(u_gpu, dev_io(xs["delta"]), dev_f32(xs["A"]), dev_f32(xs["B"]),
                    dev_f32(xs["C"]), dev_f32(xs["D"]), dev_io(xs["z"]), dev_f32(xs["delta_bias"]))
    torch.cuda.synchronize()
    assert oracle.rel_err(host64(y), y_ref) <= 1e-2


# ---------------------------------------------------------------------------
# the backward (ssm_conv1d_bwd) against oracle.conv1d_bwd
# ---------------------------------------------------------------------------

def _dout(io, shape, seed):
    n = int(np.prod(shape))
    return synth.fill(seed, synth.S_DY, 0, n, synth.NORMAL, 0.0, 1.0, dtype=io).reshape(shape)


def _check_bwd(io, batch, dim, L, K, seed, silu=True, state=True, bias=True, bld=False):
    x, wt, b, st = _inputs(io, batch, dim, L, K, seed, state)
    dout = _dout(io, (batch, dim, L), seed + 1)
    ref = oracle.conv1d_bwd(x, wt, b if bias else None, _as64(st), silu, dout)
    tr = (lambda t: t.transpose(1, 2).contiguous()) if bld else (lambda t: t)
    out = ssm.conv1d_bwd(tr(dev_io(x)), dev_f32(wt), tr(dev_io(dout)), dev_f32(b) if bias else None,
                         dev_io(st) if st is not None else None, silu=silu, bld=bld)
    torch.cuda.synchronize()
    got_dx = host64(out["dx"].transpose(1, 2) if bld else out["dx"])
    assert oracle.rel_err(got_dx, ref["dx"]) <= TOL[io]
    assert oracle.rel_err(host64(out["dweight"]), ref["dweight"]) <= TOL[io] / 10
    assert oracle.rel_err(host64(out["dbias"]), ref["dbias"]) <= TOL[io] / 10
    if K > 1:
        assert oracle.rel_err(host64(out["dstate"]), ref["dstate"]) <= TOL[io] / 10
    return out


@pytest.mark.parametrize("io", ["bf16", "f32"])
@pytest.mark.parametrize("K", [1, 2, 3, 4])
@pytest.mark.parametrize("L", [64, 67, 5])
def test_conv1d_bwd_matches_oracle(io, K, L):
    _check_bwd(io, 3, 37, L, K, seed=70 + K + L)


@pytest.mark.parametrize("case", ["no_silu", "no_state_no_bias", "long_rows", "bld", "bld_ragged",
                                  "f32_long_rows", "one_unit_and_a_bit", "long_rows_no_state"])
def test_conv1d_bwd_variants(case):
    kw = dict(no_silu=dict(silu=False), no_state_no_bias=dict(state=False, bias=False),
              long_rows=dict(L=5000), bld=dict(bld=True), bld_ragged=dict(bld=True, L=29),
              f32_long_rows=dict(io="f32", L=4100), one_unit_and_a_bit=dict(L=2056, K=3),
              long_rows_no_state=dict(L=4104, state=False))[case]
    args = dict(io="bf16", batch=2, dim=24, L=136, K=4, seed=90)
    args.update(kw)
    _check_bwd(**args)


def test_conv1d_bwd_repeats_bit_for_bit():
    """The sums over the batch are added in a fixed order."""
    a = _check_bwd("bf16", 4, 16, 100, 4, seed=95)
    b = _check_bwd("bf16", 4, 16, 100, 4, seed=95)
    for k in ("dx", "dweight", "dbias", "dstate"):
        assert torch.equal(a[k], b[k]), k


@pytest.mark.parametrize("io,L", [("bf16", 5000), ("f32", 2052)])
def test_conv1d_bwd_staged_rows_equal_the_elementwise_kernel(io, L):
    """Rows of whole 16-byte pieces in (batch, dim, L) go through the kernel that
    stages them in shared memory; the (batch, L, dim) layout takes the element-wise
    kernel.  Same arithmetic and order of sums: equal bit for bit."""
    x, wt, b, st = _inputs(io, 2, 24, L, 4, 97, True)
    dout = _dout(io, (2, 24, L), 98)
    tr = lambda t: t.transpose(1, 2).contiguous()
    args = (dev_f32(wt),)
    a = ssm.conv1d_bwd(dev_io(x), *args, dev_io(dout), dev_f32(b), dev_io(st))
    c = ssm.conv1d_bwd(tr(dev_io(x)), *args, tr(dev_io(dout)), dev_f32(b), dev_io(st), bld=True)
    torch.cuda.synchronize()
    assert torch.equal(a["dx"], c["dx"].transpose(1, 2))
    for k in ("dweight", "dbias", "dstate"):
        assert torch.equal(a[k], c[k]), k
