"""GPU parity of the two-warp-block scan kernel on small sizes.

The forward scan has two kernels: the block kernel (blocks of 32 channels that
share their conversion; every dstate and dtype) and the two-warp-block kernel
(blocks of 64 threads for 16 channels, each warp holding two of a channel's
four state groups; N = 16, bf16, zero-order hold, views TMA can stage), chosen
by size: the second when there are enough of its warps to give every SM 16.  The
test mode's kernel choice runs it here on sizes that span several blocks, chunks
and a ragged tail, against the fp64 oracle (bar 1e-2 for bf16 I/O), with the
cases its own code paths handle: steps past the sequence, channels past dim, no
gate / D / bias / softplus, a zero A (its precise per-thread loop, also through
channel-major and strided views), an initial state and a carry over two calls, a
sequence split across blocks (both passes), the channel-major layout and strided
halves of one projection (bit-equal to the time-major contiguous run), and the
training forward's saved states (the backward from them equals the backward that
recomputes them)."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_128_b300 as ssm
import synth
from _gpu import dev_f32, dev_io, host64, upload_scan

pytestmark = pytest.mark.gpu

TOL = 1e-2


@pytest.fixture(autouse=True)
def pair_kernel():
    ssm.ssm_set_test_mode(True, 1_000_000, scan_kernel=ssm.SCAN_KERNEL_PAIR)
    yield
    ssm.ssm_set_test_mode(False)


def _run(w, x, **kw):
    g = upload_scan(x)
    y, h = ssm.scan(g["u"], g["delta"], g["A"], g["B"], g["C"], g.get("D"), g.get("z"),
                    g.get("delta_bias"), **kw)
    torch.cuda.synchronize()
    return g, y, h


def _oracle(x, **kw):
    return oracle.scan(x["u"], x["delta"], x["A"], x["B"], x["C"], x.get("D"), x.get("z"),
                       x.get("delta_bias"), **kw)


@pytest.mark.parametrize("dim,L", [(8, 16), (40, 200), (72, 1000), (100, 64), (64, 1032)])
def test_ragged_sizes(dim, L):
    w = synth.scaled(synth.MAMBA_130M, batch=2, dim=dim, seqlen=L, seed=500 + dim + L)
    x = synth.make_scan_inputs(w)
    _, y, h = _run(w, x)
    y_o, h_o = _oracle(x)
    assert oracle.rel_err(host64(y), y_o) <= TOL
    assert oracle.rel_err(host64(h), h_o) <= TOL


@pytest.mark.parametrize("drop", ["z", "D", "delta_bias", "softplus"])
def test_optional_arguments(drop):
    w = synth.scaled(synth.MAMBA_130M, batch=2, dim=48, seqlen=256, seed=520)
    x = synth.make_scan_inputs(w)
    sp = drop != "softplus"
    if drop != "softplus":
        x[drop] = None
    else:  # Δ = delta as given: small positive steps, no bias
        x["delta"] = synth.f32_to_bf16(np.abs(synth.bf16_to_f32(x["delta"])) * 0.05)
        x["delta_bias"] = None
    _, y, h = _run(w, x, delta_softplus=sp)
    y_o, h_o = _oracle(x, delta_softplus=sp)
    assert oracle.rel_err(host64(y), y_o) <= TOL
    assert oracle.rel_err(host64(h), h_o) <= TOL


def test_zero_A_takes_the_precise_path():
    w = synth.scaled(synth.MAMBA_130M, batch=2, dim=32, seqlen=96, seed=530)
    x = synth.make_scan_inputs(w)
    x["A"] = x["A"].copy()
    x["A"][3, 5] = 0.0      # block 0's channels take the precise loop, the others the fast path
    _, y, h = _run(w, x)
    y_o, h_o = _oracle(x)
    assert oracle.rel_err(host64(y), y_o) <= TOL
    assert oracle.rel_err(host64(h), h_o) <= TOL


def test_initial_state_and_carry_over_two_calls():
    w = synth.scaled(synth.MAMBA_130M, batch=2, dim=40, seqlen=512, seed=540)
    x = synth.make_scan_inputs(w)
    e = synth.make_bwd_inputs(w)
    g = upload_scan(x)
    h0 = dev_f32(e["init_state"])
    y, h = ssm.scan(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"], g["delta_bias"],
                    init_state=h0)
    half = 256
    cut = lambda t, a, b: t[..., a:b].contiguous()
    y1, h1 = ssm.scan(cut(g["u"], 0, half), cut(g["delta"], 0, half), g["A"], cut(g["B"], 0, half),
                      cut(g["C"], 0, half), g["D"], cut(g["z"], 0, half), g["delta_bias"], init_state=h0)
    y2, h2 = ssm.scan(cut(g["u"], half, None), cut(g["delta"], half, None), g["A"],
                      cut(g["B"], half, None), cut(g["C"], half, None), g["D"], cut(g["z"], half, None),
                      g["delta_bias"], init_state=h1)
    torch.cuda.synchronize()
    y_o, h_o = _oracle(x, init_state=e["init_state"].astype(np.float64))
    assert oracle.rel_err(host64(y), y_o) <= TOL
    assert oracle.rel_err(host64(h), h_o) <= TOL
    assert torch.equal(torch.cat([y1, y2], dim=2), y) and torch.equal(h2, h)


def test_split_sequence_both_passes():
    w = synth.scaled(synth.MAMBA_130M, batch=1, dim=24, seqlen=8192 + 24, seed=550)
    assert ssm.ssm_scan_workspace_bytes(w.batch, w.dim, w.seqlen, 16, ssm.SSM_BF16) > \
        ssm.SCAN_STATUS_BYTES   # the plan splits the sequence
    x = synth.make_scan_inputs(w)
    _, y, h = _run(w, x)
    y_o, h_o = _oracle(x)
    assert oracle.rel_err(host64(y), y_o) <= TOL
    assert oracle.rel_err(host64(h), h_o) <= TOL


def test_channel_major_and_strided_views_are_bit_equal():
    w = synth.scaled(synth.MAMBA_130M, batch=2, dim=64, seqlen=320, seed=560)
    x = synth.make_scan_inputs(w)
    g, y0, h0 = _run(w, x)
    t = {k: g[k].transpose(1, 2).contiguous() for k in ("u", "delta", "z")}
    y1, h1 = ssm.scan(t["u"], t["delta"], g["A"], g["B"], g["C"], g["D"], t["z"], g["delta_bias"],
                      bld=True)
    xz = torch.cat([g["u"], g["z"]], dim=1)
    y2 = torch.empty_like(y0)
    h2 = torch.empty_like(h0)
    ssm.ssm_scan_fwd_strided(xz[:, :64], g["delta"], g["delta_bias"], g["A"], g["B"], g["C"],
                             g["D"], xz[:, 64:], True, y2, h2)
    torch.cuda.synchronize()
    assert torch.equal(y1.transpose(1, 2), y0) and torch.equal(h1, h0)
    assert torch.equal(y2, y0) and torch.equal(h2, h0)
    y_o, _ = _oracle(x)
    assert oracle.rel_err(host64(y0), y_o) <= TOL


def test_zero_A_channel_major_and_strided_views_are_bit_equal():
    # the precise loop reads and writes through the tensors' strides
    w = synth.scaled(synth.MAMBA_130M, batch=2, dim=48, seqlen=200, seed=565)
    x = synth.make_scan_inputs(w)
    x["A"] = x["A"].copy()
    x["A"][5, 3] = 0.0
    x["A"][40, 0] = 0.0
    g, y0, h0 = _run(w, x)
    t = {k: g[k].transpose(1, 2).contiguous() for k in ("u", "delta", "z")}
    y1, h1 = ssm.scan(t["u"], t["delta"], g["A"], g["B"], g["C"], g["D"], t["z"], g["delta_bias"],
                      bld=True)
    xz = torch.cat([g["u"], g["z"]], dim=1)
    y2 = torch.empty_like(y0)
    h2 = torch.empty_like(h0)
    ssm.ssm_scan_fwd_strided(xz[:, :48], g["delta"], g["delta_bias"], g["A"], g["B"], g["C"],
                             g["D"], xz[:, 48:], True, y2, h2)
    torch.cuda.synchronize()
    assert torch.equal(y1.transpose(1, 2), y0) and torch.equal(h1, h0)
    assert torch.equal(y2, y0) and torch.equal(h2, h0)
    y_o, h_o = _oracle(x)
    assert oracle.rel_err(host64(y0), y_o) <= TOL
    assert oracle.rel_err(host64(h0), h_o) <= TOL


def test_training_forward_saves_the_backward_states():
    w = synth.scaled(synth.MAMBA_130M, batch=2, dim=32, seqlen=400, seed=570)
    x = synth.make_scan_inputs(w)
    e = synth.make_bwd_inputs(w, init_state=False, d_final_state=False)
    g = upload_scan(x)
    dy = dev_io(e["dy"])
    y_t, h_t, saved = ssm.scan_train(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"],
                                     g["delta_bias"])
    y, h = ssm.scan(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"], g["delta_bias"])
    a = ssm.scan_bwd(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"], g["delta_bias"],
                     dy=dy, saved=saved)
    b = ssm.scan_bwd(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"], g["delta_bias"],
                     dy=dy)
    torch.cuda.synchronize()
    assert torch.equal(y_t, y) and torch.equal(h_t, h)
    for k in ("du", "ddelta", "dz", "dA", "dB", "dC"):
        assert oracle.rel_err(host64(a[k]), host64(b[k])) <= 1e-5, k
