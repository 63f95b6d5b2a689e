"""GPU parity of the scan on host buffers (``ssm_scan_fwd_host``): the copies to
and from the device happen inside the call, pipelined over units of the input.

Each case runs the oracle on the same inputs (bar: 1e-4 for float32 I/O, 1e-2 for
bfloat16) and compares with the device entry point on device copies of the inputs
(the same kernels on the same per-channel arithmetic; where the smaller units of the
host path let the scan split the sequence, the difference is rounding only, so the
bar there is the oracle's)."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_128_b300 as ssm
import synth
from _gpu import host64, upload_scan

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 1e-2}


def _host(x, pin=True):
    """Generator arrays -> host tensors (bfloat16 bits as torch.bfloat16), page-locked or not."""
    out = {}
    for k, v in x.items():
        if v is None:
            out[k] = None
            continue
        a = np.ascontiguousarray(v)
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if a.dtype == np.uint16 \
            else torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
        out[k] = t.pin_memory() if pin else t.clone()
    return out


def _oracle(x, init=None, euler=False):
    return oracle.scan(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"],
                       True, init, euler=euler)


@pytest.mark.parametrize("io,N,batch,dim,L,pin", [
    ("bf16", 16, 3, 200, 300, True),    # batch < 8: three channel blocks per row, a ragged one
    ("bf16", 16, 9, 64, 130, True),     # one unit per batch row, more units than slots
    ("bf16", 16, 2, 96, 257, False),    # pageable host memory
    ("f32", 16, 2, 40, 70, True),
    ("bf16", 64, 1, 48, 100, True),
    ("bf16", 128, 2, 24, 65, True),
])
def test_scan_host_matches_oracle_and_device_path(io, N, batch, dim, L, pin):
    w = synth.scaled(synth.MAMBA_130M, name="host_scan", batch=batch, dim=dim, seqlen=L, dstate=N,
                     io=io, seed=170 + N + dim + batch)
    x = synth.make_scan_inputs(w)
    y_ref, h_ref = _oracle(x)
    hx = _host(x, pin)
    y1, h1 = ssm.scan_host(hx["u"], hx["delta"], hx["A"], hx["B"], hx["C"], hx["D"], hx["z"],
                           hx["delta_bias"])
    assert not y1.is_cuda and y1.shape == (batch, dim, L)
    assert oracle.rel_err(y1.double().numpy(), y_ref) <= TOL[io]
    assert oracle.rel_err(h1.double().numpy(), h_ref) <= TOL[io]
    g = upload_scan(x)
    y0, h0 = ssm.scan(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"], g["delta_bias"])
    torch.cuda.synchronize()
    assert oracle.rel_err(y1.double().numpy(), host64(y0)) <= TOL[io]
    assert oracle.rel_err(h1.double().numpy(), host64(h0)) <= TOL[io]


def test_scan_host_init_state_euler_and_no_gate():
    w = synth.scaled(synth.MAMBA_130M, name="host_init", batch=2, dim=72, seqlen=90, io="f32",
                     seed=181)
    x = synth.make_scan_inputs(w)
    x["z"] = None
    x["D"] = None
    init = np.random.default_rng(5).standard_normal((2, 72, 16)).astype(np.float32)
    y_ref, h_ref = _oracle(x, init.astype(np.float64), euler=True)
    hx = _host(x)
    y1, h1 = ssm.scan_host(hx["u"], hx["delta"], hx["A"], hx["B"], hx["C"], None, None,
                           hx["delta_bias"], init_state=torch.from_numpy(init).pin_memory(),
                           euler=True)
    assert oracle.rel_err(y1.double().numpy(), y_ref) <= TOL["f32"]
    assert oracle.rel_err(h1.double().numpy(), h_ref) <= TOL["f32"]


def test_scan_host_bld_layout():
    w = synth.scaled(synth.MAMBA_130M, name="host_bld", batch=3, dim=96, seqlen=120, seed=182)
    x = synth.make_scan_inputs(w)
    y_ref, h_ref = _oracle(x)
    hx = _host(x)
    tr = lambda t: t.transpose(1, 2).contiguous().pin_memory()
    y1, h1 = ssm.scan_host(tr(hx["u"]), tr(hx["delta"]), hx["A"], hx["B"], hx["C"], hx["D"],
                           tr(hx["z"]), hx["delta_bias"], bld=True)
    assert y1.shape == (3, 120, 96)
    assert oracle.rel_err(y1.transpose(1, 2).double().numpy(), y_ref) <= TOL["bf16"]
    assert oracle.rel_err(h1.double().numpy(), h_ref) <= TOL["bf16"]


@pytest.mark.parametrize("with_init", [False, True])
def test_scan_host_empty_sequence(with_init):
    """L = 0: no steps, so the final state is the initial one (or zeros)."""
    batch, dim, N = 2, 40, 16
    u = torch.empty((batch, dim, 0), dtype=torch.bfloat16).pin_memory()
    A = -torch.arange(1, N + 1, dtype=torch.float32).repeat(dim, 1).contiguous()
    B = torch.empty((batch, N, 0), dtype=torch.float32)
    init = torch.randn((batch, dim, N), generator=torch.Generator().manual_seed(3)).pin_memory()
    y, h = ssm.scan_host(u, u, A, B, B, init_state=init if with_init else None)
    assert y.shape == (batch, dim, 0)
    assert torch.equal(h, init if with_init else torch.zeros_like(h))


@pytest.mark.slow
def test_scan_host_bench_shape_sampled():
    """The bench's Mamba-130M layer through the host path at full size (8 batch-row
    units through three slots): sampled channels against the oracle, every output
    against the device entry point."""
    w = synth.MAMBA_130M
    x = synth.make_scan_inputs(w)
    hx = _host(x)
    y1, h1 = ssm.scan_host(hx["u"], hx["delta"], hx["A"], hx["B"], hx["C"], hx["D"], hx["z"],
                           hx["delta_bias"])
    rng = np.random.default_rng(7)
    flat = np.sort(rng.choice(w.batch * w.dim, size=96, replace=False))
    bs, ds = flat // w.dim, flat % w.dim
    y_ref, h_ref = oracle.scan_rows(x["u"][bs, ds], x["delta"][bs, ds], x["z"][bs, ds], bs, ds,
                                    x["A"], x["B"], x["C"], x["D"], x["delta_bias"], True)
    assert oracle.rel_err(y1[bs, ds].double().numpy(), y_ref) <= TOL["bf16"]
    assert oracle.rel_err(h1[bs, ds].double().numpy(), h_ref) <= TOL["bf16"]
    g = upload_scan(x)
    y0, h0 = ssm.scan(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"], g["delta_bias"])
    torch.cuda.synchronize()
    assert oracle.rel_err(y1.double().numpy(), host64(y0)) <= TOL["bf16"]
    assert oracle.rel_err(h1.double().numpy(), host64(h0)) <= TOL["bf16"]


def test_scan_host_in_place_carry():
    """final_state may be init_state itself: two calls over the two halves of a
    sequence, the state carried in place in host memory, equal one call over the whole."""
    w = synth.scaled(synth.MAMBA_130M, name="host_carry", batch=2, dim=64, seqlen=160, seed=183)
    x = synth.make_scan_inputs(w)
    y_ref, h_ref = _oracle(x)
    hx = _host(x)
    state = torch.zeros((2, 64, 16), dtype=torch.float32).pin_memory()
    ws_bytes = ssm.ssm_scan_fwd_host_workspace_bytes(2, 64, 80, 16, ssm.SSM_BF16, 1)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    ys = []
    for t0 in (0, 80):
        part = {k: hx[k][:, :, t0:t0 + 80].contiguous().pin_memory() for k in ("u", "delta", "z", "B", "C")}
        y = torch.empty((2, 64, 80), dtype=torch.bfloat16).pin_memory()
        ssm.ssm_scan_fwd_host(part["u"], part["delta"], hx["delta_bias"], hx["A"], part["B"], part["C"],
                              hx["D"], part["z"], 1, y, state, state, ws, ws_bytes)
        torch.cuda.current_stream().synchronize()
        ys.append(y)
    y_all = torch.cat(ys, dim=2)
    assert oracle.rel_err(y_all.double().numpy(), y_ref) <= TOL["bf16"]
    assert oracle.rel_err(state.double().numpy(), h_ref) <= TOL["bf16"]
