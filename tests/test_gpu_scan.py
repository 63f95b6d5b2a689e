"""GPU parity of ssm_scan_fwd / ssm_scan_fwd_ex against the fp64 oracle.

Bar: max|y_gpu - y_ref| / max|y_ref| <= 1e-4 for float32 I/O and <= 1e-2 for
bfloat16 I/O, the same bound for final_state, on identical seeded inputs."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_128_b300 as ssm
import synth
from _gpu import dev_f32, dev_io, host64, upload_scan

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 1e-2}


def _oracle(x, z=True, D=True, bias=True, softplus=True, init=None):
    return oracle.scan(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"] if D else None,
                       x["z"] if z else None, x["delta_bias"] if bias else None, softplus,
                       init_state=init)


def _gpu(x, z=True, D=True, bias=True, softplus=True, init=None, split=True, short=False):
    g = upload_scan(x)
    h0 = dev_f32(init) if init is not None else None
    if short:
        y = torch.empty_like(g["u"])
        h = torch.empty(g["u"].shape[:2] + (g["A"].shape[1],), dtype=torch.float32, device="cuda")
        ssm.ssm_scan_fwd(g["u"], g["delta"], g["delta_bias"] if bias else None, g["A"], g["B"],
                         g["C"], g["D"] if D else None, g["z"] if z else None, softplus, y, h)
    else:
        y, h = ssm.scan(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"] if D else None,
                        g["z"] if z else None, g["delta_bias"] if bias else None, softplus,
                        init_state=h0, split=split)
    torch.cuda.synchronize()
    return host64(y), host64(h)


def _check(w, x, tol=None, **kw):
    tol = TOL[w.io] if tol is None else tol
    y_ref, h_ref = _oracle(x, **{k: v for k, v in kw.items() if k in ("z", "D", "bias", "softplus", "init")})
    y, h = _gpu(x, **kw)
    ey, eh = oracle.rel_err(y, y_ref), oracle.rel_err(h, h_ref)
    assert np.isfinite(y).all() and np.isfinite(h).all()
    assert ey <= tol, ("y", ey)
    assert eh <= tol, ("final_state", eh)
    return ey, eh


def test_tiny_fp32_workload():
    """batch 1, d_inner 16, L 256, N 4, fp32 I/O, seed 0 (the tiny S6 workload)."""
    ey, eh = _check(synth.TINY, synth.make_scan_inputs(synth.TINY))
    assert ey < 1e-5 and eh < 1e-5


def test_tiny_fp32_short_entry_point():
    _check(synth.TINY, synth.make_scan_inputs(synth.TINY), short=True)


@pytest.mark.parametrize("N", [1, 2, 4, 8, 16, 32, 64, 128])
@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_state_sizes(N, io):
    w = synth.scaled(synth.MAMBA_130M, batch=2, dim=72, seqlen=200, dstate=N, io=io, seed=30 + N)
    _check(w, synth.make_scan_inputs(w))


@pytest.mark.parametrize("L", [1, 7, 8, 63, 64, 65, 129, 1000, 1031])
def test_ragged_lengths(L):
    """L not a multiple of the 16-byte vector or of the chunk: element-wise path and tails."""
    w = synth.scaled(synth.MAMBA_130M, batch=2, dim=40, seqlen=L, seed=100 + L)
    _check(w, synth.make_scan_inputs(w))


@pytest.mark.parametrize("opts", [dict(z=False), dict(D=False), dict(bias=False),
                                  dict(softplus=False, bias=False), dict(z=False, D=False)])
def test_optional_arguments(opts):
    w = synth.scaled(synth.MAMBA_130M, batch=2, dim=64, seqlen=256, seed=7)
    x = synth.make_scan_inputs(w)
    if opts.get("softplus") is False:
        # Δ used as given must be a positive step size: take |Δ_raw| * 0.05
        dl = synth.bf16_to_f32(x["delta"])
        x["delta"] = synth.f32_to_bf16(np.abs(dl) * 0.05 + 1e-3)
    _check(w, x, **opts)


def test_init_state_and_chunk_carry():
    """final_state of a call over [0, L1) as init_state of a call over [L1, L) equals one
    call over [0, L) (the chunk-carried state)."""
    w = synth.scaled(synth.MAMBA_130M, batch=2, dim=96, seqlen=640, seed=9)
    x = synth.make_scan_inputs(w)
    g = upload_scan(x)
    y_full, h_full = ssm.scan(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"],
                              g["delta_bias"])
    parts, h = [], None
    for t0, t1 in ((0, 192), (192, 200), (200, 640)):
        sl = lambda k: g[k][:, :, t0:t1].contiguous()
        yk, h = ssm.scan(sl("u"), sl("delta"), g["A"], sl("B"), sl("C"), g["D"], sl("z"),
                         g["delta_bias"], init_state=h)
        parts.append(yk)
    y_cat = torch.cat(parts, dim=2)
    torch.cuda.synchronize()
    y_ref, h_ref = _oracle(x)
    assert oracle.rel_err(host64(y_cat), y_ref) <= 1e-2
    assert oracle.rel_err(host64(h), h_ref) <= 1e-2
    # the carried and one-shot GPU results agree to bf16 rounding of y
    assert oracle.rel_err(host64(y_cat), host64(y_full)) <= 1e-2
    assert oracle.rel_err(host64(h), host64(h_full)) <= 1e-5


def test_in_place_carry():
    """init_state and final_state may be the same buffer."""
    w = synth.scaled(synth.MAMBA_130M, batch=1, dim=64, seqlen=256, seed=12)
    x = synth.make_scan_inputs(w)
    g = upload_scan(x)
    rng = np.random.default_rng(0)
    h0 = rng.standard_normal((1, 64, 16)).astype(np.float32)
    h = dev_f32(h0)
    y = torch.empty_like(g["u"])
    ssm.ssm_scan_fwd_ex(g["u"], g["delta"], g["delta_bias"], g["A"], g["B"], g["C"], g["D"],
                        g["z"], True, y, h, init_state=h)
    torch.cuda.synchronize()
    y_ref, h_ref = _oracle(x, init=h0.astype(np.float64))
    assert oracle.rel_err(host64(y), y_ref) <= 1e-2
    assert oracle.rel_err(host64(h), h_ref) <= 1e-2


def test_split_sequence_matches_oracle():
    """Few channels, long sequence: the plan splits L across blocks (two passes with a
    carried state); the result still matches the oracle and the unsplit scan."""
    w = synth.scaled(synth.MAMBA_130M, batch=1, dim=96, seqlen=8192 + 40, seed=13)
    x = synth.make_scan_inputs(w)
    assert ssm.ssm_scan_workspace_bytes(1, 96, w.seqlen, 16, 1) > 0
    y_ref, h_ref = _oracle(x)
    y_s, h_s = _gpu(x, split=True)
    y_u, h_u = _gpu(x, split=False)
    assert oracle.rel_err(y_s, y_ref) <= 1e-2 and oracle.rel_err(h_s, h_ref) <= 1e-2
    assert oracle.rel_err(y_u, y_ref) <= 1e-2 and oracle.rel_err(h_u, h_ref) <= 1e-2
    assert oracle.rel_err(h_s, h_u) <= 1e-4


def test_zero_A_takes_the_limit():
    """A[d, n] = 0 (pure integrator) in some channels: B̄ = Δ B, no NaN."""
    w = synth.scaled(synth.MAMBA_130M, batch=2, dim=64, seqlen=300, seed=14)
    x = synth.make_scan_inputs(w)
    x["A"] = x["A"].copy()
    x["A"][5, :] = 0.0
    x["A"][40, 3] = 0.0
    _check(w, x)


def test_small_and_large_steps():
    """Δ spanning 1e-6 .. 50 (softplus off): the cancellation regime of B̄ and the reset
    regime of Ā."""
    w = synth.scaled(synth.MAMBA_130M, batch=1, dim=64, seqlen=256, seed=15)
    x = synth.make_scan_inputs(w)
    rng = np.random.default_rng(1)
    dl = np.exp(rng.uniform(np.log(1e-6), np.log(50.0), (1, 64, 256))).astype(np.float32)
    x["delta"] = synth.f32_to_bf16(dl)
    _check(w, x, softplus=False, bias=False)


def test_empty_and_degenerate_sizes():
    A = torch.full((8, 16), -1.0, device="cuda")
    e = torch.empty((0, 8, 10), dtype=torch.bfloat16, device="cuda")
    Bz = torch.empty((0, 16, 10), device="cuda")
    ssm.ssm_scan_fwd(e, e, None, A, Bz, Bz, None, None, True, torch.empty_like(e), None)
    # L = 0 writes final_state = init_state
    u0 = torch.empty((2, 8, 0), dtype=torch.bfloat16, device="cuda")
    B0 = torch.empty((2, 16, 0), device="cuda")
    h0 = torch.randn(2, 8, 16, device="cuda")
    h = torch.full((2, 8, 16), 7.0, device="cuda")
    ssm.ssm_scan_fwd_ex(u0, u0, None, A, B0, B0, None, None, True, torch.empty_like(u0), h,
                        init_state=h0)
    torch.cuda.synchronize()
    assert torch.equal(h, h0)
    ssm.ssm_scan_fwd_ex(u0, u0, None, A, B0, B0, None, None, True, torch.empty_like(u0), h)
    torch.cuda.synchronize()
    assert torch.count_nonzero(h).item() == 0


def test_streams_and_errors():
    w = synth.scaled(synth.MAMBA_130M, batch=1, dim=32, seqlen=64, seed=16)
    x = synth.make_scan_inputs(w)
    g = upload_scan(x)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        y, h = ssm.scan(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"], g["delta_bias"])
    s.synchronize()
    y_ref, _ = _oracle(x)
    assert oracle.rel_err(host64(y), y_ref) <= 1e-2
    with pytest.raises(ssm.SSMError) as ei:   # y overlapping u
        ssm.ssm_scan_fwd(g["u"], g["delta"], None, g["A"], g["B"], g["C"], None, None, True,
                         g["u"], None)
    assert ei.value.status == ssm.SSM_ERR_ARG
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    w2 = synth.scaled(synth.MAMBA_130M, batch=1, dim=32, seqlen=65536)
    need = ssm.ssm_scan_workspace_bytes(1, 32, 65536, 16, 1)
    assert need > 16
    u2 = torch.zeros((1, 32, 65536), dtype=torch.bfloat16, device="cuda")
    B2 = torch.zeros((1, 16, 65536), device="cuda")
    with pytest.raises(ssm.SSMError) as ei:
        ssm.ssm_scan_fwd_ex(u2, u2, None, g["A"], B2, B2, None, None, True, torch.empty_like(u2),
                            None, workspace=ws)
    assert ei.value.status == ssm.SSM_ERR_WORKSPACE
    del w2


def test_mamba130m_layer_full_size():
    """batch 8, d_inner 1536, L 2048, N 16, bf16 I/O: every output against the oracle."""
    w = synth.MAMBA_130M
    _check(w, synth.make_scan_inputs(w))


@pytest.mark.parametrize("N", [64, 128])
def test_large_state_split_plan(N):
    """N = 64 and 128 spread a channel over 8 and 16 lanes (8 states each); few
    channels and a long sequence also take the split plan."""
    w = synth.scaled(synth.MAMBA_130M, batch=1, dim=48, seqlen=4096, dstate=N, seed=200 + N)
    assert ssm.ssm_scan_workspace_bytes(1, 48, 4096, N, ssm.SSM_BF16) > 0
    _check(w, synth.make_scan_inputs(w))
