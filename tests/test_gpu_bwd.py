"""GPU parity of ssm_scan_bwd (the backward pass) against the fp64 backward oracle.

Every derivative is compared element by element: du, ddelta, dz (batch, dim, L),
dA (dim, N), dB, dC (batch, N, L), dD, dbias (dim), d_init_state (batch, dim, N).
Bar, per output: max|gpu - ref| / max|ref| <= 1e-4 for float32 I/O and <= 1e-2 for
bfloat16 I/O (the forward's bar; the bf16 outputs du/ddelta/dz are rounded to
bfloat16, a relative 2^-9 of each value).  Sizes span several chunks and channel
blocks with ragged tails."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_128_b300 as ssm
import synth
from _gpu import dev_f32, dev_io, host64, upload_scan

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 1e-2}
KEYS = ("du", "ddelta", "dz", "dA", "dB", "dC", "dD", "dbias", "dinit")


def _as64(a):
    a = np.asarray(a)
    return synth.bf16_to_f32(a).astype(np.float64) if a.dtype == np.uint16 else a.astype(np.float64)


def _run(w, z=True, D=True, bias=True, softplus=True, init=True, dfin=True, zero_a=False):
    x = synth.make_scan_inputs(w)
    if zero_a:
        x["A"][1, ::2] = 0.0           # channel 1: the A = 0 limit on half its states
    if not softplus:
        # Δ is used as given: make it a step size (positive, the recipe's range)
        dpos = (np.abs(_as64(x["delta"])) * 0.2).astype(np.float32)
        x["delta"] = dpos if w.io == "f32" else synth.f32_to_bf16(dpos)
        x["delta_bias"] = np.full_like(x["delta_bias"], 0.01)
    e = synth.make_bwd_inputs(w, init_state=init, d_final_state=dfin)
    ref = oracle.scan_bwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"] if D else None,
                          x["z"] if z else None, x["delta_bias"] if bias else None, softplus,
                          None if e["init_state"] is None else e["init_state"].astype(np.float64),
                          _as64(e["dy"]),
                          None if e["d_final_state"] is None else e["d_final_state"].astype(np.float64))
    g = upload_scan(x)
    out = ssm.scan_bwd(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"] if D else None,
                       g["z"] if z else None, g["delta_bias"] if bias else None, softplus,
                       init_state=dev_f32(e["init_state"]), dy=dev_io(e["dy"]),
                       d_final_state=dev_f32(e["d_final_state"]), want_init_grad=True)
    torch.cuda.synchronize()
    return ref, out


def _check(w, tol=None, **kw):
    tol = TOL[w.io] if tol is None else tol
    ref, out = _run(w, **kw)
    errs = {}
    for k in KEYS:
        if ref[k] is None:
            assert out[k] is None, k
            continue
        got = host64(out[k])
        assert got.shape == ref[k].shape, k
        assert np.isfinite(got).all(), k
        errs[k] = oracle.rel_err(got, ref[k])
    bad = {k: v for k, v in errs.items() if v > tol}
    assert not bad, bad
    return errs


def test_fp32_all_inputs_ragged():
    """float32 I/O, N 16: 3 channel blocks (70 = 2 x 32 + 6), 5 chunks (77 = 4 x 16 + 13)."""
    w = synth.scaled(synth.TINY, name="bwd_f32", batch=2, dim=70, seqlen=77, dstate=16, seed=31,
                     d_one=False)
    errs = _check(w)
    assert max(errs.values()) < 2e-5


def test_bf16_mamba_value_recipe():
    w = synth.scaled(synth.MAMBA_130M, name="bwd_bf16", batch=2, dim=96, seqlen=200, seed=32)
    _check(w)


@pytest.mark.parametrize("N", [1, 2, 4, 8, 32, 64, 128])
def test_bf16_every_state_size(N):
    w = synth.scaled(synth.MAMBA_130M, name="bwd_n%d" % N, batch=2, dim=150, seqlen=45,
                     dstate=N, seed=40 + N)
    _check(w)


@pytest.mark.parametrize("N", [1, 4, 64, 128])
def test_fp32_state_sizes(N):
    w = synth.scaled(synth.TINY, name="bwd_f32_n%d" % N, batch=1, dim=33, seqlen=37, dstate=N,
                     seed=50 + N, d_one=False)
    _check(w)


@pytest.mark.parametrize("variant", ["no_gate", "no_softplus", "no_D_no_bias", "no_init_no_dfinal",
                                     "zero_A"])
def test_bf16_variants(variant):
    w = synth.scaled(synth.MAMBA_130M, name="bwd_" + variant, batch=2, dim=40, seqlen=70,
                     seed=60)
    kw = dict(no_gate=dict(z=False), no_softplus=dict(softplus=False),
              no_D_no_bias=dict(D=False, bias=False),
              no_init_no_dfinal=dict(init=False, dfin=False), zero_A=dict(zero_a=True))[variant]
    _check(w, **kw)


def test_fp32_zero_A_precise_limit():
    w = synth.scaled(synth.TINY, name="bwd_f32_zeroA", batch=1, dim=20, seqlen=50, dstate=16,
                     seed=61, d_one=False)
    _check(w, zero_a=True)


def test_single_step_and_single_channel():
    for (b, d, L) in ((1, 1, 1), (3, 1, 17), (1, 5, 1)):
        w = synth.scaled(synth.MAMBA_130M, name="bwd_small", batch=b, dim=d, seqlen=L, seed=62)
        _check(w)


def test_chunked_backward_equals_one_shot():
    """A sequence split in two launches, the second's d_init_state feeding the first's
    d_final_state (and the first's final state the second's init_state), gives the
    same derivatives as one launch over the whole sequence."""
    w = synth.scaled(synth.MAMBA_130M, name="bwd_chunked", batch=2, dim=64, seqlen=96, seed=63,
                     io="f32")
    x = synth.make_scan_inputs(w)
    e = synth.make_bwd_inputs(w, init_state=False)
    g = upload_scan(x)
    dy = dev_io(e["dy"])
    dfin = dev_f32(e["d_final_state"])
    whole = ssm.scan_bwd(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"],
                         g["delta_bias"], True, dy=dy, d_final_state=dfin)
    cut = 40
    part = {k: (g[k][..., :cut].contiguous(), g[k][..., cut:].contiguous())
            for k in ("u", "delta", "z", "B", "C")}
    _, h_mid = ssm.scan(part["u"][0], part["delta"][0], g["A"], part["B"][0], part["C"][0], g["D"],
                        part["z"][0], g["delta_bias"])
    second = ssm.scan_bwd(part["u"][1], part["delta"][1], g["A"], part["B"][1], part["C"][1],
                          g["D"], part["z"][1], g["delta_bias"], True, init_state=h_mid,
                          dy=dy[..., cut:].contiguous(), d_final_state=dfin, want_init_grad=True)
    first = ssm.scan_bwd(part["u"][0], part["delta"][0], g["A"], part["B"][0], part["C"][0],
                         g["D"], part["z"][0], g["delta_bias"], True,
                         dy=dy[..., :cut].contiguous(), d_final_state=second["dinit"])
    torch.cuda.synchronize()
    for k in ("du", "ddelta", "dz", "dB", "dC"):
        got = torch.cat([first[k], second[k]], dim=-1)
        assert oracle.rel_err(host64(got), host64(whole[k])) < 1e-5, k
    for k in ("dA", "dD", "dbias"):
        assert oracle.rel_err(host64(first[k] + second[k]), host64(whole[k])) < 1e-5, k


def test_empty_sizes():
    dev = "cuda"
    A = torch.full((8, 16), -1.0, device=dev)
    # no steps: sums are zero, d_init_state = d_final_state
    u = torch.zeros((2, 8, 0), dtype=torch.bfloat16, device=dev)
    B = torch.zeros((2, 16, 0), device=dev)
    dfin = torch.randn((2, 8, 16), device=dev)
    out = ssm.scan_bwd(u, u, A, B, B, torch.ones(8, device=dev), None, None, True, dy=u,
                       d_final_state=dfin, want_init_grad=True)
    torch.cuda.synchronize()
    assert torch.equal(out["dinit"], dfin)
    assert out["dA"].abs().max().item() == 0.0 and out["dD"].abs().max().item() == 0.0
    assert out["dbias"].abs().max().item() == 0.0
    # no channels: dB and dC are zero sums
    u = torch.zeros((2, 0, 5), dtype=torch.bfloat16, device=dev)
    B = torch.randn((2, 16, 5), device=dev)
    out = ssm.scan_bwd(u, u, torch.zeros((0, 16), device=dev), B, B, dy=u)
    torch.cuda.synchronize()
    assert out["dB"].abs().max().item() == 0.0 and out["dC"].abs().max().item() == 0.0


@pytest.mark.parametrize("case", ["bf16_n16", "f32_n16", "bf16_n4", "bf16_split", "bf16_n32",
                                  "bf16_n128", "euler"])
def test_training_forward_saves_what_the_backward_recomputes(case):
    """ssm_scan_fwd_train returns the forward's results and saves the chunk-start
    states; the backward that starts from them (SSM_SAVED_STATES) gives the same
    derivatives as the backward that recomputes them (N = 32 and 128 save nothing
    and the flag changes nothing)."""
    kw = dict(bf16_n16=dict(), f32_n16=dict(io="f32"), bf16_n4=dict(dstate=4),
              bf16_split=dict(batch=1, dim=64, seqlen=8192), bf16_n32=dict(dstate=32),
              bf16_n128=dict(dstate=128, dim=40), euler=dict())[case]
    base = dict(name="bwd_saved", batch=2, dim=96, seqlen=300, seed=120)
    base.update(kw)
    w = synth.scaled(synth.MAMBA_130M, **base)
    x = synth.make_scan_inputs(w)
    e = synth.make_bwd_inputs(w)
    g = upload_scan(x)
    euler = case == "euler"
    h0 = dev_f32(e["init_state"])
    args = (g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"], g["delta_bias"], True)
    y_t, h_t, saved = ssm.scan_train(*args, init_state=h0, euler=euler)
    y_f, h_f = ssm.scan(*args, init_state=h0, euler=euler)
    kw2 = dict(init_state=h0, dy=dev_io(e["dy"]), d_final_state=dev_f32(e["d_final_state"]),
               want_init_grad=True, euler=euler)
    plain = ssm.scan_bwd(*args, **kw2)
    fast = ssm.scan_bwd(*args, saved=saved, **kw2)
    torch.cuda.synchronize()
    assert torch.equal(y_t, y_f) and torch.equal(h_t, h_f)
    # one launch: the saved states are the backward's own, bit for bit; the split plan
    # folds segment carries in another order, so a bf16 output may round differently
    tol = 2e-3 if case == "bf16_split" else 1e-6
    for k in ("du", "ddelta", "dz", "dA", "dB", "dC", "dD", "dbias", "dinit"):
        assert oracle.rel_err(host64(fast[k]), host64(plain[k])) <= tol, k


@pytest.mark.parametrize("N,L", [(1, 300), (4, 300), (8, 300), (8, 296), (16, 300)])
def test_row_lengths_that_misalign_wide_vectors(N, L):
    """Rows of bf16 whose length is a multiple of 4 but not of 8 start on 8-byte
    boundaries: the 16-byte vector path must not be taken there."""
    w = synth.scaled(synth.MAMBA_130M, name="bwd_align", batch=2, dim=40, seqlen=L, dstate=N,
                     seed=130 + N)
    _check(w)


# channels per block and steps per chunk of the backward kernel, for the expected
# workspace of an unsplit plan
_BWD_GEOM = {4: (128, 16), 16: (32, 16), 128: (16, 8)}


def _unsplit_bytes(batch, dim, L, N):
    ch, t = _BWD_GEOM[N]

    def al(x):
        return (x + 255) // 256 * 256

    nblk, nch = -(-dim // ch), -(-L // t)
    return (al(batch * nch * dim * N * 4) + 2 * al(batch * nblk * N * L * 4)
            + al(batch * dim * N * 4) + 2 * al(batch * dim * 4))


@pytest.mark.parametrize("case", ["bf16_n16", "f32_n4", "bf16_n128", "bf16_n16_bld", "euler",
                                  "zero_a", "no_states"])
def test_split_sequence_matches_oracle(case):
    """Sizes with few channel blocks and long rows, where the backward's plan splits
    the sequence into segments (each block folds the forward's and the adjoint's
    carries of the other segments): every derivative against the oracle, ragged
    last segments and chunks.  The (batch, L, dim) case must also equal the
    (batch, dim, L) run bit for bit."""
    kw = dict(bf16_n16=dict(batch=1, dim=40, seqlen=3000),
              f32_n4=dict(batch=2, dim=8, seqlen=2100, dstate=4, io="f32"),
              bf16_n128=dict(batch=1, dim=16, seqlen=1500, dstate=128),
              bf16_n16_bld=dict(batch=2, dim=40, seqlen=2100),
              euler=dict(batch=1, dim=40, seqlen=2050),
              zero_a=dict(batch=1, dim=40, seqlen=2050),
              no_states=dict(batch=1, dim=33, seqlen=2500))[case]
    base = dict(name="bwd_split", seed=170)
    base.update(kw)
    w = synth.scaled(synth.MAMBA_130M, **base)
    # the plan does split here: its workspace holds the segment carries
    assert (ssm.ssm_scan_bwd_workspace_bytes(w.batch, w.dim, w.seqlen, w.dstate)
            > _unsplit_bytes(w.batch, w.dim, w.seqlen, w.dstate))
    if case in ("bf16_n16", "f32_n4", "bf16_n128", "no_states"):
        states = case != "no_states"
        _check(w, init=states, dfin=states)
        return
    x = synth.make_scan_inputs(w)
    if case == "zero_a":
        x["A"][1, ::2] = 0.0
    e = synth.make_bwd_inputs(w)
    dy64 = _as64(e["dy"])
    euler = case == "euler"
    ref = oracle.scan_bwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                          x["delta_bias"], True, e["init_state"].astype(np.float64), dy64,
                          e["d_final_state"].astype(np.float64), euler=euler)
    g = upload_scan(x)
    kw2 = dict(init_state=dev_f32(e["init_state"]), d_final_state=dev_f32(e["d_final_state"]),
               want_init_grad=True, euler=euler)
    args = (g["A"], g["B"], g["C"], g["D"])
    out = ssm.scan_bwd(g["u"], g["delta"], *args, g["z"], g["delta_bias"], True,
                       dy=dev_io(e["dy"]), **kw2)
    if case == "bf16_n16_bld":
        def bld(t):
            return t.transpose(1, 2).contiguous()
        out1 = ssm.scan_bwd(bld(g["u"]), bld(g["delta"]), *args, bld(g["z"]), g["delta_bias"],
                            True, dy=bld(dev_io(e["dy"])), bld=True, **kw2)
        torch.cuda.synchronize()
        for k in ("du", "ddelta", "dz"):
            assert torch.equal(out1[k].transpose(1, 2), out[k]), k
        for k in ("dA", "dB", "dC", "dD", "dbias", "dinit"):
            assert torch.equal(out1[k], out[k]), k
    torch.cuda.synchronize()
    for k in KEYS:
        assert oracle.rel_err(host64(out[k]), ref[k]) <= TOL[w.io], k
