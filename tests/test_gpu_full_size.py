"""GPU parity at the full sizes of the three large workloads, against the fp64 oracle
on sampled channels (the GPU computes every channel; the oracle recomputes a seeded
sample of them one by one):

* Mamba-2.8B-shaped layer scan: batch 4, d_inner 5120, L 4096, N 16, bf16 I/O;
* million-length sequence: batch 1, d_inner 1536, L 2^20, N 16, processed as 16
  launches of 65 536 steps with the fp32 state carried between launches; y compared
  at every step t = 0 (mod 1021) and the final state;
* autoregressive decode: batch 256, d_inner 5120, N 16, 1000 single-token steps from
  the state of a 256-step prefill scan (the oracle's fp64 prefill state rounded to
  fp32 is the common start; the GPU prefill is checked against it separately).

Bar: max|gpu - oracle| / max|oracle| <= 1e-2 for bf16 I/O, for y and the states."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_128_b300 as ssm
import synth
from _gpu import dev_f32, dev_io, host64, upload_scan

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

TOL = 1e-2


def _sample_rows(batch, dim, count, seed):
    rng = np.random.default_rng(seed)
    flat = rng.choice(batch * dim, size=count, replace=False)
    flat.sort()
    return flat // dim, flat % dim


def test_mamba2p8b_layer_full_size_sampled():
    w = synth.MAMBA_2P8B
    x = synth.make_scan_inputs(w)
    g = upload_scan(x)
    y, h = ssm.scan(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"], g["delta_bias"])
    torch.cuda.synchronize()
    bs, ds = _sample_rows(w.batch, w.dim, 192, seed=2)
    y_ref, h_ref = oracle.scan_rows(x["u"][bs, ds], x["delta"][bs, ds], x["z"][bs, ds], bs, ds,
                                    x["A"], x["B"], x["C"], x["D"], x["delta_bias"], True)
    bi, di = torch.from_numpy(bs).cuda(), torch.from_numpy(ds).cuda()
    y_gpu, h_gpu = host64(y[bi, di]), host64(h[bi, di])
    assert np.isfinite(y_gpu).all() and np.isfinite(h_gpu).all()
    assert oracle.rel_err(y_gpu, y_ref) <= TOL
    assert oracle.rel_err(h_gpu, h_ref) <= TOL
    # every output is finite, not only the sampled ones
    assert torch.isfinite(y.float()).all().item() and torch.isfinite(h).all().item()


def test_million_length_carried_state_sampled():
    w = synth.MILLION
    Lc = w.seqlen // w.launches
    stride = 1021
    bs, ds = _sample_rows(w.batch, w.dim, 24, seed=3)
    A = torch.from_numpy(synth.gen_A(w.dim, w.dstate)).cuda()
    D = torch.from_numpy(synth.gen_D(w)).cuda()
    bias = torch.from_numpy(synth.gen_delta_bias(w.seed, w.dim)).cuda()
    h = None
    y_samples = []  # per launch: (rows, steps at t = 0 mod stride within the launch)
    for k in range(w.launches):
        t0 = k * Lc
        rows = {name: synth.gen_rows(w, name, 0, 0, w.dim, t0, Lc)[None] for name in ("u", "delta", "z")}
        u, dl, z = (dev_io(rows[n]) for n in ("u", "delta", "z"))
        Bk = dev_f32(synth.gen_bc(w, "B", t0, Lc))
        Ck = dev_f32(synth.gen_bc(w, "C", t0, Lc))
        y, h = ssm.scan(u, dl, A, Bk, Ck, D, z, bias, init_state=h)
        first = (-t0) % stride
        ts = torch.arange(first, Lc, stride, device="cuda")
        y_samples.append(host64(y[0][torch.from_numpy(ds).cuda()][:, ts]))
        del u, dl, z, Bk, Ck, y
    torch.cuda.synchronize()
    y_gpu = np.concatenate(y_samples, axis=1)
    h_gpu = host64(h[0][torch.from_numpy(ds).cuda()])
    # the oracle over the whole length for the sampled channels (rows regenerated one by one)
    u, dl, z = (np.concatenate([synth.gen_rows(w, n, 0, int(d), 1) for d in ds])
                for n in ("u", "delta", "z"))
    y_ref, h_ref = oracle.scan_rows(u, dl, z, bs, ds, synth.gen_A(w.dim, w.dstate),
                                    synth.gen_bc(w, "B"), synth.gen_bc(w, "C"), synth.gen_D(w),
                                    synth.gen_delta_bias(w.seed, w.dim), True, y_stride=stride)
    assert y_gpu.shape == y_ref.shape
    assert np.isfinite(y_gpu).all() and np.isfinite(h_gpu).all()
    assert oracle.rel_err(y_gpu, y_ref) <= TOL
    assert oracle.rel_err(h_gpu, h_ref) <= TOL


def test_decode_1000_steps_full_size_sampled():
    dw = synth.DECODE
    pw = synth.prefill_workload(dw)
    px = synth.make_scan_inputs(pw)
    # common start: the oracle's prefill state, rounded to fp32 (only the final state is kept)
    U = pw.batch * pw.dim
    ub, ud = np.divmod(np.arange(U), pw.dim)
    _, st_ref = oracle.scan_rows(px["u"].reshape(U, -1), px["delta"].reshape(U, -1),
                                 px["z"].reshape(U, -1), ub, ud, px["A"], px["B"], px["C"],
                                 px["D"], px["delta_bias"], True, y_stride=pw.seqlen)
    st_ref = st_ref.reshape(pw.batch, pw.dim, pw.dstate)
    st0 = st_ref.astype(np.float32)
    # the GPU prefill against it
    g = upload_scan(px)
    _, h_pre = ssm.scan(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"],
                        g["delta_bias"])
    torch.cuda.synchronize()
    assert oracle.rel_err(host64(h_pre), st_ref) <= TOL
    del g, h_pre
    A, D, bias = px["A"], px["D"], px["delta_bias"]
    gA, gD, gb = dev_f32(A), dev_f32(D), dev_f32(bias)
    state = dev_f32(st0)
    bs, ds = _sample_rows(dw.batch, dw.dim, 64, seed=4)
    bi, di = torch.from_numpy(bs).cuda(), torch.from_numpy(ds).cuda()
    # oracle state for the sampled channels
    st_o = st_ref[bs, ds].astype(np.float32).astype(np.float64)
    y_gpu, y_ref = [], []
    chunk = 50
    for s0 in range(0, dw.steps, chunk):
        n = min(chunk, dw.steps - s0)
        inp = synth.make_decode_step_inputs(dw, s0, n)
        for i in range(n):
            y = torch.empty((dw.batch, dw.dim), dtype=torch.bfloat16, device="cuda")
            ssm.ssm_state_update_ex(state, dev_io(inp["u"][i]), dev_io(inp["delta"][i]), gb, True,
                                    gA, dev_f32(inp["B"][i]), dev_f32(inp["C"][i]), gD,
                                    dev_io(inp["z"][i]), y)
            y_gpu.append(host64(y[bi, di]))
            # the oracle's step for the sampled channels: a one-step scan of those units
            yo, st_o = oracle.scan_rows(inp["u"][i][bs, ds][:, None], inp["delta"][i][bs, ds][:, None],
                                        inp["z"][i][bs, ds][:, None], bs, ds, A,
                                        inp["B"][i][:, :, None], inp["C"][i][:, :, None], D, bias,
                                        True, init_state=st_o)
            y_ref.append(yo[:, 0])
    torch.cuda.synchronize()
    y_gpu, y_ref = np.stack(y_gpu), np.stack(y_ref)
    assert np.isfinite(y_gpu).all()
    assert oracle.rel_err(y_gpu, y_ref) <= TOL
    assert oracle.rel_err(host64(state[bi, di]), st_o) <= TOL


def test_backward_mamba130m_layer_full_size_sampled():
    """The backward at the bench's layer size (batch 8, d_inner 1536, L 2048, N 16, bf16):
    dB and dC of batch row 0 in full (they sum over all 1536 channels), du, ddelta, dz
    and d_init_state of 32 sampled channels, and dA, dD, dbias of 24 sampled channels
    (they sum over the 8 batch rows)."""
    w = synth.MAMBA_130M
    x = synth.make_scan_inputs(w)
    e = synth.make_bwd_inputs(w)
    g = upload_scan(x)
    out = ssm.scan_bwd(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"],
                       g["delta_bias"], True, init_state=dev_f32(e["init_state"]),
                       dy=dev_io(e["dy"]), d_final_state=dev_f32(e["d_final_state"]),
                       want_init_grad=True)
    torch.cuda.synchronize()
    dy64 = synth.bf16_to_f32(e["dy"]).astype(np.float64)
    h0 = e["init_state"].astype(np.float64)
    dfin = e["d_final_state"].astype(np.float64)

    def rows(bs, ds):
        return oracle.scan_bwd_rows(x["u"][bs, ds], x["delta"][bs, ds], x["z"][bs, ds], bs, ds,
                                    x["A"], x["B"], x["C"], x["D"], x["delta_bias"], True,
                                    dy64[bs, ds], h0[bs, ds], dfin[bs, ds], nbatch=w.batch)

    # batch row 0, every channel: dB[0], dC[0] in full
    d_all = np.arange(w.dim)
    r0 = rows(np.zeros(w.dim, np.int64), d_all)
    assert oracle.rel_err(host64(out["dB"][0]), r0["dB"][0]) <= TOL
    assert oracle.rel_err(host64(out["dC"][0]), r0["dC"][0]) <= TOL
    bs, ds = _sample_rows(w.batch, w.dim, 32, seed=5)
    rs = rows(bs, ds)
    bi, di = torch.from_numpy(bs).cuda(), torch.from_numpy(ds).cuda()
    for k in ("du", "ddelta", "dz"):
        assert oracle.rel_err(host64(out[k][bi, di]), rs[k]) <= TOL, k
    assert oracle.rel_err(host64(out["dinit"][bi, di]), rs["dinit"]) <= TOL
    # per-channel sums over the batch for 24 channels
    dsel = np.random.default_rng(6).choice(w.dim, 24, replace=False)
    bb = np.repeat(np.arange(w.batch), len(dsel))
    dd = np.tile(dsel, w.batch)
    rc = rows(bb, dd)
    dA_ref = rc["dA_unit"].reshape(w.batch, len(dsel), w.dstate).sum(0)
    dD_ref = rc["dD_unit"].reshape(w.batch, len(dsel)).sum(0)
    db_ref = rc["dbias_unit"].reshape(w.batch, len(dsel)).sum(0)
    dsel_t = torch.from_numpy(dsel).cuda()
    assert oracle.rel_err(host64(out["dA"][dsel_t]), dA_ref) <= TOL
    assert oracle.rel_err(host64(out["dD"][dsel_t]), dD_ref) <= TOL
    assert oracle.rel_err(host64(out["dbias"][dsel_t]), db_ref) <= TOL


def test_backward_million_length_one_call_sampled():
    """The backward over the million-length sequence in one call (batch 1, d_inner 1536,
    L 2^20, N 16, bf16), where the plan splits the sequence into segments that fold
    each other's carries: du, ddelta, dz over the whole length, d_init_state, and
    (one batch row) dA, dD, dbias of 16 sampled channels against the oracle; every
    output finite.  dB and dC sum over all 1536 channels: the split cases of the
    backward's parity tests check them in full at smaller sizes."""
    w = synth.MILLION
    L, dim, N = w.seqlen, w.dim, w.dstate
    dev = "cuda"
    step = 128
    t = {k: torch.empty((1, dim, L), dtype=torch.bfloat16, device=dev)
         for k in ("u", "delta", "z", "dy")}
    for d0 in range(0, dim, step):
        for k in ("u", "delta", "z"):
            t[k][0, d0:d0 + step] = dev_io(synth.gen_rows(w, k, 0, d0, step))
        dyk = synth.fill(w.seed, synth.S_DY, d0 * L, step * L, synth.NORMAL, 0.0, 1.0,
                         dtype=w.io).reshape(step, L)
        t["dy"][0, d0:d0 + step] = dev_io(dyk)
    e = synth.make_bwd_inputs(synth.scaled(w, seqlen=1))  # init / d_final: (batch, dim, N)
    h0 = e["init_state"].astype(np.float64)
    dfin = e["d_final_state"].astype(np.float64)
    A, D = synth.gen_A(dim, N), synth.gen_D(w)
    bias = synth.gen_delta_bias(w.seed, dim)
    B, C = synth.gen_bc(w, "B"), synth.gen_bc(w, "C")
    out = ssm.scan_bwd(t["u"], t["delta"], dev_f32(A), dev_f32(B), dev_f32(C), dev_f32(D),
                       t["z"], dev_f32(bias), True, init_state=dev_f32(e["init_state"]),
                       dy=t["dy"], d_final_state=dev_f32(e["d_final_state"]),
                       want_init_grad=True)
    torch.cuda.synchronize()
    for k in ("du", "ddelta", "dz", "dA", "dB", "dC", "dD", "dbias", "dinit"):
        assert torch.isfinite(out[k].float()).all().item(), k
    bs, ds = _sample_rows(w.batch, dim, 16, seed=9)
    di = torch.from_numpy(ds).cuda()
    got = {k: host64(out[k][0][di]) for k in ("du", "ddelta", "dz", "dinit")}
    got.update({k: host64(out[k][di]) for k in ("dA", "dD", "dbias")})
    del out, t
    rows = {k: np.concatenate([synth.gen_rows(w, k, 0, int(d), 1) for d in ds])
            for k in ("u", "delta", "z")}
    dy64 = np.concatenate([synth.bf16_to_f32(synth.fill(w.seed, synth.S_DY, int(d) * L, L,
                                                        synth.NORMAL, 0.0, 1.0, dtype=w.io))
                           [None] for d in ds]).astype(np.float64)
    r = oracle.scan_bwd_rows(rows["u"], rows["delta"], rows["z"], bs, ds, A, B, C, D, bias,
                             True, dy64, h0[bs, ds], dfin[bs, ds], nbatch=1)
    for k in ("du", "ddelta", "dz", "dinit"):
        assert oracle.rel_err(got[k], r[k]) <= TOL, k
    assert oracle.rel_err(got["dA"], r["dA_unit"]) <= TOL
    assert oracle.rel_err(got["dD"], r["dD_unit"]) <= TOL
    assert oracle.rel_err(got["dbias"], r["dbias_unit"]) <= TOL


def test_conv1d_backward_at_layer_size_sampled():
    """The front end's backward at the bench's size (8 x 1536 x 2048 bf16, width 4, rows
    staged through the shared-memory ring): dx, dweight, dbias and d state of 24
    sampled channels over all 8 batch rows against the oracle; every output finite."""
    w = synth.MAMBA_130M
    x = synth.make_scan_inputs(w)
    wt = synth.fill(7, synth.S_B, 0, w.dim * 4, synth.NORMAL, 0.0, 0.5).reshape(w.dim, 4)
    bias = synth.fill(7, synth.S_D, 0, w.dim, synth.NORMAL, 0.0, 0.2)
    st = synth.fill(7, synth.S_H0, 0, w.batch * w.dim * 3, synth.NORMAL, 0.0, 1.0,
                    dtype="bf16").reshape(w.batch, w.dim, 3)
    dout = synth.make_bwd_inputs(w, init_state=False, d_final_state=False)["dy"]
    out = ssm.conv1d_bwd(dev_io(x["u"]), dev_f32(wt), dev_io(dout), dev_f32(bias), dev_io(st))
    torch.cuda.synchronize()
    for k in ("dx", "dweight", "dbias", "dstate"):
        assert torch.isfinite(out[k].float()).all().item(), k
    dsel = np.sort(np.random.default_rng(10).choice(w.dim, 24, replace=False))
    ref = oracle.conv1d_bwd(np.ascontiguousarray(x["u"][:, dsel]), wt[dsel], bias[dsel],
                            synth.bf16_to_f32(st[:, dsel]), True, np.ascontiguousarray(dout[:, dsel]))
    di = torch.from_numpy(dsel).cuda()
    assert oracle.rel_err(host64(out["dx"][:, di]), ref["dx"]) <= TOL
    assert oracle.rel_err(host64(out["dweight"][di]), ref["dweight"]) <= 1e-3
    assert oracle.rel_err(host64(out["dbias"][di]), ref["dbias"]) <= 1e-3
    assert oracle.rel_err(host64(out["dstate"][:, di]), ref["dstate"]) <= 1e-3


def test_conv1d_and_bld_scan_at_layer_size():
    """The front end at the bench's size (8 x 1536 x 2048 bf16, width 4) on 64 sampled
    rows, and the (batch, L, dim) scan of the layer equal, bit for bit, to the
    (batch, dim, L) one (which the parity tests above pin to the oracle)."""
    w = synth.MAMBA_130M
    x = synth.make_scan_inputs(w)
    wt = synth.fill(7, synth.S_B, 0, w.dim * 4, synth.NORMAL, 0.0, 0.5).reshape(w.dim, 4)
    bias = synth.fill(7, synth.S_D, 0, w.dim, synth.NORMAL, 0.0, 0.2)
    gu = dev_io(x["u"])
    out = ssm.conv1d(gu, dev_f32(wt), dev_f32(bias))
    torch.cuda.synchronize()
    bs, ds = _sample_rows(w.batch, w.dim, 64, seed=8)
    # the sampled rows as one batch row of 64 channels with their own weights
    ref, _ = oracle.conv1d(np.ascontiguousarray(x["u"][bs, ds][None]), wt[ds], bias[ds])
    got = host64(out[torch.from_numpy(bs).cuda(), torch.from_numpy(ds).cuda()])
    assert oracle.rel_err(got, ref[0]) <= TOL
    g = upload_scan(x)
    y0, h0 = ssm.scan(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"], g["delta_bias"])
    t = {k: g[k].transpose(1, 2).contiguous() for k in ("u", "delta", "z")}
    y1, h1 = ssm.scan(t["u"], t["delta"], g["A"], g["B"], g["C"], g["D"], t["z"], g["delta_bias"],
                      bld=True)
    torch.cuda.synchronize()
    assert torch.equal(y1.transpose(1, 2), y0) and torch.equal(h1, h0)
