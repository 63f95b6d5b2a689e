"""GPU parity of ssm_state_update / ssm_state_update_ex (one-token decode) against the
fp64 oracle, the decode == scan invariant, and a loop of steps replayed from a CUDA
graph."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_128_b300 as ssm
import synth
from _gpu import dev_f32, dev_io, host64, upload_scan

pytestmark = pytest.mark.gpu


def _decode_case(batch, dim, N, steps, io="bf16", seed=40):
    dw = synth.DecodeWorkload("t", batch, dim, N, steps, 32, seed, io=io)
    return dw, synth.make_decode_step_inputs(dw, 0, steps)


@pytest.mark.parametrize("N", [1, 2, 4, 8, 16, 32, 64, 128])
@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_decode_steps_match_oracle(N, io):
    dw, s = _decode_case(3, 50, N, 6, io)
    A = synth.gen_A(dw.dim, N)
    D = synth.fill(seed := 41, synth.S_D, 0, dw.dim, synth.UNIFORM, 0.5, 1.5)
    bias = synth.gen_delta_bias(seed, dw.dim)
    rng = np.random.default_rng(N)
    st0 = rng.standard_normal((dw.batch, dw.dim, N)).astype(np.float32)
    st_ref = st0.astype(np.float64)
    st = dev_f32(st0)
    gA, gD, gb = dev_f32(A), dev_f32(D), dev_f32(bias)
    tol = 1e-4 if io == "f32" else 1e-2
    for i in range(dw.steps):
        y_ref, st_ref = oracle.step(st_ref, s["u"][i], s["delta"][i], A, s["B"][i], s["C"][i], D,
                                    s["z"][i], bias, True)
        y = torch.empty(dev_io(s["u"][i]).shape, dtype=dev_io(s["u"][i]).dtype, device="cuda")
        ssm.ssm_state_update_ex(st, dev_io(s["u"][i]), dev_io(s["delta"][i]), gb, True, gA,
                                dev_f32(s["B"][i]), dev_f32(s["C"][i]), gD, dev_io(s["z"][i]), y)
        torch.cuda.synchronize()
        assert oracle.rel_err(host64(y), y_ref) <= tol
        assert oracle.rel_err(host64(st), st_ref) <= tol


def test_short_form_uses_delta_as_given():
    dw, s = _decode_case(2, 64, 16, 1)
    A = synth.gen_A(64, 16)
    dl = np.abs(synth.bf16_to_f32(s["delta"][0])) * 0.1 + 1e-3
    dl_bits = synth.f32_to_bf16(dl)
    st0 = np.zeros((2, 64, 16), np.float32) + 0.5
    y_ref, st_ref = oracle.step(st0.astype(np.float64), s["u"][0], dl_bits, A, s["B"][0],
                                s["C"][0], None, None, None, False)
    st = dev_f32(st0)
    y = torch.empty((2, 64), dtype=torch.bfloat16, device="cuda")
    ssm.ssm_state_update(st, dev_io(s["u"][0]), dev_io(dl_bits), dev_f32(A), dev_f32(s["B"][0]),
                         dev_f32(s["C"][0]), None, None, y)
    torch.cuda.synchronize()
    assert oracle.rel_err(host64(y), y_ref) <= 1e-2
    assert oracle.rel_err(host64(st), st_ref) <= 1e-2


def test_decode_steps_equal_scan_on_gpu():
    """L single-token steps from a zero state give the scan's outputs and final state."""
    w = synth.scaled(synth.MAMBA_130M, batch=2, dim=64, seqlen=40, seed=42)
    x = synth.make_scan_inputs(w)
    g = upload_scan(x)
    y_scan, h_scan = ssm.scan(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"],
                              g["delta_bias"])
    st = torch.zeros((2, 64, 16), device="cuda")
    ys = []
    for t in range(w.seqlen):
        y = torch.empty((2, 64), dtype=torch.bfloat16, device="cuda")
        ssm.ssm_state_update_ex(st, g["u"][:, :, t].contiguous(), g["delta"][:, :, t].contiguous(),
                                g["delta_bias"], True, g["A"], g["B"][:, :, t].contiguous(),
                                g["C"][:, :, t].contiguous(), g["D"], g["z"][:, :, t].contiguous(), y)
        ys.append(y)
    torch.cuda.synchronize()
    yd = host64(torch.stack(ys, dim=2))
    assert oracle.rel_err(yd, host64(y_scan)) <= 1e-2
    assert oracle.rel_err(host64(st), host64(h_scan)) <= 1e-4
    y_ref, h_ref = oracle.scan(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                               x["delta_bias"])
    assert oracle.rel_err(yd, y_ref) <= 1e-2 and oracle.rel_err(host64(st), h_ref) <= 1e-2


def test_zero_A_decode():
    dw, s = _decode_case(2, 32, 16, 1, seed=43)
    A = synth.gen_A(32, 16)
    A[3, :] = 0.0
    st0 = np.ones((2, 32, 16), np.float32)
    y_ref, st_ref = oracle.step(st0.astype(np.float64), s["u"][0], s["delta"][0], A, s["B"][0],
                                s["C"][0], None, s["z"][0], None, True)
    st = dev_f32(st0)
    y = torch.empty((2, 32), dtype=torch.bfloat16, device="cuda")
    ssm.ssm_state_update_ex(st, dev_io(s["u"][0]), dev_io(s["delta"][0]), None, True, dev_f32(A),
                            dev_f32(s["B"][0]), dev_f32(s["C"][0]), None, dev_io(s["z"][0]), y)
    torch.cuda.synchronize()
    assert oracle.rel_err(host64(y), y_ref) <= 1e-2
    assert oracle.rel_err(host64(st), st_ref) <= 1e-2


@pytest.mark.parametrize("gate,softplus", [(True, True), (False, True), (True, False)])
def test_whole_channel_blocks_with_zero_A(gate, softplus):
    """d_inner a multiple of the block's channels (192 = 3 x 64), N 16, bf16, with and
    without gate and softplus, including a channel with A = 0 states (that channel
    takes the precise flavour, the exact limit Ā = 1, B̄ = Δ B)."""
    dw, s = _decode_case(7, 192, 16, 4, "bf16", seed=44)
    A = synth.gen_A(dw.dim, 16)
    A[5, ::3] = 0.0
    D = synth.fill(45, synth.S_D, 0, dw.dim, synth.UNIFORM, 0.5, 1.5)
    bias = synth.gen_delta_bias(45, dw.dim)
    st0 = np.random.default_rng(7).standard_normal((dw.batch, dw.dim, 16)).astype(np.float32)
    st_ref = st0.astype(np.float64)
    st = dev_f32(st0)
    for i in range(dw.steps):
        dl = s["delta"][i]
        if not softplus:
            dl = synth.f32_to_bf16(np.abs(synth.bf16_to_f32(dl)) * 0.1 + 1e-3)
        z = s["z"][i] if gate else None
        y_ref, st_ref = oracle.step(st_ref, s["u"][i], dl, A, s["B"][i], s["C"][i], D, z,
                                    bias if softplus else None, softplus)
        u = dev_io(s["u"][i])
        y = torch.empty_like(u)
        ssm.ssm_state_update_ex(st, u, dev_io(dl), dev_f32(bias) if softplus else None, softplus,
                                dev_f32(A), dev_f32(s["B"][i]), dev_f32(s["C"][i]), dev_f32(D),
                                dev_io(z), y)
        torch.cuda.synchronize()
        assert oracle.rel_err(host64(y), y_ref) <= 1e-2
        assert oracle.rel_err(host64(st), st_ref) <= 1e-2
    assert ssm.ssm_status(None) == ssm.SSM_OK


def test_decode_steps_replayed_from_a_cuda_graph():
    """The decode entry point makes no synchronising call, so a loop of steps can be
    captured once in a CUDA graph and replayed: the replay equals the same steps
    launched one by one, bit for bit, and the oracle."""
    dw, s = _decode_case(4, 96, 16, 12, seed=44)
    A = dev_f32(synth.gen_A(dw.dim, 16))
    D = dev_f32(synth.fill(45, synth.S_D, 0, dw.dim, synth.UNIFORM, 0.5, 1.5))
    bias_h = synth.gen_delta_bias(45, dw.dim)
    bias = dev_f32(bias_h)
    st0 = np.random.default_rng(46).standard_normal((dw.batch, dw.dim, 16)).astype(np.float32)
    ins = [dict(u=dev_io(s["u"][i]), delta=dev_io(s["delta"][i]), z=dev_io(s["z"][i]),
                B=dev_f32(s["B"][i]), C=dev_f32(s["C"][i])) for i in range(dw.steps)]

    def run(st, ys, stream):
        for i, x in enumerate(ins):
            ssm.ssm_state_update_ex(st, x["u"], x["delta"], bias, True, A, x["B"], x["C"], D,
                                    x["z"], ys[i], stream=stream)

    st_a = dev_f32(st0)
    ys_a = [torch.empty((dw.batch, dw.dim), dtype=torch.bfloat16, device="cuda")
            for _ in range(dw.steps)]
    run(st_a, ys_a, torch.cuda.current_stream())
    st_b = dev_f32(st0)
    ys_b = [torch.empty_like(y) for y in ys_a]
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run(st_b, ys_b, torch.cuda.current_stream())
    st_b.copy_(dev_f32(st0))   # the capture recorded the steps without running them
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(st_b, st_a)
    assert all(torch.equal(yb, ya) for yb, ya in zip(ys_b, ys_a))
    st_ref = st0.astype(np.float64)
    Ah = synth.gen_A(dw.dim, 16)
    Dh = synth.fill(45, synth.S_D, 0, dw.dim, synth.UNIFORM, 0.5, 1.5)
    for i in range(dw.steps):
        y_ref, st_ref = oracle.step(st_ref, s["u"][i], s["delta"][i], Ah, s["B"][i], s["C"][i], Dh,
                                    s["z"][i], bias_h, True)
        assert oracle.rel_err(host64(ys_b[i]), y_ref) <= 1e-2
    assert oracle.rel_err(host64(st_b), st_ref) <= 1e-2
