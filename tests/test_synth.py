"""The seeded input generator: SplitMix64 words, bfloat16 rounding, slicing and
the value recipe of the workloads."""
import numpy as np
import torch

import synth

M64 = (1 << 64) - 1


def _splitmix64_reference(state, count):
    """SplitMix64 as published (Steele, Lea & Flood 2014): add the golden gamma, then mix."""
    out = []
    for _ in range(count):
        state = (state + 0x9E3779B97F4A7C15) & M64
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
        out.append(z ^ (z >> 31))
    return out


def _key(seed, stream):
    z = ((seed * 0x9E3779B97F4A7C15) & M64) ^ (stream << 40) ^ 0x5DEECE66D
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
    return z ^ (z >> 31)


def test_words_are_splitmix64_sequence():
    for seed, stream in ((0, 1), (3, 7), (12345, 15)):
        got = synth.words(seed, stream, 0, 40).tolist()
        assert got == _splitmix64_reference(_key(seed, stream), 40)
        assert synth.words(seed, stream, 17, 5).tolist() == got[17:22]


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(10000).astype(np.float32) * 10.0 ** rng.integers(-8, 8, 10000),
                        np.array([1.00390625, 1.01171875, -1.00390625, 3.0e-39, 65504.0], np.float32)])
    x = x.astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(synth.f32_to_bf16(x), ref)
    assert np.array_equal(synth.bf16_to_f32(ref), torch.from_numpy(ref.view(np.int16)).view(
        torch.bfloat16).float().numpy())


def test_rows_regenerate_any_slice():
    w = synth.scaled(synth.MAMBA_130M, batch=2, dim=32, seqlen=300)
    x = synth.make_scan_inputs(w)
    for which in ("u", "delta", "z"):
        r = synth.gen_rows(w, which, 1, 7, 4, 33, 100)
        assert np.array_equal(r, x[which][1, 7:11, 33:133])
    assert np.array_equal(synth.gen_bc(w, "B", 10, 50), x["B"][:, :, 10:60])


def test_value_recipe():
    w = synth.scaled(synth.MAMBA_130M, batch=2, dim=512, seqlen=1024)
    x = synth.make_scan_inputs(w)
    u = synth.bf16_to_f32(x["u"])
    dl = synth.bf16_to_f32(x["delta"])
    assert abs(u.mean()) < 0.01 and abs(u.std() - 1.0) < 0.01
    assert abs(dl.std() - 0.5) < 0.005
    assert x["B"].dtype == np.float32 and abs(x["C"].std() - 1.0) < 0.01
    assert np.array_equal(x["A"][3], -(np.arange(16) + 1.0))
    assert x["D"].min() >= 0.5 and x["D"].max() <= 1.5
    dt = np.log1p(np.exp(x["delta_bias"].astype(np.float64)))   # softplus(bias) = dt
    assert dt.min() >= 1e-3 * 0.999 and dt.max() <= 0.1 * 1.001
    # log-uniform: log(dt) is uniform on [ln 1e-3, ln 0.1]
    ld = (np.log(dt) - np.log(1e-3)) / (np.log(0.1) - np.log(1e-3))
    assert abs(ld.mean() - 0.5) < 0.05
    assert np.array_equal(synth.gen_D(synth.TINY), np.ones(16, np.float32))


def test_decode_inputs_slice():
    dw = synth.DecodeWorkload("d", 4, 64, 16, 5, 8, 4)
    full = synth.make_decode_step_inputs(dw, 0, 5)
    part = synth.make_decode_step_inputs(dw, 2, 2, b0=1, nb=2, d0=10, nd=20)
    for k in ("u", "delta", "z"):
        assert np.array_equal(part[k], full[k][2:4, 1:3, 10:30])
    for k in ("B", "C"):
        assert np.array_equal(part[k], full[k][2:4, 1:3])
