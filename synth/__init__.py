"""Seeded synthetic inputs for the selective-scan workloads.

This package only draws and encodes random numbers (see ``synth.c`` for the
generator's definition); it holds none of the scan's arithmetic.  The oracle
and the CUDA path both read the arrays it returns, so both sides see the same
bits.  bfloat16 tensors are returned as ``numpy.uint16`` bit patterns.

Value recipe (the Mamba page's hyper-parameter table, section 4d, and the
shape table of section 4a, "Mamba: Linear-Time Sequence Modeling" summary):

* u, z ~ N(0, 1); Δ_raw ~ N(0, σ = 0.5) (the workload text "N(0,0.25)" is
  read as a variance);
* per channel dt ~ log-uniform[1e-3, 0.1] and delta_bias = log(expm1(dt)),
  i.e. the inverse softplus of dt, computed in double and rounded to float;
* A[d, n] = -(n + 1) (S4D-Real initialisation);
* D = 1 for the tiny fp32 workload, else D ~ U(0.5, 1.5);
* B, C ~ N(0, 1) with shape (batch, N, L), shared by all channels.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libssm_synth.so")
_lib = None

# stream ids, one per tensor
S_U, S_DELTA, S_Z, S_B, S_C, S_D, S_DT = 1, 2, 3, 4, 5, 6, 7
S_DEC_U, S_DEC_DELTA, S_DEC_Z, S_DEC_B, S_DEC_C = 11, 12, 13, 14, 15
S_DY, S_DFIN, S_H0 = 21, 22, 23          # backward: upstream derivatives, initial state

NORMAL, UNIFORM, LOGUNIFORM = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile ``libssm_synth.so`` next to its source (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        u64, i64, i32, dbl, vp = (ctypes.c_uint64, ctypes.c_int64, ctypes.c_int,
                                  ctypes.c_double, ctypes.c_void_p)
        for name in ("synth_fill_f32", "synth_fill_bf16", "synth_fill_f64"):
            getattr(lib, name).argtypes = [u64, u64, u64, i64, i32, dbl, dbl, vp]
            getattr(lib, name).restype = None
        lib.synth_words.argtypes = [u64, u64, u64, i64, vp]
        lib.synth_f32_to_bf16.argtypes = [vp, i64, vp]
        _lib = lib
    return _lib


def fill(seed, stream, offset, n, kind, p0, p1, dtype="f32", out=None):
    """Draw elements ``offset .. offset+n`` of a stream into a new flat array."""
    lib = _load()
    np_dtype = {"f32": np.float32, "bf16": np.uint16, "f64": np.float64}[dtype]
    if out is None:
        out = np.empty(int(n), dtype=np_dtype)
    assert out.dtype == np_dtype and out.flags.c_contiguous and out.size == n
    fn = {"f32": lib.synth_fill_f32, "bf16": lib.synth_fill_bf16, "f64": lib.synth_fill_f64}[dtype]
    if n:
        fn(seed, stream, offset, n, kind, p0, p1, out.ctypes.data)
    return out


def words(seed, stream, offset, n):
    out = np.empty(int(n), dtype=np.uint64)
    _load().synth_words(seed, stream, offset, n, out.ctypes.data)
    return out


def f32_to_bf16(x):
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().synth_f32_to_bf16(x.ctypes.data, x.size, out.ctypes.data)
    return out


def bf16_to_f32(bits):
    """Exact widening of bfloat16 bit patterns to float32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclass(frozen=True)
class ScanWorkload:
    """One selective-scan problem: sizes, I/O precision and seed."""
    name: str
    batch: int
    dim: int          # d_inner channels
    seqlen: int
    dstate: int       # N
    io: str           # "f32" or "bf16": dtype of u, Δ_raw, z and y
    seed: int
    d_one: bool = False      # D = 1 instead of U(0.5, 1.5)
    launches: int = 1        # sequence processed in this many launches (state carried)
    sigma_delta: float = 0.5

    @property
    def channel_steps(self) -> int:
        return self.batch * self.dim * self.seqlen


@dataclass(frozen=True)
class DecodeWorkload:
    """Autoregressive decode: ``steps`` single-token state updates."""
    name: str
    batch: int
    dim: int
    dstate: int
    steps: int
    prefill_len: int
    seed: int
    io: str = "bf16"
    sigma_delta: float = 0.5


TINY = ScanWorkload("tiny_s6_fp32", 1, 16, 256, 4, "f32", 0, d_one=True)
MAMBA_130M = ScanWorkload("mamba130m_layer_scan", 8, 1536, 2048, 16, "bf16", 1)
MAMBA_2P8B = ScanWorkload("mamba2p8b_layer_scan", 4, 5120, 4096, 16, "bf16", 2)
MILLION = ScanWorkload("million_length_scan", 1, 1536, 1 << 20, 16, "bf16", 3, launches=16)
DECODE = DecodeWorkload("decode_256x5120", 256, 5120, 16, 1000, 256, 4)

WORKLOADS = {w.name: w for w in (TINY, MAMBA_130M, MAMBA_2P8B, MILLION)}


def scaled(w: ScanWorkload, **kw) -> ScanWorkload:
    """A copy of a workload with some fields replaced (smaller parity cases)."""
    d = dict(w.__dict__)
    d.update(kw)
    return ScanWorkload(**d)


def gen_A(dim, dstate):
    """S4D-Real: A[d, n] = -(n + 1)."""
    return np.ascontiguousarray(np.broadcast_to(-(np.arange(dstate, dtype=np.float32) + 1.0),
                                                (dim, dstate)))


def gen_D(w):
    if w.d_one:
        return np.ones(w.dim, dtype=np.float32)
    return fill(w.seed, S_D, 0, w.dim, UNIFORM, 0.5, 1.5)


def gen_delta_bias(seed, dim):
    """delta_bias = log(expm1(dt)), dt ~ log-uniform[1e-3, 0.1], in double then float."""
    dt = fill(seed, S_DT, 0, dim, LOGUNIFORM, 1e-3, 0.1, dtype="f64")
    return np.log(np.expm1(dt)).astype(np.float32)


def gen_rows(w: ScanWorkload, which: str, b: int, d0: int, nd: int, t0: int = 0, nt=None):
    """Rows [d0, d0+nd) of u / delta / z for batch b, time steps [t0, t0+nt)."""
    nt = w.seqlen - t0 if nt is None else nt
    stream, std = {"u": (S_U, 1.0), "delta": (S_DELTA, w.sigma_delta), "z": (S_Z, 1.0)}[which]
    out = np.empty((nd, nt), dtype=np.float32 if w.io == "f32" else np.uint16)
    for i in range(nd):
        off = ((b * w.dim) + d0 + i) * w.seqlen + t0
        fill(w.seed, stream, off, nt, NORMAL, 0.0, std, dtype=w.io, out=out[i])
    return out


def gen_bc(w: ScanWorkload, which: str, t0: int = 0, nt=None):
    """B or C, shape (batch, N, nt) float32, time steps [t0, t0+nt)."""
    nt = w.seqlen - t0 if nt is None else nt
    stream = S_B if which == "B" else S_C
    out = np.empty((w.batch, w.dstate, nt), dtype=np.float32)
    for b in range(w.batch):
        for n in range(w.dstate):
            off = (b * w.dstate + n) * w.seqlen + t0
            fill(w.seed, stream, off, nt, NORMAL, 0.0, 1.0, out=out[b, n])
    return out


def make_scan_inputs(w: ScanWorkload):
    """All inputs of a scan workload, as numpy arrays in the library's layouts:
    u, delta, z: (batch, dim, L); B, C: (batch, N, L); A: (dim, N);
    D, delta_bias: (dim,)."""
    n = w.batch * w.dim * w.seqlen
    io = w.io
    shape = (w.batch, w.dim, w.seqlen)
    u = fill(w.seed, S_U, 0, n, NORMAL, 0.0, 1.0, dtype=io).reshape(shape)
    delta = fill(w.seed, S_DELTA, 0, n, NORMAL, 0.0, w.sigma_delta, dtype=io).reshape(shape)
    z = fill(w.seed, S_Z, 0, n, NORMAL, 0.0, 1.0, dtype=io).reshape(shape)
    nbc = w.batch * w.dstate * w.seqlen
    B = fill(w.seed, S_B, 0, nbc, NORMAL, 0.0, 1.0).reshape(w.batch, w.dstate, w.seqlen)
    C = fill(w.seed, S_C, 0, nbc, NORMAL, 0.0, 1.0).reshape(w.batch, w.dstate, w.seqlen)
    return dict(u=u, delta=delta, z=z, B=B, C=C, A=gen_A(w.dim, w.dstate), D=gen_D(w),
                delta_bias=gen_delta_bias(w.seed, w.dim))


def make_bwd_inputs(w: ScanWorkload, init_state=True, d_final_state=True):
    """Inputs of the backward pass beyond the forward's: dy ~ N(0, 1) in the workload's
    I/O dtype, (batch, dim, L); d_final_state and init_state ~ N(0, 1) float32,
    (batch, dim, N) (None when not asked for)."""
    n = w.batch * w.dim * w.seqlen
    ns = w.batch * w.dim * w.dstate
    out = dict(dy=fill(w.seed, S_DY, 0, n, NORMAL, 0.0, 1.0, dtype=w.io)
               .reshape(w.batch, w.dim, w.seqlen))
    out["d_final_state"] = (fill(w.seed, S_DFIN, 0, ns, NORMAL, 0.0, 1.0)
                            .reshape(w.batch, w.dim, w.dstate) if d_final_state else None)
    out["init_state"] = (fill(w.seed, S_H0, 0, ns, NORMAL, 0.0, 1.0)
                         .reshape(w.batch, w.dim, w.dstate) if init_state else None)
    return out


def prefill_workload(dw: DecodeWorkload) -> ScanWorkload:
    """The scan whose final state starts the decode: same batch/dim/N, the
    Mamba-2.8B-layer value recipe, ``prefill_len`` steps, the decode seed."""
    return ScanWorkload(dw.name + "_prefill", dw.batch, dw.dim, dw.prefill_len, dw.dstate,
                        dw.io, dw.seed)


def make_decode_step_inputs(dw: DecodeWorkload, step0: int, nsteps: int, b0=0, nb=None,
                            d0=0, nd=None):
    """Per-step decode inputs for steps [step0, step0+nsteps): u, delta, z of
    shape (nsteps, nb, nd) and B, C of shape (nsteps, nb, N)."""
    nb = dw.batch - b0 if nb is None else nb
    nd = dw.dim - d0 if nd is None else nd
    io = dw.io
    np_io = np.float32 if io == "f32" else np.uint16
    out = {k: np.empty((nsteps, nb, nd), dtype=np_io) for k in ("u", "delta", "z")}
    streams = {"u": (S_DEC_U, 1.0), "delta": (S_DEC_DELTA, dw.sigma_delta), "z": (S_DEC_Z, 1.0)}
    for k, (s, std) in streams.items():
        for i in range(nsteps):
            if d0 == 0 and nd == dw.dim:   # whole rows: one contiguous block per step
                off = ((step0 + i) * dw.batch + b0) * dw.dim
                fill(dw.seed, s, off, nb * nd, NORMAL, 0.0, std, dtype=io,
                     out=out[k][i].reshape(-1))
                continue
            for j in range(nb):
                off = ((step0 + i) * dw.batch + b0 + j) * dw.dim + d0
                fill(dw.seed, s, off, nd, NORMAL, 0.0, std, dtype=io, out=out[k][i, j])
    for k, s in (("B", S_DEC_B), ("C", S_DEC_C)):
        arr = np.empty((nsteps, nb, dw.dstate), dtype=np.float32)
        for i in range(nsteps):
            off = ((step0 + i) * dw.batch + b0) * dw.dstate
            fill(dw.seed, s, off, nb * dw.dstate, NORMAL, 0.0, 1.0, out=arr[i].reshape(-1))
        out[k] = arr
    return out
