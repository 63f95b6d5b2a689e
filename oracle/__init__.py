"""fp64 CPU oracle for the selective state-space (S6) scan -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never does, and this
package never imports the CUDA library: the two share no code.

``ssm_oracle.c`` holds the arithmetic (the plain sequential recurrence in
double precision; its header cites the passages it follows).  This module
only marshals numpy arrays into it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssm_oracle.c")
_LIB = os.path.join(_HERE, "libssm_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``libssm_oracle.so`` next to its source (gcc -O2, OpenMP, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        lib.ssm_oracle_scan.argtypes = [i64, i64, i64, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                        i64, vp, i32, vp, i64, vp, vp, i32]
        lib.ssm_oracle_scan.restype = i32
        lib.ssm_oracle_step.argtypes = [i64, i64, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                        i32, vp, vp, i32]
        lib.ssm_oracle_step.restype = i32
        lib.ssm_oracle_scan_bwd.argtypes = [i64, i64, i64, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                            i64, vp, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                            i64, vp, vp, i32]
        lib.ssm_oracle_scan_bwd.restype = i32
        lib.ssm_oracle_conv1d.argtypes = [i64, i64, i64, i32, vp, vp, vp, vp, vp, i32, vp, vp, i32]
        lib.ssm_oracle_conv1d.restype = i32
        lib.ssm_oracle_max_threads.restype = i32
        _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().ssm_oracle_max_threads())


def _ptr(a):
    return None if a is None else a.ctypes.data


def _mode(delta_softplus, euler):
    """The oracle's mode bits: 1 = softplus on Δ, 2 = Euler B̄ = Δ B."""
    return int(bool(delta_softplus)) | (2 if euler else 0)


def _io(arr):
    if arr.dtype == np.uint16:
        return 1
    if arr.dtype == np.float32:
        return 0
    raise TypeError("u/delta/z must be float32 or bfloat16 bits (uint16), got %s" % arr.dtype)


def scan_rows(u, delta, z, unit_b, unit_d, A, B, C, D=None, delta_bias=None,
              delta_softplus=True, init_state=None, y_stride=1, nthreads=0, euler=False):
    """Scan U units given as rows.

    u, delta, z: (U, L) float32 or uint16 (bfloat16 bits); z may be None.
    unit_b, unit_d: (U,) batch / channel of each row.
    A: (dim, N) f32; B, C: (batch, N, L_B) f32 (L_B >= L; time index 0 aligned
    with column 0 of the rows); D, delta_bias: (dim,) f32 or None.
    init_state: (U, N) float64 or None.
    Returns (y, final_state): y is (U, ceil(L / y_stride)) float64 holding
    y_t for t = 0, y_stride, ...; final_state is (U, N) float64.
    """
    u = np.ascontiguousarray(u)
    delta = np.ascontiguousarray(delta)
    U, L = u.shape
    io = _io(u)
    assert delta.shape == u.shape and _io(delta) == io
    if z is not None:
        z = np.ascontiguousarray(z)
        assert z.shape == u.shape and _io(z) == io
    A = np.ascontiguousarray(A, dtype=np.float32)
    N = A.shape[1]
    B = np.ascontiguousarray(B, dtype=np.float32)
    C = np.ascontiguousarray(C, dtype=np.float32)
    assert B.shape == C.shape and B.shape[1] == N and B.shape[2] >= L
    ub = np.ascontiguousarray(unit_b, dtype=np.int64)
    ud = np.ascontiguousarray(unit_d, dtype=np.int64)
    assert ub.shape == (U,) and ud.shape == (U,)
    assert (ub >= 0).all() and (ub < B.shape[0]).all() and (ud >= 0).all() and (ud < A.shape[0]).all()
    D = None if D is None else np.ascontiguousarray(D, dtype=np.float32)
    bias = None if delta_bias is None else np.ascontiguousarray(delta_bias, dtype=np.float32)
    h0 = None
    if init_state is not None:
        h0 = np.ascontiguousarray(init_state, dtype=np.float64)
        assert h0.shape == (U, N)
    ny = (L + y_stride - 1) // y_stride
    y = np.empty((U, ny), dtype=np.float64)
    hN = np.empty((U, N), dtype=np.float64)
    rc = _load().ssm_oracle_scan(U, L, N, io, _ptr(u), _ptr(delta), _ptr(z), _ptr(ub), _ptr(ud),
                                 _ptr(bias), _ptr(A), _ptr(B), _ptr(C), B.shape[2], _ptr(D),
                                 _mode(delta_softplus, euler), _ptr(h0), int(y_stride), _ptr(y),
                                 _ptr(hN), int(nthreads))
    if rc != 0:
        raise ValueError("oracle rejected the arguments (rc=%d)" % rc)
    return y, hN


def scan(u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=True,
         init_state=None, nthreads=0, euler=False):
    """Full scan of (batch, dim, L) inputs.  Returns y (batch, dim, L) and
    final_state (batch, dim, N), both float64."""
    batch, dim, L = u.shape
    N = A.shape[1]
    bb, dd = np.meshgrid(np.arange(batch), np.arange(dim), indexing="ij")
    h0 = None if init_state is None else np.asarray(init_state, np.float64).reshape(batch * dim, N)
    y, hN = scan_rows(u.reshape(batch * dim, L), delta.reshape(batch * dim, L),
                      None if z is None else z.reshape(batch * dim, L), bb.ravel(), dd.ravel(),
                      A, B, C, D, delta_bias, delta_softplus, h0, 1, nthreads, euler)
    return y.reshape(batch, dim, L), hN.reshape(batch, dim, N)


def step(state, u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=True,
         nthreads=0, euler=False):
    """One decode step on (batch, dim, N) float64 state (returned updated, not
    modified in place) with u, delta, z of shape (batch, dim) and B, C of shape
    (batch, N).  Returns (y (batch, dim) float64, new_state)."""
    batch, dim = u.shape
    N = A.shape[1]
    st = np.array(state, dtype=np.float64, copy=True).reshape(batch * dim, N)
    bb, dd = np.meshgrid(np.arange(batch), np.arange(dim), indexing="ij")
    y = np.empty(batch * dim, dtype=np.float64)
    u_ = np.ascontiguousarray(u).reshape(-1)
    io = _io(u_)
    dl = np.ascontiguousarray(delta).reshape(-1)
    zz = None if z is None else np.ascontiguousarray(z).reshape(-1)
    ub = np.ascontiguousarray(bb.ravel(), dtype=np.int64)
    ud = np.ascontiguousarray(dd.ravel(), dtype=np.int64)
    A = np.ascontiguousarray(A, dtype=np.float32)
    B = np.ascontiguousarray(B, dtype=np.float32)
    C = np.ascontiguousarray(C, dtype=np.float32)
    D = None if D is None else np.ascontiguousarray(D, dtype=np.float32)
    bias = None if delta_bias is None else np.ascontiguousarray(delta_bias, dtype=np.float32)
    rc = _load().ssm_oracle_step(batch * dim, N, io, _ptr(u_), _ptr(dl), _ptr(zz), _ptr(ub),
                                 _ptr(ud), _ptr(bias), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                                 _mode(delta_softplus, euler), _ptr(st), _ptr(y), int(nthreads))
    if rc != 0:
        raise ValueError("oracle rejected the arguments (rc=%d)" % rc)
    return y.reshape(batch, dim), st.reshape(batch, dim, N)


def scan_bwd_rows(u, delta, z, unit_b, unit_d, A, B, C, D, delta_bias, delta_softplus,
                  dy, init_state=None, d_final_state=None, nbatch=None, nthreads=0, euler=False):
    """Backward of ``scan_rows`` for U units given as rows (same conventions; every
    row spans the whole time axis, L = u.shape[1]).

    dy: (U, L) upstream derivative of y; d_final_state: (U, N) or None.
    Returns a dict of float64 arrays: du, ddelta, dz (U, L; dz None without z);
    dA_unit (U, N), dD_unit (U,), dbias_unit (U,), dinit (U, N): per-unit terms
    (sum them by channel for the parameter gradients); dB, dC (nbatch, N, L):
    summed over the given units of each batch."""
    u = np.ascontiguousarray(u)
    delta = np.ascontiguousarray(delta)
    U, L = u.shape
    io = _io(u)
    assert delta.shape == u.shape and _io(delta) == io
    if z is not None:
        z = np.ascontiguousarray(z)
        assert z.shape == u.shape and _io(z) == io
    A = np.ascontiguousarray(A, dtype=np.float32)
    N = A.shape[1]
    B = np.ascontiguousarray(B, dtype=np.float32)
    C = np.ascontiguousarray(C, dtype=np.float32)
    assert B.shape == C.shape and B.shape[1] == N and B.shape[2] >= L
    nbatch = B.shape[0] if nbatch is None else nbatch
    ub = np.ascontiguousarray(unit_b, dtype=np.int64)
    ud = np.ascontiguousarray(unit_d, dtype=np.int64)
    assert ub.shape == (U,) and ud.shape == (U,)
    assert (ud >= 0).all() and (ud < A.shape[0]).all()
    D = None if D is None else np.ascontiguousarray(D, dtype=np.float32)
    bias = None if delta_bias is None else np.ascontiguousarray(delta_bias, dtype=np.float32)
    h0 = None if init_state is None else np.ascontiguousarray(init_state, dtype=np.float64)
    dfin = None if d_final_state is None else np.ascontiguousarray(d_final_state, dtype=np.float64)
    assert h0 is None or h0.shape == (U, N)
    assert dfin is None or dfin.shape == (U, N)
    dy = np.ascontiguousarray(dy, dtype=np.float64)
    assert dy.shape == (U, L)
    out = dict(du=np.empty((U, L)), ddelta=np.empty((U, L)),
               dz=None if z is None else np.empty((U, L)),
               dA_unit=np.empty((U, N)), dD_unit=np.empty(U), dbias_unit=np.empty(U),
               dinit=np.empty((U, N)), dB=np.empty((nbatch, N, L)), dC=np.empty((nbatch, N, L)))
    rc = _load().ssm_oracle_scan_bwd(
        U, L, N, io, _ptr(u), _ptr(delta), _ptr(z), _ptr(ub), _ptr(ud), _ptr(bias), _ptr(A),
        _ptr(B), _ptr(C), B.shape[2], _ptr(D), _mode(delta_softplus, euler), _ptr(h0), _ptr(dy),
        _ptr(dfin), _ptr(out["du"]), _ptr(out["ddelta"]), _ptr(out["dz"]), _ptr(out["dA_unit"]),
        _ptr(out["dD_unit"]), _ptr(out["dbias_unit"]), _ptr(out["dinit"]), nbatch,
        _ptr(out["dB"]), _ptr(out["dC"]), int(nthreads))
    if rc != 0:
        raise ValueError("oracle rejected the arguments (rc=%d)" % rc)
    return out


def scan_bwd(u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=True,
             init_state=None, dy=None, d_final_state=None, nthreads=0, euler=False):
    """Backward of ``scan`` for (batch, dim, L) inputs: the derivatives of
    Σ y·dy + Σ final_state·d_final_state.  Returns float64 arrays du, ddelta,
    dz (batch, dim, L), dA (dim, N), dB, dC (batch, N, L), dD, dbias (dim,) and
    dinit (batch, dim, N)."""
    batch, dim, L = u.shape
    N = A.shape[1]
    bb, dd = np.meshgrid(np.arange(batch), np.arange(dim), indexing="ij")
    U = batch * dim
    r = scan_bwd_rows(u.reshape(U, L), delta.reshape(U, L),
                      None if z is None else z.reshape(U, L), bb.ravel(), dd.ravel(), A, B, C, D,
                      delta_bias, delta_softplus, np.asarray(dy, np.float64).reshape(U, L),
                      None if init_state is None else np.asarray(init_state).reshape(U, N),
                      None if d_final_state is None else np.asarray(d_final_state).reshape(U, N),
                      batch, nthreads, euler)
    return dict(du=r["du"].reshape(batch, dim, L), ddelta=r["ddelta"].reshape(batch, dim, L),
                dz=None if z is None else r["dz"].reshape(batch, dim, L),
                dA=r["dA_unit"].reshape(batch, dim, N).sum(0),
                dD=r["dD_unit"].reshape(batch, dim).sum(0),
                dbias=r["dbias_unit"].reshape(batch, dim).sum(0),
                dinit=r["dinit"].reshape(batch, dim, N), dB=r["dB"], dC=r["dC"])


def conv1d(x, weight, bias=None, state_in=None, silu=True, nthreads=0):
    """Causal depthwise conv1d (+ SiLU) of x (batch, dim, L) (float32 or bfloat16 bits)
    with weight (dim, K) and bias (dim,); state_in (batch, dim, K-1) float64 or None
    holds the K-1 inputs before the sequence.  Returns (out (batch, dim, L) float64,
    state_out (batch, dim, K-1) float64: the last K-1 inputs)."""
    x = np.ascontiguousarray(x)
    batch, dim, L = x.shape
    io = _io(x)
    w = np.ascontiguousarray(weight, dtype=np.float32)
    K = w.shape[1]
    assert w.shape == (dim, K)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    st = None if state_in is None else np.ascontiguousarray(state_in, dtype=np.float64)
    assert st is None or st.shape == (batch, dim, K - 1)
    ud = np.ascontiguousarray(np.tile(np.arange(dim, dtype=np.int64), batch))
    out = np.empty((batch, dim, L))
    sout = np.empty((batch, dim, max(K - 1, 0)))
    rc = _load().ssm_oracle_conv1d(batch * dim, L, K, io, _ptr(x), _ptr(ud), _ptr(w), _ptr(b),
                                   _ptr(st), int(bool(silu)), _ptr(out),
                                   _ptr(sout) if K > 1 else None, int(nthreads))
    if rc != 0:
        raise ValueError("oracle rejected the arguments (rc=%d)" % rc)
    return out, sout


def _f64(arr):
    """float32 or bfloat16 bits (uint16) -> float64 (bf16 decoded exactly)."""
    arr = np.ascontiguousarray(arr)
    if arr.dtype == np.uint16:
        return (arr.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return arr.astype(np.float64)


def conv1d_bwd(x, weight, bias, state_in, silu, dout):
    """Derivatives of ``conv1d``'s output against a cotangent ``dout`` (batch, dim, L)
    (the causal depthwise conv1d + SiLU of the summary page's section 4a shape
    table, width d_conv of the configuration page), by the chain rule in fp64:

        p_t = bias + Σ_k w[k] x[t-(K-1)+k]     (x before the sequence from state_in)
        g_t = dout_t · silu'(p_t),   silu'(p) = σ(p) (1 + p (1 - σ(p)))   (g = dout without SiLU)
        dx[s]     = Σ_k w[k] g[s+(K-1)-k]      for every input position s, the K-1
                                               before the sequence giving d state_in
        dw[d,k]   = Σ_{b,t} g[b,d,t] x[b,d,t-(K-1)+k]
        dbias[d]  = Σ_{b,t} g[b,d,t]

    Returns dict(dx (batch, dim, L), dweight (dim, K), dbias (dim,),
    dstate (batch, dim, K-1)), all float64."""
    xf = _f64(x)
    batch, dim, L = xf.shape
    w = np.asarray(weight, dtype=np.float64)
    K = w.shape[1]
    st = np.zeros((batch, dim, K - 1)) if state_in is None else np.asarray(state_in, dtype=np.float64)
    xp = np.concatenate([st, xf], axis=2)          # input positions -(K-1) .. L-1
    p = np.zeros((batch, dim, L))
    for k in range(K):
        p += w[None, :, k, None] * xp[:, :, k:k + L]
    if bias is not None:
        p += np.asarray(bias, dtype=np.float64)[None, :, None]
    g = _f64(dout)
    if silu:
        sg = 1.0 / (1.0 + np.exp(-p))
        g = g * sg * (1.0 + p * (1.0 - sg))
    dxp = np.zeros_like(xp)
    dw = np.zeros((dim, K))
    for k in range(K):
        dxp[:, :, k:k + L] += w[None, :, k, None] * g
        dw[:, k] = np.sum(g * xp[:, :, k:k + L], axis=(0, 2))
    return dict(dx=dxp[:, :, K - 1:], dweight=dw, dbias=np.sum(g, axis=(0, 2)),
                dstate=dxp[:, :, :K - 1])


def ssd(x, dt, A, B, C, D=None, z=None, dt_bias=None, delta_softplus=True, init_state=None,
        euler=False, nthreads=0):
    """Mamba-2's scalar-A state space model ([C] §5.1: A_t = a_t I per head), by its
    plain recurrence: the selective scan of every channel p of head h with
    A[n] = A[h] for all n, the head's step Δ_t shared by its P channels, and the B, C of
    the head's group.  The recurrence is the scan oracle's, unchanged.

    x, z: (batch, L, H, P) float32 or bfloat16 bits; dt: (batch, L, H) same dtype;
    A, D, dt_bias: (H,) float32; B, C: (batch, L, G, N) float32; init_state:
    (batch, H, P, N) float64 or None.  Returns y (batch, L, H, P) float64 and the final
    state (batch, H, P, N) float64."""
    x = np.asarray(x)
    batch, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    assert H % G == 0 and dt.shape == (batch, L, H) and C.shape == B.shape
    hpg = H // G
    # rows: unit (b, h, p); its u is x[b, :, h, p], its Δ row dt[b, :, h]
    u = np.ascontiguousarray(np.transpose(x, (0, 2, 3, 1)).reshape(batch * H * P, L))
    dl = np.ascontiguousarray(np.repeat(np.transpose(np.asarray(dt), (0, 2, 1)), P, axis=1)
                              .reshape(batch * H * P, L))
    zz = None if z is None else np.ascontiguousarray(
        np.transpose(np.asarray(z), (0, 2, 3, 1)).reshape(batch * H * P, L))
    bb, hh, pp = np.meshgrid(np.arange(batch), np.arange(H), np.arange(P), indexing="ij")
    unit_b = (bb * G + hh // hpg).ravel()             # one "batch row" of B, C per group
    unit_d = (hh * P + pp).ravel()                     # channel d = h P + p
    A_tab = np.repeat(np.asarray(A, np.float32), P)[:, None].repeat(N, axis=1)
    Bt = np.ascontiguousarray(np.transpose(np.asarray(B, np.float32), (0, 2, 3, 1))
                              .reshape(batch * G, N, L))
    Ct = np.ascontiguousarray(np.transpose(np.asarray(C, np.float32), (0, 2, 3, 1))
                              .reshape(batch * G, N, L))
    D_tab = None if D is None else np.repeat(np.asarray(D, np.float32), P)
    bias_tab = None if dt_bias is None else np.repeat(np.asarray(dt_bias, np.float32), P)
    h0 = None if init_state is None else np.asarray(init_state, np.float64).reshape(batch * H * P, N)
    y, hN = scan_rows(u, dl, zz, unit_b, unit_d, A_tab, Bt, Ct, D_tab, bias_tab, delta_softplus,
                      h0, 1, nthreads, euler)
    y = np.transpose(y.reshape(batch, H, P, L), (0, 3, 1, 2))
    return y, hN.reshape(batch, H, P, N)


def ssd_bwd(x, dt, A, B, C, D=None, z=None, dt_bias=None, delta_softplus=True, init_state=None,
            dy=None, d_final_state=None, euler=False, nthreads=0):
    """Backward of ``ssd``: the derivatives of Σ y·dy + Σ final_state·d_final_state.
    As ``ssd`` is the selective scan of every channel (b, h, p) with the head's
    scalar A, step and D and the group's B, C tied across channels, its derivatives
    are the scan backward's per-channel terms summed over the channels that share
    each parameter: the head's P channels for d dt, dA, dD, d dt_bias; the group's
    heads and channels for dB, dC (the scan backward sums a batch row's units).

    Inputs as ``ssd``; dy (batch, L, H, P), d_final_state (batch, H, P, N) or None.
    Returns float64 dx, dz (batch, L, H, P; dz None without z), ddt (batch, L, H),
    dA, dD, ddt_bias (H,), dB, dC (batch, L, G, N), dinit (batch, H, P, N)."""
    x = np.asarray(x)
    batch, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    assert H % G == 0 and dt.shape == (batch, L, H) and C.shape == B.shape
    hpg = H // G
    U = batch * H * P
    rows = lambda a: np.ascontiguousarray(np.transpose(np.asarray(a), (0, 2, 3, 1)).reshape(U, L))
    u = rows(x)
    dl = np.ascontiguousarray(np.repeat(np.transpose(np.asarray(dt), (0, 2, 1)), P, axis=1)
                              .reshape(U, L))
    zz = None if z is None else rows(z)
    bb, hh, pp = np.meshgrid(np.arange(batch), np.arange(H), np.arange(P), indexing="ij")
    unit_b = (bb * G + hh // hpg).ravel()
    unit_d = (hh * P + pp).ravel()
    A_tab = np.repeat(np.asarray(A, np.float32), P)[:, None].repeat(N, axis=1)
    Bt = np.ascontiguousarray(np.transpose(np.asarray(B, np.float32), (0, 2, 3, 1)).reshape(batch * G, N, L))
    Ct = np.ascontiguousarray(np.transpose(np.asarray(C, np.float32), (0, 2, 3, 1)).reshape(batch * G, N, L))
    D_tab = None if D is None else np.repeat(np.asarray(D, np.float32), P)
    bias_tab = None if dt_bias is None else np.repeat(np.asarray(dt_bias, np.float32), P)
    h0 = None if init_state is None else np.asarray(init_state, np.float64).reshape(U, N)
    dfin = None if d_final_state is None else np.asarray(d_final_state, np.float64).reshape(U, N)
    r = scan_bwd_rows(u, dl, zz, unit_b, unit_d, A_tab, Bt, Ct, D_tab, bias_tab, delta_softplus,
                      rows(np.asarray(dy, np.float64)), h0, dfin, batch * G, nthreads, euler)
    back = lambda a: np.transpose(a.reshape(batch, H, P, L), (0, 3, 1, 2))
    per_head = lambda a: a.reshape(batch, H, P, -1).sum(axis=(0, 2, 3))
    bc = lambda a: np.transpose(a.reshape(batch, G, N, L), (0, 3, 1, 2))
    return dict(dx=back(r["du"]), dz=None if z is None else back(r["dz"]),
                ddt=np.transpose(r["ddelta"].reshape(batch, H, P, L).sum(axis=2), (0, 2, 1)),
                dA=per_head(r["dA_unit"]), dD=per_head(r["dD_unit"]),
                ddt_bias=per_head(r["dbias_unit"]), dB=bc(r["dB"]), dC=bc(r["dC"]),
                dinit=r["dinit"].reshape(batch, H, P, N))


def rel_err(got, ref):
    """max |got - ref| / max |ref|: the parity metric for y and final_state."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.max(np.abs(ref)) if ref.size else 0.0
    num = np.max(np.abs(got - ref)) if ref.size else 0.0
    if den == 0.0:
        return float(num)
    return float(num / den)


def scan_complex(u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=True,
                 init_state=None, euler=False):
    """The selective scan with a complex diagonal A (and complex B, C), in complex128.

    The summary page ("Mamba: Linear-Time Sequence Modeling") names complex S4 only as
    an ablation row (§5.4) and defines no complex form, so this is the plainest
    reading of its equations (2) and (4) over complex numbers, for each (b, d):
        Δ_t = softplus(delta_t + bias_d) (or delta_t + bias_d),
        Ā = exp(Δ A_{d,n}),  B̄ = (Ā - 1)/A_{d,n} (A = 0: Δ; Euler flag: Δ),
        h_t = Ā h_{t-1} + B̄ B_{b,n,t} u_t,
        y_t = Re(Σ_n C_{b,n,t} h_t[n]) + D_d u_t, then · silu(z_t),
    the real part taken once, without doubling for conjugate pairs (a caller who
    keeps one state of each conjugate pair doubles C).

    u, delta, z: (batch, dim, L) float32 or bfloat16 bits; A: (dim, N) complex;
    B, C: (batch, N, L) complex; D, delta_bias: (dim,) or None; init_state:
    (batch, dim, N) complex or None.  Returns y (batch, dim, L) float64 and the
    final state (batch, dim, N) complex128."""
    u64 = _f64(u)
    d64 = _f64(delta)
    z64 = None if z is None else _f64(z)
    batch, dim, L = u64.shape
    A = np.asarray(A, dtype=np.complex128)
    N = A.shape[1]
    B = np.asarray(B, dtype=np.complex128)
    C = np.asarray(C, dtype=np.complex128)
    bias = np.zeros(dim) if delta_bias is None else np.asarray(delta_bias, np.float64)
    Dv = np.zeros(dim) if D is None else np.asarray(D, np.float64)
    h = (np.zeros((batch, dim, N), np.complex128) if init_state is None
         else np.array(init_state, dtype=np.complex128))
    y = np.empty((batch, dim, L))
    zero = A == 0
    Asafe = np.where(zero, 1.0, A)
    for t in range(L):
        x = d64[:, :, t] + bias[None, :]
        if delta_softplus:
            dt = np.where(x > 0, x + np.log1p(np.exp(-np.abs(x))), np.log1p(np.exp(np.minimum(x, 0))))
        else:
            dt = x
        dA = dt[:, :, None] * A[None, :, :]
        Abar = np.exp(dA)
        if euler:
            Bbar = np.broadcast_to(dt[:, :, None], dA.shape).astype(np.complex128)
        else:
            Bbar = np.where(zero[None], dt[:, :, None], np.expm1(dA) / Asafe[None])
        h = Abar * h + Bbar * B[:, None, :, t] * u64[:, :, t][:, :, None]
        yt = np.real(np.sum(C[:, None, :, t] * h, axis=2)) + Dv[None, :] * u64[:, :, t]
        if z64 is not None:
            zt = z64[:, :, t]
            yt = yt * (zt / (1.0 + np.exp(-zt)))
        y[:, :, t] = yt
    return y, h
