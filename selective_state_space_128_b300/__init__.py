"""Python binding of libssm, the B300 selective state-space (S6) scan library.

Every entry point of ``include/ssm.h`` has a function of the same name here that
only marshals arguments (tensor -> device pointer, shape -> sizes, current
stream) and raises :class:`SSMError` on a non-zero status.  All arithmetic runs
in the CUDA kernels of ``libssm.so``; there is no CPU path.  PyTorch is used
only for device memory and streams.

    y, h = scan(u, delta, A, B, C, D, z, delta_bias)          # allocating helper
    ssm_scan_fwd(u, delta, delta_bias, A, B, C, D, z, True, y, h)
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libssm.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "ssm.h")

SSM_F32, SSM_BF16 = 0, 1
SSM_OK = 0
SSM_ERR_ARG, SSM_ERR_ALIGN, SSM_ERR_UNSUPPORTED, SSM_ERR_CUDA, SSM_ERR_WORKSPACE = -1, -2, -3, -4, -5
SSM_ERR_TIMEOUT = -6
SSM_SOFTPLUS, SSM_EULER_B, SSM_SAVED_STATES, SSM_LAYOUT_BLD = 1, 2, 4, 8
SSM_TEST_STALL = 16
SCAN_STATUS_BYTES = 256   # the status header at the start of a scan workspace

_lib = None


class SSMError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__("%s: %s" % (where, strerror(status)))
        self.status = status


def load():
    """Load libssm.so (built in-tree by ``python -m selective_state_space_128_b300.build``).
    Raises if it is missing: there is no fallback implementation."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("libssm.so is not built (%s); run `python -m "
                           "selective_state_space_128_b300.build`" % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    lib.ssm_strerror.argtypes = [i32]
    lib.ssm_strerror.restype = ctypes.c_char_p
    lib.ssm_version.argtypes = []
    lib.ssm_version.restype = ctypes.c_char_p
    lib.ssm_scan_fwd.argtypes = [vp] * 8 + [i32, vp, vp, i64, i64, i64, i64, i32]
    lib.ssm_scan_fwd.restype = i32
    lib.ssm_scan_workspace_bytes.argtypes = [i64, i64, i64, i64, i32]
    lib.ssm_scan_workspace_bytes.restype = sz
    lib.ssm_scan_fwd_ex.argtypes = [vp] * 8 + [i32, vp, vp, i64, i64, i64, i64, i32, vp, vp, sz, vp]
    lib.ssm_scan_fwd_ex.restype = i32
    lib.ssm_state_update.argtypes = [vp] * 9 + [i64, i64, i64, i32]
    lib.ssm_state_update.restype = i32
    lib.ssm_state_update_ex.argtypes = [vp, vp, vp, vp, i32] + [vp] * 6 + [i64, i64, i64, i32, vp]
    lib.ssm_state_update_ex.restype = i32
    lib.ssm_scan_fwd_strided.argtypes = [vp] * 8 + [i32, vp, vp, i64, i64, i64, i64, i32, vp, vp,
                                                     vp, sz, vp]
    lib.ssm_scan_fwd_strided.restype = i32
    lib.ssm_scan_fwd_complex.argtypes = [vp] * 8 + [i32, vp, vp, vp, i64, i64, i64, i64, i32, vp]
    lib.ssm_scan_fwd_complex.restype = i32
    lib.ssm_scan_fwd_noalloc.argtypes = [vp] * 8 + [i32, vp, vp, i64, i64, i64, i64, i32, vp, vp]
    lib.ssm_scan_fwd_noalloc.restype = i32
    lib.ssm_status.argtypes = [vp, vp]
    lib.ssm_status.restype = i32
    lib.ssm_set_test_mode.argtypes = [i32, i64, i64, i32]
    lib.ssm_set_test_mode.restype = i32
    lib.ssm_scan_bwd_workspace_bytes.argtypes = [i64, i64, i64, i64]
    lib.ssm_scan_bwd_workspace_bytes.restype = sz
    lib.ssm_scan_bwd.argtypes = [vp] * 8 + [i32] + [vp] * 12 + [i64, i64, i64, i64, i32, vp, sz, vp]
    lib.ssm_scan_bwd.restype = i32
    lib.ssm_scan_fwd_train.argtypes = [vp] * 8 + [i32, vp, vp, i64, i64, i64, i64, i32, vp, vp, sz,
                                                   vp, sz, vp]
    lib.ssm_scan_fwd_train.restype = i32
    lib.ssm_ssd_workspace_bytes.argtypes = [i64, i64, i64, i64, i64, i64]
    lib.ssm_ssd_workspace_bytes.restype = sz
    lib.ssm_ssd_fwd.argtypes = [vp] * 8 + [i32, vp, vp, vp, i64, i64, i64, i64, i64, i64, vp, sz, vp]
    lib.ssm_ssd_fwd.restype = i32
    lib.ssm_conv1d_fwd.argtypes = [vp, vp, vp, vp, i32, vp, vp, i64, i64, i64, i64, i32, vp]
    lib.ssm_conv1d_fwd.restype = i32
    lib.ssm_conv1d_update.argtypes = [vp, vp, vp, vp, i32, vp, i64, i64, i64, i32, vp]
    lib.ssm_conv1d_update.restype = i32
    lib.ssm_ssd_bwd_workspace_bytes.argtypes = [i64, i64, i64, i64, i64, i64]
    lib.ssm_ssd_bwd_workspace_bytes.restype = sz
    lib.ssm_ssd_bwd.argtypes = [vp] * 8 + [i32] + [vp] * 12 + [i64] * 6 + [vp, sz, vp]
    lib.ssm_ssd_bwd.restype = i32
    lib.ssm_conv1d_bwd.argtypes = [vp, vp, vp, vp, i32, vp, vp, vp, vp, vp, i64, i64, i64, i64, i32,
                                   vp]
    lib.ssm_conv1d_bwd.restype = i32
    lib.ssm_scan_fwd_host_workspace_bytes.argtypes = [i64, i64, i64, i64, i32, i32]
    lib.ssm_scan_fwd_host_workspace_bytes.restype = sz
    lib.ssm_scan_fwd_host.argtypes = [vp] * 8 + [i32, vp, vp, vp, i64, i64, i64, i64, i32, vp, sz, vp]
    lib.ssm_scan_fwd_host.restype = i32
    _lib = lib
    return lib


def strerror(status: int) -> str:
    return load().ssm_strerror(int(status)).decode()


def version() -> str:
    return load().ssm_version().decode()


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------

def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _io_dtype(t):
    import torch
    if t.dtype == torch.bfloat16:
        return SSM_BF16
    if t.dtype == torch.float32:
        return SSM_F32
    raise TypeError("u/delta/z/y must be float32 or bfloat16, got %s" % t.dtype)


def _stream(stream):
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check_dev(*ts):
    for t in ts:
        if t is None or isinstance(t, int):
            continue
        if not t.is_cuda:
            raise ValueError("libssm takes device tensors; got a tensor on %s" % t.device)
        if not t.is_contiguous():
            raise ValueError("libssm takes contiguous tensors")


def _check_dev_strided(*ts):
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("libssm takes device tensors; got a tensor on %s" % t.device)
        if t.dim() != 3:
            raise ValueError("strided views are (batch, dim, L)")


def _check_host(*ts):
    for t in ts:
        if t is None or isinstance(t, int):
            continue
        if t.is_cuda:
            raise ValueError("ssm_scan_fwd_host takes host tensors; got one on %s" % t.device)
        if not t.is_contiguous():
            raise ValueError("libssm takes contiguous tensors")


def _flags(delta_softplus, euler=False, bld=False):
    """The delta_softplus flag word: a bool (softplus on/off) or the int bits
    SSM_SOFTPLUS | SSM_EULER_B | SSM_LAYOUT_BLD; `euler` and `bld` add their bits."""
    return (int(delta_softplus) | (SSM_EULER_B if euler else 0)
            | (SSM_LAYOUT_BLD if bld else 0))


def _sizes(u, A, B):
    """(batch, dim, L) from A (dim, N) and B (batch, N, L): the same for both layouts
    of u ((batch, dim, L), or (batch, L, dim) with SSM_LAYOUT_BLD)."""
    return int(B.shape[0]), int(A.shape[0]), int(B.shape[2])


def _call(name, rc):
    if rc != SSM_OK:
        raise SSMError(rc, name)


# ---------------------------------------------------------------------------
# entry points (same names and argument order as include/ssm.h)
# ---------------------------------------------------------------------------

def ssm_scan_fwd(u, delta, delta_bias, A, B, C, D, z, delta_softplus, y, final_state):
    """Tensor form of ``ssm_scan_fwd``: sizes come from u (batch, dim, L) and A (dim, N);
    runs on the legacy default stream like the C entry point."""
    _check_dev(u, delta, delta_bias, A, B, C, D, z, y, final_state)
    batch, dim, L = _sizes(u, A, B)
    N = A.shape[1]
    rc = load().ssm_scan_fwd(_ptr(u), _ptr(delta), _ptr(delta_bias), _ptr(A), _ptr(B), _ptr(C),
                             _ptr(D), _ptr(z), _flags(delta_softplus), _ptr(y),
                             _ptr(final_state), batch, dim, L, N, _io_dtype(u))
    _call("ssm_scan_fwd", rc)


def ssm_scan_workspace_bytes(batch, dim, seqlen, dstate, io_dtype) -> int:
    return int(load().ssm_scan_workspace_bytes(batch, dim, seqlen, dstate, io_dtype))


def ssm_scan_fwd_ex(u, delta, delta_bias, A, B, C, D, z, delta_softplus, y, final_state,
                    init_state=None, workspace=None, workspace_bytes=None, stream=None):
    """Tensor form of ``ssm_scan_fwd_ex`` on the current torch stream (or ``stream``)."""
    _check_dev(u, delta, delta_bias, A, B, C, D, z, y, final_state, init_state, workspace)
    batch, dim, L = _sizes(u, A, B)
    N = A.shape[1]
    if workspace is not None and workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    rc = load().ssm_scan_fwd_ex(_ptr(u), _ptr(delta), _ptr(delta_bias), _ptr(A), _ptr(B),
                                _ptr(C), _ptr(D), _ptr(z), _flags(delta_softplus), _ptr(y),
                                _ptr(final_state), batch, dim, L, N, _io_dtype(u),
                                _ptr(init_state), _ptr(workspace), int(workspace_bytes or 0),
                                _stream(stream))
    _call("ssm_scan_fwd_ex", rc)


def ssm_scan_fwd_strided(u, delta, delta_bias, A, B, C, D, z, delta_softplus, y, final_state,
                         init_state=None, workspace=None, workspace_bytes=None, stream=None):
    """Tensor form of ``ssm_scan_fwd_strided``: u, delta, z, y are (batch, dim, L) views
    with any element strides (``tensor.stride()``); sizes from u, A and B."""
    _check_dev_strided(u, delta, z, y)
    _check_dev(delta_bias, A, B, C, D, final_state, init_state, workspace)
    batch, dim, L = int(u.shape[0]), int(u.shape[1]), int(u.shape[2])
    N = A.shape[1]
    if workspace is not None and workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    st = (ctypes.c_int64 * 12)(*(list(u.stride()) + list(delta.stride())
                                 + list(z.stride() if z is not None else (0, 0, 0))
                                 + list(y.stride())))
    rc = load().ssm_scan_fwd_strided(_ptr(u), _ptr(delta), _ptr(delta_bias), _ptr(A), _ptr(B),
                                     _ptr(C), _ptr(D), _ptr(z), _flags(delta_softplus), _ptr(y),
                                     _ptr(final_state), batch, dim, L, N, _io_dtype(u),
                                     ctypes.cast(st, ctypes.c_void_p), _ptr(init_state),
                                     _ptr(workspace), int(workspace_bytes or 0), _stream(stream))
    _call("ssm_scan_fwd_strided", rc)


def ssm_scan_fwd_host_workspace_bytes(batch, dim, seqlen, dstate, io_dtype, flags=0) -> int:
    return int(load().ssm_scan_fwd_host_workspace_bytes(batch, dim, seqlen, dstate, io_dtype,
                                                         int(flags)))


def ssm_scan_fwd_host(u, delta, delta_bias, A, B, C, D, z, flags, y, final_state, init_state,
                      workspace, workspace_bytes, stream=None):
    """Tensor form of ``ssm_scan_fwd_host``: every tensor but the (device) workspace
    lives in host memory (page-locked for overlapped copies); sizes as ssm_scan_fwd_ex."""
    _check_host(u, delta, delta_bias, A, B, C, D, z, y, final_state, init_state)
    _check_dev(workspace)
    batch, dim, L = _sizes(u, A, B)
    N = A.shape[1]
    rc = load().ssm_scan_fwd_host(_ptr(u), _ptr(delta), _ptr(delta_bias), _ptr(A), _ptr(B),
                                  _ptr(C), _ptr(D), _ptr(z), int(flags), _ptr(y),
                                  _ptr(final_state), _ptr(init_state), batch, dim, L, N,
                                  _io_dtype(u), _ptr(workspace), int(workspace_bytes or 0),
                                  _stream(stream))
    _call("ssm_scan_fwd_host", rc)


def ssm_scan_fwd_train(u, delta, delta_bias, A, B, C, D, z, delta_softplus, y, final_state,
                       init_state, workspace, workspace_bytes, bwd_workspace, bwd_workspace_bytes,
                       stream=None):
    """Tensor form of ``ssm_scan_fwd_train`` (the forward that saves the backward's
    chunk-start states into ``bwd_workspace``)."""
    _check_dev(u, delta, delta_bias, A, B, C, D, z, y, final_state, init_state, workspace,
               bwd_workspace)
    batch, dim, L = _sizes(u, A, B)
    N = A.shape[1]
    rc = load().ssm_scan_fwd_train(_ptr(u), _ptr(delta), _ptr(delta_bias), _ptr(A), _ptr(B),
                                   _ptr(C), _ptr(D), _ptr(z), _flags(delta_softplus), _ptr(y),
                                   _ptr(final_state), batch, dim, L, N, _io_dtype(u),
                                   _ptr(init_state), _ptr(workspace), int(workspace_bytes or 0),
                                   _ptr(bwd_workspace), int(bwd_workspace_bytes or 0),
                                   _stream(stream))
    _call("ssm_scan_fwd_train", rc)


def ssm_status(workspace=None, stream=None) -> int:
    """Synchronise the stream and return the device-side status (SSM_OK or
    SSM_ERR_TIMEOUT) of the last scan call on ``workspace`` (its status word), or,
    with no workspace, of the calls made without one (the library-wide word, read
    and cleared)."""
    if workspace is not None:
        _check_dev(workspace)
    return int(load().ssm_status(_ptr(workspace), _stream(stream)))


SCAN_KERNEL_AUTO, SCAN_KERNEL_BLOCK, SCAN_KERNEL_PAIR = 0, 1, 2


def ssm_set_test_mode(enable, wait_limit_ns=1000000, noalloc_limit_bytes=0,
                      scan_kernel=SCAN_KERNEL_AUTO) -> None:
    """Form of ``ssm_set_test_mode`` (the test mode: failure path, scratch limit,
    forward scan kernel choice)."""
    _call("ssm_set_test_mode", load().ssm_set_test_mode(int(bool(enable)), int(wait_limit_ns),
                                                        int(noalloc_limit_bytes),
                                                        int(scan_kernel)))


def ssm_state_update(state, u, delta, A, B, C, D, z, y):
    """Tensor form of ``ssm_state_update`` (Δ = delta as given), legacy default stream."""
    _check_dev(state, u, delta, A, B, C, D, z, y)
    batch, dim = u.shape
    N = A.shape[1]
    rc = load().ssm_state_update(_ptr(state), _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C),
                                 _ptr(D), _ptr(z), _ptr(y), batch, dim, N, _io_dtype(u))
    _call("ssm_state_update", rc)


def ssm_state_update_ex(state, u, delta, delta_bias, delta_softplus, A, B, C, D, z, y,
                        stream=None):
    """Tensor form of ``ssm_state_update_ex`` on the current torch stream (or ``stream``)."""
    _check_dev(state, u, delta, delta_bias, A, B, C, D, z, y)
    batch, dim = u.shape
    N = A.shape[1]
    rc = load().ssm_state_update_ex(_ptr(state), _ptr(u), _ptr(delta), _ptr(delta_bias),
                                    _flags(delta_softplus), _ptr(A), _ptr(B), _ptr(C),
                                    _ptr(D), _ptr(z), _ptr(y), batch, dim, N, _io_dtype(u),
                                    _stream(stream))
    _call("ssm_state_update_ex", rc)


def ssm_scan_fwd_noalloc(u, delta, delta_bias, A, B, C, D, z, delta_softplus, y, final_state,
                         init_state=None, stream=None):
    """Tensor form of ``ssm_scan_fwd_noalloc``: as ``ssm_scan_fwd_ex`` without a workspace;
    the library's fixed scratch array (SSM_STATIC_SCRATCH_BYTES per GPU) stands in for it,
    for callers that cannot allocate device memory.  Calls that may overlap on the GPU
    share that array and must be ordered (e.g. issued on one stream)."""
    _check_dev(u, delta, delta_bias, A, B, C, D, z, y, final_state, init_state)
    batch, dim, L = _sizes(u, A, B)
    N = A.shape[1]
    rc = load().ssm_scan_fwd_noalloc(_ptr(u), _ptr(delta), _ptr(delta_bias), _ptr(A), _ptr(B),
                                     _ptr(C), _ptr(D), _ptr(z), _flags(delta_softplus),
                                     _ptr(y), _ptr(final_state), batch, dim, L, N,
                                     _io_dtype(u), _ptr(init_state), _stream(stream))
    _call("ssm_scan_fwd_noalloc", rc)


def ssm_scan_bwd_workspace_bytes(batch, dim, seqlen, dstate) -> int:
    return int(load().ssm_scan_bwd_workspace_bytes(batch, dim, seqlen, dstate))


def ssm_scan_bwd(u, delta, delta_bias, A, B, C, D, z, delta_softplus, init_state, dy,
                 d_final_state, du, ddelta, dA, dB, dC, dD, dz, d_delta_bias, d_init_state,
                 workspace, workspace_bytes=None, stream=None):
    """Tensor form of ``ssm_scan_bwd`` on the current torch stream (or ``stream``)."""
    _check_dev(u, delta, delta_bias, A, B, C, D, z, init_state, dy, d_final_state, du, ddelta,
               dA, dB, dC, dD, dz, d_delta_bias, d_init_state, workspace)
    batch, dim, L = _sizes(u, A, B)
    N = A.shape[1]
    if workspace is not None and workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    rc = load().ssm_scan_bwd(_ptr(u), _ptr(delta), _ptr(delta_bias), _ptr(A), _ptr(B), _ptr(C),
                             _ptr(D), _ptr(z), _flags(delta_softplus), _ptr(init_state),
                             _ptr(dy), _ptr(d_final_state), _ptr(du), _ptr(ddelta), _ptr(dA),
                             _ptr(dB), _ptr(dC), _ptr(dD), _ptr(dz), _ptr(d_delta_bias),
                             _ptr(d_init_state), batch, dim, L, N, _io_dtype(u),
                             _ptr(workspace), int(workspace_bytes or 0), _stream(stream))
    _call("ssm_scan_bwd", rc)


def ssm_conv1d_fwd(x, weight, bias, conv_state_in, silu, out, conv_state_out, stream=None):
    """Tensor form of ``ssm_conv1d_fwd``: x (batch, dim, L), weight (dim, width)."""
    _check_dev(x, weight, bias, conv_state_in, out, conv_state_out)
    batch = x.shape[0]
    dim, L = (x.shape[2], x.shape[1]) if int(silu) & SSM_LAYOUT_BLD else (x.shape[1], x.shape[2])
    rc = load().ssm_conv1d_fwd(_ptr(x), _ptr(weight), _ptr(bias), _ptr(conv_state_in),
                               int(silu), _ptr(out), _ptr(conv_state_out), batch, dim, L,
                               weight.shape[1], _io_dtype(x), _stream(stream))
    _call("ssm_conv1d_fwd", rc)


def ssm_conv1d_bwd(x, weight, bias, conv_state_in, silu, dout, dx, dweight, dbias,
                   d_conv_state_in, stream=None):
    """Tensor form of ``ssm_conv1d_bwd``: x, dout, dx like the forward's x."""
    _check_dev(x, weight, bias, conv_state_in, dout, dx, dweight, dbias, d_conv_state_in)
    batch = x.shape[0]
    dim, L = (x.shape[2], x.shape[1]) if int(silu) & SSM_LAYOUT_BLD else (x.shape[1], x.shape[2])
    rc = load().ssm_conv1d_bwd(_ptr(x), _ptr(weight), _ptr(bias), _ptr(conv_state_in), int(silu),
                               _ptr(dout), _ptr(dx), _ptr(dweight), _ptr(dbias),
                               _ptr(d_conv_state_in), batch, dim, L, weight.shape[1], _io_dtype(x),
                               _stream(stream))
    _call("ssm_conv1d_bwd", rc)


def ssm_conv1d_update(conv_state, x, weight, bias, silu, out, stream=None):
    """Tensor form of ``ssm_conv1d_update``: x (batch, dim), conv_state (batch, dim, width-1)."""
    _check_dev(conv_state, x, weight, bias, out)
    batch, dim = x.shape
    rc = load().ssm_conv1d_update(_ptr(conv_state), _ptr(x), _ptr(weight), _ptr(bias),
                                  int(bool(silu)), _ptr(out), batch, dim, weight.shape[1],
                                  _io_dtype(x), _stream(stream))
    _call("ssm_conv1d_update", rc)


def ssm_ssd_workspace_bytes(batch, seqlen, nheads, headdim, ngroups, dstate) -> int:
    return int(load().ssm_ssd_workspace_bytes(batch, seqlen, nheads, headdim, ngroups, dstate))


def ssm_ssd_fwd(x, dt, dt_bias, A, B, C, D, z, flags, y, final_state, init_state, workspace,
                workspace_bytes=None, stream=None):
    """Tensor form of ``ssm_ssd_fwd``: x (batch, L, H, P), B (batch, L, G, N)."""
    _check_dev(x, dt, dt_bias, A, B, C, D, z, y, final_state, init_state, workspace)
    batch, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    if workspace is not None and workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    rc = load().ssm_ssd_fwd(_ptr(x), _ptr(dt), _ptr(dt_bias), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                            _ptr(z), int(flags), _ptr(y), _ptr(final_state), _ptr(init_state),
                            batch, L, H, P, G, N, _ptr(workspace), int(workspace_bytes or 0),
                            _stream(stream))
    _call("ssm_ssd_fwd", rc)


def ssm_ssd_bwd_workspace_bytes(batch, seqlen, nheads, headdim, ngroups, dstate) -> int:
    return int(load().ssm_ssd_bwd_workspace_bytes(batch, seqlen, nheads, headdim, ngroups, dstate))


def ssm_ssd_bwd(x, dt, dt_bias, A, B, C, D, z, flags, init_state, dy, d_final_state, dx, ddt, dA,
                dB, dC, dD, dz, d_dt_bias, d_init_state, workspace, workspace_bytes, stream=None):
    """Tensor form of ``ssm_ssd_bwd``; sizes from x (batch, L, H, P) and B (batch, L, G, N)."""
    _check_dev(x, dt, dt_bias, A, B, C, D, z, init_state, dy, d_final_state, dx, ddt, dA, dB, dC,
               dD, dz, d_dt_bias, d_init_state, workspace)
    batch, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    rc = load().ssm_ssd_bwd(_ptr(x), _ptr(dt), _ptr(dt_bias), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                            _ptr(z), int(flags), _ptr(init_state), _ptr(dy), _ptr(d_final_state),
                            _ptr(dx), _ptr(ddt), _ptr(dA), _ptr(dB), _ptr(dC), _ptr(dD), _ptr(dz),
                            _ptr(d_dt_bias), _ptr(d_init_state), batch, L, H, P, G, N,
                            _ptr(workspace), int(workspace_bytes or 0), _stream(stream))
    _call("ssm_ssd_bwd", rc)


def static_scratch_bytes() -> int:
    """SSM_STATIC_SCRATCH_BYTES as defined in include/ssm.h."""
    import re
    m = re.search(r"#define\s+SSM_STATIC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", open(HEADER).read())
    return int(m.group(1)) << int(m.group(2))


# ---------------------------------------------------------------------------
# allocating helpers (torch allocates; the library computes)
# ---------------------------------------------------------------------------

def scan(u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=True,
         init_state=None, split=True, stream=None, euler=False, bld=False):
    """y, final_state = scan(...): allocates y (dtype of u) and final_state (float32), and a
    workspace when the plan splits the sequence across blocks."""
    import torch
    batch, dim, L = _sizes(u, A, B)
    N = A.shape[1]
    y = torch.empty_like(u)
    h = torch.empty((batch, dim, N), dtype=torch.float32, device=u.device)
    ws = None
    if split:
        nbytes = ssm_scan_workspace_bytes(batch, dim, L, N, _io_dtype(u))
        if nbytes:
            ws = torch.empty(nbytes, dtype=torch.uint8, device=u.device)
    ssm_scan_fwd_ex(u, delta, delta_bias, A, B, C, D, z, _flags(delta_softplus, euler, bld), y,
                    h, init_state, ws, stream=stream)
    return y, h


def ssm_scan_fwd_complex(u, delta, delta_bias, A, B, C, D, z, delta_softplus, y, final_state,
                         init_state=None, stream=None):
    """Tensor form of ``ssm_scan_fwd_complex``: A (dim, N), B, C (batch, N, L) and the
    states (batch, dim, N) are torch.complex64 tensors (passed as their interleaved
    (re, im) float pairs); u, delta, z, y (batch, dim, L) in the I/O dtype."""
    _check_dev(u, delta, delta_bias, A, B, C, D, z, y, final_state, init_state)
    for t in (A, B, C, final_state, init_state):
        if t is not None and t.dtype != _torch_complex64():
            raise TypeError("A, B, C and the states must be complex64")
    batch, dim, L = int(B.shape[0]), int(A.shape[0]), int(B.shape[2])
    N = int(A.shape[1])
    rc = load().ssm_scan_fwd_complex(_ptr(u), _ptr(delta), _ptr(delta_bias), _ptr(A), _ptr(B),
                                     _ptr(C), _ptr(D), _ptr(z), _flags(delta_softplus), _ptr(y),
                                     _ptr(final_state), _ptr(init_state), batch, dim, L, N,
                                     _io_dtype(u), _stream(stream))
    _call("ssm_scan_fwd_complex", rc)


def _torch_complex64():
    import torch
    return torch.complex64


def scan_complex(u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=True,
                 init_state=None, euler=False, stream=None):
    """y, final_state = scan_complex(...): the scan with a complex diagonal A; allocates
    y (dtype of u) and the complex64 final state."""
    import torch
    batch, dim = int(B.shape[0]), int(A.shape[0])
    y = torch.empty_like(u)
    h = torch.empty((batch, dim, A.shape[1]), dtype=torch.complex64, device=u.device)
    ssm_scan_fwd_complex(u, delta, delta_bias, A, B, C, D, z, _flags(delta_softplus, euler), y,
                         h, init_state, stream)
    return y, h


def scan_host(u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=True,
              init_state=None, euler=False, bld=False, stream=None):
    """y, final_state = scan_host(...): the scan on host tensors through
    ``ssm_scan_fwd_host`` (copies pipelined against the scan inside the library);
    allocates page-locked outputs and the device workspace, waits for the stream."""
    import torch
    batch, dim, L = _sizes(u, A, B)
    N = A.shape[1]
    flags = _flags(delta_softplus, euler, bld)
    y = torch.empty(u.shape, dtype=u.dtype, pin_memory=True)
    h = torch.empty((batch, dim, N), dtype=torch.float32, pin_memory=True)
    nbytes = ssm_scan_fwd_host_workspace_bytes(batch, dim, L, N, _io_dtype(u), flags)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")
    st = stream if stream is not None else torch.cuda.current_stream()
    ssm_scan_fwd_host(u, delta, delta_bias, A, B, C, D, z, flags, y, h, init_state, ws, nbytes, st)
    st.synchronize()
    return y, h


def scan_train(u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=True,
               init_state=None, stream=None, euler=False, bld=False):
    """y, final_state, saved = scan_train(...): the forward of ``scan`` that also keeps
    what the backward needs; pass ``saved`` to ``scan_bwd(..., saved=saved)``."""
    import torch
    batch, dim, L = _sizes(u, A, B)
    N = A.shape[1]
    y = torch.empty_like(u)
    h = torch.empty((batch, dim, N), dtype=torch.float32, device=u.device)
    nbytes = ssm_scan_workspace_bytes(batch, dim, L, N, _io_dtype(u))
    ws = torch.empty(nbytes, dtype=torch.uint8, device=u.device) if nbytes else None
    bbytes = ssm_scan_bwd_workspace_bytes(batch, dim, L, N)
    bws = torch.empty(max(bbytes, 16), dtype=torch.uint8, device=u.device)
    ssm_scan_fwd_train(u, delta, delta_bias, A, B, C, D, z, _flags(delta_softplus, euler, bld),
                       y, h, init_state, ws, nbytes, bws, bbytes, stream)
    return y, h, bws


def scan_bwd(u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=True,
             init_state=None, dy=None, d_final_state=None, want_init_grad=False, stream=None,
             euler=False, saved=None, bld=False):
    """Derivatives of Σ y·dy + Σ final_state·d_final_state for the inputs of ``scan``.
    Allocates every output and the workspace; returns a dict with du, ddelta, dz (dtype of
    u; dz None without z), dA, dB, dC, dD, dbias (float32; dD / dbias always computed) and
    dinit (float32, when ``want_init_grad``)."""
    import torch
    batch, dim, L = _sizes(u, A, B)
    N = A.shape[1]
    dev = u.device
    f32 = dict(dtype=torch.float32, device=dev)
    out = dict(du=torch.empty_like(u), ddelta=torch.empty_like(u),
               dz=None if z is None else torch.empty_like(u),
               dA=torch.empty((dim, N), **f32), dB=torch.empty((batch, N, L), **f32),
               dC=torch.empty((batch, N, L), **f32), dD=torch.empty(dim, **f32),
               dbias=torch.empty(dim, **f32),
               dinit=torch.empty((batch, dim, N), **f32) if want_init_grad else None)
    nbytes = ssm_scan_bwd_workspace_bytes(batch, dim, L, N)
    flags = _flags(delta_softplus, euler, bld)
    if saved is not None:
        ws = saved
        flags |= SSM_SAVED_STATES
    else:
        ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)
    ssm_scan_bwd(u, delta, delta_bias, A, B, C, D, z, flags, init_state,
                 dy, d_final_state, out["du"], out["ddelta"], out["dA"], out["dB"], out["dC"],
                 out["dD"], out["dz"], out["dbias"], out["dinit"], ws, nbytes, stream)
    return out


def conv1d(x, weight, bias=None, conv_state=None, silu=True, want_state=False, stream=None,
           bld=False):
    """out[, new_state] = conv1d(...): causal depthwise conv1d (+ SiLU) of x (batch, dim, L),
    or (batch, L, dim) with ``bld``; conv_state (batch, dim, width-1) holds the inputs
    before the sequence."""
    import torch
    out = torch.empty_like(x)
    st = None
    if want_state:
        st = torch.empty((x.shape[0], weight.shape[0], weight.shape[1] - 1), dtype=x.dtype,
                         device=x.device)
    ssm_conv1d_fwd(x, weight, bias, conv_state, int(bool(silu)) | (SSM_LAYOUT_BLD if bld else 0),
                   out, st, stream)
    return (out, st) if want_state else out


def ssd_bwd(x, dt, A, B, C, D=None, z=None, dt_bias=None, delta_softplus=True, init_state=None,
            dy=None, d_final_state=None, euler=False, stream=None):
    """Derivatives of ``ssd``'s outputs against dy (and d_final_state): dict(dx, dz, ddt
    (bf16, like x, z, dt), dA, dD, ddt_bias (H,), dB, dC (like B, float32), dinit
    (batch, H, P, N) float32)."""
    import torch
    batch, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    f32 = dict(dtype=torch.float32, device=x.device)
    out = dict(dx=torch.empty_like(x), ddt=torch.empty_like(dt), dz=None if z is None else torch.empty_like(z),
               dA=torch.empty(H, **f32), dD=torch.empty(H, **f32), ddt_bias=torch.empty(H, **f32),
               dB=torch.empty(B.shape, **f32), dC=torch.empty(C.shape, **f32),
               dinit=torch.empty((batch, H, P, N), **f32))
    nbytes = ssm_ssd_bwd_workspace_bytes(batch, L, H, P, G, N)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=x.device)
    ssm_ssd_bwd(x, dt, dt_bias, A, B, C, D, z, _flags(delta_softplus, euler), init_state, dy,
                d_final_state, out["dx"], out["ddt"], out["dA"], out["dB"], out["dC"], out["dD"],
                out["dz"], out["ddt_bias"], out["dinit"], ws, nbytes, stream)
    return out


def conv1d_bwd(x, weight, dout, bias=None, conv_state=None, silu=True, bld=False, stream=None):
    """Derivatives of ``conv1d``'s output against ``dout``: dict(dx (like x), dweight
    (dim, width), dbias (dim,), dstate (batch, dim, width-1)), the last three float32."""
    import torch
    batch, dim, K = x.shape[0], weight.shape[0], weight.shape[1]
    dx = torch.empty_like(x)
    dw = torch.empty((dim, K), dtype=torch.float32, device=x.device)
    db = torch.empty((dim,), dtype=torch.float32, device=x.device)
    ds = torch.empty((batch, dim, K - 1), dtype=torch.float32, device=x.device) if K > 1 else None
    ssm_conv1d_bwd(x, weight, bias, conv_state, int(bool(silu)) | (SSM_LAYOUT_BLD if bld else 0),
                   dout, dx, dw, db, ds, stream)
    return dict(dx=dx, dweight=dw, dbias=db, dstate=ds)


def ssd(x, dt, A, B, C, D=None, z=None, dt_bias=None, delta_softplus=True, init_state=None,
        euler=False, stream=None):
    """y, final_state = ssd(...): Mamba-2's chunked scalar-A SSM; allocates y (bf16, like x),
    the final state (batch, H, P, N) float32 and the workspace."""
    import torch
    batch, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    y = torch.empty_like(x)
    h = torch.empty((batch, H, P, N), dtype=torch.float32, device=x.device)
    nbytes = ssm_ssd_workspace_bytes(batch, L, H, P, G, N)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=x.device)
    ssm_ssd_fwd(x, dt, dt_bias, A, B, C, D, z, _flags(delta_softplus, euler), y, h, init_state,
                ws, nbytes, stream)
    return y, h


def exported_names():
    """Entry points declared in include/ssm.h."""
    import re
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:int|size_t|const char\*)\s+(ssm_\w+)\s*\(", text, re.M)))
