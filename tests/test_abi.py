"""The C ABI without a GPU: the library loads, exports every entry point that
include/ssm.h declares, and rejects bad arguments synchronously (before any CUDA
call) with the documented status codes.  Pointers here are fake addresses that
are never dereferenced."""
import pytest

import selective_state_space_128_b300 as ssm

FAKE = 0x7F0000000000  # 16-byte aligned, never dereferenced


def lib():
    return ssm.load()


def test_exports_every_declared_symbol():
    names = ssm.exported_names()
    assert {"ssm_scan_fwd", "ssm_scan_fwd_ex", "ssm_state_update", "ssm_state_update_ex",
            "ssm_scan_workspace_bytes", "ssm_strerror", "ssm_version"} <= set(names)
    for n in names:
        assert hasattr(lib(), n), n


def test_strerror_and_version():
    assert ssm.version() == "0.1.0"
    for code in (0, -1, -2, -3, -4, -5):
        assert ssm.strerror(code).startswith("SSM_")
    assert "unknown" in ssm.strerror(42)


def _scan(**kw):
    a = dict(u=FAKE, delta=FAKE + 0x1000000, bias=None, A=FAKE + 0x2000000, B=FAKE + 0x3000000,
             C=FAKE + 0x4000000, D=None, z=None, softplus=1, y=FAKE + 0x5000000, h=None,
             batch=2, dim=64, L=128, N=16, io=ssm.SSM_BF16, init=None, ws=None, wsb=0, stream=None)
    a.update(kw)
    return lib().ssm_scan_fwd_ex(a["u"], a["delta"], a["bias"], a["A"], a["B"], a["C"], a["D"],
                                 a["z"], a["softplus"], a["y"], a["h"], a["batch"], a["dim"],
                                 a["L"], a["N"], a["io"], a["init"], a["ws"], a["wsb"], a["stream"])


def test_scan_argument_errors():
    assert _scan(u=None) == ssm.SSM_ERR_ARG
    assert _scan(y=None) == ssm.SSM_ERR_ARG
    assert _scan(A=None) == ssm.SSM_ERR_ARG
    assert _scan(io=7) == ssm.SSM_ERR_ARG
    assert _scan(batch=-1) == ssm.SSM_ERR_ARG
    assert _scan(L=-5) == ssm.SSM_ERR_ARG
    assert _scan(N=0) == ssm.SSM_ERR_ARG
    assert _scan(batch=70000) == ssm.SSM_ERR_ARG
    for n in (3, 5, 12, 256):
        assert _scan(N=n) == ssm.SSM_ERR_UNSUPPORTED
    assert _scan(u=FAKE + 2) == ssm.SSM_ERR_ALIGN
    assert _scan(z=FAKE + 0x6000008) == ssm.SSM_ERR_ALIGN
    assert _scan(h=FAKE + 0x7000004) == ssm.SSM_ERR_ALIGN
    # y overlapping an input
    assert _scan(y=FAKE + 0x100) == ssm.SSM_ERR_ARG
    # final_state overlapping init_state without being the same buffer
    assert _scan(h=FAKE + 0x8000000, init=FAKE + 0x8000010) == ssm.SSM_ERR_ARG
    # empty problems succeed without touching the device
    assert _scan(batch=0) == ssm.SSM_OK
    assert _scan(dim=0) == ssm.SSM_OK


def test_workspace_too_small_is_rejected_before_launch():
    need = ssm.ssm_scan_workspace_bytes(1, 64, 1 << 16, 16, ssm.SSM_BF16)
    assert need > 0
    rc = _scan(batch=1, dim=64, L=1 << 16, ws=FAKE + 0x9000000, wsb=need - 16)
    assert rc == ssm.SSM_ERR_WORKSPACE


def test_workspace_plan():
    hdr = ssm.SCAN_STATUS_BYTES
    # many channels: one pass, the status header only
    assert ssm.ssm_scan_workspace_bytes(8, 1536, 2048, 16, 1) == hdr
    assert ssm.ssm_scan_workspace_bytes(4, 5120, 4096, 16, 1) == hdr
    # few channels, long sequence: split with carry records after the header.  On a
    # 148-SM device a batch row of 1536 channels is 192 eight-channel warps, under 8
    # per SM, so the plan splits; it sizes the segments for 16 warps per SM:
    # ceil(148 * 16 / 192) = 13 segments, carry records of 12 of them (state + ΣΔ)
    def al(x):
        return (x + 255) // 256 * 256
    carry = al(12 * 1536 * 16 * 4) + 12 * 1536 * 4
    assert ssm.ssm_scan_workspace_bytes(1, 1536, 65536, 16, 1) == hdr + carry
    assert ssm.ssm_scan_workspace_bytes(1, 64, 100, 16, 1) == hdr   # too short to split
    assert ssm.ssm_scan_workspace_bytes(1, 64, 100, 3, 1) == 0      # unsupported N


def test_workspace_smaller_than_the_status_header_is_rejected():
    rc = _scan(ws=FAKE + 0x9000000, wsb=ssm.SCAN_STATUS_BYTES - 16)
    assert rc == ssm.SSM_ERR_WORKSPACE
    assert _scan(ws=FAKE + 0x9000008, wsb=4096) == ssm.SSM_ERR_ALIGN


def test_stall_flag_is_refused_outside_test_mode():
    """SSM_TEST_STALL (the failure-path test) is an argument error unless the test
    mode is on; the test mode checks its limits."""
    assert _scan(softplus=1 | ssm.SSM_TEST_STALL) == ssm.SSM_ERR_ARG
    l = lib()
    assert l.ssm_set_test_mode(1, 10, 0, 0) == ssm.SSM_ERR_ARG            # limit below 1 us
    assert l.ssm_set_test_mode(1, 3_000_000_000, 0, 0) == ssm.SSM_ERR_ARG  # above 2 s
    assert l.ssm_set_test_mode(1, 1_000_000, -1, 0) == ssm.SSM_ERR_ARG
    assert l.ssm_set_test_mode(1, 1_000_000, 0, 3) == ssm.SSM_ERR_ARG     # no kernel 3
    assert l.ssm_set_test_mode(0, 0, 0, 0) == ssm.SSM_OK
    assert _scan(softplus=1 | ssm.SSM_TEST_STALL) == ssm.SSM_ERR_ARG


def _upd(**kw):
    a = dict(state=FAKE, u=FAKE + 0x1000000, delta=FAKE + 0x2000000, bias=None, softplus=1,
             A=FAKE + 0x3000000, B=FAKE + 0x4000000, C=FAKE + 0x5000000, D=None, z=None,
             y=FAKE + 0x6000000, batch=4, dim=64, N=16, io=ssm.SSM_BF16, stream=None)
    a.update(kw)
    return lib().ssm_state_update_ex(a["state"], a["u"], a["delta"], a["bias"], a["softplus"],
                                     a["A"], a["B"], a["C"], a["D"], a["z"], a["y"], a["batch"],
                                     a["dim"], a["N"], a["io"], a["stream"])


def test_update_argument_errors():
    assert _upd(state=None) == ssm.SSM_ERR_ARG
    assert _upd(io=2) == ssm.SSM_ERR_ARG
    assert _upd(N=24) == ssm.SSM_ERR_UNSUPPORTED
    assert _upd(y=FAKE + 0x6000002) == ssm.SSM_ERR_ALIGN
    assert _upd(y=FAKE + 0x10) == ssm.SSM_ERR_ARG           # y overlaps the state
    assert _upd(u=FAKE + 0x40) == ssm.SSM_ERR_ARG           # state overlaps u
    assert _upd(batch=0) == ssm.SSM_OK


def test_short_forms_validate_too():
    L = lib()
    rc = L.ssm_scan_fwd(None, FAKE, None, FAKE, FAKE, FAKE, None, None, 1, FAKE, None,
                        1, 1, 1, 16, 1)
    assert rc == ssm.SSM_ERR_ARG
    rc = L.ssm_state_update(FAKE, FAKE + 0x100000, FAKE + 0x200000, FAKE + 0x300000,
                            FAKE + 0x400000, FAKE + 0x500000, None, None, FAKE + 0x600000,
                            1, 1, 7, 1)
    assert rc == ssm.SSM_ERR_UNSUPPORTED


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(ssm, "_lib", None)
    monkeypatch.setattr(ssm, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        ssm.load()


def _bwd(**kw):
    a = dict(u=FAKE, delta=FAKE + 0x1000000, bias=None, A=FAKE + 0x2000000, B=FAKE + 0x3000000,
             C=FAKE + 0x4000000, D=None, z=None, softplus=1, init=None, dy=FAKE + 0x5000000,
             dfin=None, du=FAKE + 0x6000000, ddelta=FAKE + 0x7000000, dA=FAKE + 0x8000000,
             dB=FAKE + 0x9000000, dC=FAKE + 0xA000000, dD=None, dz=None, dbias=None, dinit=None,
             batch=2, dim=64, L=128, N=16, io=ssm.SSM_BF16, ws=FAKE + 0x10000000,
             wsb=1 << 30, stream=None)
    a.update(kw)
    return lib().ssm_scan_bwd(a["u"], a["delta"], a["bias"], a["A"], a["B"], a["C"], a["D"],
                              a["z"], a["softplus"], a["init"], a["dy"], a["dfin"], a["du"],
                              a["ddelta"], a["dA"], a["dB"], a["dC"], a["dD"], a["dz"],
                              a["dbias"], a["dinit"], a["batch"], a["dim"], a["L"], a["N"],
                              a["io"], a["ws"], a["wsb"], a["stream"])


def test_backward_argument_errors():
    for name in ("u", "delta", "A", "B", "C", "dy", "du", "ddelta", "dA", "dB", "dC"):
        assert _bwd(**{name: None}) == ssm.SSM_ERR_ARG, name
    assert _bwd(io=3) == ssm.SSM_ERR_ARG
    assert _bwd(N=12) == ssm.SSM_ERR_UNSUPPORTED
    assert _bwd(N=256) == ssm.SSM_ERR_UNSUPPORTED
    assert ssm.ssm_scan_bwd_workspace_bytes(2, 64, 128, 256) == 0
    assert ssm.ssm_scan_bwd_workspace_bytes(2, 64, 128, 128) > 0  # N = 128: 8-step chunks
    # dz is required with a gate and refused without one
    assert _bwd(z=FAKE + 0xB000000) == ssm.SSM_ERR_ARG
    assert _bwd(dz=FAKE + 0xB000000) == ssm.SSM_ERR_ARG
    assert _bwd(du=FAKE + 0x6000004) == ssm.SSM_ERR_ALIGN
    assert _bwd(dinit=FAKE + 0xC000008) == ssm.SSM_ERR_ALIGN
    # outputs overlapping an input or each other
    assert _bwd(du=FAKE + 0x100) == ssm.SSM_ERR_ARG
    assert _bwd(dB=FAKE + 0x8000100) == ssm.SSM_ERR_ARG
    # the workspace is required and sized by ssm_scan_bwd_workspace_bytes
    need = ssm.ssm_scan_bwd_workspace_bytes(2, 64, 128, 16)
    assert need > 0
    assert _bwd(ws=None) == ssm.SSM_ERR_WORKSPACE
    assert _bwd(wsb=need - 1) == ssm.SSM_ERR_WORKSPACE
    assert _bwd(ws=FAKE + 0x8000000, wsb=need) == ssm.SSM_ERR_ARG   # workspace over dA


def test_backward_workspace_size():
    # checkpoints [batch][chunks][dim][N] + per-block dB/dC partials + per-row sums
    need = ssm.ssm_scan_bwd_workspace_bytes(8, 1536, 2048, 16)
    ckpt = 8 * (2048 // 16) * 1536 * 16 * 4
    parts = 2 * 8 * (1536 // 32) * 16 * 2048 * 4
    assert ckpt + parts <= need <= ckpt + parts + 8 * 1536 * 18 * 4 + 6 * 256
    assert ssm.ssm_scan_bwd_workspace_bytes(0, 1536, 2048, 16) == 0
    assert ssm.ssm_scan_bwd_workspace_bytes(8, 1536, 2048, 3) == 0


def test_backward_split_plan():
    """One batch row of 1536 channels is 48 blocks of 32 channels, under half of one
    wave of 148 SMs x 3 resident blocks: the plan splits the 2^20 steps into as
    many segments as fit in that wave, 9 of 116 512 steps (444 // 48 = 9; a
    multiple of 16), and the workspace adds the per-segment sums and the forward's
    and the adjoint's carries of 8 segments.  With 8 batch rows (384 blocks) and
    2048 steps it does not split."""
    def al(x):
        return (x + 255) // 256 * 256

    b, d, L, N = 1, 1536, 1 << 20, 16
    nseg, rows = 9, b * d
    want = (al(b * (L // 16) * d * N * 4) + 2 * al(b * (d // 32) * N * L * 4)
            + al(nseg * rows * N * 4) + 2 * al(nseg * rows * 4)
            + 2 * (al((nseg - 1) * rows * N * 4) + al((nseg - 1) * rows * 4)))
    assert ssm.ssm_scan_bwd_workspace_bytes(b, d, L, N) == want
    b, L = 8, 2048
    want = (al(b * (L // 16) * d * N * 4) + 2 * al(b * (d // 32) * N * L * 4)
            + al(b * d * N * 4) + 2 * al(b * d * 4))
    assert ssm.ssm_scan_bwd_workspace_bytes(b, d, L, N) == want


def test_conv_argument_errors():
    L_ = lib()
    ok = dict(x=FAKE, w=FAKE + 0x1000000, b=None, sin=None, silu=1, out=FAKE + 0x2000000,
              sout=None, batch=2, dim=8, L=64, K=4, io=ssm.SSM_BF16)

    def fwd(**kw):
        a = dict(ok)
        a.update(kw)
        return L_.ssm_conv1d_fwd(a["x"], a["w"], a["b"], a["sin"], a["silu"], a["out"], a["sout"],
                                 a["batch"], a["dim"], a["L"], a["K"], a["io"], None)

    assert fwd(x=None) == ssm.SSM_ERR_ARG
    assert fwd(K=5) == ssm.SSM_ERR_UNSUPPORTED
    assert fwd(K=0) == ssm.SSM_ERR_ARG
    assert fwd(out=FAKE + 0x2000004) == ssm.SSM_ERR_ALIGN
    assert fwd(out=FAKE + 0x100) == ssm.SSM_ERR_ARG                       # out over x
    assert fwd(sin=FAKE + 0x3000000, sout=FAKE + 0x3000010) == ssm.SSM_ERR_ARG  # partial overlap
    assert fwd(batch=0) == ssm.SSM_OK
    assert L_.ssm_conv1d_update(None, FAKE, FAKE + 0x1000000, None, 1, FAKE + 0x2000000, 2, 8, 4,
                                ssm.SSM_BF16, None) == ssm.SSM_ERR_ARG    # state required
    assert L_.ssm_conv1d_update(FAKE + 0x3000000, FAKE, FAKE + 0x1000000, None, 1,
                                FAKE + 0x3000010, 2, 8, 4, ssm.SSM_BF16, None) == ssm.SSM_ERR_ARG


def test_flag_word_is_checked():
    assert _scan(softplus=4) == ssm.SSM_ERR_ARG
    assert _scan(softplus=-1) == ssm.SSM_ERR_ARG
    assert _upd(softplus=8) == ssm.SSM_ERR_ARG
    assert _bwd(softplus=16) == ssm.SSM_ERR_ARG
    # the defined bits pass validation (empty problem: nothing is launched)
    for f in (0, ssm.SSM_SOFTPLUS, ssm.SSM_EULER_B, ssm.SSM_SOFTPLUS | ssm.SSM_EULER_B):
        assert _scan(softplus=f, batch=0) == ssm.SSM_OK


def test_training_forward_argument_errors():
    L_ = lib()

    def tr(**kw):
        a = dict(u=FAKE, delta=FAKE + 0x1000000, bias=None, A=FAKE + 0x2000000,
                 B=FAKE + 0x3000000, C=FAKE + 0x4000000, D=None, z=None, softplus=1,
                 y=FAKE + 0x5000000, h=None, batch=2, dim=64, L=128, N=16, io=ssm.SSM_BF16,
                 init=None, ws=None, wsb=0, bws=FAKE + 0x10000000, bwsb=1 << 30)
        a.update(kw)
        return L_.ssm_scan_fwd_train(a["u"], a["delta"], a["bias"], a["A"], a["B"], a["C"],
                                     a["D"], a["z"], a["softplus"], a["y"], a["h"], a["batch"],
                                     a["dim"], a["L"], a["N"], a["io"], a["init"], a["ws"],
                                     a["wsb"], a["bws"], a["bwsb"], None)

    need = ssm.ssm_scan_bwd_workspace_bytes(2, 64, 128, 16)
    assert tr(bws=None) == ssm.SSM_ERR_WORKSPACE
    assert tr(bwsb=need - 16) == ssm.SSM_ERR_WORKSPACE
    assert tr(bws=FAKE + 0x5000000) == ssm.SSM_ERR_ARG      # over y
    assert tr(bws=FAKE + 0x10000008) == ssm.SSM_ERR_ALIGN
    assert tr(softplus=ssm.SSM_SAVED_STATES) == ssm.SSM_ERR_ARG  # a backward-only bit
    assert _bwd(softplus=ssm.SSM_SOFTPLUS | ssm.SSM_SAVED_STATES, u=None) == ssm.SSM_ERR_ARG


def test_ssd_argument_errors():
    L_ = lib()
    args = [FAKE, FAKE + 0x100000, None, FAKE + 0x200000, FAKE + 0x300000, FAKE + 0x400000, None,
            None, 1, FAKE + 0x500000, None, None]
    ws = (FAKE + 0x10000000, 1 << 30, None)
    # headdim other than 64, dstate other than 64/128, heads not a multiple of groups
    assert L_.ssm_ssd_fwd(*args, 1, 64, 4, 32, 1, 64, *ws) == ssm.SSM_ERR_UNSUPPORTED
    assert L_.ssm_ssd_fwd(*args, 1, 64, 4, 64, 1, 32, *ws) == ssm.SSM_ERR_UNSUPPORTED
    assert L_.ssm_ssd_fwd(*args, 1, 64, 4, 64, 3, 64, *ws) == ssm.SSM_ERR_UNSUPPORTED
    assert L_.ssm_ssd_fwd(*args, 1, 64, 4, 64, 1, 64, None, 0, None) == ssm.SSM_ERR_WORKSPACE
    assert L_.ssm_ssd_fwd(*args[:8], 5, *args[9:], 1, 64, 4, 64, 1, 64, *ws) == ssm.SSM_ERR_ARG
    assert L_.ssm_ssd_fwd(*args[:9], FAKE + 0x100, *args[10:], 1, 64, 4, 64, 1, 64, *ws) == ssm.SSM_ERR_ARG
    # the states entering each of the 8 x 32 x 24 (batch, chunk, head) units as
    # bf16 (64 x 128 each), each unit's step terms (3 x 64 fp32) and each
    # (batch, chunk, group)'s C Bᵀ (64 x 64 fp32)
    units = 8 * 32 * 24
    assert ssm.ssm_ssd_workspace_bytes(8, 2048, 24, 64, 1, 128) == (
        units * 64 * 128 * 2 + units * 3 * 64 * 4 + 8 * 32 * 1 * 64 * 64 * 4)
    assert ssm.ssm_ssd_workspace_bytes(8, 2048, 24, 64, 5, 128) == 0  # 24 heads in 5 groups


def _host(**kw):
    a = dict(u=FAKE, delta=FAKE + 0x1000000, bias=None, A=FAKE + 0x2000000, B=FAKE + 0x3000000,
             C=FAKE + 0x4000000, D=None, z=None, flags=1, y=FAKE + 0x5000000, h=None, init=None,
             batch=2, dim=64, L=128, N=16, io=ssm.SSM_BF16, ws=FAKE + 0x9000000, wsb=1 << 30,
             stream=None)
    a.update(kw)
    return lib().ssm_scan_fwd_host(a["u"], a["delta"], a["bias"], a["A"], a["B"], a["C"], a["D"],
                                   a["z"], a["flags"], a["y"], a["h"], a["init"], a["batch"],
                                   a["dim"], a["L"], a["N"], a["io"], a["ws"], a["wsb"], a["stream"])


def test_scan_host_argument_errors():
    assert _host(u=None) == ssm.SSM_ERR_ARG
    assert _host(y=None) == ssm.SSM_ERR_ARG
    assert _host(io=7) == ssm.SSM_ERR_ARG
    assert _host(flags=ssm.SSM_SAVED_STATES | 1) == ssm.SSM_ERR_ARG  # a backward-only bit
    assert _host(batch=-1) == ssm.SSM_ERR_ARG
    assert _host(N=12) == ssm.SSM_ERR_UNSUPPORTED
    assert _host(ws=None) == ssm.SSM_ERR_WORKSPACE
    assert _host(wsb=1024) == ssm.SSM_ERR_WORKSPACE
    assert _host(ws=FAKE + 8) == ssm.SSM_ERR_ALIGN
    assert _host(batch=0) == ssm.SSM_OK and _host(dim=0) == ssm.SSM_OK


def test_scan_host_workspace_plan():
    # the status header, then three staging slots of a whole batch row (8 rows: one unit per
    # row): u, delta, z, y of 1536 x 2048 bf16, B and C of 16 x 2048 fp32, two states of
    # 1536 x 16 fp32; plus A, D, bias and the unit scan's carry records
    slot = 4 * 1536 * 2048 * 2 + 2 * 16 * 2048 * 4 + 2 * 1536 * 16 * 4
    params = 1536 * 16 * 4 + 2 * 1536 * 4
    hdr = ssm.SCAN_STATUS_BYTES
    carry = ssm.ssm_scan_workspace_bytes(1, 1536, 2048, 16, ssm.SSM_BF16) - hdr
    scan_ws = hdr + (carry + 255) // 256 * 256
    assert ssm.ssm_scan_fwd_host_workspace_bytes(8, 1536, 2048, 16, ssm.SSM_BF16, 1) == \
        params + scan_ws + 3 * slot
    # batch 1: the row is cut into 8 blocks of channels, so a slot is an eighth as large
    small = ssm.ssm_scan_fwd_host_workspace_bytes(1, 1536, 2048, 16, ssm.SSM_BF16, 1)
    assert small < params + scan_ws + slot
    assert ssm.ssm_scan_fwd_host_workspace_bytes(1, 64, 0, 16, ssm.SSM_BF16, 0) == \
        hdr + 64 * 16 * 4
    assert ssm.ssm_scan_fwd_host_workspace_bytes(1, 64, 10, 12, ssm.SSM_BF16, 0) == 0


def test_conv1d_bwd_argument_errors():
    def call(**kw):
        a = dict(x=FAKE, w=FAKE + 0x1000000, b=None, st=None, silu=1, dout=FAKE + 0x2000000,
                 dx=FAKE + 0x3000000, dw=FAKE + 0x4000000, db=None, ds=None, batch=2, dim=64, L=128,
                 K=4, io=ssm.SSM_BF16)
        a.update(kw)
        return lib().ssm_conv1d_bwd(a["x"], a["w"], a["b"], a["st"], a["silu"], a["dout"], a["dx"],
                                    a["dw"], a["db"], a["ds"], a["batch"], a["dim"], a["L"], a["K"],
                                    a["io"], None)
    assert call(K=5) == ssm.SSM_ERR_UNSUPPORTED
    assert call(K=0) == ssm.SSM_ERR_ARG
    assert call(io=9) == ssm.SSM_ERR_ARG
    assert call(silu=4) == ssm.SSM_ERR_ARG
    assert call(dw=None) == ssm.SSM_ERR_ARG
    assert call(dout=None) == ssm.SSM_ERR_ARG
    assert call(dx=FAKE + 0x3000008) == ssm.SSM_ERR_ALIGN
    assert call(dx=FAKE + 0x10) == ssm.SSM_ERR_ARG          # dx overlapping x
    assert call(db=FAKE + 0x4000010) == ssm.SSM_ERR_ARG     # dbias overlapping dweight


def test_ssd_bwd_argument_errors():
    def call(**kw):
        a = dict(x=FAKE, dt=FAKE + 0x1000000, bias=None, A=FAKE + 0x2000000, B=FAKE + 0x3000000,
                 C=FAKE + 0x4000000, D=None, z=None, flags=1, init=None, dy=FAKE + 0x5000000,
                 dfin=None, dx=FAKE + 0x6000000, ddt=FAKE + 0x7000000, dA=FAKE + 0x8000000,
                 dB=FAKE + 0x9000000, dC=FAKE + 0xA000000, dD=None, dz=None, dbias=None, dinit=None,
                 batch=1, L=64, H=4, P=64, G=1, N=64, ws=FAKE + 0x10000000, wsb=1 << 34)
        a.update(kw)
        return lib().ssm_ssd_bwd(a["x"], a["dt"], a["bias"], a["A"], a["B"], a["C"], a["D"], a["z"],
                                 a["flags"], a["init"], a["dy"], a["dfin"], a["dx"], a["ddt"], a["dA"],
                                 a["dB"], a["dC"], a["dD"], a["dz"], a["dbias"], a["dinit"], a["batch"],
                                 a["L"], a["H"], a["P"], a["G"], a["N"], a["ws"], a["wsb"], None)
    assert call(P=32) == ssm.SSM_ERR_UNSUPPORTED
    assert call(N=16) == ssm.SSM_ERR_UNSUPPORTED
    assert call(G=3) == ssm.SSM_ERR_UNSUPPORTED
    assert call(flags=ssm.SSM_LAYOUT_BLD) == ssm.SSM_ERR_ARG
    assert call(dz=FAKE + 0xB000000) == ssm.SSM_ERR_ARG      # dz without z
    assert call(dy=None) == ssm.SSM_ERR_ARG
    assert call(dA=None) == ssm.SSM_ERR_ARG
    assert call(dx=FAKE + 0x6000008) == ssm.SSM_ERR_ALIGN
    assert call(ws=None) == ssm.SSM_ERR_WORKSPACE
    assert call(wsb=1024) == ssm.SSM_ERR_WORKSPACE
    assert ssm.ssm_ssd_bwd_workspace_bytes(1, 64, 4, 64, 1, 64) > 0
    assert ssm.ssm_ssd_bwd_workspace_bytes(1, 64, 4, 64, 3, 64) == 0


def _strided(strides, **kw):
    import ctypes
    a = dict(u=FAKE, delta=FAKE + 0x1000000, A=FAKE + 0x2000000, B=FAKE + 0x3000000,
             C=FAKE + 0x4000000, z=FAKE + 0x6000000, softplus=1, y=FAKE + 0x5000000,
             batch=2, dim=64, L=128, N=16, io=ssm.SSM_BF16)
    a.update(kw)
    st = None if strides is None else (ctypes.c_int64 * 12)(*strides)
    return lib().ssm_scan_fwd_strided(a["u"], a["delta"], None, a["A"], a["B"], a["C"], None,
                                      a["z"], a["softplus"], a["y"], None, a["batch"], a["dim"],
                                      a["L"], a["N"], a["io"], st, None, None, 0, None)


def test_strided_argument_errors():
    dense = [64 * 128, 128, 1]
    bld = [64 * 128, 1, 64]
    # mixed orientations of u / delta / z are not supported
    assert _strided(dense + bld + dense + dense) == ssm.SSM_ERR_UNSUPPORTED
    # negative or zero strides over extents above one
    assert _strided([-1, 128, 1] + dense * 3) == ssm.SSM_ERR_ARG
    assert _strided(dense * 3 + [64 * 128, 0, 1]) == ssm.SSM_ERR_ARG
    # y writing one element twice (channel and time strides that collide)
    assert _strided(dense * 3 + [64 * 128, 1, 1]) == ssm.SSM_ERR_ARG
    # the layout flag with strides
    assert _strided(dense * 4, softplus=1 | ssm.SSM_LAYOUT_BLD) == ssm.SSM_ERR_ARG
    # y overlapping u's span
    assert _strided(dense * 4, y=FAKE + 0x200) == ssm.SSM_ERR_ARG
    # empty problems succeed without touching the device
    assert _strided(dense * 4, batch=0) == ssm.SSM_OK


def _cx(**kw):
    a = dict(u=FAKE, delta=FAKE + 0x1000000, bias=None, A=FAKE + 0x2000000, B=FAKE + 0x3000000,
             C=FAKE + 0x4000000, D=None, z=None, flags=1, y=FAKE + 0x5000000, h=None, init=None,
             batch=2, dim=64, L=128, N=16, io=ssm.SSM_BF16, stream=None)
    a.update(kw)
    return lib().ssm_scan_fwd_complex(a["u"], a["delta"], a["bias"], a["A"], a["B"], a["C"],
                                      a["D"], a["z"], a["flags"], a["y"], a["h"], a["init"],
                                      a["batch"], a["dim"], a["L"], a["N"], a["io"], a["stream"])


def test_complex_scan_argument_errors():
    assert _cx(io=3) == ssm.SSM_ERR_ARG
    assert _cx(flags=ssm.SSM_LAYOUT_BLD | 1) == ssm.SSM_ERR_ARG   # (batch, dim, L) only
    assert _cx(N=3) == ssm.SSM_ERR_UNSUPPORTED
    assert _cx(N=128) == ssm.SSM_ERR_UNSUPPORTED
    assert _cx(batch=-1) == ssm.SSM_ERR_ARG
    for name in ("u", "delta", "A", "B", "C", "y"):
        assert _cx(**{name: None}) == ssm.SSM_ERR_ARG, name
    assert _cx(B=FAKE + 0x3000008) == ssm.SSM_ERR_ALIGN
    assert _cx(h=FAKE + 0x6000004) == ssm.SSM_ERR_ALIGN
    # y over u; the final state over B; the final state partly over the initial one
    assert _cx(y=FAKE + 0x100) == ssm.SSM_ERR_ARG
    assert _cx(h=FAKE + 0x3000100) == ssm.SSM_ERR_ARG
    assert _cx(h=FAKE + 0x6000000, init=FAKE + 0x6000100) == ssm.SSM_ERR_ARG
    # nothing to do: no channel, or no step and no state asked for
    assert _cx(dim=0, u=None, delta=None, A=None, B=None, C=None, y=None) == ssm.SSM_OK
    assert _cx(L=0, h=None) == ssm.SSM_OK
